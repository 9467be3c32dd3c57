"""Host logic of bench.py, no GPU: the roofline arithmetic and the staging arena
of the end-to-end measurement.

The chunk rule's algorithmic MMA flops are recounted here product by product from
the chunked WY/UT form of the gated delta rule (chunk C = 64; per chunk and v head:
K K^T, Q K^T, W = T (beta K), U = T (beta V), W H, Q H, P (U - W H), the state
update K^T (U - W H), and the triangular solve's C^3 / 3 multiply-adds), not from
the per-token formula bench.py uses, and must agree with it; the bytes are the
reads of q, k, v (activation dtype), beta and gamma (fp32), the write of o and the
final state (and the read of an initial one).
"""
from types import SimpleNamespace

import pytest
import torch

import bench
from linear_attention_sequence_qkv_gb300.workloads import WORKLOADS, replace


def chunk_rule_flops_by_products(w, ntok):
    C, dk, dv = bench.CHUNK, w.dk, w.dv
    mm = lambda m, n, k: 2 * m * n * k
    per_chunk = (mm(C, C, dk) + mm(C, C, dk)              # K K^T, Q K^T
                 + mm(C, dk, C) + mm(C, dv, C)            # W = T (beta K), U = T (beta V)
                 + mm(C, dv, dk) + mm(C, dv, dk)          # W H, Q H
                 + mm(C, dv, C)                           # P (U - W H)
                 + mm(dk, dv, C)                          # H += K^T (U - W H)
                 + 2 * C ** 3 / 3)                        # (I + A)^{-1}, forward substitution
    return per_chunk * (ntok / C) * w.Hv


@pytest.mark.parametrize("name", ["layer_bf16", "long_gqa_bf16", "tiny_fp32"])
def test_chunk_rule_flops_match_the_products(name):
    w = WORKLOADS[name]
    ntok = w.B * w.T
    _, flops = bench.algorithmic(w, ntok, w.B, False)["chunk_rule"]
    assert flops == pytest.approx(chunk_rule_flops_by_products(w, ntok), rel=1e-12)


def test_layer_figures():
    w = WORKLOADS["layer_bf16"]
    alg = bench.algorithmic(w, 4096, 2, False)
    # q, k (2 x 6 x 256) and v (6 x 512) at 2 bytes, beta and gamma fp32 per v head,
    # o at 2 bytes, and the final fp32 state of 2 sequences x 6 heads x 256 x 512
    assert alg["chunk_rule"][0] == 4096 * (6144 * 2 + 6 * 8 + 3072 * 2) + 2 * 6 * 256 * 512 * 4
    assert alg["chunk_rule"][1] == 25_031_606_272
    # the prologue reads raw q|k|v, a, b and writes q, k, v, beta, gamma; the epilogue
    # reads o and the gate and writes out
    assert alg["prologue"][0] == 4096 * (2 * 6144 * 2 + 2 * 6 * 2 + 6 * 8)
    assert alg["epilogue"][0] == 4096 * 3 * 3072 * 2


def test_roofline_entry_takes_the_binding_resource():
    pk = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0}
    # 1 GB and 1 TFLOP: 1 ms of HBM against 10 ms of MMA -> tensor-bound
    e = bench.roofline_entry("x", 1e9, 1e12, 20.0, pk, "bf16")
    assert e["bound"] == "tensor" and e["achieved"] == pytest.approx(50.0) and e["frac"] == pytest.approx(0.5)
    # 1 GB and 1 GFLOP -> HBM-bound
    e = bench.roofline_entry("x", 1e9, 1e9, 2.0, pk, "bf16")
    assert e["bound"] == "hbm" and e["achieved"] == pytest.approx(500.0) and e["frac"] == pytest.approx(0.5)
    # fp32 activations run on the CUDA cores: never reported against the bf16 tensor peak
    assert bench.roofline_entry("x", 1e9, 1e12, 20.0, pk, "fp32")["bound"] == "hbm"


def test_chunk_segments():
    nsm = 152
    seq = lambda w: (w, SimpleNamespace(T=w.T, N=w.B), SimpleNamespace(cu_seqlens=None))
    # one 131072-token sequence, 32 transposed-chain CTAs: 2048 chunks cut into 16 segments
    assert bench.chunk_segments(*seq(WORKLOADS["long_gqa_bf16"]), nsm) == 16
    # two sequences, or short ones, or chains filling more than half of the SMs: one
    assert bench.chunk_segments(*seq(WORKLOADS["layer_bf16"]), nsm) == 1
    assert bench.chunk_segments(*seq(replace(WORKLOADS["long_gqa_bf16"], T=255 * 64)), nsm) == 1
    assert bench.chunk_segments(*seq(replace(WORKLOADS["long_gqa_bf16"], Hv=80, Hk=16)), nsm) == 1
    w = WORKLOADS["varlen_bf16"]
    assert bench.chunk_segments(w, SimpleNamespace(T=w.T, N=64), SimpleNamespace(cu_seqlens=object()), nsm) == 1


def test_arena_views():
    ts = [torch.randn(3, 5).to(torch.bfloat16), torch.arange(7, dtype=torch.int32),
          torch.randn(2, 3, 4, dtype=torch.float32), torch.zeros(0, 8, dtype=torch.float16)]
    buf, views = bench.arena(ts, "cpu")
    assert buf.dtype == torch.uint8 and buf.dim() == 1
    # byte offsets of the views in the arena (the storage is the arena's own)
    starts = [v.storage_offset() * v.element_size() for v in views]
    ends = [a + v.numel() * v.element_size() for a, v in zip(starts, views)]
    for v, t, a in zip(views, ts, starts):
        assert v.untyped_storage().data_ptr() == buf.untyped_storage().data_ptr()
        assert v.dtype == t.dtype and v.shape == t.shape and v.is_contiguous()
        assert a % 256 == 0
        v.copy_(t)
    for v, t in zip(views, ts):
        assert torch.equal(v, t)
    # back to back: each view starts at the first 256-byte boundary after the last
    assert starts[0] == 0
    for e, a in zip(ends[:-1], starts[1:]):
        assert a == (e + 255) // 256 * 256
    assert buf.numel() == ends[-1]
