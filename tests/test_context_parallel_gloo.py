"""The exchange of the sequence-sharded core across ranks, on CPU: gloo,
world size 2, the collectives of context_parallel (conv-prefix tails and the
span maps) with rank-tagged tensors. The GPU steps around them are covered by
tests/test_context_parallel_gpu.py."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from linear_attention_sequence_qkv_gb300 import context_parallel as cp
        ch, Hv, dk, dv = 12, 2, 4, 6
        T = 5 + rank
        base = 100.0 * rank
        q = (base + torch.arange(T * 4, dtype=torch.float32)).reshape(1, T, 4)
        k = (base + 50 + torch.arange(T * 4, dtype=torch.float32)).reshape(1, T, 4)
        v = (base + 70 + torch.arange(T * 4, dtype=torch.float32)).reshape(1, T, 4)
        tail = cp.tail_tokens(q, k, v)
        pre = cp.exchange_tails(tail, None)
        A = torch.full((Hv, dk, dk), float(rank + 1))
        B = torch.full((Hv, dk, dv), float(-(rank + 1)))
        A_all, B_all = cp.gather_maps(A, B, None)
        results.put((rank, tail, pre, A_all, B_all))
    finally:
        dist.destroy_process_group()


def test_exchange_two_ranks():
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        r, tail, pre, A_all, B_all = results.get(timeout=90)
        res[r] = (tail, pre, A_all, B_all)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # rank 0's prefix is zeros, rank 1's is rank 0's last three raw tokens
    assert torch.equal(res[0][1], torch.zeros(1, 3, 12))
    assert torch.equal(res[1][1][0], res[0][0])
    # the tail is the last three tokens of q | k | v
    t0 = res[0][0]
    assert t0.shape == (3, 12) and t0[0, 0].item() == 8.0 and t0[2, 4].item() == 50.0 + 4 * 4
    for r in range(2):
        A_all, B_all = res[r][2], res[r][3]
        assert A_all.shape == (2, 2, 4, 4) and B_all.shape == (2, 2, 4, 6)
        assert [A_all[s, 0, 0, 0].item() for s in range(2)] == [1.0, 2.0]
        assert [B_all[s, 0, 0, 0].item() for s in range(2)] == [-1.0, -2.0]


def test_short_span_rejected():
    from linear_attention_sequence_qkv_gb300 import context_parallel as cp
    x = torch.zeros(1, 2, 4)
    with pytest.raises(ValueError):
        cp.tail_tokens(x, x, x)
