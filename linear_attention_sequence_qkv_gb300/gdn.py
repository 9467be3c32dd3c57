"""Python binding of the C ABI in ``include/gdn.h`` (ctypes; marshalling only).

Every step of the core forward runs in ``libgdn.so``'s CUDA kernels: this
module turns torch tensors into device pointers, strides into a ``gdn_desc``,
and a torch stream into a ``cudaStream_t``. PyTorch allocates the device
memory (outputs and workspace). There is no other implementation: if the
library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgdn.so")

GDN_OK = 0
GDN_ERR_INVALID_ARG = -1
GDN_ERR_UNSUPPORTED = -2
GDN_ERR_WORKSPACE = -3
GDN_ERR_CUDA = -4
GDN_ERR_DEVICE_SEQLENS = -5
GDN_ERR_DEVICE_RANGE = -6
GDN_ERR_DEVICE_TIMEOUT = -7

GDN_F32, GDN_BF16, GDN_F16 = 0, 1, 2
DTYPE_CODES = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16, torch.float16: GDN_F16}
ACT_TORCH = {GDN_F32: torch.float32, GDN_BF16: torch.bfloat16, GDN_F16: torch.float16}

# every entry point declared in include/gdn.h
EXPORTS = ("gdn_desc_init", "gdn_workspace_bytes", "gdn_workspace_offsets", "gdn_forward",
           "gdn_prologue", "gdn_chunk_rule", "gdn_epilogue", "gdn_device_status",
           "gdn_status_string", "gdn_chunk_kernel_kind", "gdn_forward_static_ws",
           "gdn_static_ws_device_status", "gdn_set_wait_test_mode",
           "gdn_decode_workspace_bytes", "gdn_decode_step", "gdn_backward_workspace_bytes",
           "gdn_backward", "gdn_forward_with_prefix", "gdn_span_scan")

# bytes of the library's fixed device scratch used by gdn_forward_static_ws
GDN_STATIC_WORKSPACE_BYTES = 16 * 1024 * 1024


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status} ({status_string(status)})")


class gdn_desc(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("T", ctypes.c_int32), ("N", ctypes.c_int32),
        ("Hk", ctypes.c_int32), ("Hv", ctypes.c_int32), ("dk", ctypes.c_int32),
        ("dv", ctypes.c_int32), ("conv_width", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("gate_dtype", ctypes.c_int32), ("norm_w_dtype", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("q_stride_b", ctypes.c_int64), ("q_stride_t", ctypes.c_int64),
        ("k_stride_b", ctypes.c_int64), ("k_stride_t", ctypes.c_int64),
        ("v_stride_b", ctypes.c_int64), ("v_stride_t", ctypes.c_int64),
        ("a_stride_b", ctypes.c_int64), ("a_stride_t", ctypes.c_int64),
        ("b_stride_b", ctypes.c_int64), ("b_stride_t", ctypes.c_int64),
        ("gate_stride_b", ctypes.c_int64), ("gate_stride_t", ctypes.c_int64),
        ("l2_eps", ctypes.c_float), ("norm_eps", ctypes.c_float), ("scale", ctypes.c_float),
        ("reserved1", ctypes.c_int32),
    ]


class gdn_workspace_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("status", "chunk_off", "q", "k", "v", "beta", "gamma", "o", "tpt", "total")]


_lib = None


def load(path: str = LIB_PATH):
    """Load ``libgdn.so`` (built in-tree by ``build.py``) and declare its ABI."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libgdn.so not built ({path}); run linear_attention_sequence_qkv_gb300/build.py")
    L = ctypes.CDLL(path)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    dp = ctypes.POINTER(gdn_desc)
    L.gdn_desc_init.argtypes = [dp, i32, i32, i32, i32, i32, i32, i32, i32]
    L.gdn_workspace_bytes.argtypes = [dp, ctypes.POINTER(sz)]
    L.gdn_workspace_offsets.argtypes = [dp, ctypes.POINTER(gdn_workspace_layout)]
    L.gdn_forward.argtypes = [dp] + [vp] * 14 + [vp, sz, vp]
    L.gdn_prologue.argtypes = [dp] + [vp] * 9 + [vp, sz, vp]
    L.gdn_chunk_rule.argtypes = [dp, vp, vp, vp, vp, sz, vp]
    L.gdn_epilogue.argtypes = [dp, vp, vp, vp, vp, sz, vp]
    L.gdn_device_status.argtypes = [vp, ctypes.POINTER(i32), vp]
    L.gdn_status_string.argtypes = [i32]
    L.gdn_status_string.restype = ctypes.c_char_p
    L.gdn_chunk_kernel_kind.argtypes = [dp]
    L.gdn_forward_static_ws.argtypes = [dp] + [vp] * 14 + [vp]
    L.gdn_static_ws_device_status.argtypes = [ctypes.POINTER(i32), vp]
    L.gdn_set_wait_test_mode.argtypes = [i32]
    L.gdn_decode_workspace_bytes.argtypes = [dp, ctypes.POINTER(sz)]
    L.gdn_decode_step.argtypes = [dp] + [vp] * 13 + [vp, sz, vp]
    L.gdn_forward_with_prefix.argtypes = [dp] + [vp] * 15 + [vp, sz, vp]
    L.gdn_span_scan.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp]
    L.gdn_backward_workspace_bytes.argtypes = [dp, ctypes.POINTER(sz)]
    L.gdn_backward.argtypes = [dp] + [vp] * 25 + [vp, sz, vp]
    for name in EXPORTS:
        if name != "gdn_status_string":
            getattr(L, name).restype = i32
    _lib = L
    return L


def status_string(status: int) -> str:
    return load().gdn_status_string(int(status)).decode()


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int, where: str):
    if rc != GDN_OK:
        raise GdnError(rc, where)


# ------------------------------------------------------------ raw ABI calls
def gdn_desc_init(B, T, packed, Hk, Hv, dk, dv, dtype) -> gdn_desc:
    d = gdn_desc()
    _check(load().gdn_desc_init(ctypes.byref(d), B, T, packed, Hk, Hv, dk, dv, dtype),
           "gdn_desc_init")
    return d


def gdn_workspace_bytes(d: gdn_desc) -> int:
    n = ctypes.c_size_t(0)
    _check(load().gdn_workspace_bytes(ctypes.byref(d), ctypes.byref(n)), "gdn_workspace_bytes")
    return n.value


def gdn_workspace_offsets(d: gdn_desc) -> gdn_workspace_layout:
    lay = gdn_workspace_layout()
    _check(load().gdn_workspace_offsets(ctypes.byref(d), ctypes.byref(lay)), "gdn_workspace_offsets")
    return lay


def gdn_forward(d, q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w,
                cu_seqlens, initial_state, out, final_state, workspace, workspace_bytes,
                stream=None, check=True) -> int:
    rc = load().gdn_forward(ctypes.byref(d), _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(a),
                            _ptr(b), _ptr(gate), _ptr(conv_w), _ptr(A_log), _ptr(dt_bias),
                            _ptr(norm_w), _ptr(cu_seqlens), _ptr(initial_state), _ptr(out),
                            _ptr(final_state), _ptr(workspace), int(workspace_bytes),
                            _stream(stream))
    if check:
        _check(rc, "gdn_forward")
    return rc


def gdn_forward_static_ws(d, q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w,
                          cu_seqlens, initial_state, out, final_state, stream=None,
                          check=True) -> int:
    """gdn_forward on the library's fixed device scratch (no workspace argument):
    for callers that cannot allocate device memory."""
    rc = load().gdn_forward_static_ws(ctypes.byref(d), _ptr(q_raw), _ptr(k_raw), _ptr(v_raw),
                                      _ptr(a), _ptr(b), _ptr(gate), _ptr(conv_w), _ptr(A_log),
                                      _ptr(dt_bias), _ptr(norm_w), _ptr(cu_seqlens),
                                      _ptr(initial_state), _ptr(out), _ptr(final_state),
                                      _stream(stream))
    if check:
        _check(rc, "gdn_forward_static_ws")
    return rc


def gdn_static_ws_device_status(stream=None) -> int:
    """Device status word of the last gdn_forward_static_ws call on the current device."""
    st = ctypes.c_int(0)
    _check(load().gdn_static_ws_device_status(ctypes.byref(st), _stream(stream)), "gdn_static_ws_device_status")
    return st.value


def gdn_set_wait_test_mode(immediate: int) -> None:
    """Test hook: 1 makes the tensor-core kernels' main-loop waits give up at once
    unless already complete (drives the GDN_ERR_DEVICE_TIMEOUT path); 0 restores them."""
    _check(load().gdn_set_wait_test_mode(int(immediate)), "gdn_set_wait_test_mode")


def gdn_prologue(d, q_raw, k_raw, v_raw, a, b, conv_w, A_log, dt_bias, cu_seqlens,
                 workspace, workspace_bytes, stream=None, check=True) -> int:
    rc = load().gdn_prologue(ctypes.byref(d), _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(a),
                             _ptr(b), _ptr(conv_w), _ptr(A_log), _ptr(dt_bias),
                             _ptr(cu_seqlens), _ptr(workspace), int(workspace_bytes),
                             _stream(stream))
    if check:
        _check(rc, "gdn_prologue")
    return rc


def gdn_chunk_rule(d, cu_seqlens, initial_state, final_state, workspace, workspace_bytes,
                   stream=None, check=True) -> int:
    rc = load().gdn_chunk_rule(ctypes.byref(d), _ptr(cu_seqlens), _ptr(initial_state),
                               _ptr(final_state), _ptr(workspace), int(workspace_bytes),
                               _stream(stream))
    if check:
        _check(rc, "gdn_chunk_rule")
    return rc


def gdn_epilogue(d, gate, norm_w, out, workspace, workspace_bytes, stream=None, check=True) -> int:
    rc = load().gdn_epilogue(ctypes.byref(d), _ptr(gate), _ptr(norm_w), _ptr(out),
                             _ptr(workspace), int(workspace_bytes), _stream(stream))
    if check:
        _check(rc, "gdn_epilogue")
    return rc


def gdn_device_status(workspace, stream=None) -> int:
    st = ctypes.c_int(0)
    _check(load().gdn_device_status(_ptr(workspace), ctypes.byref(st), _stream(stream)),
           "gdn_device_status")
    return st.value


def gdn_chunk_kernel_kind(d: gdn_desc) -> int:
    return load().gdn_chunk_kernel_kind(ctypes.byref(d))


def gdn_decode_workspace_bytes(d: gdn_desc) -> int:
    n = ctypes.c_size_t(0)
    _check(load().gdn_decode_workspace_bytes(ctypes.byref(d), ctypes.byref(n)),
           "gdn_decode_workspace_bytes")
    return n.value


def gdn_decode_step(d, q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w,
                    conv_state, state, out, workspace, workspace_bytes, stream=None,
                    check=True) -> int:
    rc = load().gdn_decode_step(ctypes.byref(d), _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(a),
                                _ptr(b), _ptr(gate), _ptr(conv_w), _ptr(A_log), _ptr(dt_bias),
                                _ptr(norm_w), _ptr(conv_state), _ptr(state), _ptr(out),
                                _ptr(workspace), int(workspace_bytes), _stream(stream))
    if check:
        _check(rc, "gdn_decode_step")
    return rc


def gdn_forward_with_prefix(d, q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w,
                            cu_seqlens, conv_prefix, initial_state, out, final_state, workspace,
                            workspace_bytes, stream=None, check=True) -> int:
    rc = load().gdn_forward_with_prefix(ctypes.byref(d), _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(a),
                                        _ptr(b), _ptr(gate), _ptr(conv_w), _ptr(A_log), _ptr(dt_bias),
                                        _ptr(norm_w), _ptr(cu_seqlens), _ptr(conv_prefix),
                                        _ptr(initial_state), _ptr(out), _ptr(final_state), _ptr(workspace),
                                        int(workspace_bytes), _stream(stream))
    if check:
        _check(rc, "gdn_forward_with_prefix")
    return rc


def gdn_span_scan(spans, Hv, dk, dv, A, B, h0, H_in, stream=None, check=True) -> int:
    rc = load().gdn_span_scan(int(spans), int(Hv), int(dk), int(dv), _ptr(A), _ptr(B), _ptr(h0), _ptr(H_in),
                              _stream(stream))
    if check:
        _check(rc, "gdn_span_scan")
    return rc


def gdn_backward_workspace_bytes(d: gdn_desc) -> int:
    n = ctypes.c_size_t(0)
    _check(load().gdn_backward_workspace_bytes(ctypes.byref(d), ctypes.byref(n)),
           "gdn_backward_workspace_bytes")
    return n.value


def gdn_backward(d, q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w, cu_seqlens,
                 initial_state, grad_out, grad_final, dq_raw, dk_raw, dv_raw, da, db, dgate, dconv_w,
                 dA_log, ddt_bias, dnorm_w, dinitial_state, workspace, workspace_bytes, stream=None,
                 check=True) -> int:
    rc = load().gdn_backward(ctypes.byref(d), _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(a), _ptr(b),
                             _ptr(gate), _ptr(conv_w), _ptr(A_log), _ptr(dt_bias), _ptr(norm_w),
                             _ptr(cu_seqlens), _ptr(initial_state), _ptr(grad_out), _ptr(grad_final),
                             _ptr(dq_raw), _ptr(dk_raw), _ptr(dv_raw), _ptr(da), _ptr(db), _ptr(dgate),
                             _ptr(dconv_w), _ptr(dA_log), _ptr(ddt_bias), _ptr(dnorm_w),
                             _ptr(dinitial_state), _ptr(workspace), int(workspace_bytes), _stream(stream))
    if check:
        _check(rc, "gdn_backward")
    return rc


# --------------------------------------------------- tensors -> descriptor
def desc_for(q_raw, k_raw, v_raw, a, b, gate, norm_w, *, Hk, Hv, dk, dv,
             cu_seqlens=None, l2_eps=1e-6, norm_eps=1e-5, scale=1.0) -> gdn_desc:
    """Descriptor for [B, T, C] views (channel stride 1) of the given tensors."""
    B, T = q_raw.shape[0], q_raw.shape[1]
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else 0
    d = gdn_desc_init(B, T, N, Hk, Hv, dk, dv, DTYPE_CODES[q_raw.dtype])
    for name, t in (("q", q_raw), ("k", k_raw), ("v", v_raw), ("a", a), ("b", b), ("gate", gate)):
        if t.shape[-1] > 1 and t.stride(2) != 1:
            raise ValueError(f"{name}: channel dimension must be contiguous")
        setattr(d, f"{name}_stride_b", t.stride(0))
        setattr(d, f"{name}_stride_t", t.stride(1))
    d.gate_dtype = DTYPE_CODES[gate.dtype]
    d.norm_w_dtype = DTYPE_CODES[norm_w.dtype]
    d.l2_eps, d.norm_eps, d.scale = l2_eps, norm_eps, scale
    return d


@dataclass
class Buffers:
    desc: gdn_desc
    out: torch.Tensor
    final_state: Optional[torch.Tensor]
    workspace: torch.Tensor

    @property
    def ws_bytes(self) -> int:
        return self.workspace.numel()

    def ws_view(self, name: str) -> torch.Tensor:
        """Typed view of one intermediate of the workspace (see gdn_workspace_offsets)."""
        d = self.desc
        lay = gdn_workspace_offsets(d)
        ntok = d.B * d.T
        # intermediates: fp16 for bf16/fp16 activations, fp32 for fp32; the
        # cumulative decay is fp64 for fp32 activations
        st = torch.float32 if d.dtype == GDN_F32 else torch.float16
        gt = torch.float64 if d.dtype == GDN_F32 else torch.float32
        qk = (d.Hk, ntok, d.dk) if d.dtype == GDN_F32 else (2, d.Hk, ntok, d.dk)  # hi, lo planes
        shapes = {"q": (qk, st), "k": (qk, st),
                  "v": ((d.Hv, ntok, d.dv), st), "beta": ((d.Hv, ntok), torch.float32),
                  "gamma": ((d.Hv, ntok), gt), "o": ((ntok, d.Hv, d.dv), st),
                  "status": ((1,), torch.int32), "chunk_off": ((d.N + 1,), torch.int32)}
        shape, dt = shapes[name]
        off = getattr(lay, name)
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dt).element_size()
        return self.workspace[off:off + nbytes].view(dt).view(shape)


def alloc(desc: gdn_desc, device, want_final_state=True) -> Buffers:
    """Allocate out, final_state and the workspace for ``desc`` with torch."""
    act = ACT_TORCH[desc.dtype]
    out = torch.empty((desc.B, desc.T, desc.Hv, desc.dv), dtype=act, device=device)
    fin = (torch.empty((desc.N, desc.Hv, desc.dk, desc.dv), dtype=torch.float32, device=device)
           if want_final_state else None)
    ws = torch.empty(gdn_workspace_bytes(desc), dtype=torch.uint8, device=device)
    return Buffers(desc, out, fin, ws)


def make_desc(inp) -> gdn_desc:
    w = inp.w
    return desc_for(inp.q_raw, inp.k_raw, inp.v_raw, inp.a, inp.b, inp.gate, inp.norm_w,
                    Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv, cu_seqlens=inp.cu_seqlens)


def forward(inp, bufs: Optional[Buffers] = None, stream=None, want_final_state=True) -> Buffers:
    """Run the core forward on an ``Inputs``-like object whose tensors live on
    the GPU (see ``workloads.Inputs``)."""
    if bufs is None:
        bufs = alloc(make_desc(inp), inp.q_raw.device, want_final_state)
    gdn_forward(bufs.desc, inp.q_raw, inp.k_raw, inp.v_raw, inp.a, inp.b, inp.gate, inp.conv_w,
                inp.A_log, inp.dt_bias, inp.norm_w, inp.cu_seqlens, inp.initial_state,
                bufs.out, bufs.final_state, bufs.workspace, bufs.ws_bytes, stream)
    return bufs


@dataclass
class Grads:
    dq_raw: torch.Tensor
    dk_raw: torch.Tensor
    dv_raw: torch.Tensor
    da: torch.Tensor
    db: torch.Tensor
    dgate: torch.Tensor
    dconv_w: torch.Tensor
    dA_log: torch.Tensor
    ddt_bias: torch.Tensor
    dnorm_w: torch.Tensor
    dinitial_state: Optional[torch.Tensor]
    workspace: torch.Tensor


def alloc_grads(desc: gdn_desc, device, want_dinitial=True) -> Grads:
    """Gradient buffers (dense, see gdn_backward in include/gdn.h) and the workspace."""
    act = ACT_TORCH[desc.dtype]
    ntok = desc.B * desc.T
    ch_qk, ch_v = desc.Hk * desc.dk, desc.Hv * desc.dv
    f32 = dict(dtype=torch.float32, device=device)
    return Grads(
        dq_raw=torch.empty((ntok, ch_qk), dtype=act, device=device),
        dk_raw=torch.empty((ntok, ch_qk), dtype=act, device=device),
        dv_raw=torch.empty((ntok, ch_v), dtype=act, device=device),
        da=torch.empty((ntok, desc.Hv), dtype=act, device=device),
        db=torch.empty((ntok, desc.Hv), dtype=act, device=device),
        dgate=torch.empty((ntok, ch_v), dtype=ACT_TORCH[desc.gate_dtype], device=device),
        dconv_w=torch.empty((2 * ch_qk + ch_v, 4), **f32), dA_log=torch.empty(desc.Hv, **f32),
        ddt_bias=torch.empty(desc.Hv, **f32), dnorm_w=torch.empty(desc.dv, **f32),
        dinitial_state=torch.empty((desc.N, desc.Hv, desc.dk, desc.dv), **f32) if want_dinitial else None,
        workspace=torch.empty(gdn_backward_workspace_bytes(desc), dtype=torch.uint8, device=device))


def backward(inp, grad_out, grad_final=None, grads: Optional[Grads] = None, stream=None) -> Grads:
    """Gradients of sum(grad_out * out) + sum(grad_final * final_state) for an
    ``Inputs``-like object on the GPU (grad_out [B, T, Hv, dv] act dtype,
    contiguous; grad_final [N, Hv, dk, dv] fp32 or None)."""
    d = make_desc(inp)
    if grads is None:
        grads = alloc_grads(d, inp.q_raw.device)
    gdn_backward(d, inp.q_raw, inp.k_raw, inp.v_raw, inp.a, inp.b, inp.gate, inp.conv_w, inp.A_log,
                 inp.dt_bias, inp.norm_w, inp.cu_seqlens, inp.initial_state, grad_out, grad_final,
                 grads.dq_raw, grads.dk_raw, grads.dv_raw, grads.da, grads.db, grads.dgate, grads.dconv_w,
                 grads.dA_log, grads.ddt_bias, grads.dnorm_w, grads.dinitial_state, grads.workspace,
                 grads.workspace.numel(), stream)
    return grads
