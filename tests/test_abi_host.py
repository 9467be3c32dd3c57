"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point declared in include/gdn.h, and rejects bad arguments with
status codes on metadata alone, before anything is launched."""
import ctypes
import os
import re

import pytest

from linear_attention_sequence_qkv_gb300 import build, gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gdn.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(gdn_\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(gdn.EXPORTS)


def declared_arity():
    """Parameter count of every prototype in include/gdn.h."""
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    out = {}
    for m in re.finditer(r"(gdn_\w+)\s*\(", src):
        name, i, depth = m.group(1), m.end(), 1
        j = i
        while depth:
            depth += {"(": 1, ")": -1}.get(src[j], 0)
            j += 1
        params = src[i:j - 1].strip()
        if src[j:].lstrip().startswith(";") or src[j:].lstrip().startswith("{"):
            out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argument_counts_match_header(lib):
    # the ctypes declarations must take exactly the parameters the header declares
    arity = declared_arity()
    assert set(arity) == set(gdn.EXPORTS)
    for name, n in arity.items():
        assert len(getattr(lib, name).argtypes) == n, name


def test_library_is_native_and_sm103a():
    # the built library exists and was compiled for sm_103a only
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.ARCH)
    assert os.path.exists(gdn.LIB_PATH)


def test_static_workspace_size_matches_header():
    # the binding's copy of GDN_STATIC_WORKSPACE_BYTES is the header's #define
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    m = re.search(r"#define\s+GDN_STATIC_WORKSPACE_BYTES\s+\(([^)]*)\)", src)
    assert m is not None
    expr = re.sub(r"(\d+)u\b", r"\1", m.group(1))
    assert re.fullmatch(r"[\d\s*+]+", expr)
    assert eval(expr) == gdn.GDN_STATIC_WORKSPACE_BYTES


def test_struct_layout_matches_header(lib):
    # gdn_desc: 12 int32 + 12 int64 + 3 float + 1 int32 = 160 bytes
    assert ctypes.sizeof(gdn.gdn_desc) == 160
    assert ctypes.sizeof(gdn.gdn_workspace_layout) == 10 * 8


@pytest.mark.parametrize("args,status", [
    ((2, 2048, 0, 6, 6, 100, 512, gdn.GDN_BF16), gdn.GDN_ERR_UNSUPPORTED),  # dk not pow2
    ((2, 2048, 0, 6, 6, 256, 1024, gdn.GDN_BF16), gdn.GDN_ERR_UNSUPPORTED),  # dv > 512
    ((2, 2048, 0, 4, 6, 64, 64, gdn.GDN_BF16), gdn.GDN_ERR_UNSUPPORTED),    # Hv % Hk
    ((2, 2048, 0, 6, 6, 64, 64, 7), gdn.GDN_ERR_UNSUPPORTED),               # dtype
    ((0, 2048, 0, 6, 6, 64, 64, gdn.GDN_F32), gdn.GDN_ERR_INVALID_ARG),     # B
    ((2, -1, 0, 6, 6, 64, 64, gdn.GDN_F32), gdn.GDN_ERR_INVALID_ARG),       # T
    ((2, 100, 3, 6, 6, 64, 64, gdn.GDN_F32), gdn.GDN_ERR_INVALID_ARG),      # packed needs B == 1
])
def test_desc_validation(lib, args, status):
    d = gdn.gdn_desc()
    assert lib.gdn_desc_init(ctypes.byref(d), *args) == status


def test_valid_descs(lib):
    for args in ((1, 128, 0, 2, 2, 64, 64, gdn.GDN_F32), (2, 2048, 0, 6, 6, 256, 512, gdn.GDN_BF16),
                 (2, 100, 0, 6, 6, 64, 128, gdn.GDN_F16), (1, 131072, 0, 16, 32, 128, 128, gdn.GDN_BF16),
                 (1, 263156, 64, 16, 32, 128, 128, gdn.GDN_BF16), (1, 0, 0, 1, 1, 16, 16, gdn.GDN_F32)):
        gdn.gdn_desc_init(*args)


def test_conv_width_and_strides_checked(lib):
    d = gdn.gdn_desc_init(2, 100, 0, 6, 6, 64, 128, gdn.GDN_F16)
    d.conv_width = 3
    assert lib.gdn_forward(ctypes.byref(d), *([None] * 14), None, 0, None) == gdn.GDN_ERR_UNSUPPORTED
    d = gdn.gdn_desc_init(2, 100, 0, 6, 6, 64, 128, gdn.GDN_F16)
    d.q_stride_t = 6 * 64 + 3   # rows not 16-byte aligned
    assert lib.gdn_forward(ctypes.byref(d), *([None] * 14), None, 0, None) == gdn.GDN_ERR_INVALID_ARG
    d = gdn.gdn_desc_init(2, 100, 0, 6, 6, 64, 128, gdn.GDN_F16)
    d.gate_dtype = gdn.GDN_BF16
    assert lib.gdn_forward(ctypes.byref(d), *([None] * 14), None, 0, None) == gdn.GDN_ERR_UNSUPPORTED


def test_null_and_workspace_checks(lib):
    d = gdn.gdn_desc_init(1, 128, 0, 2, 2, 64, 64, gdn.GDN_F32)
    fake = 1 << 20   # never dereferenced: every call below fails its checks first
    ptrs = [fake] * 10   # q_raw .. norm_w
    # null q_raw
    rc = lib.gdn_forward(ctypes.byref(d), None, *ptrs[1:], None, None, fake, None, fake,
                         gdn.gdn_workspace_bytes(d), None)
    assert rc == gdn.GDN_ERR_INVALID_ARG
    # workspace too small
    rc = lib.gdn_forward(ctypes.byref(d), *ptrs, None, None, fake, None, fake, 256, None)
    assert rc == gdn.GDN_ERR_WORKSPACE
    # workspace misaligned
    rc = lib.gdn_forward(ctypes.byref(d), *ptrs, None, None, fake, None, fake + 16,
                         gdn.gdn_workspace_bytes(d), None)
    assert rc == gdn.GDN_ERR_WORKSPACE
    # misaligned out
    rc = lib.gdn_forward(ctypes.byref(d), *ptrs, None, None, fake + 4, None, fake,
                         gdn.gdn_workspace_bytes(d), None)
    assert rc == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_device_status(None, None, None) == gdn.GDN_ERR_INVALID_ARG


def test_workspace_layout(lib):
    d = gdn.gdn_desc_init(2, 2048, 0, 6, 6, 256, 512, gdn.GDN_BF16)
    lay = gdn.gdn_workspace_offsets(d)
    ntok = 4096
    assert lay.status == 0
    for name in ("chunk_off", "q", "k", "v", "beta", "gamma", "o", "tpt", "total"):
        assert getattr(lay, name) % 256 == 0
    assert lay.k - lay.q >= ntok * 6 * 256 * 2
    assert lay.beta - lay.v >= ntok * 6 * 512 * 2
    assert lay.tpt - lay.o >= ntok * 6 * 512 * 2
    assert lay.total - lay.tpt >= 6 * (ntok // 64) * 128 * 64 * 2
    assert gdn.gdn_workspace_bytes(d) == lay.total


def test_status_strings(lib):
    for s in (0, -1, -2, -3, -4, -5, -6, -7):
        assert gdn.status_string(s) not in ("", "unknown status")
    assert gdn.status_string(42) == "unknown status"


def test_chunk_kernel_kind(lib):
    assert gdn.gdn_chunk_kernel_kind(gdn.gdn_desc_init(1, 128, 0, 2, 2, 64, 64, gdn.GDN_F32)) == 0
    assert gdn.gdn_chunk_kernel_kind(gdn.gdn_desc_init(2, 2048, 0, 6, 6, 256, 512, gdn.GDN_BF16)) == 1
    assert gdn.gdn_chunk_kernel_kind(gdn.gdn_desc_init(2, 100, 0, 6, 6, 64, 128, gdn.GDN_F16)) == 1
    assert gdn.gdn_chunk_kernel_kind(gdn.gdn_desc_init(1, 70, 0, 1, 1, 512, 512, gdn.GDN_BF16)) == 0
    assert gdn.gdn_chunk_kernel_kind(gdn.gdn_desc_init(1, 70, 0, 1, 1, 64, 32, gdn.GDN_BF16)) == 0


def test_decode_checks(lib):
    """The decode entry rejects non-decode descriptors and bad pointers before any launch."""
    fake = 1 << 20   # never dereferenced: every call below fails its checks first
    d = gdn.gdn_desc_init(4, 1, 0, 2, 4, 64, 128, gdn.GDN_BF16)
    need = gdn.gdn_decode_workspace_bytes(d)
    # fp32 q, k, v of the token, beta and g, fp16 o, after a 256-byte status block
    B, Hk, Hv, dk, dv = 4, 2, 4, 64, 128
    assert need >= 256 + 4 * B * (2 * Hk * dk + Hv * dv + 2 * Hv) + 2 * B * Hv * dv
    args = [fake] * 13   # q_raw .. out

    def call(desc, a=None, ws=fake, nbytes=None):
        a = args if a is None else a
        return lib.gdn_decode_step(ctypes.byref(desc), *a, ws, need if nbytes is None else nbytes, None)

    multi = gdn.gdn_desc_init(4, 8, 0, 2, 4, 64, 128, gdn.GDN_BF16)   # T = 8: not a decode step
    n = ctypes.c_size_t(0)
    assert lib.gdn_decode_workspace_bytes(ctypes.byref(multi), ctypes.byref(n)) == gdn.GDN_ERR_INVALID_ARG
    assert call(multi) == gdn.GDN_ERR_INVALID_ARG
    packed = gdn.gdn_desc_init(1, 1, 4, 2, 4, 64, 128, gdn.GDN_BF16)  # cu_seqlens-style descriptor
    assert call(packed) == gdn.GDN_ERR_INVALID_ARG
    for i in range(13):                     # each pointer null in turn
        a = list(args)
        a[i] = None
        assert call(d, a) == gdn.GDN_ERR_INVALID_ARG, i
    a = list(args)
    a[12] = fake + 4                        # out not 16-byte aligned
    assert call(d, a) == gdn.GDN_ERR_INVALID_ARG
    a = list(args)
    a[11] = fake + 8                        # state not 16-byte aligned
    assert call(d, a) == gdn.GDN_ERR_INVALID_ARG
    assert call(d, nbytes=need - 1) == gdn.GDN_ERR_WORKSPACE
    assert call(d, ws=fake + 16) == gdn.GDN_ERR_WORKSPACE
    bad = gdn.gdn_desc_init(4, 1, 0, 2, 4, 64, 128, gdn.GDN_BF16)
    bad.dk = 48                             # not a power of two
    assert call(bad) == gdn.GDN_ERR_UNSUPPORTED


def test_backward_checks(lib):
    """The backward entry rejects bad pointers and workspaces before any launch."""
    fake = 1 << 20   # never dereferenced: every call below fails its checks first
    d = gdn.gdn_desc_init(2, 100, 0, 2, 4, 64, 128, gdn.GDN_BF16)
    need = gdn.gdn_backward_workspace_bytes(d)
    B, T, Hk, Hv, dk, dv = 2, 100, 2, 4, 64, 128
    ntok, slots = B * T, (B * T + 63) // 64 + B
    # the forward's workspace, then per chunk slot two states and three 64x64
    # matrices, and per token the fp32 rows of the reverse pass
    assert need >= gdn.gdn_workspace_bytes(d) + slots * Hv * (2 * dk * dv + 3 * 64 * 64) * 4 + \
        ntok * Hv * (3 * dv + 2 * dk + 4) * 4 + ntok * (2 * Hk * dk + Hv * dv) * 4
    args = [fake] * 25   # q_raw .. dinitial_state
    args[10] = None      # cu_seqlens: not packed
    optional = {10, 11, 13, 24}   # cu_seqlens, initial_state, grad_final, dinitial_state

    def call(desc, a=None, ws=fake, nbytes=None):
        a = args if a is None else a
        return lib.gdn_backward(ctypes.byref(desc), *a, ws, need if nbytes is None else nbytes, None)

    for i in range(25):
        if i in optional:
            continue
        a = list(args)
        a[i] = None
        assert call(d, a) == gdn.GDN_ERR_INVALID_ARG, i
    for i in (0, 1, 2, 6, 14, 15, 16):      # vector-loaded inputs and vector-stored input
                                            # gradients must be 16-byte aligned
        a = list(args)
        a[i] = fake + 2
        assert call(d, a) == gdn.GDN_ERR_INVALID_ARG, i
    for i in (11, 13, 24):                  # fp32 states must be 16-byte aligned
        a = list(args)
        a[i] = fake + 4
        assert call(d, a) == gdn.GDN_ERR_INVALID_ARG, i
    assert call(d, nbytes=need - 1) == gdn.GDN_ERR_WORKSPACE
    assert call(d, ws=fake + 16) == gdn.GDN_ERR_WORKSPACE
    bad = gdn.gdn_desc_init(2, 100, 0, 2, 4, 64, 128, gdn.GDN_BF16)
    bad.dv = 96                             # not a power of two
    assert call(bad) == gdn.GDN_ERR_UNSUPPORTED


def test_prefix_and_span_scan_checks(lib):
    fake = 1 << 20
    d = gdn.gdn_desc_init(2, 100, 0, 2, 4, 64, 128, gdn.GDN_BF16)
    need = gdn.gdn_workspace_bytes(d)
    args = [fake] * 15   # q_raw .. final_state
    args[10] = None      # cu_seqlens
    args[11] = fake + 8  # conv_prefix not 16-byte aligned
    assert lib.gdn_forward_with_prefix(ctypes.byref(d), *args, fake, need, None) == gdn.GDN_ERR_INVALID_ARG
    # span scan: sizes and pointers checked before any launch
    assert lib.gdn_span_scan(0, 4, 64, 64, None, None, None, None, None) == gdn.GDN_OK
    assert lib.gdn_span_scan(2, 4, 48, 64, fake, fake, None, fake, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_span_scan(2, 0, 64, 64, fake, fake, None, fake, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_span_scan(2, 4, 64, 64, None, fake, None, fake, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_span_scan(2, 4, 64, 64, fake + 4, fake, None, fake, None) == gdn.GDN_ERR_INVALID_ARG
