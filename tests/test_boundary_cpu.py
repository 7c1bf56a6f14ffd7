"""Host-side checks of the C ABI (no GPU work is ever launched here).

The library must load, export every function include/m3scan.h declares, and
reject invalid or unsupported arguments on the host with the documented
status before touching a device.
"""
import ctypes
import os
import re

import pytest

from selective_state_space_129_b300 import m3scan

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000  # aligned, never dereferenced: validation fails before any device call


def _declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(m3_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    return m3scan.load()


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert len(declared) >= 6
    raw = ctypes.CDLL(m3scan.LIB_PATH)
    for name in declared:
        assert hasattr(raw, name), name
    assert set(declared) == set(m3scan.EXPORTS)


def test_status_strings(lib):
    assert m3scan.m3_status_string(0) == "M3_OK"
    assert m3scan.m3_status_string(4) == "M3_ERR_TIMEOUT"
    assert m3scan.m3_status_string(99) == "M3_ERR_UNKNOWN"
    assert m3scan.m3_version() >= 100


def _dims(**kw):
    base = dict(batch=2, seqlen=16, heads=4, groups=2, headdim=8, dstate=8,
                act_dtype=m3scan.M3_F32)
    base.update(kw)
    return m3scan.make_dims(**base)


def _scan(lib, dims, R=1, chunk=4, **ptrs):
    p = dict(x=FAKE, dt=FAKE, A=FAKE, lam=FAKE, B=FAKE, C=FAKE, theta=FAKE, out=FAKE, fs=FAKE)
    p.update(ptrs)
    v = lambda k: ctypes.c_void_p(p[k]) if p[k] else None
    return lib.m3_scan_fwd(v("x"), v("dt"), v("A"), v("lam"), v("B"), v("C"), v("theta"),
                           ctypes.byref(dims), R, chunk, v("out"), v("fs"), None)


def _decode(lib, dims, R=1, **ptrs):
    p = dict(state=FAKE, x=FAKE, dt=FAKE, A=FAKE, lam=FAKE, Bp=0, xp=0, B=FAKE, C=FAKE,
             theta=FAKE, out=FAKE)
    p.update(ptrs)
    v = lambda k: ctypes.c_void_p(p[k]) if p[k] else None
    return lib.m3_decode_step(v("state"), v("x"), v("dt"), v("A"), v("lam"), v("Bp"), v("xp"),
                              v("B"), v("C"), v("theta"), ctypes.byref(dims), R, v("out"), None)


@pytest.mark.parametrize("missing", ["x", "dt", "A", "lam", "B", "C", "theta", "out"])
def test_scan_null_pointer(lib, missing):
    assert _scan(lib, _dims(), **{missing: 0}) == m3scan.M3_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,R,chunk,expect", [
    (dict(dstate=7), 1, 4, m3scan.M3_ERR_INVALID_ARG),        # odd N
    (dict(groups=3), 1, 4, m3scan.M3_ERR_INVALID_ARG),        # G does not divide H
    (dict(batch=-1), 1, 4, m3scan.M3_ERR_INVALID_ARG),
    (dict(seqlen=-5), 1, 4, m3scan.M3_ERR_INVALID_ARG),
    (dict(heads=0), 1, 4, m3scan.M3_ERR_INVALID_ARG),
    (dict(), 0, 4, m3scan.M3_ERR_INVALID_ARG),                # R < 1
    (dict(), 1, 0, m3scan.M3_ERR_INVALID_ARG),                # chunk < 1
    (dict(act_dtype=7), 1, 4, m3scan.M3_ERR_UNSUPPORTED),     # unknown dtype
    (dict(), 1, 5000, m3scan.M3_ERR_UNSUPPORTED),             # chunk too long
    (dict(dstate=4096, headdim=512), 1, 64, m3scan.M3_ERR_UNSUPPORTED),  # tiles exceed smem
])
def test_scan_rejects(lib, kw, R, chunk, expect):
    assert _scan(lib, _dims(**kw), R=R, chunk=chunk) == expect


def test_scan_misaligned_pointer(lib):
    assert _scan(lib, _dims(), x=FAKE + 2) == m3scan.M3_ERR_INVALID_ARG
    d = _dims(act_dtype=m3scan.M3_BF16)
    assert _scan(lib, d, x=FAKE + 1) == m3scan.M3_ERR_INVALID_ARG


def test_scan_unknown_flags_are_rejected(lib):
    for bit in (2, 4, 1 << 30):
        d = _dims()
        d.flags = bit
        assert _scan(lib, d) == m3scan.M3_ERR_INVALID_ARG
        d.flags = bit | m3scan.M3_FLAG_BC_NORM
        assert _scan(lib, d) == m3scan.M3_ERR_INVALID_ARG


def test_bc_norm_outside_the_tensor_core_prefill_is_unsupported(lib):
    # fp32 activations take the CUDA-core path, which has no fused BCNorm
    d = _dims(act_dtype=m3scan.M3_F32)
    d.flags = m3scan.M3_FLAG_BC_NORM
    assert _scan(lib, d) == m3scan.M3_ERR_UNSUPPORTED
    # a bf16 shape outside the tensor-core scope (P = 16) likewise
    d = _dims(act_dtype=m3scan.M3_BF16)
    d.flags = m3scan.M3_FLAG_BC_NORM
    assert _scan(lib, d) == m3scan.M3_ERR_UNSUPPORTED


def test_bc_norm_is_unsupported_by_decode_continuation_and_backward(lib):
    v = ctypes.c_void_p(FAKE)
    d = _dims()
    d.flags = m3scan.M3_FLAG_BC_NORM
    assert lib.m3_decode_step(v, v, v, v, v, None, None, v, v, v, ctypes.byref(d), 1, v,
                              None) == m3scan.M3_ERR_UNSUPPORTED
    assert lib.m3_decode_tokens(v, v, v, v, v, None, None, v, v, v, ctypes.byref(d), 1, v,
                                None) == m3scan.M3_ERR_UNSUPPORTED
    assert lib.m3_scan_fwd_state(v, v, v, v, v, v, v, None, None, ctypes.byref(d), 1, 4, v, v,
                                 None) == m3scan.M3_ERR_UNSUPPORTED
    assert lib.m3_scan_bwd(v, v, v, v, v, v, v, v, None, ctypes.byref(d), 1, v, v, v, v, v, v, v,
                           None, None, None) == m3scan.M3_ERR_UNSUPPORTED


def test_scan_null_dims(lib):
    v = ctypes.c_void_p(FAKE)
    assert lib.m3_scan_fwd(v, v, v, v, v, v, v, None, 1, 4, v, v, None) == \
        m3scan.M3_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,R,expect", [
    (dict(headdim=6), 1, m3scan.M3_ERR_UNSUPPORTED),   # P not a multiple of 4
    (dict(), 3, m3scan.M3_ERR_UNSUPPORTED),            # R outside {1, 2, 4}
    (dict(dstate=5), 1, m3scan.M3_ERR_INVALID_ARG),
])
def test_decode_rejects(lib, kw, R, expect):
    assert _decode(lib, _dims(**kw), R=R) == expect


def test_decode_prev_pointers_come_in_pairs(lib):
    assert _decode(lib, _dims(), Bp=FAKE) == m3scan.M3_ERR_INVALID_ARG
    assert _decode(lib, _dims(), xp=FAKE) == m3scan.M3_ERR_INVALID_ARG


def test_decode_state_alignment(lib):
    assert _decode(lib, _dims(), state=FAKE + 4) == m3scan.M3_ERR_INVALID_ARG


def _tokens(lib, dims, R=1, **ptrs):
    p = dict(state=FAKE, x=FAKE, dt=FAKE, A=FAKE, lam=FAKE, Bp=0, xp=0, B=FAKE, C=FAKE,
             theta=FAKE, out=FAKE)
    p.update(ptrs)
    v = lambda k: ctypes.c_void_p(p[k]) if p[k] else None
    return lib.m3_decode_tokens(v("state"), v("x"), v("dt"), v("A"), v("lam"), v("Bp"), v("xp"),
                                v("B"), v("C"), v("theta"), ctypes.byref(dims), R, v("out"), None)


@pytest.mark.parametrize("missing", ["state", "x", "dt", "A", "lam", "B", "C", "theta", "out"])
def test_tokens_null_pointer(lib, missing):
    assert _tokens(lib, _dims(), **{missing: 0}) == m3scan.M3_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,R,ptrs,expect", [
    (dict(headdim=6), 1, {}, m3scan.M3_ERR_UNSUPPORTED),           # P not a multiple of 4
    (dict(), 3, {}, m3scan.M3_ERR_UNSUPPORTED),                    # R outside {1, 2, 4}
    (dict(dstate=512, headdim=64), 1, {}, m3scan.M3_ERR_UNSUPPORTED),  # state above 32 KB
    (dict(), 1, dict(x=FAKE + 4), m3scan.M3_ERR_UNSUPPORTED),      # not 16-byte aligned
    (dict(seqlen=5000), 1, {}, m3scan.M3_ERR_UNSUPPORTED),         # K above 4096
    (dict(dstate=5), 1, {}, m3scan.M3_ERR_INVALID_ARG),
    (dict(seqlen=-1), 1, {}, m3scan.M3_ERR_INVALID_ARG),
    (dict(), 1, dict(Bp=FAKE), m3scan.M3_ERR_INVALID_ARG),         # B_prev without x_prev
    (dict(), 1, dict(state=FAKE + 4), m3scan.M3_ERR_INVALID_ARG),
])
def test_tokens_rejects(lib, kw, R, ptrs, expect):
    assert _tokens(lib, _dims(**kw), R=R, **ptrs) == expect


def test_tokens_empty_block_is_a_no_op(lib):
    assert _tokens(lib, _dims(seqlen=0)) == m3scan.M3_OK


def _scan_state(lib, dims, R=1, chunk=4, **ptrs):
    p = dict(x=FAKE, dt=FAKE, A=FAKE, lam=FAKE, B=FAKE, C=FAKE, theta=FAKE, Bp=0, xp=0,
             out=FAKE, state=FAKE)
    p.update(ptrs)
    v = lambda k: ctypes.c_void_p(p[k]) if p[k] else None
    return lib.m3_scan_fwd_state(v("x"), v("dt"), v("A"), v("lam"), v("B"), v("C"), v("theta"),
                                 v("Bp"), v("xp"), ctypes.byref(dims), R, chunk, v("out"),
                                 v("state"), None)


@pytest.mark.parametrize("kw,R,ptrs,expect", [
    (dict(), 1, dict(state=0), m3scan.M3_ERR_INVALID_ARG),        # the state is required
    (dict(), 1, dict(Bp=FAKE), m3scan.M3_ERR_INVALID_ARG),        # B_prev without x_prev
    (dict(), 1, dict(xp=FAKE), m3scan.M3_ERR_INVALID_ARG),
    (dict(), 1, dict(x=0), m3scan.M3_ERR_INVALID_ARG),
    (dict(), 3, {}, m3scan.M3_ERR_UNSUPPORTED),                    # R outside {1, 2, 4}
    (dict(dstate=7), 1, {}, m3scan.M3_ERR_INVALID_ARG),
])
def test_scan_state_rejects(lib, kw, R, ptrs, expect):
    assert _scan_state(lib, _dims(**kw), R=R, **ptrs) == expect


def test_scan_state_empty_block_still_checks_the_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("checked without a device")
    assert _scan_state(lib, _dims(seqlen=0)) == m3scan.M3_ERR_CUDA


def test_fault_injection_arg_rejects_valid_calls(lib, monkeypatch):
    """M3_FAULT=arg: a valid call is refused on the host, before any device work."""
    monkeypatch.setenv("M3_FAULT", "arg")
    assert _scan(lib, _dims()) == m3scan.M3_ERR_INVALID_ARG
    assert _decode(lib, _dims()) == m3scan.M3_ERR_INVALID_ARG
    assert _tokens(lib, _dims()) == m3scan.M3_ERR_INVALID_ARG
    assert _scan_state(lib, _dims()) == m3scan.M3_ERR_INVALID_ARG
    # invalid calls still report their own status first
    assert _scan(lib, _dims(dstate=7)) == m3scan.M3_ERR_INVALID_ARG
    assert _decode(lib, _dims(), R=3) == m3scan.M3_ERR_UNSUPPORTED
    monkeypatch.setenv("M3_FAULT", "no-such-mode")  # unknown values inject nothing
    import torch
    if not torch.cuda.is_available():
        assert _scan(lib, _dims()) == m3scan.M3_ERR_CUDA


def _bwd(lib, dims, R=1, **ptrs):
    names = ("x", "dt", "A", "lam", "B", "C", "theta", "dy", "dfin", "gx", "gdt", "gA", "glam",
             "gB", "gC", "gth", "gbb", "gcb")
    p = {k: FAKE for k in names}
    p.update(dfin=0, gbb=0, gcb=0)
    p.update(ptrs)
    v = lambda k: ctypes.c_void_p(p[k]) if p[k] else None
    return lib.m3_scan_bwd(v("x"), v("dt"), v("A"), v("lam"), v("B"), v("C"), v("theta"), v("dy"),
                           v("dfin"), ctypes.byref(dims), R, v("gx"), v("gdt"), v("gA"), v("glam"),
                           v("gB"), v("gC"), v("gth"), v("gbb"), v("gcb"), None)


@pytest.mark.parametrize("kw,R,ptrs,expect", [
    (dict(), 1, dict(dy=0), m3scan.M3_ERR_INVALID_ARG),
    (dict(), 1, dict(gx=0), m3scan.M3_ERR_INVALID_ARG),
    (dict(), 1, dict(dfin=FAKE + 4), m3scan.M3_ERR_INVALID_ARG),   # d_final not 16-byte aligned
    (dict(), 3, {}, m3scan.M3_ERR_UNSUPPORTED),
    (dict(headdim=6), 1, {}, m3scan.M3_ERR_UNSUPPORTED),
    (dict(dstate=512, headdim=64), 1, {}, m3scan.M3_ERR_UNSUPPORTED),
    (dict(dstate=7), 1, {}, m3scan.M3_ERR_INVALID_ARG),
])
def test_bwd_rejects(lib, kw, R, ptrs, expect):
    assert _bwd(lib, _dims(**kw), R=R, **ptrs) == expect


def test_workspace_query(lib):
    d = _dims()
    assert m3scan.m3_scan_workspace_bytes(d, 1, 4) == 0
    bad = _dims(dstate=7)
    assert m3scan.m3_scan_workspace_bytes(bad, 1, 4) == ctypes.c_size_t(-1).value


def test_valid_call_without_a_device_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present; the no-device path is not reachable")
    assert _scan(lib, _dims()) == m3scan.M3_ERR_CUDA
    assert _decode(lib, _dims()) == m3scan.M3_ERR_CUDA
    assert _tokens(lib, _dims()) == m3scan.M3_ERR_CUDA
    assert _scan_state(lib, _dims()) == m3scan.M3_ERR_CUDA
    assert _bwd(lib, _dims()) == m3scan.M3_ERR_CUDA
    assert lib.m3_device_status(None) == m3scan.M3_ERR_CUDA


# ---------------------------------------------------------------- binding checks
# The Python binding checks what a raw pointer cannot carry (device, dtype,
# shape, contiguity) before any library call.
def _prefill_args(torch, dev="cpu", b=1, L=4, H=2, G=1, P=8, N=8, R=1, act=None):
    act = act or torch.bfloat16
    f = dict(device=dev)
    return dict(x=torch.zeros(b, L, H, P, R, dtype=act, **f),
                dt=torch.zeros(b, L, H, **f), A=torch.zeros(H, **f), lam=torch.zeros(b, L, H, **f),
                B=torch.zeros(b, L, G, N, R, dtype=act, **f),
                C=torch.zeros(b, L, G, N, R, dtype=act, **f),
                theta=torch.zeros(b, L, G, N // 2, **f), R=R, chunk=4)


def test_binding_rejects_host_tensors():
    torch = pytest.importorskip("torch")
    from selective_state_space_129_b300 import m3scan
    with pytest.raises(ValueError, match="CUDA tensor"):
        m3scan.m3_scan_fwd(**_prefill_args(torch))


class _DeviceTensorStub:
    """Stands in for a CUDA tensor (no GPU here): what the checks read."""

    def __init__(self, shape, dtype, contiguous=True):
        self.is_cuda, self.shape, self.dtype, self._c = True, shape, dtype, contiguous

    def is_contiguous(self):
        return self._c


def test_binding_checks_shapes_dtypes_and_contiguity():
    torch = pytest.importorskip("torch")
    from selective_state_space_129_b300 import m3scan
    ex = m3scan._expect
    ex(_DeviceTensorStub((2, 3), torch.float32), "t", (2, 3), torch.float32)  # passes
    ex(None, "opt", (1,), torch.float32, optional=True)                       # passes
    with pytest.raises(ValueError, match="required"):
        ex(None, "t", (1,), torch.float32)
    with pytest.raises(ValueError, match="must have shape"):
        ex(_DeviceTensorStub((2, 4), torch.float32), "t", (2, 3), torch.float32)
    with pytest.raises(ValueError, match="must be torch.float32"):
        ex(_DeviceTensorStub((2, 3), torch.bfloat16), "t", (2, 3), torch.float32)
    with pytest.raises(ValueError, match="contiguous"):
        ex(_DeviceTensorStub((2, 3), torch.float32, contiguous=False), "t", (2, 3), torch.float32)


def test_decode_binding_rejects_host_state():
    torch = pytest.importorskip("torch")
    from selective_state_space_129_b300 import m3scan
    b, H, G, P, N, R = 1, 2, 1, 8, 8, 1
    with pytest.raises(ValueError, match="CUDA tensor"):
        m3scan.m3_decode_step(torch.zeros(b, H, N, P), torch.zeros(b, H, P, R, dtype=torch.bfloat16),
                              torch.zeros(b, H), torch.zeros(H), torch.zeros(b, H),
                              torch.zeros(b, G, N, R, dtype=torch.bfloat16),
                              torch.zeros(b, G, N, R, dtype=torch.bfloat16),
                              torch.zeros(b, G, N // 2), R=R)


def test_bwd_workspace_query(lib):
    q = m3scan.m3_scan_bwd_workspace_bytes
    assert q(_dims(dstate=7), 1) == ctypes.c_size_t(-1).value
    assert q(_dims(batch=0), 1) == 0
    # fp32: the CUDA-core kernel's checkpoints, (ceil(L / 64) + 64) N P floats per (b, h)
    assert q(_dims(), 1) == 4 * (1 + 64) * 8 * 8 * 2 * 4
    # bf16, P 64, N 128, L 2048: the larger of the CUDA-core kernel's scratch and the
    # tensor-core path's (two [N][P] states and 2 + N scalars per chunk of 64 / R tokens)
    d = _dims(batch=2, seqlen=2048, heads=4, groups=1, headdim=64, dstate=128,
              act_dtype=m3scan.M3_BF16)
    simt = 4 * (32 + 64) * 128 * 64 * 8
    for R in (1, 2, 4):
        tc = 4 * 8 * (2048 * R // 64) * (2 * 128 * 64 + 128 + 2)
        assert q(d, R) == max(simt, tc)


def test_bwd_caller_workspace_checked_on_the_host(lib):
    d = _dims(batch=2, seqlen=2048, heads=4, groups=1, headdim=64, dstate=128,
              act_dtype=m3scan.M3_BF16)
    need = m3scan.m3_scan_bwd_workspace_bytes(d, 1)
    d.workspace, d.workspace_bytes = FAKE, need - 16
    assert _bwd(lib, d) == m3scan.M3_ERR_INVALID_ARG    # too small
    d.workspace, d.workspace_bytes = FAKE + 8, need
    assert _bwd(lib, d) == m3scan.M3_ERR_INVALID_ARG    # not 16-byte aligned
