"""Python binding of libm3scan.so (argument marshalling only).

The names mirror the C ABI in include/m3scan.h. Tensors are PyTorch CUDA
tensors (PyTorch supplies device memory and streams); every step of the scan
runs in the library's CUDA kernels. There is no CPU fallback: if the library
cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libm3scan.so")

M3_OK, M3_ERR_INVALID_ARG, M3_ERR_UNSUPPORTED, M3_ERR_CUDA, M3_ERR_TIMEOUT = range(5)
M3_F32, M3_BF16 = 0, 1
M3_FLAG_BC_NORM = 1  # m3_dims.flags: BCNorm B and C inside the prefill

# Exported entry points (kept in step with include/m3scan.h).
EXPORTS = ("m3_scan_fwd", "m3_scan_fwd_noalloc", "m3_decode_step", "m3_scan_workspace_bytes",
           "m3_status_string", "m3_device_status", "m3_version", "m3_decode_tokens",
           "m3_scan_fwd_state", "m3_scan_bwd", "m3_scan_bwd_workspace_bytes")


class M3Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s" % (where, m3_status_string(status)))


class m3_dims(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int64),
        ("seqlen", ctypes.c_int64),
        ("heads", ctypes.c_int64),
        ("groups", ctypes.c_int64),
        ("headdim", ctypes.c_int64),
        ("dstate", ctypes.c_int64),
        ("act_dtype", ctypes.c_int32),
        ("flags", ctypes.c_int32),
        ("B_bias", ctypes.c_void_p),
        ("C_bias", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
    ]


_lib = None


def load(path: str = LIB_PATH):
    """Load the library (once). Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libm3scan.so is not built (%s); run "
                           "`python -m selective_state_space_129_b300.build`" % path)
    lib = ctypes.CDLL(path)
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    dims_p = ctypes.POINTER(m3_dims)
    lib.m3_scan_fwd.argtypes = [vp] * 7 + [dims_p, i32, i32, vp, vp, vp]
    lib.m3_scan_fwd.restype = i32
    lib.m3_scan_fwd_noalloc.argtypes = [vp] * 7 + [dims_p, i32, i32, vp, vp, vp]
    lib.m3_scan_fwd_noalloc.restype = i32
    lib.m3_decode_step.argtypes = [vp] * 10 + [dims_p, i32, vp, vp]
    lib.m3_decode_step.restype = i32
    lib.m3_decode_tokens.argtypes = [vp] * 10 + [dims_p, i32, vp, vp]
    lib.m3_decode_tokens.restype = i32
    lib.m3_scan_fwd_state.argtypes = [vp] * 9 + [dims_p, i32, i32, vp, vp, vp]
    lib.m3_scan_fwd_state.restype = i32
    lib.m3_scan_bwd.argtypes = [vp] * 9 + [dims_p, i32] + [vp] * 10
    lib.m3_scan_bwd.restype = i32
    lib.m3_scan_workspace_bytes.argtypes = [dims_p, i32, i32]
    lib.m3_scan_workspace_bytes.restype = ctypes.c_size_t
    lib.m3_scan_bwd_workspace_bytes.argtypes = [dims_p, i32]
    lib.m3_scan_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.m3_status_string.argtypes = [i32]
    lib.m3_status_string.restype = ctypes.c_char_p
    lib.m3_device_status.argtypes = [vp]
    lib.m3_device_status.restype = i32
    lib.m3_version.argtypes = []
    lib.m3_version.restype = i32
    _lib = lib
    return lib


def m3_status_string(status: int) -> str:
    return load().m3_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _expect(t, name, shape, dtype, optional=False):
    """The C ABI takes plain pointers to row-major contiguous device arrays:
    check what a pointer cannot carry (device, dtype, shape, contiguity)."""
    if t is None:
        if optional:
            return
        raise ValueError("%s is required" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _check_prefill(x, dt, A, lam, B, C, theta, R, out, final_state, B_bias, C_bias):
    import torch
    if x.dim() != 5 or B.dim() != 5:
        raise ValueError("x must be [b,L,H,P,R] and B [b,L,G,N,R]")
    b, L, H, P, R_ = x.shape
    if R_ != R:
        raise ValueError("x.shape[-1] must equal R")
    G, N = B.shape[2], B.shape[3]
    f32, act = torch.float32, x.dtype
    _expect(x, "x", (b, L, H, P, R), act)
    _expect(dt, "dt", (b, L, H), f32)
    _expect(lam, "lam", (b, L, H), f32)
    _expect(A, "A", (H,), f32)
    _expect(B, "B", (b, L, G, N, R), act)
    _expect(C, "C", (b, L, G, N, R), act)
    _expect(theta, "theta", (b, L, G, N // 2), f32)
    _expect(B_bias, "B_bias", (H, N, R), f32, optional=True)
    _expect(C_bias, "C_bias", (H, N, R), f32, optional=True)
    _expect(out, "out", (b, L, H, P, R), act, optional=True)
    _expect(final_state, "final_state", (b, H, N, P), f32, optional=True)
    return b, L, H, P, G, N


def _stream_handle(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _act_dtype(t):
    import torch
    if t.dtype == torch.bfloat16:
        return M3_BF16
    if t.dtype == torch.float32:
        return M3_F32
    raise TypeError("activations must be float32 or bfloat16, got %s" % t.dtype)


def make_dims(batch, seqlen, heads, groups, headdim, dstate, act_dtype, B_bias=None,
              C_bias=None, workspace=None, flags=0):
    d = m3_dims()
    d.batch, d.seqlen, d.heads, d.groups, d.headdim, d.dstate = (
        int(batch), int(seqlen), int(heads), int(groups), int(headdim), int(dstate))
    d.act_dtype = int(act_dtype)
    d.flags = int(flags)
    d.B_bias = None if B_bias is None else B_bias.data_ptr()
    d.C_bias = None if C_bias is None else C_bias.data_ptr()
    d.workspace = None if workspace is None else workspace.data_ptr()
    d.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return d


def _check(status, where):
    if status != M3_OK:
        raise M3Error(status, where)


def m3_scan_workspace_bytes(dims: m3_dims, R: int, chunk: int) -> int:
    return int(load().m3_scan_workspace_bytes(ctypes.byref(dims), int(R), int(chunk)))


def m3_scan_bwd_workspace_bytes(dims: m3_dims, R: int) -> int:
    return int(load().m3_scan_bwd_workspace_bytes(ctypes.byref(dims), int(R)))


def m3_scan_fwd(x, dt, A, lam, B, C, theta, R, chunk, out=None, final_state=None,
                B_bias=None, C_bias=None, workspace=None, stream=None, want_state=True,
                bc_norm=False):
    """Prefill. Shapes: x [b,L,H,P,R], dt/lam [b,L,H], A [H], B/C [b,L,G,N,R],
    theta [b,L,G,N/2]. Returns (out, final_state). ``bc_norm``: B and C are
    un-normalised and the kernel applies BCNorm to them (M3_FLAG_BC_NORM)."""
    import torch
    lib = load()
    b, L, H, P, G, N = _check_prefill(x, dt, A, lam, B, C, theta, R, out, final_state, B_bias,
                                      C_bias)
    if workspace is not None and not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    if out is None:
        out = torch.empty_like(x)
    if final_state is None and want_state:
        final_state = torch.empty((b, H, N, P), dtype=torch.float32, device=x.device)
    dims = make_dims(b, L, H, G, P, N, _act_dtype(x), B_bias, C_bias, workspace,
                     flags=M3_FLAG_BC_NORM if bc_norm else 0)
    st = lib.m3_scan_fwd(_ptr(x), _ptr(dt), _ptr(A), _ptr(lam), _ptr(B), _ptr(C), _ptr(theta),
                         ctypes.byref(dims), int(R), int(chunk), _ptr(out), _ptr(final_state),
                         _stream_handle(stream))
    _check(st, "m3_scan_fwd")
    return out, final_state


def m3_scan_fwd_state(x, dt, A, lam, B, C, theta, R, chunk, state, B_prev=None, x_prev=None,
                      out=None, B_bias=None, C_bias=None, workspace=None, stream=None):
    """Prefill that continues a sequence from ``state`` [b,H,N,P] fp32, which is
    updated in place to the state after the block; B_prev [b,G,N,R] / x_prev
    [b,H,P,R] are the token before the block (or None). Returns out."""
    import torch
    lib = load()
    if state is None:
        raise ValueError("state is required")
    b, L, H, P, G, N = _check_prefill(x, dt, A, lam, B, C, theta, R, out, state, B_bias, C_bias)
    _expect(B_prev, "B_prev", (b, G, N, R), x.dtype, optional=True)
    _expect(x_prev, "x_prev", (b, H, P, R), x.dtype, optional=True)
    if workspace is not None and not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    if out is None:
        out = torch.empty_like(x)
    dims = make_dims(b, L, H, G, P, N, _act_dtype(x), B_bias, C_bias, workspace)
    st = lib.m3_scan_fwd_state(_ptr(x), _ptr(dt), _ptr(A), _ptr(lam), _ptr(B), _ptr(C),
                               _ptr(theta), _ptr(B_prev), _ptr(x_prev), ctypes.byref(dims),
                               int(R), int(chunk), _ptr(out), _ptr(state), _stream_handle(stream))
    _check(st, "m3_scan_fwd_state")
    return out


def m3_scan_bwd(x, dt, A, lam, B, C, theta, dy, R, d_final=None, B_bias=None, C_bias=None,
                stream=None, workspace=None):
    """Gradients of <y, dy> + <h_final, d_final> of a prefill from a zero state.
    Returns a dict of fp32 tensors: x, dt, A, lam, B, C, theta and, when the
    biases are given, B_bias, C_bias. ``workspace``: a device tensor of at least
    m3_scan_bwd_workspace_bytes bytes, or None (the library allocates it)."""
    import torch
    lib = load()
    b, L, H, P, G, N = _check_prefill(x, dt, A, lam, B, C, theta, R, dy, None, B_bias, C_bias)
    _expect(d_final, "d_final", (b, H, N, P), torch.float32, optional=True)
    f = dict(dtype=torch.float32, device=x.device)
    g = dict(x=torch.empty(b, L, H, P, R, **f), dt=torch.empty(b, L, H, **f),
             A=torch.empty(H, **f), lam=torch.empty(b, L, H, **f),
             B=torch.empty(b, L, G, N, R, **f), C=torch.empty(b, L, G, N, R, **f),
             theta=torch.empty(b, L, G, N // 2, **f))
    if B_bias is not None:
        g["B_bias"] = torch.empty(H, N, R, **f)
    if C_bias is not None:
        g["C_bias"] = torch.empty(H, N, R, **f)
    dims = make_dims(b, L, H, G, P, N, _act_dtype(x), B_bias, C_bias, workspace)
    st = lib.m3_scan_bwd(_ptr(x), _ptr(dt), _ptr(A), _ptr(lam), _ptr(B), _ptr(C), _ptr(theta),
                         _ptr(dy), _ptr(d_final), ctypes.byref(dims), int(R), _ptr(g["x"]),
                         _ptr(g["dt"]), _ptr(g["A"]), _ptr(g["lam"]), _ptr(g["B"]), _ptr(g["C"]),
                         _ptr(g["theta"]), _ptr(g.get("B_bias")), _ptr(g.get("C_bias")),
                         _stream_handle(stream))
    _check(st, "m3_scan_bwd")
    return g


def m3_scan_fwd_noalloc(x, dt, A, lam, B, C, theta, R, chunk, out, final_state, B_bias=None,
                        C_bias=None, stream=None, bc_norm=False):
    """Prefill like m3_scan_fwd into caller-allocated ``out`` / ``final_state``
    (``final_state`` may be None); the library allocates no device memory (its
    scratch is a fixed 32 MiB array; larger needs raise M3Error)."""
    lib = load()
    if out is None:
        raise ValueError("out is required")
    b, L, H, P, G, N = _check_prefill(x, dt, A, lam, B, C, theta, R, out, final_state, B_bias,
                                      C_bias)
    dims = make_dims(b, L, H, G, P, N, _act_dtype(x), B_bias, C_bias,
                     flags=M3_FLAG_BC_NORM if bc_norm else 0)
    st = lib.m3_scan_fwd_noalloc(_ptr(x), _ptr(dt), _ptr(A), _ptr(lam), _ptr(B), _ptr(C),
                                 _ptr(theta), ctypes.byref(dims), int(R), int(chunk), _ptr(out),
                                 _ptr(final_state), _stream_handle(stream))
    _check(st, "m3_scan_fwd_noalloc")
    return out, final_state


def m3_decode_step(state, x, dt, A, lam, B, C, theta, R, B_prev=None, x_prev=None, out=None,
                   B_bias=None, C_bias=None, stream=None):
    """One decode token; ``state`` [b,H,N,P] fp32 is updated in place. Returns out [b,H,P,R]."""
    import torch
    lib = load()
    if x.dim() != 4 or B.dim() != 4:
        raise ValueError("x must be [b,H,P,R] and B [b,G,N,R]")
    b, H, P, R_ = x.shape
    if R_ != R:
        raise ValueError("x.shape[-1] must equal R")
    G, N = B.shape[1], B.shape[2]
    f32, act = torch.float32, x.dtype
    _expect(state, "state", (b, H, N, P), f32)
    _expect(x, "x", (b, H, P, R), act)
    _expect(dt, "dt", (b, H), f32)
    _expect(lam, "lam", (b, H), f32)
    _expect(A, "A", (H,), f32)
    _expect(B, "B", (b, G, N, R), act)
    _expect(C, "C", (b, G, N, R), act)
    _expect(theta, "theta", (b, G, N // 2), f32)
    _expect(B_prev, "B_prev", (b, G, N, R), act, optional=True)
    _expect(x_prev, "x_prev", (b, H, P, R), act, optional=True)
    _expect(B_bias, "B_bias", (H, N, R), f32, optional=True)
    _expect(C_bias, "C_bias", (H, N, R), f32, optional=True)
    _expect(out, "out", (b, H, P, R), act, optional=True)
    if out is None:
        out = torch.empty_like(x)
    dims = make_dims(b, 1, H, G, P, N, _act_dtype(x), B_bias, C_bias)
    st = lib.m3_decode_step(_ptr(state), _ptr(x), _ptr(dt), _ptr(A), _ptr(lam), _ptr(B_prev),
                            _ptr(x_prev), _ptr(B), _ptr(C), _ptr(theta), ctypes.byref(dims),
                            int(R), _ptr(out), _stream_handle(stream))
    _check(st, "m3_decode_step")
    return out


def m3_decode_tokens(state, x, dt, A, lam, B, C, theta, R, B_prev=None, x_prev=None, out=None,
                     B_bias=None, C_bias=None, stream=None):
    """K consecutive decode tokens; ``state`` [b,H,N,P] fp32 is updated in place.

    x [b,K,H,P,R], dt / lam [b,K,H], B / C [b,K,G,N,R], theta [b,K,G,N/2];
    B_prev [b,G,N,R] / x_prev [b,H,P,R] are the token before the block (or
    None). Returns out [b,K,H,P,R]."""
    import torch
    lib = load()
    if x.dim() != 5 or B.dim() != 5:
        raise ValueError("x must be [b,K,H,P,R] and B [b,K,G,N,R]")
    b, K, H, P, R_ = x.shape
    if R_ != R:
        raise ValueError("x.shape[-1] must equal R")
    G, N = B.shape[2], B.shape[3]
    f32, act = torch.float32, x.dtype
    _expect(state, "state", (b, H, N, P), f32)
    _expect(x, "x", (b, K, H, P, R), act)
    _expect(dt, "dt", (b, K, H), f32)
    _expect(lam, "lam", (b, K, H), f32)
    _expect(A, "A", (H,), f32)
    _expect(B, "B", (b, K, G, N, R), act)
    _expect(C, "C", (b, K, G, N, R), act)
    _expect(theta, "theta", (b, K, G, N // 2), f32)
    _expect(B_prev, "B_prev", (b, G, N, R), act, optional=True)
    _expect(x_prev, "x_prev", (b, H, P, R), act, optional=True)
    _expect(B_bias, "B_bias", (H, N, R), f32, optional=True)
    _expect(C_bias, "C_bias", (H, N, R), f32, optional=True)
    _expect(out, "out", (b, K, H, P, R), act, optional=True)
    if out is None:
        out = torch.empty_like(x)
    dims = make_dims(b, K, H, G, P, N, _act_dtype(x), B_bias, C_bias)
    st = lib.m3_decode_tokens(_ptr(state), _ptr(x), _ptr(dt), _ptr(A), _ptr(lam), _ptr(B_prev),
                              _ptr(x_prev), _ptr(B), _ptr(C), _ptr(theta), ctypes.byref(dims),
                              int(R), _ptr(out), _stream_handle(stream))
    _check(st, "m3_decode_tokens")
    return out


def m3_device_status(stream=None) -> int:
    return int(load().m3_device_status(_stream_handle(stream)))


def m3_version() -> int:
    return int(load().m3_version())
