"""ctypes wrapper around the fp64 CPU oracle (``m3oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline / reference leg are the only callers. The product library never
imports this module, and this module never imports the product library.

Every function takes numpy arrays in the same layouts as the C ABI of the GPU
library (row-major, contiguous):

    x, y            [b, L, H, P, R]
    dt, lam         [b, L, H]
    A               [H]
    B, C            [b, L, G, N, R]
    theta           [b, L, G, N/2]
    B_bias, C_bias  [H, N, R] or None
    state           [b, H, N, P]

and computes in IEEE double. See ``m3oracle.c`` for the equations and their
sources on the Mamba-3 pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "m3oracle.c")
_LIB = os.path.join(_HERE, "libm3oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over (batch, head))."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall", "-Wextra",
             "-Wno-unused-parameter", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    scan_args = [i64] * 7 + [dp] * 9 + [dp, dp, ctypes.c_int]
    for name in ("m3o_scan_seq", "m3o_scan_rope"):
        fn = getattr(lib, name)
        fn.argtypes = scan_args
        fn.restype = ctypes.c_int
    lib.m3o_scan_chunked.argtypes = [i64] * 8 + [dp] * 9 + [dp, dp, ctypes.c_int]
    lib.m3o_scan_chunked.restype = ctypes.c_int
    lib.m3o_decode_step.argtypes = [i64] * 6 + [dp] * 12 + [dp, ctypes.c_int]
    lib.m3o_decode_step.restype = ctypes.c_int
    lib.m3o_bc_norm.argtypes = [i64] * 5 + [dp, dp, ctypes.c_double]
    lib.m3o_bc_norm.restype = ctypes.c_int
    lib.m3o_max_threads.argtypes = []
    lib.m3o_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(_LIB)
    return _lib


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_load().m3o_max_threads())


def _dims(x, B, theta):
    b, L, H, P, R = x.shape
    G, N = B.shape[2], B.shape[3]
    assert B.shape == (b, L, G, N, R), B.shape
    assert theta.shape == (b, L, G, N // 2), theta.shape
    return b, L, H, G, P, N, R


def _scan(fn_name, x, dt, A, lam, B, C, theta, B_bias=None, C_bias=None, chunk=None,
          nthreads=0, want_state=True, lib=None):
    x, dt, A, lam, B, C, theta = map(_f64, (x, dt, A, lam, B, C, theta))
    B_bias, C_bias = _f64(B_bias), _f64(C_bias)
    b, L, H, G, P, N, R = _dims(x, B, theta)
    y = np.zeros_like(x)
    st = np.zeros((b, H, N, P), dtype=np.float64) if want_state else None
    lib = lib or _load()
    fn = getattr(lib, fn_name)
    head = [b, L, H, G, P, N, R] + ([chunk] if chunk is not None else [])
    rc = fn(*head, _ptr(x), _ptr(dt), _ptr(A), _ptr(lam), _ptr(B), _ptr(C), _ptr(theta),
            _ptr(B_bias), _ptr(C_bias), _ptr(y), _ptr(st), int(nthreads))
    if rc != 0:
        raise ValueError("%s rejected its dimensions" % fn_name)
    return y, st


def scan_seq(x, dt, A, lam, B, C, theta, B_bias=None, C_bias=None, nthreads=0):
    """Explicit-rotation sequential recurrence; returns (y, final_state)."""
    return _scan("m3o_scan_seq", x, dt, A, lam, B, C, theta, B_bias, C_bias, nthreads=nthreads)


def scan_rope(x, dt, A, lam, B, C, theta, B_bias=None, C_bias=None, nthreads=0):
    """Prop. 3 form (cumulative rotation on B/C); returns (y, final_state)."""
    return _scan("m3o_scan_rope", x, dt, A, lam, B, C, theta, B_bias, C_bias, nthreads=nthreads)


def scan_chunked(x, dt, A, lam, B, C, theta, chunk, B_bias=None, C_bias=None, nthreads=0):
    """Chunked SSD form with materialised intra-chunk mask; returns (y, final_state)."""
    return _scan("m3o_scan_chunked", x, dt, A, lam, B, C, theta, B_bias, C_bias,
                 chunk=int(chunk), nthreads=nthreads)


BC_NORM_EPS = 1e-6


def bc_norm(Bm, eps=BC_NORM_EPS, lib=None):
    """BCNorm of B or C [b, L, G, N, R]: each (b, t, g, r) vector over N divided
    by its root mean square (plus eps under the root), no weight. Returns a new
    fp64 array; the scan with BCNorm is the scan of these normalised B and C."""
    a = _f64(Bm)
    b, L, G, N, R = a.shape
    out = np.zeros_like(a)
    rc = (lib or _load()).m3o_bc_norm(b, L, G, N, R, _ptr(a), _ptr(out), float(eps))
    if rc != 0:
        raise ValueError("m3o_bc_norm rejected its arguments")
    return out


def decode_step(state, x, dt, A, lam, B, C, theta, B_prev=None, x_prev=None,
                B_bias=None, C_bias=None, nthreads=0):
    """One decode token. Returns (y, new_state); ``state`` is not modified.

    Per-token layouts: state [b,H,N,P], x/x_prev [b,H,P,R], dt/lam [b,H],
    B/C/B_prev [b,G,N,R], theta [b,G,N/2].
    """
    st = _f64(state).copy()
    x, dt, A, lam, B, C, theta = map(_f64, (x, dt, A, lam, B, C, theta))
    B_prev, x_prev, B_bias, C_bias = map(_f64, (B_prev, x_prev, B_bias, C_bias))
    b, H, P, R = x.shape
    G, N = B.shape[1], B.shape[2]
    y = np.zeros_like(x)
    rc = _load().m3o_decode_step(b, H, G, P, N, R, _ptr(st), _ptr(x), _ptr(dt), _ptr(A),
                                 _ptr(lam), _ptr(B_prev), _ptr(x_prev), _ptr(B), _ptr(C),
                                 _ptr(theta), _ptr(B_bias), _ptr(C_bias), _ptr(y),
                                 int(nthreads))
    if rc != 0:
        raise ValueError("m3o_decode_step rejected its arguments")
    return y, st


def decode_tokens(state, x, dt, A, lam, B, C, theta, B_prev=None, x_prev=None,
                  B_bias=None, C_bias=None, nthreads=0):
    """K consecutive decode tokens of every (batch, head): the decode step
    applied to tokens t = 0 .. K-1 in order, token t's previous token being
    token t-1 of the block (the given B_prev / x_prev for t = 0; None for the
    first token of a sequence). Returns (y, new_state); ``state`` is not
    modified.

    Layouts: state [b,H,N,P]; x, y [b,K,H,P,R]; dt, lam [b,K,H];
    B, C [b,K,G,N,R]; theta [b,K,G,N/2]; B_prev [b,G,N,R], x_prev [b,H,P,R].
    """
    x, dt, lam, B, C, theta = map(_f64, (x, dt, lam, B, C, theta))
    K = x.shape[1]
    st = _f64(state)
    ys = []
    for t in range(K):
        bp, xp = (B_prev, x_prev) if t == 0 else (B[:, t - 1], x[:, t - 1])
        y, st = decode_step(st, x[:, t], dt[:, t], A, lam[:, t], B[:, t], C[:, t], theta[:, t],
                            B_prev=bp, x_prev=xp, B_bias=B_bias, C_bias=C_bias,
                            nthreads=nthreads)
        ys.append(y)
    y = np.stack(ys, axis=1) if ys else np.zeros_like(x)
    return y, st


class Oracle:
    """The same entry points bound to a given build of ``m3oracle.c``.

    The module-level functions use the default build; tests that plant
    mistakes in a copy of the oracle source bind the mutant build here.
    """

    def __init__(self, lib_path: str):
        self._lib = _bind(lib_path)

    def scan_seq(self, x, dt, A, lam, B, C, theta, B_bias=None, C_bias=None, nthreads=0):
        return _scan("m3o_scan_seq", x, dt, A, lam, B, C, theta, B_bias, C_bias,
                     nthreads=nthreads, lib=self._lib)

    def scan_rope(self, x, dt, A, lam, B, C, theta, B_bias=None, C_bias=None, nthreads=0):
        return _scan("m3o_scan_rope", x, dt, A, lam, B, C, theta, B_bias, C_bias,
                     nthreads=nthreads, lib=self._lib)

    def scan_chunked(self, x, dt, A, lam, B, C, theta, chunk, B_bias=None, C_bias=None,
                     nthreads=0):
        return _scan("m3o_scan_chunked", x, dt, A, lam, B, C, theta, B_bias, C_bias,
                     chunk=int(chunk), nthreads=nthreads, lib=self._lib)

    def bc_norm(self, Bm, eps=BC_NORM_EPS):
        return bc_norm(Bm, eps, lib=self._lib)


def build_variant(src_text: str, out_path: str) -> str:
    """Compile a modified copy of the oracle source (used to plant mistakes)."""
    src_path = out_path + ".c"
    with open(src_path, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", src_path,
                           "-o", out_path, "-lm"])
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()
