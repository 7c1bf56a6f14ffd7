"""Seeded synthetic inputs for the Mamba-3 scan (prefill and decode).

This module is the only thing the CPU oracle and the CUDA path share. It draws
random numbers and rounds them to the activation dtype; it holds none of the
scan's arithmetic (no bias add, no discretisation, no rotation).

Recipe (numpy PCG64, seed = workload index unless given; draw order
A, dt, lambda, theta, B, C, B_bias, C_bias, x):

    A       = -exp(U(0, ln 16))            per head            -> A in [-16, -1]
    dt      = softplus(N(-1, 0.5))          per (b, t, h)
    lambda  = sigmoid(N(0, 1))              per (b, t, h)
    theta   = U(-pi, pi)                    per (b, t, g, k), k < N/2
    B, C    = N(0,1)/sqrt(N)  (tiny case)   or  RMS-normalised N(0,1) over N
              per (b, t, g, r): v / sqrt(mean(v^2) + 1e-6)
    biases  = N(0, 0.1)                     per (h, n, r)
    x       = N(0, 1)

Activations (x, B, C) are rounded to bf16 (round-to-nearest-even) when the
workload is bf16; every array is returned as float32 holding exactly the value
the kernels see. dt, lambda, theta, A and the biases stay fp32.

Parity stress case (state tracking, the R(pi x_t) construction on the
"Mamba-3: Improved Sequence Modeling using State Space Principles" (papernotes.org), sec. 2): A = 0, bits ~ Bernoulli(0.5) per (b, t),
dt drawn per (b, t) and shared by all heads, theta = pi * bit / dt for every
state pair, and an impulse input: x is N(0,1) at t = 0 and zero after.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class ScanShape:
    batch: int
    seqlen: int
    heads: int
    groups: int
    headdim: int   # P
    dstate: int    # N
    R: int = 1
    chunk: int = 64
    bf16: bool = True
    rms_bc: bool = True   # RMS-normalised B/C (else N(0,1)/sqrt(N))

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen


# The workloads. Index 0 is the tiny fp32 case; 1 and 2 are the 1.5B-layer
# prefill shapes; 3 is batched decode; 4 is the long-context sweep.
TINY = ScanShape(1, 64, 2, 1, 16, 16, R=1, chunk=16, bf16=False, rms_bc=False)
PREFILL_SISO = ScanShape(8, 2048, 32, 1, 64, 128, R=1, chunk=64)
PREFILL_MIMO = ScanShape(8, 2048, 32, 1, 64, 128, R=4, chunk=16)
DECODE_SISO = ScanShape(128, 1, 32, 1, 64, 128, R=1, chunk=1)
DECODE_MIMO = ScanShape(128, 1, 32, 1, 64, 128, R=4, chunk=1)
DECODE_STEPS = 1024
LONG_MIMO_N128 = ScanShape(1, 65536, 32, 1, 64, 128, R=4, chunk=16)
LONG_SISO_N64 = ScanShape(1, 65536, 32, 1, 64, 64, R=1, chunk=64)
LONG_SISO_N128 = ScanShape(1, 65536, 32, 1, 64, 128, R=1, chunk=64)

WORKLOADS = {
    "tiny": (0, TINY),
    "prefill_siso": (1, PREFILL_SISO),
    "prefill_mimo": (2, PREFILL_MIMO),
    "decode_siso": (3, DECODE_SISO),
    "decode_mimo": (3, DECODE_MIMO),
    "long_mimo_n128": (4, LONG_MIMO_N128),
    "long_siso_n64": (4, LONG_SISO_N64),
    "long_siso_n128": (4, LONG_SISO_N128),
}


def to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16 (ties to even); returns float32."""
    a = np.array(a, dtype=np.float32, copy=True, order="C")
    u = a.view(np.uint32)  # finite inputs: the sum below cannot overflow 32 bits
    bias = (u >> 16) & 1
    bias += 0x7FFF
    u += bias
    u &= np.uint32(0xFFFF0000)
    return a


def _softplus(v):
    return np.logaddexp(0.0, v)


def _sigmoid(v):
    return 1.0 / (1.0 + np.exp(-v))


def _bc(rng, shape, n_axis_len, rms, dtype_f32=True):
    v = rng.standard_normal(shape, dtype=np.float32)
    if rms:
        # shape [..., N, R]: normalise over N for each (.., r)
        ms = np.mean(v.astype(np.float64) ** 2, axis=-2, keepdims=True)
        v = (v / np.sqrt(ms + 1e-6)).astype(np.float32)
    else:
        v = (v / math.sqrt(n_axis_len)).astype(np.float32)
    return v


def scan_inputs(shape: ScanShape, seed: int, parity: bool = False) -> dict:
    """Prefill inputs for ``shape`` (float32 arrays, bf16-exact where bf16)."""
    b, L, H, G, P, N, R = (shape.batch, shape.seqlen, shape.heads, shape.groups,
                           shape.headdim, shape.dstate, shape.R)
    rng = np.random.Generator(np.random.PCG64(seed))
    rnd = to_bf16 if shape.bf16 else (lambda a: np.ascontiguousarray(a, np.float32))
    A = (-np.exp(rng.uniform(0.0, math.log(16.0), size=H))).astype(np.float32)
    if parity:
        A = np.zeros(H, np.float32)
        dt1 = _softplus(rng.normal(-1.0, 0.5, size=(b, L, 1))).astype(np.float32)
        dt = np.ascontiguousarray(np.broadcast_to(dt1, (b, L, H)))
    else:
        dt = _softplus(rng.normal(-1.0, 0.5, size=(b, L, H))).astype(np.float32)
    lam = _sigmoid(rng.normal(0.0, 1.0, size=(b, L, H))).astype(np.float32)
    if parity:
        bits = (rng.uniform(size=(b, L)) < 0.5).astype(np.float32)
        th1 = (np.float32(math.pi) * bits / dt[:, :, 0]).astype(np.float32)
        theta = np.ascontiguousarray(
            np.broadcast_to(th1[:, :, None, None], (b, L, G, N // 2))).astype(np.float32)
    else:
        bits = None
        theta = rng.uniform(-math.pi, math.pi, size=(b, L, G, N // 2)).astype(np.float32)
    Bm = rnd(_bc(rng, (b, L, G, N, R), N, shape.rms_bc))
    Cm = rnd(_bc(rng, (b, L, G, N, R), N, shape.rms_bc))
    B_bias = rng.normal(0.0, 0.1, size=(H, N, R)).astype(np.float32)
    C_bias = rng.normal(0.0, 0.1, size=(H, N, R)).astype(np.float32)
    x = rng.standard_normal((b, L, H, P, R), dtype=np.float32)
    if parity:
        x[:, 1:] = 0.0
    x = rnd(x)
    out = dict(x=x, dt=dt, A=A, lam=lam, B=Bm, C=Cm, theta=theta, B_bias=B_bias,
               C_bias=C_bias)
    if bits is not None:
        out["bits"] = bits
    return out


def decode_inputs(shape: ScanShape, seed: int, step: int) -> dict:
    """Per-token inputs for decode step ``step`` (drawn as in the prefill recipe).

    A and the biases depend on ``seed`` only; the per-token tensors on
    (seed, step). Layouts: x [b,H,P,R], dt/lam [b,H], B/C [b,G,N,R],
    theta [b,G,N/2].
    """
    b, H, G, P, N, R = (shape.batch, shape.heads, shape.groups, shape.headdim,
                        shape.dstate, shape.R)
    rnd = to_bf16 if shape.bf16 else (lambda a: np.ascontiguousarray(a, np.float32))
    rng0 = np.random.Generator(np.random.PCG64(seed))
    A = (-np.exp(rng0.uniform(0.0, math.log(16.0), size=H))).astype(np.float32)
    B_bias = rng0.normal(0.0, 0.1, size=(H, N, R)).astype(np.float32)
    C_bias = rng0.normal(0.0, 0.1, size=(H, N, R)).astype(np.float32)
    rng = np.random.Generator(np.random.PCG64([seed, step + 1]))
    dt = _softplus(rng.normal(-1.0, 0.5, size=(b, H))).astype(np.float32)
    lam = _sigmoid(rng.normal(0.0, 1.0, size=(b, H))).astype(np.float32)
    theta = rng.uniform(-math.pi, math.pi, size=(b, G, N // 2)).astype(np.float32)
    Bm = rnd(_bc(rng, (b, G, N, R), N, shape.rms_bc))
    Cm = rnd(_bc(rng, (b, G, N, R), N, shape.rms_bc))
    x = rnd(rng.standard_normal((b, H, P, R), dtype=np.float32))
    return dict(x=x, dt=dt, A=A, lam=lam, B=Bm, C=Cm, theta=theta, B_bias=B_bias,
                C_bias=C_bias)


def small_shape(**kw) -> ScanShape:
    """A ScanShape with small defaults, for tests."""
    base = dict(batch=1, seqlen=16, heads=2, groups=1, headdim=8, dstate=8, R=1, chunk=4,
                bf16=False, rms_bc=False)
    base.update(kw)
    return ScanShape(**base)
