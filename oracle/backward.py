"""Gradients of the Mamba-3 scan: a plain fp64 PyTorch CPU definition.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: the tests are its only
callers; the product library never imports it and it never imports the
product library. It is the checker of the library's backward kernel
(m3_scan_bwd; tests/test_gpu_parity.py, test_backward_matches_the_gradient_oracle).

The forward is the sequential recurrence with explicit 2x2 rotations of the
state (Prop. 1 and the rotation, sec. 4.1 and 4.2 of the page
"MAMBA-3: IMPROVED SEQUENCE MODELING USING STATE SPACE PRINCIPLES" (aipaper.cc); the rotation
matrix, sec. 2.2 of "State Space Models 家族对比分析：S4 → Mamba → Mamba-2 → Mamba-3" (metaphor-xennon blog);
MIMO rank R, sec. 3 of "Mamba-3: Improved Sequence Modeling using State Space Principles" (papernotes.org)),
written here with torch tensor operations so that autograd differentiates it:

    U_t = (B_t + B_bias) x_t^T,  G_t = h_{t-1} + beta_hat_t U_{t-1}
    h_t = alpha_t Rot(Delta_t theta_t) G_t + gamma_t U_t,  y_t = (C_t + C_bias)^T h_t
    alpha_t = exp(Delta_t A),  beta_hat_t = (1 - lambda_t) Delta_t,  gamma_t = lambda_t Delta_t

with rotating pairs (2k, 2k+1) and [[cos, -sin], [sin, cos]]. The gradients
are those of a scalar loss <y, dy> + <h_final, dh> with respect to every input
(x, dt, A, lambda, B, C, theta, the biases, the entering state, and B_prev /
x_prev of a continued sequence). Layouts are those of ``oracle.py``.
Pinned in tests/test_oracle_backward.py: the forward against the C oracle,
the gradients against central finite differences of the C oracle.
"""
from __future__ import annotations

import torch

_F64 = torch.float64


def _t(a, grad=True):
    if a is None:
        return None
    t = torch.as_tensor(a).to(_F64).clone()
    t.requires_grad_(grad)
    return t


def scan_forward(x, dt, A, lam, B, C, theta, B_bias=None, C_bias=None, state0=None,
                 B_prev=None, x_prev=None):
    """Sequential forward on torch tensors (any dtype is promoted to fp64 by
    the caller). Returns (y [b,L,H,P,R], final state [b,H,N,P])."""
    b, L, H, P, R = x.shape
    G, N = B.shape[2], B.shape[3]
    gidx = torch.arange(H) // (H // G)  # group of each head
    Bh = B[:, :, gidx]                 # [b,L,H,N,R]
    Ch = C[:, :, gidx]
    th = theta[:, :, gidx]             # [b,L,H,N/2]
    if B_bias is not None:
        Bh = Bh + B_bias
    if C_bias is not None:
        Ch = Ch + C_bias
    h = torch.zeros(b, H, N, P, dtype=_F64) if state0 is None else state0
    if B_prev is not None:
        Bp = B_prev[:, gidx] + (B_bias if B_bias is not None else 0.0)
        Uprev = torch.einsum("bhnr,bhpr->bhnp", Bp, x_prev)
    else:
        Uprev = torch.zeros(b, H, N, P, dtype=_F64)
    ys = []
    for t in range(L):
        U = torch.einsum("bhnr,bhpr->bhnp", Bh[:, t], x[:, t])
        d, lm = dt[:, t], lam[:, t]                 # [b,H]
        alpha = torch.exp(d * A)
        gamma, bhat = lm * d, (1.0 - lm) * d
        Gs = h + bhat[..., None, None] * Uprev
        phi = d[..., None] * th[:, t]                # [b,H,N/2]
        c, s = torch.cos(phi)[..., None], torch.sin(phi)[..., None]
        g0, g1 = Gs[:, :, 0::2], Gs[:, :, 1::2]
        r0, r1 = c * g0 - s * g1, s * g0 + c * g1
        rot = torch.stack((r0, r1), dim=3).reshape(b, H, N, P)
        h = alpha[..., None, None] * rot + gamma[..., None, None] * U
        ys.append(torch.einsum("bhnr,bhnp->bhpr", Ch[:, t], h))
        Uprev = U
    y = torch.stack(ys, dim=1) if ys else torch.zeros(b, 0, H, P, R, dtype=_F64)
    return y, h


def scan_grads(x, dt, A, lam, B, C, theta, dy, dh=None, B_bias=None, C_bias=None, state0=None,
               B_prev=None, x_prev=None):
    """Gradients of <y, dy> + <h_final, dh> with respect to every given input.

    Returns a dict keyed by input name (x, dt, A, lam, B, C, theta and, when
    given, B_bias, C_bias, state0, B_prev, x_prev) of fp64 numpy arrays.
    """
    named = dict(x=x, dt=dt, A=A, lam=lam, B=B, C=C, theta=theta, B_bias=B_bias, C_bias=C_bias,
                 state0=state0, B_prev=B_prev, x_prev=x_prev)
    ts = {k: _t(v) for k, v in named.items()}
    y, hf = scan_forward(**ts)
    loss = (y * _t(dy, False)).sum()
    if dh is not None:
        loss = loss + (hf * _t(dh, False)).sum()
    keys = [k for k, v in ts.items() if v is not None]
    grads = torch.autograd.grad(loss, [ts[k] for k in keys], allow_unused=True)
    out = {}
    for k, g in zip(keys, grads):
        out[k] = (torch.zeros_like(ts[k]) if g is None else g).detach().numpy()
    return out
