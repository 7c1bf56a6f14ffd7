"""Pins for the gradient oracle (oracle/backward.py), CPU only.

The torch forward is checked against the C oracle (a separate implementation
of the same recurrence), and every gradient against central finite
differences of the C oracle's loss, so that autograd is never checked
against itself.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import backward  # noqa: E402


def _inputs(seed, b=1, L=6, H=2, G=1, P=3, N=4, R=2, cont=True):
    rng = np.random.default_rng(seed)
    d = dict(
        x=rng.standard_normal((b, L, H, P, R)),
        dt=np.log1p(np.exp(rng.normal(-1.0, 0.5, (b, L, H)))),
        A=-np.exp(rng.uniform(0, math.log(16), H)),
        lam=1 / (1 + np.exp(-rng.standard_normal((b, L, H)))),
        B=rng.standard_normal((b, L, G, N, R)) / math.sqrt(N),
        C=rng.standard_normal((b, L, G, N, R)) / math.sqrt(N),
        theta=rng.uniform(-math.pi, math.pi, (b, L, G, N // 2)),
        B_bias=rng.normal(0, 0.1, (H, N, R)),
        C_bias=rng.normal(0, 0.1, (H, N, R)),
    )
    if cont:
        d["state0"] = rng.standard_normal((b, H, N, P))
        d["B_prev"] = rng.standard_normal((b, G, N, R)) / math.sqrt(N)
        d["x_prev"] = rng.standard_normal((b, H, P, R))
    return d


def _c_loss(orc, d, dy, dh):
    """<y, dy> + <h_final, dh> from the C oracle (the decode step token by
    token, from the given state and previous token)."""
    b, L, H, P, R = d["x"].shape
    N = d["B"].shape[3]
    st0 = d.get("state0", np.zeros((b, H, N, P)))
    y, hf = orc.decode_tokens(st0, d["x"], d["dt"], d["A"], d["lam"], d["B"], d["C"], d["theta"],
                              B_prev=d.get("B_prev"), x_prev=d.get("x_prev"),
                              B_bias=d.get("B_bias"), C_bias=d.get("C_bias"))
    return float(np.sum(y * dy) + np.sum(hf * dh))


def test_torch_forward_matches_the_c_oracle(orc):
    d = _inputs(1, b=2, L=9, H=4, G=2, P=3, N=6, R=2, cont=False)
    y, hf = backward.scan_forward(**{k: torch.as_tensor(v) for k, v in d.items()})
    y_ref, hf_ref = orc.scan_seq(d["x"], d["dt"], d["A"], d["lam"], d["B"], d["C"], d["theta"],
                                 d["B_bias"], d["C_bias"])
    assert np.allclose(y.numpy(), y_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(hf.numpy(), hf_ref, rtol=1e-12, atol=1e-12)


def test_torch_forward_continues_from_a_state(orc):
    d = _inputs(2)
    y, hf = backward.scan_forward(**{k: torch.as_tensor(v) for k, v in d.items()})
    y_ref, hf_ref = orc.decode_tokens(d["state0"], d["x"], d["dt"], d["A"], d["lam"], d["B"],
                                      d["C"], d["theta"], B_prev=d["B_prev"], x_prev=d["x_prev"],
                                      B_bias=d["B_bias"], C_bias=d["C_bias"])
    assert np.allclose(y.numpy(), y_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(hf.numpy(), hf_ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("R", [1, 2])
def test_gradients_match_finite_differences(orc, R):
    d = _inputs(3 + R, R=R)
    rng = np.random.default_rng(10 + R)
    b, L, H, P, _ = d["x"].shape
    N = d["B"].shape[3]
    dy = rng.standard_normal((b, L, H, P, R))
    dh = rng.standard_normal((b, H, N, P))
    g = backward.scan_grads(dy=dy, dh=dh, **d)
    assert set(g) == set(d)
    eps = 1e-6
    for name, arr in d.items():
        flat = arr.reshape(-1)
        for i in rng.choice(flat.size, size=min(4, flat.size), replace=False):
            plus = {k: v.copy() for k, v in d.items()}
            minus = {k: v.copy() for k, v in d.items()}
            plus[name].reshape(-1)[i] += eps
            minus[name].reshape(-1)[i] -= eps
            fd = (_c_loss(orc, plus, dy, dh) - _c_loss(orc, minus, dy, dh)) / (2 * eps)
            ad = g[name].reshape(-1)[i]
            assert abs(ad - fd) <= 1e-6 * max(1.0, abs(fd)), (name, int(i), ad, fd)


def test_gradient_of_a_sequence_start_has_no_previous_token_terms():
    """Without a previous token the first token's beta term is absent: the
    gradient with respect to lambda_0 comes from gamma_0 alone, so moving
    lambda_0 changes y_0 through gamma_0 B_0 x_0^T only (a closed form)."""
    d = _inputs(7, L=1, H=1, P=2, N=2, R=1, cont=False)
    dy = np.ones((1, 1, 1, 2, 1))
    g = backward.scan_grads(dy=dy, **d)
    # y_0 = C0^T (gamma_0 U_0): d y / d lambda_0 = dt_0 C0^T U_0, summed over p
    Bb = d["B"][0, 0, 0, :, 0] + d["B_bias"][0, :, 0]
    Cb = d["C"][0, 0, 0, :, 0] + d["C_bias"][0, :, 0]
    U = np.outer(Bb, d["x"][0, 0, 0, :, 0])
    expect = d["dt"][0, 0, 0] * float(Cb @ U @ np.ones(2))
    assert g["lam"][0, 0, 0] == pytest.approx(expect, rel=1e-12)
