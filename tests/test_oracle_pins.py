"""Pins for the CPU oracle: facts fixed by the Mamba-3 pages and by mathematics.

Each test checks the oracle against something other than itself: a special
case that reduces to another recurrence, a closed form, an invariant, an
independent formulation, or a hand-derived fixture. Chosen so that a dropped
term, a wrong sign or index, or a transposed operand fails at least one.
"""
import cmath
import math
import os

import numpy as np
import pytest

import m3synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_inputs(seed, b=2, L=20, H=4, G=2, P=3, N=4, R=1, bias=True):
    rng = np.random.default_rng(seed)
    d = dict(
        x=rng.standard_normal((b, L, H, P, R)),
        dt=np.log1p(np.exp(rng.normal(-1.0, 0.5, (b, L, H)))),
        A=-np.exp(rng.uniform(0, math.log(16), H)),
        lam=1 / (1 + np.exp(-rng.standard_normal((b, L, H)))),
        B=rng.standard_normal((b, L, G, N, R)) / math.sqrt(N),
        C=rng.standard_normal((b, L, G, N, R)) / math.sqrt(N),
        theta=rng.uniform(-math.pi, math.pi, (b, L, G, N // 2)),
        B_bias=rng.normal(0, 0.1, (H, N, R)) if bias else None,
        C_bias=rng.normal(0, 0.1, (H, N, R)) if bias else None,
    )
    return d


def _rel(a, b):
    return float(np.linalg.norm(np.ravel(a - b)) / max(np.linalg.norm(np.ravel(b)), 1e-300))


# ---------------------------------------------------------------------------
# 1. lambda = 1, theta = 0, R = 1 reduces to the Mamba-2 Euler recurrence
#    ("MAMBA-3: IMPROVED SEQUENCE MODELING USING STATE SPACE PRINCIPLES" (aipaper.cc), sec. 4.1: "When lambda_t = 1, this rule reduces to Mamba-2's
#    Euler method"; the Euler rule h_t = e^{Delta A} h_{t-1} + Delta B_t x_t).
# ---------------------------------------------------------------------------
def test_euler_reduction(orc):
    d = _rand_inputs(1)
    d["lam"][:] = 1.0
    d["theta"][:] = 0.0
    y, st = orc.scan_seq(**d)
    b, L, H, P, R = d["x"].shape
    G, N = d["B"].shape[2], d["B"].shape[3]
    y_ref = np.zeros_like(y)
    st_ref = np.zeros((b, H, N, P))
    for bi in range(b):
        for h in range(H):
            g = h // (H // G)
            hs = np.zeros((N, P))
            for t in range(L):
                Bt = d["B"][bi, t, g, :, 0] + d["B_bias"][h, :, 0]
                Ct = d["C"][bi, t, g, :, 0] + d["C_bias"][h, :, 0]
                dl = d["dt"][bi, t, h]
                hs = math.exp(dl * d["A"][h]) * hs + dl * np.outer(Bt, d["x"][bi, t, h, :, 0])
                y_ref[bi, t, h, :, 0] = Ct @ hs
            st_ref[bi, h] = hs
    assert _rel(y, y_ref) < 1e-13
    assert _rel(st, st_ref) < 1e-13


# ---------------------------------------------------------------------------
# 2. Convergence order on a smooth complex ODE with a closed-form solution.
#    h'(tau) = (A + i w) h + b u(tau), u = sin(W tau), h(0) = 0.
#    The exponential-trapezoidal rule (lambda = 1/2) is second order, the
#    exponential-Euler rule (lambda = 1) first order ("Mamba-3: Improved Sequence Modeling using State Space Principles" (papernotes.org), sec. 1:
#    local error O(Delta^2) vs O(Delta^3)). A non-uniform grid pins that beta
#    uses the current step's Delta, and the complex rate pins that the
#    previous-input term is rotated as well.
# ---------------------------------------------------------------------------
def _ode_error(orc, K, lam_val, T=2.0, A=-1.0, w=2.0, W=3.0, b=(0.7, -0.4)):
    u = np.arange(K + 1) / K
    tau = T * (u + 0.3 * np.sin(2 * math.pi * u) / (2 * math.pi))
    dts = np.diff(tau)                     # token t covers (tau_t, tau_{t+1}]
    L = K
    x = np.sin(W * tau[1:]).reshape(1, L, 1, 1, 1)
    dt = dts.reshape(1, L, 1)
    lam = np.full((1, L, 1), lam_val)
    Bm = np.tile(np.array(b).reshape(1, 1, 1, 2, 1), (1, L, 1, 1, 1))
    Cm = np.tile(np.array([1.0, 0.0]).reshape(1, 1, 1, 2, 1), (1, L, 1, 1, 1))
    theta = np.full((1, L, 1, 1), w)
    _, st = orc.scan_seq(x, dt, np.array([A]), lam, Bm, Cm, theta)
    h_num = st[0, 0, 0, 0] + 1j * st[0, 0, 1, 0]
    z = complex(A, w)
    bc = complex(*b)
    e = lambda s: cmath.exp(s * T)
    h_ex = bc / 2j * ((e(1j * W) - e(z)) / (1j * W - z) - (e(-1j * W) - e(z)) / (-1j * W - z))
    return abs(h_num - h_ex)


@pytest.mark.parametrize("lam_val,order", [(0.5, 2.0), (1.0, 1.0)])
def test_convergence_order(orc, lam_val, order):
    errs = [_ode_error(orc, K, lam_val) for K in (64, 128, 256, 512)]
    rates = [math.log2(errs[i] / errs[i + 1]) for i in range(len(errs) - 1)]
    assert all(abs(r - order) < 0.15 for r in rates), (errs, rates)


# ---------------------------------------------------------------------------
# 3. Constant inputs: geometric series closed form. With z = alpha e^{i phi}
#    per state pair, h_t = z^t gamma U + (z beta_hat + gamma) U (1 - z^t)/(1 - z).
#    Pins the rotation direction ([[c,-s],[s,c]] = multiplication by e^{i phi},
#    "State Space Models 家族对比分析：S4 → Mamba → Mamba-2 → Mamba-3" (metaphor-xennon blog), sec. 2.2) and the weights of both input terms.
# ---------------------------------------------------------------------------
def test_geometric_series(orc):
    rng = np.random.default_rng(3)
    L, P, N, R = 12, 3, 6, 2
    dt0, lam0, A0 = 0.37, 0.3, -0.8
    th = rng.uniform(-math.pi, math.pi, N // 2)
    Bv = rng.standard_normal((N, R))
    Cv = rng.standard_normal((N, R))
    xv = rng.standard_normal((P, R))
    x = np.tile(xv, (1, L, 1, 1, 1)).reshape(1, L, 1, P, R)
    dt = np.full((1, L, 1), dt0)
    lam = np.full((1, L, 1), lam0)
    Bm = np.tile(Bv, (1, L, 1, 1, 1)).reshape(1, L, 1, N, R)
    Cm = np.tile(Cv, (1, L, 1, 1, 1)).reshape(1, L, 1, N, R)
    theta = np.tile(th, (1, L, 1, 1)).reshape(1, L, 1, N // 2)
    y, _ = orc.scan_seq(x, dt, np.array([A0]), lam, Bm, Cm, theta)
    alpha, gamma, bhat = math.exp(dt0 * A0), lam0 * dt0, (1 - lam0) * dt0
    Ureal = Bv @ xv.T                                  # N x P
    Uc = Ureal[0::2] + 1j * Ureal[1::2]                # pairs -> complex, (N/2) x P
    z = alpha * np.exp(1j * dt0 * th)[:, None]
    for t in range(L):
        hc = z ** t * gamma * Uc + (z * bhat + gamma) * Uc * (1 - z ** t) / (1 - z)
        hr = np.empty((N, P))
        hr[0::2], hr[1::2] = hc.real, hc.imag
        y_ex = (Cv.T @ hr).T                           # P x R
        assert np.allclose(y[0, t, 0], y_ex, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# 4. Prop. 3 ("MAMBA-3: IMPROVED SEQUENCE MODELING USING STATE SPACE PRINCIPLES" (aipaper.cc), sec. 4.2): the real SSM with the cumulative rotation
#    applied to B and C equals the complex (explicitly rotated) SSM.
# ---------------------------------------------------------------------------
def test_rope_form_equals_explicit_rotation(orc):
    d = _rand_inputs(4, b=2, L=40, H=4, G=2, P=5, N=8, R=2)
    y1, s1 = orc.scan_seq(**d)
    y2, s2 = orc.scan_rope(**d)
    assert _rel(y2, y1) < 1e-12
    assert _rel(s2, s1) < 1e-12


# ---------------------------------------------------------------------------
# 5. Parity ("Mamba-3: Improved Sequence Modeling using State Space Principles" (papernotes.org), sec. 2, rotation R(pi x_t)); hand fixture.
# ---------------------------------------------------------------------------
def _read_kv(path):
    out = {}
    for line in open(path):
        line = line.split("#")[0].strip()
        if "=" in line:
            k, v = line.split("=", 1)
            out[k.strip()] = v.strip()
    return out


def test_parity_fixture(orc):
    kv = _read_kv(os.path.join(GOLDEN, "parity_bits.txt"))
    bits = np.array([int(s) for s in kv["bits"].split()], dtype=np.float64)
    signs = np.array([1.0 if s == "+" else -1.0 for s in kv["signs"].split()])
    L = len(bits)
    rng = np.random.default_rng(5)
    N, P, R = 6, 4, 1
    dt = np.log1p(np.exp(rng.normal(-1, 0.5, L))).reshape(1, L, 1)
    lam = rng.uniform(0.1, 0.9, (1, L, 1))
    theta = np.tile((math.pi * bits / dt[0, :, 0])[:, None], (1, N // 2)).reshape(1, L, 1, N // 2)
    Bv = rng.standard_normal((N, R))
    Cv = rng.standard_normal((N, R))
    x = np.zeros((1, L, 1, P, R))
    x[0, 0, 0] = rng.standard_normal((P, R))
    Bm = np.tile(Bv, (1, L, 1, 1, 1)).reshape(1, L, 1, N, R)
    Cm = np.tile(Cv, (1, L, 1, 1, 1)).reshape(1, L, 1, N, R)
    y, _ = orc.scan_seq(x, dt, np.zeros(1), lam, Bm, Cm, theta)
    U0 = Bv @ x[0, 0, 0].T
    base = (lam[0, 0, 0] * dt[0, 0, 0] + (1 - lam[0, 1, 0]) * dt[0, 1, 0]) * (Cv.T @ U0).T
    for t in range(1, L):
        ratio = y[0, t, 0] / base
        assert np.allclose(ratio, signs[t - 1], rtol=1e-9, atol=0), (t, ratio)
    assert np.allclose(y[0, 0, 0], lam[0, 0, 0] * dt[0, 0, 0] * (Cv.T @ U0).T, rtol=1e-12)


# ---------------------------------------------------------------------------
# 6. Rotation preserves the norm: with A = 0 and no input after t = 0, the
#    state only rotates from t = 2 on.
# ---------------------------------------------------------------------------
def test_rotation_preserves_norm(orc):
    d = _rand_inputs(6, b=1, L=12, H=2, G=1, P=3, N=8, R=2)
    d["A"][:] = 0.0
    d["x"][:, 1:] = 0.0
    norms = []
    for Lp in range(2, 12):
        sub = {k: (v[:, :Lp] if (v is not None and k not in ("A", "B_bias", "C_bias")) else v)
               for k, v in d.items()}
        _, st = orc.scan_seq(**sub)
        norms.append(np.linalg.norm(st, axis=(2, 3)))
    norms = np.array(norms)
    assert np.allclose(norms, norms[0:1], rtol=1e-13)


# ---------------------------------------------------------------------------
# 7. Chunked SSD form equals the sequential recurrence for any chunk size,
#    including a partial last chunk and a chunk longer than the sequence.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [1, 2, 4, 16, 64, 50])
@pytest.mark.parametrize("R", [1, 3])
def test_chunked_equals_sequential(orc, chunk, R):
    d = _rand_inputs(7 + R, b=2, L=50, H=4, G=2, P=5, N=8, R=R)
    y1, s1 = orc.scan_seq(**d)
    y2, s2 = orc.scan_chunked(chunk=chunk, **d)
    assert _rel(y2, y1) < 1e-11
    assert _rel(s2, s1) < 1e-11


# ---------------------------------------------------------------------------
# 8. Structured-mask form:
#    "Mamba-3: Improved Sequence Modeling using State Space Principles" (papernotes.org), sec. 1;
#    "Mamba-3: Improved Sequence Modeling using State Space Principles" (bud-325 notes), Key claims:
#    the whole-sequence mask is (1-semiseparable decay) @ (2-band matrix) with
#    gamma_s on the diagonal and beta_{s'} on the sub-diagonal; Y = (M o C B^T) X
#    in the frame rotated by the cumulative angle (SSD form,
#    "State Space Models 家族对比分析：S4 → Mamba → Mamba-2 → Mamba-3" (metaphor-xennon blog), sec. 1.3). Built densely here with numpy.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("rotate", [False, True])
def test_dense_mask_product_form(orc, rotate):
    d = _rand_inputs(8, b=1, L=24, H=1, G=1, P=4, N=6, R=1)
    if not rotate:
        d["theta"][:] = 0.0
    y, _ = orc.scan_seq(**d)
    L = d["x"].shape[1]
    dt, lam, A = d["dt"][0, :, 0], d["lam"][0, :, 0], d["A"][0]
    alpha = np.exp(dt * A)
    Ldec = np.zeros((L, L))
    for t in range(L):
        for s in range(t + 1):
            Ldec[t, s] = np.prod(alpha[s + 1:t + 1])
    band = np.diag(lam * dt)
    for s in range(1, L):
        band[s, s - 1] = (1 - lam[s]) * dt[s] * alpha[s]
    M = Ldec @ band
    Bt = d["B"][0, :, 0, :, 0] + d["B_bias"][0, :, 0]
    Ct = d["C"][0, :, 0, :, 0] + d["C_bias"][0, :, 0]
    Phi = np.cumsum(dt[:, None] * d["theta"][0, :, 0], axis=0)     # L x N/2
    c, s = np.cos(Phi), np.sin(Phi)

    def rot_minus(V):   # Rot(-Phi_t) per token on pairs
        W = np.empty_like(V)
        W[:, 0::2] = c * V[:, 0::2] + s * V[:, 1::2]
        W[:, 1::2] = -s * V[:, 0::2] + c * V[:, 1::2]
        return W

    Bq, Cq = rot_minus(Bt), rot_minus(Ct)
    Y = (M * (Cq @ Bq.T)) @ d["x"][0, :, 0, :, 0]
    assert np.allclose(Y, y[0, :, 0, :, 0], rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# 9. MIMO = sum of R^2 SISO calls ("Mamba-3: Improved Sequence Modeling using State Space Principles" (papernotes.org), sec. 3): output column r'
#    equals sum over r of the SISO scan with (B_r, x_r, C_r').
# ---------------------------------------------------------------------------
def test_mimo_is_sum_of_siso(orc):
    R = 3
    d = _rand_inputs(9, b=1, L=30, H=2, G=1, P=4, N=6, R=R)
    y, st = orc.scan_seq(**d)
    y_sum = np.zeros_like(y)
    st_sum = np.zeros_like(st)
    for r in range(R):
        for r2 in range(R):
            sub = dict(d)
            sub["x"] = d["x"][..., r:r + 1]
            sub["B"] = d["B"][..., r:r + 1]
            sub["C"] = d["C"][..., r2:r2 + 1]
            sub["B_bias"] = d["B_bias"][..., r:r + 1]
            sub["C_bias"] = d["C_bias"][..., r2:r2 + 1]
            ys, ss = orc.scan_seq(**sub)
            y_sum[..., r2] += ys[..., 0]
            if r2 == 0:
                st_sum += ss
    assert _rel(y_sum, y) < 1e-12
    assert _rel(st_sum, st) < 1e-12


# ---------------------------------------------------------------------------
# 10. Prefill then one decode step equals prefill of one more token.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("R", [1, 2])
def test_prefill_then_decode(orc, R):
    d = _rand_inputs(10, b=2, L=17, H=4, G=2, P=3, N=6, R=R)
    y_full, st_full = orc.scan_seq(**d)
    pre = {k: (v[:, :16] if k in ("x", "dt", "lam", "B", "C", "theta") else v)
           for k, v in d.items()}
    _, st16 = orc.scan_seq(**pre)
    t = 16
    y1, st17 = orc.decode_step(
        st16, d["x"][:, t], d["dt"][:, t], d["A"], d["lam"][:, t], d["B"][:, t], d["C"][:, t],
        d["theta"][:, t], B_prev=d["B"][:, t - 1], x_prev=d["x"][:, t - 1],
        B_bias=d["B_bias"], C_bias=d["C_bias"])
    assert _rel(y1, y_full[:, t]) < 1e-12
    assert _rel(st17, st_full) < 1e-12
    # the first token decoded from a zero state equals a length-1 prefill
    y0, s0 = orc.decode_step(
        np.zeros_like(st16), d["x"][:, 0], d["dt"][:, 0], d["A"], d["lam"][:, 0], d["B"][:, 0],
        d["C"][:, 0], d["theta"][:, 0], B_bias=d["B_bias"], C_bias=d["C_bias"])
    one = {k: (v[:, :1] if k in ("x", "dt", "lam", "B", "C", "theta") else v) for k, v in d.items()}
    y_one, s_one = orc.scan_seq(**one)
    assert _rel(y0, y_one[:, 0]) < 1e-13 and _rel(s0, s_one) < 1e-13


# ---------------------------------------------------------------------------
# 10b. K decode tokens in one block continue a prefill exactly: prefill of
#      L tokens, then tokens L .. L+K-1 decoded together, equals the prefill
#      of L + K tokens (outputs of the decoded tokens and the final state);
#      from a zero state with no previous token it equals a K-token prefill.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("R", [1, 4])
def test_decode_tokens_continue_prefill(orc, R):
    import oracle.oracle as om
    L, K = 11, 5
    d = _rand_inputs(12, b=2, L=L + K, H=4, G=2, P=3, N=6, R=R)
    seq = ("x", "dt", "lam", "B", "C", "theta")
    y_full, st_full = orc.scan_seq(**d)
    _, stL = orc.scan_seq(**{k: (v[:, :L] if k in seq else v) for k, v in d.items()})
    blk = {k: d[k][:, L:] for k in seq}
    y, st = om.decode_tokens(stL, blk["x"], blk["dt"], d["A"], blk["lam"], blk["B"], blk["C"],
                             blk["theta"], B_prev=d["B"][:, L - 1], x_prev=d["x"][:, L - 1],
                             B_bias=d["B_bias"], C_bias=d["C_bias"])
    assert y.shape == y_full[:, L:].shape
    assert _rel(y, y_full[:, L:]) < 1e-12
    assert _rel(st, st_full) < 1e-12
    first = {k: d[k][:, :K] for k in seq}
    y0, s0 = om.decode_tokens(np.zeros_like(stL), first["x"], first["dt"], d["A"], first["lam"],
                              first["B"], first["C"], first["theta"], B_bias=d["B_bias"],
                              C_bias=d["C_bias"])
    y_pre, s_pre = orc.scan_seq(**{k: (v[:, :K] if k in seq else v) for k, v in d.items()})
    assert _rel(y0, y_pre) < 1e-12 and _rel(s0, s_pre) < 1e-12


# ---------------------------------------------------------------------------
# 11. Hand-derived two-token example (fixture).
# ---------------------------------------------------------------------------
def _ev(expr):
    return float(eval(expr, {"__builtins__": {}}, {"log": math.log, "pi": math.pi}))


def _rows(s):
    return [[_ev(v) for v in row.split(",")] for row in s.split(";")]


def test_hand_two_tokens(orc):
    kv = _read_kv(os.path.join(GOLDEN, "hand_two_tokens.txt"))
    L = 2
    x = np.array(_rows(kv["x"])).reshape(1, L, 1, 1, 1)
    dt = np.array(_rows(kv["dt"])).reshape(1, L, 1)
    lam = np.array(_rows(kv["lam"])).reshape(1, L, 1)
    theta = np.array(_rows(kv["theta"])).reshape(1, L, 1, 1)
    Bm = np.array(_rows(kv["B"])).reshape(1, L, 1, 2, 1)
    Cm = np.array(_rows(kv["C"])).reshape(1, L, 1, 2, 1)
    A = np.array([_ev(kv["A"])])
    for fn in (orc.scan_seq, orc.scan_rope):
        y, st = fn(x, dt, A, lam, Bm, Cm, theta)
        assert np.allclose(y.ravel(), np.array(_rows(kv["y"])).ravel(), atol=1e-14)
        assert np.allclose(st.ravel(), np.array(_rows(kv["final_state"])).ravel(), atol=1e-14)
    y, st = orc.scan_chunked(x, dt, A, lam, Bm, Cm, theta, chunk=2)
    assert np.allclose(y.ravel(), np.array(_rows(kv["y"])).ravel(), atol=1e-14)


# ---------------------------------------------------------------------------
# 12. Regression samples written by tests/golden/make_golden.py (oracle only).
# ---------------------------------------------------------------------------
def test_tiny_workload_samples(orc):
    path = os.path.join(GOLDEN, "tiny_oracle_samples.txt")
    inp = m3synth.scan_inputs(m3synth.TINY, seed=0)
    y, st = orc.scan_seq(inp["x"], inp["dt"], inp["A"], inp["lam"], inp["B"], inp["C"],
                         inp["theta"], inp["B_bias"], inp["C_bias"])
    n = 0
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        kind, idx, val = line.split()
        ix = tuple(int(v) for v in idx.split(","))
        got = y[ix] if kind == "y" else st[ix]
        assert abs(got - float(val)) <= 1e-12 * max(1.0, abs(float(val))), (kind, ix, got, val)
        n += 1
    assert n >= 16


def test_generator_is_bf16_exact_and_seeded():
    a = m3synth.scan_inputs(m3synth.small_shape(bf16=True, rms_bc=True), seed=11)
    b = m3synth.scan_inputs(m3synth.small_shape(bf16=True, rms_bc=True), seed=11)
    for k in a:
        assert np.array_equal(a[k], b[k])
    for k in ("x", "B", "C"):
        assert np.array_equal(m3synth.to_bf16(a[k]), a[k])
    # ties to even: 1 + 2^-8 lies halfway between two bf16 values -> rounds to 1
    v = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8], np.float32)
    assert m3synth.to_bf16(v).tolist() == [1.0, 1.0 + 2.0 ** -6]


# ---------------------------------------------------------------------------
# BCNorm ("Mamba-3: Improved Sequence Modeling using State Space Principles" (papernotes.org), sec. 4; "Mamba-3: Improved Sequence Modeling using State Space Principles" (bud-325 notes), Key claims): RMS normalisation
# over N per (b, t, g, r) with no weight, eps = 1e-6 under the root.
# ---------------------------------------------------------------------------
def _read_bc_fixture():
    import math as m
    vals = {}
    with open(os.path.join(GOLDEN, "bc_norm_hand.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rhs = line.partition("=")
            rows = [[eval(v, {"sqrt": m.sqrt}) for v in row.split(",")] for row in rhs.split(";")]
            vals[key.strip()] = np.array(rows, dtype=np.float64)
    return vals


def test_bc_norm_hand_fixture(orc):
    fx = _read_bc_fixture()
    got = orc.bc_norm(fx["in"].reshape(1, 1, 1, 4, 2))
    assert np.allclose(got.reshape(4, 2), fx["out"], rtol=1e-14, atol=0)


def test_bc_norm_invariants(orc):
    rng = np.random.default_rng(7)
    v = rng.standard_normal((2, 5, 3, 16, 4)) * rng.uniform(0.01, 10.0, (2, 5, 3, 1, 4))
    out = orc.bc_norm(v)
    ms = np.mean(v * v, axis=3, keepdims=True)
    # mean square of every normalised vector over N is ms / (ms + eps)
    assert np.allclose(np.mean(out * out, axis=3, keepdims=True), ms / (ms + 1e-6), rtol=1e-12)
    # direction is kept and each vector is normalised on its own: the ratio
    # out / in is one positive constant per (b, t, g, r)
    ratio = out / v
    assert np.all(ratio > 0)
    assert np.allclose(ratio, ratio[:, :, :, :1, :], rtol=1e-12)
    # every rank is normalised on its own: R = 4 equals four R = 1 calls
    for r in range(4):
        assert np.allclose(orc.bc_norm(v[..., r:r + 1])[..., 0], out[..., r], rtol=1e-14)


def test_bc_norm_matches_the_input_recipe(orc):
    """The input generator's RMS normalisation (the workloads' recipe, written
    separately) and the oracle's agree on the same raw draw."""
    rng = np.random.Generator(np.random.PCG64(11))
    raw = rng.standard_normal((2, 9, 1, 128, 4), dtype=np.float32)
    rng = np.random.Generator(np.random.PCG64(11))
    recipe = m3synth._bc(rng, (2, 9, 1, 128, 4), 128, rms=True)
    assert np.allclose(orc.bc_norm(raw), recipe, rtol=2e-7, atol=0)
