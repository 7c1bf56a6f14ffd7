"""GPU parity of the rank-4 decode step whose update runs on the tensor cores.

bf16 activations with R = 4 and P = 64 take the mma.sync kernel when N is a
multiple of 16 up to 128: the rank-8 update U [x_prev | x]^T is computed in bf16 with U split
into high and low bf16 parts. The split leaves U about 16 bits, so the fp32
state stays within 1e-4 of the fp64 oracle (max error over RMS) after several
steps; a kernel that dropped the low part would miss that bar by an order of
magnitude. Other N fall back to the FMA streaming kernel and must agree all
the same.
"""
import numpy as np
import pytest

import m3synth
from gpu_util import assert_bf16_out, max_over_rms, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import selective_state_space_129_b300 as m3  # noqa: E402

STATE_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m3.load()
    yield
    assert m3.m3_device_status() == 0


def _run(orc, batch, H, G, N, bias, steps, seed):
    shape = m3synth.ScanShape(batch, 1, H, G, 64, N, R=4, chunk=1, bf16=True)
    st_ref = 0.5 * np.random.default_rng(seed).standard_normal((batch, H, N, 64))
    st = torch.from_numpy(st_ref.astype(np.float32)).cuda()
    st_ref = st.cpu().numpy().astype(np.float64)
    prev, prev_h = None, None
    worst = 0.0
    for i in range(steps):
        s_ = m3synth.decode_inputs(shape, seed=seed, step=i)
        if not bias:
            s_["B_bias"] = s_["C_bias"] = None
        d = to_device({k: v for k, v in s_.items() if v is not None}, True)
        kw = dict(B_prev=prev["B"], x_prev=prev["x"]) if prev is not None else {}
        out = m3.m3_decode_step(st, d["x"], d["dt"], d["A"], d["lam"], d["B"], d["C"],
                                d["theta"], R=4, B_bias=d.get("B_bias"), C_bias=d.get("C_bias"),
                                **kw)
        okw = dict(B_prev=prev_h["B"], x_prev=prev_h["x"]) if prev_h is not None else {}
        y_ref, st_ref = orc.decode_step(st_ref, s_["x"], s_["dt"], s_["A"], s_["lam"], s_["B"],
                                        s_["C"], s_["theta"], B_bias=s_["B_bias"],
                                        C_bias=s_["C_bias"], **okw)
        torch.cuda.synchronize()
        assert_bf16_out(out.float().cpu().numpy(), y_ref, "y step %d" % i)
        e = max_over_rms(st.cpu().numpy(), st_ref)
        worst = max(worst, e)
        assert e <= STATE_TOL, "state after step %d: max|err|/RMS %.3e" % (i, e)
        prev, prev_h = d, s_
    assert m3.m3_device_status() == m3.M3_OK
    return worst


@pytest.mark.parametrize("N", [16, 48, 96, 128])
@pytest.mark.parametrize("bias", [True, False], ids=["bias", "nobias"])
def test_decode_rank4_mma(orc, N, bias):
    """One to eight row tiles of 16 state rows; 4 x 2 heads in two groups, three
    steps (the first without a previous token)."""
    worst = _run(orc, 4, 8, 2, N, bias, 3, seed=90 + N)
    print("decode R=4 N=%d %s: state max|err|/RMS %.2e" % (N, "bias" if bias else "nobias", worst))


def test_decode_rank4_many_units_per_cta(orc):
    """batch 80 x 8 heads at N = 16: 640 units, more than two per CTA of the
    persistent grid, so both stages are refilled several times."""
    _run(orc, 80, 8, 1, 16, True, 2, seed=97)


@pytest.mark.parametrize("N", [40, 144, 256])
def test_decode_rank4_other_state_sizes_fall_back(orc, N):
    """N = 40 (not a multiple of 16), 144 and 256 (above 128) take the FMA
    streaming kernel, to the same bar."""
    _run(orc, 2, 4, 1, N, True, 2, seed=98)


# ---------------------------------------------------------------- K tokens per call
def _run_tokens(orc, batch, K, H, G, N, bias, prev, seed):
    shape = m3synth.ScanShape(batch, K, H, G, 64, N, R=4, chunk=1, bf16=True)
    inp = m3synth.scan_inputs(shape, seed=seed)
    if not bias:
        inp["B_bias"] = inp["C_bias"] = None
    st0 = (0.5 * np.random.default_rng(seed).standard_normal((batch, H, N, 64))).astype(np.float32)
    pv = m3synth.decode_inputs(shape, seed=seed + 1, step=0) if prev else None
    d = to_device({k: v for k, v in inp.items() if v is not None}, True)
    kw = {}
    if pv is not None:
        dp = to_device(pv, True)
        kw = dict(B_prev=dp["B"], x_prev=dp["x"])
    st = torch.from_numpy(st0).cuda()
    out = m3.m3_decode_tokens(st, d["x"], d["dt"], d["A"], d["lam"], d["B"], d["C"], d["theta"],
                              R=4, B_bias=d.get("B_bias"), C_bias=d.get("C_bias"), **kw)
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    okw = dict(B_prev=pv["B"], x_prev=pv["x"]) if pv is not None else {}
    y_ref, st_ref = orc.decode_tokens(st0, inp["x"], inp["dt"], inp["A"], inp["lam"], inp["B"],
                                      inp["C"], inp["theta"], B_bias=inp["B_bias"],
                                      C_bias=inp["C_bias"], **okw)
    assert_bf16_out(out.float().cpu().numpy(), y_ref, "y")
    e = max_over_rms(st.cpu().numpy(), st_ref)
    assert e <= STATE_TOL, "state after %d tokens: max|err|/RMS %.3e" % (K, e)
    return e


@pytest.mark.parametrize("N,K,bias,prev", [
    (16, 1, True, True),     # one token through the K-token kernel
    (48, 5, False, False),   # no bias, no token before the block
    (128, 8, True, True),    # the serving block: one window of eight tokens
    (128, 16, True, True),   # three windows of tables (7, 7, 2 tokens)
    (64, 24, True, False),   # two windows at N = 64
])
def test_decode_tokens_rank4_mma(orc, N, K, bias, prev):
    e = _run_tokens(orc, 3, K, 8, 2, N, bias, prev, seed=200 + N + K)
    print("decode tokens R=4 N=%d K=%d: state max|err|/RMS %.2e" % (N, K, e))
