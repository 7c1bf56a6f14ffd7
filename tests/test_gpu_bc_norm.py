"""GPU parity of the prefill with BCNorm fused into its prologue
(M3_FLAG_BC_NORM): the kernel takes un-normalised B and C; the oracle is the
sequential scan of the oracle's own BCNorm of them ("Mamba-3: Improved Sequence
Modeling using State Space Principles" (papernotes.org), sec. 4).

The raw B and C are the workload recipe's vectors times a random positive
scale per (b, t, g, r) vector (0.05 .. 20), rounded to bf16, so that the
normalisation changes every vector. Tolerances are those of tests/gpu_util.py.
"""
import numpy as np
import pytest

import m3synth
from gpu_util import assert_bf16, assert_bf16_out, head_slice, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import selective_state_space_129_b300 as m3  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m3.load()
    yield
    assert m3.m3_device_status() == 0


def _raw_bc(inp, seed):
    """Replace B and C by un-normalised bf16 vectors (recipe vector times a
    per-vector scale); returns the dict (modified in place)."""
    rng = np.random.default_rng(seed)
    for k in ("B", "C"):
        v = inp[k]
        s = rng.uniform(0.05, 20.0, size=v.shape[:3] + (1,) + v.shape[4:]).astype(np.float32)
        inp[k] = m3synth.to_bf16(v * s)
    return inp


def _oracle_bc(orc, inp):
    return orc.scan_seq(inp["x"], inp["dt"], inp["A"], inp["lam"], orc.bc_norm(inp["B"]),
                        orc.bc_norm(inp["C"]), inp["theta"], inp["B_bias"], inp["C_bias"],
                        nthreads=0)


def _gpu_bc(inp, shape):
    d = to_device(inp, True)
    out, fs = m3.m3_scan_fwd(d["x"], d["dt"], d["A"], d["lam"], d["B"], d["C"], d["theta"],
                             R=shape.R, chunk=shape.chunk, B_bias=d["B_bias"],
                             C_bias=d["C_bias"], bc_norm=True)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), fs.cpu().numpy()


CASES = [
    # L, chunk, R, G, H, N
    (200, 64, 1, 1, 2, 128),   # three chunks and a ragged tail
    (77, 64, 1, 2, 4, 64),
    (97, 32, 2, 2, 4, 64),
    (150, 32, 2, 1, 2, 128),
    (83, 16, 4, 2, 4, 128),
    (64, 16, 4, 1, 2, 64),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "L%d_Q%d_R%d_G%d_H%d_N%d" % c)
def test_bc_norm_prefill_small(orc, case):
    L, Q, R, G, H, N = case
    shape = m3synth.ScanShape(2, L, H, G, 64, N, R=R, chunk=Q, bf16=True, rms_bc=True)
    inp = _raw_bc(m3synth.scan_inputs(shape, seed=700 + L + R), seed=L)
    y, fs = _gpu_bc(inp, shape)
    y_ref, fs_ref = _oracle_bc(orc, inp)
    assert_bf16_out(y, y_ref, "y")
    assert_bf16(fs, fs_ref, "final_state")


@pytest.mark.parametrize("name", ["prefill_siso", "prefill_mimo"])
def test_bc_norm_prefill_1p5b_sampled(orc, name):
    """The 1.5B-layer SISO and MIMO workloads at full size, four sampled heads."""
    idx, shape = m3synth.WORKLOADS[name]
    inp = _raw_bc(m3synth.scan_inputs(shape, seed=idx), seed=idx)
    y, fs = _gpu_bc(inp, shape)
    rng = np.random.default_rng(21)
    for _ in range(4):
        b, h = int(rng.integers(shape.batch)), int(rng.integers(shape.heads))
        y_ref, fs_ref = _oracle_bc(orc, head_slice(inp, b, h))
        assert_bf16_out(y[b:b + 1, :, h:h + 1], y_ref, "y[b=%d,h=%d]" % (b, h))
        assert_bf16(fs[b:b + 1, h:h + 1], fs_ref, "state[b=%d,h=%d]" % (b, h))


@pytest.mark.parametrize("L,R", [(3000, 1), (1000, 4)], ids=["R1", "R4"])
def test_bc_norm_segmented_prefill(orc, L, R):
    """Few sequences, so the call runs segmented (state-only pass, combine,
    full pass), each pass normalising B (and C) itself; SISO and MIMO R = 4."""
    Q = 64 // R
    shape = m3synth.ScanShape(1, L, 2, 1, 64, 128, R=R, chunk=Q, bf16=True, rms_bc=True)
    dims = m3.make_dims(1, L, 2, 1, 64, 128, m3.M3_BF16)
    assert m3.m3_scan_workspace_bytes(dims, R, Q) > 0, "expected a segmented launch"
    inp = _raw_bc(m3synth.scan_inputs(shape, seed=77), seed=78)
    y, fs = _gpu_bc(inp, shape)
    y_ref, fs_ref = _oracle_bc(orc, inp)
    assert_bf16_out(y, y_ref, "y")
    assert_bf16(fs, fs_ref, "final_state")


def test_bc_norm_of_normalised_inputs_changes_little():
    """Inputs already RMS-normalised: with and without the flag the results
    agree to the kernels' rounding (the normalisation is then ~ identity)."""
    shape = m3synth.ScanShape(2, 256, 4, 1, 64, 128, R=1, chunk=64, bf16=True, rms_bc=True)
    d = to_device(m3synth.scan_inputs(shape, seed=9), True)
    args = (d["x"], d["dt"], d["A"], d["lam"], d["B"], d["C"], d["theta"])
    kw = dict(R=1, chunk=64, B_bias=d["B_bias"], C_bias=d["C_bias"])
    y0, s0 = m3.m3_scan_fwd(*args, **kw)
    y1, s1 = m3.m3_scan_fwd(*args, bc_norm=True, **kw)
    torch.cuda.synchronize()
    a, b = y0.float(), y1.float()
    rms = float(a.pow(2).mean().sqrt())
    # both outputs are bf16-stored: allow each its half-ulp rounding beyond the bound
    excess = (b - a).abs() - 2.0 ** -8 * (a.abs() + b.abs())
    assert float(excess.max()) <= 2e-2 * rms
