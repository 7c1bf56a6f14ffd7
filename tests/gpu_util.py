"""Shared helpers for the GPU parity tests: seeded inputs to device tensors,
oracle calls on the same values, and the error measures the tests assert on.

Tolerances (stated once, used by every parity test):
  fp32 mode   relative L2 error  <= 1e-5
  bf16 mode   max |error|        <= 2e-2 * RMS(oracle output)
Both follow from the scan's precision contract: fp32 inputs with fp32
arithmetic, or bf16 inputs with fp32 state and accumulation.

An output stored in bf16 also carries its own storage rounding, up to half a
bf16 ulp (2^-8 |y|) per element, which no kernel can avoid; for bf16-stored
outputs the tolerance above is applied to what is left after that bound:
  max_i ( |got_i - ref_i| - 2^-8 |ref_i| ) <= 2e-2 * RMS(ref).
fp32 outputs (the final state) get the plain bound.
"""
import numpy as np

F32_REL_L2 = 1e-5
BF16_MAX_OVER_RMS = 2e-2


def to_device(inp, bf16, device="cuda"):
    import torch
    act = torch.bfloat16 if bf16 else torch.float32
    out = {}
    for k, v in inp.items():
        if k == "bits":
            continue
        t = torch.from_numpy(np.ascontiguousarray(v))
        if k in ("x", "B", "C"):
            t = t.to(act)
        out[k] = t.to(device)
    return out


def head_slice(inp, b, h):
    """Inputs of one (batch row, head) as a 1-batch, 1-head, 1-group problem."""
    H = inp["x"].shape[2]
    G = inp["B"].shape[2]
    g = h // (H // G)
    return dict(
        x=inp["x"][b:b + 1, :, h:h + 1], dt=inp["dt"][b:b + 1, :, h:h + 1],
        A=inp["A"][h:h + 1], lam=inp["lam"][b:b + 1, :, h:h + 1],
        B=inp["B"][b:b + 1, :, g:g + 1], C=inp["C"][b:b + 1, :, g:g + 1],
        theta=inp["theta"][b:b + 1, :, g:g + 1],
        B_bias=inp["B_bias"][h:h + 1], C_bias=inp["C_bias"][h:h + 1])


def rel_l2(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))


def max_over_rms(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return float(np.max(np.abs(got - ref)) / max(rms, 1e-300))


def assert_f32(got, ref, what=""):
    e = rel_l2(got, ref)
    assert e <= F32_REL_L2, "%s: relative L2 error %.3e > %.1e" % (what, e, F32_REL_L2)


BF16_HALF_ULP = 2.0 ** -8


def max_over_rms_bf16_stored(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    excess = np.abs(got - ref) - BF16_HALF_ULP * np.abs(ref)
    return float(np.max(excess) / max(rms, 1e-300))


def assert_bf16(got, ref, what=""):
    """fp32-stored result of a bf16-input computation."""
    e = max_over_rms(got, ref)
    assert e <= BF16_MAX_OVER_RMS, "%s: max|err|/RMS %.3e > %.1e" % (what, e, BF16_MAX_OVER_RMS)


def assert_bf16_out(got, ref, what=""):
    """bf16-stored output: the tolerance applies beyond the storage rounding."""
    e = max_over_rms_bf16_stored(got, ref)
    assert e <= BF16_MAX_OVER_RMS, "%s: max(|err| - 2^-8|y|)/RMS %.3e > %.1e" % (
        what, e, BF16_MAX_OVER_RMS)
