"""m3_scan_fwd_noalloc: the prefill for callers that cannot let the library
allocate device memory (their own allocator owns the GPU's memory, or a device
allocation's latency or failure is not acceptable where they call from).

The entry point is called through the C ABI on a problem that needs scratch
(a segmented scan: few sequences, many chunks), twice in a row on different
inputs -- the second call runs over the first one's leftovers in the shared
scratch array -- and each result is checked against m3_scan_fwd's (which
allocates its scratch) within the tolerance the parity tests use. A problem
that needs more scratch than the fixed array is refused without a launch.
This file is collected last, after every other test.
"""
import ctypes

import numpy as np
import pytest

import m3synth
from gpu_util import assert_bf16, assert_bf16_out, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import selective_state_space_129_b300 as m3  # noqa: E402


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_the_allocating_entry_point_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = m3.load()
    L, Q, R, H, N, P = 2048, 64, 1, 2, 128, 64
    shape = m3synth.ScanShape(1, L, H, 1, P, N, R=R, chunk=Q, bf16=True, rms_bc=True)
    dims = m3.make_dims(1, L, H, 1, P, N, m3.M3_BF16)
    assert m3.m3_scan_workspace_bytes(dims, R, Q) > 0, "this shape must need scratch"
    stream = torch.cuda.current_stream()
    for seed in (41, 42):
        d = to_device(m3synth.scan_inputs(shape, seed=seed), True)
        y_ref, fs_ref = m3.m3_scan_fwd(d["x"], d["dt"], d["A"], d["lam"], d["B"], d["C"],
                                       d["theta"], R=R, chunk=Q, B_bias=d["B_bias"],
                                       C_bias=d["C_bias"], stream=stream)
        y = torch.full_like(d["x"], float("nan"))
        fs = torch.full_like(fs_ref, float("nan"))
        dd = m3.make_dims(1, L, H, 1, P, N, m3.M3_BF16, d["B_bias"], d["C_bias"])
        st = lib.m3_scan_fwd_noalloc(_ptr(d["x"]), _ptr(d["dt"]), _ptr(d["A"]), _ptr(d["lam"]),
                                     _ptr(d["B"]), _ptr(d["C"]), _ptr(d["theta"]),
                                     ctypes.byref(dd), R, Q, _ptr(y), _ptr(fs),
                                     ctypes.c_void_p(stream.cuda_stream))
        assert st == m3.M3_OK, m3.m3_status_string(st)
        torch.cuda.synchronize()
        assert_bf16_out(y.float().cpu().numpy(), y_ref.float().cpu().numpy().astype(np.float64),
                        "y (seed %d)" % seed)
        assert_bf16(fs.cpu().numpy(), fs_ref.cpu().numpy().astype(np.float64),
                    "final_state (seed %d)" % seed)
    assert m3.m3_device_status() == m3.M3_OK


def test_noalloc_refuses_scratch_beyond_its_array():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = m3.load()
    # b1 L65536 H32 N128 R1: a segmented scan that needs more than 32 MiB of
    # scratch; the call is refused before any pointer is used
    dims = m3.make_dims(1, 65536, 32, 1, 64, 128, m3.M3_BF16)
    assert m3.m3_scan_workspace_bytes(dims, 1, 64) > (32 << 20)
    fake = ctypes.c_void_p(0x10000)
    st = lib.m3_scan_fwd_noalloc(fake, fake, fake, fake, fake, fake, fake, ctypes.byref(dims), 1, 64,
                                 fake, fake, None)
    assert st == m3.M3_ERR_UNSUPPORTED
