"""Mamba-3 selective-SSM scan for B300 (sm_103a): prefill and decode.

The compute lives in libm3scan.so (CUDA kernels behind the C ABI declared in
include/m3scan.h); ``m3scan`` is its thin ctypes binding.
"""
from .m3scan import (  # noqa: F401
    M3_BF16, M3_ERR_CUDA, M3_ERR_INVALID_ARG, M3_ERR_TIMEOUT, M3_ERR_UNSUPPORTED, M3_F32, M3_OK,
    M3Error, m3_decode_step, m3_decode_tokens, m3_device_status, m3_scan_fwd, m3_scan_fwd_noalloc,
    m3_scan_fwd_state, m3_scan_bwd,
    m3_scan_workspace_bytes, m3_scan_bwd_workspace_bytes, m3_status_string, m3_version, make_dims, load)
