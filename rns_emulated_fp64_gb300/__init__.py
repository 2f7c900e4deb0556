"""Ozaki Scheme II emulated FP64 GEMM on GB300 (sm_103a).

The compute lives in libos2 (CUDA kernels behind the C ABI of include/os2.h);
this package is its Python binding.  See ``binding.gemm``.
"""
from .binding import (GEMM_S8_SYNC, GEMM_SIMT, GEMM_TC, GEMM_TC_1SM, GEMM_TC_I8, MODE_ACCURATE, MODE_FAST, OUT_MODP_INT8,  # noqa: F401
                      OUT_RAW_INT32, Os2Error, alloc_workspace, crt, gemm, gemm_host,
                      gemm_residues, get_status, host_workspace_size, launch_count, load,
                      matmul, moduli, profile_start, profile_stop, residues, scale, sgemm,
                      set_gemm_variant, status_string, workspace_size, zgemm,
                      complex_workspace_size, wait_selftest, ERR_TIMEOUT, peak_probe,
                      PROBE_F16_1SM, PROBE_F16_2SM, PROBE_S8_SYNC, set_crt_variant,
                      CRT_TC, CRT_SIMT, CRT_AUTO, scale_bounds, exponents_from_bounds,
                      gemm_exponents)
