"""Exact, IO-aware, tiled attention (FlashAttention) for GB300 (sm_103a).

The computation lives in ``libfa_gb300.so`` (C ABI: include/fa.h): a
tcgen05/TMA/TMEM forward and backward kernel for bf16/fp16, an E4M3 (FP8)
forward with its quantiser, CUDA-core kernels for float32, and small
HBM-bound helper kernels.  This package is a thin
ctypes binding plus the seeded synthetic workload generators.
"""
from ._lib import (FAError, bwd, check_status, dropout_mask, fwd, load, make_params,  # noqa: F401
                   status_string, EXPORTED, DTYPE_CODE)
from ._lib import bwd_noalloc, noalloc_check_status, noalloc_scratch, selftest_wait_timeout  # noqa: F401
from ._lib import fp8_layout, fp8_quantize, fp8_views, fwd_fp8  # noqa: F401
from ._build import build, LIB  # noqa: F401
