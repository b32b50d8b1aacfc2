"""GB300-native low-M split-K bf16 GEMM: C[M,N] = A[M,K] . W[N,K]^T.

The compute lives in ``liblowm_gemm.so`` (CUDA C++ for sm_103a, built by
``split_bf16_gemm_swap_gb300.build``); :mod:`.lowm` is its ctypes binding and
:mod:`.inputs` draws the seeded synthetic operands.  Importing the package
does not load the library; the first call does, and fails loudly if it is
missing.
"""
from .lowm import (  # noqa: F401
    ABI_FUNCTIONS, LOWM_FLAG_A_BEFORE_PDL_WAIT, LOWM_FLAG_W_BEFORE_PDL_WAIT, LOWM_OK, LowmError, gemm,
    lowm_gemm_bf16, lowm_gemm_bf16_debug, lowm_gemm_bf16_ex, lowm_gemm_bf16_host,
    lowm_gemm_query_tactic, lowm_gemm_query_tactic_ex, lowm_gemm_sync_status, lowm_status_string, lowm_tmem_hog_launch,
)
