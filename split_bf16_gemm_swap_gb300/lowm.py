"""ctypes binding of the C ABI in ``include/lowm_gemm.h``.

Argument marshalling only: every function here forwards to the function of
the same name in ``liblowm_gemm.so``, where all of the GEMM runs in CUDA
kernels.  Pointer arguments accept a torch tensor (its ``data_ptr()``) or a
plain integer address; ``stream`` accepts a ``torch.cuda.Stream``, a raw
``cudaStream_t`` integer, or None (torch's current stream on the current
device).  There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblowm_gemm.so")

LOWM_OK = 0
LOWM_ERR_INVALID_ARGUMENT = 1
LOWM_ERR_UNSUPPORTED_SHAPE = 2
LOWM_ERR_MISALIGNED = 3
LOWM_ERR_UNSUPPORTED_ARCH = 4
LOWM_ERR_CUDA = 5
LOWM_ERR_TIMEOUT = 6

LOWM_FLAG_W_BEFORE_PDL_WAIT = 1
LOWM_FLAG_A_BEFORE_PDL_WAIT = 2

# Exported C functions, in header order.
ABI_FUNCTIONS = (
    "lowm_gemm_bf16",
    "lowm_gemm_bf16_ex",
    "lowm_gemm_query_tactic",
    "lowm_gemm_query_tactic_ex",
    "lowm_status_string",
    "lowm_gemm_sync_status",
    "lowm_gemm_bf16_host",
    "lowm_gemm_bf16_debug",
    "lowm_tmem_hog_launch",
)


class lowm_tactic_t(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in
                ("tile_n", "m_pad", "split_k", "stages", "block_k", "tiles", "num_clusters", "ctas", "smem_bytes",
                 "pdl", "persistent", "tiles_per_cluster", "kb_per_stage", "mma_issuers", "w_prefetch_stages",
                 "mbox_in_ring", "l2_prefetch_stages", "l2_before_wait_stages")]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class lowm_debug_opts_t(ctypes.Structure):
    _fields_ = [
        ("stall_warp_mask", ctypes.c_uint),
        ("stall_rank_mask", ctypes.c_uint),
        ("stall_ns", ctypes.c_uint),
        ("full_smem", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("drop_mailbox", ctypes.c_int),
        ("reduce_timeout_ns", ctypes.c_ulonglong),
        ("probes", ctypes.c_void_p),
        ("c_f32", ctypes.c_void_p),
        ("timeline", ctypes.c_void_p),
        ("flags", ctypes.c_uint),
    ]


class LowmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__("%s: %s (status %d)" % (where, status_string(status), status))


_lib = None


def lib():
    """Load ``liblowm_gemm.so`` once; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("liblowm_gemm.so is not built (run split_bf16_gemm_swap_gb300.build.build() "
                               "or __graft_entry__.build()); there is no fallback path")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
        L.lowm_gemm_bf16.argtypes = [vp, vp, vp, i, i, i, i, vp]
        L.lowm_gemm_bf16.restype = st
        L.lowm_gemm_bf16_ex.argtypes = [vp, vp, vp, i, i, i, i, ctypes.c_uint, vp]
        L.lowm_gemm_bf16_ex.restype = st
        L.lowm_gemm_query_tactic.argtypes = [i, i, i, i, ctypes.POINTER(lowm_tactic_t)]
        L.lowm_gemm_query_tactic.restype = st
        L.lowm_gemm_query_tactic_ex.argtypes = [i, i, i, i, ctypes.c_uint, ctypes.POINTER(lowm_tactic_t)]
        L.lowm_gemm_query_tactic_ex.restype = st
        L.lowm_status_string.argtypes = [st]
        L.lowm_status_string.restype = ctypes.c_char_p
        L.lowm_gemm_sync_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
        L.lowm_gemm_sync_status.restype = st
        L.lowm_gemm_bf16_host.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, vp]
        L.lowm_gemm_bf16_host.restype = st
        L.lowm_gemm_bf16_debug.argtypes = [vp, vp, vp, i, i, i, i, vp, ctypes.POINTER(lowm_debug_opts_t)]
        L.lowm_gemm_bf16_debug.restype = st
        L.lowm_tmem_hog_launch.argtypes = [vp, i, i, i]
        L.lowm_tmem_hog_launch.restype = st
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr() or None
    return int(x) or None


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream or None
    return int(s) or None


def status_string(status: int) -> str:
    return lib().lowm_status_string(int(status)).decode()


def lowm_status_string(status: int) -> str:
    return status_string(status)


def lowm_gemm_bf16(A, W, C, M: int, N: int, K: int, split_k: int = 0, stream=None) -> int:
    return lib().lowm_gemm_bf16(_ptr(A), _ptr(W), _ptr(C), int(M), int(N), int(K), int(split_k), _stream(stream))


def lowm_gemm_bf16_ex(A, W, C, M: int, N: int, K: int, split_k: int = 0, flags: int = 0, stream=None) -> int:
    return lib().lowm_gemm_bf16_ex(_ptr(A), _ptr(W), _ptr(C), int(M), int(N), int(K), int(split_k), int(flags),
                                   _stream(stream))


def lowm_gemm_query_tactic(M: int, N: int, K: int, split_k: int = 0):
    """Return ``(status, tactic dict or None)``."""
    t = lowm_tactic_t()
    s = lib().lowm_gemm_query_tactic(int(M), int(N), int(K), int(split_k), ctypes.byref(t))
    return s, (t.as_dict() if s == LOWM_OK else None)


def lowm_gemm_query_tactic_ex(M: int, N: int, K: int, split_k: int = 0, flags: int = 0):
    """Return ``(status, tactic dict or None)`` for a launch with these flags."""
    t = lowm_tactic_t()
    s = lib().lowm_gemm_query_tactic_ex(int(M), int(N), int(K), int(split_k), int(flags), ctypes.byref(t))
    return s, (t.as_dict() if s == LOWM_OK else None)


def lowm_gemm_sync_status(stream=None):
    """Return ``(status, detail bits)``."""
    d = ctypes.c_uint(0)
    s = lib().lowm_gemm_sync_status(_stream(stream), ctypes.byref(d))
    return s, d.value


def lowm_gemm_bf16_host(A_host, W_host, C_host, A_dev, W_dev, C_dev, M, N, K, split_k=0, stream=None) -> int:
    return lib().lowm_gemm_bf16_host(_ptr(A_host), _ptr(W_host), _ptr(C_host), _ptr(A_dev), _ptr(W_dev),
                                     _ptr(C_dev), int(M), int(N), int(K), int(split_k), _stream(stream))


def lowm_gemm_bf16_debug(A, W, C, M, N, K, split_k=0, stream=None, *, stall_warp_mask=0, stall_rank_mask=0,
                         stall_ns=0, full_smem=0, stages=0, drop_mailbox=0, reduce_timeout_ns=0, probes=None,
                         c_f32=None, timeline=None, flags=0) -> int:
    o = lowm_debug_opts_t(int(stall_warp_mask), int(stall_rank_mask), int(stall_ns), int(full_smem), int(stages),
                          int(drop_mailbox), int(reduce_timeout_ns), _ptr(probes), _ptr(c_f32), _ptr(timeline),
                          int(flags))
    return lib().lowm_gemm_bf16_debug(_ptr(A), _ptr(W), _ptr(C), int(M), int(N), int(K), int(split_k),
                                      _stream(stream), ctypes.byref(o))


def lowm_tmem_hog_launch(stream=None, ctas: int = 1024, ncols: int = 256, iters: int = 1) -> int:
    return lib().lowm_tmem_hog_launch(_stream(stream), int(ctas), int(ncols), int(iters))


def gemm(A, W, C=None, split_k: int = 0, stream=None, flags: int = 0):
    """C = A . W^T for CUDA bf16 tensors A [M,K], W [N,K]; allocates C if not given.

    flags: LOWM_FLAG_* for lowm_gemm_bf16_ex (LOWM_FLAG_W_BEFORE_PDL_WAIT when
    the kernel that precedes this launch on the stream does not write W).
    """
    import torch
    if A.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise TypeError("A and W must be bfloat16")
    if A.dim() != 2 or W.dim() != 2 or A.shape[1] != W.shape[1]:
        raise ValueError("A must be [M,K] and W [N,K]")
    if not (A.is_cuda and W.is_cuda and A.is_contiguous() and W.is_contiguous()):
        raise ValueError("A and W must be contiguous CUDA tensors")
    M, K = A.shape
    N = W.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    s = lowm_gemm_bf16_ex(A, W, C, M, N, K, split_k, flags, stream)
    if s != LOWM_OK:
        raise LowmError(s, "lowm_gemm_bf16_ex")
    return C
