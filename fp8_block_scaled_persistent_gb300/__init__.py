"""Python binding of the GB300 FP8 block-scaled GEMM library.

Argument marshalling only: each function takes torch tensors that already live
on the GPU, passes their device pointers and the current CUDA stream to the C
ABI of ``libfp8gemm.so`` (declared in ``include/fp8gemm.h``) and returns its
status code.  Every step of the computation runs in the library's CUDA
kernels; there is no fallback.  Importing works without a GPU; calling a GEMM
needs the built library (``__graft_entry__.build()`` or
``python fp8_block_scaled_persistent_gb300/build.py``) and a CUDA device.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8gemm.so")
# the bounds-checking build (every kernel compiled with FP8G_DEBUG_BOUNDS=1);
# FP8G_LIBRARY=debug in the environment makes library() load it instead
DEBUG_LIB_PATH = os.path.join(_HERE, "libfp8gemm_debug.so")

FP8G_OK = 0
FP8G_ERR_INVALID_ARG = 1
FP8G_ERR_UNSUPPORTED = 2
FP8G_ERR_MISALIGNED = 3
FP8G_ERR_CUDA = 4
FP8G_ERR_TIMEOUT = 5
FP8G_ERR_BAD_GROUP = 6
FP8G_ERR_WORKSPACE = 7
FP8G_ERR_SCRATCH_LIMIT = 8
FP8G_ERR_BOUNDS = 9

FP8G_KIND_NT = 0
FP8G_KIND_GROUPED_CONTIGUOUS = 1
FP8G_KIND_GROUPED_MASKED = 2

# every symbol the header declares, in declaration order
EXPORTS = (
    "fp8_gemm_nt", "fp8_gemm_nt_accumulate", "fp8_gemm_nt_ue8m0", "fp8_gemm_grouped_contiguous",
    "fp8_gemm_grouped_masked",
    "fp8_gemm_workspace_size", "fp8_gemm_get_device_error", "fp8_gemm_status_string",
    "fp8_gemm_sfa_ld", "fp8_gemm_set_override", "fp8_gemm_set_pair_mode", "fp8_gemm_set_narrow_mode",
    "fp8_gemm_workspace_size_for",
    "fp8_gemm_set_wait_timeout_ns", "fp8_gemm_nt_noalloc", "fp8_gemm_version",
)

_lock = threading.Lock()
_lib = None


class Fp8GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


def library(path: str | None = None):
    """The loaded C library (raises if it has not been built).  The
    bounds-checking build is loaded instead when FP8G_LIBRARY=debug."""
    global _lib
    if path is None:
        path = DEBUG_LIB_PATH if os.environ.get("FP8G_LIBRARY") == "debug" else LIB_PATH
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"libfp8gemm.so is not built ({path}); run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        vp, sz, i, u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint64
        lib.fp8_gemm_nt.argtypes = [vp, vp, vp, vp, vp, i, i, i, vp, sz, vp]
        lib.fp8_gemm_nt_accumulate.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, vp, sz, vp]
        lib.fp8_gemm_nt_accumulate.restype = i
        lib.fp8_gemm_nt_ue8m0.argtypes = [vp, vp, vp, vp, vp, i, i, i, vp]
        lib.fp8_gemm_nt_ue8m0.restype = i
        lib.fp8_gemm_grouped_contiguous.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, vp, sz, vp]
        lib.fp8_gemm_grouped_masked.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, vp, sz, vp]
        for f in ("fp8_gemm_nt", "fp8_gemm_grouped_contiguous", "fp8_gemm_grouped_masked"):
            getattr(lib, f).restype = i
        lib.fp8_gemm_workspace_size.argtypes = [i, i, i, i, i]
        lib.fp8_gemm_workspace_size.restype = sz
        lib.fp8_gemm_workspace_size_for.argtypes = [i, i, i, i, i]
        lib.fp8_gemm_workspace_size_for.restype = sz
        lib.fp8_gemm_get_device_error.argtypes = [vp]
        lib.fp8_gemm_get_device_error.restype = i
        lib.fp8_gemm_status_string.argtypes = [i]
        lib.fp8_gemm_status_string.restype = ctypes.c_char_p
        lib.fp8_gemm_sfa_ld.argtypes = [i]
        lib.fp8_gemm_sfa_ld.restype = i
        lib.fp8_gemm_set_override.argtypes = [i, i]
        lib.fp8_gemm_set_override.restype = i
        lib.fp8_gemm_set_pair_mode.argtypes = [i]
        lib.fp8_gemm_set_pair_mode.restype = i
        lib.fp8_gemm_set_narrow_mode.argtypes = [i]
        lib.fp8_gemm_set_narrow_mode.restype = i
        lib.fp8_gemm_set_wait_timeout_ns.argtypes = [u64]
        lib.fp8_gemm_set_wait_timeout_ns.restype = i
        lib.fp8_gemm_nt_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, vp]
        lib.fp8_gemm_nt_noalloc.restype = i
        lib.fp8_gemm_version.argtypes = []
        lib.fp8_gemm_version.restype = i
        _lib = lib
        return lib


# ------------------------------------------------------------------ marshalling

def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ws(workspace):
    if workspace is None:
        return None, 0
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def fp8_gemm_nt(A, SFA, B, SFB, D, M, N, K, workspace=None, stream=None) -> int:
    """D[M][N] (bf16) = A[M][K] (e4m3) x B[N][K]^T with SFA [K/128][sfa_ld(M)]
    and SFB [ceil(N/128)][K/128] fp32 scales.  Returns the status code."""
    wp, wb = _ws(workspace)
    return library().fp8_gemm_nt(_ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(D),
                                 int(M), int(N), int(K), wp, wb, _stream(stream))


def fp8_gemm_nt_accumulate(A, SFA, B, SFB, C, D, M, N, K, workspace=None, stream=None) -> int:
    """D[M][N] (bf16) = C[M][N] (fp32) + the plain product of fp8_gemm_nt.
    C must not overlap D.  Returns the status code."""
    wp, wb = _ws(workspace)
    return library().fp8_gemm_nt_accumulate(_ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(C), _ptr(D),
                                             int(M), int(N), int(K), wp, wb, _stream(stream))


def fp8_gemm_nt_ue8m0(A, SFA_e, B, SFB_e, D, M, N, K, stream=None) -> int:
    """D[M][N] (bf16) = A x B^T with power-of-two scales given as UE8M0 bytes:
    SFA_e uint8 [K/128][sfa_ld(M)], SFB_e uint8 [ceil(N/128)][K/128].
    Returns the status code."""
    return library().fp8_gemm_nt_ue8m0(_ptr(A), _ptr(SFA_e), _ptr(B), _ptr(SFB_e), _ptr(D),
                                       int(M), int(N), int(K), _stream(stream))


def fp8_gemm_grouped_contiguous(A, SFA, B, SFB, D, m_indices, M_total, N, K, G,
                                workspace=None, stream=None) -> int:
    wp, wb = _ws(workspace)
    return library().fp8_gemm_grouped_contiguous(
        _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(D), _ptr(m_indices),
        int(M_total), int(N), int(K), int(G), wp, wb, _stream(stream))


def fp8_gemm_grouped_masked(A, SFA, B, SFB, D, masked_m, G, M_max, N, K,
                            workspace=None, stream=None) -> int:
    wp, wb = _ws(workspace)
    return library().fp8_gemm_grouped_masked(
        _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(D), _ptr(masked_m),
        int(G), int(M_max), int(N), int(K), wp, wb, _stream(stream))


def fp8_gemm_workspace_size(kind, M, N, K, G=1) -> int:
    return int(library().fp8_gemm_workspace_size(int(kind), int(M), int(N), int(K), int(G)))


def fp8_gemm_workspace_size_for(M, N, K, block_n, split_ctas) -> int:
    return int(library().fp8_gemm_workspace_size_for(int(M), int(N), int(K), int(block_n),
                                                     int(split_ctas)))


def fp8_gemm_get_device_error(stream=None) -> int:
    return library().fp8_gemm_get_device_error(_stream(stream))


def fp8_gemm_status_string(status: int) -> str:
    return library().fp8_gemm_status_string(int(status)).decode()


status_string = fp8_gemm_status_string


def fp8_gemm_sfa_ld(M) -> int:
    return library().fp8_gemm_sfa_ld(int(M))


def fp8_gemm_set_override(block_n=0, split_ctas=0) -> int:
    return library().fp8_gemm_set_override(int(block_n), int(split_ctas))


def fp8_gemm_set_pair_mode(mode=0) -> int:
    """1: unsplit calls run on CTA pairs (256 x 128 tiles over two SMs; the
    power-of-two-scale GEMM on 256 x 256 tiles), 2: A-sharing clusters,
    0: automatic choice (pairs only for the power-of-two-scale GEMM with
    M > 128), -1: never.  Returns the status code."""
    return library().fp8_gemm_set_pair_mode(int(mode))


def fp8_gemm_set_narrow_mode(mode=0) -> int:
    """1: every plain GEMM with M <= 128 runs on the narrow-slice kernel (one
    CTA per 96-column slice and K half, the two CTAs of a slice a cluster
    trading halves over distributed shared memory), 0: automatic choice,
    -1: never.
    Returns the status code."""
    return library().fp8_gemm_set_narrow_mode(int(mode))


def fp8_gemm_set_wait_timeout_ns(ns) -> int:
    return library().fp8_gemm_set_wait_timeout_ns(int(ns))


def fp8_gemm_nt_noalloc(A, SFA, B, SFB, D, M, N, K, stream=None) -> int:
    """fp8_gemm_nt without a workspace, for callers that cannot call
    cudaMalloc (code inside an allocator callback, plug-ins whose host
    framework owns all device memory, loops that forbid allocation after
    start-up).  The split-K scratch is a 24 MiB static device array inside the
    library, so nothing is allocated per call.  Calls that overlap on the GPU
    race on that one array; make the first call on a device before any
    stream capture (it looks up the array's address)."""
    return library().fp8_gemm_nt_noalloc(_ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(D),
                                         int(M), int(N), int(K), _stream(stream))


def fp8_gemm_version() -> int:
    return library().fp8_gemm_version()


def check(status: int, what: str = "fp8 gemm") -> None:
    """Raise Fp8GemmError unless status is FP8G_OK."""
    if status != FP8G_OK:
        raise Fp8GemmError(status, what)
