"""CPU oracle for the FP8 (E4M3) GEMM with fine-grained scaling.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product library never
imports this package and this package never imports the product library.

The arithmetic lives in ``fp8_oracle.c`` (plain C, fp64, one loop per output
element).  This module only compiles it (gcc, no fast-math, no FMA
contraction, so x86 and Arm give the same bits) and marshals numpy arrays.
Row-parallel drivers split rows over threads; every element is still computed
by the same single-threaded loop, so results do not depend on the split.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off",
          "-fno-fast-math", "-fexcess-precision=standard"]


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle (gcc) into ``out`` (default ``oracle/liboracle.so``)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    u8p = ctypes.POINTER(ctypes.c_uint8)
    f32p = ctypes.POINTER(ctypes.c_float)
    f64p = ctypes.POINTER(ctypes.c_double)
    i32p = ctypes.POINTER(ctypes.c_int)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    I = ctypes.c_int
    lib.oracle_e4m3_to_f64.restype = ctypes.c_double
    lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_f64_to_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_f64_to_bf16_rne.argtypes = [ctypes.c_double]
    lib.oracle_bf16_to_f64.restype = ctypes.c_double
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_element_f64.restype = ctypes.c_double
    lib.oracle_element_f64.argtypes = [u8p, u8p, f32p, ctypes.c_long, f32p, I]
    lib.oracle_gemm_nt.restype = None
    lib.oracle_gemm_nt.argtypes = [u8p, f32p, u8p, f32p, I, I, I, u16p, f64p]
    lib.oracle_gemm_nt_rows.restype = None
    lib.oracle_gemm_nt_rows.argtypes = [u8p, f32p, u8p, f32p, I, I, I,
                                        i32p, I, u16p, f64p]
    lib.oracle_gemm_nt_acc_rows.restype = None
    lib.oracle_gemm_nt_acc_rows.argtypes = [u8p, f32p, u8p, f32p, f32p, I, I, I,
                                            i32p, I, u16p, f64p]
    lib.oracle_ue8m0_to_f64.restype = ctypes.c_double
    lib.oracle_ue8m0_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_gemm_nt_ue8m0_rows.restype = None
    lib.oracle_gemm_nt_ue8m0_rows.argtypes = [u8p, u8p, u8p, u8p, I, I, I, i32p, I, u16p, f64p]
    lib.oracle_gemm_grouped_contiguous_rows.restype = None
    lib.oracle_gemm_grouped_contiguous_rows.argtypes = [
        u8p, f32p, u8p, f32p, i32p, I, I, I, I, i32p, I, u16p]
    lib.oracle_gemm_grouped_masked_rows.restype = None
    lib.oracle_gemm_grouped_masked_rows.argtypes = [
        u8p, f32p, u8p, f32p, i32p, I, I, I, I, I, i32p, I, u16p]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def load_variant(path: str):
    """Load another build of the oracle's source (the tests use this to show
    that the pins reject copies with a planted mistake)."""
    return _bind(ctypes.CDLL(path))


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u8(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        a = a.view(np.uint8)
    return a


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


# --------------------------------------------------------------------------
# scalar codecs

def e4m3_to_f64(code: int, lib=None) -> float:
    return (lib or _load()).oracle_e4m3_to_f64(int(code) & 0xFF)


def f64_to_bf16(x: float, lib=None) -> int:
    return int((lib or _load()).oracle_f64_to_bf16_rne(float(x)))


def bf16_to_f64(h: int, lib=None) -> float:
    return (lib or _load()).oracle_bf16_to_f64(int(h) & 0xFFFF)


def element(A, SFA, B, SFB, M, N, K, m, n, lib=None) -> float:
    """Unrounded fp64 value of D[m][n] for the plain layout."""
    lib = lib or _load()
    A, B, SFA, SFB = _u8(A), _u8(B), _f32(SFA), _f32(SFB)
    ld = (M + 3) // 4 * 4
    kb = K // 128
    a_row = A.reshape(-1)[m * K:(m + 1) * K]
    b_row = B.reshape(-1)[n * K:(n + 1) * K]
    sfa = SFA.reshape(-1)[m:]
    sfb = SFB.reshape(-1)[(n // 128) * kb:]
    return lib.oracle_element_f64(_ptr(a_row, ctypes.c_uint8), _ptr(b_row, ctypes.c_uint8),
                                  _ptr(sfa, ctypes.c_float), ld,
                                  _ptr(sfb, ctypes.c_float), K)


# --------------------------------------------------------------------------
# GEMM drivers

def _split(rows: np.ndarray, threads: int):
    threads = max(1, min(threads, len(rows)))
    return [c for c in np.array_split(rows, threads) if len(c)]


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def gemm_nt(A, SFA, B, SFB, M, N, K, want_acc=False, lib=None):
    """Full product (single thread).  Returns D bits (uint16 [M][N]) and,
    if asked, the unrounded fp64 values."""
    lib = lib or _load()
    A, B, SFA, SFB = _u8(A), _u8(B), _f32(SFA), _f32(SFB)
    D = np.empty((M, N), np.uint16)
    acc = np.empty((M, N), np.float64) if want_acc else None
    lib.oracle_gemm_nt(_ptr(A, ctypes.c_uint8), _ptr(SFA, ctypes.c_float),
                       _ptr(B, ctypes.c_uint8), _ptr(SFB, ctypes.c_float),
                       M, N, K, _ptr(D, ctypes.c_uint16),
                       _ptr(acc, ctypes.c_double) if want_acc else None)
    return (D, acc) if want_acc else D


def gemm_nt_rows(A, SFA, B, SFB, M, N, K, rows, threads=1, want_acc=False, lib=None):
    """Rows ``rows`` of the plain product, split over ``threads`` threads."""
    lib = lib or _load()
    A, B, SFA, SFB = _u8(A), _u8(B), _f32(SFA), _f32(SFB)
    rows = _i32(rows)
    D = np.empty((len(rows), N), np.uint16)
    acc = np.empty((len(rows), N), np.float64) if want_acc else None

    def run(chunk_start, chunk):
        lib.oracle_gemm_nt_rows(
            _ptr(A, ctypes.c_uint8), _ptr(SFA, ctypes.c_float),
            _ptr(B, ctypes.c_uint8), _ptr(SFB, ctypes.c_float), M, N, K,
            _ptr(chunk, ctypes.c_int), len(chunk),
            _ptr(D[chunk_start:], ctypes.c_uint16),
            _ptr(acc[chunk_start:], ctypes.c_double) if want_acc else None)

    _run_chunks(rows, threads, run)
    return (D, acc) if want_acc else D


def gemm_nt_acc_rows(A, SFA, B, SFB, C, M, N, K, rows, threads=1, want_acc=False, lib=None):
    """Rows ``rows`` of the plain product plus the fp32 addend ``C`` [M][N]."""
    lib = lib or _load()
    A, B, SFA, SFB, C = _u8(A), _u8(B), _f32(SFA), _f32(SFB), _f32(C)
    assert C.size == M * N, "C must be [M][N]"
    rows = _i32(rows)
    D = np.empty((len(rows), N), np.uint16)
    acc = np.empty((len(rows), N), np.float64) if want_acc else None

    def run(chunk_start, chunk):
        lib.oracle_gemm_nt_acc_rows(
            _ptr(A, ctypes.c_uint8), _ptr(SFA, ctypes.c_float),
            _ptr(B, ctypes.c_uint8), _ptr(SFB, ctypes.c_float),
            _ptr(C, ctypes.c_float), M, N, K,
            _ptr(chunk, ctypes.c_int), len(chunk),
            _ptr(D[chunk_start:], ctypes.c_uint16),
            _ptr(acc[chunk_start:], ctypes.c_double) if want_acc else None)

    _run_chunks(rows, threads, run)
    return (D, acc) if want_acc else D


def ue8m0_to_f64(e: int, lib=None) -> float:
    return (lib or _load()).oracle_ue8m0_to_f64(int(e) & 0xFF)


def gemm_nt_ue8m0_rows(A, SFA_e, B, SFB_e, M, N, K, rows, threads=1, want_acc=False, lib=None):
    """Rows ``rows`` of the plain product with UE8M0 exponent-byte scales
    (SFA_e uint8 [K/128][round_up(M,4)], SFB_e uint8 [ceil(N/128)][K/128])."""
    lib = lib or _load()
    A, B, SFA_e, SFB_e = _u8(A), _u8(B), _u8(SFA_e), _u8(SFB_e)
    rows = _i32(rows)
    D = np.empty((len(rows), N), np.uint16)
    acc = np.empty((len(rows), N), np.float64) if want_acc else None

    def run(chunk_start, chunk):
        lib.oracle_gemm_nt_ue8m0_rows(
            _ptr(A, ctypes.c_uint8), _ptr(SFA_e, ctypes.c_uint8),
            _ptr(B, ctypes.c_uint8), _ptr(SFB_e, ctypes.c_uint8), M, N, K,
            _ptr(chunk, ctypes.c_int), len(chunk),
            _ptr(D[chunk_start:], ctypes.c_uint16),
            _ptr(acc[chunk_start:], ctypes.c_double) if want_acc else None)

    _run_chunks(rows, threads, run)
    return (D, acc) if want_acc else D


def _run_chunks(rows, threads, fn):
    chunks = _split(rows, threads)
    starts = np.cumsum([0] + [len(c) for c in chunks[:-1]])
    if len(chunks) <= 1:
        for s, c in zip(starts, chunks):
            fn(int(s), np.ascontiguousarray(c))
        return
    with ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        futs = [ex.submit(fn, int(s), np.ascontiguousarray(c))
                for s, c in zip(starts, chunks)]
        for f in futs:
            f.result()


def gemm_grouped_contiguous_rows(A, SFA, B, SFB, m_indices, M_total, N, K, G,
                                 rows, threads=1, D_init=None, lib=None):
    """Rows ``rows`` of the contiguous grouped product.  Rows whose group is
    out of range keep ``D_init``'s value (zeros when not given)."""
    lib = lib or _load()
    A, B, SFA, SFB = _u8(A), _u8(B), _f32(SFA), _f32(SFB)
    layout = _i32(m_indices)
    rows = _i32(rows)
    if D_init is None:
        D = np.zeros((len(rows), N), np.uint16)
    else:
        D = np.ascontiguousarray(D_init, dtype=np.uint16).copy()

    def run(s, chunk):
        lib.oracle_gemm_grouped_contiguous_rows(
            _ptr(A, ctypes.c_uint8), _ptr(SFA, ctypes.c_float),
            _ptr(B, ctypes.c_uint8), _ptr(SFB, ctypes.c_float),
            _ptr(layout, ctypes.c_int), M_total, N, K, G,
            _ptr(chunk, ctypes.c_int), len(chunk), _ptr(D[s:], ctypes.c_uint16))

    _run_chunks(rows, threads, run)
    return D


def gemm_grouped_masked_rows(A, SFA, B, SFB, masked_m, G, M_max, N, K, g, rows,
                             threads=1, D_init=None, lib=None):
    """Rows ``rows`` of group ``g`` of the masked grouped product.  Rows at or
    beyond the group's count keep ``D_init``'s value (zeros when not given)."""
    lib = lib or _load()
    A, B, SFA, SFB = _u8(A), _u8(B), _f32(SFA), _f32(SFB)
    counts = _i32(masked_m)
    rows = _i32(rows)
    if D_init is None:
        D = np.zeros((len(rows), N), np.uint16)
    else:
        D = np.ascontiguousarray(D_init, dtype=np.uint16).copy()

    def run(s, chunk):
        lib.oracle_gemm_grouped_masked_rows(
            _ptr(A, ctypes.c_uint8), _ptr(SFA, ctypes.c_float),
            _ptr(B, ctypes.c_uint8), _ptr(SFB, ctypes.c_float),
            _ptr(counts, ctypes.c_int), G, M_max, N, K, g,
            _ptr(chunk, ctypes.c_int), len(chunk), _ptr(D[s:], ctypes.c_uint16))

    _run_chunks(rows, threads, run)
    return D
