"""Seeded synthetic inputs for the FP8 block-scaled GEMM.

This module is shared by the tests (for both the CUDA path and the CPU
oracle), the benchmark and the smoke check.  It only draws random numbers and
prepares quantised inputs; it contains none of the GEMM's arithmetic.

Recipe (every workload, seed 0 unless a test says otherwise):

* Random numbers come from a counter-based generator: SplitMix64 (Steele,
  Lea & Flood, "Fast splittable pseudorandom number generators", 2014), whose
  i-th output from state ``s`` is ``mix64(s + (i+1) * 0x9E3779B97F4A7C15)``.
  Each tensor has its own stream (state ``key(seed, stream)``), so any slice
  of any tensor can be drawn on its own and in parallel.
* N(0,1) values: Box-Muller, cosine branch, from two consecutive 64-bit draws
  (53-bit uniforms, the first shifted by half an ulp away from 0), computed in
  fp64 and rounded to fp32.
* Quantisation: A (rows x K) gets one fp32 scale per row per 128-wide K block,
  B (N x K) one per 128 x 128 block; ``scale = amax / 448`` in fp32 (448 is
  the largest E4M3FN value), ``q = e4m3(x / scale)`` with the division in fp32
  and round-to-nearest-even encoding, saturating at +-448.  A block whose amax
  is 0 gets scale 1 (its codes are all zero whatever the scale).
* Group sizes (contiguous): uniform integers in [1024, 6144], rounded up to a
  multiple of 128; counts (masked): uniform integers in [0, M_max].
* The fp32 addend C of the accumulate variant: sqrt(K) * N(0,1), the spread
  of the product itself (a sum of K products of two N(0,1) values).
* Power-of-two (UE8M0) scales: the same blocks, with scale = 2^j for the
  smallest integer j such that amax / 2^j <= 448 (amax / 448 formed in fp64),
  stored as the byte e = 127 + j (clamped to 0..254); a zero block gets e = 127.
  q = e4m3(x / 2^j), where the division is exact.

Layouts (all C-contiguous):
  A    uint8 [rows][K]          masked: [G][M_max][K]
  SFA  fp32  [K/128][ld]        masked: [G][K/128][ld], ld = round_up(rows, 4)
  B    uint8 [G][N][K]          (G = 1 for the plain GEMM)
  SFB  fp32  [G][ceil(N/128)][K/128]
  D    bf16  [rows][N]          masked: [G][M_max][N]
  C    fp32  [rows][N]          (accumulate variant only)
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
E4M3_MAX = 448.0

STREAM_A = 1
STREAM_B = 2
STREAM_GROUPS = 3
STREAM_C = 4

_CHUNK = 1 << 22


def _threads() -> int:
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return 4


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([(seed * 0x9E3779B97F4A7C15 + stream * 0xD1B54A32D192ED03)
                      & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _mix64(s)[0]


def raw_u64(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of the SplitMix64 stream with state key."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix64(key + i * GOLDEN)


def _normal_chunk(key, start, count) -> np.ndarray:
    z = raw_u64(key, 2 * start, 2 * count)
    z1 = z[0::2] >> np.uint64(11)
    z2 = z[1::2] >> np.uint64(11)
    u1 = (z1.astype(np.float64) + 0.5) * (2.0 ** -53)
    u2 = z2.astype(np.float64) * (2.0 ** -53)
    return (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)).astype(np.float32)


def normal_f32(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    """``count`` N(0,1) fp32 values, elements start .. start+count-1 of the stream."""
    key = stream_key(seed, stream)
    out = np.empty(count, np.float32)
    spans = [(s, min(_CHUNK, count - s)) for s in range(0, count, _CHUNK)]

    def fill(span):
        s, c = span
        out[s:s + c] = _normal_chunk(key, start + s, c)

    if len(spans) > 1:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, spans))
    else:
        for sp in spans:
            fill(sp)
    return out


def uniform_ints(seed: int, stream: int, count: int, lo: int, hi: int) -> np.ndarray:
    """``count`` integers uniform in [lo, hi] (modulo reduction of 64-bit draws)."""
    z = raw_u64(stream_key(seed, stream), 0, count)
    return (lo + (z % np.uint64(hi - lo + 1)).astype(np.int64)).astype(np.int64)


# --------------------------------------------------------------------------
# E4M3FN encoding of fp32 values (input preparation)

def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest E4M3FN code (ties to even), saturating
    at +-448.  Returns uint8 codes."""
    y = np.asarray(y, dtype=np.float32)
    flat = y.reshape(-1)
    out = np.empty(flat.shape, np.uint8)
    spans = [(s, min(_CHUNK, flat.size - s)) for s in range(0, flat.size, _CHUNK)]

    def enc(span):
        s, c = span
        out[s:s + c] = _e4m3_encode_chunk(flat[s:s + c])

    if len(spans) > 1:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(enc, spans))
    else:
        for sp in spans:
            enc(sp)
    return out.reshape(y.shape)


def _e4m3_encode_chunk(y: np.ndarray) -> np.ndarray:
    sign = np.signbit(y)
    a = np.minimum(np.abs(y.astype(np.float64)), E4M3_MAX)
    _, E = np.frexp(a)                       # a = f * 2^E, f in [0.5, 1)
    lead = E - 1
    qexp = np.where(lead >= -6, lead - 3, -9)  # weight of the last mantissa bit
    n = np.rint(np.ldexp(a, -qexp))           # rint: ties to even
    v = np.ldexp(n, qexp)
    _, Ev = np.frexp(v)
    leadv = Ev - 1
    normal = v >= 2.0 ** -6
    e_field = np.where(normal, leadv + 7, 0)
    mant = np.where(normal, np.ldexp(v, -leadv) * 8.0 - 8.0, np.ldexp(v, 9))
    code = (e_field.astype(np.int64) << 3) | mant.astype(np.int64)
    code = np.where(v == 0, 0, code)
    return (code | (sign.astype(np.int64) << 7)).astype(np.uint8)


# --------------------------------------------------------------------------
# block quantisation

def quantize_rows_1x128(x: np.ndarray):
    """x: fp32 [rows][K] -> (codes uint8 [rows][K], scales fp32 [rows][K/128])."""
    rows, K = x.shape
    kb = K // 128
    xb = x.reshape(rows, kb, 128)
    amax = np.abs(xb).max(axis=2)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = (xb / scale[:, :, None]).astype(np.float32)
    return e4m3_encode(y).reshape(rows, K), scale


def quantize_blocks_128x128(x: np.ndarray):
    """x: fp32 [N][K] -> (codes uint8 [N][K], scales fp32 [ceil(N/128)][K/128])."""
    N, K = x.shape
    kb = K // 128
    nb = (N + 127) // 128
    pad = nb * 128 - N
    xp = np.concatenate([x, np.zeros((pad, K), np.float32)]) if pad else x
    amax = np.abs(xp.reshape(nb, 128, kb, 128)).max(axis=(1, 3))
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    full = np.repeat(np.repeat(scale, 128, axis=0), 128, axis=1)[:N]
    y = (x / full).astype(np.float32)
    return e4m3_encode(y), scale


def ue8m0_exponents(amax: np.ndarray) -> np.ndarray:
    """UE8M0 bytes e = 127 + j, j the smallest integer with amax / 2^j <= 448
    (amax / 448 in fp64); 127 where amax is 0."""
    r = np.asarray(amax, np.float64) / E4M3_MAX
    f, E = np.frexp(np.where(r > 0, r, 1.0))      # r = f * 2^E, f in [0.5, 1)
    j = np.where(f == 0.5, E - 1, E)              # 2^j >= r, and 2^(j-1) < r
    e = np.where(r > 0, 127 + j, 127)
    return np.clip(e, 0, 254).astype(np.uint8)


def quantize_rows_1x128_ue8m0(x: np.ndarray):
    """x: fp32 [rows][K] -> (codes uint8 [rows][K], UE8M0 bytes [rows][K/128])."""
    rows, K = x.shape
    xb = x.reshape(rows, K // 128, 128)
    e = ue8m0_exponents(np.abs(xb).max(axis=2))
    scale = np.ldexp(np.float32(1.0), e.astype(np.int32) - 127).astype(np.float32)
    y = (xb / scale[:, :, None]).astype(np.float32)
    return e4m3_encode(y).reshape(rows, K), e


def quantize_blocks_128x128_ue8m0(x: np.ndarray):
    """x: fp32 [N][K] -> (codes uint8 [N][K], UE8M0 bytes [ceil(N/128)][K/128])."""
    N, K = x.shape
    kb, nb = K // 128, (N + 127) // 128
    pad = nb * 128 - N
    xp = np.concatenate([x, np.zeros((pad, K), np.float32)]) if pad else x
    e = ue8m0_exponents(np.abs(xp.reshape(nb, 128, kb, 128)).max(axis=(1, 3)))
    scale = np.ldexp(np.float32(1.0), e.astype(np.int32) - 127).astype(np.float32)
    full = np.repeat(np.repeat(scale, 128, axis=0), 128, axis=1)[:N]
    return e4m3_encode((x / full).astype(np.float32)), e


def sfa_ld(rows: int) -> int:
    return (rows + 3) // 4 * 4


def sfa_m_major(scale_rows: np.ndarray, rows: int) -> np.ndarray:
    """[rows][kb] per-row scales -> M-major [kb][round_up(rows, 4)] (pad 0)."""
    kb = scale_rows.shape[1]
    out = np.zeros((kb, sfa_ld(rows)), np.float32)
    out[:, :rows] = scale_rows.T
    return out


# --------------------------------------------------------------------------
# problems

@dataclass
class Problem:
    kind: str                       # "nt" | "nt_acc" | "contiguous" | "masked"
    M: int                          # nt: M; contiguous: M_total; masked: M_max
    N: int
    K: int
    G: int
    A: np.ndarray
    SFA: np.ndarray
    B: np.ndarray
    SFB: np.ndarray
    m_indices: np.ndarray | None = None   # contiguous, int32 [M_total]
    masked_m: np.ndarray | None = None    # masked, int32 [G]
    C: np.ndarray | None = None           # nt_acc: fp32 addend [M][N]
    # nt_ue8m0: SFA and SFB hold UE8M0 exponent bytes (uint8) instead of fp32
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def kb(self) -> int:
        return self.K // 128

    @property
    def nb(self) -> int:
        return (self.N + 127) // 128

    def d_shape(self):
        if self.kind == "masked":
            return (self.G, self.M, self.N)
        return (self.M, self.N)

    def valid_rows(self) -> int:
        if self.kind == "masked":
            return int(np.minimum(np.maximum(self.masked_m, 0), self.M).sum())
        if self.kind == "contiguous":
            return int(((self.m_indices >= 0) & (self.m_indices < self.G)).sum())
        return self.M

    def flops(self) -> int:
        return 2 * self.valid_rows() * self.N * self.K

    @property
    def scale_bytes(self) -> int:
        return 1 if self.kind == "nt_ue8m0" else 4

    def algorithmic_bytes(self) -> int:
        """A + SFA + B + SFB + D (+ the group layout, + C), valid rows only;
        a group's B counts once if the group has any valid row."""
        kb, nb, N, K, sb = self.kb, self.nb, self.N, self.K, self.scale_bytes
        rows = self.valid_rows()
        per_row = K + sb * kb + 2 * N
        if self.kind == "masked":
            live = int((self.masked_m > 0).sum())
            return rows * per_row + live * (N * K + 4 * nb * kb) + 4 * self.G
        if self.kind == "contiguous":
            live = len(set(int(g) for g in np.unique(self.m_indices) if 0 <= g < self.G))
            return rows * per_row + live * (N * K + 4 * nb * kb) + 4 * self.M
        c_bytes = 4 * rows * N if self.C is not None else 0
        return rows * per_row + N * K + sb * nb * kb + c_bytes


def _quant_A(x: np.ndarray):
    q, s = quantize_rows_1x128(x)
    return q, s


def make_nt(M: int, N: int, K: int, seed: int = 0, name: str = "") -> Problem:
    a = normal_f32(seed, STREAM_A, M * K).reshape(M, K)
    b = normal_f32(seed, STREAM_B, N * K).reshape(N, K)
    qa, sa = _quant_A(a)
    qb, sb = quantize_blocks_128x128(b)
    return Problem("nt", M, N, K, 1, qa, sfa_m_major(sa, M), qb.reshape(1, N, K),
                   sb.reshape(1, *sb.shape), name=name or f"nt_{M}x{N}x{K}")


def make_nt_acc(M: int, N: int, K: int, seed: int = 0, name: str = "") -> Problem:
    """The plain problem of make_nt plus an fp32 addend C [M][N]."""
    p = make_nt(M, N, K, seed, name or f"acc_{M}x{N}x{K}")
    p.kind = "nt_acc"
    p.C = (normal_f32(seed, STREAM_C, M * N) * np.float32(math.sqrt(K))).reshape(M, N)
    return p


def make_nt_ue8m0(M: int, N: int, K: int, seed: int = 0, name: str = "") -> Problem:
    """The plain problem's A and B values with power-of-two scales: SFA and
    SFB hold UE8M0 bytes, SFA M-major [K/128][round_up(M,4)] (pad 127)."""
    a = normal_f32(seed, STREAM_A, M * K).reshape(M, K)
    b = normal_f32(seed, STREAM_B, N * K).reshape(N, K)
    qa, ea = quantize_rows_1x128_ue8m0(a)
    qb, eb = quantize_blocks_128x128_ue8m0(b)
    sfa = np.full((K // 128, sfa_ld(M)), 127, np.uint8)
    sfa[:, :M] = ea.T
    return Problem("nt_ue8m0", M, N, K, 1, qa, sfa, qb.reshape(1, N, K), eb.reshape(1, *eb.shape),
                   name=name or f"ue8m0_{M}x{N}x{K}")


def make_contiguous(group_rows, N: int, K: int, seed: int = 0, name: str = "") -> Problem:
    """``group_rows``: rows per group, each a multiple of 128."""
    group_rows = [int(r) for r in group_rows]
    assert all(r % 128 == 0 for r in group_rows)
    G = len(group_rows)
    M = sum(group_rows)
    a = normal_f32(seed, STREAM_A, M * K).reshape(M, K)
    qa, sa = _quant_A(a)
    qbs, sbs = [], []
    for g in range(G):
        b = normal_f32(seed, STREAM_B, N * K, start=g * N * K).reshape(N, K)
        qb, sb = quantize_blocks_128x128(b)
        qbs.append(qb)
        sbs.append(sb)
    layout = np.repeat(np.arange(G, dtype=np.int32), group_rows).astype(np.int32)
    return Problem("contiguous", M, N, K, G, qa, sfa_m_major(sa, M), np.stack(qbs),
                   np.stack(sbs), m_indices=layout, name=name or f"contiguous_g{G}_{N}x{K}",
                   meta={"group_rows": group_rows})


def make_masked(counts, M_max: int, N: int, K: int, seed: int = 0, name: str = "") -> Problem:
    counts = np.asarray(counts, dtype=np.int32)
    G = len(counts)
    a = normal_f32(seed, STREAM_A, G * M_max * K).reshape(G * M_max, K)
    qa, sa = _quant_A(a)
    sfa = np.stack([sfa_m_major(sa[g * M_max:(g + 1) * M_max], M_max) for g in range(G)])
    qbs, sbs = [], []
    for g in range(G):
        b = normal_f32(seed, STREAM_B, N * K, start=g * N * K).reshape(N, K)
        qb, sb = quantize_blocks_128x128(b)
        qbs.append(qb)
        sbs.append(sb)
    return Problem("masked", M_max, N, K, G, qa.reshape(G, M_max, K), sfa, np.stack(qbs),
                   np.stack(sbs), masked_m=counts, name=name or f"masked_g{G}_{M_max}x{N}x{K}")


def contiguous_group_rows(G: int, lo: int = 1024, hi: int = 6144, seed: int = 0):
    r = uniform_ints(seed, STREAM_GROUPS, G, lo, hi)
    return [int((v + 127) // 128 * 128) for v in r]


def masked_counts(G: int, M_max: int, seed: int = 0):
    return uniform_ints(seed, STREAM_GROUPS, G, 0, M_max).astype(np.int32)


# --------------------------------------------------------------------------
# the five workload families of the method's evaluation

WORKLOADS = {
    "single_128x256x512": lambda seed=0: make_nt(128, 256, 512, seed, "single_128x256x512"),
    "dense_4096x7168x2048": lambda seed=0: make_nt(4096, 7168, 2048, seed, "dense_4096x7168x2048"),
    "dense_4096x24576x1536": lambda seed=0: make_nt(4096, 24576, 1536, seed, "dense_4096x24576x1536"),
    "smallm_64x7168x16384": lambda seed=0: make_nt(64, 7168, 16384, seed, "smallm_64x7168x16384"),
    "smallm_128x7168x16384": lambda seed=0: make_nt(128, 7168, 16384, seed, "smallm_128x7168x16384"),
    "contiguous_g8_n4096_k7168": lambda seed=0: make_contiguous(
        contiguous_group_rows(8, seed=seed), 4096, 7168, seed, "contiguous_g8_n4096_k7168"),
    "masked_g16_m256_n7168_k2048": lambda seed=0: make_masked(
        masked_counts(16, 256, seed=seed), 256, 7168, 2048, seed, "masked_g16_m256_n7168_k2048"),
    # the accumulate variant (D = bf16(C + A B^T)) on the first dense shape
    "acc_4096x7168x2048": lambda seed=0: make_nt_acc(4096, 7168, 2048, seed, "acc_4096x7168x2048"),
    # power-of-two (UE8M0) scales on the dense shapes
    "ue8m0_4096x7168x2048": lambda seed=0: make_nt_ue8m0(4096, 7168, 2048, seed, "ue8m0_4096x7168x2048"),
    "ue8m0_4096x24576x1536": lambda seed=0: make_nt_ue8m0(4096, 24576, 1536, seed, "ue8m0_4096x24576x1536"),
}


def make(name: str, seed: int = 0) -> Problem:
    return WORKLOADS[name](seed)


def exact_integer_problem(M: int, N: int, K: int, seed: int = 0, vmax: int = 4,
                          kind: str = "nt", G: int = 1) -> Problem:
    """Small-integer E4M3 values in [-vmax, vmax] (all exact in E4M3) with
    power-of-two scales in [2^-2, 2^2].  Every 128-term partial is an integer
    of magnitude <= 128 * vmax^2, every scaled term a multiple of 2^-4, so
    for K/128 < 32 (vmax = 4) every fp32 partial and running sum is exact and
    the only rounding anywhere is the final one to bf16."""
    kb, nb = K // 128, (N + 127) // 128
    za = raw_u64(stream_key(seed, 11), 0, M * K)
    zb = raw_u64(stream_key(seed, 12), 0, G * N * K)
    va = (za % np.uint64(2 * vmax + 1)).astype(np.int64) - vmax
    vb = (zb % np.uint64(2 * vmax + 1)).astype(np.int64) - vmax
    qa = e4m3_encode(va.astype(np.float32)).reshape(M, K)
    qb = e4m3_encode(vb.astype(np.float32)).reshape(G, N, K)
    ea = (raw_u64(stream_key(seed, 13), 0, M * kb) % np.uint64(5)).astype(np.int64) - 2
    eb = (raw_u64(stream_key(seed, 14), 0, G * nb * kb) % np.uint64(5)).astype(np.int64) - 2
    sa = np.ldexp(np.float32(1.0), ea).astype(np.float32).reshape(M, kb)
    sb = np.ldexp(np.float32(1.0), eb).astype(np.float32).reshape(G, nb, kb)
    return Problem(kind, M, N, K, G, qa, sfa_m_major(sa, M), qb, sb,
                   name=f"exact_{M}x{N}x{K}",
                   meta={"va": va.reshape(M, K), "vb": vb.reshape(G, N, K),
                         "sa_rows": sa, "sb": sb})
