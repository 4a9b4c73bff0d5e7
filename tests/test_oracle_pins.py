"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test ties the oracle to something it does not compute itself: the
format's named special values, a library cast (torch's float8_e4m3fn and
bfloat16 conversions), a second formulation (dequantise then matmul), closed
forms for small integers, hand-worked elements, the scale-doubling invariant
and grouped-to-dense reductions.  ``test_oracle_mutants.py`` shows that these
pins reject copies of the oracle with plausible planted mistakes.
"""
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers

def torch_decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """Library decode: reinterpret bytes as torch.float8_e4m3fn, widen to f64."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_bf16_bits(values_f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(values_f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)


def dequant_matmul(p: wl.Problem, g: int = 0):
    """Second formulation: dequantise every element with its own scale, then a
    plain fp64 matmul (numpy).  Returns fp64 [M][N]."""
    M, N, K = p.M, p.N, p.K
    kb = K // 128
    a = torch_decode_e4m3(p.A.reshape(-1, K)[:M])
    b = torch_decode_e4m3(p.B[g])
    sfa = p.SFA.reshape(kb, -1)[:, :M].T.astype(np.float64)          # [M][kb]
    sfb = p.SFB[g].astype(np.float64)                                # [nb][kb]
    a_s = a * np.repeat(sfa, 128, axis=1)
    b_s = b * np.repeat(np.repeat(sfb, 128, axis=0), 128, axis=1)[:N]
    return a_s @ b_s.T


def oracle_lib_or(lib):
    return lib


# ---------------------------------------------------------------- E4M3 decode

def test_e4m3_decode_exhaustive_matches_library(lib=None):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch_decode_e4m3(codes)
    for c in range(256):
        v = oracle.e4m3_to_f64(c, lib=lib)
        if np.isnan(ref[c]):
            assert np.isnan(v), f"code {c:#x}: expected NaN, got {v}"
        else:
            assert v == ref[c] and np.signbit(v) == np.signbit(ref[c]), (c, v, ref[c])


def test_e4m3_special_values_golden(lib=None):
    path = os.path.join(GOLDEN, "e4m3fn_special_values.txt")
    n = 0
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        code_hex, value = line.split()
        v = oracle.e4m3_to_f64(int(code_hex, 16), lib=lib)
        if value == "nan":
            assert np.isnan(v), code_hex
        else:
            want = float(value)
            assert v == want and np.signbit(v) == np.signbit(want), (code_hex, v, want)
        n += 1
    assert n >= 15


def test_e4m3_nan_codes_are_exactly_two(lib=None):
    nans = [c for c in range(256) if np.isnan(oracle.e4m3_to_f64(c, lib=lib))]
    assert nans == [0x7F, 0xFF]


# ---------------------------------------------------------------- bf16 rounding

def _random_finite_f32(n, seed):
    z = wl.raw_u64(wl.stream_key(seed, 99), 0, n)
    bits = (z & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    f = bits.view(np.float32)
    return f[np.isfinite(f)]


def test_bf16_rne_matches_library_on_f32_values(lib=None):
    # values exact in fp32 have a single rounding either way, so the library's
    # fp32 -> bf16 cast (round-to-nearest-even) is a valid reference.
    vals = _random_finite_f32(200_000, 1)
    # add every bf16 tie pattern around a few exponents, plus subnormals
    extra = []
    for e in (-133, -127, -126, -10, 0, 1, 7, 100, 127):
        for mant in range(0, 128, 7):
            base = (1 + mant / 128) * 2.0 ** e
            for off in (-2 ** -9, 2 ** -9, 2 ** -8 - 2 ** -16):
                extra.append(base * (1 + off))
    extra += [2.0 ** -149, 3 * 2.0 ** -149, 2.0 ** -133, 1.5 * 2.0 ** -133, 3.3895e38]
    vals = np.concatenate([vals, np.array(extra, np.float32)])
    vals = vals[np.isfinite(vals)]
    ref = torch_bf16_bits(vals)
    got = np.array([oracle.f64_to_bf16(float(v), lib=lib) for v in vals], np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert len(bad) == 0, [(float(vals[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_bf16_rne_fp64_only_cases(lib=None):
    """Cases where rounding through fp32 first would give a different answer:
    the oracle must round fp64 directly."""
    f = lambda x: oracle.f64_to_bf16(x, lib=lib)
    assert f(1.0 + 2 ** -8) == 0x3F80                   # exact tie -> even (down)
    assert f(1.0 + 3 * 2 ** -8) == 0x3F82               # exact tie -> even (up)
    assert f(1.0 + 2 ** -8 + 2 ** -40) == 0x3F81        # just above a tie: up
    assert f(1.0 + 2 ** -8 - 2 ** -40) == 0x3F80        # just below a tie: down
    assert f(-(1.0 + 2 ** -8 + 2 ** -40)) == 0xBF81
    assert f(2.0 ** 128) == 0x7F80                      # overflow -> +Inf
    assert f(-(2.0 ** 128)) == 0xFF80
    assert f((2 - 2 ** -8) * 2.0 ** 127) == 0x7F80       # ties past max -> Inf
    assert f((2 - 2 ** -7) * 2.0 ** 127) == 0x7F7F       # largest finite
    assert f(2.0 ** -134) == 0x0000                      # half the min subnormal: tie -> 0
    assert f(2.0 ** -134 + 2.0 ** -160) == 0x0001
    assert f(-0.0) == 0x8000
    assert f(float("nan")) == 0x7FC0


def test_e4m3_quantise_dequantise_round_trips(lib=None):
    """The input generator's encoder against the oracle's decoder:
    encode(decode(q)) == q for every non-NaN code, and for values inside the
    finite range decode(encode(x)) is within half an E4M3 ulp of x, ties
    going to the code with an even mantissa."""
    codes = [q for q in range(256) if q not in (0x7F, 0xFF)]
    dec = np.array([oracle.e4m3_to_f64(q, lib=lib) for q in codes])
    assert np.array_equal(wl.e4m3_encode(dec.astype(np.float32)), np.array(codes, np.uint8))
    x = np.concatenate([wl.normal_f32(0, 60, 20_000) * 60, wl.normal_f32(0, 61, 20_000) * 0.02,
                        # exact midpoints between neighbouring codes (ties)
                        ((dec[1:120] + dec[2:121]) / 2).astype(np.float32)]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    q = wl.e4m3_encode(x)
    back = np.array([oracle.e4m3_to_f64(int(c), lib=lib) for c in q])
    a = np.abs(x.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    ulp = 2.0 ** (e - 3)                 # 3 mantissa bits; subnormals share 2^-9
    err = np.abs(back - x)
    assert (err <= ulp / 2).all()
    tie = err == ulp / 2
    assert tie.any() and ((q[tie] & 1) == 0).all()


def test_bf16_decode_roundtrip(lib=None):
    for h in range(0, 0x10000, 37):
        v = oracle.bf16_to_f64(h, lib=lib)
        if np.isnan(v):
            continue
        assert oracle.f64_to_bf16(v, lib=lib) == h


# ---------------------------------------------------------------- hand-worked

def _parse_hand_cases():
    cases = []
    for line in open(os.path.join(GOLDEN, "hand_worked_elements.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = [x.strip() for x in line.split("|")]
        name, K, N, n = f[0], int(f[1]), int(f[2]), int(f[3])
        a_codes = [int(x, 16) for x in f[4].split(",") if x]
        b_codes = [int(x, 16) for x in f[5].split(",") if x]
        sfa = [float(x) for x in f[6].split(",") if x]
        sfb = [[float(x) for x in blk.split(",") if x] for blk in f[7].split("/")]
        cases.append((name, K, N, n, a_codes, b_codes, sfa, sfb, int(f[8], 16)))
    return cases


@pytest.mark.parametrize("case", _parse_hand_cases(), ids=lambda c: c[0])
def test_hand_worked_elements(case, lib=None):
    name, K, N, n, a_codes, b_codes, sfa, sfb, want = case
    kb, nb = K // 128, (N + 127) // 128
    M = 1
    A = np.repeat(np.array(a_codes, np.uint8), 128).reshape(1, K)
    B = np.zeros((N, K), np.uint8)
    B[n] = np.repeat(np.array(b_codes, np.uint8), 128)
    SFA = np.zeros((kb, 4), np.float32)
    SFA[:, 0] = sfa
    SFB = np.ones((nb, kb), np.float32)
    for j, blk in enumerate(sfb):
        SFB[j] = blk
    D = oracle.gemm_nt(A, SFA, B, SFB, M, N, K, lib=lib)
    assert D[0, n] == want, f"{name}: got {D[0, n]:#06x}, want {want:#06x}"


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("M,N,K", [(5, 200, 256), (3, 130, 384), (8, 64, 128)])
def test_brute_force_against_dequant_matmul(M, N, K, lib=None):
    p = wl.make_nt(M, N, K, seed=7)
    D, acc = oracle.gemm_nt(p.A, p.SFA, p.B, p.SFB, M, N, K, want_acc=True, lib=lib)
    ref = dequant_matmul(p)
    np.testing.assert_allclose(acc, ref, rtol=1e-12, atol=1e-300)
    # D equals the rounding of the reference except where the reference sits
    # within a few fp64 ulps of a bf16 rounding boundary.
    ref_bits = np.array([oracle.f64_to_bf16(v, lib=lib) for v in ref.reshape(-1)],
                        np.uint16).reshape(M, N)
    mism = np.nonzero(D != ref_bits)
    for i, j in zip(*mism):
        lo = oracle.bf16_to_f64(int(min(D[i, j], ref_bits[i, j])), lib=lib)
        hi = oracle.bf16_to_f64(int(max(D[i, j], ref_bits[i, j])), lib=lib)
        mid = (lo + hi) / 2
        assert abs(ref[i, j] - mid) <= 1e-12 * abs(mid), (i, j)


# ---------------------------------------------------------------- exact integers

def _exact_value(p, m, n):
    """Exact value of D[m][n] as a Fraction from integer arithmetic."""
    kb = p.K // 128
    va, vb = p.meta["va"], p.meta["vb"][0]
    sa, sb = p.meta["sa_rows"], p.meta["sb"][0]
    total = Fraction(0)
    for k in range(kb):
        s = int(np.dot(va[m, 128 * k:128 * (k + 1)], vb[n, 128 * k:128 * (k + 1)]))
        total += Fraction(float(sa[m, k])) * Fraction(float(sb[n // 128, k])) * s
    return total


@pytest.mark.parametrize("M,N,K", [(6, 256, 512), (4, 384, 1024)])
def test_exact_integer_closed_form(M, N, K, lib=None):
    p = wl.exact_integer_problem(M, N, K, seed=3)
    # the generator's codes decode to the intended integers (library decode)
    assert np.array_equal(torch_decode_e4m3(p.A), p.meta["va"].astype(np.float64))
    D, acc = oracle.gemm_nt(p.A, p.SFA, p.B, p.SFB, M, N, K, want_acc=True, lib=lib)
    exact = np.array([[float(_exact_value(p, m, n)) for n in range(N)] for m in range(M)])
    assert np.array_equal(acc, exact)
    # each exact value is exact in fp32 (multiple of 2^-4, magnitude < 2^20),
    # so the library's fp32 -> bf16 cast rounds it exactly once
    assert np.array_equal(exact.astype(np.float32).astype(np.float64), exact)
    assert np.array_equal(D, torch_bf16_bits(exact.astype(np.float32)))


# ---------------------------------------------------------------- the fp32 addend

def test_acc_zero_addend_equals_plain(lib=None):
    p = wl.make_nt(5, 200, 256, seed=21)
    D0, acc0 = oracle.gemm_nt(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, want_acc=True, lib=lib)
    C = np.zeros((p.M, p.N), np.float32)
    D1, acc1 = oracle.gemm_nt_acc_rows(p.A, p.SFA, p.B, p.SFB, C, p.M, p.N, p.K,
                                       np.arange(p.M), want_acc=True, lib=lib)
    assert np.array_equal(D0, D1) and np.array_equal(acc0, acc1)


def test_acc_zero_product_rounds_the_addend_like_library(lib=None):
    """Every A code zero: D is C rounded to bf16, which the library's fp32 ->
    bf16 cast (round to nearest even) decides.  M != N, so a transposed or
    wrongly strided C is caught; zeros are left out (0 + -0 is +0)."""
    M, N, K = 6, 272, 256
    p = wl.make_nt(M, N, K, seed=22)
    vals = _random_finite_f32(4 * M * N, 23)
    vals = vals[vals != 0][:M * N]
    assert vals.size == M * N
    C = vals.reshape(M, N)
    D = oracle.gemm_nt_acc_rows(np.zeros_like(p.A), p.SFA, p.B, p.SFB, C, M, N, K,
                                np.arange(M), lib=lib)
    assert np.array_equal(D, torch_bf16_bits(C))
    # only the listed rows, in the listed order
    sel = np.array([4, 0], np.int32)
    Ds = oracle.gemm_nt_acc_rows(np.zeros_like(p.A), p.SFA, p.B, p.SFB, C, M, N, K, sel, lib=lib)
    assert np.array_equal(Ds, D[sel])


@pytest.mark.parametrize("M,N,K", [(6, 256, 512), (5, 384, 1024)])
def test_acc_exact_integer_closed_form(M, N, K, lib=None):
    """Small integers with power-of-two scales plus an integer addend: every
    result is exact in fp32, so D must be the library's cast of the closed
    form, and the unrounded value the closed form itself."""
    p = wl.exact_integer_problem(M, N, K, seed=5)
    z = wl.raw_u64(wl.stream_key(5, 15), 0, M * N)
    # integers in [-64, 64] plus sixteenths: up to 11 significant bits, more
    # than bf16 holds, so the addend must enter the sum unrounded
    C = (((z % np.uint64(129)).astype(np.int64) - 64) +
         ((z >> np.uint64(32)) % np.uint64(16)).astype(np.int64) / 16.0).astype(np.float32).reshape(M, N)
    D, acc = oracle.gemm_nt_acc_rows(p.A, p.SFA, p.B, p.SFB, C, M, N, K, np.arange(M),
                                     want_acc=True, lib=lib)
    exact = np.array([[float(Fraction(float(C[m, n])) + _exact_value(p, m, n)) for n in range(N)]
                      for m in range(M)])
    assert np.array_equal(acc, exact)
    assert np.array_equal(exact.astype(np.float32).astype(np.float64), exact)
    assert np.array_equal(D, torch_bf16_bits(exact.astype(np.float32)))


# ---------------------------------------------------------------- UE8M0 scales

def test_ue8m0_decode_exhaustive(lib=None):
    """Every UE8M0 byte against the MX format's closed form 2^(e - 127)
    (Python's ldexp, not the oracle's); 0xFF is NaN."""
    import math
    for e in range(255):
        assert oracle.ue8m0_to_f64(e, lib=lib) == math.ldexp(1.0, e - 127), e
    assert math.isnan(oracle.ue8m0_to_f64(255, lib=lib))


def test_ue8m0_reduces_to_fp32_scales(lib=None):
    """With the exponent bytes decoded to fp32 outside the oracle (numpy
    ldexp), the fp32-scale oracle must give the same values and bits: the
    UE8M0 form reads the same layouts with the same indices."""
    p = wl.make_nt_ue8m0(70, 300, 384, seed=16)
    dec = lambda e: np.ldexp(np.float32(1.0), e.astype(np.int32) - 127).astype(np.float32)  # noqa: E731
    rows = np.arange(p.M, dtype=np.int32)
    D, acc = oracle.gemm_nt_ue8m0_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows,
                                       want_acc=True, lib=lib)
    D32, acc32 = oracle.gemm_nt(p.A, dec(p.SFA), p.B, dec(p.SFB), p.M, p.N, p.K, want_acc=True, lib=lib)
    assert np.array_equal(acc, acc32) and np.array_equal(D, D32)


@pytest.mark.parametrize("M,N,K", [(6, 256, 512), (5, 384, 1024)])
def test_ue8m0_exact_integer_closed_form(M, N, K, lib=None):
    """Small integers with UE8M0 exponents 124..130: the exact value from
    integer arithmetic, rounded once by the library's fp32 -> bf16 cast."""
    p = wl.exact_integer_problem(M, N, K, seed=6)
    kb, nb = K // 128, (N + 127) // 128
    ea = (wl.raw_u64(wl.stream_key(6, 17), 0, M * kb) % np.uint64(7)).astype(np.int64) + 124
    eb = (wl.raw_u64(wl.stream_key(6, 18), 0, nb * kb) % np.uint64(7)).astype(np.int64) + 124
    SFA = np.full((kb, (M + 3) // 4 * 4), 127, np.uint8)
    SFA[:, :M] = ea.reshape(M, kb).T
    SFB = eb.reshape(nb, kb).astype(np.uint8)
    D, acc = oracle.gemm_nt_ue8m0_rows(p.A, SFA, p.B[0], SFB, M, N, K, np.arange(M, dtype=np.int32),
                                       want_acc=True, lib=lib)
    va, vb = p.meta["va"], p.meta["vb"][0]
    exact = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            for k in range(kb):
                s = int(np.dot(va[m, 128 * k:128 * (k + 1)], vb[n, 128 * k:128 * (k + 1)]))
                tot += Fraction(2) ** (int(ea[m * kb + k]) - 127 + int(eb[(n // 128) * kb + k]) - 127) * s
            exact[m, n] = float(tot)
    assert np.array_equal(acc, exact)
    assert np.array_equal(exact.astype(np.float32).astype(np.float64), exact)
    assert np.array_equal(D, torch_bf16_bits(exact.astype(np.float32)))


# ---------------------------------------------------------------- invariants

def _block_partial(p, m, n, k, g=0):
    a = torch_decode_e4m3(p.A.reshape(-1, p.K)[m, 128 * k:128 * (k + 1)])
    b = torch_decode_e4m3(p.B[g][n, 128 * k:128 * (k + 1)])
    return float(np.dot(a, b))      # exact: <= 128 terms of <= 8-bit products


def test_doubling_one_b_scale_changes_exactly_its_block(lib=None):
    p = wl.make_nt(4, 300, 384, seed=5)
    M, N, K = p.M, p.N, p.K
    _, acc0 = oracle.gemm_nt(p.A, p.SFA, p.B, p.SFB, M, N, K, want_acc=True, lib=lib)
    j, k = 1, 2
    SFB2 = p.SFB.copy()
    SFB2[0, j, k] *= 2
    _, acc1 = oracle.gemm_nt(p.A, p.SFA, p.B, SFB2, M, N, K, want_acc=True, lib=lib)
    for m in range(M):
        for n in range(N):
            if n // 128 != j:
                assert acc1[m, n] == acc0[m, n]
            else:
                want = float(p.SFA[k, m]) * float(p.SFB[0, j, k]) * _block_partial(p, m, n, k)
                d = acc1[m, n] - acc0[m, n]
                assert abs(d - want) <= 1e-12 * (abs(acc0[m, n]) + abs(want) + 1e-30), (m, n)


def test_doubling_one_a_scale_changes_exactly_its_row(lib=None):
    p = wl.make_nt(5, 200, 256, seed=6)
    M, N, K = p.M, p.N, p.K
    _, acc0 = oracle.gemm_nt(p.A, p.SFA, p.B, p.SFB, M, N, K, want_acc=True, lib=lib)
    m0, k = 3, 1
    SFA2 = p.SFA.copy()
    SFA2[k, m0] *= 2
    _, acc1 = oracle.gemm_nt(p.A, SFA2, p.B, p.SFB, M, N, K, want_acc=True, lib=lib)
    for m in range(M):
        for n in range(N):
            if m != m0:
                assert acc1[m, n] == acc0[m, n]
            else:
                want = float(p.SFA[k, m]) * float(p.SFB[0, n // 128, k]) * _block_partial(p, m, n, k)
                d = acc1[m, n] - acc0[m, n]
                assert abs(d - want) <= 1e-12 * (abs(acc0[m, n]) + abs(want) + 1e-30), (m, n)


def test_contiguous_single_group_equals_dense(lib=None):
    p = wl.make_nt(256, 160, 256, seed=8)
    dense = oracle.gemm_nt(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, lib=lib)
    layout = np.zeros(p.M, np.int32)
    D = oracle.gemm_grouped_contiguous_rows(p.A, p.SFA, p.B, p.SFB, layout, p.M, p.N, p.K, 1,
                                            np.arange(p.M), lib=lib)
    assert np.array_equal(D, dense)


def test_contiguous_rows_use_their_own_group(lib=None):
    p = wl.make_contiguous([128, 256, 128], 136, 256, seed=9)
    rows = np.arange(p.M)
    D = oracle.gemm_grouped_contiguous_rows(p.A, p.SFA, p.B, p.SFB, p.m_indices, p.M, p.N, p.K,
                                            p.G, rows, lib=lib)
    start = 0
    for g, r in enumerate(p.meta["group_rows"]):
        # the rows of group g against B[g], as a plain GEMM over those rows
        sub_rows = np.arange(start, start + r)
        sfa = np.zeros((p.kb, wl.sfa_ld(r)), np.float32)
        sfa[:, :r] = p.SFA[:, sub_rows]
        want = oracle.gemm_nt(p.A[sub_rows], sfa, p.B[g], p.SFB[g], r, p.N, p.K, lib=lib)
        assert np.array_equal(D[sub_rows], want), g
        start += r


def test_contiguous_negative_group_leaves_rows(lib=None):
    p = wl.make_contiguous([128, 128], 64, 128, seed=10)
    layout = p.m_indices.copy()
    layout[:128] = -1
    init = np.full((p.M, p.N), 0x7FA5, np.uint16)
    D = oracle.gemm_grouped_contiguous_rows(p.A, p.SFA, p.B, p.SFB, layout, p.M, p.N, p.K, p.G,
                                            np.arange(p.M), D_init=init, lib=lib)
    assert (D[:128] == 0x7FA5).all()
    assert not (D[128:] == 0x7FA5).any()


def test_masked_full_counts_equal_per_group_dense(lib=None):
    G, M_max, N, K = 3, 136, 144, 256
    p = wl.make_masked([M_max] * G, M_max, N, K, seed=11)
    for g in range(G):
        D = oracle.gemm_grouped_masked_rows(p.A, p.SFA, p.B, p.SFB, p.masked_m, G, M_max, N, K,
                                            g, np.arange(M_max), lib=lib)
        want = oracle.gemm_nt(p.A[g], p.SFA[g], p.B[g], p.SFB[g], M_max, N, K, lib=lib)
        assert np.array_equal(D, want), g


def test_masked_rows_beyond_count_untouched(lib=None):
    G, M_max, N, K = 2, 64, 32, 128
    p = wl.make_masked([0, 17], M_max, N, K, seed=12)
    init = np.full((M_max, N), 0x7FA5, np.uint16)
    D0 = oracle.gemm_grouped_masked_rows(p.A, p.SFA, p.B, p.SFB, p.masked_m, G, M_max, N, K, 0,
                                         np.arange(M_max), D_init=init, lib=lib)
    assert (D0 == 0x7FA5).all()
    D1 = oracle.gemm_grouped_masked_rows(p.A, p.SFA, p.B, p.SFB, p.masked_m, G, M_max, N, K, 1,
                                         np.arange(M_max), D_init=init, lib=lib)
    assert (D1[17:] == 0x7FA5).all() and not (D1[:17] == 0x7FA5).any()


def test_row_driver_threads_bitwise(lib=None):
    p = wl.make_nt(64, 256, 256, seed=13)
    D1 = oracle.gemm_nt(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, lib=lib)
    rows = np.arange(p.M)
    D4 = oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows, threads=4, lib=lib)
    assert np.array_equal(D1, D4)
    sel = np.array([63, 0, 17])
    Ds = oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, sel, threads=2, lib=lib)
    assert np.array_equal(Ds, D1[sel])


def test_acc_row_driver_threads_bitwise(lib=None):
    p = wl.make_nt_acc(40, 272, 384, seed=15)
    rows = np.arange(p.M)
    one, acc1 = oracle.gemm_nt_acc_rows(p.A, p.SFA, p.B, p.SFB, p.C, p.M, p.N, p.K, rows,
                                        threads=1, want_acc=True, lib=lib)
    four, acc4 = oracle.gemm_nt_acc_rows(p.A, p.SFA, p.B, p.SFB, p.C, p.M, p.N, p.K, rows,
                                         threads=4, want_acc=True, lib=lib)
    assert np.array_equal(one, four) and np.array_equal(acc1, acc4)


def test_element_matches_full_product(lib=None):
    p = wl.make_nt(3, 260, 384, seed=14)
    _, acc = oracle.gemm_nt(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, want_acc=True, lib=lib)
    for m, n in [(0, 0), (2, 259), (1, 128), (1, 127)]:
        assert oracle.element(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, m, n, lib=lib) == acc[m, n]
