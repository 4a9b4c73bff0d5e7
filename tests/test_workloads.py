"""Checks of the seeded input generator (no GPU)."""
import numpy as np
import torch

import workloads as wl


def test_e4m3_encode_matches_library_cast():
    # library reference: torch's fp32 -> float8_e4m3fn cast (round to nearest
    # even) of values already clamped to the finite range
    x = np.concatenate([
        wl.normal_f32(0, 50, 100_000) * 100,
        wl.normal_f32(0, 51, 50_000) * 0.01,
        np.array([0.0, -0.0, 448.0, -448.0, 449.0, 500.0, 2 ** -10, 2 ** -9, 3 * 2 ** -10,
                  1.0625, 1.1875, 2 ** -6 * (1 - 2 ** -5)], np.float32)])
    x = x.astype(np.float32)
    got = wl.e4m3_encode(x)
    ref = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(got != ref)[0]
    assert len(bad) == 0, [(float(x[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_quantise_recipe():
    x = wl.normal_f32(0, 1, 4 * 256).reshape(4, 256)
    q, s = wl.quantize_rows_1x128(x)
    amax = np.abs(x.reshape(4, 2, 128)).max(axis=2)
    assert np.array_equal(s, (amax / np.float32(448)).astype(np.float32))
    deq = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    # every block reaches +-448 at its maximum and round-trips within half an ulp
    assert (np.abs(deq.reshape(4, 2, 128)).max(axis=2) == 448).all()
    rel = np.abs(deq * np.repeat(s, 128, axis=1) - x) / np.maximum(np.abs(x), 1e-30)
    assert np.median(rel) < 2 ** -4


def test_quantise_blocks_ragged_n():
    x = wl.normal_f32(0, 2, 200 * 256).reshape(200, 256)
    q, s = wl.quantize_blocks_128x128(x)
    assert s.shape == (2, 2) and q.shape == (200, 256)
    assert s[1, 0] == np.float32(np.abs(x[128:, :128]).max() / np.float32(448))


def test_zero_block_gets_unit_scale():
    x = np.zeros((2, 128), np.float32)
    q, s = wl.quantize_rows_1x128(x)
    assert (s == 1).all() and (q == 0).all()


def test_generator_deterministic_and_sliceable():
    a = wl.normal_f32(0, 1, 10_000)
    b = wl.normal_f32(0, 1, 10_000)
    assert np.array_equal(a, b)
    c = wl.normal_f32(0, 1, 3000, start=4000)
    assert np.array_equal(a[4000:7000], c)
    assert abs(float(a.mean())) < 0.05 and abs(float(a.std()) - 1) < 0.05


def test_group_recipes():
    rows = wl.contiguous_group_rows(8)
    assert len(rows) == 8 and all(1024 <= r <= 6144 and r % 128 == 0 for r in rows)
    counts = wl.masked_counts(16, 256)
    assert len(counts) == 16 and counts.min() >= 0 and counts.max() <= 256


def test_problem_accounting():
    p = wl.make_nt(128, 256, 512)
    assert p.flops() == 2 * 128 * 256 * 512
    assert p.algorithmic_bytes() == 264_224


def test_addend_recipe():
    """The accumulate variant's C: fp32 [M][N], sqrt(K) * N(0,1) from its own
    stream, the plain problem's A and B unchanged, C counted in the bytes."""
    M, N, K = 130, 256, 1024
    p = wl.make_nt_acc(M, N, K, seed=3)
    q = wl.make_nt(M, N, K, seed=3)
    assert p.kind == "nt_acc" and p.C.shape == (M, N) and p.C.dtype == np.float32
    assert np.array_equal(p.A, q.A) and np.array_equal(p.B, q.B)
    assert np.array_equal(p.C, wl.make_nt_acc(M, N, K, seed=3).C)
    want = (wl.normal_f32(3, wl.STREAM_C, M * N) * np.float32(np.sqrt(K))).reshape(M, N)
    assert np.array_equal(p.C, want)
    assert 0.9 * np.sqrt(K) < p.C.std() < 1.1 * np.sqrt(K)
    assert p.flops() == q.flops()
    assert p.algorithmic_bytes() == q.algorithmic_bytes() + 4 * M * N


def test_ue8m0_quantise_recipe():
    """Power-of-two scales: each is the smallest 2^j with amax / 2^j <= 448,
    so no block saturates and its largest element lands in the top binade
    [224, 448]; a zero block gets the byte 127 (scale 1)."""
    x = wl.normal_f32(0, 70, 8 * 512).reshape(8, 512) * np.float32(3.7)
    x[3, 128:256] = 0
    q, e = wl.quantize_rows_1x128_ue8m0(x)
    assert e.dtype == np.uint8 and e.shape == (8, 4) and e[3, 1] == 127
    scale = np.ldexp(1.0, e.astype(np.int64) - 127)
    amax = np.abs(x.reshape(8, 4, 128)).astype(np.float64).max(axis=2)
    live = amax > 0
    assert (amax[live] / scale[live] <= 448).all() and (amax[live] / scale[live] > 224).all()
    deq = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy().reshape(8, 4, 128)
    top = np.abs(deq).max(axis=2)
    assert ((top[live] >= 224) & (top[live] <= 448)).all()
    # the byte rule at exact powers of two: amax = 448 * 2^j gives j itself
    assert list(wl.ue8m0_exponents(np.array([448.0, 896.0, 224.0, 448.0 * 2 ** -20, 0.0]))) == \
        [127, 128, 126, 107, 127]
    p = wl.make_nt_ue8m0(130, 200, 384, seed=4)
    assert p.kind == "nt_ue8m0" and p.SFA.dtype == np.uint8 and p.SFB.shape == (1, 2, 3)
    assert (p.SFA[:, 130:] == 127).all()
    assert p.algorithmic_bytes() == 130 * (384 + 3 + 2 * 200) + 200 * 384 + 2 * 3
