"""Parity of the CUDA path with the CPU oracle, through the C ABI.

Small problems are compared element by element (every element of D); the
full-size workloads are compared on sampled rows (every element of each
sampled row), in the launch configuration the benchmark uses.  The bound is
the method's stated tolerance (tests/tolerance.py).  Exact small-integer
inputs must match bit for bit.  Rows the method must leave untouched are
checked bit-exactly against a sentinel fill.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests import gpu_util as gu
from tests.tolerance import check

pytestmark = pytest.mark.gpu

THREADS = oracle.default_threads()


@pytest.fixture(autouse=True)
def _reset_overrides():
    import fp8_block_scaled_persistent_gb300 as fg
    fg.fp8_gemm_set_override(0, 0)
    yield
    fg.fp8_gemm_set_override(0, 0)
    assert fg.fp8_gemm_get_device_error() == 0


def _full_ref(p):
    return oracle.gemm_nt(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K)


# ------------------------------------------------------------------ plain GEMM

def test_single_workload_elementwise():
    p = wl.make("single_128x256x512")
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    check(got, _full_ref(p), p.name)


@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("M,N,K", [
    (1, 16, 128), (63, 48, 256), (64, 128, 128), (65, 144, 384), (127, 256, 256),
    (129, 272, 640), (200, 512, 512), (256, 400, 1024), (300, 96, 256)])
def test_edge_shapes(M, N, K, block_n):
    import fp8_block_scaled_persistent_gb300 as fg
    fg.fp8_gemm_set_override(block_n, -1)
    p = wl.make_nt(M, N, K, seed=M * 7 + N)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    check(got, _full_ref(p), f"{M}x{N}x{K} bn{block_n}")


@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (130, 384, 1024), (7, 272, 3968)])
def test_exact_integers_bit_identical(M, N, K, block_n):
    import fp8_block_scaled_persistent_gb300 as fg
    fg.fp8_gemm_set_override(block_n, -1)
    p = wl.exact_integer_problem(M, N, K, seed=M + N)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    assert np.array_equal(got, _full_ref(p))


def test_output_guard_bands_untouched():
    """Canaries before and after D stay bit-identical (ragged M and N)."""
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    p = wl.make_nt(131, 208, 256, seed=3)
    t = gu.dev_tensors(p)
    pad = 4096
    buf = torch.empty(pad + p.M * p.N + pad, dtype=torch.int16, device="cuda")
    buf.fill_(np.int16(np.uint16(gu.SENTINEL).view(np.int16)))
    D = buf[pad:pad + p.M * p.N].view(torch.bfloat16).view(p.M, p.N)
    assert gu.call(p, t, D) == 0
    assert fg.fp8_gemm_get_device_error() == 0
    host = buf.cpu().numpy().view(np.uint16)
    assert (host[:pad] == gu.SENTINEL).all() and (host[-pad:] == gu.SENTINEL).all()
    check(host[pad:-pad].reshape(p.M, p.N), _full_ref(p), "guarded")


def test_deterministic():
    p = wl.make_nt(256, 512, 2048, seed=4)
    a, _, _ = gu.run(p)
    b, _, _ = gu.run(p)
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ split-K schedule

@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("M,N,K,P", [
    (64, 256, 2048, 7), (128, 512, 4096, 24), (100, 384, 1536, 5), (128, 128, 1024, 3),
    (64, 1024, 8192, 152), (1, 128, 512, 4)])
def test_split_k_matches_oracle(M, N, K, P, block_n):
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    assert fg.fp8_gemm_set_override(block_n, P) == 0
    p = wl.make_nt(M, N, K, seed=M + K)
    n = fg.fp8_gemm_workspace_size_for(M, N, K, block_n, P)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    got, st, dst = gu.run(p, workspace=ws)
    assert st == 0 and dst == 0
    check(got, _full_ref(p), f"split {M}x{N}x{K} P={P} bn{block_n}")
    # the tickets are back at zero, and a second run gives the same bits
    ntiles = ((M + 127) // 128) * ((N + block_n - 1) // block_n)
    assert int(ws[: ntiles * 8 * 4].view(torch.int32).abs().sum()) == 0
    again, st2, _ = gu.run(p, workspace=ws)
    assert st2 == 0 and np.array_equal(got, again)


@pytest.mark.parametrize("block_n", [128, 256])
def test_split_k_exact_integers_bit_identical(block_n):
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    M, N, K, P = 128, 256, 3968, 9
    assert fg.fp8_gemm_set_override(block_n, P) == 0
    p = wl.exact_integer_problem(M, N, K, seed=5)
    ws = torch.zeros(fg.fp8_gemm_workspace_size_for(M, N, K, block_n, P), dtype=torch.uint8, device="cuda")
    got, st, dst = gu.run(p, workspace=ws)
    assert st == 0 and dst == 0
    assert np.array_equal(got, _full_ref(p))


def test_forced_split_without_workspace_is_rejected():
    import fp8_block_scaled_persistent_gb300 as fg
    assert fg.fp8_gemm_set_override(128, 8) == 0
    p = wl.make_nt(64, 128, 1024, seed=6)
    _, st, _ = gu.run(p, workspace=None)
    assert st == fg.FP8G_ERR_WORKSPACE


# ------------------------------------------------------------------ grouped, contiguous

def test_contiguous_elementwise():
    p = wl.make_contiguous([128, 256, 128, 384], 272, 512, seed=21)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    ref = oracle.gemm_grouped_contiguous_rows(p.A, p.SFA, p.B, p.SFB, p.m_indices, p.M, p.N, p.K,
                                              p.G, np.arange(p.M), threads=THREADS)
    check(got, ref, "contiguous")


def test_contiguous_skips_negative_blocks_and_flags_bad_ones():
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    p = wl.make_contiguous([128, 128, 256], 128, 256, seed=22)
    layout = p.m_indices.copy()
    layout[0:128] = -1          # skipped, untouched, no error
    t = gu.dev_tensors(p)
    D = gu.new_d(p)
    lay = torch.from_numpy(layout).cuda()
    assert gu.call(p, t, D, layout=lay) == 0
    assert fg.fp8_gemm_get_device_error() == 0
    got = gu.bits(D)
    assert (got[:128] == gu.SENTINEL).all()
    ref = oracle.gemm_grouped_contiguous_rows(p.A, p.SFA, p.B, p.SFB, layout, p.M, p.N, p.K, p.G,
                                              np.arange(128, p.M), threads=THREADS)
    check(got[128:], ref, "contiguous -1")
    layout[128:256] = 7         # out of range: skipped and flagged
    lay = torch.from_numpy(layout).cuda()
    D = gu.new_d(p)
    assert gu.call(p, t, D, layout=lay) == 0
    assert fg.fp8_gemm_get_device_error() == fg.FP8G_ERR_BAD_GROUP
    got = gu.bits(D)
    assert (got[:256] == gu.SENTINEL).all()
    check(got[256:], ref[128:], "contiguous bad group")


def test_contiguous_single_group_equals_plain():
    p = wl.make_nt(384, 256, 512, seed=23)
    dense, _, _ = gu.run(p)
    q = wl.Problem("contiguous", p.M, p.N, p.K, 1, p.A, p.SFA, p.B, p.SFB,
                   m_indices=np.zeros(p.M, np.int32))
    got, st, dst = gu.run(q)
    assert st == 0 and dst == 0
    assert np.array_equal(got, dense)


# ------------------------------------------------------------------ grouped, masked

@pytest.mark.parametrize("counts,M_max", [([0, 1, 130, 200], 200), ([256, 255, 128, 17], 256)])
def test_masked_elementwise_and_untouched(counts, M_max):
    p = wl.make_masked(counts, M_max, 272, 512, seed=31)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    for g, c in enumerate(counts):
        assert (got[g, c:] == gu.SENTINEL).all(), f"group {g} rows beyond {c} were written"
        if c:
            ref = oracle.gemm_grouped_masked_rows(p.A, p.SFA, p.B, p.SFB, p.masked_m, p.G, M_max,
                                                  p.N, p.K, g, np.arange(c), threads=THREADS)
            check(got[g, :c], ref, f"masked g{g}")


def test_masked_count_above_max_is_clamped_and_flagged():
    import fp8_block_scaled_persistent_gb300 as fg
    p = wl.make_masked([300, 5], 256, 128, 256, seed=32)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == fg.FP8G_ERR_BAD_GROUP
    ref = oracle.gemm_grouped_masked_rows(p.A, p.SFA, p.B, p.SFB, np.array([256, 5], np.int32), 2,
                                          256, p.N, p.K, 0, np.arange(256), threads=THREADS)
    check(got[0], ref, "clamped group")
    assert (got[1, 5:] == gu.SENTINEL).all()


def test_masked_all_zero_counts_write_nothing():
    p = wl.make_masked([0, 0, 0], 128, 256, 256, seed=33)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    assert (got == gu.SENTINEL).all()


# ------------------------------------------------------------------ full-size workloads

FULL = ["dense_4096x7168x2048", "dense_4096x24576x1536", "smallm_64x7168x16384",
        "smallm_128x7168x16384", "contiguous_g8_n4096_k7168", "masked_g16_m256_n7168_k2048"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows(name):
    p = wl.make(name)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    if p.kind == "nt":
        rows = gu.sample_rows(p.M, 10, seed=1, must=(0, p.M - 1, 127, 128))
        ref = oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows, threads=THREADS)
        check(got[rows], ref, name)
    elif p.kind == "contiguous":
        # every group's first and last row, the first row of the group's
        # second 128-row block, and random rows
        starts = np.cumsum([0] + p.meta["group_rows"][:-1])
        ends = starts + np.array(p.meta["group_rows"]) - 1
        must = list(starts) + list(ends) + [s + 128 for s in starts if s + 128 <= p.M - 1]
        rows = gu.sample_rows(p.M, 16, seed=2, must=must)
        ref = oracle.gemm_grouped_contiguous_rows(p.A, p.SFA, p.B, p.SFB, p.m_indices, p.M, p.N,
                                                  p.K, p.G, rows, threads=THREADS)
        check(got[rows], ref, name)
    else:
        for g in range(p.G):
            c = int(p.masked_m[g])
            assert (got[g, c:] == gu.SENTINEL).all(), f"{name}: group {g} rows beyond {c} written"
        # every live group: its first and last valid row, both sides of the
        # 128-row boundary when the count crosses it, and random valid rows
        for g in np.nonzero(p.masked_m)[0]:
            c = int(p.masked_m[g])
            must = (0, c - 1) + ((127, 128) if c > 128 else ())
            rows = gu.sample_rows(c, 3, seed=int(g), must=must)
            ref = oracle.gemm_grouped_masked_rows(p.A, p.SFA, p.B, p.SFB, p.masked_m, p.G, p.M,
                                                  p.N, p.K, int(g), rows, threads=THREADS)
            check(got[g][rows], ref, f"{name} g{g}")
    again, _, _ = gu.run(p)
    assert np.array_equal(got, again), f"{name}: not deterministic"


@pytest.mark.parametrize("M", [384, 1280])
def test_automatic_pair_choice_padding(M):
    """The automatic choice leaves a problem on one CTA when 256-row pair
    tiles would pad M by more than an eighth (384 rows: 512 computed), and
    takes pairs when they do not (1280 rows); both agree with the oracle on
    sampled rows, and with the one-CTA kernel (pair mode -1) within the
    tolerance."""
    import fp8_block_scaled_persistent_gb300 as fg
    p = wl.make_nt(M, 24576, 1024, seed=M)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    rows = gu.sample_rows(p.M, 8, seed=3, must=(0, 127, 128, 255, 256, p.M - 1))
    ref = oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows, threads=THREADS)
    check(got[rows], ref, f"automatic {M}")
    assert fg.fp8_gemm_set_pair_mode(-1) == fg.FP8G_OK
    try:
        one, st, dst = gu.run(p)
    finally:
        fg.fp8_gemm_set_pair_mode(0)
    assert st == 0 and dst == 0
    check(one[rows], ref, f"one CTA {M}")


@pytest.mark.parametrize("name", ["dense_4096x7168x2048", "dense_4096x24576x1536"])
def test_full_size_dense_one_cta(name):
    """The dense workloads on the one-CTA kernel (pair mode -1; the automatic
    choice runs them on CTA pairs), sampled rows against the oracle."""
    import fp8_block_scaled_persistent_gb300 as fg
    assert fg.fp8_gemm_set_pair_mode(-1) == fg.FP8G_OK
    try:
        p = wl.make(name)
        got, st, dst = gu.run(p)
    finally:
        fg.fp8_gemm_set_pair_mode(0)
    assert st == 0 and dst == 0
    rows = gu.sample_rows(p.M, 10, seed=4, must=(0, 127, 128, 255, 256, p.M - 1))
    ref = oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows, threads=THREADS)
    check(got[rows], ref, f"{name} one CTA")
