"""Parity of the accumulate variant, D = bf16(C + A B^T scaled), with the CPU
oracle, through the C ABI (fp8_gemm_nt_accumulate).

Small problems are compared element by element, across 128- and 256-column
tiles, ragged edges and the split-K schedule (where only the tile's storing
CTA may add C); the full-size workload on sampled rows.  Inputs whose every
fp32 step is exact must match bit for bit, a zero addend must reproduce
fp8_gemm_nt's bits, and a zero product must give C rounded to bf16.
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


def _ref(p, rows=None):
    rows = np.arange(p.M) if rows is None else rows
    return oracle.gemm_nt_acc_rows(p.A, p.SFA, p.B, p.SFB, p.C, p.M, p.N, p.K, rows, threads=THREADS)


def _split_ws(p, block_n, P):
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    assert fg.fp8_gemm_set_override(block_n, P) == 0
    n = fg.fp8_gemm_workspace_size_for(p.M, p.N, p.K, block_n, P)
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def _exact_with_addend(M, N, K, seed):
    """Small integers with power-of-two scales, and an addend of integers in
    [-64, 64] plus sixteenths: every fp32 partial and running sum is exact."""
    p = wl.exact_integer_problem(M, N, K, seed=seed)
    z = wl.raw_u64(wl.stream_key(seed, 16), 0, M * N)
    p.C = (((z % np.uint64(129)).astype(np.int64) - 64) +
           ((z >> np.uint64(32)) % np.uint64(16)).astype(np.int64) / 16.0).astype(np.float32).reshape(M, N)
    p.kind = "nt_acc"
    return p


@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("M,N,K", [
    (1, 16, 128), (65, 144, 384), (129, 272, 640), (200, 512, 512), (300, 96, 256)])
def test_edge_shapes(M, N, K, block_n):
    import fp8_block_scaled_persistent_gb300 as fg
    fg.fp8_gemm_set_override(block_n, -1)
    p = wl.make_nt_acc(M, N, K, seed=M * 5 + N)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    check(got, _ref(p), f"acc {M}x{N}x{K} bn{block_n}")


@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("split", [0, 9])
def test_exact_integers_bit_identical(block_n, split):
    import fp8_block_scaled_persistent_gb300 as fg
    p = _exact_with_addend(130, 384, 3968, seed=7)
    if split:
        ws = _split_ws(p, block_n, split)
    else:
        fg.fp8_gemm_set_override(block_n, -1)
        ws = None
    got, st, dst = gu.run(p, workspace=ws)
    assert st == 0 and dst == 0
    assert np.array_equal(got, _ref(p))


@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("M,N,K,P", [
    (64, 256, 2048, 7), (100, 384, 1536, 5), (1, 128, 512, 4), (64, 1024, 8192, 152)])
def test_split_k_matches_oracle(M, N, K, P, block_n):
    import torch
    p = wl.make_nt_acc(M, N, K, seed=M + K)
    ws = _split_ws(p, block_n, P)
    got, st, dst = gu.run(p, workspace=ws)
    assert st == 0 and dst == 0
    check(got, _ref(p), f"acc split {M}x{N}x{K} P={P} bn{block_n}")
    ntiles = ((M + 127) // 128) * ((N + block_n - 1) // block_n)
    assert int(ws[: ntiles * 8 * 4].view(torch.int32).abs().sum()) == 0
    again, st2, _ = gu.run(p, workspace=ws)
    assert st2 == 0 and np.array_equal(got, again)


@pytest.mark.parametrize("split", [0, 6])
def test_zero_addend_reproduces_the_plain_bits(split):
    """C = 0: the accumulator starts from +0 either way, so the bits are
    fp8_gemm_nt's."""
    p = wl.make_nt_acc(192, 640, 1024, seed=11)
    p.C = np.zeros_like(p.C)
    plain = wl.make_nt(192, 640, 1024, seed=11)
    ws = _split_ws(p, 128, split) if split else None
    got, st, dst = gu.run(p, workspace=ws)
    assert st == 0 and dst == 0
    base, st, dst = gu.run(plain, workspace=ws)
    assert st == 0 and dst == 0
    assert np.array_equal(got, base)


@pytest.mark.parametrize("split", [0, 5])
def test_zero_product_gives_the_addend_rounded(split):
    """Every A code zero: D = RNE(C) bit for bit (the library's fp32 -> bf16
    cast), ragged in both dimensions; C itself is left unchanged."""
    import torch
    p = wl.make_nt_acc(130, 272, 512, seed=12)
    p.A = np.zeros_like(p.A)
    assert (p.C != 0).all()
    ws = _split_ws(p, 128, split) if split else None
    t = gu.dev_tensors(p)
    D = gu.new_d(p)
    assert gu.call(p, t, D, workspace=ws) == 0
    import fp8_block_scaled_persistent_gb300 as fg
    assert fg.fp8_gemm_get_device_error() == 0
    want = torch.from_numpy(p.C).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(gu.bits(D), want)
    assert np.array_equal(t["C"].cpu().numpy(), p.C)


def test_full_size_sampled_rows():
    p = wl.make("acc_4096x7168x2048")
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    rows = gu.sample_rows(p.M, 10, seed=3, must=(0, p.M - 1, 127, 128))
    check(got[rows], _ref(p, rows), p.name)
    again, _, _ = gu.run(p)
    assert np.array_equal(got, again), "not deterministic"


def test_full_size_one_cta():
    """The full-size workload on the one-CTA kernel (pair mode -1; the
    automatic choice runs it on CTA pairs), sampled rows against the oracle."""
    import fp8_block_scaled_persistent_gb300 as fg
    assert fg.fp8_gemm_set_pair_mode(-1) == fg.FP8G_OK
    try:
        p = wl.make("acc_4096x7168x2048")
        got, st, dst = gu.run(p)
    finally:
        fg.fp8_gemm_set_pair_mode(0)
    assert st == 0 and dst == 0
    rows = gu.sample_rows(p.M, 10, seed=5, must=(0, 127, 128, 255, 256, p.M - 1))
    check(got[rows], _ref(p, rows), f"{p.name} one CTA")


def test_pair_addend_ragged_edges():
    """The addend on CTA pairs with 256-column tiles (the addend/store warp
    copies C through the staging area), forced by pair mode 1: ragged M and
    N, a pair whose second CTA has no rows, K below and above 8 blocks."""
    import fp8_block_scaled_persistent_gb300 as fg
    assert fg.fp8_gemm_set_pair_mode(1) == fg.FP8G_OK
    try:
        for (M, N, K) in [(100, 272, 640), (300, 528, 1024), (513, 256, 2304), (256, 784, 1280)]:
            p = wl.make_nt_acc(M, N, K, seed=M + N + K)
            got, st, dst = gu.run(p)
            assert st == 0 and dst == 0
            check(got, _ref(p), f"pair acc {M}x{N}x{K}")
    finally:
        fg.fp8_gemm_set_pair_mode(0)
