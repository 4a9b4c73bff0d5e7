"""Parity of fp8_gemm_nt_ue8m0 (power-of-two scales applied by the tensor
cores' block-scaled MMA) with the oracle's UE8M0 mode, through the C ABI.

Element by element on ragged shapes (M and N tails, one and many K blocks,
K block counts that leave a partial scale chunk), bit for bit on exact
small-integer inputs with exponents 124..130, the scale-doubling invariant
(raising one B block's exponent by one doubles exactly that block's columns),
determinism, a CUDA graph replay, and the full-size dense shapes on sampled
rows; each on the one-CTA kernel and on CTA pairs.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests import gpu_util as gu
from tests.tolerance import check

pytestmark = pytest.mark.gpu

THREADS = oracle.default_threads()


@pytest.fixture(autouse=True, params=[-1, 1], ids=["one_cta", "pair"])
def cta_mode(request):
    """Every test runs on the one-CTA kernel (128 x 256 tiles,
    fp8_gemm_set_pair_mode(-1)) and on CTA pairs (256 x 256 tiles,
    fp8_gemm_set_pair_mode(1))."""
    import fp8_block_scaled_persistent_gb300 as fg
    assert fg.fp8_gemm_set_pair_mode(request.param) == fg.FP8G_OK
    yield request.param
    fg.fp8_gemm_set_pair_mode(0)
    assert fg.fp8_gemm_get_device_error() == 0


def _ref(p, rows=None):
    rows = np.arange(p.M, dtype=np.int32) if rows is None else rows
    return oracle.gemm_nt_ue8m0_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows, threads=THREADS)


def _exact_problem(M, N, K, seed):
    """Small integers (exact in E4M3) with UE8M0 exponents 124..130: every
    fp32 partial sum is exact, so the GPU must match the oracle bit for bit."""
    q = wl.exact_integer_problem(M, N, K, seed=seed)
    kb, nb = K // 128, (N + 127) // 128
    ea = (wl.raw_u64(wl.stream_key(seed, 17), 0, M * kb) % np.uint64(7)).astype(np.int64) + 124
    eb = (wl.raw_u64(wl.stream_key(seed, 18), 0, nb * kb) % np.uint64(7)).astype(np.int64) + 124
    SFA = np.full((kb, (M + 3) // 4 * 4), 127, np.uint8)
    SFA[:, :M] = ea.reshape(M, kb).T
    SFB = eb.reshape(1, nb, kb).astype(np.uint8)
    return wl.Problem("nt_ue8m0", M, N, K, 1, q.A, SFA, q.B, SFB, name=f"ue8m0 exact {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [
    (1, 16, 128), (63, 48, 256), (128, 256, 512), (129, 272, 640), (200, 512, 1024),
    (256, 400, 1536), (300, 96, 2304), (520, 1040, 2048), (64, 7168, 16384)])
def test_ue8m0_shapes(M, N, K):
    p = wl.make_nt_ue8m0(M, N, K, seed=M * 3 + N)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    check(got, _ref(p), f"ue8m0 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (130, 384, 1024), (7, 272, 3968), (256, 512, 2048)])
def test_ue8m0_exact_integers_bit_identical(M, N, K):
    p = _exact_problem(M, N, K, seed=M + N)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    assert np.array_equal(got, _ref(p))


def test_ue8m0_scale_doubling_moves_one_block():
    """Raising the exponent of B block (1, k) by one doubles exactly the
    contribution of that block: with integer inputs the difference of the
    two results is that block's partial sum, exactly, and only in its 128
    columns."""
    M, N, K = 128, 384, 512
    p = _exact_problem(M, N, K, seed=9)
    base, st, _ = gu.run(p)
    assert st == 0
    q = wl.Problem("nt_ue8m0", M, N, K, 1, p.A, p.SFA, p.B, p.SFB.copy(), name="doubled")
    q.SFB[0, 1, 2] += 1
    got, st, _ = gu.run(q)
    assert st == 0
    assert np.array_equal(got, _ref(q))
    changed = np.any(got != base, axis=0)
    assert not changed[:128].any() and not changed[256:].any()
    assert changed[128:256].any()


def test_ue8m0_deterministic():
    p = wl.make_nt_ue8m0(384, 1024, 2048, seed=4)
    a, _, _ = gu.run(p)
    b, _, _ = gu.run(p)
    assert np.array_equal(a, b)


def test_ue8m0_graph_replay_bit_identical():
    """Two shapes captured into one CUDA graph on a side stream replay, twice,
    to the eager calls' bits (the pair path launches clusters of two)."""
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    probs = [wl.make_nt_ue8m0(300, 528, 2304, seed=6), wl.make_nt_ue8m0(64, 256, 512, seed=7)]
    tens = [gu.dev_tensors(p) for p in probs]
    side = torch.cuda.Stream()
    ref = [gu.new_d(p) for p in probs]
    with torch.cuda.stream(side):
        for p, t, D in zip(probs, tens, ref):
            assert gu.call(p, t, D, stream=side) == 0
    side.synchronize()
    assert fg.fp8_gemm_get_device_error(side) == 0
    ref_bits = [gu.bits(D) for D in ref]
    outs = [gu.new_d(p) for p in probs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for p, t, D in zip(probs, tens, outs):
            assert gu.call(p, t, D, stream=side) == 0
    for _ in range(2):
        for D in outs:
            D.view(torch.int16).fill_(np.int16(np.uint16(gu.SENTINEL).view(np.int16)))
        g.replay()
        torch.cuda.synchronize()
        assert fg.fp8_gemm_get_device_error() == 0
        for i, (D, r) in enumerate(zip(outs, ref_bits)):
            assert np.array_equal(gu.bits(D), r), f"replay output {i}"
    check(ref_bits[0], _ref(probs[0]), "ue8m0 graph 300x528x2304")


def test_ue8m0_argument_checks():
    import fp8_block_scaled_persistent_gb300 as fg
    import torch
    p = wl.make_nt_ue8m0(128, 256, 512, seed=1)
    t = gu.dev_tensors(p)
    D = gu.new_d(p)
    assert fg.fp8_gemm_nt_ue8m0(t["A"], None, t["B"], t["SFB"], D, 128, 256, 512) == fg.FP8G_ERR_INVALID_ARG
    assert fg.fp8_gemm_nt_ue8m0(t["A"], t["SFA"], t["B"], t["SFB"], D, 128, 256, 500) == fg.FP8G_ERR_UNSUPPORTED
    assert fg.fp8_gemm_nt_ue8m0(t["A"], t["SFA"], t["B"], t["SFB"], D, 128, 250, 512) == fg.FP8G_ERR_UNSUPPORTED
    assert fg.fp8_gemm_nt_ue8m0(t["A"], t["SFA"], t["B"], t["SFB"], D, 0, 256, 512) == fg.FP8G_OK
    torch.cuda.synchronize()
    assert (gu.bits(D) == gu.SENTINEL).all()


@pytest.mark.parametrize("name", ["ue8m0_4096x7168x2048", "ue8m0_4096x24576x1536"])
def test_ue8m0_full_size_sampled_rows(name):
    p = wl.make(name)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    rows = gu.sample_rows(p.M, 12, seed=1, must=(0, 127, 128, p.M - 1))
    check(got[rows], _ref(p, rows), name)
    again, _, _ = gu.run(p)
    assert np.array_equal(got, again)
