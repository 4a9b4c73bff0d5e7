"""Parity of the CTA-pair kernel (clusters of two CTAs sharing 256 x 128
tiles through tcgen05.mma.cta_group::2) with the CPU oracle, through the C
ABI with fp8_gemm_set_pair_mode(1).

Every test runs with both pair tile widths.  Covers the plain GEMM on ragged shapes (pair tiles whose second CTA has few
or no rows, column tails), exact small-integer inputs bit for bit, the
contiguous layout with pair tiles whose two 128-row blocks belong to
different groups (the second pass), skipped and out-of-range blocks, the
masked layout with counts on both sides of 128 and 256 (rows past a count
untouched), the fp32 addend (at 256-column tiles copied through the staging
area by the addend/store warp), guard bands, determinism, a CUDA graph
replay, and the full-size workloads on sampled rows.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests import gpu_util as gu
from tests.tolerance import check

pytestmark = pytest.mark.gpu

THREADS = oracle.default_threads()


@pytest.fixture(autouse=True, params=[128, 256], ids=["pair256x128", "pair256x256"])
def pair_bn(request):
    """Every test runs with both pair tile widths (256 x 128 and 256 x 256);
    splitting K is forbidden so that the pair kernel is what runs."""
    import fp8_block_scaled_persistent_gb300 as fg
    assert fg.fp8_gemm_set_override(request.param, -1) == fg.FP8G_OK
    assert fg.fp8_gemm_set_pair_mode(1) == fg.FP8G_OK
    yield request.param
    fg.fp8_gemm_set_pair_mode(0)
    fg.fp8_gemm_set_override(0, 0)
    assert fg.fp8_gemm_get_device_error() == 0


def _ref(p):
    return oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, np.arange(p.M), threads=THREADS)


def test_pair_mode_argument_checks():
    import fp8_block_scaled_persistent_gb300 as fg
    assert fg.fp8_gemm_set_pair_mode(3) == fg.FP8G_ERR_INVALID_ARG
    assert fg.fp8_gemm_set_pair_mode(-2) == fg.FP8G_ERR_INVALID_ARG


@pytest.mark.parametrize("M,N,K", [
    (1, 16, 128), (63, 48, 256), (128, 128, 128), (129, 272, 640), (200, 512, 512),
    (256, 400, 1024), (300, 96, 256), (384, 256, 1536), (520, 1040, 2048), (1000, 144, 384)])
def test_pair_plain_shapes(M, N, K):
    p = wl.make_nt(M, N, K, seed=M * 5 + N)
    got, st, dst = gu.run(p, workspace=None)
    assert st == 0 and dst == 0
    check(got, _ref(p), f"pair {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(256, 256, 512), (130, 384, 1024), (512, 128, 3968)])
def test_pair_exact_integers_bit_identical(M, N, K):
    p = wl.exact_integer_problem(M, N, K, seed=M + N + 1)
    got, st, dst = gu.run(p, workspace=None)
    assert st == 0 and dst == 0
    assert np.array_equal(got, _ref(p))


def test_pair_guard_bands_and_determinism():
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    p = wl.make_nt(387, 208, 768, seed=3)
    t = gu.dev_tensors(p)
    pad = 4096
    buf = torch.empty(pad + p.M * p.N + pad, dtype=torch.int16, device="cuda")
    buf.fill_(np.int16(np.uint16(gu.SENTINEL).view(np.int16)))
    D = buf[pad:pad + p.M * p.N].view(torch.bfloat16).view(p.M, p.N)
    assert gu.call(p, t, D) == 0
    assert fg.fp8_gemm_get_device_error() == 0
    host = buf.cpu().numpy().view(np.uint16)
    assert (host[:pad] == gu.SENTINEL).all() and (host[-pad:] == gu.SENTINEL).all()
    first = host[pad:-pad].reshape(p.M, p.N).copy()
    check(first, _ref(p), "pair guarded")
    assert gu.call(p, t, D) == 0
    assert np.array_equal(gu.bits(D), first)


def test_pair_contiguous_straddling_pairs():
    # 128-row blocks: groups 0 | 1 1 | 2 | 3 3 3: pair tiles (0,1), (1,2),
    # (3,3), (3,-): the first two need the second pass
    p = wl.make_contiguous([128, 256, 128, 384], 272, 512, seed=21)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    ref = oracle.gemm_grouped_contiguous_rows(p.A, p.SFA, p.B, p.SFB, p.m_indices, p.M, p.N, p.K,
                                              p.G, np.arange(p.M), threads=THREADS)
    check(got, ref, "pair contiguous")


def test_pair_contiguous_skipped_and_bad_blocks():
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    p = wl.make_contiguous([128, 128, 256, 128], 128, 256, seed=22)
    layout = p.m_indices.copy()
    layout[0:128] = -1              # first block of the first pair skipped
    layout[384:512] = -1            # second block of the second pair skipped
    t = gu.dev_tensors(p)
    D = gu.new_d(p)
    assert gu.call(p, t, D, layout=torch.from_numpy(layout).cuda()) == 0
    assert fg.fp8_gemm_get_device_error() == 0
    got = gu.bits(D)
    assert (got[:128] == gu.SENTINEL).all() and (got[384:512] == gu.SENTINEL).all()
    live = np.r_[128:384, 512:640]
    ref = oracle.gemm_grouped_contiguous_rows(p.A, p.SFA, p.B, p.SFB, layout, p.M, p.N, p.K, p.G,
                                              live, threads=THREADS)
    check(got[live], ref, "pair contiguous -1")
    layout[128:256] = 9             # out of range: skipped and flagged
    D = gu.new_d(p)
    assert gu.call(p, t, D, layout=torch.from_numpy(layout).cuda()) == 0
    assert fg.fp8_gemm_get_device_error() == fg.FP8G_ERR_BAD_GROUP
    got = gu.bits(D)
    assert (got[:256] == gu.SENTINEL).all()
    live2 = np.r_[256:384, 512:640]
    ref2 = oracle.gemm_grouped_contiguous_rows(p.A, p.SFA, p.B, p.SFB, layout, p.M, p.N, p.K, p.G,
                                               live2, threads=THREADS)
    check(got[live2], ref2, "pair contiguous bad group")


@pytest.mark.parametrize("counts,M_max", [([0, 1, 130, 200], 200), ([256, 255, 128, 17], 256),
                                          ([300, 0, 257, 511], 512)])
def test_pair_masked_elementwise_and_untouched(counts, M_max):
    import fp8_block_scaled_persistent_gb300 as fg
    p = wl.make_masked(counts, M_max, 272, 512, seed=31)
    got, st, dst = gu.run(p)
    assert st == 0
    assert dst == (fg.FP8G_ERR_BAD_GROUP if max(counts) > M_max else 0)
    for g, c in enumerate(counts):
        c = min(c, M_max)
        assert (got[g, c:] == gu.SENTINEL).all(), f"group {g} rows beyond {c} were written"
        if c:
            cc = np.minimum(p.masked_m, M_max).astype(np.int32)
            ref = oracle.gemm_grouped_masked_rows(p.A, p.SFA, p.B, p.SFB, cc, p.G, M_max,
                                                  p.N, p.K, g, np.arange(c), threads=THREADS)
            check(got[g, :c], ref, f"pair masked g{g}")


@pytest.mark.parametrize("M,N,K", [(256, 512, 1024), (300, 272, 640)])
def test_pair_accumulate(M, N, K):
    a = wl.make_nt_acc(M, N, K, seed=M + 3)
    got, st, dst = gu.run(a, workspace=None)
    assert st == 0 and dst == 0
    ref = oracle.gemm_nt_acc_rows(a.A, a.SFA, a.B, a.SFB, a.C, a.M, a.N, a.K, np.arange(a.M),
                                  threads=THREADS)
    check(got, ref, f"pair accumulate {M}x{N}x{K}")


def test_pair_graph_replay_bit_identical():
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    probs = [wl.make_nt(512, 1024, 1024, seed=41), wl.make_masked([5, 200, 0], 256, 256, 512, seed=43),
             wl.make_contiguous([128, 256], 256, 512, seed=44), wl.make_nt_acc(300, 528, 1280, seed=45)]
    tens = [gu.dev_tensors(p) for p in probs]
    side = torch.cuda.Stream()
    ref = [gu.new_d(p) for p in probs]
    with torch.cuda.stream(side):
        for p, t, D in zip(probs, tens, ref):
            assert gu.call(p, t, D, stream=side) == 0
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


FULL = ["dense_4096x7168x2048", "dense_4096x24576x1536", "contiguous_g8_n4096_k7168",
        "masked_g16_m256_n7168_k2048", "acc_4096x7168x2048"]


@pytest.mark.parametrize("name", FULL)
def test_pair_full_size_sampled_rows(name):
    p = wl.make(name)
    got, st, dst = gu.run(p, workspace=None)
    assert st == 0 and dst == 0
    if p.kind == "nt":
        rows = gu.sample_rows(p.M, 12, seed=1, must=(0, 127, 128, 255, 256, p.M - 1))
        ref = oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows, threads=THREADS)
        check(got[rows], ref, name)
    elif p.kind == "nt_acc":
        rows = gu.sample_rows(p.M, 12, seed=1, must=(0, 127, 128, 255, 256, p.M - 1))
        ref = oracle.gemm_nt_acc_rows(p.A, p.SFA, p.B, p.SFB, p.C, p.M, p.N, p.K, rows, threads=THREADS)
        check(got[rows], ref, name)
    elif p.kind == "contiguous":
        starts = np.cumsum([0] + p.meta["group_rows"][:-1])
        ends = starts + np.array(p.meta["group_rows"]) - 1
        rows = gu.sample_rows(p.M, 16, seed=2, must=list(starts) + list(ends))
        ref = oracle.gemm_grouped_contiguous_rows(p.A, p.SFA, p.B, p.SFB, p.m_indices, p.M, p.N,
                                                  p.K, p.G, rows, threads=THREADS)
        check(got[rows], ref, name)
    else:
        for g in range(p.G):
            c = int(p.masked_m[g])
            assert (got[g, c:] == gu.SENTINEL).all(), f"{name}: group {g} rows beyond {c} written"
        for g in np.nonzero(p.masked_m)[0]:
            c = int(p.masked_m[g])
            must = (0, c - 1) + ((127, 128) if c > 128 else ())
            rows = gu.sample_rows(c, 3, seed=int(g), must=must)
            ref = oracle.gemm_grouped_masked_rows(p.A, p.SFA, p.B, p.SFB, p.masked_m, p.G, p.M,
                                                  p.N, p.K, int(g), rows, threads=THREADS)
            check(got[g][rows], ref, f"{name} g{g}")
    again, _, _ = gu.run(p, workspace=None)
    assert np.array_equal(got, again), f"{name}: not deterministic"
