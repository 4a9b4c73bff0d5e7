"""Parity of the A-sharing clusters (fp8_gemm_set_pair_mode(2)): two
one-CTA kernels computing neighbouring n-blocks of one m-block, the first
copying each A tile into the second one's shared memory over DSMEM.

Element by element against the oracle: ragged plain shapes (including an
odd number of 256-column blocks, where the second CTA of the last cluster
has no columns and stores nothing), exact small integers bit for bit, the
contiguous layout with skipped and out-of-range blocks, the masked layout
with rows past each count untouched, repeatability, and the full-size
contiguous workload on sampled rows.  The addend variant is not shared and
must still match.
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
def _share_mode():
    import fp8_block_scaled_persistent_gb300 as fg
    assert fg.fp8_gemm_set_override(0, -1) == fg.FP8G_OK       # unsplit schedules
    assert fg.fp8_gemm_set_pair_mode(2) == fg.FP8G_OK
    yield
    fg.fp8_gemm_set_pair_mode(0)
    fg.fp8_gemm_set_override(0, 0)
    assert fg.fp8_gemm_get_device_error() == 0


def _ref(p):
    return oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, np.arange(p.M), threads=THREADS)


@pytest.mark.parametrize("M,N,K", [
    (1, 16, 128), (128, 256, 512), (129, 528, 640), (200, 512, 1024), (300, 1040, 256), (384, 784, 1536)])
def test_share_plain_shapes(M, N, K):
    p = wl.make_nt(M, N, K, seed=M * 11 + N)
    got, st, dst = gu.run(p, workspace=None)
    assert st == 0 and dst == 0
    check(got, _ref(p), f"share {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (130, 528, 1024)])
def test_share_exact_integers_bit_identical(M, N, K):
    p = wl.exact_integer_problem(M, N, K, seed=M + N + 2)
    got, st, dst = gu.run(p, workspace=None)
    assert st == 0 and dst == 0
    assert np.array_equal(got, _ref(p))


def test_share_contiguous_with_skipped_and_bad_blocks():
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    p = wl.make_contiguous([128, 256, 128, 384], 528, 512, seed=25)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    ref = oracle.gemm_grouped_contiguous_rows(p.A, p.SFA, p.B, p.SFB, p.m_indices, p.M, p.N, p.K,
                                              p.G, np.arange(p.M), threads=THREADS)
    check(got, ref, "share contiguous")
    layout = p.m_indices.copy()
    layout[0:128] = -1
    layout[128:256] = 11
    t = gu.dev_tensors(p)
    D = gu.new_d(p)
    assert gu.call(p, t, D, layout=torch.from_numpy(layout).cuda()) == 0
    assert fg.fp8_gemm_get_device_error() == fg.FP8G_ERR_BAD_GROUP
    got = gu.bits(D)
    assert (got[:256] == gu.SENTINEL).all()
    check(got[256:], ref[256:], "share contiguous skipped")


@pytest.mark.parametrize("counts,M_max", [([0, 1, 130, 200], 200), ([256, 255, 128, 17], 256)])
def test_share_masked_elementwise_and_untouched(counts, M_max):
    p = wl.make_masked(counts, M_max, 784, 512, seed=35)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    for g, c in enumerate(counts):
        assert (got[g, c:] == gu.SENTINEL).all(), f"group {g} rows beyond {c} were written"
        if c:
            ref = oracle.gemm_grouped_masked_rows(p.A, p.SFA, p.B, p.SFB, p.masked_m, p.G, M_max,
                                                  p.N, p.K, g, np.arange(c), threads=THREADS)
            check(got[g, :c], ref, f"share masked g{g}")


def test_share_repeatable_and_addend_unaffected():
    p = wl.make_nt(512, 1024, 2048, seed=7)
    a, _, _ = gu.run(p, workspace=None)
    b, _, _ = gu.run(p, workspace=None)
    assert np.array_equal(a, b)
    q = wl.make_nt_acc(256, 512, 1024, seed=8)
    got, st, dst = gu.run(q, workspace=None)
    assert st == 0 and dst == 0
    ref = oracle.gemm_nt_acc_rows(q.A, q.SFA, q.B, q.SFB, q.C, q.M, q.N, q.K, np.arange(q.M), threads=THREADS)
    check(got, ref, "addend with sharing requested")


@pytest.mark.parametrize("name", ["contiguous_g8_n4096_k7168", "dense_4096x7168x2048"])
def test_share_full_size_sampled_rows(name):
    p = wl.make(name)
    got, st, dst = gu.run(p, workspace=None)
    assert st == 0 and dst == 0
    if p.kind == "contiguous":
        starts = np.cumsum([0] + p.meta["group_rows"][:-1])
        ends = starts + np.array(p.meta["group_rows"]) - 1
        rows = gu.sample_rows(p.M, 16, seed=2, must=list(starts) + list(ends))
        ref = oracle.gemm_grouped_contiguous_rows(p.A, p.SFA, p.B, p.SFB, p.m_indices, p.M, p.N,
                                                  p.K, p.G, rows, threads=THREADS)
    else:
        rows = gu.sample_rows(p.M, 12, seed=1, must=(0, 127, 128, p.M - 1))
        ref = oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows, threads=THREADS)
    check(got[rows], ref, name)
