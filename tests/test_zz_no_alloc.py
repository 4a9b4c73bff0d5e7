"""fp8_gemm_nt_noalloc: the plain GEMM for callers that cannot call cudaMalloc.

Some callers cannot hand the library a workspace because they may not
allocate device memory at all: code that runs inside an allocator or
memory-pool callback, plug-ins whose host framework owns every device
allocation, loops that forbid allocation once started.  For them the split-K
schedule's scratch lives in a 24 MiB static device array inside the library.

These tests call the entry point through the C ABI and compare its output,
on two calls in a row, with fp8_gemm_nt given a workspace.  Both run the
same split-K schedule, whose reduction order is fixed, so the outputs must
be identical bit for bit; every shape below is one that splits, so the
static scratch is really used.  The file is named to be collected last, so a
run that stops at the first failure has already run every other test.
"""
import numpy as np
import pytest

import workloads as wl
from tests import gpu_util as gu
from tests.tolerance import check

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset():
    # the split-K schedule throughout (the scratch array is what these tests
    # exercise); the narrow-slice kernel's own no-alloc case is in
    # test_gpu_narrow.py
    import fp8_block_scaled_persistent_gb300 as fg
    fg.fp8_gemm_set_override(0, 0)
    fg.fp8_gemm_set_narrow_mode(-1)
    yield
    fg.fp8_gemm_set_override(0, 0)
    fg.fp8_gemm_set_narrow_mode(0)


@pytest.mark.parametrize("M,N,K", [(128, 7168, 16384), (64, 1024, 4096), (300, 512, 1024)])
def test_noalloc_matches_workspace_entry_point(M, N, K):
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    import oracle
    # the shape splits K, so the schedule goes through the scratch
    assert fg.fp8_gemm_workspace_size(fg.FP8G_KIND_NT, M, N, K, 1) > 0
    p = wl.make_nt(M, N, K, seed=M + N + K)
    t = gu.dev_tensors(p)

    # the existing entry point, with the workspace it asks for
    ws = gu.workspace_for(p)
    D_ref = gu.new_d(p)
    assert gu.call(p, t, D_ref, workspace=ws) == fg.FP8G_OK
    assert fg.fp8_gemm_get_device_error() == fg.FP8G_OK
    ref = gu.bits(D_ref)
    # and that output is right (sampled rows against the oracle)
    rows = gu.sample_rows(M, 8, seed=1, must=(0, M - 1))
    check(ref[rows], oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, M, N, K, rows,
                                         threads=oracle.default_threads()), f"{M}x{N}x{K}")

    # the allocation-free entry point, twice in a row (the static scratch keeps
    # the first call's contents when the second one starts)
    for call in range(2):
        D = gu.new_d(p)
        st = fg.fp8_gemm_nt_noalloc(t["A"], t["SFA"], t["B"], t["SFB"], D, M, N, K)
        assert st == fg.FP8G_OK, fg.fp8_gemm_status_string(st)
        assert fg.fp8_gemm_get_device_error() == fg.FP8G_OK
        got = gu.bits(D)
        assert np.array_equal(got, ref), f"noalloc call {call + 1} {M}x{N}x{K} differs from fp8_gemm_nt"
    torch.cuda.synchronize()


def test_noalloc_rejects_a_split_beyond_its_scratch():
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    p = wl.make_nt(128, 2048, 8192, seed=9)
    t = gu.dev_tensors(p)
    D = gu.new_d(p)
    # 152 CTAs with 256-column tiles need 2 x 152 slots of 128 KiB: more than
    # the 24 MiB array
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert fg.fp8_gemm_set_override(256, sms) == fg.FP8G_OK
    assert fg.fp8_gemm_workspace_size_for(p.M, p.N, p.K, 256, sms) > 24 << 20
    st = fg.fp8_gemm_nt_noalloc(t["A"], t["SFA"], t["B"], t["SFB"], D, p.M, p.N, p.K)
    assert st == fg.FP8G_ERR_SCRATCH_LIMIT
    assert "static" in fg.fp8_gemm_status_string(st)
    torch.cuda.synchronize()
    assert (gu.bits(D) == gu.SENTINEL).all()      # nothing was launched


def test_forced_split_beyond_the_sm_count_is_refused():
    """A split schedule needs all its CTAs resident at once; a forced count
    above the SM count is refused before anything is launched."""
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    p = wl.make_nt(128, 2048, 8192, seed=9)
    t = gu.dev_tensors(p)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert fg.fp8_gemm_set_override(128, sms + 1) == fg.FP8G_OK
    ws = torch.zeros(fg.fp8_gemm_workspace_size_for(p.M, p.N, p.K, 128, sms + 1), dtype=torch.uint8,
                     device="cuda")
    D = gu.new_d(p)
    assert gu.call(p, t, D, workspace=ws) == fg.FP8G_ERR_UNSUPPORTED
    assert fg.fp8_gemm_nt_noalloc(t["A"], t["SFA"], t["B"], t["SFB"], D, p.M, p.N, p.K) == \
        fg.FP8G_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert (gu.bits(D) == gu.SENTINEL).all()
