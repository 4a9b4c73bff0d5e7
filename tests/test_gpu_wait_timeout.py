"""A bounded wait that runs out, on the GPU, without any fault.

The split-K schedule's reducing CTA waits for a counter that the other
contributors of its tile bump.  Here the counters are poisoned (a large
negative start) so that they never reach their target: the wait is a flag
that nothing sets.  With a short wait limit the kernel must record
FP8G_ERR_TIMEOUT, drain its copies and MMAs, free its tensor memory and
return; the context must stay usable, and the next call with a clean
workspace must give the right answer.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests import gpu_util as gu
from tests.tolerance import check

pytestmark = pytest.mark.gpu


def test_reducer_wait_runs_out_and_reports_timeout():
    import torch
    import fp8_block_scaled_persistent_gb300 as fg

    # 8 tiles of 128 columns, 64 K blocks: fewer tiles than SMs -> split-K
    p = wl.make_nt(128, 1024, 8192, seed=3, name="timeout_probe")
    t = gu.dev_tensors(p)
    ws = gu.workspace_for(p)
    assert ws is not None, "this shape is expected to use the split-K schedule"
    tiles = (p.N + 127) // 128
    counter_bytes = tiles * 8 * 4

    # the reference result, through the normal path
    D_ref = gu.new_d(p)
    assert gu.call(p, t, D_ref, workspace=ws) == fg.FP8G_OK
    assert fg.fp8_gemm_get_device_error() == fg.FP8G_OK

    try:
        assert fg.fp8_gemm_set_wait_timeout_ns(2_000_000) == fg.FP8G_OK     # 2 ms
        ws[:counter_bytes].fill_(0x80)          # every counter starts at -2139062144
        D = gu.new_d(p)
        assert gu.call(p, t, D, workspace=ws) == fg.FP8G_OK                # the launch itself is fine
        assert fg.fp8_gemm_get_device_error() == fg.FP8G_ERR_TIMEOUT
        # the sticky error was read and cleared; the context still works
        torch.cuda.synchronize()
    finally:
        fg.fp8_gemm_set_wait_timeout_ns(2_000_000_000)
        ws.zero_()
        torch.cuda.synchronize()

    D2 = gu.new_d(p)
    assert gu.call(p, t, D2, workspace=ws) == fg.FP8G_OK
    assert fg.fp8_gemm_get_device_error() == fg.FP8G_OK
    assert np.array_equal(gu.bits(D2), gu.bits(D_ref))
    rows = gu.sample_rows(p.M, 6, seed=5, must=(0, p.M - 1))
    ref = oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows, threads=8)
    check(gu.bits(D2)[rows], ref, "timeout_probe after recovery")
