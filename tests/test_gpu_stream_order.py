"""The kernel is launched as a programmatic dependent of the previous kernel
on the stream and waits for it before touching global memory: inputs that the
previous kernel writes must be the ones the GEMM reads, and a GEMM's output
must be complete for the kernel after it."""
import numpy as np
import pytest

import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_inputs_written_just_before_are_read():
    import torch
    import fp8_block_scaled_persistent_gb300 as fg

    p1 = wl.make_nt(512, 2048, 4096, seed=11, name="order_a")
    p2 = wl.make_nt(512, 2048, 4096, seed=12, name="order_b")
    t1, t2 = gu.dev_tensors(p1), gu.dev_tensors(p2)
    ref1, ref2 = gu.new_d(p1), gu.new_d(p2)
    assert gu.call(p1, t1, ref1) == fg.FP8G_OK
    assert gu.call(p2, t2, ref2) == fg.FP8G_OK
    torch.cuda.synchronize()

    work = {k: v.clone() for k, v in t1.items()}
    D = gu.new_d(p1)
    for i in range(20):
        src, ref = (t2, ref2) if i % 2 else (t1, ref1)
        # the copies are kernels (or copy engines) right before the GEMM
        for k in work:
            work[k].copy_(src[k])
        assert gu.call(p1, work, D) == fg.FP8G_OK
        # the GEMM's output feeds a kernel right after it
        got = D.clone()
        torch.cuda.synchronize()
        assert np.array_equal(gu.bits(got), gu.bits(ref)), f"iteration {i}"
    assert fg.fp8_gemm_get_device_error() == fg.FP8G_OK


def test_back_to_back_gemms_chain_through_device_memory():
    import torch
    import fp8_block_scaled_persistent_gb300 as fg

    # GEMM 2 reads as its B operand the bytes GEMM 1 wrote as D (a bf16 output
    # reinterpreted as e4m3 bytes: the values are meaningless, the order is not)
    p1 = wl.make_nt(256, 1024, 2048, seed=21, name="chain_1")
    t1 = gu.dev_tensors(p1)
    p2 = wl.make_nt(128, 256, 1024, seed=22, name="chain_2")
    t2 = gu.dev_tensors(p2)
    D1 = gu.new_d(p1)
    D2 = gu.new_d(p2)
    b2c = torch.empty((p2.N, p2.K), dtype=torch.uint8, device="cuda")
    t2b = dict(t2)
    t2b["B"] = b2c

    def run_chain():
        D1.fill_(0)
        assert gu.call(p1, t1, D1) == fg.FP8G_OK
        b2c.copy_(D1.view(torch.uint8).reshape(-1)[: p2.N * p2.K].view(p2.N, p2.K))
        assert gu.call(p2, t2b, D2) == fg.FP8G_OK
        torch.cuda.synchronize()
        return gu.bits(D2).copy()

    first = run_chain()
    for _ in range(5):
        assert np.array_equal(run_chain(), first)
    assert fg.fp8_gemm_get_device_error() == fg.FP8G_OK
