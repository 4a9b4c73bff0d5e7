"""The entry points can be captured in a CUDA graph and replayed.

No call reads the device-side group layouts on the host or synchronises, so a
sequence of calls -- split-K with its workspace, the plain schedule, the
masked layout, the accumulate variant and the allocation-free entry point --
records into one graph.  Every replay must give exactly the bits of the eager
calls (the split-K counters are back at zero after each launch, so a replay
starts from the same state), and rows the masked layout must leave untouched
stay untouched.
"""
import numpy as np
import pytest

import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_capture_and_replay_bit_identical():
    import torch
    import fp8_block_scaled_persistent_gb300 as fg

    probs = [
        wl.make_nt(128, 1024, 8192, seed=41),            # split-K schedule
        wl.make_nt(384, 768, 1024, seed=42),             # one CTA per tile
        wl.make_masked([5, 200, 0], 256, 256, 512, seed=43),
        wl.make_nt_acc(256, 512, 1024, seed=44),
    ]
    noalloc = wl.make_nt(64, 512, 4096, seed=45)         # split-K through the static scratch
    side = torch.cuda.Stream()
    tens = [gu.dev_tensors(p) for p in probs]
    wss = [gu.workspace_for(p) for p in probs]
    t_na = gu.dev_tensors(noalloc)

    def run_all(outs, D_na, stream):
        for p, t, ws, D in zip(probs, tens, wss, outs):
            assert gu.call(p, t, D, workspace=ws, stream=stream) == fg.FP8G_OK
        assert fg.fp8_gemm_nt_noalloc(t_na["A"], t_na["SFA"], t_na["B"], t_na["SFB"], D_na,
                                      noalloc.M, noalloc.N, noalloc.K, stream=stream) == fg.FP8G_OK

    # eager reference (also the first call of every kind on this device)
    ref = [gu.new_d(p) for p in probs]
    ref_na = gu.new_d(noalloc)
    with torch.cuda.stream(side):
        run_all(ref, ref_na, side)
    assert fg.fp8_gemm_get_device_error(side) == fg.FP8G_OK
    ref_bits = [gu.bits(D) for D in ref] + [gu.bits(ref_na)]

    outs = [gu.new_d(p) for p in probs]
    D_na = gu.new_d(noalloc)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        run_all(outs, D_na, side)
    for rep in range(3):
        for D in outs + [D_na]:
            D.view(torch.int16).fill_(np.int16(np.uint16(gu.SENTINEL).view(np.int16)))
        graph.replay()
        torch.cuda.synchronize()
        assert fg.fp8_gemm_get_device_error() == fg.FP8G_OK
        got = [gu.bits(D) for D in outs] + [gu.bits(D_na)]
        for i, (g, r) in enumerate(zip(got, ref_bits)):
            assert np.array_equal(g, r), f"replay {rep}: output {i} differs from the eager run"
    # the masked rows beyond each count are still the sentinel
    m = probs[2]
    for g in range(m.G):
        assert (got[2][g, int(m.masked_m[g]):] == gu.SENTINEL).all()
