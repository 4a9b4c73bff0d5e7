"""The narrow-slice kernel (plain GEMM with M <= 128: one CTA per narrow
column slice and K part) against the oracle, through the C ABI.

fp8_gemm_set_narrow_mode(1) forces it wherever it applies (M <= 128, K >= 512).
It runs 96-column slices (which straddle the 128-column scale blocks) in two
K parts: the two CTAs of a slice are a cluster and trade halves of their fp32
partials over distributed shared memory (no workspace); A boxes of 64 rows
for M <= 64, 128 above.  The cases
cover both, ragged M, N not a multiple of the slice width, K block counts
that leave a partial last copy or an empty second K part, more work units
than SMs (CTAs take units in turn), exact integers (bit-identical), the
allocation-free entry point, a CUDA graph, and the full-size small-M
workloads under the automatic choice, on the split-K schedule as well.
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
def _narrow():
    import fp8_block_scaled_persistent_gb300 as fg
    fg.fp8_gemm_set_override(0, 0)
    assert fg.fp8_gemm_set_narrow_mode(1) == fg.FP8G_OK
    yield
    fg.fp8_gemm_set_narrow_mode(0)
    fg.fp8_gemm_set_override(0, 0)
    assert fg.fp8_gemm_get_device_error() == 0


def _ref(p):
    return oracle.gemm_nt(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K)


@pytest.mark.parametrize("M,N,K", [
    (1, 16, 512), (17, 64, 640), (63, 48, 1024), (64, 128, 512), (64, 336, 2560),
    (65, 144, 1536), (100, 400, 2688), (127, 1024, 768), (128, 256, 4096), (128, 80, 896)])
def test_narrow_shapes(M, N, K):
    p = wl.make_nt(M, N, K, seed=M * 5 + N + K)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    check(got, _ref(p), f"narrow {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(8, 64 * 200, 512), (100, 96 * 100, 1024)])
def test_narrow_more_units_than_sms(M, N, K):
    """200 work units: with one CTA per SM some CTAs take two in turn (with
    two K parts, both CTAs of a slice in the same round)."""
    p = wl.make_nt(M, N, K, seed=11)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    check(got, _ref(p), f"narrow {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (64, 192, 1664), (7, 272, 3968)])
def test_narrow_exact_integers_bit_identical(M, N, K):
    p = wl.exact_integer_problem(M, N, K, seed=M + N)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    assert np.array_equal(got, _ref(p))


def test_narrow_guard_bands_untouched():
    """Canaries before and after D stay bit-identical (ragged M, N % 64 != 0)."""
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    p = wl.make_nt(77, 208, 1024, seed=3)
    t = gu.dev_tensors(p)
    pad = 4096
    buf = torch.empty(pad + p.M * p.N + pad, dtype=torch.int16, device="cuda")
    buf.fill_(np.int16(np.uint16(gu.SENTINEL).view(np.int16)))
    D = buf[pad:pad + p.M * p.N].view(torch.bfloat16).view(p.M, p.N)
    assert gu.call(p, t, D) == 0
    assert fg.fp8_gemm_get_device_error() == 0
    host = buf.cpu().numpy().view(np.uint16)
    assert (host[:pad] == gu.SENTINEL).all() and (host[-pad:] == gu.SENTINEL).all()
    check(host[pad:-pad].reshape(p.M, p.N), _ref(p), "narrow guarded")


def test_narrow_noalloc_bit_identical():
    import fp8_block_scaled_persistent_gb300 as fg
    p = wl.make_nt(96, 1024, 4096, seed=12)
    t = gu.dev_tensors(p)
    D_ref = gu.new_d(p)
    # no workspace: the narrow-slice kernel needs none, so both calls run it
    assert gu.call(p, t, D_ref) == 0
    ref = gu.bits(D_ref)
    D = gu.new_d(p)
    assert fg.fp8_gemm_nt_noalloc(t["A"], t["SFA"], t["B"], t["SFB"], D, p.M, p.N, p.K) == 0
    assert fg.fp8_gemm_get_device_error() == 0
    assert np.array_equal(gu.bits(D), ref)
    rows = np.array([0, 1, 47, 95], dtype=np.int32)
    check(ref[rows], oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows, threads=THREADS),
          "narrow noalloc")


def test_narrow_graph_replay_bit_identical():
    """Both instantiations (64- and 128-row A boxes) captured into one CUDA
    graph on a side stream replay, twice, to the eager calls' bits."""
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    probs = [wl.make_nt(64, 512, 2048, seed=6), wl.make_nt(128, 320, 1536, seed=7)]
    tens = [gu.dev_tensors(p) for p in probs]
    wss = [None, None]      # the narrow-slice kernel needs no workspace
    side = torch.cuda.Stream()
    ref = [gu.new_d(p) for p in probs]
    with torch.cuda.stream(side):
        for p, t, D, ws in zip(probs, tens, ref, wss):
            assert gu.call(p, t, D, workspace=ws, stream=side) == 0
    side.synchronize()
    assert fg.fp8_gemm_get_device_error(side) == 0
    ref_bits = [gu.bits(D) for D in ref]
    outs = [gu.new_d(p) for p in probs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for p, t, D, ws in zip(probs, tens, outs, wss):
            assert gu.call(p, t, D, workspace=ws, stream=side) == 0
    for _ in range(2):
        for D in outs:
            D.view(torch.int16).fill_(np.int16(np.uint16(gu.SENTINEL).view(np.int16)))
        g.replay()
        torch.cuda.synchronize()
        assert fg.fp8_gemm_get_device_error() == 0
        for i, (D, r) in enumerate(zip(outs, ref_bits)):
            assert np.array_equal(gu.bits(D), r), f"replay output {i}"
    for p, r in zip(probs, ref_bits):
        check(r, _ref(p), f"narrow graph {p.M}x{p.N}x{p.K}")


def test_narrow_mode_off_and_overrides_keep_the_other_schedules():
    """Mode -1 and a forced split both take the split-K schedule (its
    workspace counters are used and left at zero); results agree with the
    narrow kernel's to within the tolerance."""
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    p = wl.make_nt(64, 1024, 8192, seed=13)
    narrow, st, _ = gu.run(p)
    assert st == 0
    ref = _ref(p)
    check(narrow, ref, "narrow")
    for setup in ((-1, None), (1, (128, 16))):
        fg.fp8_gemm_set_narrow_mode(setup[0])
        if setup[1]:
            fg.fp8_gemm_set_override(*setup[1])
        ws = gu.workspace_for(p) if not setup[1] else torch.zeros(
            fg.fp8_gemm_workspace_size_for(p.M, p.N, p.K, *setup[1]), dtype=torch.uint8, device="cuda")
        assert ws is not None
        got, st, dst = gu.run(p, workspace=ws)
        assert st == 0 and dst == 0
        check(got, ref, f"split, narrow mode {setup[0]}")
        fg.fp8_gemm_set_override(0, 0)
        fg.fp8_gemm_set_narrow_mode(1)


@pytest.mark.parametrize("mode", [0, -1], ids=["automatic", "split"])
@pytest.mark.parametrize("name", ["smallm_64x7168x16384", "smallm_128x7168x16384"])
def test_full_size_small_m(name, mode):
    """The small-M workloads as the benchmark runs them (automatic choice:
    the narrow kernel) and on the split-K schedule, sampled rows against the
    oracle, and a second run bit-identical."""
    import fp8_block_scaled_persistent_gb300 as fg
    fg.fp8_gemm_set_narrow_mode(mode)
    p = wl.make(name)
    got, st, dst = gu.run(p)
    assert st == 0 and dst == 0
    rows = gu.sample_rows(p.M, 10, seed=1, must=(0, 31, 32, p.M - 1))
    ref = oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows, threads=THREADS)
    check(got[rows], ref, f"{name} mode {mode}")
    again, _, _ = gu.run(p)
    assert np.array_equal(got, again), f"{name}: not deterministic"
