"""The bounds-checking build (libfp8gemm_debug.so, every kernel compiled with
FP8G_DEBUG_BOUNDS=1) runs the edge shapes of every path with no failed check.

In that build each kernel checks the invariants its memory accesses rely on
(a work unit starts inside the problem; group, K-block, split-slot and
counter indices are in range; every store stays inside D) and records
FP8G_ERR_BOUNDS, skipping the access, when one fails.  The cases below run
in a child process that loads the checking build (FP8G_LIBRARY=debug): the
plain GEMM at both tile widths with ragged M and N, split-K, the
narrow-slice kernel (both A box heights, more slices than SMs), the addend,
both grouped layouts with skipped blocks and short groups, the CTA-pair and
A-sharing modes, and the power-of-two-scale entry point.  Every result must
match the oracle and the device error must stay FP8G_OK.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import os, sys
import numpy as np
import torch
sys.path.insert(0, os.environ["FP8G_ROOT"])
import fp8_block_scaled_persistent_gb300 as fg
import oracle
import workloads as wl
from tests import gpu_util as gu
from tests.tolerance import check

lib = fg.library()
assert lib._name.endswith("libfp8gemm_debug.so"), lib._name
T = oracle.default_threads()
cases = 0

def run(p, what):
    global cases
    got, st, dst = gu.run(p)
    assert st == 0, (what, st)
    assert dst == 0, (what, fg.fp8_gemm_status_string(dst))
    rows = np.arange(p.M if p.kind != "masked" else 0, dtype=np.int32)
    if p.kind == "nt":
        check(got, oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows, threads=T), what)
    elif p.kind == "nt_acc":
        check(got, oracle.gemm_nt_acc_rows(p.A, p.SFA, p.B, p.SFB, p.C, p.M, p.N, p.K, rows, threads=T), what)
    elif p.kind == "nt_ue8m0":
        check(got, oracle.gemm_nt_ue8m0_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows, threads=T), what)
    elif p.kind == "contiguous":
        live = np.nonzero(p.m_indices >= 0)[0].astype(np.int32)
        ref = oracle.gemm_grouped_contiguous_rows(p.A, p.SFA, p.B, p.SFB, p.m_indices, p.M, p.N, p.K, p.G,
                                                  live, threads=T)
        check(got[live], ref, what)
    else:
        for g in range(p.G):
            c = int(p.masked_m[g])
            assert (got[g, c:] == gu.SENTINEL).all(), what
            if c:
                ref = oracle.gemm_grouped_masked_rows(p.A, p.SFA, p.B, p.SFB, p.masked_m, p.G, p.M, p.N, p.K,
                                                      g, np.arange(c, dtype=np.int32), threads=T)
                check(got[g, :c], ref, what)
    cases += 1

shapes = [(1, 16, 128), (63, 48, 256), (129, 272, 640), (300, 528, 512), (256, 400, 1024)]
for bn in (128, 256):
    fg.fp8_gemm_set_override(bn, -1)
    for M, N, K in shapes:
        run(wl.make_nt(M, N, K, seed=M + N), f"plain bn{bn} {M}x{N}x{K}")
fg.fp8_gemm_set_override(0, 0)
fg.fp8_gemm_set_narrow_mode(-1)
for M, N, K in [(64, 1024, 8192), (100, 384, 1536), (1, 128, 512)]:
    run(wl.make_nt(M, N, K, seed=K), f"split {M}x{N}x{K}")
fg.fp8_gemm_set_narrow_mode(1)
for M, N, K in [(1, 16, 512), (63, 336, 2560), (100, 400, 2688), (128, 64 * 160, 512)]:
    run(wl.make_nt(M, N, K, seed=K + 1), f"narrow {M}x{N}x{K}")
fg.fp8_gemm_set_narrow_mode(0)
run(wl.make_nt_acc(130, 272, 640, seed=3), "addend")
c = wl.make_contiguous([128, 256, 128, 384], 272, 512, seed=21)
c.m_indices[128:256] = -1
run(c, "contiguous")
run(wl.make_masked([0, 1, 130, 200], 200, 272, 512, seed=31), "masked")
for mode, bn in ((1, 128), (1, 256), (2, 256)):
    fg.fp8_gemm_set_pair_mode(mode)
    fg.fp8_gemm_set_override(bn, -1)
    run(wl.make_nt(300, 528, 512, seed=7), f"mode{mode} bn{bn} plain")
    run(wl.make_contiguous([128, 256, 128], 528, 256, seed=8), f"mode{mode} bn{bn} contiguous")
    run(wl.make_masked([5, 200, 0, 256], 256, 528, 256, seed=9), f"mode{mode} bn{bn} masked")
fg.fp8_gemm_set_pair_mode(0)
fg.fp8_gemm_set_override(0, 0)
for mode in (-1, 1):
    fg.fp8_gemm_set_pair_mode(mode)
    for M, N, K in [(63, 48, 256), (300, 528, 2304)]:
        run(wl.make_nt_ue8m0(M, N, K, seed=M), f"ue8m0 mode{mode} {M}x{N}x{K}")
fg.fp8_gemm_set_pair_mode(0)
torch.cuda.synchronize()
print("debug build ok", cases)
'''


def test_bounds_checking_build_runs_every_path_clean():
    env = dict(os.environ, FP8G_LIBRARY="debug", FP8G_ROOT=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True, env=env, cwd=ROOT,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "debug build ok" in r.stdout
