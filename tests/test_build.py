"""Build checks that need no GPU: the register budget of every kernel.

The kernel hands registers from its control warpgroup to its two epilogue
warpgroups with setmaxnreg.  The request must fit the block's launch
allocation (384 threads x the registers ptxas assigned at launch), or the
epilogue's increase would wait forever; and no kernel should spill.
"""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "fp8_block_scaled_persistent_gb300", "csrc")
KERNEL = os.path.join(CSRC, "gemm_kernel.cuh")
PAIR_KERNEL = os.path.join(CSRC, "gemm_kernel_pair.cuh")


def _const(name, path=KERNEL):
    m = re.search(rf"constexpr int {name} = (\d+);", open(path).read())
    assert m, name
    return int(m.group(1))


@pytest.fixture(scope="module")
def ptxas_report():
    from fp8_block_scaled_persistent_gb300 import build
    build.build(force=not os.path.exists(build.PTXAS_LOG))
    text = open(build.PTXAS_LOG).read()
    entries = re.split(r"Compiling entry function '", text)[1:]
    out = {}
    for e in entries:
        name = e.split("'")[0]
        regs = int(re.search(r"Used (\d+) registers", e).group(1))
        spill = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", e)
        out[name] = (regs, int(spill.group(1)), int(spill.group(2)))
    assert out, "no kernels in the ptxas report"
    return out


def test_register_reallocation_fits_the_launch_allocation(ptxas_report):
    threads, ctl, epi, launch = (_const("kNumThreads"), _const("kRegsCtl"), _const("kRegsEpi"),
                                 _const("kLaunchRegs"))
    assert threads == 384
    kernels = [n for n in ptxas_report if "fp8_gemm_kernel" in n]
    # plain and addend: 2 tile widths x split or not; grouped: 2 x 2; A-sharing clusters: plain and grouped
    assert len(kernels) == 15
    for name in kernels:
        regs = ptxas_report[name][0]
        assert regs == launch, f"{name}: launched with {regs} registers, expected {launch}"
        assert 128 * ctl + 256 * epi <= threads * regs, name
        assert ctl % 8 == 0 and epi % 8 == 0 and 24 <= ctl <= epi <= 256


def test_pair_kernel_register_split_fits(ptxas_report):
    threads, launch = _const("kNumThreads"), _const("kLaunchRegs")
    text = open(PAIR_KERNEL).read()
    ctl = re.search(r"kRegsCtl = BN == 128 \? (\d+) : (\d+);", text)
    epi = re.search(r"kRegsEpi = BN == 128 \? (\d+) : (\d+);", text)
    assert ctl and epi
    kernels = [n for n in ptxas_report if "fp8_gemm_pair_kernel" in n]
    assert len(kernels) == 8        # 2 tile widths x plain, addend, contiguous, masked
    for name in kernels:
        regs = ptxas_report[name][0]
        assert regs == launch, f"{name}: launched with {regs} registers, expected {launch}"
        i = 0 if "ILi128E" in name else 1
        c, e = int(ctl.group(1 + i)), int(epi.group(1 + i))
        assert 128 * c + 256 * e <= threads * regs, name
        assert c % 8 == 0 and e % 8 == 0 and 24 <= c <= e <= 256


def test_kernels_do_not_spill(ptxas_report):
    for name, (_, st, ld) in ptxas_report.items():
        assert st == 0 and ld == 0, f"{name}: {st} B spill stores, {ld} B spill loads"
