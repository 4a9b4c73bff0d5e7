"""The C ABI without a GPU: the library loads, exports every symbol that
include/fp8gemm.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import fp8_block_scaled_persistent_gb300 as fg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8gemm.h")


@pytest.fixture(scope="module")
def lib():
    from fp8_block_scaled_persistent_gb300 import build
    build.build()
    return fg.library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(fp8_gemm_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_entry_points():
    names = header_functions()
    for f in ("fp8_gemm_nt", "fp8_gemm_grouped_contiguous", "fp8_gemm_grouped_masked"):
        assert f in names
    assert sorted(names) == sorted(fg.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for s in range(0, 10):
        assert fg.fp8_gemm_status_string(s)
    assert fg.fp8_gemm_status_string(999) == "unknown status"


def test_sfa_ld(lib):
    assert [fg.fp8_gemm_sfa_ld(m) for m in (0, 1, 4, 5, 64, 65)] == [0, 4, 4, 8, 64, 68]


FAKE = 1 << 20   # a 16-byte aligned non-null address; never dereferenced


@pytest.mark.parametrize("args,status", [
    ((0, FAKE, FAKE, FAKE, FAKE, 128, 256, 512), fg.FP8G_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, -1, 256, 512), fg.FP8G_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 128, 256, 0), fg.FP8G_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 128, 256, 500), fg.FP8G_ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 128, 250, 512), fg.FP8G_ERR_UNSUPPORTED),
    ((FAKE + 8, FAKE, FAKE, FAKE, FAKE, 128, 256, 512), fg.FP8G_ERR_MISALIGNED),
    ((FAKE, FAKE, FAKE, FAKE, FAKE + 2, 128, 256, 512), fg.FP8G_ERR_MISALIGNED),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 0, 256, 512), fg.FP8G_OK),       # empty: no-op
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 128, 0, 512), fg.FP8G_OK),
])
def test_nt_validation(lib, args, status):
    assert fg.fp8_gemm_nt(*args, workspace=None, stream=0) == status


def test_nt_accumulate_validation(lib):
    a = fg.fp8_gemm_nt_accumulate
    M, N, K = 128, 256, 512
    assert a(FAKE, FAKE, FAKE, FAKE, 0, FAKE, M, N, K, stream=0) == fg.FP8G_ERR_INVALID_ARG      # no C
    assert a(FAKE, FAKE, FAKE, FAKE, FAKE + 4, FAKE, M, N, K, stream=0) == fg.FP8G_ERR_MISALIGNED
    assert a(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, M, N, 500, stream=0) == fg.FP8G_ERR_UNSUPPORTED
    c = FAKE + (1 << 24)
    # C [M][N] fp32 and D [M][N] bf16 overlapping, either way round
    assert a(FAKE, FAKE, FAKE, FAKE, c, c + 4 * M * N - 16, M, N, K, stream=0) == fg.FP8G_ERR_INVALID_ARG
    assert a(FAKE, FAKE, FAKE, FAKE, c, c - 2 * M * N + 16, M, N, K, stream=0) == fg.FP8G_ERR_INVALID_ARG
    assert a(FAKE, FAKE, FAKE, FAKE, c, c, 0, N, K, stream=0) == fg.FP8G_OK        # empty: no-op


def test_grouped_validation(lib):
    c = fg.fp8_gemm_grouped_contiguous
    assert c(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 256, 256, 512, 2, stream=0) == fg.FP8G_ERR_INVALID_ARG
    assert c(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 256, 256, 512, 0, stream=0) == fg.FP8G_ERR_INVALID_ARG
    assert c(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 200, 256, 512, 2, stream=0) == fg.FP8G_ERR_UNSUPPORTED
    assert c(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, 256, 256, 512, 2, stream=0) == fg.FP8G_ERR_MISALIGNED
    m = fg.fp8_gemm_grouped_masked
    assert m(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 2, 256, 256, 512, stream=0) == fg.FP8G_ERR_INVALID_ARG
    assert m(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, -1, 256, 256, 512, stream=0) == fg.FP8G_ERR_INVALID_ARG
    assert m(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 256, 256, 384 + 1, stream=0) == fg.FP8G_ERR_UNSUPPORTED
    assert m(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 0, 256, 512, stream=0) == fg.FP8G_OK


def test_overrides_and_timeout_validation(lib):
    assert fg.fp8_gemm_set_override(100, 0) == fg.FP8G_ERR_INVALID_ARG
    assert fg.fp8_gemm_set_override(256, 4) == fg.FP8G_OK
    assert fg.fp8_gemm_set_override(128, 4) == fg.FP8G_OK
    assert fg.fp8_gemm_set_override(0, 0) == fg.FP8G_OK
    for bad in (-2, 2, 64):
        assert fg.fp8_gemm_set_narrow_mode(bad) == fg.FP8G_ERR_INVALID_ARG
    for good in (-1, 1, 0):
        assert fg.fp8_gemm_set_narrow_mode(good) == fg.FP8G_OK
    assert fg.fp8_gemm_set_wait_timeout_ns(10) == fg.FP8G_ERR_INVALID_ARG
    assert fg.fp8_gemm_set_wait_timeout_ns(2_000_000_000) == fg.FP8G_OK


def test_workspace_sizes_host_only(lib):
    # small-M problems split K across SMs (128-column tiles), large ones do not
    assert fg.fp8_gemm_workspace_size(0, 128, 7168, 16384, 1) == \
        fg.fp8_gemm_workspace_size_for(128, 7168, 16384, 128, 152)
    assert fg.fp8_gemm_workspace_size(0, 4096, 7168, 2048, 1) == 0
    assert fg.fp8_gemm_workspace_size(1, 4096, 7168, 2048, 8) == 0
    n = fg.fp8_gemm_workspace_size_for(128, 256, 1024, 128, 10)
    assert n == 256 + 2 * 10 * 128 * 128 * 4
    assert fg.fp8_gemm_version() == 10000


@pytest.mark.parametrize("value,dense,smallm", [
    ("", 0, "auto"),
    ("128,8", "forced", "forced_small"),
    ("256,-1", 0, 0),
    ("bogus", 0, "auto"),
    ("100,4", 0, "auto"),
    ("128,8x", 0, "auto"),
])
def test_force_config_environment(lib, value, dense, smallm):
    """FP8G_FORCE_CONFIG sets the tuning overrides when the library loads;
    malformed values leave the automatic choice.  Observed through the
    workspace sizes the schedule choice implies (no GPU needed)."""
    import subprocess
    import sys
    code = ("import fp8_block_scaled_persistent_gb300 as fg; "
            "print(fg.fp8_gemm_workspace_size(0, 4096, 7168, 2048, 1), "
            "fg.fp8_gemm_workspace_size(0, 128, 7168, 16384, 1))")
    env = dict(os.environ, FP8G_FORCE_CONFIG=value, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                         cwd=ROOT, check=True).stdout.split()
    got_dense, got_small = int(out[0]), int(out[1])
    want = {
        0: 0,
        "auto": fg.fp8_gemm_workspace_size(0, 128, 7168, 16384, 1),
        "forced": fg.fp8_gemm_workspace_size_for(4096, 7168, 2048, 128, 8),
        "forced_small": fg.fp8_gemm_workspace_size_for(128, 7168, 16384, 128, 8),
    }
    assert got_dense == want[dense] and got_small == want[smallm]
