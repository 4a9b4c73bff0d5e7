"""The C ABI from C itself: include/fp8gemm.h compiles as strict C99 and as
C++, and a C program linked against libfp8gemm.so calls the host-only entry
points and the argument checks (which return before any CUDA call, so no GPU
is needed)."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
PKG = os.path.join(ROOT, "fp8_block_scaled_persistent_gb300")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "fp8gemm.h"

#define CHECK(cond) do { if (!(cond)) { printf("failed: %s\n", #cond); return 1; } } while (0)

int main(void)
{
    /* a 16-byte aligned address that is never dereferenced */
    static float buf[64] __attribute__((aligned(16)));
    const void *p = buf;
    CHECK(fp8_gemm_version() == 10000);
    CHECK(fp8_gemm_sfa_ld(5) == 8 && fp8_gemm_sfa_ld(0) == 0);
    CHECK(strcmp(fp8_gemm_status_string(999), "unknown status") == 0);
    CHECK(fp8_gemm_status_string(FP8G_OK) != NULL);
    CHECK(fp8_gemm_nt(NULL, buf, p, buf, buf, 128, 256, 512, NULL, 0, NULL) == FP8G_ERR_INVALID_ARG);
    CHECK(fp8_gemm_nt(p, buf, p, buf, buf, 128, 256, 500, NULL, 0, NULL) == FP8G_ERR_UNSUPPORTED);
    CHECK(fp8_gemm_nt(p, buf, p, buf, buf, 0, 256, 512, NULL, 0, NULL) == FP8G_OK);
    CHECK(fp8_gemm_nt_accumulate(p, buf, p, buf, NULL, buf, 128, 256, 512, NULL, 0, NULL)
          == FP8G_ERR_INVALID_ARG);
    CHECK(fp8_gemm_grouped_contiguous(p, buf, p, buf, buf, NULL, 256, 256, 512, 2, NULL, 0, NULL)
          == FP8G_ERR_INVALID_ARG);
    CHECK(fp8_gemm_grouped_masked(p, buf, p, buf, buf, (const int *)p, 2, 256, 250, 512, NULL, 0, NULL)
          == FP8G_ERR_UNSUPPORTED);
    CHECK(fp8_gemm_nt_noalloc(p, buf, p, buf, buf, 128, 256, 500, NULL) == FP8G_ERR_UNSUPPORTED);
    CHECK(fp8_gemm_set_override(100, 0) == FP8G_ERR_INVALID_ARG);
    CHECK(fp8_gemm_set_override(0, 0) == FP8G_OK);
    CHECK(fp8_gemm_set_narrow_mode(2) == FP8G_ERR_INVALID_ARG);
    CHECK(fp8_gemm_set_narrow_mode(-1) == FP8G_OK);
    CHECK(fp8_gemm_set_narrow_mode(0) == FP8G_OK);
    CHECK(fp8_gemm_set_wait_timeout_ns(10) == FP8G_ERR_INVALID_ARG);
    CHECK(fp8_gemm_workspace_size_for(128, 256, 1024, 128, 10) == 256 + 2 * 10 * 128 * 128 * 4);
    printf("ok\n");
    return 0;
}
"""


@pytest.fixture(scope="module")
def lib_dir():
    from fp8_block_scaled_persistent_gb300 import build
    build.build()
    return PKG


@pytest.mark.parametrize("compiler,flags", [
    ("gcc", ["-x", "c", "-std=c99", "-pedantic-errors", "-Wall", "-Wextra", "-Werror"]),
    ("g++", ["-x", "c++", "-std=c++17", "-Wall", "-Wextra", "-Werror"]),
])
def test_header_compiles_links_and_validates(tmp_path, lib_dir, compiler, flags):
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    # the GNU alignment attribute is fine under -pedantic-errors in C99 mode
    subprocess.run([compiler, *flags, "-I", INCLUDE, str(src), "-o", str(exe),
                    "-L", lib_dir, "-lfp8gemm", "-Wl,-rpath," + lib_dir], check=True)
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
