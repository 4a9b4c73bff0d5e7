"""Property-based pins of the oracle (CPU only; skipped where hypothesis is
not installed): for random small shapes, random E4M3 codes (NaN codes left
out) and random positive fp32 scales, the blocked oracle equals an
independent dequantise-then-matmul formulation in fp64, for the plain, the
addend and both grouped layouts."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from tests.test_oracle_pins import torch_decode_e4m3  # noqa: E402

SETTINGS = dict(max_examples=25, deadline=None, derandomize=True)


def _codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint16).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38          # NaN codes -> 1.0
    return c


def _scales(rng, shape):
    return (2.0 ** rng.uniform(-12, 12, size=shape)).astype(np.float32)


def _dequant(A, SFA, B, SFB, M, N, K):
    kb = K // 128
    a = torch_decode_e4m3(A) * np.repeat(SFA[:, :M].T.astype(np.float64), 128, axis=1)
    b = torch_decode_e4m3(B) * np.repeat(np.repeat(SFB.astype(np.float64), 128, axis=0)[:N], 128, axis=1)
    assert a.shape == (M, K) and b.shape == (N, K) and kb == SFA.shape[0]
    return a @ b.T


shapes = st.tuples(st.integers(1, 9), st.integers(1, 300), st.sampled_from([128, 256, 384]),
                   st.integers(0, 2 ** 31))


@settings(**SETTINGS)
@given(shapes)
def test_plain_and_addend_match_dequantised_matmul(shape):
    M, N, K, seed = shape
    rng = np.random.default_rng(seed)
    kb, nb, ld = K // 128, (N + 127) // 128, (M + 3) // 4 * 4
    A, B = _codes(rng, (M, K)), _codes(rng, (N, K))
    SFA = np.zeros((kb, ld), np.float32)
    SFA[:, :M] = _scales(rng, (kb, M))
    SFB = _scales(rng, (nb, kb))
    ref = _dequant(A, SFA, B, SFB, M, N, K)
    _, acc = oracle.gemm_nt(A, SFA, B, SFB, M, N, K, want_acc=True)
    np.testing.assert_allclose(acc, ref, rtol=1e-11, atol=1e-290)
    C = rng.standard_normal((M, N)).astype(np.float32)
    _, acc_c = oracle.gemm_nt_acc_rows(A, SFA, B, SFB, C, M, N, K, np.arange(M, dtype=np.int32),
                                       want_acc=True)
    np.testing.assert_allclose(acc_c, ref + C.astype(np.float64), rtol=1e-11,
                               atol=1e-11 * (np.abs(ref).max() + 1))


@settings(**SETTINGS)
@given(st.tuples(st.integers(1, 4), st.integers(1, 150), st.sampled_from([128, 256]),
                 st.integers(0, 2 ** 31)))
def test_grouped_layouts_match_dequantised_matmul(shape):
    G, N, K, seed = shape
    rng = np.random.default_rng(seed)
    kb, nb = K // 128, (N + 127) // 128
    B = _codes(rng, (G, N, K))
    SFB = _scales(rng, (G, nb, kb))
    # contiguous: 128-row blocks with random groups (some -1: skipped)
    blocks = int(rng.integers(1, 4))
    Mt = 128 * blocks
    A = _codes(rng, (Mt, K))
    SFA = _scales(rng, (kb, Mt))
    grp = rng.integers(-1, G, size=blocks)
    layout = np.repeat(grp, 128).astype(np.int32)
    rows = rng.choice(Mt, size=min(Mt, 12), replace=False).astype(np.int32)
    D = oracle.gemm_grouped_contiguous_rows(A, SFA, B, SFB, layout, Mt, N, K, G, rows,
                                            D_init=np.full((len(rows), N), 0x7FA5, np.uint16))
    for i, m in enumerate(rows):
        g = layout[m]
        if g < 0:
            assert (D[i] == 0x7FA5).all()
            continue
        ref = _dequant(A[m:m + 1], SFA[:, m:m + 1], B[g], SFB[g], 1, N, K)[0]
        want = np.array([oracle.f64_to_bf16(v) for v in ref], np.uint16)
        close = np.abs(np.array([oracle.bf16_to_f64(int(x)) for x in D[i]]) - ref) <= \
            np.abs(np.array([oracle.bf16_to_f64(int(x)) for x in want]) - ref) + 1e-12 * np.abs(ref)
        assert close.all()
    # masked: M_max rows per group, random counts
    M_max = int(rng.integers(1, 40))
    ld = (M_max + 3) // 4 * 4
    Am = _codes(rng, (G, M_max, K))
    SFAm = np.zeros((G, kb, ld), np.float32)
    SFAm[:, :, :M_max] = _scales(rng, (G, kb, M_max))
    counts = rng.integers(0, M_max + 1, size=G).astype(np.int32)
    for g in range(G):
        r = np.arange(M_max, dtype=np.int32)
        Dm = oracle.gemm_grouped_masked_rows(Am, SFAm, B, SFB, counts, G, M_max, N, K, g, r,
                                             D_init=np.full((M_max, N), 0x7FA5, np.uint16))
        c = int(counts[g])
        assert (Dm[c:] == 0x7FA5).all()
        if c:
            ref = _dequant(Am[g, :c], SFAm[g], B[g], SFB[g], c, N, K)
            want = np.array([[oracle.f64_to_bf16(v) for v in row] for row in ref], np.uint16)
            got = Dm[:c]
            gd = np.vectorize(lambda x: oracle.bf16_to_f64(int(x)))(got)
            wd = np.vectorize(lambda x: oracle.bf16_to_f64(int(x)))(want)
            assert (np.abs(gd - ref) <= np.abs(wd - ref) + 1e-12 * np.abs(ref)).all()
