"""Pins for the oracle's GEMM  D(m,n) = C(m,n) + sum_k A(m,k) B(n,k).

Each check is chosen so that a plausible slip in the triple loop fails one of
them: closed forms with identity / permutation / all-ones operands (a dropped
C, a sign, B(k,n) instead of B(n,k), swapped m and n), K-major versus
MN-major storage of the same matrices and NaN in the leading-dimension slack
(a wrong view), exact integer brute force on the pages' 16x8x16 atom and
32x16x16 four-warp tile, and float64 BLAS matmul on random values.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

K_MAJOR, MN_MAJOR = oracle.MAJOR_K, oracle.MAJOR_MN


def h(x):
    return np.asarray(x, dtype=np.float16)


def storage(mat, major, ld, fill=np.nan):
    """Lay out the logical (rows, cols) fp16 matrix with the given major and ld."""
    rows, cols = mat.shape
    if major == K_MAJOR:
        st = np.full((rows, ld), fill, np.float16)
        st[:, :cols] = mat
    else:
        st = np.full((cols, ld), fill, np.float16)
        st[:, :rows] = mat.T
    return st.reshape(-1)


def run(A, B, C=None, a_major=K_MAJOR, b_major=K_MAJOR, pad=0, threads=None):
    M, K = A.shape
    N = B.shape[0]
    ldA = (K if a_major == K_MAJOR else M) + pad
    ldB = (K if b_major == K_MAJOR else N) + pad
    sa, sb = storage(A, a_major, ldA), storage(B, b_major, ldB)
    sc = None if C is None else np.ascontiguousarray(C, np.float16).reshape(-1)
    return oracle.gemm_tn(M, N, K, sa, ldA, a_major, sb, ldB, b_major, sc, N,
                          nthreads=threads)


def rnd(shape, seed, lo=-1.0, hi=1.0):
    return h(np.random.default_rng(seed).uniform(lo, hi, shape))


@pytest.mark.parametrize("a_major", [K_MAJOR, MN_MAJOR])
@pytest.mark.parametrize("b_major", [K_MAJOR, MN_MAJOR])
def test_identity_a_gives_c_plus_b_transposed(a_major, b_major):
    M = K = 24
    N = 17
    A = h(np.eye(M))
    B = rnd((N, K), 1)
    C = rnd((M, N), 2)
    d, _ = run(A, B, C, a_major, b_major, pad=3)
    # D(m,n) = C(m,n) + B(n,m): transposed, not B itself
    assert np.array_equal(d, C.astype(np.float64) + B.T.astype(np.float64))


@pytest.mark.parametrize("b_major", [K_MAJOR, MN_MAJOR])
def test_identity_b_gives_c_plus_a(b_major):
    M, N = 13, 20
    K = N
    A = rnd((M, K), 3)
    B = h(np.eye(N))
    C = rnd((M, N), 4)
    d, _ = run(A, B, C, K_MAJOR, b_major, pad=5)
    assert np.array_equal(d, C.astype(np.float64) + A.astype(np.float64))


def test_permutation_a():
    M = K = 32
    N = 9
    pi = np.random.default_rng(5).permutation(K)
    A = np.zeros((M, K), np.float16)
    A[np.arange(M), pi] = 1
    B = rnd((N, K), 6)
    C = rnd((M, N), 7)
    d, _ = run(A, B, C, MN_MAJOR, K_MAJOR)
    want = C.astype(np.float64) + B[:, pi].T.astype(np.float64)
    assert np.array_equal(d, want)


def test_negated_permutation_detects_sign():
    M = K = 8
    N = 8
    A = -h(np.eye(8))
    B = rnd((N, K), 8)
    C = h(np.zeros((M, N)))
    d, _ = run(A, B, C)
    assert np.array_equal(d, -B.T.astype(np.float64))


@pytest.mark.parametrize("K", [1, 16, 100, 2048])
def test_all_ones_gives_c_plus_k(K):
    M, N = 5, 7
    C = rnd((M, N), 9, -4, 4)
    d, d16 = run(h(np.ones((M, K))), h(np.ones((N, K))), C)
    assert np.array_equal(d, C.astype(np.float64) + K)
    assert np.array_equal(d16, (C.astype(np.float64) + K).astype(np.float16).view(np.uint16))


def test_no_c_means_zero_c():
    A, B = rnd((6, 10), 10), rnd((4, 10), 11)
    d0, _ = run(A, B, None)
    d1, _ = run(A, B, h(np.zeros((6, 4))))
    assert np.array_equal(d0, d1)


def _brute(A, B, C):
    """Exact rational triple loop (fractions), independent of the float path."""
    M, K = A.shape
    N = B.shape[0]
    out = np.empty((M, N), dtype=object)
    for m in range(M):
        for n in range(N):
            s = Fraction(float(C[m, n]))
            for k in range(K):
                s += Fraction(float(A[m, k])) * Fraction(float(B[n, k]))
            out[m, n] = s
    return out


@pytest.mark.parametrize("shape", [(16, 8, 16), (32, 16, 16)])
def test_brute_force_on_the_atom_and_four_warp_tile(shape):
    M, N, K = shape
    rng = np.random.default_rng(M * N * K)
    A = h(rng.integers(-2, 3, (M, K)))
    B = h(rng.integers(-2, 3, (N, K)))
    C = h(rng.integers(-4, 5, (M, N)))
    want = _brute(A, B, C)
    for am in (K_MAJOR, MN_MAJOR):
        for bm in (K_MAJOR, MN_MAJOR):
            d, d16 = run(A, B, C, am, bm, pad=8)
            assert all(Fraction(d[i, j]) == want[i, j] for i in range(M) for j in range(N))
            assert np.array_equal(d16.view(np.float16).astype(np.float64), d)


def test_brute_force_real_values_exact():
    # fp16 x fp16 products are exact in fp64; with K=16 the sum is too
    M, N, K = 16, 8, 16
    A, B, C = rnd((M, K), 20), rnd((N, K), 21), rnd((M, N), 22)
    d, _ = run(A, B, C)
    want = _brute(A, B, C)
    err = max(abs(Fraction(d[i, j]) - want[i, j]) for i in range(M) for j in range(N))
    assert err <= Fraction(1, 2 ** 40)


def test_matches_float64_blas_on_random_shapes():
    rng = np.random.default_rng(30)
    for M, N, K in [(1, 1, 1), (3, 5, 7), (64, 48, 80), (129, 65, 300), (200, 160, 512)]:
        A = h(rng.uniform(-1, 1, (M, K)))
        B = h(rng.uniform(-1, 1, (N, K)))
        C = h(rng.uniform(-1, 1, (M, N)))
        d, _ = run(A, B, C, MN_MAJOR, K_MAJOR, pad=4)
        ref = A.astype(np.float64) @ B.astype(np.float64).T + C.astype(np.float64)
        assert np.allclose(d, ref, rtol=1e-12, atol=1e-12)


def test_blas_route_agrees_with_triple_loop():
    rng = np.random.default_rng(31)
    M, N, K = 70, 50, 130
    A = h(rng.uniform(-1, 1, (M, K)))
    B = h(rng.uniform(-1, 1, (N, K)))
    C = h(rng.uniform(-1, 1, (M, N)))
    for am, bm in [(K_MAJOR, K_MAJOR), (MN_MAJOR, K_MAJOR), (K_MAJOR, MN_MAJOR)]:
        ldA = (K if am == K_MAJOR else M) + 2
        ldB = (K if bm == K_MAJOR else N) + 6
        sa, sb = storage(A, am, ldA), storage(B, bm, ldB)
        sc = C.reshape(-1)
        d, _ = oracle.gemm_tn(M, N, K, sa, ldA, am, sb, ldB, bm, sc, N)
        d2 = oracle.gemm_tn_blas(M, N, K, sa, ldA, am, sb, ldB, bm, sc, N)
        assert np.allclose(d, d2, rtol=1e-12, atol=1e-12)


def test_majorness_and_slack_do_not_change_the_result():
    rng = np.random.default_rng(40)
    M, N, K = 37, 29, 45
    A = h(rng.uniform(-1, 1, (M, K)))
    B = h(rng.uniform(-1, 1, (N, K)))
    C = h(rng.uniform(-1, 1, (M, N)))
    ref, _ = run(A, B, C)
    for am in (K_MAJOR, MN_MAJOR):
        for bm in (K_MAJOR, MN_MAJOR):
            for pad in (0, 1, 11):
                d, _ = run(A, B, C, am, bm, pad=pad)  # slack is NaN-poisoned
                assert np.array_equal(d, ref)


def test_thread_count_does_not_change_the_result():
    rng = np.random.default_rng(41)
    A = h(rng.uniform(-1, 1, (33, 200)))
    B = h(rng.uniform(-1, 1, (21, 200)))
    C = h(rng.uniform(-1, 1, (33, 21)))
    d1, _ = run(A, B, C, threads=1)
    d7, _ = run(A, B, C, threads=7)
    assert np.array_equal(d1, d7)


def test_sampled_equals_full():
    rng = np.random.default_rng(42)
    M, N, K = 40, 30, 70
    A = h(rng.uniform(-1, 1, (M, K)))
    B = h(rng.uniform(-1, 1, (N, K)))
    C = h(rng.uniform(-1, 1, (M, N)))
    d, d16 = run(A, B, C, MN_MAJOR, K_MAJOR)
    rows = rng.integers(0, M, 100)
    cols = rng.integers(0, N, 100)
    sa = storage(A, MN_MAJOR, M)
    sb = storage(B, K_MAJOR, K)
    s64, s16 = oracle.gemm_tn_sampled(M, N, K, sa, M, MN_MAJOR, sb, K, K_MAJOR,
                                      C.reshape(-1), N, rows, cols)
    assert np.array_equal(s64, d[rows, cols])
    assert np.array_equal(s16, d16[rows, cols])


def test_degenerate_sizes():
    A = h(np.zeros((3, 0)))
    B = h(np.zeros((4, 0)))
    C = rnd((3, 4), 50)
    d, d16 = oracle.gemm_tn(3, 4, 0, A.reshape(-1), 1, K_MAJOR, B.reshape(-1), 1, K_MAJOR,
                            C.reshape(-1), 4)
    assert np.array_equal(d, C.astype(np.float64))
    assert np.array_equal(d16, C.view(np.uint16))
    d, _ = oracle.gemm_tn(0, 4, 5, np.zeros(0, np.float16), 5, K_MAJOR,
                          rnd((4, 5), 51).reshape(-1), 5, K_MAJOR, None, 4)
    assert d.shape == (0, 4)


# ----------------------------------------------------------------------------
# general element strides ("CuTe Layout to Tensor Core", sections 1-2)

def test_strided_matches_gathered_copy_with_no_unit_stride():
    """A view with neither mode stride-1 equals the product of its gathered
    (numpy fancy-indexed) contiguous copy: a library gather, not the loop."""
    rng = np.random.default_rng(60)
    M, N, K = 21, 13, 37
    sAm, sAk, sBn, sBk, sCm, sCn = 3 * 2 * K + 5, 3, 2, 2 * N + 7, 1, M + 9
    XA = h(rng.uniform(-1, 1, (M - 1) * sAm + (K - 1) * sAk + 1))
    XB = h(rng.uniform(-1, 1, (N - 1) * sBn + (K - 1) * sBk + 1))
    XC = h(rng.uniform(-1, 1, (M - 1) * sCm + (N - 1) * sCn + 1))
    d, d16 = oracle.gemm_tn_strided(M, N, K, XA, sAm, sAk, XB, sBn, sBk, XC, sCm, sCn)
    a = XA[np.arange(M)[:, None] * sAm + np.arange(K)[None, :] * sAk]
    b = XB[np.arange(N)[:, None] * sBn + np.arange(K)[None, :] * sBk]
    c = XC[np.arange(M)[:, None] * sCm + np.arange(N)[None, :] * sCn]
    d_ref, _ = run(a, b, c)
    assert np.array_equal(d, d_ref)
    assert np.allclose(d, a.astype(np.float64) @ b.astype(np.float64).T + c.astype(np.float64),
                       rtol=1e-12, atol=1e-12)


def test_strided_equals_ld_major_form():
    rng = np.random.default_rng(61)
    M, N, K = 19, 23, 41
    A = h(rng.uniform(-1, 1, (M, K)))
    B = h(rng.uniform(-1, 1, (N, K)))
    C = h(rng.uniform(-1, 1, (M, N)))
    sa = storage(A, MN_MAJOR, M + 3)
    sb = storage(B, K_MAJOR, K + 5)
    d1, _ = oracle.gemm_tn(M, N, K, sa, M + 3, MN_MAJOR, sb, K + 5, K_MAJOR, C.reshape(-1), N)
    d2, _ = oracle.gemm_tn_strided(M, N, K, sa, 1, M + 3, sb, K + 5, 1, C.reshape(-1), N, 1)
    assert np.array_equal(d1, d2)


def test_broadcast_rows_closed_form():
    """Stride 0 along M repeats one row of A: every row of D is C's row plus
    the same vector B.a (computed here by BLAS)."""
    rng = np.random.default_rng(62)
    M, N, K = 7, 11, 29
    a_row = h(rng.uniform(-1, 1, K))
    B = h(rng.uniform(-1, 1, (N, K)))
    C = h(rng.uniform(-1, 1, (M, N)))
    d, _ = oracle.gemm_tn_strided(M, N, K, a_row, 0, 1, B.reshape(-1), K, 1, C.reshape(-1), N, 1)
    v = B.astype(np.float64) @ a_row.astype(np.float64)
    assert np.allclose(d, C.astype(np.float64) + v[None, :], rtol=1e-12, atol=1e-12)


def test_column_major_d_is_the_transpose_layout():
    rng = np.random.default_rng(63)
    M, N, K = 9, 6, 17
    A = h(rng.integers(-2, 3, (M, K)))
    B = h(rng.integers(-2, 3, (N, K)))
    C = h(rng.integers(-4, 5, (M, N)))
    CT = np.ascontiguousarray(C.T)  # C/D stored column-major: C(m,n) at n*M + m
    d, _ = oracle.gemm_tn_strided(M, N, K, A.reshape(-1), K, 1, B.reshape(-1), K, 1,
                                  CT.reshape(-1), 1, M)
    want = _brute(A, B, C)
    assert all(Fraction(d[i, j]) == want[i, j] for i in range(M) for j in range(N))
