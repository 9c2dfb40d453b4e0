"""Pins for the oracle's scaled, batched form
D(l,m,n) = alpha * sum_k A(l,m,k) B(l,n,k) + beta * C(l,m,n).

The simple_gemm page's cuBLAS comparison (section 8.1) defines the alpha /
beta form; local_tile's extra modes (section 4) carry the batch coordinate.
Each check would fail on a plausible slip: alpha and beta swapped or one of
them dropped (distinct non-unit scalars, closed forms with identity
operands), B(k,n) for B(n,k) (identity A gives B transposed), a batch stride
applied to the wrong operand or not at all (float64 einsum over batches
with different strides, and a shared operand with stride 0), and the BLAS
conventions the page leaves implicit: alpha == 0 reads neither A nor B and
beta == 0 does not read C (NaN there must not reach D).
"""
import numpy as np
import pytest

import oracle

K_MAJOR, MN_MAJOR = oracle.MAJOR_K, oracle.MAJOR_MN


def h(x):
    return np.asarray(x, dtype=np.float16)


def rnd(shape, seed, lo=-1.0, hi=1.0):
    return h(np.random.default_rng(seed).uniform(lo, hi, shape))


def ints(shape, seed, lo=-3, hi=4):
    return h(np.random.default_rng(seed).integers(lo, hi, shape))


def batched_storage(mats, major, ld, stride, fill=np.nan):
    """Lay out L logical (rows, cols) matrices, matrix l starting at l*stride."""
    L, rows, cols = mats.shape
    per = (rows if major == K_MAJOR else cols) * ld
    assert stride == 0 or stride >= per
    size = (L - 1) * stride + per if L else 0
    st = np.full(max(size, 1), fill, np.float16)
    for l in range(L):
        blk = np.full((rows, ld) if major == K_MAJOR else (cols, ld), fill, np.float16)
        if major == K_MAJOR:
            blk[:, :cols] = mats[l]
        else:
            blk[:, :rows] = mats[l].T
        st[l * stride:l * stride + per] = blk.reshape(-1)
    return st


def run(alpha, A, B, beta, C, a_major=K_MAJOR, b_major=K_MAJOR, pad=0, gap=0, ldc_pad=0):
    L, M, K = A.shape
    N = B.shape[1]
    ldA = (K if a_major == K_MAJOR else M) + pad
    ldB = (K if b_major == K_MAJOR else N) + pad
    sA = ((M if a_major == K_MAJOR else K) * ldA + gap) if L > 1 else 0
    sB = ((N if b_major == K_MAJOR else K) * ldB + gap) if L > 1 else 0
    ldC = N + ldc_pad
    sC = (M * ldC + gap) if L > 1 else 0
    a = batched_storage(A, a_major, ldA, sA)
    b = batched_storage(B, b_major, ldB, sB)
    c = None if C is None else batched_storage(C, K_MAJOR, ldC, sC)
    return oracle.gemm_tn_general(M, N, K, alpha, a, ldA, a_major, b, ldB, b_major, beta, c,
                                  ldC, L, sA, sB, sC)


def expected(alpha, A, B, beta, C):
    """float64 einsum: an independent library route for the same definition."""
    A64, B64 = A.astype(np.float64), B.astype(np.float64)
    out = alpha * np.einsum("lmk,lnk->lmn", A64, B64)
    if beta != 0:
        out = out + beta * C.astype(np.float64)
    return out


@pytest.mark.parametrize("a_major", [K_MAJOR, MN_MAJOR])
@pytest.mark.parametrize("b_major", [K_MAJOR, MN_MAJOR])
def test_batched_integers_equal_einsum_exactly(a_major, b_major):
    L, M, N, K = 3, 13, 9, 21
    A, B, C = ints((L, M, K), 1), ints((L, N, K), 2), ints((L, M, N), 3)
    d, d16 = run(-2.0, A, B, 0.5, C, a_major, b_major, pad=5, gap=7, ldc_pad=3)
    ref = expected(-2.0, A, B, 0.5, C)
    assert np.array_equal(d, ref)
    assert np.array_equal(d16, ref.astype(np.float16).view(np.uint16))


def test_real_values_match_einsum():
    L, M, N, K = 4, 17, 23, 150
    A, B, C = rnd((L, M, K), 4), rnd((L, N, K), 5), rnd((L, M, N), 6)
    d, _ = run(0.75, A, B, -1.25, C, pad=2, gap=1)
    np.testing.assert_allclose(d, expected(0.75, A, B, -1.25, C), rtol=1e-12, atol=1e-12)


def test_identity_a_closed_form_separates_alpha_and_beta():
    # A = I: D = alpha * B^T + beta * C; alpha 3, beta -5 cannot be confused
    M = K = 12
    N = 7
    A = h(np.eye(M))[None]
    B, C = ints((1, N, K), 7), ints((1, M, N), 8)
    d, _ = run(3.0, A, B, -5.0, C)
    assert np.array_equal(d[0], 3.0 * B[0].T.astype(np.float64) - 5.0 * C[0])


def test_alpha_zero_reads_neither_a_nor_b():
    L, M, N, K = 2, 5, 6, 8
    A = h(np.full((L, M, K), np.nan))
    B = h(np.full((L, N, K), np.inf))
    C = ints((L, M, N), 9)
    d, _ = run(0.0, A, B, 2.0, C)
    assert np.array_equal(d, 2.0 * C.astype(np.float64))


def test_beta_zero_does_not_read_c():
    L, M, N, K = 2, 5, 6, 8
    A, B = ints((L, M, K), 10), ints((L, N, K), 11)
    C = h(np.full((L, M, N), np.nan))
    d, _ = run(1.5, A, B, 0.0, C)
    assert np.isfinite(d).all()
    assert np.array_equal(d, expected(1.5, A, B, 0.0, None))
    d2, _ = run(1.5, A, B, 0.0, None)
    assert np.array_equal(d, d2)


def test_empty_k_gives_beta_c():
    L, M, N = 2, 4, 3
    A, B = h(np.zeros((L, M, 0))), h(np.zeros((L, N, 0)))
    C = ints((L, M, N), 12)
    d, _ = run(7.0, A, B, -1.0, C)
    assert np.array_equal(d, -C.astype(np.float64))


def test_shared_operand_with_zero_batch_stride():
    L, M, N, K = 3, 6, 5, 9
    A = ints((L, M, K), 13)
    B1 = ints((1, N, K), 14)
    C = ints((L, M, N), 15)
    ldB = K
    b = batched_storage(B1, K_MAJOR, ldB, 0)
    sA = M * K
    a = batched_storage(A, K_MAJOR, K, sA)
    c = batched_storage(C, K_MAJOR, N, M * N)
    d, _ = oracle.gemm_tn_general(M, N, K, 1.0, a, K, K_MAJOR, b, ldB, K_MAJOR, 1.0, c, N, L,
                                  sA, 0, M * N)
    assert np.array_equal(d, expected(1.0, A, np.repeat(B1, L, axis=0), 1.0, C))


def test_unit_scalars_agree_with_the_unscaled_oracle():
    # alpha = beta = 1 is the definition D = C + A.B^T of the unscaled oracle
    M, N, K = 19, 11, 40
    A, B, C = ints((1, M, K), 16), ints((1, N, K), 17), ints((1, M, N), 18)
    d, d16 = run(1.0, A, B, 1.0, C, pad=1)
    d1, d161 = oracle.gemm_tn(M, N, K, A[0].reshape(-1), K, K_MAJOR, B[0].reshape(-1), K,
                              K_MAJOR, C[0].reshape(-1), N)
    assert np.array_equal(d[0], d1) and np.array_equal(d16[0], d161)


def test_rounding_is_once_from_the_fp64_value():
    # s = 2049 is not an fp16 value.  Scaled by 3 and rounded once it gives
    # 6147 -> 6148 (quantum 4); rounding s first would give 2048 * 3 = 6144.
    K = 2049
    A = h(np.ones((1, 1, K)))
    B = h(np.ones((1, 1, K)))
    d, d16 = run(3.0, A, B, 0.0, None)
    assert d[0, 0, 0] == 6147.0
    assert d16[0, 0, 0] == np.float16(6148.0).view(np.uint16)


def test_degenerate_sizes():
    A, B = h(np.zeros((0, 3, 4))), h(np.zeros((0, 2, 4)))
    d, d16 = run(1.0, A, B, 0.0, None)
    assert d.shape == (0, 3, 2)


def test_signed_zero_of_a_lone_term():
    # A zero sum scaled by a negative alpha with no C term is -0 (P alone);
    # adding a +0 C term (beta != 0) gives +0 by IEEE addition; beta * C alone
    # keeps -0 when alpha == 0; with both terms absent D is +0.
    M, N, K = 3, 4, 5
    A = h(np.zeros((1, M, K)))
    B = ints((1, N, K), 19)
    C = h(np.zeros((1, M, N)))
    neg0 = np.float16(-0.0).view(np.uint16)
    pos0 = np.float16(0.0).view(np.uint16)
    _, d16 = run(-1.0, A, B, 0.0, None)
    assert (d16 == neg0).all()
    _, d16 = run(-1.0, A, B, 1.0, C)
    assert (d16 == pos0).all()
    _, d16 = run(0.0, A, B, -2.0, C)
    assert (d16 == neg0).all()
    _, d16 = run(0.0, A, B, 0.0, None)
    assert (d16 == pos0).all()
    # K == 0 leaves the product term out even for a negative alpha
    _, d16 = run(-3.0, h(np.zeros((1, M, 0))), h(np.zeros((1, N, 0))), 0.0, None)
    assert (d16 == pos0).all()
