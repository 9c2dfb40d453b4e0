"""GPU parity of the cluster-reduced skinny kernel: each 128-row tile of B
gets a cluster of 2, 4 or 8 CTAs that split its K loop, and the partial
sums are added through the cluster's shared memory in rank order, with C
added once (the make_tiled_mma page's K split across workers).  Every MMA
width it serves (up to 64), every cluster size, K a multiple of 64 (K-chunk
boxes) or not (2-D boxes), ragged N; integer values bit-exact against the
oracle, real values within the fp32-accumulation tolerance and
deterministic; the shapes it leaves to the contiguous split."""
import numpy as np
import pytest
import torch

import oracle
from dense_fp16_tensor_gb300 import binding as gb
from dense_fp16_tensor_gb300 import workloads as wl
from parity import check, np_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp16_tensor_gb300 as g
    g.build()
    gb.lib()


CLUSTER = "gemm_tn_skinny_cluster_kernel"


def run(M, N, K, dist="int1", cdist="int4", seed=0, alpha=1.0, beta=1.0, opts=None):
    ldA = (K + 7) // 8 * 8
    ldB = (K + 7) // 8 * 8 + 8           # rows of B off the 128-byte grid
    A_st = wl.operand(M, K, ldA, 0, dist if dist != "normal_k" else "normal", 40 + seed, K)
    B_st = wl.operand(N, K, ldB, 0, dist, 41 + seed, K)
    C_st = wl.operand(M, N, N, 0, cdist, 42 + seed)
    dev = torch.device("cuda")
    A, B, C = A_st.to(dev), B_st.to(dev), C_st.to(dev)
    D = torch.full((M, N), -3.0, dtype=torch.float16, device=dev)
    st = gb.gemm_tn_batched_ex(M, N, K, 1, alpha, A.data_ptr(), ldA, 0, 0, B.data_ptr(), ldB, 0, 0,
                               beta, C.data_ptr(), N, 0, D.data_ptr(), N, 0, gb.ACC_F32,
                               torch.cuda.current_stream().cuda_stream,
                               dict(path=gb.PATH_SKINNY, sync_check=1, **(opts or {})))
    assert st == gb.OK, gb.gemm_tn_status_string(st)
    kernels = gb.gemm_tn_last_kernels()
    torch.cuda.synchronize()
    d64, d16 = oracle.gemm_tn_general(M, N, K, alpha, np_bits(A_st), ldA, 0, np_bits(B_st), ldB, 0,
                                      beta, np_bits(C_st), N, 1, 0, 0, 0)
    return np_bits(D.cpu()), d64, d16, kernels


# (N, K): 64 tiles (pairs), 32 tiles (four), 8 tiles (eight); K a multiple
# of 64 or not
SHAPES = [(8192, 3000), (4000, 4096), (1000, 1088), (1000, 2500)]


@pytest.mark.parametrize("M", [1, 16, 17, 48, 64])
def test_cluster_skinny_integers_bit_exact(M):
    for N, K in SHAPES:
        got, d64, d16, k = run(M, N, K, seed=M)
        assert k == CLUSTER, k
        check(got.reshape(1, M, N), d64, d16, K, 0, True, f"cluster M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K", [(65, 1000, 3000), (128, 8192, 2048), (256, 1000, 3000),
                                   (16, 16384, 2048)])
def test_split_kernel_where_the_cluster_is_not_chosen(M, N, K):
    # MMA widths above 64, or one CTA per tile: the contiguous split
    got, d64, d16, k = run(M, N, K, seed=M + 3)
    assert k == "gemm_tn_skinny_kernel+gemm_tn_splitk_reduce_kernel", k
    check(got.reshape(1, M, N), d64, d16, K, 0, True, f"split M={M} N={N} K={K}")


def test_cluster_skinny_real_values_deterministic_and_scaled():
    for M, N, K in ((16, 8192, 8192), (64, 4000, 4096), (40, 1000, 3000)):
        a = run(M, N, K, dist="normal_k", cdist="u11", seed=7, alpha=-2.0, beta=0.5)
        b = run(M, N, K, dist="normal_k", cdist="u11", seed=7, alpha=-2.0, beta=0.5)
        assert a[3] == CLUSTER
        assert np.array_equal(a[0], b[0]), "rank-ordered reduction must be deterministic"
        check(a[0].reshape(1, M, N), a[1], a[2], K, 0, False, f"cluster real M={M}")
    # beta = 0: C is not read (NaN there cannot reach D)
    got, d64, d16, k = run(32, 2048, 4096, cdist="int4", seed=9, alpha=3.0, beta=0.0)
    check(got.reshape(1, 32, 2048), d64, d16, 4096, 0, True, "cluster beta 0")


def test_cluster_skinny_timeout_reports_and_recovers():
    M, N, K = 16, 1000, 2048  # eight CTAs per cluster: every peer must get through
    A = torch.zeros(M, K, dtype=torch.float16, device="cuda")
    B = torch.zeros(N, K, dtype=torch.float16, device="cuda")
    CD = torch.zeros(M, N, dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = gb.gemm_tn_ex(M, N, K, A.data_ptr(), K, 0, B.data_ptr(), K, 0, CD.data_ptr(), N, 0, s,
                       dict(path=gb.PATH_SKINNY, test_stall=1, timeout_ns=20_000_000,
                            sync_check=1))
    assert st == gb.ERR_DEVICE_TIMEOUT, gb.gemm_tn_status_string(st)
    assert gb.gemm_tn_check_device_error(s)[0] == gb.OK
    got, d64, d16, k = run(M, N, K, seed=11)
    assert k == CLUSTER
    check(got.reshape(1, M, N), d64, d16, K, 0, True, "cluster after timeout")
