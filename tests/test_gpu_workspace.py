"""Workspace exhaustion, injected on the host.

The test-only option ``test_fail_alloc`` makes every workspace request of
one call fail as an exhausted memory pool would (no device fault is
involved: the request is refused before anything is enqueued).  The
library's contract for that case:

  * a workspace the caller asked for -- the skinny path's contiguous split
    (an explicit split count), an explicit K split of the 128-row or
    CTA-pair kernel, the forced repack route of the strided entry point --
    makes the call return GEMM_TN_ERR_NO_MEMORY and leaves D untouched;
  * a workspace the library chose by itself -- an automatic K split,
    stream-K, the automatic repack route -- is dropped: the call runs the
    kernel that needs none and D matches the oracle bit for bit (integer
    inputs).
"""
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


FAIL = dict(test_fail_alloc=1)


def _problem(M, N, K, L=1, seed=0):
    """Integer-valued K-major operands (every partial sum exact), C in {-4..4}."""
    A_st = wl.batched_operand(L, M, K, K, 0, M * K, "int1", 1300 + seed, K)
    B_st = wl.batched_operand(L, N, K, K, 0, N * K, "int1", 1400 + seed, K)
    C_st = wl.batched_operand(L, M, N, N, 0, M * N, "int4", 1500 + seed)
    return A_st, B_st, C_st


def _run(M, N, K, L, opts, seed=0):
    """In-place batched call (alpha = beta = 1, D = C); returns status,
    kernels, D's bits and the operands' storage."""
    A_st, B_st, C_st = _problem(M, N, K, L, seed)
    dev = torch.device("cuda")
    A, B, CD = A_st.to(dev), B_st.to(dev), C_st.to(dev)
    st = gb.gemm_tn_batched_ex(M, N, K, L, 1.0, A.data_ptr(), K, M * K, 0, B.data_ptr(), K,
                               N * K, 0, 1.0, CD.data_ptr(), N, M * N, CD.data_ptr(), N, M * N,
                               gb.ACC_F32, torch.cuda.current_stream().cuda_stream, opts)
    kernels = gb.gemm_tn_last_kernels() if st == gb.OK else ""
    torch.cuda.synchronize()
    return st, kernels, np_bits(CD.cpu()), (A_st, B_st, C_st)


def _oracle(M, N, K, L, ops):
    A_st, B_st, C_st = ops
    return oracle.gemm_tn_general(M, N, K, 1.0, np_bits(A_st), K, 0, np_bits(B_st), K, 0, 1.0,
                                  np_bits(C_st), N, L, M * K, N * K, M * N)


@pytest.mark.parametrize("what,M,N,K,opts", [
    ("skinny split path", 16, 2048, 4096, dict(split_k=64)),
    ("explicit 128-row split", 512, 512, 4096, dict(path=gb.PATH_LARGE, tile_kernel=1,
                                                      tile_n=128, split_k=4)),
    ("explicit pair split", 512, 512, 4096, dict(path=gb.PATH_LARGE, tile_kernel=2,
                                                   split_k=2)),
])
def test_requested_workspace_fails_cleanly(what, M, N, K, opts):
    st, _, got, ops = _run(M, N, K, 1, dict(FAIL, **opts))
    assert st == gb.ERR_NO_MEMORY, f"{what}: {gb.gemm_tn_status_string(st)}"
    assert gb.gemm_tn_last_launch_count() == 0
    assert np.array_equal(got, np_bits(ops[2])), f"{what}: D changed"
    # the same call without the injected failure succeeds and is exact
    st, _, got, ops = _run(M, N, K, 1, opts)
    assert st == gb.OK
    d64, d16 = _oracle(M, N, K, 1, ops)
    check(got.reshape(1, M, N), d64, d16, K, 0, True, what)


@pytest.mark.parametrize("what,M,N,K,L,opts,split_kernels,plain_kernels", [
    # 16 tiles of 128 x 128 on 152 SMs, K = 8192: the library splits K by itself
    ("automatic 128-row split", 512, 512, 8192, 1, dict(path=gb.PATH_LARGE),
     "gemm_tn_large_kernel<128>+gemm_tn_tile_reduce_kernel", "gemm_tn_large_kernel<128>"),
    # 20 pair tiles with K = 8192: the library splits the pair tiles' K loops
    ("automatic pair split", 256, 256, 8192, 20, {},
     "gemm_tn_large2_kernel<deep>+gemm_tn_tile_reduce_kernel", "gemm_tn_large2_kernel<deep>"),
    # 192 tiles of 256 x 256: one full wave plus 40, split only with stream-K
    ("stream-K", 3072, 4096, 1024, 1, dict(path=gb.PATH_LARGE, tile_kernel=3, stream_k=1),
     "memset+gemm_tn_wide_kernel", "gemm_tn_wide_kernel"),
])
def test_chosen_workspace_is_dropped(what, M, N, K, L, opts, split_kernels, plain_kernels):
    st, k_split, got_split, ops = _run(M, N, K, L, opts, seed=1)
    assert st == gb.OK and k_split == split_kernels, (what, k_split)
    st, k_plain, got_plain, ops = _run(M, N, K, L, dict(FAIL, **opts), seed=1)
    assert st == gb.OK, f"{what}: {gb.gemm_tn_status_string(st)}"
    assert k_plain == plain_kernels, (what, k_plain)
    d64, d16 = _oracle(M, N, K, L, ops)
    check(got_plain.reshape(L, M, N), d64, d16, K, 0, True, f"{what}, no workspace")
    assert np.array_equal(got_plain, got_split)


def test_skinny_cluster_path_needs_no_workspace():
    # the library's skinny choice reduces the K split in a cluster: no pool
    st, k, got, ops = _run(16, 2048, 4096, 1, dict(FAIL), seed=3)
    assert st == gb.OK and k == "gemm_tn_skinny_cluster_kernel", (st, k)
    d64, d16 = _oracle(16, 2048, 4096, 1, ops)
    check(got.reshape(1, 16, 2048), d64, d16, 4096, 0, True, "skinny cluster, no pool")


def _strided(opts, M=256, N=320, K=264, seed=2):
    """Views TMA cannot read (leading dimensions K+1 and N+3)."""
    ldA, ldB, ldC = K + 1, K + 1, N + 3
    A_st = wl.draw((M * ldA,), "int1", 1600 + seed)
    B_st = wl.draw((N * ldB,), "int1", 1700 + seed)
    C_st = wl.draw((M * ldC,), "int4", 1800 + seed)
    dev = torch.device("cuda")
    A, B, CD = A_st.to(dev), B_st.to(dev), C_st.to(dev)
    st = gb.gemm_tn_strided_ex(M, N, K, A.data_ptr(), ldA, 1, B.data_ptr(), ldB, 1,
                               CD.data_ptr(), ldC, 1, gb.ACC_F32,
                               torch.cuda.current_stream().cuda_stream, opts)
    kernels = gb.gemm_tn_last_kernels() if st == gb.OK else ""
    torch.cuda.synchronize()
    got = np_bits(CD.cpu())
    d64, d16 = oracle.gemm_tn_strided(M, N, K, np_bits(A_st), ldA, 1, np_bits(B_st), ldB, 1,
                                      np_bits(C_st), ldC, 1)
    idx = np.arange(M)[:, None] * ldC + np.arange(N)[None, :]
    return st, kernels, got, got[idx], d64, d16, np_bits(C_st)


def test_strided_routes_without_workspace():
    # forced repack: the workspace is the caller's request
    st, _, got, _, _, _, c0 = _strided(dict(FAIL, path=gb.PATH_STRIDED_REPACK))
    assert st == gb.ERR_NO_MEMORY
    assert np.array_equal(got, c0), "D changed"
    # automatic route on a problem large enough for repacking: falls back to
    # the copy producer, which needs no workspace
    st, k, _, view, d64, d16, _ = _strided(FAIL)
    assert st == gb.OK and k.startswith("gemm_tn_strided_kernel"), k
    check(view, d64, d16, 264, 0, True, "strided fallback")
    st, k, _, view2, _, _, _ = _strided({})
    assert st == gb.OK and k.startswith("repack2d_kernel+"), k
    assert np.array_equal(view, view2)
