"""gemm_tn_skinny_noalloc: the skinny path for callers that cannot let a
library allocate device memory for them (latency-sensitive loops in which
cudaMalloc/cudaFree would synchronise the device, processes whose allocator
already holds nearly all device memory).  Its split-K partial sums live in a
fixed array compiled into the library instead of a cudaMalloc'd workspace.

This file is collected last on purpose (pytest orders files by name), and it
must pass both on its own in a fresh process and after the other tests.  Each
case calls the allocation-free entry point twice in a row through the C ABI
and compares both results with gemm_tn's on the same inputs, within the fp32
accumulation tolerance the parity tests use.
"""
import numpy as np
import pytest
import torch

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


def _inputs(M, N, K, seed):
    A_st = wl.operand(M, K, K, 0, "normal", seed, K)
    B_st = wl.operand(N, K, K, 0, "normal_k", seed + 1, K)
    C_st = wl.operand(M, N, N, 0, "u11", seed + 2)
    return A_st, B_st, C_st


@pytest.mark.parametrize("M,N,K", [(16, 16384, 16384), (40, 1000, 3000), (64, 4096, 1024)])
def test_noalloc_matches_gemm_tn_twice(M, N, K):
    dev = torch.device("cuda")
    A_st, B_st, C_st = _inputs(M, N, K, 600 + M)
    A, B = A_st.to(dev), B_st.to(dev)
    s = torch.cuda.current_stream().cuda_stream

    ref = C_st.to(dev)
    st = gb.gemm_tn(M, N, K, A.data_ptr(), K, 0, B.data_ptr(), K, 0, ref.data_ptr(), N, 0, s)
    assert st == gb.OK, gb.gemm_tn_status_string(st)
    torch.cuda.synchronize()
    ref64 = ref.cpu().double().numpy()

    for call in range(2):  # the second call reuses the array the first one left behind
        out = C_st.to(dev)
        st = gb.gemm_tn_skinny_noalloc(M, N, K, A.data_ptr(), K, 0, B.data_ptr(), K, 0,
                                       out.data_ptr(), N, 0, s)
        assert st == gb.OK, gb.gemm_tn_status_string(st)
        assert gb.gemm_tn_last_launch_count() == 2
        torch.cuda.synchronize()
        check(np_bits(out.cpu()), ref64, None, K, 0, False, f"noalloc call {call}")


def test_noalloc_rejects_what_it_cannot_serve():
    dev = torch.device("cuda")
    s = torch.cuda.current_stream().cuda_stream
    A = torch.zeros(64, 64, dtype=torch.float16, device=dev)
    B = torch.zeros(1 << 20, 64, dtype=torch.float16, device=dev)
    CD = torch.zeros(64, 1 << 20, dtype=torch.float16, device=dev)
    # M = 64, N = 2^20, K = 64: far more partial-sum scratch than the fixed array holds
    st = gb.gemm_tn_skinny_noalloc(64, 1 << 20, 64, A.data_ptr(), 64, 0, B.data_ptr(), 64, 0,
                                   CD.data_ptr(), 1 << 20, 0, s)
    assert st == gb.ERR_INVALID_ARG
    # outside the skinny path's restrictions
    assert gb.gemm_tn_skinny_noalloc(65, 64, 64, A.data_ptr(), 64, 0, B.data_ptr(), 64, 0,
                                     CD.data_ptr(), 64, 0, s) == gb.ERR_INVALID_ARG
    assert gb.gemm_tn_skinny_noalloc(16, 64, 64, A.data_ptr(), 64, 0, B.data_ptr(), 64, 0,
                                     CD.data_ptr(), 64, 1, s) == gb.ERR_INVALID_ARG
    assert gb.gemm_tn_last_launch_count() == 0
