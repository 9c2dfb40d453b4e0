"""gemm_tn_skinny_noalloc: the skinny path for callers that cannot let a
library allocate device memory for them (latency-sensitive loops in which
cudaMalloc/cudaFree would synchronise the device, processes whose allocator
already holds nearly all device memory).  Its split-K partial sums live in a
fixed array compiled into the library instead of a cudaMalloc'd workspace.

This file is collected last on purpose (pytest orders files by name), and it
must pass both on its own in a fresh process and after the other tests.

Every case makes two calls in a row through the C ABI, and the two calls
leave different contents in the shared array (other values, or a larger
problem before a smaller one), so that a partial sum the second call failed
to write would show up as the first call's stale value.  Each result is
checked against the CPU oracle -- bit for bit on integer-valued inputs,
within the fp32-accumulation tolerance of the parity tests on real values --
and against gemm_tn's skinny path with the same split over one CTA per SM on
the same inputs, which runs the same kernels and so must agree bit for bit.
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


def _inputs(M, N, K, seed, integer):
    if integer:  # every partial sum exact in fp32: the result is unique
        return (wl.operand(M, K, K, 0, "int1", seed), wl.operand(N, K, K, 0, "int1", seed + 1),
                wl.operand(M, N, N, 0, "int4", seed + 2))
    return (wl.operand(M, K, K, 0, "normal", seed, K), wl.operand(N, K, K, 0, "normal_k", seed + 1, K),
            wl.operand(M, N, N, 0, "u11", seed + 2))


def _call_and_check(M, N, K, seed, integer, what):
    dev = torch.device("cuda")
    s = torch.cuda.current_stream().cuda_stream
    A_st, B_st, C_st = _inputs(M, N, K, seed, integer)
    A, B = A_st.to(dev), B_st.to(dev)

    out = C_st.to(dev)
    st = gb.gemm_tn_skinny_noalloc(M, N, K, A.data_ptr(), K, 0, B.data_ptr(), K, 0,
                                   out.data_ptr(), N, 0, s)
    assert st == gb.OK, gb.gemm_tn_status_string(st)
    assert gb.gemm_tn_last_launch_count() == 2
    assert gb.gemm_tn_last_kernels() == "gemm_tn_skinny_kernel+gemm_tn_splitk_reduce_kernel"
    torch.cuda.synchronize()
    got = np_bits(out.cpu())

    d64, d16 = oracle.gemm_tn(M, N, K, np_bits(A_st), K, 0, np_bits(B_st), K, 0,
                              np_bits(C_st), N)
    check(got, d64, d16, K, 0, integer, what)

    # gemm_tn's skinny path with the contiguous split over one CTA per SM:
    # the same kernels and split, a pooled workspace
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ref = C_st.to(dev)
    st = gb.gemm_tn_ex(M, N, K, A.data_ptr(), K, 0, B.data_ptr(), K, 0, ref.data_ptr(), N, 0, s,
                       dict(path=gb.PATH_SKINNY, split_k=sms))
    assert st == gb.OK, gb.gemm_tn_status_string(st)
    assert gb.gemm_tn_last_kernels() == "gemm_tn_skinny_kernel+gemm_tn_splitk_reduce_kernel"
    torch.cuda.synchronize()
    assert np.array_equal(got, np_bits(ref.cpu())), f"{what}: differs from gemm_tn's skinny path"


@pytest.mark.parametrize("M,N,K", [(16, 16384, 16384), (40, 1000, 3000), (64, 4096, 1024)])
def test_noalloc_real_values_two_calls(M, N, K):
    # the second call draws other values, so stale partial sums would be wrong ones
    for call in range(2):
        _call_and_check(M, N, K, 600 + 10 * M + 5 * call, False, f"noalloc {M}x{N}x{K} call {call}")


def test_noalloc_integers_larger_problem_first():
    # M = 64 over N = 8192 fills ~9.6 MB of the array; the M = 16 call after it
    # uses far less, and must not pick up anything the first call left behind
    _call_and_check(64, 8192, 4096, 700, True, "noalloc integers M=64")
    _call_and_check(16, 2048, 8192, 710, True, "noalloc integers M=16 after M=64")


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
