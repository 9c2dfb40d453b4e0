"""GPU parity of the stream-K split in the 256x256 tile kernel.

The last, partial wave of tiles is cut into K ranges shared by several CTAs;
every contributor writes a partial sum and the last one to arrive adds them
in a fixed order plus C (once).  Forced on shapes where many CTAs share a
tile, checked bit-exactly on integer inputs against the oracle and against
the unsplit kernel, and for determinism on real inputs.
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


def run(M, N, K, A_st, ldA, a_major, B_st, ldB, b_major, C_st, ldC, accum, stream_k):
    dev = torch.device("cuda")
    A, Bm, CD = A_st.to(dev), B_st.to(dev), C_st.to(dev)
    st = gb.gemm_tn_ex(M, N, K, A.data_ptr(), ldA, a_major, Bm.data_ptr(), ldB, b_major,
                       CD.data_ptr(), ldC, accum, torch.cuda.current_stream().cuda_stream,
                       {"path": gb.PATH_LARGE, "tile_kernel": gb.TILE_WIDE,
                        "stream_k": stream_k, "sync_check": 1})
    assert st == gb.OK, gb.gemm_tn_status_string(st)
    kernels = gb.gemm_tn_last_kernels()
    torch.cuda.synchronize()
    return np_bits(CD.cpu()), kernels


SHAPES = [  # (M, N, K): tiles of 256x256 vs 152 SMs, K blocks of 64
    (300, 520, 700),      # 6 tiles, 11 K blocks: ~12 contributors per tile
    (256, 256, 4096),     # 1 tile, 64 K blocks over every SM
    (1000, 1500, 1000),   # 24 tiles, ragged M/N/K
    (4000, 3000, 2500),   # 192 tiles: one full wave + 40 split tiles
]


@pytest.mark.parametrize("a_major,b_major", [(0, 0), (1, 0)])
@pytest.mark.parametrize("shape", SHAPES)
def test_stream_k_integer_bit_exact(shape, a_major, b_major):
    M, N, K = shape
    ldA = ((K if a_major == 0 else M) + 7) // 8 * 8
    ldB = ((K if b_major == 0 else N) + 7) // 8 * 8
    ldC = (N + 7) // 8 * 8
    A_st = wl.operand(M, K, ldA, a_major, "int1", 71)
    B_st = wl.operand(N, K, ldB, b_major, "int1", 72)
    C_st = wl.operand(M, N, ldC, 0, "int4", 73)  # NaN slack: never read, never written
    d_split, k_split = run(M, N, K, A_st, ldA, a_major, B_st, ldB, b_major, C_st, ldC, 0, 1)
    assert k_split == "memset+gemm_tn_wide_kernel"
    d_plain, k_plain = run(M, N, K, A_st, ldA, a_major, B_st, ldB, b_major, C_st, ldC, 0, -1)
    assert k_plain == "gemm_tn_wide_kernel"
    assert np.array_equal(d_split, d_plain)
    d64, d16 = oracle.gemm_tn(M, N, K, np_bits(A_st), ldA, a_major, np_bits(B_st), ldB, b_major,
                              np_bits(C_st), ldC)
    check(d_split[:M, :N], d64, d16, K, 0, True, f"stream-K {shape}")
    assert np.array_equal(d_split[:, N:], np_bits(C_st)[:, N:]), "slack written"


def test_stream_k_real_values_tolerance_and_determinism():
    M, N, K = 1000, 1504, 3000
    A_st = wl.operand(M, K, K, 0, "u11", 81)
    B_st = wl.operand(N, K, K, 0, "u11", 82)
    C_st = wl.operand(M, N, N, 0, "u11", 83)
    d1, _ = run(M, N, K, A_st, K, 0, B_st, K, 0, C_st, N, 0, 1)
    d2, _ = run(M, N, K, A_st, K, 0, B_st, K, 0, C_st, N, 0, 1)
    assert np.array_equal(d1, d2)  # fixed summation order: same bits every call
    d64, d16 = oracle.gemm_tn(M, N, K, np_bits(A_st), K, 0, np_bits(B_st), K, 0,
                              np_bits(C_st), N)
    check(d1, d64, d16, K, 0, False, "stream-K real")


def test_stream_k_not_used_for_fp16_accumulation():
    M, N, K = 300, 520, 704
    A_st = wl.operand(M, K, K, 0, "int1", 91)
    B_st = wl.operand(N, K, K, 0, "int1", 92)
    C_st = wl.operand(M, N, N, 0, "int4", 93)
    d, kernels = run(M, N, K, A_st, K, 0, B_st, K, 0, C_st, N, 1, 1)
    assert kernels == "gemm_tn_wide_kernel"
    d64, d16 = oracle.gemm_tn(M, N, K, np_bits(A_st), K, 0, np_bits(B_st), K, 0,
                              np_bits(C_st), N)
    check(d, d64, d16, K, 1, True, "fp16 accumulation unsplit")


def test_stream_k_timeout_path_reports_and_recovers():
    M, N, K = 300, 520, 704
    A_st = wl.operand(M, K, K, 0, "int1", 95)
    B_st = wl.operand(N, K, K, 0, "int1", 96)
    C_st = wl.operand(M, N, N, 0, "int4", 97)
    dev = torch.device("cuda")
    A, Bm, CD = A_st.to(dev), B_st.to(dev), C_st.to(dev)
    st = gb.gemm_tn_ex(M, N, K, A.data_ptr(), K, 0, Bm.data_ptr(), K, 0, CD.data_ptr(), N, 0,
                       torch.cuda.current_stream().cuda_stream,
                       {"path": gb.PATH_LARGE, "tile_kernel": gb.TILE_WIDE, "stream_k": 1,
                        "test_stall": 1, "timeout_ns": 20_000_000, "sync_check": 1})
    assert st == gb.ERR_DEVICE_TIMEOUT
    d, _ = run(M, N, K, A_st, K, 0, B_st, K, 0, C_st, N, 0, 1)
    d64, d16 = oracle.gemm_tn(M, N, K, np_bits(A_st), K, 0, np_bits(B_st), K, 0,
                              np_bits(C_st), N)
    check(d, d64, d16, K, 0, True, "after timeout")
