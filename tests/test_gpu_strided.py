"""GPU parity of gemm_tn_strided (arbitrary element strides, copy-producer
kernel) against the oracle's strided triple loop, through the C ABI.

Views cover what the TMA kernels cannot take: odd leading dimensions,
operands offset by one element (2-byte alignment only), modes with no unit
stride, column-major C/D and a broadcast (stride-0) operand.  Integer inputs
are compared bit for bit; real inputs within the fp32 / fp16 accumulation
tolerances.
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


def extent(rows, cols, s_r, s_c):
    return (rows - 1) * s_r + (cols - 1) * s_c + 1


# (name, A strides, B strides, C strides, element offsets of A/B/C) as functions of M, N, K
VIEWS = {
    "odd_ld_k_major": lambda M, N, K: ((K + 3, 1), (K + 5, 1), (N + 1, 1), (0, 0, 0)),
    "odd_ld_mn_major": lambda M, N, K: ((1, M + 3), (1, N + 7), (N + 3, 1), (0, 0, 0)),
    "offset_by_one": lambda M, N, K: ((K, 1), (K, 1), (N, 1), (1, 3, 1)),
    "no_unit_stride": lambda M, N, K: ((2 * K + 1, 2), (3, 3 * N + 2), (2 * N + 2, 2), (0, 1, 0)),
    "column_major_d": lambda M, N, K: ((K, 1), (1, N), (1, M + 2), (0, 0, 0)),
    "broadcast_a_rows": lambda M, N, K: ((0, 1), (K + 1, 1), (N, 1), (0, 0, 0)),
}


def run_case(M, N, K, view, accum, dist_ab, dist_c, seed, route=gb.PATH_STRIDED_COPY):
    (sAm, sAk), (sBn, sBk), (sCm, sCn), (oA, oB, oC) = VIEWS[view](M, N, K)
    XA = wl.draw((oA + extent(M, K, sAm, sAk),), dist_ab, seed)
    XB = wl.draw((oB + extent(N, K, sBn, sBk),), dist_ab, seed + 1)
    XC = wl.draw((oC + extent(M, N, sCm, sCn),), dist_c, seed + 2)
    dev = torch.device("cuda")
    dA, dB, dC = XA.to(dev), XB.to(dev), XC.to(dev)
    s = torch.cuda.current_stream().cuda_stream
    st = gb.gemm_tn_strided_ex(M, N, K, dA.data_ptr() + 2 * oA, sAm, sAk, dB.data_ptr() + 2 * oB,
                               sBn, sBk, dC.data_ptr() + 2 * oC, sCm, sCn, accum, s,
                               {"path": route})
    assert st == gb.OK, gb.gemm_tn_status_string(st)
    kernels = gb.gemm_tn_last_kernels()
    if route == gb.PATH_STRIDED_COPY:
        assert kernels.startswith("gemm_tn_strided_kernel"), kernels
    elif route == gb.PATH_STRIDED_REPACK:
        assert "gemm_tn_strided_kernel" not in kernels and kernels
    torch.cuda.synchronize()
    out = np_bits(dC.cpu())
    d64, d16 = oracle.gemm_tn_strided(M, N, K, np_bits(XA)[oA:], sAm, sAk, np_bits(XB)[oB:],
                                      sBn, sBk, np_bits(XC)[oC:], sCm, sCn)
    got = out[oC + np.arange(M)[:, None] * sCm + np.arange(N)[None, :] * sCn]
    # elements of the C storage outside the view stay untouched
    mask = np.ones(out.size, bool)
    mask[(oC + np.arange(M)[:, None] * sCm + np.arange(N)[None, :] * sCn).reshape(-1)] = False
    assert np.array_equal(out[mask], np_bits(XC)[mask])
    return got, d64, d16


ROUTES = [gb.PATH_STRIDED_COPY, gb.PATH_STRIDED_REPACK]


@pytest.mark.parametrize("route", ROUTES)
@pytest.mark.parametrize("view", sorted(VIEWS))
@pytest.mark.parametrize("accum", [0, 1])
def test_strided_views_integer_bit_exact(view, accum, route):
    for i, (M, N, K) in enumerate([(1, 1, 1), (17, 129, 65), (200, 300, 130), (130, 260, 513)]):
        got, d64, d16 = run_case(M, N, K, view, accum, "int2", "int4", 500 + 10 * i, route)
        check(got, d64, d16, K, accum, True, f"{view} {M}x{N}x{K}")


@pytest.mark.parametrize("route", ROUTES)
@pytest.mark.parametrize("accum", [0, 1])
def test_strided_real_values_tolerance(accum, route):
    M, N, K = 384, 520, 1000
    for view in ("no_unit_stride", "odd_ld_mn_major"):
        got, d64, d16 = run_case(M, N, K, view, accum, "u11", "u11", 900, route)
        check(got, d64, d16, K, accum, False, f"{view} real")


def test_strided_auto_route_picks_repack_for_large_problems():
    M, N, K = 256, 512, 768
    got, d64, d16 = run_case(M, N, K, "odd_ld_k_major", 0, "int1", "int4", 950, gb.PATH_AUTO)
    assert gb.gemm_tn_last_kernels().startswith("repack2d_kernel+")
    check(got, d64, d16, K, 0, True, "auto route")


@pytest.mark.parametrize("view,variant", [("odd_ld_k_major", "<rows>"), ("offset_by_one", "<rows>"),
                                          ("odd_ld_mn_major", ""), ("no_unit_stride", "")])
def test_copy_route_variant(view, variant):
    # stride-1 K modes for both operands (any ld, any 2-byte offset) take the
    # row-class TMA variant; other views gather through the strides
    M, N, K = 300, 280, 700
    got, d64, d16 = run_case(M, N, K, view, 0, "int1", "int4", 1950)
    assert gb.gemm_tn_last_kernels() == "gemm_tn_strided_kernel" + variant
    check(got, d64, d16, K, 0, True, f"copy route {view}")


@pytest.mark.parametrize("view", ["odd_ld_k_major", "offset_by_one"])
@pytest.mark.parametrize("accum", [0, 1])
def test_copy_route_rows_k_multiple_of_64(view, accum):
    # the row-class variant shifts each row by its offset in the boxes; with K
    # a multiple of 64 the last K block's final elements come from the row
    # itself (no box past the end), so such K need their own cases, over
    # several 256 x 256 tiles and ragged M / N
    for i, (M, N, K) in enumerate([(520, 300, 256), (264, 520, 64), (300, 280, 1024)]):
        got, d64, d16 = run_case(M, N, K, view, accum, "int2", "int4", 2100 + 10 * i)
        assert gb.gemm_tn_last_kernels() == "gemm_tn_strided_kernel<rows>"
        check(got, d64, d16, K, accum, True, f"rows {view} {M}x{N}x{K}")


@pytest.mark.parametrize("accum", [0, 1])
def test_copy_route_rows_real_values(accum):
    # real values through the row-class variant (the class order of the
    # stage rows must not change what is summed)
    M, N, K = 384, 520, 1000
    for view in ("odd_ld_k_major", "offset_by_one"):
        got, d64, d16 = run_case(M, N, K, view, accum, "u11", "u11", 2300)
        assert gb.gemm_tn_last_kernels() == "gemm_tn_strided_kernel<rows>"
        check(got, d64, d16, K, accum, False, f"rows real {view}")


def test_copy_route_rows_smallest_views():
    # the row-class variant takes M, N >= 8: exactly one row per class, one K
    # element, and a single partial K block
    for i, (M, N, K) in enumerate([(8, 8, 1), (8, 300, 7), (300, 8, 64), (9, 17, 129)]):
        got, d64, d16 = run_case(M, N, K, "odd_ld_k_major", 0, "int2", "int4", 2400 + 10 * i)
        assert gb.gemm_tn_last_kernels() == "gemm_tn_strided_kernel<rows>"
        check(got, d64, d16, K, 0, True, f"rows small {M}x{N}x{K}")
