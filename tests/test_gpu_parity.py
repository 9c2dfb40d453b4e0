"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Inputs come from dense_fp16_tensor_gb300.workloads (seeded, CPU-drawn, the
same bits on both sides).  The oracle (oracle/) computes the exact fp64
value; tests/parity.py holds the acceptance tolerances.
"""
import math

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
    yield


def run_gpu(M, N, K, A_st, ldA, a_major, B_st, ldB, b_major, C_st, ldC, accum, opts=None,
            guard_rows=0):
    """Copy storage to the device, run gemm_tn(_ex), return D storage (CPU) and the status.

    With guard_rows, CD is embedded between guard_rows rows of sentinel values
    above and below; the sentinels are checked to be untouched.
    """
    dev = torch.device("cuda")
    A = A_st.to(dev)
    Bm = B_st.to(dev)
    if guard_rows:
        sent = torch.full((guard_rows, ldC), -77.0, dtype=torch.float16)
        big = torch.cat([sent, C_st, sent]).to(dev)
        CD = big[guard_rows:guard_rows + C_st.shape[0]]
    else:
        CD = C_st.to(dev).contiguous()
    stream = torch.cuda.current_stream().cuda_stream
    args = (M, N, K, A.data_ptr(), ldA, a_major, Bm.data_ptr(), ldB, b_major,
            CD.data_ptr(), ldC, accum, stream)
    st = gb.gemm_tn_ex(*args, opts=opts) if opts else gb.gemm_tn(*args)
    torch.cuda.synchronize()
    if guard_rows:
        out = big.cpu()
        assert torch.equal(out[:guard_rows].view(torch.int16), sent.view(torch.int16))
        assert torch.equal(out[guard_rows + C_st.shape[0]:].view(torch.int16),
                           sent.view(torch.int16))
        return out[guard_rows:guard_rows + C_st.shape[0]], st
    return CD.cpu(), st


def oracle_full(w, A_st, B_st, C_st):
    return oracle.gemm_tn(w.M, w.N, w.K, np_bits(A_st), w.ldA, w.a_major,
                          np_bits(B_st), w.ldB, w.b_major, np_bits(C_st), w.ldC)


def result_view(D_st, M, N):
    return np_bits(D_st)[:M, :N]


def slack_untouched(D_st, C_st, N):
    if D_st.shape[1] > N:
        assert torch.equal(D_st[:, N:].view(torch.int16), C_st[:, N:].view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "tiny_int", "square1024", "ragged", "skinny"])
def test_workload_full_parity(name):
    w = wl.WORKLOADS[name]
    A_st, B_st, C_st = wl.make_inputs(w)
    D_st, st = run_gpu(w.M, w.N, w.K, A_st, w.ldA, w.a_major, B_st, w.ldB, w.b_major,
                       C_st, w.ldC, w.accum, guard_rows=3)
    assert st == gb.OK, gb.gemm_tn_status_string(st)
    assert gb.gemm_tn_check_device_error(torch.cuda.current_stream().cuda_stream)[0] == gb.OK
    d64, d16 = oracle_full(w, A_st, B_st, C_st)
    check(result_view(D_st, w.M, w.N), d64, d16, w.K, w.accum, w.exact, name)
    slack_untouched(D_st, C_st, w.N)


def test_large_8192_sampled_and_full():
    w = wl.WORKLOADS["large"]
    A_st, B_st, C_st = wl.make_inputs(w)
    D_st, st = run_gpu(w.M, w.N, w.K, A_st, w.ldA, w.a_major, B_st, w.ldB, w.b_major,
                       C_st, w.ldC, w.accum)
    assert st == gb.OK
    rows, cols = wl.sample_positions(w, 1024)
    s64, s16 = oracle.gemm_tn_sampled(w.M, w.N, w.K, np_bits(A_st), w.ldA, w.a_major,
                                      np_bits(B_st), w.ldB, w.b_major, np_bits(C_st), w.ldC,
                                      rows.numpy(), cols.numpy())
    d = np_bits(D_st)
    check(d[rows.numpy(), cols.numpy()], s64, s16, w.K, w.accum, False, "large sampled")
    full = oracle.gemm_tn_blas(w.M, w.N, w.K, np_bits(A_st), w.ldA, w.a_major,
                               np_bits(B_st), w.ldB, w.b_major, np_bits(C_st), w.ldC)
    check(d, full, None, w.K, w.accum, False, "large full")


SWEEP = [1, 15, 16, 17, 63, 127, 129, 200]


KERNEL_NAMES = {(1, 0): "gemm_tn_large_kernel<256>", (1, 128): "gemm_tn_large_kernel<128>",
                (1, 64): "gemm_tn_large_kernel<64>", (2, 0): "gemm_tn_large2_kernel",
                (3, 0): "gemm_tn_wide_kernel"}  # (shapes here are too small for stream-K)


@pytest.mark.parametrize("tile_kernel,tile_n", list(KERNEL_NAMES))
@pytest.mark.parametrize("accum", [0, 1])
@pytest.mark.parametrize("a_major,b_major", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_ragged_sweep(accum, a_major, b_major, tile_kernel, tile_n):
    """Tails in M, N and K across both majors and every tile kernel (single
    CTA 128x256, 128x128 and 128x64, CTA pair 256x256, single CTA 256x256),
    integer values: bit-exact."""
    rng = np.random.default_rng(100 + 10 * accum + 2 * a_major + b_major)
    cases = [(M, N, K) for M in (1, 17, 129, 200) for N in (1, 16, 129, 300)
             for K in (1, 15, 64, 129)]
    for M, N, K in cases:
        pad = 8
        ldA = ((K if a_major == 0 else M) + 7) // 8 * 8 + pad
        ldB = ((K if b_major == 0 else N) + 7) // 8 * 8 + pad
        ldC = (N + 7) // 8 * 8 + 8
        A_st = wl.operand(M, K, ldA, a_major, "int2", int(rng.integers(1 << 30)))
        B_st = wl.operand(N, K, ldB, b_major, "int2", int(rng.integers(1 << 30)))
        # NaN in C's slack: the kernels must neither read it nor write it
        C_st = wl.operand(M, N, ldC, 0, "int4", int(rng.integers(1 << 30)))
        D_st, st = run_gpu(M, N, K, A_st, ldA, a_major, B_st, ldB, b_major, C_st, ldC, accum,
                           opts={"path": gb.PATH_LARGE, "tile_kernel": tile_kernel,
                                 "tile_n": tile_n},
                           guard_rows=2)
        assert st == gb.OK, (M, N, K, gb.gemm_tn_status_string(st))
        assert gb.gemm_tn_last_kernels() == KERNEL_NAMES[(tile_kernel, tile_n)]
        d64, d16 = oracle.gemm_tn(M, N, K, np_bits(A_st), ldA, a_major, np_bits(B_st), ldB,
                                  b_major, np_bits(C_st), ldC)
        check(result_view(D_st, M, N), d64, d16, K, accum, True, f"{M}x{N}x{K}")
        slack_untouched(D_st, C_st, N)


@pytest.mark.parametrize("a_major,b_major", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_pair_deep_stages_k_tails(a_major, b_major):
    """The CTA pair's 128-deep stages (two 64-deep sub-blocks per operand,
    from K = 1024 on): K ending inside the first sub-block of the last stage
    (its second sub-block lies wholly past K), inside the second, and on
    stage and sub-block boundaries; ragged M and N; K-major leading
    dimensions multiples of 64.  Integer values: bit-exact.  Operands whose
    rows are off the 128-byte grid run both depths (128 by default, 64 on
    request)."""
    rng = np.random.default_rng(700 + 2 * a_major + b_major)
    M, N = 300, 520
    for K in (1024, 1030, 1088, 1100, 1152, 1190):
        ldA = (K + 63) // 64 * 64 if a_major == 0 else (M + 7) // 8 * 8 + 8
        ldB = (K + 63) // 64 * 64 if b_major == 0 else (N + 7) // 8 * 8 + 8
        A_st = wl.operand(M, K, ldA, a_major, "int1", int(rng.integers(1 << 30)))
        B_st = wl.operand(N, K, ldB, b_major, "int1", int(rng.integers(1 << 30)))
        C_st = wl.operand(M, N, N + 8, 0, "int4", int(rng.integers(1 << 30)))
        d64, d16 = oracle.gemm_tn(M, N, K, np_bits(A_st), ldA, a_major, np_bits(B_st), ldB,
                                  b_major, np_bits(C_st), N + 8)
        D_st, st = run_gpu(M, N, K, A_st, ldA, a_major, B_st, ldB, b_major, C_st, N + 8, 0,
                           opts={"path": gb.PATH_LARGE, "tile_kernel": 2}, guard_rows=2)
        assert st == gb.OK, (K, gb.gemm_tn_status_string(st))
        assert gb.gemm_tn_last_kernels() == "gemm_tn_large2_kernel<deep>"
        check(result_view(D_st, M, N), d64, d16, K, 0, True, f"deep K={K}")
        slack_untouched(D_st, C_st, N)
    # K-major operands with rows off the 128-byte grid
    K = 1100
    A_st = wl.operand(M, K, K + 4, 0, "int1", 5)
    B_st = wl.operand(N, K, K + 12, 0, "int1", 6)
    C_st = wl.operand(M, N, N, 0, "int4", 7)
    d64, d16 = oracle.gemm_tn(M, N, K, np_bits(A_st), K + 4, 0, np_bits(B_st), K + 12, 0,
                              np_bits(C_st), N)
    for k_stage, name in ((0, "gemm_tn_large2_kernel<deep>"), (64, "gemm_tn_large2_kernel")):
        D_st, st = run_gpu(M, N, K, A_st, K + 4, 0, B_st, K + 12, 0, C_st, N, 0,
                           opts={"path": gb.PATH_LARGE, "tile_kernel": 2, "k_stage": k_stage})
        assert st == gb.OK
        assert gb.gemm_tn_last_kernels() == name
        check(result_view(D_st, M, N), d64, d16, K, 0, True, f"off-grid rows K=1100 {name}")


@pytest.mark.parametrize("tile_n", [128, 160, 192, 224, 256])
@pytest.mark.parametrize("a_major,b_major", [(0, 0), (1, 0), (0, 1)])
def test_pair_tile_widths(tile_n, a_major, b_major):
    """The CTA-pair kernel at every tile width it runs (B's rows split
    bn / 2 per CTA, the last epilogue chunk 32 wide for odd multiples of 32):
    ragged M, N and K over several tiles, both accumulations, 64- and
    128-deep stages; integer values, bit-exact.  With an N-major B only the
    widths that are whole 64-element boxes per CTA run; the others are
    rejected."""
    M, N = 530, 3 * tile_n + 72
    for K, k_stage in ((300, 64), (1100, 128)):
        ldA = ((K if a_major == 0 else M) + 7) // 8 * 8 + 8
        ldB = (K + 63) // 64 * 64 if b_major == 0 else N + 8
        A_st = wl.operand(M, K, ldA, a_major, "int1", 900 + tile_n + K)
        B_st = wl.operand(N, K, ldB, b_major, "int1", 901 + tile_n + K)
        C_st = wl.operand(M, N, N + 8, 0, "int4", 902 + tile_n + K)
        d64, d16 = oracle.gemm_tn(M, N, K, np_bits(A_st), ldA, a_major, np_bits(B_st), ldB,
                                  b_major, np_bits(C_st), N + 8)
        for accum in (0, 1):
            opts = {"path": gb.PATH_LARGE, "tile_kernel": 2, "tile_n": tile_n,
                    "k_stage": k_stage}
            D_st, st = run_gpu(M, N, K, A_st, ldA, a_major, B_st, ldB, b_major, C_st, N + 8,
                               accum, opts=opts, guard_rows=2)
            if b_major == 1 and tile_n % 128 != 0:
                assert st == gb.ERR_INVALID_ARG
                continue
            assert st == gb.OK, gb.gemm_tn_status_string(st)
            assert gb.gemm_tn_last_kernels() == ("gemm_tn_large2_kernel<deep>" if k_stage == 128
                                                 else "gemm_tn_large2_kernel")
            check(result_view(D_st, M, N), d64, d16, K, accum, True,
                  f"pair bn={tile_n} K={K} acc={accum}")
            slack_untouched(D_st, C_st, N)


def test_pair_tile_width_of_the_ragged_workload_real_values():
    """The ragged workload on 256 x 224 pair tiles (the width the library
    picks for it) against the 256-wide ones and the oracle's tolerance."""
    w = wl.WORKLOADS["ragged"]
    A_st, B_st, C_st = wl.make_inputs(w)
    d64, d16 = oracle_full(w, A_st, B_st, C_st)
    for tile_n in (224, 256):
        D_st, st = run_gpu(w.M, w.N, w.K, A_st, w.ldA, w.a_major, B_st, w.ldB, w.b_major,
                           C_st, w.ldC, w.accum,
                           opts={"path": gb.PATH_LARGE, "tile_kernel": 2, "tile_n": tile_n})
        assert st == gb.OK
        check(result_view(D_st, w.M, w.N), d64, d16, w.K, w.accum, False, f"ragged bn={tile_n}")


@pytest.mark.parametrize("tile_n,tile_kernel", [(64, 1), (128, 1), (256, 1), (256, 2),
                                                 (256, 3)])
def test_large_path_real_values_every_tile_kernel(tile_n, tile_kernel):
    M, N, K = 300, 520, 700
    ldA, ldB = K + 12, N + 8
    A_st = wl.operand(M, K, ldA, 0, "u11", 11)
    B_st = wl.operand(N, K, ldB, 1, "u11", 12)  # B MN-major
    C_st = wl.operand(M, N, N, 0, "u11", 13)
    for accum in (0, 1):
        D_st, st = run_gpu(M, N, K, A_st, ldA, 0, B_st, ldB, 1, C_st, N, accum,
                           opts={"path": gb.PATH_LARGE, "tile_n": tile_n,
                                 "tile_kernel": tile_kernel})
        assert st == gb.OK, gb.gemm_tn_status_string(st)
        d64, d16 = oracle.gemm_tn(M, N, K, np_bits(A_st), ldA, 0, np_bits(B_st), ldB, 1,
                                  np_bits(C_st), N)
        check(result_view(D_st, M, N), d64, d16, K, accum, False, f"tile_n={tile_n}")


@pytest.mark.parametrize("M", [1, 16, 17, 40, 64, 65, 96, 100, 128, 129, 192, 200, 256])
def test_skinny_path_shapes_and_splits(M):
    """Skinny path: every M bucket, ragged N and K, several split counts;
    integer values so that every split must give the same bits (C once)."""
    N, K = 1000, 3000
    A_st = wl.operand(M, K, K, 0, "int1", 21 + M)
    B_st = wl.operand(N, K, K + 8, 0, "int1", 22 + M)
    C_st = wl.operand(M, N, N, 0, "int4", 23 + M)
    d64, d16 = oracle.gemm_tn(M, N, K, np_bits(A_st), K, 0, np_bits(B_st), K + 8, 0,
                              np_bits(C_st), N)
    outs = []
    for split in (1, 7, 64, 0):
        D_st, st = run_gpu(M, N, K, A_st, K, 0, B_st, K + 8, 0, C_st, N, 0,
                           opts={"path": gb.PATH_SKINNY, "split_k": split})
        assert st == gb.OK
        if split or M > 64:  # the contiguous split and its reduction kernel
            assert gb.gemm_tn_last_launch_count() == 2
            assert gb.gemm_tn_last_kernels() == "gemm_tn_skinny_kernel+gemm_tn_splitk_reduce_kernel"
        else:  # the library's choice up to M = 64: K split inside a cluster per tile
            assert gb.gemm_tn_last_launch_count() == 1
            assert gb.gemm_tn_last_kernels() == "gemm_tn_skinny_cluster_kernel"
        check(result_view(D_st, M, N), d64, d16, K, 0, True, f"skinny M={M} split={split}")
        outs.append(D_st)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_skinny_real_values_tolerance():
    w = wl.WORKLOADS["skinny"]
    M, N, K = 16, 2048, 16384
    A_st = wl.operand(M, K, K, 0, "normal", 31, K)
    B_st = wl.operand(N, K, K, 0, "normal_k", 32, K)
    C_st = wl.operand(M, N, N, 0, "u11", 33)
    D_st, st = run_gpu(M, N, K, A_st, K, 0, B_st, K, 0, C_st, N, 0)
    assert st == gb.OK
    d64, d16 = oracle.gemm_tn(M, N, K, np_bits(A_st), K, 0, np_bits(B_st), K, 0,
                              np_bits(C_st), N)
    check(result_view(D_st, M, N), d64, d16, K, 0, False, "skinny real")


def test_degenerate_calls_launch_nothing():
    dev = torch.device("cuda")
    CD = torch.randn(8, 8, device=dev).half()
    before = CD.clone()
    A = torch.zeros(8, 8, device=dev, dtype=torch.float16)
    s = torch.cuda.current_stream().cuda_stream
    # K = 0: D = C
    assert gb.gemm_tn(8, 8, 0, A.data_ptr(), 8, 0, A.data_ptr(), 8, 0, CD.data_ptr(), 8, 0, s) == 0
    assert gb.gemm_tn_last_launch_count() == 0
    # M = 0 / N = 0: no-op
    assert gb.gemm_tn(0, 8, 8, A.data_ptr(), 8, 0, A.data_ptr(), 8, 0, CD.data_ptr(), 8, 0, s) == 0
    assert gb.gemm_tn(8, 0, 8, A.data_ptr(), 8, 0, A.data_ptr(), 8, 0, CD.data_ptr(), 8, 0, s) == 0
    torch.cuda.synchronize()
    assert torch.equal(CD, before)


def test_bounded_wait_expires_and_reports_instead_of_hanging():
    """A producer that withholds one stage makes the consumer's bounded wait
    run out: the call reports GEMM_TN_ERR_DEVICE_TIMEOUT, the kernel frees its
    resources, and the next call on the same context is correct."""
    M, N, K = 256, 256, 512
    A_st = wl.operand(M, K, K, 0, "int1", 41)
    B_st = wl.operand(N, K, K, 0, "int1", 42)
    C_st = wl.operand(M, N, N, 0, "int4", 43)
    for path, m, pair in ((gb.PATH_LARGE, M, 1), (gb.PATH_LARGE, M, 2), (gb.PATH_LARGE, M, 3),
                          (gb.PATH_SKINNY, 16, 0)):
        _, st = run_gpu(m, N, K, A_st, K, 0, B_st, K, 0, C_st, N, 0,
                        opts={"path": path, "test_stall": 1, "timeout_ns": 20_000_000,
                              "sync_check": 1, "tile_kernel": pair})
        assert st == gb.ERR_DEVICE_TIMEOUT, gb.gemm_tn_status_string(st)
        assert gb.gemm_tn_check_device_error(torch.cuda.current_stream().cuda_stream)[0] == gb.OK
        D_st, st = run_gpu(m, N, K, A_st, K, 0, B_st, K, 0, C_st, N, 0,
                           opts={"path": path, "sync_check": 1, "tile_kernel": pair})
        assert st == gb.OK
        d64, d16 = oracle.gemm_tn(m, N, K, np_bits(A_st), K, 0, np_bits(B_st), K, 0,
                                  np_bits(C_st), N)
        check(result_view(D_st, m, N), d64, d16, K, 0, True, "after timeout")


def test_tensor_front_end_matches_oracle():
    import dense_fp16_tensor_gb300 as g
    dev = torch.device("cuda")
    M, N, K = 136, 96, 200
    A_st = wl.draw((K, M), "int2", 51)               # stored K rows of M: M-major
    B_st = wl.draw((N, K), "int2", 52)               # K-major
    C_st = wl.draw((M, N), "int4", 53)
    A = A_st.to(dev).t()                             # (M,K):(1,M) view
    D = C_st.to(dev)
    g.gemm(A, B_st.to(dev), D, accum="f32")
    torch.cuda.synchronize()
    d64, d16 = oracle.gemm_tn(M, N, K, np_bits(A_st), M, 1, np_bits(B_st), K, 0,
                              np_bits(C_st), N)
    check(np_bits(D.cpu()), d64, d16, K, 0, True, "tensor front end")


def test_skinny_calls_on_two_streams_do_not_share_scratch():
    """Two skinny problems enqueued on two streams without ordering between
    them: each must still match the oracle (each call has its own workspace)."""
    dev = torch.device("cuda")
    M, N, K = 16, 4096, 8192
    probs = []
    for seed in (71, 81):
        A_st = wl.operand(M, K, K, 0, "int1", seed)
        B_st = wl.operand(N, K, K, 0, "int1", seed + 1)
        C_st = wl.operand(M, N, N, 0, "int4", seed + 2)
        probs.append((A_st, B_st, C_st, A_st.to(dev), B_st.to(dev), C_st.to(dev)))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for rep in range(3):
        outs = []
        for (A_st, B_st, C_st, A, Bm, C), s in zip(probs, streams):
            CD = C.clone()
            torch.cuda.synchronize()
            outs.append(CD)
        for (A_st, B_st, C_st, A, Bm, C), s, CD in zip(probs, streams, outs):
            st = gb.gemm_tn(M, N, K, A.data_ptr(), K, 0, Bm.data_ptr(), K, 0, CD.data_ptr(), N, 0,
                            s.cuda_stream)
            assert st == gb.OK
        torch.cuda.synchronize()
        for (A_st, B_st, C_st, A, Bm, C), CD in zip(probs, outs):
            d64, d16 = oracle.gemm_tn(M, N, K, np_bits(A_st), K, 0, np_bits(B_st), K, 0,
                                      np_bits(C_st), N)
            check(np_bits(CD.cpu()), d64, d16, K, 0, True, f"two streams rep {rep}")
