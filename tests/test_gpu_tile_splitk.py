"""GPU parity of the K split in the 128-row tile kernel: for problems whose
tiles would leave more than half the SMs idle, each tile's K loop is cut
over several CTAs, every split stores an fp32 partial tile, and a second
kernel adds the splits in a fixed order plus beta * C once (the
make_tiled_mma page's K split across workers: the partial sums are reduced
and C is added once).  Integer-valued inputs make every case bit-exact
against the oracle; real values are checked for determinism and tolerance.
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


def up8(x):
    return (x + 7) // 8 * 8


def run(M, N, K, L, alpha, beta, dist="int1", cdist="int4", acc=0, opts=None, seed=0,
        am=0, bm=0):
    ldA = up8(K if am == 0 else M) + 8
    ldB = up8(K if bm == 0 else N) + 8
    ldC, ldD = up8(N) + 8, up8(N) + 16
    per = lambda rows, cols, ld, major: (rows if major == 0 else cols) * ld
    sA = per(M, K, ldA, am) + 16 if L > 1 else 0
    sB = per(N, K, ldB, bm) + 16 if L > 1 else 0
    sC = M * ldC + 16 if L > 1 else 0
    sD = M * ldD + 32 if L > 1 else 0
    A_st = wl.batched_operand(L, M, K, ldA, am, sA, dist, 500 + seed, K)
    B_st = wl.batched_operand(L, N, K, ldB, bm, sB, dist, 600 + seed, K)
    C_st = wl.batched_operand(L, M, N, ldC, 0, sC, cdist, 700 + seed)
    D0 = wl.batched_operand(L, M, N, ldD, 0, sD, "int4", 800 + seed)
    dev = torch.device("cuda")
    A, B, C, D = A_st.to(dev), B_st.to(dev), C_st.to(dev), D0.to(dev)
    st = gb.gemm_tn_batched_ex(M, N, K, L, alpha, A.data_ptr(), ldA, sA, am, B.data_ptr(), ldB,
                               sB, bm, beta, C.data_ptr(), ldC, sC, D.data_ptr(), ldD, sD, acc,
                               torch.cuda.current_stream().cuda_stream,
                               dict(sync_check=1, **(opts or {})))
    assert st == gb.OK, gb.gemm_tn_status_string(st)
    kernels = gb.gemm_tn_last_kernels()
    torch.cuda.synchronize()
    bits = np_bits(D.cpu())
    got = np.stack([bits[l * sD + np.arange(M)[:, None] * ldD + np.arange(N)[None, :]]
                    for l in range(L)])
    d64, d16 = oracle.gemm_tn_general(M, N, K, alpha, np_bits(A_st), ldA, am, np_bits(B_st), ldB,
                                      bm, beta, np_bits(C_st), ldC, L, sA, sB, sC)
    # nothing outside D's views changed
    mask = np.zeros(bits.size, bool)
    for l in range(L):
        mask[(l * sD + np.arange(M)[:, None] * ldD + np.arange(N)[None, :]).reshape(-1)] = True
    assert np.array_equal(bits[~mask], np_bits(D0)[~mask]), "wrote outside D's views"
    return got, d64, d16, kernels


SPLIT = "gemm_tn_large_kernel<128>+gemm_tn_tile_reduce_kernel"


@pytest.mark.parametrize("shape", [(512, 512, 8192), (1024, 1024, 4096), (300, 200, 5000),
                                   (128, 128, 64 * 40), (100, 260, 2600)])
def test_automatic_split_integers_bit_exact(shape):
    M, N, K = shape
    # the tile path (M <= 256 would otherwise take the skinny path)
    got, d64, d16, k = run(M, N, K, 1, 1.0, 1.0, seed=1, opts=dict(path=gb.PATH_LARGE))
    assert k == SPLIT, k
    check(got, d64, d16, K, 0, True, f"split {shape}")


@pytest.mark.parametrize("am,bm", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_split_with_scalars_batches_and_majors(am, bm):
    got, d64, d16, k = run(200, 300, 3000, 2, -2.0, 0.5, seed=2, am=am, bm=bm)
    assert k == SPLIT, k
    check(got, d64, d16, 3000, 0, True, f"split batched {am}{bm}")


def test_split_beta_zero_and_real_values_deterministic():
    # the tile path (M <= 256 with this N would otherwise take the skinny path)
    o = dict(path=gb.PATH_LARGE)
    a = run(256, 384, 6000, 1, 0.75, 0.0, dist="u11", cdist="u11", seed=3, opts=o)
    b = run(256, 384, 6000, 1, 0.75, 0.0, dist="u11", cdist="u11", seed=3, opts=o)
    assert a[3] == SPLIT
    assert np.array_equal(a[0], b[0])  # fixed summation order
    check(a[0], a[1], a[2], 6000, 0, False, "split real")


def test_explicit_split_count_on_a_larger_problem():
    got, d64, d16, k = run(1000, 1200, 2048, 1, 1.0, 1.0, seed=4,
                           opts=dict(path=gb.PATH_LARGE, tile_kernel=1, tile_n=256, split_k=3))
    assert k == "gemm_tn_large_kernel<256>+gemm_tn_tile_reduce_kernel", k
    check(got, d64, d16, 2048, 0, True, "explicit split 3")


def test_fp16_accumulation_is_never_split():
    got, d64, d16, k = run(512, 512, 4096, 1, 1.0, 1.0, acc=1, seed=5)
    # 16 tiles of 128 x 128 would leave most SMs idle: 128 x 64 tiles, unsplit
    assert k == "gemm_tn_large_kernel<64>", k
    check(got, d64, d16, 4096, 1, True, "fp16 accumulation unsplit")


def test_split_timeout_reports_and_recovers():
    M, N, K = 512, 512, 8192
    dev = torch.device("cuda")
    A = wl.draw((M * K,), "int1", 900).to(dev)
    B = wl.draw((N * K,), "int1", 901).to(dev)
    C = wl.draw((M * N,), "int4", 902).to(dev)
    D = torch.empty_like(C)
    st = gb.gemm_tn_batched_ex(M, N, K, 1, 1.0, A.data_ptr(), K, 0, 0, B.data_ptr(), K, 0, 0, 1.0,
                               C.data_ptr(), N, 0, D.data_ptr(), N, 0, 0,
                               torch.cuda.current_stream().cuda_stream,
                               dict(test_stall=1, timeout_ns=20_000_000, sync_check=1))
    assert st == gb.ERR_DEVICE_TIMEOUT
    got, d64, d16, k = run(M, N, K, 1, 1.0, 1.0, seed=6)
    assert k == SPLIT
    check(got, d64, d16, K, 0, True, "after timeout")


# --- the same K split in the CTA-pair kernel (split_k with tile_kernel 2):
# each unit stores its two CTAs' rows as two 128-row partial tiles, and the
# same reduction adds the splits in order.

PAIR_SPLIT = "gemm_tn_large2_kernel{}+gemm_tn_tile_reduce_kernel"


@pytest.mark.parametrize("M,N,K,L,am,bm,splits,deep", [
    (300, 520, 3000, 1, 0, 0, 3, True),     # K-major rows on the 128-byte grid: deep stages
    (500, 260, 2500, 1, 0, 0, 2, True),     # ld 2512: off the 128-byte grid, deep stages
    (256, 2048, 4088, 1, 0, 0, 2, True),
    (300, 300, 2000, 1, 1, 1, 3, True),     # both operands M/N-major
    (130, 700, 1100, 1, 1, 0, 5, True),     # splits of 1-2 K blocks of 128; last split short
    (130, 700, 900, 1, 1, 0, 5, False),     # K < 1024: 64-deep stages, splits of 3 blocks
])
def test_pair_split_integers_bit_exact(M, N, K, L, am, bm, splits, deep):
    got, d64, d16, k = run(M, N, K, L, 1.0, 1.0, seed=10 + splits, am=am, bm=bm,
                           opts=dict(path=gb.PATH_LARGE, tile_kernel=2, split_k=splits))
    assert k == PAIR_SPLIT.format("<deep>" if deep else ""), k
    check(got, d64, d16, K, 0, True, f"pair split {M}x{N}x{K} s={splits}")


def test_pair_split_batched_scalars_and_determinism():
    o = dict(path=gb.PATH_LARGE, tile_kernel=2, split_k=4)
    got, d64, d16, k = run(200, 300, 3000, 2, -2.0, 0.5, seed=20, opts=o)
    assert k == PAIR_SPLIT.format("<deep>"), k
    check(got, d64, d16, 3000, 0, True, "pair split batched")
    a = run(520, 260, 3000, 1, 0.75, 0.0, dist="u11", cdist="u11", seed=21, opts=o)
    b = run(520, 260, 3000, 1, 0.75, 0.0, dist="u11", cdist="u11", seed=21, opts=o)
    assert np.array_equal(a[0], b[0])  # fixed summation order
    check(a[0], a[1], a[2], 3000, 0, False, "pair split real")


def test_pair_split_timeout_reports_and_recovers():
    M, N, K = 512, 512, 8192
    dev = torch.device("cuda")
    A = wl.draw((M * K,), "int1", 910).to(dev)
    B = wl.draw((N * K,), "int1", 911).to(dev)
    C = wl.draw((M * N,), "int4", 912).to(dev)
    D = torch.empty_like(C)
    st = gb.gemm_tn_batched_ex(M, N, K, 1, 1.0, A.data_ptr(), K, 0, 0, B.data_ptr(), K, 0, 0, 1.0,
                               C.data_ptr(), N, 0, D.data_ptr(), N, 0, 0,
                               torch.cuda.current_stream().cuda_stream,
                               dict(path=gb.PATH_LARGE, tile_kernel=2, split_k=2, test_stall=1,
                                    timeout_ns=20_000_000, sync_check=1))
    assert st == gb.ERR_DEVICE_TIMEOUT
    got, d64, d16, k = run(M, N, K, 1, 1.0, 1.0, seed=22,
                           opts=dict(path=gb.PATH_LARGE, tile_kernel=2, split_k=2))
    assert k == PAIR_SPLIT.format("<deep>"), k
    check(got, d64, d16, K, 0, True, "pair split after timeout")


# --- the pair kernel's last-wave split: after the rounds of whole 256 x 256
# tiles, the tiles of the last, partial round run as K splits over the pairs
# that would otherwise idle, and the same reduction adds their partials.

@pytest.mark.parametrize("M,N,K,L,am,bm", [
    (2560, 2048, 4096, 1, 0, 0),    # 80 tiles: one round of 76, then 4 tiles x 4 splits
    (1280, 2048, 4096, 2, 1, 0),    # two problems of 40 tiles, M-major A
    (2400, 2100, 3000, 1, 0, 1),    # 90 tiles: 14 x 3 splits; ragged edges, N-major B
])
def test_pair_last_wave_split_integers_bit_exact(M, N, K, L, am, bm):
    o = dict(path=gb.PATH_LARGE, tile_kernel=2, tile_n=256)
    got, d64, d16, k = run(M, N, K, L, 1.0, 1.0, seed=30, am=am, bm=bm, opts=o)
    assert k == PAIR_SPLIT.format("<deep>"), k
    check(got, d64, d16, K, 0, True, f"last-wave split {M}x{N}x{K}xL{L}")
    # the same call without the split: the same bits
    got2, _, _, k2 = run(M, N, K, L, 1.0, 1.0, seed=30, am=am, bm=bm,
                         opts=dict(o, stream_k=-1))
    assert k2 == "gemm_tn_large2_kernel<deep>", k2
    assert np.array_equal(got, got2)


def test_pair_last_wave_split_scaled_real_values():
    o = dict(path=gb.PATH_LARGE, tile_kernel=2, tile_n=256)
    a = run(2560, 2048, 4096, 1, -0.5, 2.0, dist="u11", cdist="u11", seed=31, opts=o)
    b = run(2560, 2048, 4096, 1, -0.5, 2.0, dist="u11", cdist="u11", seed=31, opts=o)
    assert np.array_equal(a[0], b[0])  # fixed summation order
    check(a[0], a[1], a[2], 4096, 0, False, "last-wave split real")
