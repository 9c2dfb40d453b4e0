"""Seeded random configurations of the scaled, batched entry point against the
oracle, bit for bit: sizes with ragged tails, both majors per operand,
batches with gaps and shared operands, alpha / beta including 0, fp32 and
fp16 accumulation, and every path control (automatic, each tile kernel,
stream-K, explicit K splits of the 128-row and pair kernels, the skinny
path).  Operands are integers in
{-1, 0, 1} and C in {-4..4}, so every result is exact up to the final
rounding, which both sides take once from the same value (fp16
accumulation only where its partial sums stay within 2048).  Each case also
checks that nothing outside D's views was written.
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


def draw_case(rng):
    L = int(rng.choice([1, 1, 2, 3]))
    acc = int(rng.choice([0, 0, 0, 1]))
    kmax = 2048 if acc == 1 else 3000
    while True:
        M, N = int(rng.integers(1, 700)), int(rng.integers(1, 700))
        K = int(rng.integers(1, kmax + 1))
        if M * N * K * L <= 1.5e8:
            break
    am, bm = int(rng.integers(0, 2)), int(rng.integers(0, 2))
    alpha = float(rng.choice([1.0, 2.0, -1.0, 0.5, 0.0]))
    beta = float(rng.choice([1.0, 0.0, -0.5, 2.0]))
    opts = {}
    mode = rng.choice(["auto", "tile1", "tile1_split", "pair", "pair_split", "wide", "wide_sk",
                       "skinny"])
    if mode == "tile1":
        opts = dict(path=gb.PATH_LARGE, tile_kernel=1, tile_n=int(rng.choice([64, 128, 256])))
    elif mode == "tile1_split":
        opts = dict(path=gb.PATH_LARGE, tile_kernel=1, split_k=int(rng.integers(2, 5)))
    elif mode == "pair":
        opts = dict(path=gb.PATH_LARGE, tile_kernel=2)
    elif mode == "pair_split":
        opts = dict(path=gb.PATH_LARGE, tile_kernel=2, split_k=int(rng.integers(2, 6)))
    elif mode == "wide":
        opts = dict(path=gb.PATH_LARGE, tile_kernel=3)
    elif mode == "wide_sk":
        opts = dict(path=gb.PATH_LARGE, tile_kernel=3, stream_k=1)
    elif mode == "skinny":
        if M <= 128 and am == 0 and bm == 0 and acc == 0 and L == 1:
            opts = dict(path=gb.PATH_SKINNY)
    shared = {x: L > 1 and rng.random() < 0.25 for x in "ABC"}
    return M, N, K, L, am, bm, acc, alpha, beta, opts, shared, str(mode)


CASES = [draw_case(np.random.default_rng(10_000 + i)) for i in range(96)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}xL{c[3]}-{c[11]}")
def test_random_configuration_bit_exact(case):
    M, N, K, L, am, bm, acc, alpha, beta, opts, shared, mode = case
    ldA = up8(K if am == 0 else M) + 8
    ldB = up8(K if bm == 0 else N) + 8
    ldC, ldD = up8(N) + 8, up8(N) + 16
    per = lambda rows, cols, ld, major: (rows if major == 0 else cols) * ld
    sA = 0 if (L == 1 or shared["A"]) else per(M, K, ldA, am) + 24
    sB = 0 if (L == 1 or shared["B"]) else per(N, K, ldB, bm) + 40
    sC = 0 if (L == 1 or shared["C"]) else M * ldC + 8
    sD = M * ldD + 16 if L > 1 else 0
    seed = abs(hash((M, N, K, L))) % 100_000
    A_st = wl.batched_operand(L, M, K, ldA, am, sA, "int1", seed + 1, K)
    B_st = wl.batched_operand(L, N, K, ldB, bm, sB, "int1", seed + 2, K)
    C_st = wl.batched_operand(L, M, N, ldC, 0, sC, "int4", seed + 3)
    D0 = wl.batched_operand(L, M, N, ldD, 0, sD, "int4", seed + 4)
    dev = torch.device("cuda")
    A, B, C, D = A_st.to(dev), B_st.to(dev), C_st.to(dev), D0.to(dev)
    st = gb.gemm_tn_batched_ex(M, N, K, L, alpha, A.data_ptr(), ldA, sA, am, B.data_ptr(), ldB,
                               sB, bm, beta, C.data_ptr(), ldC, sC, D.data_ptr(), ldD, sD, acc,
                               torch.cuda.current_stream().cuda_stream,
                               dict(sync_check=1, **opts))
    assert st == gb.OK, (gb.gemm_tn_status_string(st), case)
    torch.cuda.synchronize()
    bits = np_bits(D.cpu())
    idx = [l * sD + np.arange(M)[:, None] * ldD + np.arange(N)[None, :] for l in range(L)]
    got = np.stack([bits[i] for i in idx])
    d64, d16 = oracle.gemm_tn_general(M, N, K, alpha, np_bits(A_st), ldA, am, np_bits(B_st), ldB,
                                      bm, beta, np_bits(C_st), ldC, L, sA, sB, sC)
    check(got, d64, d16, K, acc, True, f"{case} kernels {gb.gemm_tn_last_kernels()}")
    mask = np.zeros(bits.size, bool)
    for i in idx:
        mask[i.reshape(-1)] = True
    assert np.array_equal(bits[~mask], np_bits(D0)[~mask]), f"{case}: wrote outside D's views"
