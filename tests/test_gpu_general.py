"""GPU parity of the scaled and batched entry points,
D_l = alpha * A_l.B_l^T + beta * C_l, against the oracle's general form.

Integer-valued operands with scalars whose products stay exact make every
path bit-exact (the oracle rounds the exact value once); real values are
held to the acceptance tolerances.  Every call also checks that nothing
outside D's views changed (NaN-poisoned slack and gaps between problems),
and the BLAS conventions: alpha == 0 or K == 0 reads neither A nor B,
beta == 0 does not read C.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_fp16_tensor_gb300 import binding as gb
from dense_fp16_tensor_gb300 import workloads as wl
from parity import check, np_bits

pytestmark = pytest.mark.gpu

K_MAJ, MN_MAJ = 0, 1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp16_tensor_gb300 as g
    g.build()
    gb.lib()


def per_view(rows, cols, ld, major):
    return (rows if major == K_MAJ else cols) * ld


class Case:
    """Storage and strides of one batched call (CPU tensors)."""

    def __init__(self, M, N, K, L, am=K_MAJ, bm=K_MAJ, dist="int1", cdist="int4", pad=8, gap=16,
                 shared_a=False, shared_b=False, shared_c=False, in_place=False, c=True, seed=0):
        self.M, self.N, self.K, self.L = M, N, K, L
        self.am, self.bm = am, bm
        up8 = lambda x: (x + 7) // 8 * 8
        self.ldA = up8(K if am == K_MAJ else M) + pad
        self.ldB = up8(K if bm == K_MAJ else N) + pad
        self.ldC = up8(N) + pad
        self.ldD = self.ldC if in_place else up8(N) + 2 * pad
        self.sA = 0 if shared_a or L == 1 else per_view(M, K, self.ldA, am) + gap
        self.sB = 0 if shared_b or L == 1 else per_view(N, K, self.ldB, bm) + gap
        self.sC = 0 if shared_c or L == 1 else M * self.ldC + gap
        self.sD = self.sC if in_place else (0 if L == 1 else M * self.ldD + 2 * gap)
        self.A = wl.batched_operand(L, M, K, self.ldA, am, self.sA, dist, 100 + seed, K)
        self.B = wl.batched_operand(L, N, K, self.ldB, bm, self.sB, dist, 200 + seed, K)
        self.C = wl.batched_operand(L, M, N, self.ldC, K_MAJ, self.sC, cdist, 300 + seed) if c else None
        self.in_place = in_place
        if in_place:
            self.D0 = self.C.clone()
        else:
            self.D0 = wl.batched_operand(L, M, N, self.ldD, K_MAJ, self.sD, "int4", 400 + seed)

    def run(self, alpha, beta, acc=0, opts=None, pass_a=True, pass_b=True, pass_c=True):
        dev = torch.device("cuda")
        A = self.A.to(dev) if pass_a else None
        B = self.B.to(dev) if pass_b else None
        C = self.C.to(dev) if (pass_c and self.C is not None) else None
        D = C if self.in_place else self.D0.to(dev)
        ptr = lambda t: t.data_ptr() if t is not None else 0
        st = gb.gemm_tn_batched_ex(self.M, self.N, self.K, self.L, alpha, ptr(A), self.ldA,
                                   self.sA, self.am, ptr(B), self.ldB, self.sB, self.bm, beta,
                                   ptr(C), self.ldC, self.sC, ptr(D), self.ldD, self.sD, acc,
                                   torch.cuda.current_stream().cuda_stream,
                                   dict(sync_check=1, **(opts or {})))
        assert st == gb.OK, gb.gemm_tn_status_string(st)
        kernels = gb.gemm_tn_last_kernels()
        torch.cuda.synchronize()
        return D.cpu(), kernels

    def expect(self, alpha, beta):
        c = np_bits(self.C) if (self.C is not None and beta != 0) else None
        return oracle.gemm_tn_general(self.M, self.N, self.K, alpha, np_bits(self.A), self.ldA,
                                      self.am, np_bits(self.B), self.ldB, self.bm, beta, c,
                                      self.ldC, self.L, self.sA, self.sB, self.sC)

    def views(self, D):
        """(L, M, N) bits of D's views and a mask of the storage they cover."""
        bits = np_bits(D)
        out = np.empty((self.L, self.M, self.N), np.uint16)
        mask = np.zeros(bits.size, bool)
        for l in range(self.L):
            base = l * self.sD
            idx = base + np.arange(self.M)[:, None] * self.ldD + np.arange(self.N)[None, :]
            out[l] = bits[idx]
            mask[idx.reshape(-1)] = True
        return out, mask, bits

    def verify(self, D, alpha, beta, acc, exact, what):
        got, mask, bits = self.views(D)
        d64, d16 = self.expect(alpha, beta)
        check(got, d64, d16, self.K, acc, exact, what)
        before = np_bits(self.D0)
        bad = np.flatnonzero(~mask & (bits != before))
        where = [(int(i // self.sD) if self.sD else 0, int(i % self.sD // self.ldD) if self.sD
                  else int(i // self.ldD), int(i % self.ldD)) for i in bad[:6]]
        assert bad.size == 0, (f"{what}: {bad.size} elements written outside D's views, first "
                               f"(problem, row, col) {where}")


SCALARS = [(2.0, -0.5), (-1.0, 0.0), (0.5, 2.0), (1.0, 1.0)]


@pytest.mark.parametrize("alpha,beta", SCALARS)
@pytest.mark.parametrize("tile", [gb.TILE_SINGLE, gb.TILE_PAIR, gb.TILE_WIDE])
@pytest.mark.parametrize("acc", [0, 1])
def test_scaled_integers_bit_exact(alpha, beta, tile, acc):
    cs = Case(300, 520, 700, 1, seed=1)
    D, k = cs.run(alpha, beta, acc, dict(path=gb.PATH_LARGE, tile_kernel=tile))
    assert "gemm_tn" in k
    cs.verify(D, alpha, beta, acc, True, f"scaled tile={tile} acc={acc} a={alpha} b={beta}")


@pytest.mark.parametrize("am,bm", [(K_MAJ, K_MAJ), (MN_MAJ, K_MAJ), (K_MAJ, MN_MAJ),
                                   (MN_MAJ, MN_MAJ)])
@pytest.mark.parametrize("tile", [gb.TILE_SINGLE, gb.TILE_PAIR, gb.TILE_WIDE])
def test_batched_integers_bit_exact(am, bm, tile):
    cs = Case(264, 392, 328, 3, am, bm, seed=2)
    D, k = cs.run(-2.0, 0.5, 0, dict(path=gb.PATH_LARGE, tile_kernel=tile))
    cs.verify(D, -2.0, 0.5, 0, True, f"batched {am}{bm} tile={tile}")


@pytest.mark.parametrize("shared", ["a", "b", "c"])
def test_batched_shared_operand(shared):
    cs = Case(200, 300, 256, 4, shared_a=shared == "a", shared_b=shared == "b",
              shared_c=shared == "c", seed=3)
    D, _ = cs.run(1.0, 1.0, 0)
    cs.verify(D, 1.0, 1.0, 0, True, f"shared {shared}")


def test_batched_in_place_and_fp16_accumulation():
    cs = Case(333, 257, 450, 2, in_place=True, seed=4)
    D, _ = cs.run(0.5, 2.0, 1)
    cs.verify(D, 0.5, 2.0, 1, True, "in place, fp16 accumulation")


def test_batched_real_values_tolerance():
    cs = Case(520, 700, 1500, 3, dist="u11", cdist="u11", seed=5)
    for acc in (0, 1):
        D, _ = cs.run(0.75, -1.25, acc)
        cs.verify(D, 0.75, -1.25, acc, False, f"real acc={acc}")


def test_batched_small_m_runs_the_tile_kernel():
    cs = Case(16, 1000, 512, 4, seed=6)
    D, k = cs.run(2.0, 1.0, 0)
    assert k.startswith("gemm_tn_large_kernel"), k
    cs.verify(D, 2.0, 1.0, 0, True, "batched M=16")


def test_skinny_path_scaled_separate_d():
    # both skinny kernels: the cluster-reduced one (the library's choice here
    # up to M = 64) and the contiguous split with its reduction kernel
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for M in (16, 40, 64, 160, 256):
        cs = Case(M, 1000, 3000, 1, seed=7 + M)
        D, k = cs.run(0.5, -2.0, 0, dict(path=gb.PATH_SKINNY))
        assert k == ("gemm_tn_skinny_cluster_kernel" if M <= 64 else
                     "gemm_tn_skinny_kernel+gemm_tn_splitk_reduce_kernel"), k
        cs.verify(D, 0.5, -2.0, 0, True, f"skinny auto M={M}")
        D, k = cs.run(0.5, -2.0, 0, dict(path=gb.PATH_SKINNY, split_k=sms))
        assert k == "gemm_tn_skinny_kernel+gemm_tn_splitk_reduce_kernel", k
        cs.verify(D, 0.5, -2.0, 0, True, f"skinny split M={M}")


def test_stream_k_with_batches_and_scalars():
    cs = Case(300, 520, 700, 2, seed=8)
    D, k = cs.run(-1.0, 0.25, 0, dict(path=gb.PATH_LARGE, tile_kernel=gb.TILE_WIDE, stream_k=1))
    assert k == "memset+gemm_tn_wide_kernel", k
    cs.verify(D, -1.0, 0.25, 0, True, "stream-K batched")


def test_beta_zero_does_not_read_c():
    cs = Case(200, 300, 256, 2, seed=9)
    cs.C = torch.full_like(cs.C, float("nan"))
    D, _ = cs.run(3.0, 0.0, 0)
    cs.verify(D, 3.0, 0.0, 0, True, "beta 0, NaN C")
    D2, _ = cs.run(3.0, 0.0, 0, pass_c=False)  # C pointer NULL
    assert torch.equal(D.view(torch.int16), D2.view(torch.int16))
    cs1 = Case(40, 500, 2000, 1, seed=10)     # skinny path, C NULL
    for extra in ({}, {"split_k": torch.cuda.get_device_properties(0).multi_processor_count}):
        D3, k = cs1.run(1.0, 0.0, 0, dict(path=gb.PATH_SKINNY, **extra), pass_c=False)
        assert k.startswith("gemm_tn_skinny"), k
        cs1.verify(D3, 1.0, 0.0, 0, True, f"skinny beta 0 {k}")


@pytest.mark.parametrize("beta", [0.0, 1.0, -0.5])
def test_alpha_zero_and_empty_k(beta):
    cs = Case(130, 270, 96, 3, seed=11)
    cs.A = torch.full_like(cs.A, float("nan"))
    D, k = cs.run(0.0, beta, 0, pass_b=False)
    assert k == "gemm_tn_scale_kernel", k
    cs.verify(D, 0.0, beta, 0, True, f"alpha 0, beta {beta}")
    ce = Case(130, 270, 0, 2, seed=12)
    D, k = ce.run(2.0, beta, 0, pass_a=False, pass_b=False)
    assert k == "gemm_tn_scale_kernel", k
    ce.verify(D, 2.0, beta, 0, True, f"K 0, beta {beta}")


def test_empty_k_in_place_with_unit_beta_launches_nothing():
    cs = Case(64, 64, 0, 1, in_place=True, seed=13)
    D, k = cs.run(1.0, 1.0, 0, pass_a=False, pass_b=False)
    assert k == "" and gb.gemm_tn_last_launch_count() == 0
    assert torch.equal(D.view(torch.int16), cs.C.view(torch.int16))


def test_scaled_entry_point_matches_batched():
    cs = Case(300, 400, 500, 1, seed=14)
    dev = torch.device("cuda")
    A, B, C = cs.A.to(dev), cs.B.to(dev), cs.C.to(dev)
    D = cs.D0.to(dev)
    st = gb.gemm_tn_scaled(cs.M, cs.N, cs.K, 1.5, A.data_ptr(), cs.ldA, cs.am, B.data_ptr(),
                           cs.ldB, cs.bm, -1.0, C.data_ptr(), cs.ldC, D.data_ptr(), cs.ldD, 0,
                           torch.cuda.current_stream().cuda_stream)
    assert st == gb.OK
    torch.cuda.synchronize()
    cs.verify(D.cpu(), 1.5, -1.0, 0, True, "gemm_tn_scaled")


def test_batched_timeout_reports_and_recovers():
    cs = Case(300, 520, 704, 2, seed=15)
    dev = torch.device("cuda")
    A, B, C, D = cs.A.to(dev), cs.B.to(dev), cs.C.to(dev), cs.D0.to(dev)
    st = gb.gemm_tn_batched_ex(cs.M, cs.N, cs.K, cs.L, 2.0, A.data_ptr(), cs.ldA, cs.sA, 0,
                               B.data_ptr(), cs.ldB, cs.sB, 0, 1.0, C.data_ptr(), cs.ldC, cs.sC,
                               D.data_ptr(), cs.ldD, cs.sD, 0,
                               torch.cuda.current_stream().cuda_stream,
                               dict(path=gb.PATH_LARGE, tile_kernel=gb.TILE_WIDE, test_stall=1,
                                    timeout_ns=20_000_000, sync_check=1))
    assert st == gb.ERR_DEVICE_TIMEOUT
    D, _ = cs.run(2.0, 1.0, 0)
    cs.verify(D, 2.0, 1.0, 0, True, "after timeout")


def test_unscaled_entry_point_unchanged_by_general_form():
    # gemm_tn is the batch-1, alpha = beta = 1, in-place case: same bits
    cs = Case(520, 700, 900, 1, in_place=True, dist="u11", cdist="u11", seed=16)
    dev = torch.device("cuda")
    A, B = cs.A.to(dev), cs.B.to(dev)
    CD = cs.C.to(dev)
    assert gb.gemm_tn(cs.M, cs.N, cs.K, A.data_ptr(), cs.ldA, 0, B.data_ptr(), cs.ldB, 0,
                      CD.data_ptr(), cs.ldC, 0, torch.cuda.current_stream().cuda_stream) == gb.OK
    D, _ = cs.run(1.0, 1.0, 0)
    torch.cuda.synchronize()
    assert torch.equal(CD.cpu().view(torch.int16), D.view(torch.int16))


def test_batched_large_sampled_rows():
    """Two 4096^3 problems (16 x 16 tiles each, several waves), scaled, separate
    D, real values: whole rows of D checked against the oracle's general form
    evaluated on those rows only."""
    M = N = K = 4096
    L = 2
    dev = torch.device("cuda")
    A_st = wl.draw((L * M * K,), "u11", 501)
    B_st = wl.draw((L * N * K,), "u11", 502)
    C_st = wl.draw((L * M * N,), "u11", 503)
    A, B, C = A_st.to(dev), B_st.to(dev), C_st.to(dev)
    D = torch.empty(L * M * N, dtype=torch.float16, device=dev)
    st = gb.gemm_tn_batched(M, N, K, L, 0.5, A.data_ptr(), K, M * K, 0, B.data_ptr(), K, N * K,
                            0, -1.0, C.data_ptr(), N, M * N, D.data_ptr(), N, M * N, 0,
                            torch.cuda.current_stream().cuda_stream)
    assert st == gb.OK
    torch.cuda.synchronize()
    d = np_bits(D.cpu())
    a, b, c = np_bits(A_st), np_bits(B_st), np_bits(C_st)
    rng = np.random.default_rng(7)
    for l in range(L):
        for m0 in sorted(rng.choice(M - 1, 3, replace=False)):
            rows = 2
            ao = l * M * K + m0 * K
            co = l * M * N + m0 * N
            d64, d16 = oracle.gemm_tn_general(rows, N, K, 0.5, a[ao:ao + rows * K], K, 0,
                                              b[l * N * K:(l + 1) * N * K], K, 0, -1.0,
                                              c[co:co + rows * N], N)
            got = d[co:co + rows * N].reshape(1, rows, N)
            check(got, d64, d16, K, 0, False, f"problem {l} rows {m0}..{m0 + rows}")


@pytest.mark.parametrize("case", ["wide", "single", "scale", "skinny", "skinny_split", "streamk",
                                  "tile_split", "pair_split"])
def test_graph_capture_replays_match_eager(case):
    """A call captured into a CUDA graph (after one eager call has set the
    library up) replays to the same bits as the eager call.  The tile-kernel
    scale-only and cluster-reduced skinny paths allocate nothing per call;
    the split skinny path's workspace comes from the library's pool in
    stream order, which capture records as graph memory nodes."""
    M, N, K, L = {"skinny": (16, 1000, 3000, 1), "skinny_split": (16, 1000, 3000, 1),
                  "tile_split": (300, 200, 4000, 1),
                  "pair_split": (300, 520, 3000, 1)}.get(case, (520, 392, 328, 2))
    tile = {"wide": gb.TILE_WIDE, "single": gb.TILE_SINGLE, "scale": gb.TILE_WIDE,
            "skinny": 0, "skinny_split": 0, "streamk": gb.TILE_WIDE,
            "tile_split": gb.TILE_SINGLE, "pair_split": gb.TILE_PAIR}[case]
    path = gb.PATH_SKINNY if case.startswith("skinny") else gb.PATH_LARGE
    split = {"tile_split": 3, "pair_split": 3, "skinny_split": 64}.get(case, 0)
    alpha = 0.0 if case == "scale" else -2.0
    cs = Case(M, N, K, L, seed=20)
    dev = torch.device("cuda")
    A, B, C = cs.A.to(dev), cs.B.to(dev), cs.C.to(dev)
    D_eager, D_graph = cs.D0.to(dev), cs.D0.to(dev)

    def call(D, stream):
        return gb.gemm_tn_batched_ex(M, N, K, L, alpha, A.data_ptr(), cs.ldA, cs.sA, 0,
                                     B.data_ptr(), cs.ldB, cs.sB, 0, 0.5, C.data_ptr(), cs.ldC,
                                     cs.sC, D.data_ptr(), cs.ldD, cs.sD, 0, stream,
                                     dict(path=path, tile_kernel=tile,
                                          stream_k=1 if case == "streamk" else 0,
                                          split_k=split))
    assert call(D_eager, torch.cuda.current_stream().cuda_stream) == gb.OK
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        assert call(D_graph, torch.cuda.current_stream().cuda_stream) == gb.OK
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(D_graph.view(torch.int16), D_eager.view(torch.int16))
    cs.verify(D_graph.cpu(), alpha, 0.5, 0, True, f"graph replay {case}")


@pytest.mark.parametrize("route", ["repack", "copy"])
def test_graph_capture_of_the_strided_routes(route):
    """gemm_tn_strided captured and replayed: the repack route (pooled
    buffers, copy kernels, tile kernel, scatter of D) and the copy-producer
    kernel."""
    M, N, K = 300, 260, 200
    dev = torch.device("cuda")
    ld = K + 1  # not TMA-expressible: forces the repack route
    A_st = wl.draw((M * ld,), "int1", 31)
    B_st = wl.draw((N * ld,), "int1", 32)
    C_st = wl.draw((M * (N + 1),), "int4", 33)
    A, B = A_st.to(dev), B_st.to(dev)
    D1, D2 = C_st.to(dev), C_st.to(dev)

    path = gb.PATH_STRIDED_REPACK if route == "repack" else gb.PATH_STRIDED_COPY

    def call(D, stream):
        return gb.gemm_tn_strided_ex(M, N, K, A.data_ptr(), ld, 1, B.data_ptr(), ld, 1,
                                     D.data_ptr(), N + 1, 1, 0, stream, {"path": path})
    assert call(D1, torch.cuda.current_stream().cuda_stream) == gb.OK
    assert ("repack" in gb.gemm_tn_last_kernels()) == (route == "repack")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        assert call(D2, torch.cuda.current_stream().cuda_stream) == gb.OK
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(D1.view(torch.int16), D2.view(torch.int16))
    d64, d16 = oracle.gemm_tn_strided(M, N, K, np_bits(A_st), ld, 1, np_bits(B_st), ld, 1,
                                      np_bits(C_st), N + 1, 1)
    got = np_bits(D2.cpu())[:M * (N + 1)].reshape(M, N + 1)[:, :N]
    check(got, d64, d16, K, 0, True, f"strided graph replay ({route})")


def test_tensor_front_end_scaled_and_batched():
    """dense_fp16_tensor_gb300.gemm_scaled: 3-D batches (B shared through
    expand, stride 0), a separate output allocated by the call, and a 2-D
    in-place call with out = C."""
    import dense_fp16_tensor_gb300 as g
    dev = torch.device("cuda")
    L, M, N, K = 3, 136, 200, 96
    A = wl.draw((L, M, K), "int1", 41).to(dev)
    B1 = wl.draw((N, K), "int1", 42).to(dev)
    C = wl.draw((L, M, N), "int4", 43).to(dev)
    D = g.gemm_scaled(A, B1.unsqueeze(0).expand(L, N, K), C, alpha=2.0, beta=-1.0)
    torch.cuda.synchronize()
    assert D.shape == (L, M, N)
    _, ref16 = oracle.gemm_tn_general(M, N, K, 2.0, np_bits(A.cpu()), K, 0, np_bits(B1.cpu()), K,
                                      0, -1.0, np_bits(C.cpu()), N, L, M * K, 0, M * N)
    assert np.array_equal(np_bits(D.cpu()).reshape(L, M, N), ref16)
    # one problem, in place: C <- 0.5 * A0 . B1^T + 1 * C
    C0 = C[1].clone()
    out = g.gemm_scaled(A[0], B1, C0, alpha=0.5, out=C0)
    torch.cuda.synchronize()
    assert out.data_ptr() == C0.data_ptr()
    _, ref16 = oracle.gemm_tn_general(M, N, K, 0.5, np_bits(A[0].cpu()), K, 0, np_bits(B1.cpu()),
                                      K, 0, 1.0, np_bits(C[1].cpu()), N)
    assert np.array_equal(np_bits(C0.cpu()), ref16[0])


def test_concurrent_calls_from_host_threads():
    """Four host threads, each with its own stream, call the scaled entry point
    (tile path with K split, skinny path, 256x256 tiles) at the same time;
    every result matches the oracle (workspaces are per call, the library's
    per-thread state is thread-local)."""
    import threading
    dev = torch.device("cuda")
    shapes = [(512, 512, 8192), (48, 2000, 4096), (600, 700, 2048), (300, 260, 5000)]
    cases = [Case(M, N, K, 1, seed=60 + i) for i, (M, N, K) in enumerate(shapes)]
    inputs = [(cs.A.to(dev), cs.B.to(dev), cs.C.to(dev), cs.D0.to(dev)) for cs in cases]
    torch.cuda.synchronize()
    errors, kernels = [], {}

    def work(i):
        try:
            cs = cases[i]
            A, B, C, D = inputs[i]
            s = torch.cuda.Stream()
            for _ in range(5):
                st = gb.gemm_tn_batched_ex(cs.M, cs.N, cs.K, 1, -1.0, A.data_ptr(), cs.ldA, 0, 0,
                                           B.data_ptr(), cs.ldB, 0, 0, 2.0, C.data_ptr(), cs.ldC,
                                           0, D.data_ptr(), cs.ldD, 0, 0, s.cuda_stream, None)
                assert st == gb.OK, gb.gemm_tn_status_string(st)
            kernels[i] = gb.gemm_tn_last_kernels()
            s.synchronize()
        except Exception as e:  # reported below
            errors.append((i, repr(e)))
    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert "tile_reduce" in kernels[0] and "skinny" in kernels[1], kernels
    for i, cs in enumerate(cases):
        cs.verify(inputs[i][3].cpu(), -1.0, 2.0, 0, True, f"thread {i}")


def test_batch_strides_beyond_32_bits():
    """Problem 1's A and D start more than 2^31 elements (4 GiB) after
    problem 0's: the batch offsets go through 64-bit arithmetic in the tensor
    maps, the epilogue and the checks."""
    M, N, K, L = 256, 264, 128, 2
    big = (1 << 31) + 64            # elements, a multiple of 8
    dev = torch.device("cuda")
    A = torch.zeros(big + M * K, dtype=torch.float16, device=dev)
    Dbuf = torch.zeros(big + 64 + M * N, dtype=torch.float16, device=dev)
    A0 = wl.draw((M * K,), "int1", 71)
    A1 = wl.draw((M * K,), "int1", 72)
    A[:M * K] = A0.to(dev)
    A[big:big + M * K] = A1.to(dev)
    B = wl.draw((N * K,), "int1", 73).to(dev)
    C = wl.draw((M * N,), "int4", 74).to(dev)
    sD = big + 64
    for tile in (gb.TILE_SINGLE, gb.TILE_PAIR, gb.TILE_WIDE):
        st = gb.gemm_tn_batched_ex(M, N, K, L, 2.0, A.data_ptr(), K, big, 0, B.data_ptr(), K, 0, 0,
                                   -1.0, C.data_ptr(), N, 0, Dbuf.data_ptr(), N, sD, 0,
                                   torch.cuda.current_stream().cuda_stream,
                                   dict(path=gb.PATH_LARGE, tile_kernel=tile, sync_check=1))
        assert st == gb.OK, gb.gemm_tn_status_string(st)
        torch.cuda.synchronize()
        for l, Al in enumerate((A0, A1)):
            got = np_bits(Dbuf[l * sD:l * sD + M * N].cpu()).reshape(1, M, N)
            d64, d16 = oracle.gemm_tn_general(M, N, K, 2.0, np_bits(Al), K, 0, np_bits(B.cpu()),
                                              K, 0, -1.0, np_bits(C.cpu()), N)
            check(got, d64, d16, K, 0, True, f"problem {l} tile {tile}")
    del A, Dbuf
    torch.cuda.empty_cache()
