"""gemm_tn_host: the scaled GEMM with A, B, C and D in host memory, the copies
in and out overlapped with the GEMMs of panels of M (a copy-in stream, the
caller's stream, a copy-out stream).

Each case is checked against the CPU oracle -- bit for bit on integer-valued
inputs (every partial sum exact), within the parity tolerances on real
values -- and against gemm_tn_scaled on device copies of the same arrays,
which runs the same kernels panel by panel and must agree bit for bit on
integer inputs.  The host arrays carry NaN slack past each row; D's slack
and rows must be untouched outside the view.  Panel sizes are forced small
so that the ring of three device slots is reused many times, with a ragged
last panel.
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


def _case(M, N, K, a_major=0, b_major=0, accum=0, alpha=1.0, beta=1.0, in_place=False,
          panel_rows=0, integer=True, pinned=True, seed=0, ready=0):
    dist, cdist = ("int1", "int4") if integer else ("normal_k", "u11")
    ldA = (K if a_major == 0 else M) + 5
    ldB = (K if b_major == 0 else N) + 3
    ldC, ldD = N + 7, (N + 7 if in_place else N + 2)
    A = wl.operand(M, K, ldA, a_major, dist, 2100 + seed, K)
    B = wl.operand(N, K, ldB, b_major, dist, 2200 + seed, K)
    C = wl.operand(M, N, ldC, 0, cdist, 2300 + seed)
    D = C.clone() if in_place else torch.full((M, ldD), float("nan"), dtype=torch.float16)
    if pinned:
        A, B, C, D = A.pin_memory(), B.pin_memory(), C.pin_memory(), D.pin_memory()
    C0, D0 = C.clone(), D.clone()
    Dout = C if in_place else D
    s = torch.cuda.current_stream().cuda_stream
    st = gb.gemm_tn_host(M, N, K, alpha, A.data_ptr(), ldA, a_major, B.data_ptr(), ldB, b_major,
                         beta, C.data_ptr(), ldC, Dout.data_ptr(), ldC if in_place else ldD,
                         accum, s, dict(host_panel_rows=panel_rows, host_inputs_ready=ready))
    assert st == gb.OK, gb.gemm_tn_status_string(st)
    kernels = gb.gemm_tn_last_kernels()
    torch.cuda.synchronize()
    got = np_bits(Dout)[:, :N]
    d64, d16 = oracle.gemm_tn_general(M, N, K, alpha, np_bits(A), ldA, a_major, np_bits(B), ldB,
                                      b_major, beta, np_bits(C0), ldC)
    what = f"host {M}x{N}x{K} a{a_major} b{b_major} acc{accum} panels of {panel_rows}"
    check(got.reshape(1, M, N), d64, d16, K, accum, integer, what)
    # nothing past each row of D is written; C is read only
    assert np.array_equal(np_bits(Dout)[:, N:], np_bits(C0 if in_place else D0)[:, N:]), \
        f"{what}: D's slack changed"
    if not in_place:
        assert np.array_equal(np_bits(C), np_bits(C0)), f"{what}: C changed"
    if integer:
        # gemm_tn_scaled on device copies (rows padded to a multiple of 8)
        dev = torch.device("cuda")

        def dev_copy(t, inner):
            ld = (inner + 7) // 8 * 8
            out = torch.zeros(t.shape[0], max(ld, 8), dtype=torch.float16, device=dev)
            out[:, :inner] = t[:, :inner].to(dev)
            return out, max(ld, 8)
        dA, lA = dev_copy(A, K if a_major == 0 else M)
        dB, lB = dev_copy(B, K if b_major == 0 else N)
        dC, lC = dev_copy(C0, N)
        dD = torch.zeros_like(dC)
        st = gb.gemm_tn_scaled(M, N, K, alpha, dA.data_ptr(), lA, a_major, dB.data_ptr(), lB,
                               b_major, beta, dC.data_ptr(), lC, dD.data_ptr(), lC, accum, s)
        assert st == gb.OK, gb.gemm_tn_status_string(st)
        torch.cuda.synchronize()
        assert np.array_equal(np_bits(dD.cpu())[:, :N], got), f"{what}: differs from device call"
    return kernels


@pytest.mark.parametrize("a_major,b_major", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("accum", [0, 1])
def test_host_panels_integers_bit_exact(a_major, b_major, accum):
    # 700 rows in panels of 64: eleven panels, the last of 60 rows, three slots reused
    _case(700, 300, 520, a_major, b_major, accum, panel_rows=64, seed=a_major + 2 * b_major)


@pytest.mark.parametrize("M,N,K,panel_rows", [(1, 1, 1, 0), (17, 9, 33, 8), (1030, 260, 200, 0),
                                              (2056, 520, 640, 0), (300, 2000, 4096, 128)])
def test_host_shapes(M, N, K, panel_rows):
    _case(M, N, K, panel_rows=panel_rows, seed=M)


def test_host_in_place_scaled_and_real_values():
    _case(500, 384, 1000, alpha=-2.0, beta=0.5, in_place=True, panel_rows=96, seed=5)
    _case(640, 256, 2048, integer=False, panel_rows=200, seed=6)
    _case(640, 256, 2048, accum=1, integer=False, panel_rows=200, seed=7)


def test_host_degenerate_terms():
    _case(200, 100, 64, beta=0.0, panel_rows=64, seed=8)        # C not read
    _case(200, 100, 64, alpha=0.0, beta=3.0, panel_rows=64, seed=9)  # no product term
    _case(200, 100, 0, panel_rows=64, seed=10)                  # K = 0: D = C


def test_host_inputs_ready_sizes_and_growth():
    # calls of growing size (the workspaces grow between them) and shrinking
    # size with the inputs declared ready, in place and not
    for i, (M, N, K) in enumerate([(100, 80, 64), (1500, 300, 700), (2100, 260, 520),
                                   (300, 100, 100)]):
        _case(M, N, K, in_place=bool(i % 2), panel_rows=0 if i != 1 else 128, seed=40 + i,
              ready=1)


def test_host_pageable_memory():
    _case(300, 200, 256, panel_rows=64, pinned=False, seed=11)


def test_host_workspace_exhaustion_enqueues_nothing():
    M, N, K = 256, 128, 128
    A = wl.operand(M, K, K, 0, "int1", 1).pin_memory()
    B = wl.operand(N, K, K, 0, "int1", 2).pin_memory()
    C = wl.operand(M, N, N, 0, "int4", 3).pin_memory()
    D = torch.full((M, N), 7.0, dtype=torch.float16).pin_memory()
    s = torch.cuda.current_stream().cuda_stream
    st = gb.gemm_tn_host(M, N, K, 1.0, A.data_ptr(), K, 0, B.data_ptr(), K, 0, 1.0, C.data_ptr(),
                         N, D.data_ptr(), N, 0, s, dict(test_fail_alloc=1))
    assert st == gb.ERR_NO_MEMORY
    assert gb.gemm_tn_last_launch_count() == 0
    torch.cuda.synchronize()
    assert bool((D == 7.0).all())


@pytest.mark.parametrize("ready", [0, 1])
def test_host_calls_back_to_back_on_one_stream(ready):
    # several calls queued before one synchronisation: each call's device
    # slots, the two alternating workspaces and the shared copy streams must
    # not mix up the calls (with host_inputs_ready the copies in of a call
    # start before the previous call has finished)
    M, N, K = 384, 256, 512
    s = torch.cuda.current_stream().cuda_stream
    outs = []
    for c in range(4):
        A = wl.operand(M, K, K, 0, "int1", 40 + c).pin_memory()
        B = wl.operand(N, K, K, 0, "int1", 50 + c).pin_memory()
        C = wl.operand(M, N, N, 0, "int4", 60 + c).pin_memory()
        D = torch.empty(M, N, dtype=torch.float16).pin_memory()
        st = gb.gemm_tn_host(M, N, K, 1.0, A.data_ptr(), K, 0, B.data_ptr(), K, 0, 1.0,
                             C.data_ptr(), N, D.data_ptr(), N, 0, s,
                             dict(host_panel_rows=64, host_inputs_ready=ready))
        assert st == gb.OK
        outs.append((A, B, C, D))
    torch.cuda.synchronize()
    for A, B, C, D in outs:
        d64, d16 = oracle.gemm_tn_general(M, N, K, 1.0, np_bits(A), K, 0, np_bits(B), K, 0, 1.0,
                                          np_bits(C), N)
        check(np_bits(D).reshape(1, M, N), d64, d16, K, 0, True, "back to back")


def test_host_call_captured_in_a_cuda_graph():
    # the copy streams join the capture through the call's events; the
    # workspace becomes a graph memory node; replays copy the host arrays as
    # they are at replay time
    M, N, K = 520, 264, 384
    A = wl.operand(M, K, K, 0, "int1", 70).pin_memory()
    B = wl.operand(N, K, K, 0, "int1", 71).pin_memory()
    C = wl.operand(M, N, N, 0, "int4", 72).pin_memory()
    D = torch.empty(M, N, dtype=torch.float16).pin_memory()

    def call(stream):
        return gb.gemm_tn_host(M, N, K, 1.0, A.data_ptr(), K, 0, B.data_ptr(), K, 0, 1.0,
                               C.data_ptr(), N, D.data_ptr(), N, 0, stream,
                               dict(host_panel_rows=128))
    assert call(torch.cuda.current_stream().cuda_stream) == gb.OK  # eager first call
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        assert call(torch.cuda.current_stream().cuda_stream) == gb.OK
    for rep in range(2):
        # new host values between replays
        A.copy_(wl.operand(M, K, K, 0, "int1", 80 + rep))
        D.fill_(0.0)
        g.replay()
        torch.cuda.synchronize()
        d64, d16 = oracle.gemm_tn_general(M, N, K, 1.0, np_bits(A), K, 0, np_bits(B), K, 0, 1.0,
                                          np_bits(C), N)
        check(np_bits(D).reshape(1, M, N), d64, d16, K, 0, True, f"graph replay {rep}")


def test_host_calls_from_two_threads():
    # each thread on its own stream with its own arrays; the library's copy
    # streams are shared, so the calls are serialised while they enqueue
    import threading
    M, N, K = 384, 200, 256
    results, errors = {}, []

    def worker(t):
        try:
            s = torch.cuda.Stream()
            for c in range(3):
                A = wl.operand(M, K, K, 0, "int1", 900 + 10 * t + c).pin_memory()
                B = wl.operand(N, K, K, 0, "int1", 950 + 10 * t + c).pin_memory()
                C = wl.operand(M, N, N, 0, "int4", 990 + 10 * t + c).pin_memory()
                D = torch.empty(M, N, dtype=torch.float16).pin_memory()
                st = gb.gemm_tn_host(M, N, K, 1.0, A.data_ptr(), K, 0, B.data_ptr(), K, 0, 1.0,
                                     C.data_ptr(), N, D.data_ptr(), N, 0, s.cuda_stream,
                                     dict(host_panel_rows=64))
                assert st == gb.OK, st
                results[(t, c)] = (A, B, C, D)
            s.synchronize()
        except Exception as e:  # reported by the main thread
            errors.append(e)
    ths = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in ths:
        th.start()
    for th in ths:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for (t, c), (A, B, C, D) in results.items():
        d64, d16 = oracle.gemm_tn_general(M, N, K, 1.0, np_bits(A), K, 0, np_bits(B), K, 0, 1.0,
                                          np_bits(C), N)
        check(np_bits(D).reshape(1, M, N), d64, d16, K, 0, True, f"thread {t} call {c}")


def test_host_tensor_front_end():
    import dense_fp16_tensor_gb300 as g
    M, N, K = 300, 200, 256
    A = wl.operand(M, K, K, 0, "int1", 1200).pin_memory()
    Bt = wl.operand(N, K, N, 1, "int1", 1201)   # stored (K, N): an N-major view of B
    Bv = Bt.t()                                  # (N, K) with strides (1, N)
    C = wl.operand(M, N, N, 0, "int4", 1202).pin_memory()
    D = g.gemm_host(A, Bv, C, alpha=2.0, beta=-1.0, host_panel_rows=64)
    d64, d16 = oracle.gemm_tn_general(M, N, K, 2.0, np_bits(A), K, 0, np_bits(Bt), N, 1, -1.0,
                                      np_bits(C), N)
    check(np_bits(D).reshape(1, M, N), d64, d16, K, 0, True, "tensor front end")
