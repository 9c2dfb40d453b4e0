"""Phase trace (gemm_tn_options.trace, gemm_tn_trace_read): every CTA of a
traced launch stamps its phases in order, the CTAs' work units add up to
the problem's tiles, and tracing leaves the result unchanged (integer
inputs, bit-exact against the oracle)."""
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


ORDER = ("entry", "ready", "first_stage", "last_mma", "exit")


@pytest.mark.parametrize("M,N,K,opts,tiles", [
    (1000, 704, 640, dict(path=gb.PATH_LARGE, tile_kernel=1, tile_n=128), 8 * 6),
    (1000, 704, 640, dict(path=gb.PATH_LARGE, tile_kernel=2, tile_n=256), 4 * 3),
    (1000, 704, 640, dict(path=gb.PATH_LARGE, tile_kernel=3), 4 * 3),
    (16, 4096, 4096, dict(path=gb.PATH_SKINNY), None),
])
def test_traced_launch_records_every_cta_in_order(M, N, K, opts, tiles):
    dev = torch.device("cuda")
    s = torch.cuda.current_stream().cuda_stream
    A_st = wl.operand(M, K, K, 0, "int1", 61)
    B_st = wl.operand(N, K, K, 0, "int1", 62)
    C_st = wl.operand(M, N, N, 0, "int4", 63)
    A, B, CD = A_st.to(dev), B_st.to(dev), C_st.to(dev)
    st = gb.gemm_tn_ex(M, N, K, A.data_ptr(), K, 0, B.data_ptr(), K, 0, CD.data_ptr(), N, 0, s,
                       dict(trace=1, **opts))
    assert st == gb.OK, gb.gemm_tn_status_string(st)
    st, recs = gb.gemm_tn_trace_read(s)
    assert st == gb.OK
    assert recs, "no CTA recorded"
    busy = [r for r in recs if r["units"] > 0]
    assert busy
    for r in busy:
        t = [r[f] for f in ORDER]
        assert all(x > 0 for x in t), r
        assert t == sorted(t), r
        assert r["first_acc"] == 0 or r["first_stage"] <= r["first_acc"] <= r["exit"], r
    if tiles is not None:
        # (the pair kernel counts a tile once, on the even CTA of its pair)
        assert sum(r["units"] for r in recs) == tiles
    assert len({r["sm"] for r in recs}) == len(recs)  # one CTA per SM (persistent grids)
    d64, d16 = oracle.gemm_tn(M, N, K, np_bits(A_st), K, 0, np_bits(B_st), K, 0, np_bits(C_st), N)
    check(np_bits(CD.cpu()), d64, d16, K, 0, True, f"traced {opts}")


def test_untraced_launch_leaves_the_last_trace_alone():
    dev = torch.device("cuda")
    s = torch.cuda.current_stream().cuda_stream
    M, N, K = 256, 256, 256
    A = torch.zeros(M, K, dtype=torch.float16, device=dev)
    CD = torch.zeros(M, N, dtype=torch.float16, device=dev)
    o = dict(path=gb.PATH_LARGE, tile_kernel=1, tile_n=128)
    assert gb.gemm_tn_ex(M, N, K, A.data_ptr(), K, 0, A.data_ptr(), K, 0, CD.data_ptr(), N, 0, s,
                         dict(trace=1, **o)) == gb.OK
    st, first = gb.gemm_tn_trace_read(s)
    assert gb.gemm_tn_ex(M, N, K, A.data_ptr(), K, 0, A.data_ptr(), K, 0, CD.data_ptr(), N, 0, s,
                         o) == gb.OK
    st, second = gb.gemm_tn_trace_read(s)
    assert st == gb.OK and first == second and len(first) == 4
