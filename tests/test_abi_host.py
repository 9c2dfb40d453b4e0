"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, loads, exports every function include/gemm_tn.h declares, and
rejects bad arguments before it touches the device (the pointers below are
never dereferenced: validation returns first)."""
import ctypes
import os
import re

import pytest

import dense_fp16_tensor_gb300 as g
from dense_fp16_tensor_gb300 import binding as gb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    g.build()
    return gb.lib()


def header_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"GEMM_TN_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = header_functions()
    assert set(gb.EXPORTED) <= set(names)
    for n in names:
        assert hasattr(lib, n), n  # ctypes resolves it with dlsym


def test_status_strings(lib):
    for s, name in [(0, "GEMM_TN_OK"), (1, "GEMM_TN_ERR_INVALID_ARG"),
                    (2, "GEMM_TN_ERR_ALIGNMENT"), (5, "GEMM_TN_ERR_DEVICE_TIMEOUT"),
                    (99, "GEMM_TN_ERR_UNKNOWN")]:
        assert gb.gemm_tn_status_string(s) == name


def test_plan_path(lib):
    P = gb.gemm_tn_plan_path
    assert P(16, 16384, 16384, 0, 0) == gb.PATH_SKINNY
    # long enough K for the skinny path: 2048 up to M = 32, 4096 up to 64, 8192 above
    assert P(32, 100, 2048, 0, 0) == gb.PATH_SKINNY
    assert P(32, 100, 2047, 0, 0) == gb.PATH_LARGE
    assert P(33, 100, 2048, 0, 0) == gb.PATH_LARGE
    assert P(64, 100, 4096, 0, 0) == gb.PATH_SKINNY
    assert P(64, 100, 4095, 0, 0) == gb.PATH_LARGE
    assert P(128, 100, 8192, 0, 0) == gb.PATH_SKINNY
    assert P(128, 100, 8191, 0, 0) == gb.PATH_LARGE
    assert P(32, 16, 16, 0, 0) == gb.PATH_LARGE        # the tiny workload
    # M up to 192 at any N; up to 256 while N <= 14336
    assert P(192, 65536, 8192, 0, 0) == gb.PATH_SKINNY
    assert P(193, 14336, 8192, 0, 0) == gb.PATH_SKINNY
    assert P(256, 14336, 8192, 0, 0) == gb.PATH_SKINNY
    assert P(193, 14337, 8192, 0, 0) == gb.PATH_LARGE
    assert P(257, 100, 8192, 0, 0) == gb.PATH_LARGE
    assert P(16, 100, 8192, 1, 0) == gb.PATH_LARGE     # M-major A
    assert P(8192, 8192, 8192, 0, 0) == gb.PATH_LARGE


P = 0x7F0000000000  # a 16-byte aligned fake device address, never dereferenced


def call(M=64, N=64, K=64, A=P, ldA=64, am=0, B=P + (1 << 20), ldB=64, bm=0,
         CD=P + (2 << 20), ldC=64, acc=0, opts=None):
    return gb.gemm_tn_ex(M, N, K, A, ldA, am, B, ldB, bm, CD, ldC, acc, None, opts)


@pytest.mark.parametrize("kw,status", [
    (dict(M=-1), gb.ERR_INVALID_ARG),
    (dict(K=1 << 31), gb.ERR_INVALID_ARG),
    (dict(ldA=63), gb.ERR_INVALID_ARG),                  # K-major A needs ldA >= K
    (dict(am=1, ldA=32), gb.ERR_INVALID_ARG),            # M-major A needs ldA >= M
    (dict(ldB=8), gb.ERR_INVALID_ARG),
    (dict(ldC=56), gb.ERR_INVALID_ARG),
    (dict(am=2), gb.ERR_INVALID_ARG),
    (dict(acc=3), gb.ERR_INVALID_ARG),
    (dict(A=0), gb.ERR_INVALID_ARG),
    (dict(CD=0), gb.ERR_INVALID_ARG),
    (dict(CD=P), gb.ERR_INVALID_ARG),                    # CD overlaps A
    (dict(CD=P + (1 << 20) + 128), gb.ERR_INVALID_ARG),  # CD overlaps B
    (dict(A=P + 8), gb.ERR_ALIGNMENT),
    (dict(CD=P + (2 << 20) + 2), gb.ERR_ALIGNMENT),
    (dict(ldA=68), gb.ERR_ALIGNMENT),
    (dict(ldC=68), gb.ERR_ALIGNMENT),
    (dict(opts=gb.make_options(path=7)), gb.ERR_INVALID_ARG),
    (dict(opts=gb.make_options(tile_n=96)), gb.ERR_INVALID_ARG),
    (dict(opts=gb.make_options(tile_n=300)), gb.ERR_INVALID_ARG),
    (dict(opts=gb.make_options(k_stage=32)), gb.ERR_INVALID_ARG),
    (dict(M=264, opts=gb.make_options(path=2)), gb.ERR_INVALID_ARG),  # skinny needs M <= 256
])
def test_argument_errors_return_before_any_device_work(lib, kw, status):
    assert call(**kw) == status
    assert gb.gemm_tn_last_launch_count() == 0
    assert gb.gemm_tn_last_kernels() == ""


def test_noop_sizes_return_ok_without_a_device(lib):
    assert call(M=0) == gb.OK
    assert call(N=0) == gb.OK
    assert call(K=0) == gb.OK  # D = C: nothing to launch
    assert gb.gemm_tn_last_launch_count() == 0


def test_null_operands_allowed_when_k_is_zero(lib):
    assert call(K=0, A=0, B=0) == gb.OK


def test_tensor_front_end_major_inference():
    torch = pytest.importorskip("torch")
    from dense_fp16_tensor_gb300.tensor_api import operand_view
    a = torch.zeros(4, 16, dtype=torch.float16)
    assert operand_view(a, "A") == (gb.MAJOR_K, 16)
    assert operand_view(torch.zeros(16, 24, dtype=torch.float16).t(), "A") == (gb.MAJOR_MN, 24)
    st = torch.zeros(40, 32, dtype=torch.float16)
    assert operand_view(st[:, :20], "A") == (gb.MAJOR_K, 32)   # padded ld
    with pytest.raises(ValueError):
        operand_view(torch.zeros(8, 8, 2, dtype=torch.float16)[:, :, 0], "A")


def scall(M=64, N=64, K=64, A=P, sAm=64, sAk=1, B=P + (1 << 20), sBn=64, sBk=1,
          CD=P + (2 << 20), sCm=64, sCn=1, acc=0):
    return gb.gemm_tn_strided(M, N, K, A, sAm, sAk, B, sBn, sBk, CD, sCm, sCn, acc, None)


@pytest.mark.parametrize("kw,status", [
    (dict(M=-1), gb.ERR_INVALID_ARG),
    (dict(sAk=-1), gb.ERR_INVALID_ARG),
    (dict(sCm=0), gb.ERR_INVALID_ARG),               # two rows of D on the same elements
    (dict(sCm=32, sCn=1), gb.ERR_INVALID_ARG),       # rows of 64 overlap with stride 32
    (dict(sCm=1, sCn=1), gb.ERR_INVALID_ARG),
    (dict(CD=P), gb.ERR_INVALID_ARG),                # overlaps A
    (dict(A=0), gb.ERR_INVALID_ARG),
    (dict(acc=2), gb.ERR_INVALID_ARG),
    (dict(A=P + 1), gb.ERR_ALIGNMENT),               # fp16 needs 2-byte alignment
    (dict(CD=P + (2 << 20) + 3), gb.ERR_ALIGNMENT),
])
def test_strided_argument_errors(lib, kw, status):
    assert scall(**kw) == status
    assert gb.gemm_tn_last_launch_count() == 0


def test_strided_noop_sizes(lib):
    assert scall(M=0) == gb.OK
    assert scall(K=0, A=0, B=0) == gb.OK
    assert scall(M=1, sCm=0, K=0) == gb.OK  # one row: a zero row stride is fine


def test_strided_ex_rejects_tile_paths(lib):
    for path in (gb.PATH_LARGE, gb.PATH_SKINNY, 9):
        assert gb.gemm_tn_strided_ex(64, 64, 64, P, 64, 1, P + (1 << 20), 64, 1, P + (2 << 20),
                                     64, 1, 0, None, {"path": path}) == gb.ERR_INVALID_ARG


# --- scaled / batched form: argument checks (no device needed) -------------

MB = 1 << 20


def bcall(M=64, N=64, K=64, L=2, alpha=1.0, A=P, ldA=64, sA=64 * 64, am=0, B=P + 4 * MB,
          ldB=64, sB=64 * 64, bm=0, beta=1.0, C=P + 8 * MB, ldC=64, sC=64 * 64,
          D=P + 12 * MB, ldD=64, sD=64 * 64, acc=0):
    return gb.gemm_tn_batched_ex(M, N, K, L, alpha, A, ldA, sA, am, B, ldB, sB, bm, beta, C,
                                 ldC, sC, D, ldD, sD, acc, None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(L=-1), gb.ERR_INVALID_ARG),
    (dict(C=0), gb.ERR_INVALID_ARG),                      # beta != 0 needs C
    (dict(D=0), gb.ERR_INVALID_ARG),
    (dict(sD=64 * 64 - 8), gb.ERR_INVALID_ARG),           # the problems' D overlap
    (dict(sA=64 * 63), gb.ERR_INVALID_ARG),               # A views overlap (not 0)
    (dict(sB=-64 * 64), gb.ERR_INVALID_ARG),
    (dict(sC=-8), gb.ERR_INVALID_ARG),
    (dict(D=P + 8 * MB + 128), gb.ERR_INVALID_ARG),       # D overlaps C, not in place
    (dict(D=P + 8 * MB, ldD=72, sD=72 * 64), gb.ERR_INVALID_ARG),  # same base, other view
    (dict(D=P + 4096 * 2), gb.ERR_INVALID_ARG),           # D overlaps problem 1's A
    (dict(D=P + 4 * MB + 64 * 64 * 2), gb.ERR_INVALID_ARG),  # D overlaps problem 1's B
    (dict(sA=64 * 64 + 4), gb.ERR_ALIGNMENT),
    (dict(sC=12), gb.ERR_ALIGNMENT),
    (dict(sD=64 * 64 + 4), gb.ERR_ALIGNMENT),
    (dict(C=P + 8 * MB + 2, L=1), gb.ERR_ALIGNMENT),
    (dict(ldD=60), gb.ERR_INVALID_ARG),
    (dict(sC=(1 << 61) + 8), gb.ERR_INVALID_ARG),          # byte extents past 64 bits
    (dict(L=3, sD=1 << 61), gb.ERR_INVALID_ARG),
    (dict(L=1 << 30, sA=1 << 40), gb.ERR_INVALID_ARG),
])
def test_batched_argument_checks(lib, kw, status):
    assert bcall(**kw) == status


def test_batched_checks_that_pass_reach_the_device(lib):
    # Arguments that validate: without a GPU the call fails at device setup
    # (GEMM_TN_ERR_CUDA), not at an argument check.  With a GPU these calls
    # would enqueue kernels on the fake addresses, so the test runs only on
    # a host without one.
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: valid calls would launch on fake addresses")
    ok_like = {gb.OK, gb.ERR_CUDA}
    assert bcall() in ok_like
    assert bcall(beta=0.0, C=0) in ok_like                  # C unused when beta == 0
    assert bcall(alpha=0.0, A=0, B=0) in ok_like            # A, B unused when alpha == 0
    assert bcall(K=0, A=0, B=0) in ok_like                  # empty sum
    assert bcall(C=P + 12 * MB) in ok_like                  # D == C in place
    assert bcall(sA=0, sB=0, sC=0) in ok_like               # shared A, B, C
    assert bcall(L=1, sD=0, sA=8, sB=8) in ok_like          # strides unused for one problem


def test_scaled_is_one_problem(lib):
    st = gb.gemm_tn_scaled(64, 64, 64, 2.0, P, 64, 0, P + 4 * MB, 64, 0, 0.5, P + 8 * MB, 64,
                           P + 8 * MB + 64, 64, 0, None)
    assert st == gb.ERR_INVALID_ARG                          # D overlaps C
    st = gb.gemm_tn_scaled(0, 64, 64, 2.0, P, 64, 0, P + 4 * MB, 64, 0, 0.5, 0, 64, 0, 64, 0,
                           None)
    assert st == gb.OK                                       # M == 0: no-op


def test_tensor_front_end_checks_before_the_device():
    import torch
    from dense_fp16_tensor_gb300 import tensor_api
    A = torch.zeros((2, 16, 32), dtype=torch.float16)
    B = torch.zeros((3, 24, 32), dtype=torch.float16)
    with pytest.raises(ValueError, match="batch sizes disagree"):
        tensor_api.gemm_scaled(A, B)
    with pytest.raises(ValueError, match="K mismatch"):
        tensor_api.gemm_scaled(A, torch.zeros((2, 24, 16), dtype=torch.float16))
    with pytest.raises(ValueError, match="beta != 0 needs C"):
        tensor_api.gemm_scaled(A, B[:2], beta=1.0)
    with pytest.raises(TypeError, match="CUDA"):
        tensor_api.gemm_scaled(A, B[:2], out=torch.zeros((2, 16, 24), dtype=torch.float16))


def _host(M=64, N=48, K=32, alpha=1.0, A=0x10000, ldA=32, a_major=0, B=0x20000, ldB=32,
          b_major=0, beta=1.0, C=0x30000, ldC=48, D=0x40000, ldD=48, accum=0, opts=None):
    return gb.gemm_tn_host(M, N, K, alpha, A, ldA, a_major, B, ldB, b_major, beta, C, ldC, D,
                           ldD, accum, None, opts)


@pytest.mark.parametrize("kw", [
    dict(M=-1), dict(K=1 << 31), dict(a_major=2), dict(b_major=-1), dict(accum=5),
    dict(ldA=31), dict(a_major=1, ldA=63), dict(b_major=1, ldB=47), dict(ldC=47), dict(ldD=47),
    dict(D=0), dict(A=0), dict(C=0),
    dict(opts=gb.make_options(host_panel_rows=-8)), dict(opts=gb.make_options(tile_n=96)),
    # C and D overlapping other than exactly, or exactly with another ld
    dict(C=0x40000 + 2 * 48), dict(C=0x40000, ldC=56, ldD=56 + 8),
    # D overlapping A or B (D is written while later panels of A are read)
    dict(D=0x10000 + 64),
])
def test_host_entry_point_rejects_bad_arguments_before_device_work(lib, kw):
    assert _host(**kw) == gb.ERR_INVALID_ARG


def test_host_entry_point_noops(lib):
    assert _host(M=0) == gb.OK
    assert _host(N=0, D=0) == gb.OK


def test_host_front_end_argument_checks():
    import torch

    from dense_fp16_tensor_gb300 import tensor_api
    A = torch.zeros((32, 16), dtype=torch.float16)
    B = torch.zeros((24, 16), dtype=torch.float16)
    with pytest.raises(ValueError):
        tensor_api.gemm_host(A, torch.zeros((24, 8), dtype=torch.float16))   # K mismatch
    with pytest.raises(ValueError):
        tensor_api.gemm_host(A, B, beta=1.0)                                   # beta without C
    with pytest.raises(ValueError):
        tensor_api.gemm_host(A, B, torch.zeros((32, 25), dtype=torch.float16))  # C shape
    with pytest.raises(TypeError):
        tensor_api.gemm_host(A.float(), B)
    assert tensor_api._host_view(A, "A") == (gb.MAJOR_K, 16)
    assert tensor_api._host_view(A.t(), "A") == (gb.MAJOR_MN, 16)
    assert tensor_api._host_view(torch.zeros((32, 20), dtype=torch.float16)[:, :16], "A") == \
        (gb.MAJOR_K, 20)
