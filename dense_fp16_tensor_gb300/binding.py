"""Thin ctypes binding of libgemm_tn.so (include/gemm_tn.h).

The functions keep the C names and arguments; this module only marshals
arguments.  Every step of the computation runs in the library's CUDA
kernels.  There is no fallback: if the library is missing or cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

MAJOR_K, MAJOR_MN = 0, 1
ACC_F32, ACC_F16 = 0, 1
PATH_AUTO, PATH_LARGE, PATH_SKINNY = 0, 1, 2
PATH_STRIDED_COPY, PATH_STRIDED_REPACK = 3, 4

OK = 0
ERR_INVALID_ARG = 1
ERR_ALIGNMENT = 2
ERR_UNSUPPORTED = 3
ERR_CUDA = 4
ERR_DEVICE_TIMEOUT = 5
ERR_NO_MEMORY = 6

# Every symbol declared in include/gemm_tn.h.
EXPORTED = ("gemm_tn", "gemm_tn_ex", "gemm_tn_check_device_error", "gemm_tn_plan_path",
            "gemm_tn_last_launch_count", "gemm_tn_status_string", "gemm_tn_skinny_noalloc",
            "gemm_tn_last_kernels", "gemm_tn_strided", "gemm_tn_strided_ex",
            "gemm_tn_scaled", "gemm_tn_batched", "gemm_tn_batched_ex", "gemm_tn_trace_read",
            "gemm_tn_host")

# Phase-trace record layout (gemm_tn_trace_read).
TRACE_SLOTS = 12
TRACE_CTAS = 512
TRACE_FIELDS = ("entry", "ready", "first_stage", "last_mma", "first_acc", "last_chunk",
                "stores_done", "exit", "sm", "units", "cycles_entry", "cycles_exit")

# Size of the fixed scratch array behind gemm_tn_skinny_noalloc (bytes).
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


class GemmTnOptions(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("split_k", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("sync_check", ctypes.c_int), ("timeout_ns", ctypes.c_uint64),
                ("test_stall", ctypes.c_int), ("tile_kernel", ctypes.c_int),
                ("stream_k", ctypes.c_int), ("test_fail_alloc", ctypes.c_int),
                ("k_stage", ctypes.c_int), ("trace", ctypes.c_int),
                ("host_panel_rows", ctypes.c_int), ("host_inputs_ready", ctypes.c_int)]


class GemmTnError(RuntimeError):
    def __init__(self, status: int, what: str = "gemm_tn"):
        self.status = status
        super().__init__(f"{what} failed: {gemm_tn_status_string(status)} ({status})")


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run dense_fp16_tensor_gb300.build() "
                               "(nvcc, sm_103a) first; there is no fallback path")
        L = ctypes.CDLL(path)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        gemm_args = [i64, i64, i64, vp, i64, i32, vp, i64, i32, vp, i64, i32, vp]
        L.gemm_tn.restype = i32
        L.gemm_tn.argtypes = gemm_args
        L.gemm_tn_ex.restype = i32
        L.gemm_tn_ex.argtypes = gemm_args + [ctypes.POINTER(GemmTnOptions)]
        L.gemm_tn_check_device_error.restype = i32
        L.gemm_tn_check_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        L.gemm_tn_plan_path.restype = i32
        L.gemm_tn_plan_path.argtypes = [i64, i64, i64, i32, i32]
        L.gemm_tn_last_launch_count.restype = i32
        L.gemm_tn_last_launch_count.argtypes = []
        L.gemm_tn_status_string.restype = ctypes.c_char_p
        L.gemm_tn_status_string.argtypes = [i32]
        L.gemm_tn_strided.restype = i32
        L.gemm_tn_strided.argtypes = [i64, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64, i64,
                                      i32, vp]
        L.gemm_tn_strided_ex.restype = i32
        L.gemm_tn_strided_ex.argtypes = [i64, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64,
                                         i64, i32, vp, ctypes.POINTER(GemmTnOptions)]
        L.gemm_tn_last_kernels.restype = ctypes.c_char_p
        L.gemm_tn_last_kernels.argtypes = []
        L.gemm_tn_trace_read.restype = i32
        L.gemm_tn_trace_read.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64), i32,
                                         ctypes.POINTER(ctypes.c_int)]
        L.gemm_tn_skinny_noalloc.restype = i32
        L.gemm_tn_skinny_noalloc.argtypes = gemm_args
        f32 = ctypes.c_float
        batched_args = [i64, i64, i64, i64, f32, vp, i64, i64, i32, vp, i64, i64, i32,
                        f32, vp, i64, i64, vp, i64, i64, i32, vp]
        L.gemm_tn_batched.restype = i32
        L.gemm_tn_batched.argtypes = batched_args
        L.gemm_tn_batched_ex.restype = i32
        L.gemm_tn_batched_ex.argtypes = batched_args + [ctypes.POINTER(GemmTnOptions)]
        L.gemm_tn_scaled.restype = i32
        L.gemm_tn_scaled.argtypes = [i64, i64, i64, f32, vp, i64, i32, vp, i64, i32, f32,
                                     vp, i64, vp, i64, i32, vp]
        L.gemm_tn_host.restype = i32
        L.gemm_tn_host.argtypes = [i64, i64, i64, f32, vp, i64, i32, vp, i64, i32, f32,
                                   vp, i64, vp, i64, i32, vp, ctypes.POINTER(GemmTnOptions)]
        _lib = L
        return L


def gemm_tn(M, N, K, A, ldA, a_major, B, ldB, b_major, CD, ldC, accum_dtype, stream) -> int:
    """C ``gemm_tn``: pointers and the stream are integers (device addresses,
    cudaStream_t).  Returns the gemm_tn_status."""
    return lib().gemm_tn(M, N, K, A, ldA, a_major, B, ldB, b_major, CD, ldC, accum_dtype,
                         stream)


TILE_AUTO, TILE_SINGLE, TILE_PAIR, TILE_WIDE = 0, 1, 2, 3


def make_options(path=0, split_k=0, tile_n=0, sync_check=0, timeout_ns=0, test_stall=0,
                 tile_kernel=0, stream_k=0, test_fail_alloc=0, k_stage=0, trace=0,
                 host_panel_rows=0, host_inputs_ready=0):
    return GemmTnOptions(path, split_k, tile_n, sync_check, timeout_ns, test_stall, tile_kernel,
                         stream_k, test_fail_alloc, k_stage, trace, host_panel_rows,
                         host_inputs_ready)


def gemm_tn_ex(M, N, K, A, ldA, a_major, B, ldB, b_major, CD, ldC, accum_dtype, stream,
               opts=None) -> int:
    """C ``gemm_tn_ex``; ``opts`` is a GemmTnOptions, a dict of its fields, or None."""
    if isinstance(opts, dict):
        opts = make_options(**opts)
    p = ctypes.byref(opts) if opts is not None else None
    return lib().gemm_tn_ex(M, N, K, A, ldA, a_major, B, ldB, b_major, CD, ldC, accum_dtype,
                            stream, p)


def gemm_tn_scaled(M, N, K, alpha, A, ldA, a_major, B, ldB, b_major, beta, C, ldC, D, ldD,
                   accum_dtype, stream) -> int:
    """C ``gemm_tn_scaled``: D = alpha * A.B^T + beta * C (C may be 0 when
    beta == 0)."""
    return lib().gemm_tn_scaled(M, N, K, alpha, A, ldA, a_major, B, ldB, b_major, beta, C, ldC,
                                D, ldD, accum_dtype, stream)


def gemm_tn_host(M, N, K, alpha, A, ldA, a_major, B, ldB, b_major, beta, C, ldC, D, ldD,
                 accum_dtype, stream, opts=None) -> int:
    """C ``gemm_tn_host``: the scaled form with A, B, C and D given as HOST
    addresses (page-locked memory for overlapped copies); ``opts`` as for
    :func:`gemm_tn_ex`.  The host arrays must stay untouched until the
    stream has passed the call."""
    if isinstance(opts, dict):
        opts = make_options(**opts)
    p = ctypes.byref(opts) if opts is not None else None
    return lib().gemm_tn_host(M, N, K, alpha, A, ldA, a_major, B, ldB, b_major, beta, C, ldC,
                              D, ldD, accum_dtype, stream, p)


def gemm_tn_batched(M, N, K, batch, alpha, A, ldA, strideA, a_major, B, ldB, strideB, b_major,
                    beta, C, ldC, strideC, D, ldD, strideD, accum_dtype, stream) -> int:
    """C ``gemm_tn_batched``: D_l = alpha * A_l.B_l^T + beta * C_l, operand l
    starting l * stride elements after the base pointer."""
    return lib().gemm_tn_batched(M, N, K, batch, alpha, A, ldA, strideA, a_major, B, ldB,
                                 strideB, b_major, beta, C, ldC, strideC, D, ldD, strideD,
                                 accum_dtype, stream)


def gemm_tn_batched_ex(M, N, K, batch, alpha, A, ldA, strideA, a_major, B, ldB, strideB,
                       b_major, beta, C, ldC, strideC, D, ldD, strideD, accum_dtype, stream,
                       opts=None) -> int:
    """C ``gemm_tn_batched_ex``; ``opts`` as for :func:`gemm_tn_ex`."""
    if isinstance(opts, dict):
        opts = make_options(**opts)
    p = ctypes.byref(opts) if opts is not None else None
    return lib().gemm_tn_batched_ex(M, N, K, batch, alpha, A, ldA, strideA, a_major, B, ldB,
                                    strideB, b_major, beta, C, ldC, strideC, D, ldD, strideD,
                                    accum_dtype, stream, p)


def gemm_tn_check_device_error(stream) -> tuple[int, int]:
    d = ctypes.c_uint32(0)
    s = lib().gemm_tn_check_device_error(stream, ctypes.byref(d))
    return s, d.value


def gemm_tn_trace_read(stream, max_ctas=TRACE_CTAS):
    """C ``gemm_tn_trace_read``: returns (status, records) where records is a
    list of one dict per CTA with an entry stamp (fields TRACE_FIELDS plus
    "cta")."""
    n = max(0, min(int(max_ctas), TRACE_CTAS))
    buf = (ctypes.c_uint64 * (n * TRACE_SLOTS))()
    rec = ctypes.c_int(0)
    st = lib().gemm_tn_trace_read(stream, buf, n, ctypes.byref(rec))
    out = []
    if st == OK:
        for c in range(n):
            row = buf[c * TRACE_SLOTS:(c + 1) * TRACE_SLOTS]
            if row[0]:
                d = dict(zip(TRACE_FIELDS, row))
                d["cta"] = c
                out.append(d)
    return st, out


def gemm_tn_plan_path(M, N, K, a_major, b_major) -> int:
    return lib().gemm_tn_plan_path(M, N, K, a_major, b_major)


def gemm_tn_last_launch_count() -> int:
    return lib().gemm_tn_last_launch_count()


def gemm_tn_strided(M, N, K, A, sAm, sAk, B, sBn, sBk, CD, sCm, sCn, accum_dtype,
                    stream) -> int:
    """C ``gemm_tn_strided``: operands as pointers plus element strides."""
    return lib().gemm_tn_strided(M, N, K, A, sAm, sAk, B, sBn, sBk, CD, sCm, sCn, accum_dtype,
                                 stream)


def gemm_tn_strided_ex(M, N, K, A, sAm, sAk, B, sBn, sBk, CD, sCm, sCn, accum_dtype,
                       stream, opts=None) -> int:
    """C ``gemm_tn_strided_ex``; ``opts`` as for :func:`gemm_tn_ex`."""
    if isinstance(opts, dict):
        opts = make_options(**opts)
    p = ctypes.byref(opts) if opts is not None else None
    return lib().gemm_tn_strided_ex(M, N, K, A, sAm, sAk, B, sBn, sBk, CD, sCm, sCn,
                                    accum_dtype, stream, p)


def gemm_tn_last_kernels() -> str:
    return lib().gemm_tn_last_kernels().decode()


def gemm_tn_status_string(status: int) -> str:
    return lib().gemm_tn_status_string(status).decode()


def gemm_tn_skinny_noalloc(M, N, K, A, ldA, a_major, B, ldB, b_major, CD, ldC, accum_dtype,
                           stream) -> int:
    """C ``gemm_tn_skinny_noalloc``: the skinny path (M <= 64, K-major A and B,
    fp32 accumulation) for callers that cannot have device memory allocated on
    their behalf -- latency-sensitive loops where cudaMalloc/cudaFree would
    synchronise the device, or processes whose allocator already holds nearly
    all device memory.  Its partial sums live in a fixed 16 MiB array inside
    the library instead of a cudaMalloc'd workspace; larger problems are
    rejected with GEMM_TN_ERR_INVALID_ARG.  Calls that overlap on the GPU share
    that array and race.  Returns the gemm_tn_status."""
    return lib().gemm_tn_skinny_noalloc(M, N, K, A, ldA, a_major, B, ldB, b_major, CD, ldC,
                                        accum_dtype, stream)
