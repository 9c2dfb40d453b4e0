"""CPU oracle for the fp16 TN GEMM  D(m,n) = C(m,n) + sum_k A(m,k) * B(n,k).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
never imports it, and it imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain C, fp64): a shape:stride layout
evaluator, an IEEE binary16 codec and the triple loop.  This module only
builds that file with gcc, marshals numpy arrays into it, and adds one
library route for full-size checks:

* ``gemm_tn_blas`` -- the same definition with float64 BLAS matmul as its
  one step (used where the triple loop would take minutes, e.g. 8192^3).

``gemm_tn_general`` is the scaled, batched form D = alpha A.B^T + beta C over
a batch of (ld, major) views ("cute(7) simple_gemm", section 8.1's cuBLAS
call and section 4's extra modes), with the BLAS conventions for alpha == 0
and beta == 0.

Operand convention ("Reading CuTe's make_tiled_mma", section "Fix the
matrices and directions first"): A is (M,K), B is (N,K), C/D are (M,N) and
D(m,n) = C(m,n) + sum_k A(m,k) B(n,k).  Memory views ("CuTe Layout to Tensor
Core", sections 1-2): an operand whose K mode is contiguous is
(rows,K):(ld,1); one whose M (or N) mode is contiguous is (rows,K):(1,ld).

Pins: every function here is checked against values printed on the pages,
closed forms, invariants or library routines in ``tests/test_oracle_*.py``;
no function is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

MAJOR_K = 0
MAJOR_MN = 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no GPU, no CUDA)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-fvisibility=hidden", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, i32 = ctypes.c_int64, ctypes.c_int
        vp = ctypes.c_void_p
        lib.oracle_layout_offset.restype = i64
        lib.oracle_layout_offset.argtypes = [i32, vp, vp, i32, vp, vp]
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_double_to_half_rne.restype = ctypes.c_uint16
        lib.oracle_double_to_half_rne.argtypes = [ctypes.c_double]
        lib.oracle_gemm_tn.restype = i32
        lib.oracle_gemm_tn.argtypes = [i64, i64, i64, vp, i64, i32, vp, i64, i32,
                                       vp, i64, vp, vp, i32]
        lib.oracle_gemm_tn_strided.restype = i32
        lib.oracle_gemm_tn_strided.argtypes = [i64, i64, i64, vp, i64, i64, vp, i64, i64,
                                               vp, i64, i64, vp, vp, i32]
        lib.oracle_gemm_tn_sampled.restype = i32
        lib.oracle_gemm_tn_sampled.argtypes = [i64, i64, i64, vp, i64, i32, vp, i64,
                                               i32, vp, i64, i64, vp, vp, vp, vp, i32]
        lib.oracle_gemm_tn_general.restype = i32
        lib.oracle_gemm_tn_general.argtypes = [i64, i64, i64, i64, ctypes.c_double,
                                               vp, i64, i64, i64, vp, i64, i64, i64,
                                               ctypes.c_double, vp, i64, i64, i64,
                                               vp, vp, i32]
        _lib = lib
        return lib


# --------------------------------------------------------------------------
# Layouts
# --------------------------------------------------------------------------

def _flatten(x):
    if isinstance(x, (tuple, list)):
        out = []
        for e in x:
            out.extend(_flatten(e))
        return out
    return [int(x)]


def layout_offset(shape, stride, coord) -> int:
    """Evaluate the shape:stride layout at ``coord``.

    ``shape``/``stride`` are nested tuples of equal structure.  ``coord`` is
    either one integer (decoded over the whole shape, first mode fastest) or
    a tuple with one integer per top-level mode (each decoded over that mode's
    own, possibly nested, shape).  Raises ValueError when out of range.
    """
    lib = _load()
    if isinstance(shape, (tuple, list)):
        top_shapes = list(shape)
        top_strides = list(stride)
    else:
        top_shapes, top_strides = [shape], [stride]
    flat_shape, flat_stride, mode_len = [], [], []
    for s, d in zip(top_shapes, top_strides):
        fs, fd = _flatten(s), _flatten(d)
        if len(fs) != len(fd):
            raise ValueError("shape and stride differ in structure")
        flat_shape += fs
        flat_stride += fd
        mode_len.append(len(fs))
    if isinstance(coord, (tuple, list)):
        coords = [int(c) for c in coord]
        if len(coords) != len(mode_len):
            raise ValueError("coordinate rank does not match the layout")
    else:
        coords = [int(coord)]
        mode_len = [len(flat_shape)]
    a_shape = (ctypes.c_int64 * len(flat_shape))(*flat_shape)
    a_stride = (ctypes.c_int64 * len(flat_stride))(*flat_stride)
    a_len = (ctypes.c_int * len(mode_len))(*mode_len)
    a_coord = (ctypes.c_int64 * len(coords))(*coords)
    off = lib.oracle_layout_offset(len(flat_shape), a_shape, a_stride,
                                   len(mode_len), a_len, a_coord)
    if off < 0:
        raise ValueError(f"coordinate {coord} outside layout {shape}:{stride}")
    return int(off)


def layout_size(shape) -> int:
    n = 1
    for s in _flatten(shape):
        n *= s
    return n


# --------------------------------------------------------------------------
# binary16 codec
# --------------------------------------------------------------------------

def half_to_double(bits: int) -> float:
    return float(_load().oracle_half_to_double(int(bits) & 0xFFFF))


def double_to_half(x: float) -> int:
    return int(_load().oracle_double_to_half_rne(float(x)))


# --------------------------------------------------------------------------
# GEMM
# --------------------------------------------------------------------------

def _bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError("operands are raw binary16: pass float16 or uint16 arrays")
    return x


def _ptr(x):
    return None if x is None else x.ctypes.data


def default_threads() -> int:
    return os.cpu_count() or 1


def gemm_tn(M, N, K, A, ldA, a_major, B, ldB, b_major, C=None, ldC=None,
            want_f16=True, nthreads=None):
    """Full D = C + A.B^T by the triple loop.

    ``A``, ``B``, ``C`` are flat (or any-shape, contiguous) float16/uint16
    arrays holding the operands' storage; the views are formed from
    (ld, major) as in the module docstring.  Returns ``(d64, d16bits)``:
    d64 is the exact fp64 value (M,N), d16bits its binary16 round-to-nearest-
    even bit pattern (or None).
    """
    lib = _load()
    A, B = _bits(A), _bits(B)
    C = None if C is None else _bits(C)
    _check_extent(M, K, A, ldA, a_major, "A")
    _check_extent(N, K, B, ldB, b_major, "B")
    if C is not None:
        ldC = N if ldC is None else ldC
        _check_extent(M, N, C, ldC, MAJOR_K, "C")
    d64 = np.empty((M, N), np.float64)
    d16 = np.empty((M, N), np.uint16) if want_f16 else None
    lib.oracle_gemm_tn(M, N, K, _ptr(A), ldA, a_major, _ptr(B), ldB, b_major,
                       _ptr(C), ldC or 0, _ptr(d64), _ptr(d16),
                       nthreads or default_threads())
    return d64, d16


def _check_strided(rows, cols, X, s_r, s_c, name):
    if rows == 0 or cols == 0:
        return
    if s_r < 0 or s_c < 0:
        raise ValueError(f"{name}: negative strides are not supported")
    need = (rows - 1) * s_r + (cols - 1) * s_c + 1
    if X.size < need:
        raise ValueError(f"{name}: storage holds {X.size} elements, view needs {need}")


def gemm_tn_strided(M, N, K, A, sAm, sAk, B, sBn, sBk, C=None, sCm=0, sCn=1, want_f16=True,
                    nthreads=None):
    """Full D = C + A.B^T over arbitrary element strides:
    A(m,k) = A[m*sAm + k*sAk], B(n,k) = B[n*sBn + k*sBk], C(m,n) = C[m*sCm + n*sCn].
    Returns ``(d64, d16bits)`` like :func:`gemm_tn`."""
    lib = _load()
    A, B = _bits(A), _bits(B)
    C = None if C is None else _bits(C)
    _check_strided(M, K, A, sAm, sAk, "A")
    _check_strided(N, K, B, sBn, sBk, "B")
    if C is not None:
        _check_strided(M, N, C, sCm, sCn, "C")
    d64 = np.empty((M, N), np.float64)
    d16 = np.empty((M, N), np.uint16) if want_f16 else None
    lib.oracle_gemm_tn_strided(M, N, K, _ptr(A), sAm, sAk, _ptr(B), sBn, sBk, _ptr(C), sCm,
                               sCn, _ptr(d64), _ptr(d16), nthreads or default_threads())
    return d64, d16


def gemm_tn_sampled(M, N, K, A, ldA, a_major, B, ldB, b_major, C, ldC,
                    rows, cols, nthreads=None):
    """D at the listed (rows[s], cols[s]) positions; returns (d64, d16bits)."""
    lib = _load()
    A, B = _bits(A), _bits(B)
    C = None if C is None else _bits(C)
    _check_extent(M, K, A, ldA, a_major, "A")
    _check_extent(N, K, B, ldB, b_major, "B")
    if C is not None:
        _check_extent(M, N, C, ldC, MAJOR_K, "C")
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape or rows.ndim != 1:
        raise ValueError("rows/cols must be equal-length 1-D")
    if len(rows) and (rows.min() < 0 or rows.max() >= M or cols.min() < 0 or cols.max() >= N):
        raise ValueError("sample outside D")
    d64 = np.empty(len(rows), np.float64)
    d16 = np.empty(len(rows), np.uint16)
    lib.oracle_gemm_tn_sampled(M, N, K, _ptr(A), ldA, a_major, _ptr(B), ldB, b_major,
                               _ptr(C), ldC or 0, len(rows), _ptr(rows), _ptr(cols),
                               _ptr(d64), _ptr(d16), nthreads or default_threads())
    return d64, d16


def gemm_tn_general(M, N, K, alpha, A, ldA, a_major, B, ldB, b_major, beta, C=None,
                    ldC=None, batch=1, strideA=0, strideB=0, strideC=0, want_f16=True,
                    nthreads=None):
    """D(l) = alpha * A(l).B(l)^T + beta * C(l) for l < batch.

    Operand l's view is the (ld, major) view of the storage starting at
    element l * stride (a stride may be 0: the operand is shared).  alpha == 0
    leaves A and B unread, beta == 0 leaves C unread (C may be None).
    Returns ``(d64, d16bits)`` of shape (batch, M, N)."""
    lib = _load()
    A, B = _bits(A).reshape(-1), _bits(B).reshape(-1)
    C = None if C is None else _bits(C).reshape(-1)
    if beta != 0 and C is None:
        raise ValueError("beta != 0 needs C")
    vA = (ldA, 1) if a_major == MAJOR_K else (1, ldA)
    vB = (ldB, 1) if b_major == MAJOR_K else (1, ldB)
    ldC = N if ldC is None else ldC
    for l in (0, batch - 1) if batch > 0 else ():
        if alpha != 0:
            _check_strided(M, K, A[l * strideA:], vA[0], vA[1], "A")
            _check_strided(N, K, B[l * strideB:], vB[0], vB[1], "B")
        if beta != 0:
            _check_strided(M, N, C[l * strideC:], ldC, 1, "C")
    d64 = np.empty((batch, M, N), np.float64)
    d16 = np.empty((batch, M, N), np.uint16) if want_f16 else None
    lib.oracle_gemm_tn_general(M, N, K, batch, float(alpha),
                               _ptr(A), vA[0], vA[1], strideA,
                               _ptr(B), vB[0], vB[1], strideB,
                               float(beta), _ptr(C), ldC, 1, strideC,
                               _ptr(d64), _ptr(d16), nthreads or default_threads())
    return d64, d16


def _check_extent(rows, cols, X, ld, major, name):
    """The storage must cover the view: cosize of (rows,cols):(ld,1) or (1,ld)."""
    if rows == 0 or cols == 0:
        return
    inner = cols if major == MAJOR_K else rows
    outer = rows if major == MAJOR_K else cols
    if ld < inner:
        raise ValueError(f"{name}: ld={ld} < contiguous extent {inner}")
    need = (outer - 1) * ld + inner
    if X.size < need:
        raise ValueError(f"{name}: storage holds {X.size} elements, view needs {need}")


def view(X, rows, cols, ld, major) -> np.ndarray:
    """The (rows, cols) logical view of flat storage X as float64 (exact)."""
    X = _bits(X).reshape(-1).view(np.float16)
    _check_extent(rows, cols, X, ld, major, "view")
    es = X.itemsize
    strides = (ld * es, es) if major == MAJOR_K else (es, ld * es)
    v = np.lib.stride_tricks.as_strided(X, shape=(rows, cols), strides=strides,
                                        writeable=False)
    return v.astype(np.float64)


def gemm_tn_blas(M, N, K, A, ldA, a_major, B, ldB, b_major, C=None, ldC=None):
    """D = C + A.B^T in float64 with a BLAS matmul as the one step.

    Used for full-size checks where the triple loop would take minutes; it
    agrees with ``gemm_tn`` to fp64 rounding (pinned in the tests).
    """
    a = view(A, M, K, ldA, a_major)
    b = view(B, N, K, ldB, b_major)
    d = a @ b.T
    if C is not None:
        d += view(C, M, N, ldC if ldC is not None else N, MAJOR_K)
    return d
