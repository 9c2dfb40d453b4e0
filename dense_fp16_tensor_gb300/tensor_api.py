"""torch-tensor front end of gemm_tn: reads pointers, strides and the current
stream from torch tensors and calls the C ABI.  torch provides device memory
and streams only."""
from __future__ import annotations

import torch

from . import binding as B

_ACC = {"f32": B.ACC_F32, "fp32": B.ACC_F32, "float32": B.ACC_F32,
        "f16": B.ACC_F16, "fp16": B.ACC_F16, "float16": B.ACC_F16}


def _round8(x: int) -> int:
    return (x + 7) // 8 * 8


def operand_view(t: torch.Tensor, name: str):
    """(major, ld) for a 2-D fp16 view (rows, K) with one stride-1 mode.

    K-major when the K mode is stride-1: (rows,K):(ld,1); MN-major when the
    rows mode is: (rows,K):(1,ld).  A mode of size one may take any stride,
    so the candidate whose leading dimension is legal is chosen.
    """
    if t.dim() != 2 or t.dtype != torch.float16:
        raise TypeError(f"{name} must be a 2-D float16 tensor")
    rows, k = t.shape
    s0, s1 = t.stride()
    cands = []
    if s1 == 1 or k == 1:
        cands.append((B.MAJOR_K, s0 if rows > 1 else _round8(k), k))
    if s0 == 1 or rows == 1:
        cands.append((B.MAJOR_MN, s1 if k > 1 else _round8(rows), rows))
    for major, ld, inner in cands:
        if ld >= inner and ld % 8 == 0:
            return major, ld
    if cands:
        return cands[0][0], cands[0][1]
    raise ValueError(f"{name}: neither mode is stride-1 (strides {t.stride()})")


def gemm(A: torch.Tensor, Bm: torch.Tensor, CD: torch.Tensor, accum: str = "f32",
         stream: torch.cuda.Stream | None = None, **options) -> torch.Tensor:
    """CD <- CD + A . Bm^T in place (A (M,K), Bm (N,K), CD (M,N), all fp16 CUDA).

    Raises GemmTnError on a non-OK status.  ``options`` are gemm_tn_options
    fields (path, split_k, tile_n, sync_check, timeout_ns).
    """
    M, K = A.shape
    N, K2 = Bm.shape
    if K2 != K or tuple(CD.shape) != (M, N):
        raise ValueError(f"shape mismatch: A {tuple(A.shape)}, B {tuple(Bm.shape)}, CD {tuple(CD.shape)}")
    if CD.dtype != torch.float16 or CD.dim() != 2:
        raise TypeError("CD must be a 2-D float16 tensor")
    if not (A.is_cuda and Bm.is_cuda and CD.is_cuda):
        raise ValueError("A, B and CD must be CUDA tensors")
    if CD.stride(1) != 1 and N > 1:
        raise ValueError("CD must be row-major (stride-1 N mode)")
    a_major, ldA = operand_view(A, "A")
    b_major, ldB = operand_view(Bm, "B")
    ldC = CD.stride(0) if M > 1 else _round8(N)
    s = stream if stream is not None else torch.cuda.current_stream(CD.device)
    acc = _ACC[accum] if isinstance(accum, str) else int(accum)
    args = (M, N, K, A.data_ptr(), ldA, a_major, Bm.data_ptr(), ldB, b_major,
            CD.data_ptr(), ldC, acc, s.cuda_stream)
    if options:
        st = B.gemm_tn_ex(*args, opts=options)
    else:
        st = B.gemm_tn(*args)
    if st != B.OK:
        raise B.GemmTnError(st)
    return CD


def _per_problem(t: torch.Tensor | None, name: str):
    """(2-D view of problem 0, batch stride, batch size or None) of a 2-D or 3-D tensor."""
    if t is None:
        return None, 0, None
    if t.dim() == 3:
        return t[0], t.stride(0) if t.shape[0] > 1 else 0, t.shape[0]
    if t.dim() == 2:
        return t, 0, None
    raise TypeError(f"{name} must be 2-D or 3-D")


def gemm_scaled(A: torch.Tensor, Bm: torch.Tensor, C: torch.Tensor | None = None, *,
                alpha: float = 1.0, beta: float | None = None, out: torch.Tensor | None = None,
                accum: str = "f32", stream: torch.cuda.Stream | None = None,
                **options) -> torch.Tensor:
    """out <- alpha * A . Bm^T + beta * C (gemm_tn_batched).

    2-D operands are one problem: A (M,K), Bm (N,K), C and out (M,N).  Any
    3-D operand makes a batch: A (L,M,K), Bm (L,N,K), C and out (L,M,N); a
    2-D operand (or a 3-D one expanded along the batch, stride 0) is shared
    by every problem.  beta defaults to 1 with C and 0 without; out is
    allocated when not given (and may be C itself, for in place).
    """
    A2, sA, LA = _per_problem(A, "A")
    B2, sB, LB = _per_problem(Bm, "B")
    C2, sC, LC = _per_problem(C, "C")
    O2, sO, LO = _per_problem(out, "out")
    sizes = {x for x in (LA, LB, LC, LO) if x is not None}
    if len(sizes) > 1:
        raise ValueError(f"batch sizes disagree: {sorted(sizes)}")
    L = sizes.pop() if sizes else None
    M, K = A2.shape
    N, K2 = B2.shape
    if K2 != K:
        raise ValueError(f"K mismatch: A {tuple(A.shape)}, B {tuple(Bm.shape)}")
    if beta is None:
        beta = 1.0 if C is not None else 0.0
    if beta != 0 and C is None:
        raise ValueError("beta != 0 needs C")
    if out is None:
        shape = (L, M, N) if L is not None else (M, N)
        out = torch.empty(shape, dtype=torch.float16, device=A.device)
        O2, sO, _ = _per_problem(out, "out")
    for t, name in ((A, "A"), (Bm, "B"), (C, "C"), (out, "out")):
        if t is not None and (t.dtype != torch.float16 or not t.is_cuda):
            raise TypeError(f"{name} must be a float16 CUDA tensor")
    for t2, name in ((C2, "C"), (O2, "out")):
        if t2 is not None and (tuple(t2.shape) != (M, N) or (t2.stride(1) != 1 and N > 1)):
            raise ValueError(f"{name} must be (M, N) row-major per problem")
    a_major, ldA = operand_view(A2, "A")
    b_major, ldB = operand_view(B2, "B")
    ldC = (C2.stride(0) if M > 1 else _round8(N)) if C2 is not None else N
    ldD = O2.stride(0) if M > 1 else _round8(N)
    s = stream if stream is not None else torch.cuda.current_stream(out.device)
    acc = _ACC[accum] if isinstance(accum, str) else int(accum)
    st = B.gemm_tn_batched_ex(M, N, K, L if L is not None else 1, float(alpha), A2.data_ptr(),
                              ldA, sA, a_major, B2.data_ptr(), ldB, sB, b_major, float(beta),
                              C2.data_ptr() if C2 is not None else 0, ldC, sC, O2.data_ptr(),
                              ldD, sO, acc, s.cuda_stream, options or None)
    if st != B.OK:
        raise B.GemmTnError(st)
    return out


def _host_view(t: torch.Tensor, name: str):
    """(major, ld) of a 2-D fp16 host operand (rows, K): any leading dimension
    at least its row, one stride-1 mode."""
    if t.dim() != 2 or t.dtype != torch.float16:
        raise TypeError(f"{name} must be a 2-D float16 tensor")
    rows, k = t.shape
    s0, s1 = t.stride()
    if s1 == 1 or k == 1:
        return B.MAJOR_K, max(s0, k) if rows > 1 else max(k, 1)
    if s0 == 1 or rows == 1:
        return B.MAJOR_MN, max(s1, rows) if k > 1 else max(rows, 1)
    raise ValueError(f"{name}: neither mode is stride-1 (strides {t.stride()})")


def gemm_host(A: torch.Tensor, Bm: torch.Tensor, C: torch.Tensor | None = None, *,
              alpha: float = 1.0, beta: float | None = None, out: torch.Tensor | None = None,
              accum: str = "f32", stream: torch.cuda.Stream | None = None,
              synchronize: bool = True, **options) -> torch.Tensor:
    """out <- alpha * A . Bm^T + beta * C with every tensor in host memory
    (gemm_tn_host): A (M,K), Bm (N,K), C and out (M,N) fp16 CPU tensors,
    page-locked (``pin_memory()``) for the copies to overlap the GEMMs.  out
    is allocated (page-locked) when not given and may be C itself.  The
    copies and GEMMs are enqueued on ``stream`` (default: the current
    stream); with ``synchronize`` (default) the call waits for them, else
    the caller must synchronise the stream before reading out or touching
    the inputs.  ``options`` are gemm_tn_options fields (host_panel_rows,
    tile_kernel, ...)."""
    if A.is_cuda or Bm.is_cuda or (C is not None and C.is_cuda) or \
            (out is not None and out.is_cuda):
        raise ValueError("gemm_host takes CPU tensors (use gemm / gemm_scaled on CUDA tensors)")
    M, K = A.shape
    N, K2 = Bm.shape
    if K2 != K:
        raise ValueError(f"K mismatch: A {tuple(A.shape)}, B {tuple(Bm.shape)}")
    if beta is None:
        beta = 1.0 if C is not None else 0.0
    if beta != 0 and C is None:
        raise ValueError("beta != 0 needs C")
    a_major, ldA = _host_view(A, "A")
    b_major, ldB = _host_view(Bm, "B")

    def check_mn(t, name):
        if t is not None and (t.dtype != torch.float16 or tuple(t.shape) != (M, N) or
                              (t.stride(1) != 1 and N > 1)):
            raise ValueError(f"{name} must be an (M, N) row-major float16 tensor")
    check_mn(C, "C")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16).pin_memory()
    check_mn(out, "out")
    ldC = max(C.stride(0), N) if C is not None and M > 1 else N
    ldD = max(out.stride(0), N) if M > 1 else N
    s = stream if stream is not None else torch.cuda.current_stream()
    acc = _ACC[accum] if isinstance(accum, str) else int(accum)
    st = B.gemm_tn_host(M, N, K, float(alpha), A.data_ptr(), ldA, a_major, Bm.data_ptr(), ldB,
                        b_major, float(beta), C.data_ptr() if C is not None else 0, ldC,
                        out.data_ptr(), ldD, acc, s.cuda_stream, options or None)
    if st != B.OK:
        raise B.GemmTnError(st, "gemm_tn_host")
    if synchronize:
        s.synchronize()
    return out
