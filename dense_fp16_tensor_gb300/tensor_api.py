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
