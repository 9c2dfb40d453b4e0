"""Shared helpers of the parity tests: the acceptance tolerances and a call of
the GPU path through the C ABI on stored operands.

Tolerances (the acceptance bar for this GEMM):
  * integer-valued inputs:            bit-exact against the oracle's
                                      round-to-nearest-even fp16 result
  * fp32 accumulation:                |d - ref| <= 1e-2 + 2^-9 |ref|
  * fp16 accumulation, real values:   |d - ref| <= 2^-7 sqrt(K/16) max(1, |ref|)
ref is the oracle's exact fp64 value.
"""
import math

import numpy as np

ACC_F32, ACC_F16 = 0, 1


def tol(ref: np.ndarray, K: int, accum: int) -> np.ndarray:
    a = np.abs(ref)
    if accum == ACC_F32:
        return 1e-2 + 2.0 ** -9 * a
    return 2.0 ** -7 * math.sqrt(max(K, 1) / 16) * np.maximum(1.0, a)


def check(d16: np.ndarray, ref64: np.ndarray, ref16: np.ndarray | None, K: int, accum: int,
          exact: bool, what: str = ""):
    """Assert parity of the GPU fp16 result d16 (uint16 bits or float16)."""
    d16 = np.asarray(d16)
    if d16.dtype == np.float16:
        d16 = d16.view(np.uint16)
    if exact:
        assert ref16 is not None
        bad = np.flatnonzero(d16.reshape(-1) != ref16.reshape(-1))
        assert bad.size == 0, (f"{what}: {bad.size} elements differ bit-wise, first at flat "
                               f"{bad[:5].tolist()}: got {d16.reshape(-1)[bad[:5]].view(np.float16)} "
                               f"want {ref16.reshape(-1)[bad[:5]].view(np.float16)}")
        return 0.0
    d = d16.view(np.float16).astype(np.float64)
    assert np.all(np.isfinite(d)), f"{what}: non-finite values in D"
    err = np.abs(d - ref64)
    t = tol(ref64, K, accum)
    bad = np.flatnonzero((err > t).reshape(-1))
    assert bad.size == 0, (f"{what}: {bad.size} elements out of tolerance; worst err "
                           f"{err.max():.3e}, first flat {bad[:5].tolist()}")
    return float((err / t).max()) if err.size else 0.0


def np_bits(t):
    """uint16 numpy view of a CPU fp16 torch tensor."""
    return t.contiguous().view(__import__("torch").int16).numpy().view(np.uint16)
