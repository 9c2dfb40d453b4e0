"""Seeded synthetic inputs for the TN GEMM workloads.

This module only draws numbers and lays them out in memory; it holds none of
the GEMM's arithmetic, and both the oracle-side tests and the GPU side take
their inputs from it.  Values are drawn on the CPU with a seeded
``torch.Generator`` in fp32 and rounded to fp16 (round to nearest even), so
both sides see identical bits.

Seeds: A = 1000 + index, B = 2000 + index, C = 3000 + index, sample
positions = 4000 + index, where index is the workload's number below.
Values are drawn in storage order (row by row of the stored array), and any
leading-dimension slack is filled with NaN so that a read outside the
logical view shows up in D.

Workloads (sizes, majors and value distributions):
  1 tiny        M=32 N=16 K=16, A,B K-major (ld 16), C=0, U[-1,1], fp32 acc
  1 tiny_int    same shapes, values in {-2..2}: exact
  2 square1024  M=N=K=1024, K-major ld=1024, A,B in {-1,0,1}, C in {-4..4},
                fp16 accumulation: exact
  3 ragged      M=4000 N=3000 K=2500, A M-major (M,K):(1,4096), B K-major
                (N,K):(2504,1), CD ld=3000, A,B,C U[-1,1], fp32 acc
  4 skinny      M=16 N=K=16384, K-major, A ~ N(0,1), B ~ N(0,1/K), C=0, fp32 acc
  5 large       M=N=K=8192, K-major, U[-1,1], C=0, fp32 acc
"""
from __future__ import annotations

import dataclasses
import math

import torch

MAJOR_K, MAJOR_MN = 0, 1
ACC_F32, ACC_F16 = 0, 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    M: int
    N: int
    K: int
    a_major: int
    ldA: int
    b_major: int
    ldB: int
    ldC: int
    accum: int
    a_dist: str
    b_dist: str
    c_dist: str
    exact: bool = False  # integer-valued inputs: the result must be bit-exact

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def min_bytes(self) -> int:
        """Algorithmic HBM bytes: A and B read once, C read once, D written once."""
        return 2 * (self.M * self.K + self.N * self.K + 2 * self.M * self.N)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny", 1, 32, 16, 16, MAJOR_K, 16, MAJOR_K, 16, 16, ACC_F32,
                 "u11", "u11", "zero"),
        Workload("tiny_int", 1, 32, 16, 16, MAJOR_K, 16, MAJOR_K, 16, 16, ACC_F32,
                 "int2", "int2", "zero", exact=True),
        Workload("square1024", 2, 1024, 1024, 1024, MAJOR_K, 1024, MAJOR_K, 1024, 1024, ACC_F16,
                 "int1", "int1", "int4", exact=True),
        Workload("ragged", 3, 4000, 3000, 2500, MAJOR_MN, 4096, MAJOR_K, 2504, 3000, ACC_F32,
                 "u11", "u11", "u11"),
        Workload("skinny", 4, 16, 16384, 16384, MAJOR_K, 16384, MAJOR_K, 16384, 16384, ACC_F32,
                 "normal", "normal_k", "zero"),
        Workload("large", 5, 8192, 8192, 8192, MAJOR_K, 8192, MAJOR_K, 8192, 8192, ACC_F32,
                 "u11", "u11", "zero"),
    ]
}


def storage_shape(rows: int, cols: int, ld: int, major: int) -> tuple[int, int]:
    """Shape of the stored 2-D array of a (rows, cols) view: (rows, ld) when
    the cols mode is contiguous, (cols, ld) when the rows mode is."""
    return (rows, ld) if major == MAJOR_K else (cols, ld)


def draw(shape, dist: str, seed: int, K: int = 1) -> torch.Tensor:
    """fp16 values of the named distribution, drawn in fp32 on the CPU."""
    g = torch.Generator().manual_seed(seed)
    n = math.prod(shape)
    if dist == "zero":
        x = torch.zeros(n)
    elif dist == "u11":
        x = torch.rand(n, generator=g) * 2 - 1
    elif dist == "normal":
        x = torch.randn(n, generator=g)
    elif dist == "normal_k":
        x = torch.randn(n, generator=g) * (1.0 / math.sqrt(K))
    elif dist.startswith("int"):
        r = int(dist[3:])
        x = torch.randint(-r, r + 1, (n,), generator=g).float()
    else:
        raise ValueError(dist)
    return x.reshape(shape).half()


def operand(rows: int, cols: int, ld: int, major: int, dist: str, seed: int,
            K: int = 1, poison: bool = True) -> torch.Tensor:
    """Stored array of a (rows, cols) operand; slack beyond the view is NaN."""
    outer, _ = storage_shape(rows, cols, ld, major)
    inner = cols if major == MAJOR_K else rows
    vals = draw((outer, inner), dist, seed, K)
    if ld == inner:
        return vals
    st = torch.full((outer, ld), float("nan") if poison else 0.0, dtype=torch.float16)
    st[:, :inner] = vals
    return st


def batched_operand(L: int, rows: int, cols: int, ld: int, major: int, stride: int, dist: str,
                    seed: int, K: int = 1, poison: bool = True) -> torch.Tensor:
    """Flat storage of L (rows, cols) operands, operand l at element l * stride
    (stride 0: one operand shared by all).  Slack and gaps are NaN."""
    outer, _ = storage_shape(rows, cols, ld, major)
    per = outer * ld
    n = max(per, (L - 1) * stride + per) if L > 0 else per
    st = torch.full((n,), float("nan") if poison else 0.0, dtype=torch.float16)
    for l in range(L if stride else 1):
        st[l * stride:l * stride + per] = operand(rows, cols, ld, major, dist, seed + 7919 * l, K,
                                                 poison).reshape(-1)
    return st


def view(storage: torch.Tensor, rows: int, cols: int, ld: int, major: int) -> torch.Tensor:
    """The logical (rows, cols) view of a stored operand (no copy)."""
    strides = (ld, 1) if major == MAJOR_K else (1, ld)
    return storage.as_strided((rows, cols), strides)


def make_inputs(w: Workload):
    """CPU fp16 storage for A, B and C/D of workload ``w``: (A_st, B_st, CD_st)."""
    A = operand(w.M, w.K, w.ldA, w.a_major, w.a_dist, 1000 + w.index, w.K)
    B = operand(w.N, w.K, w.ldB, w.b_major, w.b_dist, 2000 + w.index, w.K)
    C = operand(w.M, w.N, w.ldC, MAJOR_K, w.c_dist, 3000 + w.index, w.K)
    return A, B, C


def sample_positions(w: Workload, count: int = 1024):
    """Seeded output positions (rows, cols) for sampled checks."""
    g = torch.Generator().manual_seed(4000 + w.index)
    rows = torch.randint(0, w.M, (count,), generator=g)
    cols = torch.randint(0, w.N, (count,), generator=g)
    return rows, cols
