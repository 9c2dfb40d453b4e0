// scale.cuh -- D = beta * C without a product term, sm_103a.
//
// When alpha == 0 or K == 0 the product term of D = alpha * A.B^T + beta * C
// is absent (an empty sum; A and B are not read), and the result is beta * C
// rounded to fp16, or zero when beta == 0 (C not read).  One thread writes 8
// consecutive columns of one row of one problem, with 16-byte accesses where
// the row has 8 more columns; the grid strides over (problem, row, group).
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace gemm_tn_dev {

constexpr int kScaleThreads = 256;

__global__ void __launch_bounds__(kScaleThreads)
    gemm_tn_scale_kernel(int M, int N, int L, const EpiArgs e) {
  const int64_t groups = (N + 7) / 8;
  const int64_t total = static_cast<int64_t>(L) * M * groups;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t lm = i / groups;
    const int n = static_cast<int>(i - lm * groups) * 8;
    const int64_t l = lm / M, m = lm - l * M;
    const __half* c = e.read_c ? e.C + l * e.sC + m * e.ldC + n : nullptr;
    __half* d = e.D + l * e.sD + m * e.ldD + n;
    if (n + 8 <= N) {
      uint4 cv = make_uint4(0u, 0u, 0u, 0u);
      if (e.read_c) cv = *reinterpret_cast<const uint4*>(c);
      const __half2* ch = reinterpret_cast<const __half2*>(&cv);
      uint4 o;
      __half2* oh = reinterpret_cast<__half2*>(&o);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 cf = __half22float2(ch[j]);
        oh[j] = __floats2half2_rn(e.beta * cf.x, e.beta * cf.y);
      }
      *reinterpret_cast<uint4*>(d) = o;
    } else {
      for (int j = 0; n + j < N; ++j)
        d[j] = __float2half_rn(e.read_c ? e.beta * __half2float(c[j]) : 0.f);
    }
  }
}

}  // namespace gemm_tn_dev
