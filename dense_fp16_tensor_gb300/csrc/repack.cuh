// repack.cuh -- copy between two strided 2-D fp16 views.
//
//   dst(r,c) = src(r,c)   for r < rows, c < cols
//   src(r,c) = src[r*s_sr + c*s_sc],  dst(r,c) = dst[r*s_dr + c*s_dc]
//
// Used by the general-stride GEMM to turn an operand view that TMA cannot
// describe into a row-major buffer it can (and to scatter D back).  Each
// block moves one 64 x 64 tile through shared memory: it reads with
// consecutive threads along the source's unit-stride mode (or along columns
// when neither mode has unit stride) and writes with consecutive threads
// along the destination's, so both sides are coalesced for the usual layouts.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

namespace gemm_tn_dev {

constexpr int kRepackTile = 64;
constexpr int kRepackThreads = 256;

__global__ void __launch_bounds__(kRepackThreads)
    repack2d_kernel(const __half* __restrict__ src, int64_t s_sr, int64_t s_sc,
                    __half* __restrict__ dst, int64_t s_dr, int64_t s_dc, int rows, int cols) {
  __shared__ unsigned short tile[kRepackTile][kRepackTile + 2];
  const int r0 = static_cast<int>(blockIdx.y) * kRepackTile;
  const int c0 = static_cast<int>(blockIdx.x) * kRepackTile;
  const unsigned short* s = reinterpret_cast<const unsigned short*>(src);
  unsigned short* d = reinterpret_cast<unsigned short*>(dst);
  const bool src_rows_fast = (s_sr == 1 && s_sc != 1);  // consecutive threads along r
  const bool dst_rows_fast = (s_dr == 1 && s_dc != 1);
  for (int i = threadIdx.x; i < kRepackTile * kRepackTile; i += kRepackThreads) {
    const int a = i % kRepackTile, b = i / kRepackTile;
    const int r = src_rows_fast ? a : b, c = src_rows_fast ? b : a;
    const int gr = r0 + r, gc = c0 + c;
    if (gr < rows && gc < cols)
      tile[r][c] = s[static_cast<int64_t>(gr) * s_sr + static_cast<int64_t>(gc) * s_sc];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kRepackTile * kRepackTile; i += kRepackThreads) {
    const int a = i % kRepackTile, b = i / kRepackTile;
    const int r = dst_rows_fast ? a : b, c = dst_rows_fast ? b : a;
    const int gr = r0 + r, gc = c0 + c;
    if (gr < rows && gc < cols)
      d[static_cast<int64_t>(gr) * s_dr + static_cast<int64_t>(gc) * s_dc] = tile[r][c];
  }
}

// 16 bytes at a 2-byte aligned address, read / written with the widest
// accesses the alignment allows, never outside [p, p + 16).
__device__ __forceinline__ uint4 ld16_any(const unsigned short* p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  if ((a & 15u) == 0) return *reinterpret_cast<const uint4*>(p);
  if ((a & 7u) == 0) {
    const uint2 lo = reinterpret_cast<const uint2*>(p)[0], hi = reinterpret_cast<const uint2*>(p)[1];
    return make_uint4(lo.x, lo.y, hi.x, hi.y);
  }
  if ((a & 3u) == 0) {
    const unsigned* w = reinterpret_cast<const unsigned*>(p);
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  const unsigned* w = reinterpret_cast<const unsigned*>(p + 1);
  const uint32_t h0 = p[0], h7 = p[7], w0 = w[0], w1 = w[1], w2 = w[2];
  return make_uint4(h0 | (w0 << 16), (w0 >> 16) | (w1 << 16), (w1 >> 16) | (w2 << 16),
                    (w2 >> 16) | (h7 << 16));
}

__device__ __forceinline__ void st16_any(unsigned short* p, uint4 v) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  if ((a & 15u) == 0) {
    *reinterpret_cast<uint4*>(p) = v;
  } else if ((a & 7u) == 0) {
    reinterpret_cast<uint2*>(p)[0] = make_uint2(v.x, v.y);
    reinterpret_cast<uint2*>(p)[1] = make_uint2(v.z, v.w);
  } else if ((a & 3u) == 0) {
    unsigned* w = reinterpret_cast<unsigned*>(p);
    w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
  } else {
    unsigned* w = reinterpret_cast<unsigned*>(p + 1);
    p[0] = static_cast<unsigned short>(v.x);
    w[0] = (v.x >> 16) | (v.y << 16);
    w[1] = (v.y >> 16) | (v.z << 16);
    w[2] = (v.z >> 16) | (v.w << 16);
    p[7] = static_cast<unsigned short>(v.w >> 16);
  }
}

// dst(r, c) = src(r, c) when both views have unit column stride: each thread
// moves 8 consecutive columns of one row (blockIdx.y selects the row).
__global__ void __launch_bounds__(kRepackThreads)
    repack_rows_kernel(const __half* __restrict__ src, int64_t s_sr, __half* __restrict__ dst,
                       int64_t s_dr, int rows, int cols) {
  const unsigned short* s =
      reinterpret_cast<const unsigned short*>(src) + static_cast<int64_t>(blockIdx.y) * s_sr;
  unsigned short* d = reinterpret_cast<unsigned short*>(dst) + static_cast<int64_t>(blockIdx.y) * s_dr;
  for (int c = 8 * (static_cast<int>(blockIdx.x) * kRepackThreads + static_cast<int>(threadIdx.x));
       c < cols; c += 8 * kRepackThreads * static_cast<int>(gridDim.x)) {
    if (c + 8 <= cols) {
      st16_any(d + c, ld16_any(s + c));
    } else {
      for (int j = c; j < cols; ++j) d[j] = s[j];
    }
  }
}

}  // namespace gemm_tn_dev
