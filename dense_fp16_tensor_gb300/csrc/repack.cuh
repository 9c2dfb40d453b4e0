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

#include "shift.cuh"

namespace gemm_tn_dev {

constexpr int kRepackTile = 64;
constexpr int kRepackThreads = 256;

__global__ void __launch_bounds__(kRepackThreads)
    repack2d_kernel(const __half* __restrict__ src, int64_t s_sr, int64_t s_sc,
                    __half* __restrict__ dst, int64_t s_dr, int64_t s_dc, int rows, int cols) {
  __shared__ unsigned short tile[kRepackTile][kRepackTile + 2];
  // launched as a programmatic dependent: resident while the kernel before
  // it drains, touching memory only once that kernel has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
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

// dst(r, c) = src(r, c) when both views have unit column stride (any 2-byte
// alignment of either row): blockIdx.y selects the row, each thread builds
// whole 16-byte words of the destination row at their aligned addresses
// from the two aligned 16-byte source words under them (shift_window
// when the two rows are misaligned differently), so every load and every
// interior store is one aligned vector access.  Source words are read only
// where they hold bytes of the row (an aligned word never crosses a page);
// the partial words at the two ends of the destination row are written
// element by element.  A thread handles kRowWords words, kRepackThreads
// apart, with all their loads issued before the first store, so that enough
// bytes are in flight to stream at HBM rate.
constexpr int kRowWords = 4;

__global__ void __launch_bounds__(kRepackThreads)
    repack_rows_kernel(const __half* __restrict__ src, int64_t s_sr, __half* __restrict__ dst,
                       int64_t s_dr, int rows, int cols) {
  (void)rows;
  // a programmatic dependent launch, as repack2d_kernel
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const unsigned short* s =
      reinterpret_cast<const unsigned short*>(src) + static_cast<int64_t>(blockIdx.y) * s_sr;
  unsigned short* d = reinterpret_cast<unsigned short*>(dst) + static_cast<int64_t>(blockIdx.y) * s_dr;
  const uintptr_t sb = reinterpret_cast<uintptr_t>(s), db = reinterpret_cast<uintptr_t>(d);
  const uintptr_t s_end = sb + 2 * static_cast<uintptr_t>(cols);  // one past the row's bytes
  const uintptr_t d_end = db + 2 * static_cast<uintptr_t>(cols);
  const int a_d = static_cast<int>(db & 15u);
  // destination word w covers bytes [d0 + 16 w, d0 + 16 w + 16); element j of
  // the row sits at byte 2 j + a_d of that range, fed from source byte
  // sb + 2 j, i.e. source bytes [sb - a_d + 16 w, ... + 16)
  const uintptr_t d0 = db - a_d;
  const int words = static_cast<int>((d_end - d0 + 15) / 16);
  const intptr_t src_off = static_cast<intptr_t>(sb) - a_d;  // source byte of dst byte d0
  const int sh = static_cast<int>(static_cast<uintptr_t>(src_off) & 15u);
  constexpr int kSpan = kRepackThreads * kRowWords;  // words per block and round
  for (int w0 = static_cast<int>(blockIdx.x) * kSpan + static_cast<int>(threadIdx.x); w0 < words;
       w0 += kSpan * static_cast<int>(gridDim.x)) {
    uint4 lo[kRowWords], hi[kRowWords];
#pragma unroll
    for (int i = 0; i < kRowWords; ++i) {
      const int w = w0 + i * kRepackThreads;
      const uintptr_t a0 = (src_off + 16 * static_cast<intptr_t>(w)) & ~static_cast<uintptr_t>(15);
      lo[i] = make_uint4(0u, 0u, 0u, 0u);
      hi[i] = lo[i];
      if (w < words && a0 + 16 > sb && a0 < s_end) lo[i] = *reinterpret_cast<const uint4*>(a0);
      if (w < words && sh != 0 && a0 + 32 > sb && a0 + 16 < s_end)
        hi[i] = *reinterpret_cast<const uint4*>(a0 + 16);
    }
#pragma unroll
    for (int i = 0; i < kRowWords; ++i) {
      const int w = w0 + i * kRepackThreads;
      if (w >= words) break;
      const uint4 v = sh ? shift_window(lo[i], hi[i], sh) : lo[i];
      const uintptr_t dw = d0 + 16 * static_cast<uintptr_t>(w);
      if (dw >= db && dw + 16 <= d_end) {
        *reinterpret_cast<uint4*>(dw) = v;
      } else {
        const unsigned short* vh = reinterpret_cast<const unsigned short*>(&v);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uintptr_t a = dw + 2 * e;
          if (a >= db && a < d_end) *reinterpret_cast<unsigned short*>(a) = vh[e];
        }
      }
    }
  }
}

}  // namespace gemm_tn_dev
