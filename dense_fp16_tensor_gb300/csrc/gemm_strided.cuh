// gemm_strided.cuh -- the TN GEMM for operand views TMA cannot describe.
//
// The layout page (sections 1-2) lets an operand be any shape:stride view;
// the tile kernels need one stride-1 mode, 16-byte aligned rows and 16-byte
// aligned leading dimensions for TMA.  This kernel takes arbitrary element
// strides for A (M,K), B (N,K) and C/D (M,N) and keeps everything after the
// copy the same:
//
//   warps 0-3   copy producer: each thread gathers 16-byte K-chunks (8 fp16
//               along K) of A and B rows through the strides, four chunks in
//               flight at a time -- for a contiguous chunk the widest loads
//               its alignment allows, else eight 2-byte loads -- and writes
//               them to the 128B-swizzled
//               K-major layout the TMA unit would produce (row r, chunk j at
//               byte r*128 + 16*(j ^ (r%8))), zero outside the matrix; then
//               fence.proxy.async and one arrival per thread on `full`.
//   warp 4      TMEM allocation and the single MMA-issuing thread
//               (tcgen05.mma M=128, N=256, K=16, always K-major descriptors).
//   warps 5-8   epilogue: tcgen05.ld, + C, round, element-wise strided D.
//
// 128 x 256 tiles, 4 stages of 48 KiB, two TMEM accumulators, persistent
// grid, bounded waits; no asynchronous copies, so an abort only has to drain
// the MMAs.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace gemm_tn_dev {

constexpr int kStrBM = 128;
constexpr int kStrBN = 256;
constexpr int kStrBK = 64;
constexpr int kStrStages = 4;
constexpr int kStrProducers = 128;  // four warps
constexpr int kStrThreads = 288;    // 4 producer warps, MMA warp, 4 epilogue warps

struct StridedArgs {
  int M, N, K;
  const __half* A;
  int64_t sAm, sAk;
  const __half* B;
  int64_t sBn, sBk;
  __half* CD;
  int64_t sCm, sCn;
  int acc_f16;
  int tiles_m, tiles_n, num_tiles, k_blocks;
  int group_m;
  uint64_t timeout_ns;
};

struct StridedSmem {
  static constexpr uint32_t kABytes = kStrBM * kStrBK * 2;  // 16 KiB
  static constexpr uint32_t kBBytes = kStrBN * kStrBK * 2;  // 32 KiB
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kBarOffset = kStrStages * kStageBytes;
  static constexpr uint32_t kNumBars = 2 * kStrStages + 5;
  static constexpr uint32_t kCtlOffset = kBarOffset + kNumBars * 8;
  static constexpr uint32_t kBytes = kCtlOffset + 16;
  static constexpr uint32_t kDynamicBytes = kBytes + 1024;
};

// 16 contiguous bytes at a 2-byte aligned address, with the widest loads
// the alignment allows (never touching bytes outside [src, src + 16)).
__device__ __forceinline__ uint4 load16_contiguous(const __half* src) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(src);
  if ((a & 15u) == 0) return __ldg(reinterpret_cast<const uint4*>(src));
  uint4 v;
  if ((a & 7u) == 0) {
    const uint2 lo = __ldg(reinterpret_cast<const uint2*>(src));
    const uint2 hi = __ldg(reinterpret_cast<const uint2*>(src + 4));
    v = make_uint4(lo.x, lo.y, hi.x, hi.y);
  } else if ((a & 3u) == 0) {
    const unsigned* w = reinterpret_cast<const unsigned*>(src);
    v = make_uint4(__ldg(w), __ldg(w + 1), __ldg(w + 2), __ldg(w + 3));
  } else {  // 2 mod 4: one halfword, three words, one halfword
    const unsigned short* hs = reinterpret_cast<const unsigned short*>(src);
    const unsigned* w = reinterpret_cast<const unsigned*>(src + 1);
    const uint32_t h0 = __ldg(hs), h7 = __ldg(hs + 7);
    const uint32_t w0 = __ldg(w), w1 = __ldg(w + 1), w2 = __ldg(w + 2);
    v.x = h0 | (w0 << 16);
    v.y = (w0 >> 16) | (w1 << 16);
    v.z = (w1 >> 16) | (w2 << 16);
    v.w = (w2 >> 16) | (h7 << 16);
  }
  return v;
}

// Eight consecutive-k elements X(row, k0..k0+7) of a (rows, K) view with
// strides (s_row, s_k); zeros outside the matrix.
__device__ __forceinline__ uint4 gather_chunk(const __half* X, int64_t s_row, int64_t s_k,
                                              int rows, int K, int row, int k0) {
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (row >= rows || k0 >= K) return v;
  const __half* src = X + static_cast<int64_t>(row) * s_row + static_cast<int64_t>(k0) * s_k;
  if (s_k == 1 && k0 + 8 <= K) return load16_contiguous(src);
  unsigned short h[8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
    h[j] = (k0 + j < K) ? __ldg(reinterpret_cast<const unsigned short*>(src + j * s_k)) : 0;
  v.x = h[0] | (static_cast<uint32_t>(h[1]) << 16);
  v.y = h[2] | (static_cast<uint32_t>(h[3]) << 16);
  v.z = h[4] | (static_cast<uint32_t>(h[5]) << 16);
  v.w = h[6] | (static_cast<uint32_t>(h[7]) << 16);
  return v;
}

// Fill `rows` x 64 of one operand's stage in the K-major 128B-swizzled
// layout.  Chunk q of this thread's share covers row (q / 8) and K-chunk
// (q % 8) when K is the contiguous mode, else row (q % rows) so that
// neighbouring threads read neighbouring rows.  Chunks are gathered four at
// a time so that their loads are in flight together.
__device__ __forceinline__ void fill_operand(uint8_t* dst, const __half* X, int64_t s_row,
                                             int64_t s_k, int rows_total, int K, int row0,
                                             int k0, int rows, int tid) {
  const bool k_fast = (s_k == 1) || (s_row != 1 && s_k <= s_row);
  constexpr int kBatch = 4;
  for (int q0 = tid; q0 < rows * 8; q0 += kBatch * kStrProducers) {
    uint4 v[kBatch];
    int off[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int q = q0 + b * kStrProducers;
      off[b] = -1;
      v[b] = make_uint4(0u, 0u, 0u, 0u);
      if (q < rows * 8) {
        const int r = k_fast ? q >> 3 : q % rows;
        const int j = k_fast ? q & 7 : q / rows;
        v[b] = gather_chunk(X, s_row, s_k, rows_total, K, row0 + r, k0 + 8 * j);
        off[b] = r * 128 + 16 * (j ^ (r & 7));
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b)
      if (off[b] >= 0) *reinterpret_cast<uint4*>(dst + off[b]) = v[b];
  }
}

__global__ void __launch_bounds__(kStrThreads, 1) gemm_tn_strided_kernel(const StridedArgs p) {
  using L = StridedSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;                                // stage s at s * kABytes
  uint8_t* sB = smem + kStrStages * L::kABytes;      // stage s at s * kBBytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kCtlOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kCtlOffset + 4);

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + kStrStages);
  const uint32_t tfull0 = smem_u32(bars + 2 * kStrStages);
  const uint32_t tempty0 = smem_u32(bars + 2 * kStrStages + 2);
  const uint32_t drain = smem_u32(bars + 2 * kStrStages + 4);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStrStages; ++s) {
      mbar_init(full0 + 8 * s, kStrProducers);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(tmem_slot), 2 * kStrBN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp < 4) {
    // ------------------------------------------------------------ copy producer
    const int tid = static_cast<int>(threadIdx.x);
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
      int tm, tn;
      tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        if (!wait_bounded(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.timeout_ns,
                          timeout_code(kRoleProducer, stage))) {
          ok = false;
          break;
        }
        const int k0 = kb * kStrBK;
        fill_operand(sA + stage * L::kABytes, p.A, p.sAm, p.sAk, p.M, p.K, tm * kStrBM, k0,
                     kStrBM, tid);
        fill_operand(sB + stage * L::kBBytes, p.B, p.sBn, p.sBk, p.N, p.K, tn * kStrBN, k0,
                     kStrBN, tid);
        fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
        mbar_arrive(full0 + 8 * stage);
        if (++stage == kStrStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 4) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc_f16(kStrBM, kStrBN, !p.acc_f16, 0, 0);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        if (!wait_bounded(tempty0 + 8 * acc, acc_phase ^ 1u, abort_flag, p.timeout_ns,
                          timeout_code(kRoleMma, 0x200 + acc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kStrBN;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_bounded(full0 + 8 * stage, phase, abort_flag, p.timeout_ns,
                            timeout_code(kRoleMma, stage))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * L::kABytes);
          const uint32_t b_base = smem_u32(sB + stage * L::kBBytes);
#pragma unroll
          for (int k = 0; k < kStrBK / 16; ++k)
            mma_f16(d_tmem, make_sw128_desc(a_base + k * 32, 16, 1024),
                    make_sw128_desc(b_base + k * 32, 16, 1024), idesc, (kb | k) != 0);
          mma_commit(empty0 + 8 * stage);
          if (++stage == kStrStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * acc);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok || *abort_flag) {
        mma_commit(drain);
        wait_bounded(drain, 0, abort_flag, p.timeout_ns, timeout_code(kRoleMma, 0x300), false);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t quad = static_cast<uint32_t>(warp & 3);
    const int row_in_tile = static_cast<int>(quad * 32 + lane);
    uint32_t acc = 0, acc_phase = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int tm, tn;
      tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
      if (!wait_bounded(tfull0 + 8 * acc, acc_phase, abort_flag, p.timeout_ns,
                        timeout_code(kRoleEpilogue, acc)))
        break;
      tc_fence_after();
      const int m = tm * kStrBM + row_in_tile;
      const uint32_t t_row = tmem_base + ((quad * 32) << 16) + acc * kStrBN;
#pragma unroll 1
      for (int c = 0; c < kStrBN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        tmem_wait_ld();
        if (m < p.M) {
          __half* row = p.CD + static_cast<int64_t>(m) * p.sCm;
          const int n0 = tn * kStrBN + c * 32;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int n = n0 + j;
            if (n < p.N) {
              __half* d = row + static_cast<int64_t>(n) * p.sCn;
              if (p.acc_f16)
                *d = __hadd(__ushort_as_half(static_cast<unsigned short>(r[j])), *d);
              else
                *d = __float2half_rn(__uint_as_float(r[j]) + __half2float(*d));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * kStrBN);
  }
}

}  // namespace gemm_tn_dev
