// gemm_wide.cuh -- persistent tcgen05 TN GEMM with 256 x 256 tiles on one CTA.
//
// Same computation as gemm_large.cuh (the CTA tiling and K-block loop of the
// layout page, section 4 "local_tile"), arranged for the SM's operand
// ingress rather than for accumulator double-buffering:
//
//   * per 64-deep K block the producer loads one 256 x 64 box of A and one
//     256 x 64 box of B (64 KiB, 3 stages); every 16-deep step issues two
//     tcgen05.mma (M = 128, N = 256) that share the B slice, one per
//     128-row half of A, into TMEM columns [0,256) and [256,512).  Per SM
//     that is 62.5 bytes of operands per clock of tensor work, against 96 for
//     128 x 256 tiles, which a GB300 SM's TMA ingress (measured ~70-80 B/clk)
//     cannot sustain.
//   * the tile's accumulator fills all 512 TMEM columns, so it is not double
//     buffered and the epilogue is on the critical path.  Eight epilogue
//     warps (two per TMEM lane quadrant, one per 128-row half) each drain a
//     32 x 256 block in four 32 x 64 chunks through a 4 KiB staging buffer
//     with the 128-byte swizzle: C rows arrive with coalesced 128-byte loads
//     (the first chunk's before the accumulator is even ready, the others
//     one chunk ahead), each lane adds its TMEM row in the swizzled layout
//     (conflict-free), and D leaves by TMA store, which also clips the tails.
//     The next tile's C rows are prefetched into L2 during its main loop, and
//     the TMA ring keeps loading the next tile's first stages meanwhile.
//
// Waits are bounded and abort as in gemm_large.cuh.
#pragma once

#include <cuda_fp16.h>

#include "gemm_large.cuh"

namespace gemm_tn_dev {

constexpr int kWideBM = 256;
constexpr int kWideBN = 256;
constexpr int kWideBK = 64;
constexpr int kWideStages = 3;
constexpr int kWideThreads = 320;  // producer warp, MMA warp, 8 epilogue warps
constexpr uint32_t kWideTmemCols = 512;

constexpr int kWideEpiWarps = 8;
constexpr uint32_t kWideStagingBytes = 32 * 128;  // 32 rows x 64 fp16, 128-byte swizzle

struct WideSmem {
  static constexpr uint32_t kABytes = kWideBM * kWideBK * 2;  // 32 KiB
  static constexpr uint32_t kBBytes = kWideBN * kWideBK * 2;  // 32 KiB
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kStagingOffset = kWideStages * kStageBytes;  // 1024-aligned
  static constexpr uint32_t kBarOffset = kStagingOffset + kWideEpiWarps * kWideStagingBytes;
  // full[S], empty[S], tmem_full, tmem_empty, drain
  static constexpr uint32_t kNumBars = 2 * kWideStages + 3;
  static constexpr uint32_t kCtlOffset = kBarOffset + kNumBars * 8;
  static constexpr uint32_t kBytes = kCtlOffset + 16;
  static constexpr uint32_t kDynamicBytes = kBytes + 1024;
};

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)),
               "r"(bytes)
               : "memory");
}

// Eight fp16 values of C (uint4) plus eight accumulator words -> eight fp16 of D.
__device__ __forceinline__ uint4 add_c8(bool acc_f16, const uint32_t* r, uint4 c) {
  const __half2* ch = reinterpret_cast<const __half2*>(&c);
  uint4 o;
  __half2* oh = reinterpret_cast<__half2*>(&o);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = r[2 * j], hi = r[2 * j + 1];
    if (acc_f16) {
      const __half2 acc = __halves2half2(__ushort_as_half(static_cast<unsigned short>(lo)),
                                         __ushort_as_half(static_cast<unsigned short>(hi)));
      oh[j] = __hadd2(acc, ch[j]);
    } else {
      const float2 cf = __half22float2(ch[j]);
      oh[j] = __floats2half2_rn(__uint_as_float(lo) + cf.x, __uint_as_float(hi) + cf.y);
    }
  }
  return o;
}

// One 16-byte piece of a 32 x 64 C chunk for the coalesced load pattern:
// load i (0..7) of lane l covers row 4i + l/8, columns 8*(l%8) .. +8.
__device__ __forceinline__ uint4 load_c_piece(const LargeArgs& p, int m, int n) {
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (m < p.M && n < p.N) {
    const __half* src = p.CD + static_cast<int64_t>(m) * p.ldC + n;
    if (n + 8 <= p.N) {
      v = *reinterpret_cast<const uint4*>(src);
    } else {
      __half* vh = reinterpret_cast<__half*>(&v);
      for (int j = 0; j < 8 && n + j < p.N; ++j) vh[j] = src[j];
    }
  }
  return v;
}

__global__ void __launch_bounds__(kWideThreads, 1)
    gemm_tn_wide_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmD, const LargeArgs p) {
  using L = WideSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // stage s: A box at s*kStageBytes, B box right after (both 1024-aligned)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kCtlOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kCtlOffset + 4);

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + kWideStages);
  const uint32_t tfull = smem_u32(bars + 2 * kWideStages);
  const uint32_t tempty = smem_u32(bars + 2 * kWideStages + 1);
  const uint32_t drain = smem_u32(bars + 2 * kWideStages + 2);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWideStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 8);  // eight epilogue warps
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kWideTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, issued_mask = 0, issued_parity = 0;
      bool ok = true;
      int local = 0;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x, ++local) {
        int tm, tn;
        tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_bounded(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.timeout_ns,
                            timeout_code(kRoleProducer, stage))) {
            ok = false;
            break;
          }
          if (!(p.test_stall && local == 0 && kb == 0)) {
            const uint32_t fb = full0 + 8 * stage;
            const uint32_t a_dst = smem_u32(smem + stage * L::kStageBytes);
            const uint32_t b_dst = a_dst + L::kABytes;
            mbar_arrive_expect_tx(fb, L::kStageBytes);
            const int k0 = kb * kWideBK;
            if (!p.a_mn) {
              tma_load_2d(a_dst, &tmA, fb, k0, tm * kWideBM);
            } else {
#pragma unroll
              for (int i = 0; i < kWideBM / 64; ++i)
                tma_load_2d(a_dst + i * 8192, &tmA, fb, tm * kWideBM + 64 * i, k0);
            }
            if (!p.b_mn) {
              tma_load_2d(b_dst, &tmB, fb, k0, tn * kWideBN);
            } else {
#pragma unroll
              for (int i = 0; i < kWideBN / 64; ++i)
                tma_load_2d(b_dst + i * 8192, &tmB, fb, tn * kWideBN + 64 * i, k0);
            }
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == kWideStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok || *abort_flag) {
        for (int s = 0; s < kWideStages; ++s)
          if (issued_mask >> s & 1u)
            wait_bounded(full0 + 8 * s, issued_parity >> s & 1u, abort_flag, p.timeout_ns,
                         timeout_code(kRoleProducer, 0x100 + s), false);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc_f16(128, kWideBN, !p.acc_f16, p.a_mn, p.b_mn);
      uint32_t stage = 0, phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        if (!wait_bounded(tempty, acc_phase ^ 1u, abort_flag, p.timeout_ns,
                          timeout_code(kRoleMma, 0x200))) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_bounded(full0 + 8 * stage, phase, abort_flag, p.timeout_ns,
                            timeout_code(kRoleMma, stage))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + stage * L::kStageBytes);
          const uint32_t b_base = a_base + L::kABytes;
#pragma unroll
          for (int k = 0; k < kWideBK / 16; ++k) {
            const uint64_t bd = p.b_mn ? make_sw128_desc(b_base + k * 2048, 8192, 1024)
                                       : make_sw128_desc(b_base + k * 32, 16, 1024);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              // rows [128h, 128h+128) of the A box: 16 KiB further in both layouts
              const uint32_t ah = a_base + h * 16384;
              const uint64_t ad = p.a_mn ? make_sw128_desc(ah + k * 2048, 8192, 1024)
                                         : make_sw128_desc(ah + k * 32, 16, 1024);
              mma_f16(tmem_base + h * kWideBN, ad, bd, idesc, (kb | k) != 0);
            }
          }
          mma_commit(empty0 + 8 * stage);
          if (++stage == kWideStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull);
        acc_phase ^= 1u;
      }
      if (!ok || *abort_flag) {
        mma_commit(drain);
        wait_bounded(drain, 0, abort_flag, p.timeout_ns, timeout_code(kRoleMma, 0x300), false);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;                                // 0..7
    const int half = ew >> 2;                               // 128-row half of the tile
    const uint32_t quad = static_cast<uint32_t>(warp & 3);  // TMEM lanes 32*quad ..
    const int row0 = half * 128 + static_cast<int>(quad * 32);  // first tile row of this warp
    uint8_t* stg = smem + L::kStagingOffset + ew * kWideStagingBytes;
    const uint32_t stg_u32 = smem_u32(stg);
    // coalesced pattern: piece i of lane l is row 4i + l/8, 16-byte segment l%8
    const int prow = static_cast<int>(lane >> 3), pseg = static_cast<int>(lane & 7);
    auto load_chunk = [&](int tm, int tn, int c, uint4 (&v)[8]) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        v[i] = load_c_piece(p, tm * kWideBM + row0 + 4 * i + prow, tn * kWideBN + 64 * c + 8 * pseg);
    };
    auto stage_chunk = [&](const uint4 (&v)[8]) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = 4 * i + prow;
        *reinterpret_cast<uint4*>(stg + r * 128 + 16 * (pseg ^ (r & 7))) = v[i];
      }
    };
    // Warm L2 with this warp's C rows of a tile (one row per lane).
    auto prefetch_c = [&](int t2) {
      if (t2 >= p.num_tiles) return;
      int tm2, tn2;
      tile_coords(t2, p.tiles_m, p.tiles_n, p.group_m, tm2, tn2);
      const int m2 = tm2 * kWideBM + row0 + static_cast<int>(lane);
      const int n2 = tn2 * kWideBN;
      if (m2 < p.M && n2 < p.N) {
        const uint32_t bytes = static_cast<uint32_t>(min(kWideBN, p.N - n2) * 2) & ~15u;
        if (bytes) prefetch_l2(p.CD + static_cast<int64_t>(m2) * p.ldC + n2, bytes);
      }
    };
    prefetch_c(static_cast<int>(blockIdx.x));
    uint32_t acc_phase = 0;
    uint4 cnext[8];
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int tm, tn;
      tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
      // C of the first two chunks does not depend on the MMAs: fetch it now
      // (once the previous tile's last store has finished reading staging).
      load_chunk(tm, tn, 0, cnext);
      if (lane == 0) bulk_wait_group_read0();
      __syncwarp();
      stage_chunk(cnext);
      load_chunk(tm, tn, 1, cnext);
      __syncwarp();
      if (!wait_bounded(tfull, acc_phase, abort_flag, p.timeout_ns,
                        timeout_code(kRoleEpilogue, 0)))
        break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((quad * 32) << 16) + half * kWideBN;
      const int m_row0 = tm * kWideBM + row0;
#pragma unroll 1
      for (int c = 0; c < kWideBN / 64; ++c) {
        uint32_t r[64];
        tmem_ld_32x32b_x32(t_row + c * 64, *reinterpret_cast<uint32_t(*)[32]>(r));
        tmem_ld_32x32b_x32(t_row + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
        tmem_wait_ld();
        if (c == kWideBN / 64 - 1) {
          // every TMEM column of this warp is in registers: hand the
          // accumulator back so the next tile's MMAs can start
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty);
        }
        if (c > 0) {
          // the previous chunk's store must have read the staging buffer
          if (lane == 0) bulk_wait_group_read0();
          __syncwarp();
          stage_chunk(cnext);
          if (c + 1 < kWideBN / 64) load_chunk(tm, tn, c + 1, cnext);
          __syncwarp();
        }
        // row `lane` of the chunk: D = C + acc in the swizzled layout
        uint8_t* my_row = stg + lane * 128;
#pragma unroll
        for (int s8 = 0; s8 < 8; ++s8) {
          uint4* q = reinterpret_cast<uint4*>(my_row + 16 * (s8 ^ static_cast<int>(lane & 7)));
          *q = add_c8(p.acc_f16, r + 8 * s8, *q);
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int n0 = tn * kWideBN + 64 * c;
        if (lane == 0 && m_row0 < p.M && n0 < p.N) {
          tma_store_2d(&tmD, stg_u32, n0, m_row0);
          bulk_commit_group();
        }
      }
      acc_phase ^= 1u;
      prefetch_c(t + static_cast<int>(gridDim.x));
    }
    if (lane == 0) bulk_wait_group0();  // all D stores performed before exit
    __syncwarp();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kWideTmemCols);
  }
}

}  // namespace gemm_tn_dev
