// gemm_large.cuh -- persistent, warp-specialised tcgen05 TN GEMM for sm_103a.
//
// Computes D(m,n) = C(m,n) + sum_k A(m,k) B(n,k) over 128 x BN output tiles
// (in general D = alpha * A.B^T + beta * C, over a batch of problems; see
// EpiArgs)
// (the CTA tiling and K-block loop of "CuTe Layout to Tensor Core", section
// 4 "local_tile", and "cute(7) simple_gemm", section "3.4 the K loop"), with
// the data movement redone for GB300:
//
//   warp 0      TMA producer: per K block of 64, one A box (128 x 64) and one
//               B box (BN x 64) into a 128B-swizzled stage of a kStages ring,
//               completion counted on the stage's `full` mbarrier.  Out-of-
//               range rows / columns / K are zero-filled by the TMA unit, so
//               ragged M, N and K need no special case in the main loop.
//   warp 1      allocates 2*BN TMEM columns (two accumulators) and one lane
//               issues tcgen05.mma (M=128, N=BN, K=16, four per stage); each
//               stage is released with tcgen05.commit -> `empty`, each tile
//               with tcgen05.commit -> `tmem_full`.
//   warps 2-5   epilogue: tcgen05.ld 32 columns at a time, add C in the
//               accumulator's precision, round to fp16, predicated 16-byte
//               stores; arrive `tmem_empty` so the MMA warp can reuse the
//               accumulator while the next tile's main loop runs.
//
// Tiles are handed out round-robin (t = blockIdx.x, += gridDim.x) in a
// grouped raster.  Every wait is bounded (see wait_bounded); on expiry the
// kernel records the failure, drains its own copies and MMAs in flight,
// frees its TMEM and returns.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace gemm_tn_dev {

constexpr int kLargeBM = 128;
constexpr int kLargeBK = 64;
constexpr int kLargeStages = 4;
constexpr int kLargeThreads = 192;

struct LargeArgs {
  int M, N, K;
  EpiArgs e;           // C, D, alpha, beta
  int batch;           // problems; tile t belongs to problem t / tiles_per_batch
  int tiles_per_batch;  // tiles_m * tiles_n
  int a_batched, b_batched;  // operand maps carry a batch coordinate (else it is 0)
  int acc_f16;
  int a_mn, b_mn;
  int tiles_m, tiles_n, num_tiles, k_blocks;  // num_tiles = batch * tiles_per_batch
  int group_m;
  uint64_t timeout_ns;
  int test_stall;
  // Stream-K (256 x 256 kernel only): tiles [sk_tile0, num_tiles) are cut
  // into contiguous (tile, K-block) ranges of sk_per units, CTA c owning
  // units [c * sk_per, min((c + 1) * sk_per, sk_units)).  sk_tile0 ==
  // num_tiles means no split tiles.  (sk_per * (gridDim.x + 1) < 2^31.)
  int sk_tile0;
  int sk_max_segs;     // split-tile segments one CTA can hold
  int sk_units;        // (num_tiles - sk_tile0) * k_blocks
  int sk_per;          // units per CTA
  float* sk_partials;  // [gridDim.x * sk_max_segs] slots of 256 x 256 fp32
  int* sk_counters;    // [(num_tiles - sk_tile0) * 8], zero on entry
};

template <int BN>
struct LargeSmem {
  static constexpr uint32_t kABytes = kLargeBM * kLargeBK * 2;  // 16 KiB
  static constexpr uint32_t kBBytes = BN * kLargeBK * 2;        // 16 / 32 KiB
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kBarOffset = kLargeStages * kStageBytes;
  // full[S], empty[S], tmem_full[2], tmem_empty[2], drain
  static constexpr uint32_t kNumBars = 2 * kLargeStages + 5;
  static constexpr uint32_t kCtlOffset = kBarOffset + kNumBars * 8;
  static constexpr uint32_t kBytes = kCtlOffset + 16;
  static constexpr uint32_t kDynamicBytes = kBytes + 1024;  // + alignment slack
};

// Batch and tile coordinates of tile t (grouped raster inside each problem).
__device__ __forceinline__ void batch_tile(const LargeArgs& p, int t, int& tb, int& tm,
                                           int& tn) {
  tb = p.batch > 1 ? t / p.tiles_per_batch : 0;
  tile_coords(t - tb * p.tiles_per_batch, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
}

// Epilogue of one 32-column chunk for one row of problem tb:
// D = alpha * acc + beta * C, fp16 out.
__device__ __forceinline__ void store_chunk(const LargeArgs& p, int tb, int m, int n0,
                                            const uint32_t (&r)[32]) {
  if (m >= p.M || n0 >= p.N) return;
  const EpiArgs& e = p.e;
  const __half* crow = e.C + tb * e.sC + static_cast<int64_t>(m) * e.ldC;
  __half* drow = e.D + tb * e.sD + static_cast<int64_t>(m) * e.ldD;
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const int n = n0 + 8 * v;
    if (n + 8 <= p.N) {
      uint4 c = make_uint4(0u, 0u, 0u, 0u);
      if (e.read_c) c = *reinterpret_cast<const uint4*>(crow + n);
      const __half2* ch = reinterpret_cast<const __half2*>(&c);
      uint4 o;
      __half2* oh = reinterpret_cast<__half2*>(&o);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo = r[8 * v + 2 * j], hi = r[8 * v + 2 * j + 1];
        if (p.acc_f16) {
          const __half2 acc = __halves2half2(__ushort_as_half(static_cast<unsigned short>(lo)),
                                             __ushort_as_half(static_cast<unsigned short>(hi)));
          oh[j] = epi_f16x2(e, acc, ch[j]);
        } else {
          oh[j] = epi_f32x2(e, __uint_as_float(lo), __uint_as_float(hi), ch[j]);
        }
      }
      *reinterpret_cast<uint4*>(drow + n) = o;
    } else {
      for (int j = 0; j < 8 && n + j < p.N; ++j) {
        const __half c = e.read_c ? crow[n + j] : __ushort_as_half(0);
        drow[n + j] = epi_one(e, p.acc_f16, r[8 * v + j], c);
      }
    }
  }
}

template <int BN>
__global__ void __launch_bounds__(kLargeThreads, 1)
    gemm_tn_large_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB, const LargeArgs p) {
  using L = LargeSmem<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;                                  // stage s at s * kABytes
  uint8_t* sB = smem + kLargeStages * L::kABytes;      // stage s at s * kBBytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kCtlOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kCtlOffset + 4);

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + kLargeStages);
  const uint32_t tfull0 = smem_u32(bars + 2 * kLargeStages);
  const uint32_t tempty0 = smem_u32(bars + 2 * kLargeStages + 2);
  const uint32_t drain = smem_u32(bars + 2 * kLargeStages + 4);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kLargeStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;  // per stage: loads issued, their parity
      bool ok = true;
      int local = 0;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x, ++local) {
        int tb, tm, tn;
        batch_tile(p, t, tb, tm, tn);
        const int za = p.a_batched ? tb : 0, zb = p.b_batched ? tb : 0;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_bounded(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.timeout_ns,
                            timeout_code(kRoleProducer, stage))) {
            ok = false;
            break;
          }
          const bool withhold = p.test_stall && local == 0 && kb == 0;
          if (!withhold) {
            const uint32_t fb = full0 + 8 * stage;
            const uint32_t a_dst = smem_u32(sA + stage * L::kABytes);
            const uint32_t b_dst = smem_u32(sB + stage * L::kBBytes);
            mbar_arrive_expect_tx(fb, L::kStageBytes);
            const int k0 = kb * kLargeBK;
            if (!p.a_mn) {
              tma_load_3d(a_dst, &tmA, fb, k0, tm * kLargeBM, za);
            } else {
#pragma unroll
              for (int i = 0; i < kLargeBM / 64; ++i)
                tma_load_3d(a_dst + i * 8192, &tmA, fb, tm * kLargeBM + 64 * i, k0, za);
            }
            if (!p.b_mn) {
              tma_load_3d(b_dst, &tmB, fb, k0, tn * BN, zb);
            } else {
#pragma unroll
              for (int i = 0; i < BN / 64; ++i)
                tma_load_3d(b_dst + i * 8192, &tmB, fb, tn * BN + 64 * i, k0, zb);
            }
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == kLargeStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok || *abort_flag) {
        // Let every copy this thread issued land before the CTA can exit.
        for (int s = 0; s < kLargeStages; ++s)
          if (issued_mask >> s & 1u)
            wait_bounded(full0 + 8 * s, issued_parity >> s & 1u, abort_flag, p.timeout_ns,
                         timeout_code(kRoleProducer, 0x100 + s), false);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc_f16(kLargeBM, BN, !p.acc_f16, p.a_mn, p.b_mn);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        if (!wait_bounded(tempty0 + 8 * acc, acc_phase ^ 1u, abort_flag, p.timeout_ns,
                          timeout_code(kRoleMma, 0x200 + acc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
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
          for (int k = 0; k < kLargeBK / 16; ++k) {
            const uint64_t ad = p.a_mn ? make_sw128_desc(a_base + k * 2048, 8192, 1024)
                                       : make_sw128_desc(a_base + k * 32, 16, 1024);
            const uint64_t bd = p.b_mn ? make_sw128_desc(b_base + k * 2048, 8192, 1024)
                                       : make_sw128_desc(b_base + k * 32, 16, 1024);
            mma_f16(d_tmem, ad, bd, idesc, (kb | k) != 0);
          }
          mma_commit(empty0 + 8 * stage);  // stage free once these MMAs have read it
          if (++stage == kLargeStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * acc);  // accumulator complete
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok || *abort_flag) {
        // Wait until every MMA issued so far has finished with TMEM and smem.
        mma_commit(drain);
        wait_bounded(drain, 0, abort_flag, p.timeout_ns, timeout_code(kRoleMma, 0x300), false);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t quad = static_cast<uint32_t>(warp & 3);  // TMEM lanes 32*quad ..
    const int row_in_tile = static_cast<int>(quad * 32 + lane);
    uint32_t acc = 0, acc_phase = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int tb, tm, tn;
      batch_tile(p, t, tb, tm, tn);
      if (!wait_bounded(tfull0 + 8 * acc, acc_phase, abort_flag, p.timeout_ns,
                        timeout_code(kRoleEpilogue, acc)))
        break;
      tc_fence_after();
      const int m = tm * kLargeBM + row_in_tile;
      const uint32_t t_row = tmem_base + ((quad * 32) << 16) + acc * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        tmem_wait_ld();
        store_chunk(p, tb, m, tn * BN + c * 32, r);
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
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * BN);
  }
}

}  // namespace gemm_tn_dev
