// gemm_large.cuh -- persistent, warp-specialised tcgen05 TN GEMM for sm_103a.
//
// Computes D(m,n) = C(m,n) + sum_k A(m,k) B(n,k) over 128 x BN output tiles
// (in general D = alpha * A.B^T + beta * C over a batch of problems, see
// EpiArgs; the CTA tiling and K-block loop of "CuTe Layout to Tensor Core",
// section 4 "local_tile", and "cute(7) simple_gemm", section "3.4 the K
// loop"), with the data movement redone for GB300:
//
//   warp 0      TMA producer: per K block of 64, one A box (128 x 64) and one
//               B box (BN x 64) into a 128B-swizzled stage of a 4-stage ring,
//               completion counted on the stage's `full` mbarrier.  Out-of-
//               range rows / columns / K are zero-filled by the TMA unit, so
//               ragged M, N and K need no special case in the main loop.
//               With KO (BN = 128, K-major A and B, K a multiple of 64) a
//               stage covers 128 of K and each operand arrives as one
//               {64, 128, 2} box over a map whose third dimension steps K by
//               64: three stages of two 32 KiB boxes, which a GB300 SM takes
//               in about twice as fast as four 16 KiB boxes.
//   warp 1      allocates 2*BN TMEM columns (two accumulators) and one lane
//               issues tcgen05.mma (M=128, N=BN, K=16, four per stage); each
//               stage is released with tcgen05.commit -> `empty`, each tile
//               with tcgen05.commit -> `tmem_full`.
//   warps 2-9   epilogue (staged, shared with the other tile kernels), two
//               warps per TMEM lane quadrant, each on one half of the
//               tile's columns: C of the next tile arrives in coalesced
//               32 x 64 chunks into the warp's 128-byte-swizzled staging
//               buffer while its MMAs run; per chunk tcgen05.ld 64 columns,
//               combine with the staged C (epi_f32x2 / epi_f16x2),
//               TMA-store the chunk; arrive `tmem_empty` once the warp's
//               columns are read, so the MMA warp reuses the accumulator
//               while the epilogue finishes.
//
// Work units (tiles, or (tile, K range) pairs when ks_splits > 1) are handed
// out round-robin (u = blockIdx.x, += gridDim.x) in a grouped raster; a
// split unit stores its fp32 partial tile for gemm_tn_tile_reduce_kernel.
// Every wait is bounded (see wait_bounded); on expiry the kernel records the
// failure, drains its own copies and MMAs in flight, frees its TMEM and
// returns.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace gemm_tn_dev {

constexpr int kLargeBM = 128;
constexpr int kLargeBK = 64;   // K per stage (and per p.k_blocks unit) without KO
constexpr int kLargeThreads = 320;  // producer warp, MMA warp, 8 epilogue warps

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
  // Split-K of the 128-row kernel: each tile's K blocks are cut into
  // ks_splits ranges of ks_kb_per blocks (the last may be shorter); work
  // unit u is split u % ks_splits of tile u / ks_splits.  With ks_splits > 1
  // each unit stores its fp32 partial tile to ks_ws (layout at
  // ks_partial_index) and gemm_tn_tile_reduce_kernel adds the splits.
  int ks_splits;       // 1 = no split
  int ks_kb_per;
  float* ks_ws;
  // CTA-pair kernel: with ks_splits > 1, tiles [0, ks_tile0) run whole and
  // only tiles [ks_tile0, num_tiles) are split (0: every tile is split).
  // The reduction kernel's tile t is the partial slot of split tile t, and
  // ks_tile0 there is the first split tile in its own (128-row) raster.
  // The 128-row kernel splits every tile (ks_tile0 = 0).
  int ks_tile0;
  // CTA-pair kernel: output tile width (a multiple of 32 in [64, 256]; 256
  // whenever ks_splits > 1).  The other kernels use their compile-time width.
  int bn;
  int trace;           // phase trace on (see trace_mark)
};

// Epilogue warps of the 128 x BN kernel: two per TMEM lane quadrant, each
// draining one half of the tile's columns, for BN >= 128; one per quadrant
// over all 64 columns for BN = 64.
template <int BN>
struct LargeEpi {
  static constexpr int kWarps = BN >= 128 ? 8 : 4;
  static constexpr int kColsPerWarp = BN >= 128 ? BN / 2 : BN;
  static constexpr int kChunks = kColsPerWarp / 64;  // 64-column chunks per warp
  static_assert(BN == 64 || BN == 128 || BN == 256, "tile widths 64, 128 and 256");
};

template <int BN, bool KO = false>
struct LargeSmem {
  static_assert(!KO || BN <= 128, "K-chunk boxes only with 128 x 128 and 128 x 64 tiles");
  static constexpr int kBK = KO ? 128 : kLargeBK;    // K per stage
  // 3 stages of 64 KiB (KO, 128 wide), 4 of 48 KiB (KO, 64 wide), 4 of 48 /
  // 32 KiB (256 / 128 wide), 6 of 24 KiB (64 wide)
  static constexpr int kStages = KO ? (BN == 64 ? 4 : 3) : (BN == 64 ? 6 : 4);
  static constexpr uint32_t kABytes = kLargeBM * kBK * 2;  // 16 / 32 KiB
  static constexpr uint32_t kBBytes = BN * kBK * 2;        // 8 - 32 KiB
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  // epilogue staging: one buffer of 32 rows x 64 fp16 per epilogue warp
  // (1024-aligned)
  static constexpr uint32_t kStagingOffset = kStages * kStageBytes;
  static constexpr uint32_t kBarOffset = kStagingOffset + LargeEpi<BN>::kWarps * 32 * 128;
  // full[S], empty[S], tmem_full[2], tmem_empty[2], drain
  static constexpr uint32_t kNumBars = 2 * kStages + 5;
  static constexpr uint32_t kCtlOffset = kBarOffset + kNumBars * 8;
  static constexpr uint32_t kBytes = kCtlOffset + 16;
  static constexpr uint32_t kDynamicBytes = kBytes + 1024;  // + alignment slack
  static_assert(kDynamicBytes <= 232448, "over the 227 KiB of shared memory per CTA");
};

// Batch and tile coordinates of tile t (grouped raster inside each problem).
__device__ __forceinline__ void batch_tile(const LargeArgs& p, int t, int& tb, int& tm,
                                           int& tn) {
  tb = p.batch > 1 ? t / p.tiles_per_batch : 0;
  tile_coords(t - tb * p.tiles_per_batch, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
}

// Split-K partial tile of unit u (128 x bn fp32): float4 of row 32q + lane,
// columns 64c + 4g .. +3 (q: TMEM lane quadrant, c: 64-column chunk, g: group
// of 4 columns) at this index, so that a warp's stores and the reduction's
// loads move whole 512-byte lines.
__device__ __forceinline__ int64_t ks_partial_index(int64_t u, int bn, int q, int c, int g,
                                                    int lane) {
  return (((u * 4 + q) * (bn / 64) + c) * 16 + g) * 32 + lane;
}

// Eight fp16 values of C (uint4) plus eight accumulator words -> eight fp16
// of D = alpha * acc + beta * C.
__device__ __forceinline__ uint4 add_c8(const LargeArgs& p, const uint32_t* r, uint4 c) {
  const __half2* ch = reinterpret_cast<const __half2*>(&c);
  uint4 o;
  __half2* oh = reinterpret_cast<__half2*>(&o);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = r[2 * j], hi = r[2 * j + 1];
    if (p.acc_f16) {
      const __half2 acc = __halves2half2(__ushort_as_half(static_cast<unsigned short>(lo)),
                                         __ushort_as_half(static_cast<unsigned short>(hi)));
      oh[j] = epi_f16x2(p.e, acc, ch[j]);
    } else {
      oh[j] = epi_f32x2(p.e, __uint_as_float(lo), __uint_as_float(hi), ch[j]);
    }
  }
  return o;
}

// One 16-byte piece of a 32 x 64 C chunk for the coalesced load pattern:
// load i (0..7) of lane l covers row 4i + l/8, columns 8*(l%8) .. +8.
// cb is problem tb's C; zeros when C is not read.
__device__ __forceinline__ uint4 load_c_piece(const LargeArgs& p, const __half* cb, int m, int n) {
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (p.e.read_c && m < p.M && n < p.N) {
    const __half* src = cb + static_cast<int64_t>(m) * p.e.ldC + n;
    if (n + 8 <= p.N) {
      v = *reinterpret_cast<const uint4*>(src);
    } else {
      __half* vh = reinterpret_cast<__half*>(&v);
      for (int j = 0; j < 8 && n + j < p.N; ++j) vh[j] = src[j];
    }
  }
  return v;
}

// ---------------------------------------------------------------------------
// Staged epilogue of one warp: 32 rows x 64 columns per chunk.
//
// C arrives in a coalesced pattern (8 lanes per 128-byte row segment) into a
// 128-byte-swizzled staging buffer; each lane then adds its own TMEM row to
// its staged row (conflict-free thanks to the swizzle) and the chunk leaves
// by one TMA store, which also clips the row tail.  A right edge with N not
// a multiple of 8 is copied out with plain stores instead, because a TMA
// store writes whole 16-byte pieces.
constexpr uint32_t kStagingBytes = 32 * 128;  // 32 rows x 64 fp16

// C pieces of the chunk with rows m_base.., columns n_base..: piece i of lane
// l is row 4i + l/8, 16-byte segment l%8.
__device__ __forceinline__ void epi_load_c(const LargeArgs& p, const __half* cb, int m_base,
                                           int n_base, uint32_t lane, uint4 (&v)[8]) {
  const int prow = static_cast<int>(lane >> 3), pseg = static_cast<int>(lane & 7);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = load_c_piece(p, cb, m_base + 4 * i + prow, n_base + 8 * pseg);
}

// (Nothing to stage when C is not read: the add then skips the buffer.)
__device__ __forceinline__ void epi_stage_c(const LargeArgs& p, uint8_t* stg, uint32_t lane,
                                            const uint4 (&v)[8]) {
  if (!p.e.read_c) return;
  const int prow = static_cast<int>(lane >> 3), pseg = static_cast<int>(lane & 7);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 4 * i + prow;
    *reinterpret_cast<uint4*>(stg + r * 128 + 16 * (pseg ^ (r & 7))) = v[i];
  }
}

// Plain-store copy of this lane's staged row, columns [n0, n0 + ncols), for
// a chunk that a TMA store of 64 columns would overrun: a right edge with
// N % 8 != 0, or the 32-column last chunk of a tile whose width is not a
// multiple of 64 (kept out of line: it runs at most once per tile row).
__device__ __noinline__ void epi_store_ragged(const LargeArgs& p, const uint8_t* my_row,
                                              uint32_t lane, int tb, int m, int n0, int ncols) {
  if (m >= p.M || ncols <= 0) return;
  __half* drow = p.e.D + tb * p.e.sD + static_cast<int64_t>(m) * p.e.ldD + n0;
  for (int s8 = 0; 8 * s8 < ncols; ++s8) {
    const uint4 v =
        *reinterpret_cast<const uint4*>(my_row + 16 * (s8 ^ static_cast<int>(lane & 7)));
    if (8 * s8 + 8 <= ncols) {
      *reinterpret_cast<uint4*>(drow + 8 * s8) = v;
    } else {
      const __half* vh = reinterpret_cast<const __half*>(&v);
      for (int j = 0; 8 * s8 + j < ncols; ++j) drow[8 * s8 + j] = vh[j];
    }
  }
}

// Combine this lane's accumulator row r (64 words) with its staged C row
// (or scale it alone when C is not read: nothing was staged then),
// then store the chunk whose first element is D(m_row0, n0) of problem tb;
// only its first `width` columns (64, or 32 for the last chunk of a tile
// whose width is an odd multiple of 32) belong to the tile.  Returns (in
// lane 0) whether the chunk left by a TMA store, i.e. whether one bulk
// group now reads the staging buffer.
__device__ __forceinline__ bool epi_store_chunk(const LargeArgs& p, const CUtensorMap* tmD,
                                                uint8_t* stg, uint32_t stg_u32, uint32_t lane,
                                                int tb, int m_row0, int n0,
                                                const uint32_t (&r)[64], int width = 64) {
  uint8_t* my_row = stg + lane * 128;
  if (p.e.read_c) {
#pragma unroll
    for (int s8 = 0; s8 < 8; ++s8) {
      uint4* q = reinterpret_cast<uint4*>(my_row + 16 * (s8 ^ static_cast<int>(lane & 7)));
      *q = add_c8(p, r + 8 * s8, *q);
    }
  } else {
#pragma unroll
    for (int s8 = 0; s8 < 8; ++s8)
      *reinterpret_cast<uint4*>(my_row + 16 * (s8 ^ static_cast<int>(lane & 7))) =
          add_c8(p, r + 8 * s8, make_uint4(0u, 0u, 0u, 0u));
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (width < 64 || (n0 + 64 > p.N && (p.N & 7))) {
    epi_store_ragged(p, my_row, lane, tb, m_row0 + static_cast<int>(lane), n0,
                     min(width, p.N - n0));
  } else if (lane == 0 && m_row0 < p.M && n0 < p.N) {
    tma_store_3d(tmD, stg_u32, n0, m_row0, tb);
    bulk_commit_group();
    return true;
  }
  return false;
}

// KO: stages of 128 of K loaded as K-chunk boxes (see the header); p.k_blocks
// then counts blocks of 128.
template <int BN, bool KO = false>
__global__ void __launch_bounds__(kLargeThreads, 1)
    gemm_tn_large_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmD, const LargeArgs p) {
  using L = LargeSmem<BN, KO>;
  constexpr int kStages = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;                             // stage s at s * kABytes
  uint8_t* sB = smem + kStages * L::kABytes;      // stage s at s * kBBytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kCtlOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kCtlOffset + 4);

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + kStages);
  const uint32_t tfull0 = smem_u32(bars + 2 * kStages);
  const uint32_t tempty0 = smem_u32(bars + 2 * kStages + 2);
  const uint32_t drain = smem_u32(bars + 2 * kStages + 4);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  // The next kernel in the stream (this call's reduction, or the next
  // call's kernel) may become resident now; it waits for this grid's
  // completion before it touches memory.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    trace_entry(p.trace);
    trace_value(p.trace, kTrSm, sm_id());
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, LargeEpi<BN>::kWarps);  // one arrival per epilogue warp
    }
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
    tmem_alloc(smem_u32(tmem_slot), 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Programmatic dependent launch: the kernel before this one in the stream
  // (which may write A, B or C, or read a workspace this call reuses) must
  // be complete before any global memory is touched.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) trace_mark(p.trace, kTrReady);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;  // per stage: loads issued, their parity
      bool ok = true;
      int local = 0;
      const int units = p.num_tiles * p.ks_splits;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++local) {
        const int t = u / p.ks_splits, sp = u - t * p.ks_splits;
        const int kb0 = sp * p.ks_kb_per, kb1 = min(kb0 + p.ks_kb_per, p.k_blocks);
        int tb, tm, tn;
        batch_tile(p, t, tb, tm, tn);
        const int za = p.a_batched ? tb : 0, zb = p.b_batched ? tb : 0;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bounded(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.timeout_ns,
                            timeout_code(kRoleProducer, stage))) {
            ok = false;
            break;
          }
          const bool withhold = p.test_stall && local == 0 && kb == kb0;
          if (!withhold) {
            const uint32_t fb = full0 + 8 * stage;
            const uint32_t a_dst = smem_u32(sA + stage * L::kABytes);
            const uint32_t b_dst = smem_u32(sB + stage * L::kBBytes);
            mbar_arrive_expect_tx(fb, L::kStageBytes);
            if constexpr (KO) {
              // K chunks 2kb and 2kb+1 (the second zero-filled past K)
              tma_load_4d(a_dst, &tmA, fb, 0, tm * kLargeBM, 2 * kb, za);
              tma_load_4d(b_dst, &tmB, fb, 0, tn * BN, 2 * kb, zb);
            } else {
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
            }
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok || *abort_flag) {
        // Let every copy this thread issued land before the CTA can exit.
        for (int s = 0; s < kStages; ++s)
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
      bool ok = true, first_stage = true;
      int done = 0;
      const int units = p.num_tiles * p.ks_splits;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++done) {
        const int sp = u % p.ks_splits;
        const int kb0 = sp * p.ks_kb_per, kb1 = min(kb0 + p.ks_kb_per, p.k_blocks);
        if (!wait_bounded(tempty0 + 8 * acc, acc_phase ^ 1u, abort_flag, p.timeout_ns,
                          timeout_code(kRoleMma, 0x200 + acc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bounded(full0 + 8 * stage, phase, abort_flag, p.timeout_ns,
                            timeout_code(kRoleMma, stage))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (first_stage) {
            trace_mark(p.trace, kTrFirstStage);
            first_stage = false;
          }
          const uint32_t a_base = smem_u32(sA + stage * L::kABytes);
          const uint32_t b_base = smem_u32(sB + stage * L::kBBytes);
#pragma unroll
          for (int k = 0; k < L::kBK / 16; ++k) {
            uint64_t ad, bd;
            if constexpr (KO) {
              // K chunk k/4 of each operand is a 128-row SW128 block
              ad = make_sw128_desc(a_base + (k >> 2) * (kLargeBM * 128) + (k & 3) * 32, 16, 1024);
              bd = make_sw128_desc(b_base + (k >> 2) * (BN * 128) + (k & 3) * 32, 16, 1024);
            } else {
              ad = p.a_mn ? make_sw128_desc(a_base + k * 2048, 8192, 1024)
                          : make_sw128_desc(a_base + k * 32, 16, 1024);
              bd = p.b_mn ? make_sw128_desc(b_base + k * 2048, 8192, 1024)
                          : make_sw128_desc(b_base + k * 32, 16, 1024);
            }
            mma_f16(d_tmem, ad, bd, idesc, (kb != kb0) || (k != 0));
          }
          mma_commit(empty0 + 8 * stage);  // stage free once these MMAs have read it
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * acc);  // accumulator complete
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      trace_mark(p.trace, kTrLastMma);
      trace_value(p.trace, kTrUnits, static_cast<uint64_t>(done));
      if (!ok || *abort_flag) {
        // Wait until every MMA issued so far has finished with TMEM and smem.
        mma_commit(drain);
        wait_bounded(drain, 0, abort_flag, p.timeout_ns, timeout_code(kRoleMma, 0x300), false);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Staged: C of the next tile is fetched (coalesced) while its MMAs run;
    // per 64-column chunk the accumulator row is added to the staged C row
    // and the chunk leaves by TMA store.  Eight warps, two per TMEM lane
    // quadrant, each drain one half of the tile's columns through one
    // staging buffer, so that an accumulator is free again after
    // BN / 128 chunk times.
    const uint32_t quad = static_cast<uint32_t>(warp & 3);  // TMEM lanes 32*quad ..
    const int ew = warp - 2;                                // 0..7
    const int half = ew >> 2;                               // column half of the tile
    const int row0 = static_cast<int>(quad * 32);            // first tile row of this warp
    using E = LargeEpi<BN>;
    constexpr int kChunks = E::kChunks;                      // 64-column chunks per warp
    const int col0 = half * E::kColsPerWarp;                 // first tile column of this warp
    // with 64-wide tiles the second warp of each quadrant has no columns
    const bool epi_active = ew < E::kWarps;
    uint8_t* stg = smem + L::kStagingOffset + (epi_active ? ew : 0) * kStagingBytes;
    const uint32_t stg_u32 = smem_u32(stg);
    uint32_t acc = 0, acc_phase = 0;
    uint4 cnext[8];
    const int units = epi_active ? p.num_tiles * p.ks_splits : 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      if (p.ks_splits > 1) {
        // split-K unit: this warp's 32 rows x kColsPerWarp of the fp32 partial tile -> ks_ws
        if (!wait_bounded(tfull0 + 8 * acc, acc_phase, abort_flag, p.timeout_ns,
                          timeout_code(kRoleEpilogue, acc)))
          break;
        tc_fence_after();
        const uint32_t t_row = tmem_base + ((quad * 32) << 16) + acc * BN + col0;
        float4* ws4 = reinterpret_cast<float4*>(p.ks_ws);
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c) {
          uint32_t r[64];
          tmem_ld_32x32b_x32(t_row + c * 64, *reinterpret_cast<uint32_t(*)[32]>(r));
          tmem_ld_32x32b_x32(t_row + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
          tmem_wait_ld();
          if (c == kChunks - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
          }
          const int gc = half * kChunks + c;  // chunk of the tile
#pragma unroll
          for (int g = 0; g < 16; ++g)
            ws4[ks_partial_index(u, BN, static_cast<int>(quad), gc, g, static_cast<int>(lane))] =
                make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                            __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3]));
        }
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
        continue;
      }
      const int t = u;
      int tb, tm, tn;
      batch_tile(p, t, tb, tm, tn);
      const __half* cb = p.e.read_c ? p.e.C + tb * p.e.sC : nullptr;
      const int m_base = tm * kLargeBM + row0, n_base = tn * BN + col0;
      // chunk 0 of C staged (and chunk 1 in registers)
      epi_load_c(p, cb, m_base, n_base, lane, cnext);
      if (lane == 0) bulk_wait_group_read0();  // the last store has read the buffer
      __syncwarp();
      epi_stage_c(p, stg, lane, cnext);
      if (kChunks > 1) epi_load_c(p, cb, m_base, n_base + 64, lane, cnext);
      __syncwarp();
      if (!wait_bounded(tfull0 + 8 * acc, acc_phase, abort_flag, p.timeout_ns,
                        timeout_code(kRoleEpilogue, acc)))
        break;
      tc_fence_after();
      if (ew == 0 && lane == 0 && u == static_cast<int>(blockIdx.x))
        trace_mark(p.trace, kTrFirstAcc);
      const uint32_t t_row = tmem_base + ((quad * 32) << 16) + acc * BN + col0;
#pragma unroll 1
      for (int c = 0; c < kChunks; ++c) {
        if (c > 0) {
          if (lane == 0) bulk_wait_group_read0();
          __syncwarp();
          epi_stage_c(p, stg, lane, cnext);
          if (c + 1 < kChunks) epi_load_c(p, cb, m_base, n_base + 64 * (c + 1), lane, cnext);
          __syncwarp();
        }
        uint32_t r[64];
        tmem_ld_32x32b_x32(t_row + c * 64, *reinterpret_cast<uint32_t(*)[32]>(r));
        tmem_ld_32x32b_x32(t_row + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
        tmem_wait_ld();
        if (c == kChunks - 1) {
          // every column of this warp's share is in registers: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
        }
        epi_store_chunk(p, &tmD, stg, stg_u32, lane, tb, m_base, n_base + 64 * c, r);
      }
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (ew == 0 && lane == 0) trace_mark(p.trace, kTrLastChunk);
    if (lane == 0) bulk_wait_group0();  // all D stores performed before exit
    if (ew == 0 && lane == 0) trace_mark(p.trace, kTrStoresDone);
    __syncwarp();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) trace_exit(p.trace);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * BN);
  }
}

// Sum of the split-K partials of one 32 x 64 piece of a tile, in split order,
// then the epilogue: D = alpha * sum + beta * C (see EpiArgs).  Block
// (piece, tile): piece = quadrant q (32 rows) x chunk c (64 columns).  The
// partial float4s are read in their stored order (whole lines), the sums go
// through shared memory, and C / D move as 16-byte row segments.  Launched
// as a programmatic dependent of the split kernel.
constexpr int kTileReduceThreads = 256;

template <int BN>
__global__ void __launch_bounds__(kTileReduceThreads)
    gemm_tn_tile_reduce_kernel(const LargeArgs p) {
  // The next call's kernels may become resident now (they wait for this
  // grid's completion before touching memory).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ float sum[32][64 + 4];
  const int t = static_cast<int>(blockIdx.y);  // partial slot (split tile t of the launch)
  const int piece = static_cast<int>(blockIdx.x);
  const int q = piece / (BN / 64), c = piece - q * (BN / 64);
  const float4* ws4 = reinterpret_cast<const float4*>(p.ks_ws);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int f = static_cast<int>(threadIdx.x) + h * kTileReduceThreads;  // 0..511
    const int g = f >> 5, lane = f & 31;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp = 0; sp < p.ks_splits; ++sp) {
      const float4 v = __ldcg(ws4 + ks_partial_index(static_cast<int64_t>(t) * p.ks_splits + sp,
                                                     BN, q, c, g, lane));
      a.x += v.x;
      a.y += v.y;
      a.z += v.z;
      a.w += v.w;
    }
    sum[lane][4 * g] = a.x;
    sum[lane][4 * g + 1] = a.y;
    sum[lane][4 * g + 2] = a.z;
    sum[lane][4 * g + 3] = a.w;
  }
  __syncthreads();
  int tb, tm, tn;
  batch_tile(p, p.ks_tile0 + t, tb, tm, tn);
  const int r = static_cast<int>(threadIdx.x) >> 3, seg = static_cast<int>(threadIdx.x) & 7;
  const int m = tm * kLargeBM + 32 * q + r, n = tn * BN + 64 * c + 8 * seg;
  if (m >= p.M || n >= p.N) return;
  const EpiArgs& e = p.e;
  const __half* crow = e.read_c ? e.C + tb * e.sC + static_cast<int64_t>(m) * e.ldC : nullptr;
  __half* drow = e.D + tb * e.sD + static_cast<int64_t>(m) * e.ldD;
  if (n + 8 <= p.N) {
    uint4 cv = make_uint4(0u, 0u, 0u, 0u);
    if (e.read_c) cv = *reinterpret_cast<const uint4*>(crow + n);
    const __half2* ch = reinterpret_cast<const __half2*>(&cv);
    uint4 o;
    __half2* oh = reinterpret_cast<__half2*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      oh[j] = epi_f32x2(e, sum[r][8 * seg + 2 * j], sum[r][8 * seg + 2 * j + 1], ch[j]);
    *reinterpret_cast<uint4*>(drow + n) = o;
  } else {
    for (int j = 0; n + j < p.N; ++j) {
      const __half cj = e.read_c ? crow[n + j] : __ushort_as_half(0);
      drow[n + j] = epi_one(e, false, __float_as_uint(sum[r][8 * seg + j]), cj);
    }
  }
}

}  // namespace gemm_tn_dev
