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
//     (conflict-free), and D leaves by TMA store, which also clips the tails
//     (all but a right edge with N % 8 != 0: the TMA store writes whole
//     16-byte pieces, so that chunk is copied out with plain stores).
//     The next tile's C rows are prefetched into L2 during its main loop, and
//     the TMA ring keeps loading the next tile's first stages meanwhile.
//
// Stream-K (the make_tiled_mma page's K split across workers, "Thread groups
// along K, and the loop along K": partial sums must be reduced and C added
// once): whole tiles go round-robin; the tiles of the last, partial wave
// (t >= sk_tile0) are cut into contiguous (tile, K-block) ranges of equal
// length, one per CTA.  A CTA whose range covers a whole tile finishes it directly.
// Otherwise each of its epilogue warps writes its 32 x 256 slab of the fp32
// partial sum, fences, and takes a ticket on the (tile, slab) counter; the
// warp that takes the last ticket adds the slab's partials of all
// contributors in CTA order (deterministic), adds C once, rounds and stores
// D.  A warp that finds every other contributor already done skips its own
// partial and finishes from TMEM; the sum, and its order, are the same.  No
// CTA ever waits for another.  Partials are stored in 4-column groups
// (float4 per lane, lanes on consecutive rows) so that every store and load
// moves whole lines.
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
constexpr uint32_t kWideStagingBytes = kStagingBytes;
// Stream-K partials: one 32-row x 64-column fp32 block of a warp's slab is
// 8 KiB, stored as [column group g (16)][lane (32)] float4.
constexpr uint32_t kSkBlockBytes = 32 * 64 * 4;
constexpr int kFinBufs = 3;  // finisher landing buffers per epilogue warp

struct WideSmem {
  static constexpr uint32_t kABytes = kWideBM * kWideBK * 2;  // 32 KiB
  static constexpr uint32_t kBBytes = kWideBN * kWideBK * 2;  // 32 KiB
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kStagingOffset = kWideStages * kStageBytes;  // 1024-aligned
  static constexpr uint32_t kBarOffset = kStagingOffset + kWideEpiWarps * kWideStagingBytes;
  // full[S], empty[S], tmem_full, tmem_empty, drain, then the stream-K
  // finisher's landing-zone barriers (kFinBufs per epilogue warp)
  static constexpr uint32_t kFinBar0 = 2 * kWideStages + 3;
  static constexpr uint32_t kNumBars = kFinBar0 + kWideEpiWarps * kFinBufs;
  static constexpr uint32_t kCtlOffset = kBarOffset + kNumBars * 8;
  static constexpr uint32_t kBytes = kCtlOffset + 16;
  static constexpr uint32_t kDynamicBytes = kBytes + 1024;
};

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)),
               "r"(bytes)
               : "memory");
}

// One item of CTA c's work list: whole tiles first (round-robin), then the
// pieces of split tiles in its stream-K range.  slot < 0: the CTA computes
// the whole tile (direct epilogue); slot >= 0: partial sum, stored in slot.
struct WideItem {
  int tile, kb0, kb1, slot;
};

// First unit of CTA c's stream-K range.
__device__ __forceinline__ int sk_begin(const LargeArgs& p, int c) {
  return min(c * p.sk_per, p.sk_units);
}

__device__ __forceinline__ bool wide_item(const LargeArgs& p, int c, int G, int idx,
                                          WideItem& it) {
  const int n_dp = c < p.sk_tile0 ? (p.sk_tile0 - 1 - c) / G + 1 : 0;
  if (idx < n_dp) {
    it.tile = c + idx * G;
    it.kb0 = 0;
    it.kb1 = p.k_blocks;
    it.slot = -1;
    return true;
  }
  if (p.sk_units == 0) return false;
  const int j = idx - n_dp;
  const int ub = sk_begin(p, c), ue = sk_begin(p, c + 1);
  if (ue <= ub) return false;
  const int kb = p.k_blocks;
  const int ft = ub / kb;
  if (j > (ue - 1) / kb - ft) return false;
  const int rt = ft + j;
  const int t0 = rt * kb;
  const int lo = max(ub, t0), hi = min(ue, t0 + kb);
  it.tile = p.sk_tile0 + rt;
  it.kb0 = lo - t0;
  it.kb1 = hi - t0;
  it.slot = (it.kb0 == 0 && it.kb1 == kb) ? -1 : c * p.sk_max_segs + j;
  return true;
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
  const int cta = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
  // The next kernel in the stream (this call's reduction, or the next
  // call's kernel) may become resident now; it waits for this grid's
  // completion before it touches memory.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    trace_entry(p.trace);
    trace_value(p.trace, kTrSm, sm_id());
    for (int s = 0; s < kWideStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 8);  // eight epilogue warps
    mbar_init(drain, 1);
    for (int b = 0; b < kWideEpiWarps * kFinBufs; ++b) mbar_init(smem_u32(bars + L::kFinBar0 + b), 1);
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
  // Programmatic dependent launch: the kernel before this one in the stream
  // (which may write A, B or C, or read a workspace this call reuses) must
  // be complete before any global memory is touched.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) trace_mark(p.trace, kTrReady);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, issued_mask = 0, issued_parity = 0;
      bool ok = true;
      WideItem it;
      for (int idx = 0; ok && wide_item(p, cta, G, idx, it); ++idx) {
        int tb, tm, tn;
        batch_tile(p, it.tile, tb, tm, tn);
        const int za = p.a_batched ? tb : 0, zb = p.b_batched ? tb : 0;
        for (int kb = it.kb0; kb < it.kb1; ++kb) {
          if (!wait_bounded(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.timeout_ns,
                            timeout_code(kRoleProducer, stage))) {
            ok = false;
            break;
          }
          if (!(p.test_stall && idx == 0 && kb == it.kb0)) {
            const uint32_t fb = full0 + 8 * stage;
            const uint32_t a_dst = smem_u32(smem + stage * L::kStageBytes);
            const uint32_t b_dst = a_dst + L::kABytes;
            mbar_arrive_expect_tx(fb, L::kStageBytes);
            const int k0 = kb * kWideBK;
            if (!p.a_mn) {
              tma_load_3d(a_dst, &tmA, fb, k0, tm * kWideBM, za);
            } else {
#pragma unroll
              for (int i = 0; i < kWideBM / 64; ++i)
                tma_load_3d(a_dst + i * 8192, &tmA, fb, tm * kWideBM + 64 * i, k0, za);
            }
            if (!p.b_mn) {
              tma_load_3d(b_dst, &tmB, fb, k0, tn * kWideBN, zb);
            } else {
#pragma unroll
              for (int i = 0; i < kWideBN / 64; ++i)
                tma_load_3d(b_dst + i * 8192, &tmB, fb, tn * kWideBN + 64 * i, k0, zb);
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
      bool ok = true, first_stage = true;
      int done = 0;
      WideItem it;
      for (int idx = 0; ok && wide_item(p, cta, G, idx, it); ++idx, ++done) {
        if (!wait_bounded(tempty, acc_phase ^ 1u, abort_flag, p.timeout_ns,
                          timeout_code(kRoleMma, 0x200))) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = it.kb0; kb < it.kb1; ++kb) {
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
              mma_f16(tmem_base + h * kWideBN, ad, bd, idesc, (kb != it.kb0) || (k != 0));
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
      trace_mark(p.trace, kTrLastMma);
      trace_value(p.trace, kTrUnits, static_cast<uint64_t>(done));
      if (!ok || *abort_flag) {
        mma_commit(drain);
        wait_bounded(drain, 0, abort_flag, p.timeout_ns, timeout_code(kRoleMma, 0x300), false);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;                                // 0..7: the warp's slab
    const int half = ew >> 2;                               // 128-row half of the tile
    const uint32_t quad = static_cast<uint32_t>(warp & 3);  // TMEM lanes 32*quad ..
    const int row0 = half * 128 + static_cast<int>(quad * 32);  // first tile row of this warp
    const int trow = row0 + static_cast<int>(lane);             // this lane's tile row
    uint8_t* stg = smem + L::kStagingOffset + ew * kWideStagingBytes;
    const uint32_t stg_u32 = smem_u32(stg);
    int tb = 0, tm = 0, tn = 0;
    const __half* cb = p.e.C;  // problem tb's C
    uint4 cnext[8];
    auto load_chunk = [&](int c, uint4 (&v)[8]) {
      epi_load_c(p, cb, tm * kWideBM + row0, tn * kWideBN + 64 * c, lane, v);
    };
    auto stage_chunk = [&](const uint4 (&v)[8]) { epi_stage_c(p, stg, lane, v); };
    // C of chunks 0 and 1 (0 staged, 1 in registers), once the previous
    // tile's last store has finished reading the staging buffer.
    auto preload_c = [&]() {
      load_chunk(0, cnext);
      if (lane == 0) bulk_wait_group_read0();
      __syncwarp();
      stage_chunk(cnext);
      load_chunk(1, cnext);
      __syncwarp();
    };
    // D = alpha * acc + beta * C for chunk c (64 columns) of this warp's
    // slab; acc words are fp32 (or fp16 in the low half) in r[0..64).
    auto emit_chunk = [&](int c, const uint32_t (&r)[64]) {
      if (c > 0) {
        if (lane == 0) bulk_wait_group_read0();  // previous store has read staging
        __syncwarp();
        stage_chunk(cnext);
        if (c + 1 < kWideBN / 64) load_chunk(c + 1, cnext);
        __syncwarp();
      }
      epi_store_chunk(p, &tmD, stg, stg_u32, lane, tb, tm * kWideBM + row0, tn * kWideBN + 64 * c,
                      r);
    };
    auto load_tmem_chunk = [&](int c, uint32_t (&r)[64]) {
      const uint32_t t_row = tmem_base + ((quad * 32) << 16) + half * kWideBN;
      tmem_ld_32x32b_x32(t_row + c * 64, *reinterpret_cast<uint32_t(*)[32]>(r));
      tmem_ld_32x32b_x32(t_row + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
      tmem_wait_ld();
      if (c == kWideBN / 64 - 1) {
        // every TMEM column of this warp is in registers: hand the
        // accumulator back so the next item's MMAs can start
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty);
      }
    };
    // Warm L2 with this warp's C rows of a whole tile (one row per lane).
    auto prefetch_c = [&](int idx2) {
      WideItem nx;
      if (!wide_item(p, cta, G, idx2, nx)) return;
      int tb2, tm2, tn2;
      batch_tile(p, nx.tile, tb2, tm2, tn2);
      const int m2 = tm2 * kWideBM + trow;
      const int n2 = tn2 * kWideBN;
      if (p.e.read_c && m2 < p.M && n2 < p.N) {
        const uint32_t bytes = static_cast<uint32_t>(min(kWideBN, p.N - n2) * 2) & ~15u;
        if (bytes)
          prefetch_l2(p.e.C + tb2 * p.e.sC + static_cast<int64_t>(m2) * p.e.ldC + n2, bytes);
      }
    };
    prefetch_c(0);
    uint32_t acc_phase = 0;
    WideItem it;
    for (int idx = 0; wide_item(p, cta, G, idx, it); ++idx) {
      batch_tile(p, it.tile, tb, tm, tn);
      cb = p.e.read_c ? p.e.C + tb * p.e.sC : nullptr;
      // C does not depend on the MMAs: fetch it now (for a partial tile too,
      // in case this warp turns out to finish it; the staging buffer is
      // otherwise idle on such an item)
      preload_c();
      WideItem nx;
      const bool last_item = !wide_item(p, cta, G, idx + 1, nx);
      if (!wait_bounded(tfull, acc_phase, abort_flag, p.timeout_ns,
                        timeout_code(kRoleEpilogue, 0)))
        break;
      if (ew == 0 && lane == 0 && idx == 0) trace_mark(p.trace, kTrFirstAcc);
      tc_fence_after();
      if (it.slot < 0) {
#pragma unroll 1
        for (int c = 0; c < kWideBN / 64; ++c) {
          uint32_t r[64];
          load_tmem_chunk(c, r);
          emit_chunk(c, r);
        }
        acc_phase ^= 1u;
        prefetch_c(idx + 1);
        continue;
      }
      // Stream-K state of a partial tile.
      int rt = 0, c_first = 0, c_last = 0, n_mem = 0, n_loads = 0;
      bool own_in_tmem = true, staged = false;
      const uint32_t zone = smem_u32(smem + ew * (kFinBufs * kSkBlockBytes));
      const uint32_t fbar = smem_u32(bars + L::kFinBar0 + ew * kFinBufs);
      // this warp's 8 KiB block (slab ew, chunk c) of contributor c2's slot
      auto block_of = [&](int c2, int c) -> const float4* {
        const int j2 = rt - (c2 * p.sk_per) / p.k_blocks;
        return reinterpret_cast<const float4*>(p.sk_partials) +
               static_cast<int64_t>(c2 * p.sk_max_segs + j2) * (kWideBM * kWideBN / 4) +
               (ew * 4 + c) * (kSkBlockBytes / 16);
      };
      // bulk load i: chunk i / n_mem of the (i % n_mem)-th contributor kept in memory
      auto issue = [&](int i) {
        const int c = i / n_mem;
        int c2 = c_first + (i - c * n_mem);
        if (own_in_tmem && c2 >= cta) ++c2;  // skip this CTA's own term
        const int buf = i % kFinBufs;
        mbar_arrive_expect_tx(fbar + 8 * buf, kSkBlockBytes);
        bulk_load_g2s(zone + buf * kSkBlockBytes, block_of(c2, c), kSkBlockBytes, fbar + 8 * buf);
      };
      {
        // partial tile.  Contributors: CTAs c_first..c_last, every one with
        // a non-empty share.
        rt = it.tile - p.sk_tile0;
        const int u0 = rt * p.k_blocks;
        c_first = u0 / p.sk_per;
        c_last = (u0 + p.k_blocks - 1) / p.sk_per;
        const int n_contrib = c_last - c_first + 1;
        int* counter = p.sk_counters + rt * 8 + ew;
        // If every other contributor has already published its slab, this
        // warp finishes the slab straight from TMEM (no partial of its own
        // goes through memory); no other warp can then reach the last ticket.
        const int done = ld_acquire_gpu(counter);  // every lane acquires for its own loads
        bool finish = done == n_contrib - 1;
        own_in_tmem = finish;
        if (!finish) {
          // publish this slab's fp32 partial sum, then take a ticket
          float4* part = reinterpret_cast<float4*>(p.sk_partials) +
                         static_cast<int64_t>(it.slot) * (kWideBM * kWideBN / 4);
#pragma unroll 1
          for (int c = 0; c < kWideBN / 64; ++c) {
            uint32_t r[64];
            load_tmem_chunk(c, r);
            float4* dst = part + (ew * 4 + c) * (kSkBlockBytes / 16) + lane;
#pragma unroll
            for (int g = 0; g < 16; ++g)
              dst[32 * g] = make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                                        __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3]));
          }
          __threadfence();
          __syncwarp();
          int ticket = 0;
          if (lane == 0) ticket = atomicAdd(counter, 1);
          ticket = __shfl_sync(0xffffffffu, ticket, 0);
          finish = ticket == n_contrib - 1;
          if (finish) __threadfence();
        }
        if (!finish) {
          acc_phase ^= 1u;
          prefetch_c(idx + 1);
          continue;
        }
        // This warp finishes the slab: every other contributor's slab is in
        // memory.  On the CTA's last item the main-loop stages are idle (its
        // MMAs have completed), so the blocks come in by bulk copy, three in
        // flight per warp; otherwise by plain loads.
        staged = last_item;
        n_mem = n_contrib - (own_in_tmem ? 1 : 0);
        n_loads = n_mem * (kWideBN / 64);
        if (staged && lane == 0) {
          fence_proxy_async_global();
          for (int i = 0; i < min(kFinBufs, n_loads); ++i) issue(i);
        }
      }
      bool ok = true;
      int next = 0;  // next bulk load to consume
#pragma unroll 1
      for (int c = 0; c < kWideBN / 64; ++c) {
        uint32_t r[64];
        {
          // all terms in CTA order (this CTA's own from TMEM or from memory)
          float4 acc[16];
#pragma unroll
          for (int g = 0; g < 16; ++g) acc[g] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
          for (int c2 = c_first; c2 <= c_last; ++c2) {
            if (own_in_tmem && c2 == cta) {
              // 16 columns at a time: a whole 64-column chunk next to acc
              // and the held C chunk would not fit the register budget
              const uint32_t t_row = tmem_base + ((quad * 32) << 16) + half * kWideBN + c * 64;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                uint32_t t[16];
                tmem_ld_32x32b_x16(t_row + 16 * q, t);
                tmem_wait_ld();
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                  acc[4 * q + g].x += __uint_as_float(t[4 * g]);
                  acc[4 * q + g].y += __uint_as_float(t[4 * g + 1]);
                  acc[4 * q + g].z += __uint_as_float(t[4 * g + 2]);
                  acc[4 * q + g].w += __uint_as_float(t[4 * g + 3]);
                }
              }
              if (c == kWideBN / 64 - 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty);
              }
            } else if (staged) {
              const int buf = next % kFinBufs;
              if (!wait_bounded(fbar + 8 * buf, static_cast<uint32_t>(next / kFinBufs) & 1u,
                                abort_flag, p.timeout_ns, timeout_code(kRoleEpilogue, 0x10),
                                false)) {
                // give the copies still in flight a bounded chance to land
                for (int i = next + 1; i < min(next + kFinBufs, n_loads); ++i)
                  wait_bounded(fbar + 8 * (i % kFinBufs), static_cast<uint32_t>(i / kFinBufs) & 1u,
                               abort_flag, p.timeout_ns, timeout_code(kRoleEpilogue, 0x11), false);
                ok = false;
                break;
              }
              const float4* blk =
                  reinterpret_cast<const float4*>(smem + ew * (kFinBufs * kSkBlockBytes) +
                                                  buf * kSkBlockBytes) +
                  lane;
#pragma unroll
              for (int g = 0; g < 16; ++g) {
                const float4 v = blk[32 * g];
                acc[g].x += v.x;
                acc[g].y += v.y;
                acc[g].z += v.z;
                acc[g].w += v.w;
              }
              __syncwarp();  // every lane has read the buffer before it is refilled
              if (lane == 0 && next + kFinBufs < n_loads) {
                fence_proxy_async_smem();
                issue(next + kFinBufs);
              }
              ++next;
            } else {
              const float4* src = block_of(c2, c) + lane;
              // two halves of eight column groups keep the registers in
              // budget next to the C chunk held for the next store
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                float4 v[8];
#pragma unroll
                for (int g = 0; g < 8; ++g) v[g] = __ldcg(src + 32 * (8 * h + g));
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                  acc[8 * h + g].x += v[g].x;
                  acc[8 * h + g].y += v[g].y;
                  acc[8 * h + g].z += v[g].z;
                  acc[8 * h + g].w += v[g].w;
                }
              }
            }
          }
          if (!ok) break;
#pragma unroll
          for (int g = 0; g < 16; ++g) {
            r[4 * g] = __float_as_uint(acc[g].x);
            r[4 * g + 1] = __float_as_uint(acc[g].y);
            r[4 * g + 2] = __float_as_uint(acc[g].z);
            r[4 * g + 3] = __float_as_uint(acc[g].w);
          }
        }
        emit_chunk(c, r);
      }
      if (!ok) break;
      acc_phase ^= 1u;
      prefetch_c(idx + 1);
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
    tmem_dealloc(tmem_base, kWideTmemCols);
  }
}

}  // namespace gemm_tn_dev
