// gemm_large2.cuh -- persistent tcgen05 TN GEMM on CTA pairs (cta_group::2).
//
// Same computation and tiling scheme as gemm_large.cuh, but two CTAs on two
// SMs (a cluster of 2) compute one 256 x 256 output tile together:
//
//   * CTA r of the pair TMA-loads rows [128r, 128r+128) of the tile's A block
//     and rows [128r, 128r+128) of its B block into its own ring, so each SM
//     pulls 64 B per clock of tensor work instead of 96 B with 128 x 256
//     single-CTA tiles.  With DEEP the ring has 3 stages of 128 of K (two
//     64-deep sub-blocks per operand, each loaded as in the 64-deep layout;
//     64 KiB per CTA), and a sub-block past K is zero-filled by the copy;
//     otherwise 6 stages of one 64-deep K block.  Deep stages halve the
//     stage hand-offs per byte and win from K = 1024 on.
//   * One thread of the even CTA issues tcgen05.mma.cta_group::2 with
//     M = 256, N = 256, K = 16: the instruction reads A from both CTAs'
//     shared memory (split along M) and B from both (split along N), and
//     writes rows [128r, 128r+128) of D into CTA r's tensor memory.
//   * Stage completion: both CTAs' copies of a stage count their bytes on
//     the even CTA's `full` barrier (cta_group::2 loads may signal a barrier
//     in the peer CTA), which the even CTA's producer arms with the bytes of
//     the whole pair stage; so the MMA thread sees a stage as soon as the
//     last of its four boxes has landed, with no hop through the odd CTA.
//     The MMA thread releases a stage in both CTAs with one multicast
//     tcgen05.commit; accumulators are handed to both CTAs' epilogues the
//     same way, and the sixteen epilogue warps of the pair return an
//     accumulator by arriving on the even CTA's `tmem_empty`.
//   * Each CTA's epilogue is the staged one of gemm_large.cuh on its 128
//     rows of the tile, with two accumulators so it overlaps the next
//     tile's main loop; eight warps, two per TMEM lane quadrant, each drain
//     one 128-column half, so that an accumulator is free again after two
//     chunk times (with short K loops the drain, not the MMA, set the pace).
//   * The tile width p.bn is chosen per call (256, 224, 192, 160 or 128):
//     each CTA holds bn / 2 rows of B, the MMA runs with N = bn, and the
//     epilogue drains bn columns in 64-column chunks (the last one 32 wide
//     when bn is an odd multiple of 32), so that the number of tiles can be
//     matched to the number of pairs.
//   * Work units are tiles, or with ks_splits > 1 (tile, K range) pairs
//     (the make_tiled_mma page's K split across workers): a split unit's
//     CTAs store their fp32 rows as 128-row partial tiles 2t and 2t + 1, and
//     gemm_tn_tile_reduce_kernel adds the splits in order and C once.
//
// Every wait is bounded; a CTA that gives up raises its own and its peer's
// abort flag, both drain what they issued, free the pair's TMEM and return.
#pragma once

#include "gemm_large.cuh"

namespace gemm_tn_dev {

constexpr int kPairBM = 256;   // output rows per tile (128 per CTA)
constexpr int kPairBN = 256;   // widest tile (B rows: 128 per CTA); p.bn may be narrower
constexpr int kPairThreads = 320;  // producer warp, MMA warp, 8 epilogue warps
constexpr uint32_t kPairTmemCols = 512;  // two 256-column fp32 accumulators

template <bool DEEP = false>
struct PairSmem {
  static constexpr int kBK = DEEP ? 128 : 64;  // K per stage (= p.k_blocks unit)
  static constexpr int kStages = DEEP ? 3 : 6;
  static constexpr uint32_t kABytes = 128 * kBK * 2;  // 16 / 32 KiB
  static constexpr uint32_t kBBytes = 128 * kBK * 2;  // 16 / 32 KiB
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  // epilogue staging: 8 warps x 32 rows x 64 fp16 (1024-aligned)
  static constexpr uint32_t kStagingOffset = kStages * kStageBytes;
  static constexpr uint32_t kBarOffset = kStagingOffset + 8 * kStagingBytes;
  static constexpr uint32_t kNumBars = 2 * kStages + 5;
  static constexpr uint32_t kCtlOffset = kBarOffset + kNumBars * 8;
  static constexpr uint32_t kBytes = kCtlOffset + 16;
  static constexpr uint32_t kDynamicBytes = kBytes + 1024;
  static_assert(kDynamicBytes <= 232448, "over the 227 KiB of shared memory per CTA");
};

// Work units: with ks_splits == 1 unit u is tile u; otherwise units below
// ks_tile0 are whole tiles and unit ks_tile0 + v is split v % ks_splits of
// tile ks_tile0 + v / ks_splits.  Sets the tile, its K blocks [kb0, kb1) and
// the partial slot of a split unit (-1 for a whole tile).
__device__ __forceinline__ void pair_unit(const LargeArgs& p, int u, int& t, int& kb0, int& kb1,
                                          int64_t& slot) {
  if (p.ks_splits <= 1 || u < p.ks_tile0) {
    t = u;
    kb0 = 0;
    kb1 = p.k_blocks;
    slot = -1;
    return;
  }
  const int v = u - p.ks_tile0;
  const int j = v / p.ks_splits, sp = v - j * p.ks_splits;
  t = p.ks_tile0 + j;
  kb0 = sp * p.ks_kb_per;
  kb1 = min(kb0 + p.ks_kb_per, p.k_blocks);
  slot = static_cast<int64_t>(j) * p.ks_splits + sp;  // split tile j, split sp
}

__device__ __forceinline__ int pair_units(const LargeArgs& p) {
  return p.ks_splits > 1 ? p.ks_tile0 + (p.num_tiles - p.ks_tile0) * p.ks_splits : p.num_tiles;
}

template <bool DEEP = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    gemm_tn_large2_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmD, const LargeArgs p) {
  using L = PairSmem<DEEP>;
  constexpr int kPairStages = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // stage s: A half at s*kStageBytes, B half right after (both 1024-aligned)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kCtlOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kCtlOffset + 4);

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + kPairStages);
  const uint32_t tfull0 = smem_u32(bars + 2 * kPairStages);
  const uint32_t tempty0 = smem_u32(bars + 2 * kPairStages + 2);
  const uint32_t drain = smem_u32(bars + 2 * kPairStages + 4);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs, 1: peer
  const bool leader = rank == 0;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int num_pairs = static_cast<int>(gridDim.x >> 1);
  const int units = pair_units(p);  // work units, round-robin over the pairs
  // The next kernel in the stream (this call's reduction, or the next
  // call's kernel) may become resident now; it waits for this grid's
  // completion before it touches memory.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    trace_entry(p.trace);
    trace_value(p.trace, kTrSm, sm_id());
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(full0 + 8 * s, 1);  // the even CTA's arming; both CTAs' bytes (odd: unused)
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 16);  // the pair's sixteen epilogue warps
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
    tmem_alloc_pair(smem_u32(tmem_slot), kPairTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t peer_abort = mapa_shared(smem_u32(smem + L::kCtlOffset), rank ^ 1u);
  // Programmatic dependent launch: the kernel before this one in the stream
  // (which may write A, B or C, or read a workspace this call reuses) must
  // be complete before any global memory is touched.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) trace_mark(p.trace, kTrReady);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // Both CTAs' copies signal the even CTA's full barrier; only the even
      // CTA arms it (arrival plus the pair stage's bytes).  A copy of the odd
      // CTA may land before the arming: the barrier's transaction count then
      // runs below zero for a while, and the phase still cannot complete
      // without the arrival.  Neither CTA can start a stage's next phase
      // before the MMA thread has released the stage in both (the multicast
      // commit on `empty`), which it does only after the phase completed, so
      // no copy can count against the wrong phase.
      const uint32_t full_pair0 = mapa_shared(full0, 0);
      // bytes of one pair stage: each CTA's A box(es) and its bn / 2 rows of
      // B (K-major: one box of bn / 2 rows; M/N-major: 64-wide boxes, the
      // last possibly reaching past this CTA's rows)
      const int b_half = p.bn / 2;
      const int b_boxes_mn = (b_half + 63) / 64;
      const uint32_t b_sub_bytes = p.b_mn ? b_boxes_mn * 8192u : b_half * 128u;
      const uint32_t pair_stage_bytes = 2u * (L::kBK / 64) * (16384u + b_sub_bytes);
      uint32_t stage = 0, phase = 0, issued_mask = 0, issued_parity = 0;
      bool ok = true;
      int local = 0;
      for (int u = pair; ok && u < units; u += num_pairs, ++local) {
        int t, kb0, kb1;
        int64_t slot;
        pair_unit(p, u, t, kb0, kb1, slot);
        int tb, tm, tn;
        batch_tile(p, t, tb, tm, tn);
        const int za = p.a_batched ? tb : 0, zb = p.b_batched ? tb : 0;
        const int a_row = tm * kPairBM + 128 * static_cast<int>(rank);
        const int b_row = tn * p.bn + b_half * static_cast<int>(rank);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bounded(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.timeout_ns,
                            timeout_code(kRoleProducer, stage), true, peer_abort)) {
            ok = false;
            break;
          }
          if (!(p.test_stall && local == 0 && kb == kb0)) {
            const uint32_t fb = full_pair0 + 8 * stage;
            const uint32_t a_dst = smem_u32(smem + stage * L::kStageBytes);
            const uint32_t b_dst = a_dst + L::kABytes;
            if (leader) mbar_arrive_expect_tx(full0 + 8 * stage, pair_stage_bytes);
            // 64-deep sub-blocks, 16 KiB apart; rows past M / N and K past the
            // end (up to a whole sub-block) are zero-filled
#pragma unroll
            for (int sub = 0; sub < L::kBK / 64; ++sub) {
              const int k0 = kb * L::kBK + 64 * sub;
              const uint32_t as = a_dst + sub * 16384, bs = b_dst + sub * 16384;
              if (!p.a_mn) {
                tma_load_3d_pair(as, &tmA, fb, k0, a_row, za);
              } else {
                tma_load_3d_pair(as, &tmA, fb, a_row, k0, za);
                tma_load_3d_pair(as + 8192, &tmA, fb, a_row + 64, k0, za);
              }
              if (!p.b_mn) {
                tma_load_3d_pair(bs, &tmB, fb, k0, b_row, zb);
              } else {
                tma_load_3d_pair(bs, &tmB, fb, b_row, k0, zb);
                if (b_boxes_mn > 1) tma_load_3d_pair(bs + 8192, &tmB, fb, b_row + 64, k0, zb);
              }
            }
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok || *abort_flag) {
        // Give every copy still in flight time to land before the CTA can
        // leave.  The even CTA sees its stages complete on `full` (which
        // also counts the odd CTA's bytes, so a phase the odd CTA never
        // loaded runs to the limit).  The odd CTA cannot watch its copies
        // directly; a stage it loaded is known landed once the MMA thread
        // has released it (`empty`), else it waits out the limit.
        for (int s = 0; s < kPairStages; ++s)
          if (issued_mask >> s & 1u)
            wait_bounded(leader ? full0 + 8 * s : empty0 + 8 * s, issued_parity >> s & 1u,
                         abort_flag, p.timeout_ns, timeout_code(kRoleProducer, 0x100 + s), false,
                         peer_abort);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t idesc = make_idesc_f16(kPairBM, p.bn, !p.acc_f16, p.a_mn, p.b_mn);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, first_stage = true;
      int done = 0;
      for (int u = pair; ok && u < units; u += num_pairs, ++done) {
        int t, kb0, kb1;
        int64_t slot;
        pair_unit(p, u, t, kb0, kb1, slot);
        if (!wait_bounded<true>(tempty0 + 8 * acc, acc_phase ^ 1u, abort_flag, p.timeout_ns,
                                timeout_code(kRoleMma, 0x200 + acc), true, peer_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kPairBN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bounded<true>(full0 + 8 * stage, phase, abort_flag, p.timeout_ns,
                                  timeout_code(kRoleMma, stage), true, peer_abort)) {
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
          for (int k = 0; k < L::kBK / 16; ++k) {
            // 16-deep step k: sub-block k / 4 (16 KiB further per sub-block),
            // step k % 4 in it
            const uint32_t as = a_base + (k >> 2) * 16384, bs = b_base + (k >> 2) * 16384;
            const int kk = k & 3;
            const uint64_t ad = p.a_mn ? make_sw128_desc(as + kk * 2048, 8192, 1024)
                                       : make_sw128_desc(as + kk * 32, 16, 1024);
            const uint64_t bd = p.b_mn ? make_sw128_desc(bs + kk * 2048, 8192, 1024)
                                       : make_sw128_desc(bs + kk * 32, 16, 1024);
            mma_f16_pair(d_tmem, ad, bd, idesc, (kb != kb0) || (k != 0));
          }
          mma_commit_pair_mc(empty0 + 8 * stage, 0x3);  // free the stage in both CTAs
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair_mc(tfull0 + 8 * acc, 0x3);  // accumulator ready in both CTAs
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      trace_mark(p.trace, kTrLastMma);
      trace_value(p.trace, kTrUnits, static_cast<uint64_t>(done));
      if (!ok || *abort_flag) {
        mma_commit_pair(drain);
        wait_bounded(drain, 0, abort_flag, p.timeout_ns, timeout_code(kRoleMma, 0x300), false,
                     peer_abort);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Staged as in the single-CTA kernels: this CTA's 128 rows of the pair
    // tile, C fetched while the tile's MMAs run, 64-column chunks stored by
    // TMA from one staging buffer per warp; the accumulator goes back to the
    // even CTA's MMA thread.
    const uint32_t quad = static_cast<uint32_t>(warp & 3);  // TMEM lanes 32*quad ..
    const int ew = warp - 2;                                // 0..7
    // The tile's bn columns form ceil(bn / 64) chunks of 64 (the last 32
    // wide when bn is an odd multiple of 32); the first warp of a quadrant
    // drains the first half of the chunks, the second the rest.
    const int tile_chunks = (p.bn + 63) / 64;
    const int half_chunks = (tile_chunks + 1) / 2;
    const int chunk0 = (ew >> 2) * half_chunks;
    const int nchunks = min(half_chunks, tile_chunks - chunk0);  // this warp's chunks
    const int col0 = chunk0 * 64;                            // first tile column of this warp
    const int row0 = static_cast<int>(rank * 128 + quad * 32);  // first tile row of this warp
    uint8_t* stg = smem + L::kStagingOffset + ew * kStagingBytes;
    const uint32_t stg_u32 = smem_u32(stg);
    const uint32_t leader_tempty0 = mapa_shared(tempty0, 0);
    uint32_t acc = 0, acc_phase = 0;
    uint4 cnext[8];
    for (int u = pair; u < units; u += num_pairs) {
      int t, kb0, kb1;
      int64_t slot;
      pair_unit(p, u, t, kb0, kb1, slot);
      if (slot >= 0) {
        // K-split unit: this warp's 32 x 128 of the fp32 partial, stored as
        // part of 128-row partial tile 2j + rank of split sp (slot = j *
        // ks_splits + sp; the reduction's view of the split pair tile)
        if (!wait_bounded(tfull0 + 8 * acc, acc_phase, abort_flag, p.timeout_ns,
                          timeout_code(kRoleEpilogue, acc), true, peer_abort))
          break;
        tc_fence_after();
        // (split units always have bn = 256: two whole chunks per warp)
        const uint32_t t_row = tmem_base + ((quad * 32) << 16) + acc * kPairBN + col0;
        const int64_t jj = slot / p.ks_splits, sp = slot - jj * p.ks_splits;
        const int64_t ur = (2 * jj + rank) * p.ks_splits + sp;
        float4* ws4 = reinterpret_cast<float4*>(p.ks_ws);
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
          uint32_t r[64];
          tmem_ld_32x32b_x32(t_row + c * 64, *reinterpret_cast<uint32_t(*)[32]>(r));
          tmem_ld_32x32b_x32(t_row + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
          tmem_wait_ld();
          if (c == nchunks - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(leader_tempty0 + 8 * acc);
          }
          const int gc = col0 / 64 + c;  // chunk of the tile row
#pragma unroll
          for (int g = 0; g < 16; ++g)
            ws4[ks_partial_index(ur, kPairBN, static_cast<int>(quad), gc, g, static_cast<int>(lane))] =
                make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                            __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3]));
        }
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
        continue;
      }
      int tb, tm, tn;
      batch_tile(p, t, tb, tm, tn);
      const __half* cb = p.e.read_c ? p.e.C + tb * p.e.sC : nullptr;
      const int m_base = tm * kPairBM + row0, n_base = tn * p.bn + col0;
      epi_load_c(p, cb, m_base, n_base, lane, cnext);
      if (lane == 0) bulk_wait_group_read0();  // the last store has read the buffer
      __syncwarp();
      epi_stage_c(p, stg, lane, cnext);
      if (nchunks > 1) epi_load_c(p, cb, m_base, n_base + 64, lane, cnext);
      __syncwarp();
      if (!wait_bounded(tfull0 + 8 * acc, acc_phase, abort_flag, p.timeout_ns,
                        timeout_code(kRoleEpilogue, acc), true, peer_abort))
        break;
      tc_fence_after();
      if (ew == 0 && lane == 0 && u == pair) trace_mark(p.trace, kTrFirstAcc);
      if (nchunks <= 0) {
        // no columns for this warp (a tile narrower than the host ever
        // picks): still return the accumulator in this phase
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(leader_tempty0 + 8 * acc);
      }
      const uint32_t t_row = tmem_base + ((quad * 32) << 16) + acc * kPairBN + col0;
#pragma unroll 1
      for (int c = 0; c < nchunks; ++c) {
        if (c > 0) {
          if (lane == 0) bulk_wait_group_read0();
          __syncwarp();
          epi_stage_c(p, stg, lane, cnext);
          if (c + 1 < nchunks) epi_load_c(p, cb, m_base, n_base + 64 * (c + 1), lane, cnext);
          __syncwarp();
        }
        // (the last chunk of a 32-column remainder reads 32 accumulator
        // columns past the tile; they lie inside the 256-column buffer and
        // are not stored)
        uint32_t r[64];
        tmem_ld_32x32b_x32(t_row + c * 64, *reinterpret_cast<uint32_t(*)[32]>(r));
        tmem_ld_32x32b_x32(t_row + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
        tmem_wait_ld();
        if (c == nchunks - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(leader_tempty0 + 8 * acc);
        }
        epi_store_chunk(p, &tmD, stg, stg_u32, lane, tb, m_base, n_base + 64 * c, r,
                        min(64, p.bn - (col0 + 64 * c)));
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
  cluster_sync();  // no CTA leaves while its peer's MMAs or arrivals may touch it
  if (threadIdx.x == 0) trace_exit(p.trace);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kPairTmemCols);
  }
}

}  // namespace gemm_tn_dev
