// gemm_skinny_cluster.cuh -- HBM-streaming path for skinny M with the K
// split reduced inside a thread-block cluster (sm_103a).
//
// The same swapped-operand product as gemm_skinny.cuh ("Reading CuTe's
// make_tiled_mma", section "Fix the matrices and directions first"):
//
//     D^T(n,m) = sum_k B(n,k) * A(m,k)      (MMA M = 128 rows of B,
//                                            MMA N = M rounded up to 16)
//
// but each 128-row tile of B gets one cluster of `cs` CTAs (cs = 1..8), and
// CTA r of the cluster runs the K blocks [r * kb / cs, (r + 1) * kb / cs).
// After its MMAs every CTA parks its fp32 partial sum (128 x MP) in its own
// shared memory (the idle operand ring), the cluster synchronises, and CTA r
// finishes rows [r * 128 / cs, (r + 1) * 128 / cs) of the tile: it reads the
// cs partials of each output from the cluster's shared memory in rank order
// (distributed shared memory), adds them, then applies the epilogue with C
// exactly once -- the rule of the same page's section "Thread groups along
// K, and the loop along K" for a K split: reduce the partial sums, add the
// initial C once.  The fixed rank order makes the result deterministic.
// There is no workspace and no second kernel.
//
// Operands arrive by TMA into the 128B-swizzled layout of gemm_skinny.cuh,
// in deeper stages (cluster_sub).  With `ko` (K a multiple of 64) each
// operand of a stage is one K-chunk box {64, rows, sub} (a GB300 SM takes
// fewer, larger boxes in faster); otherwise one 2-D box per 64-deep
// sub-block.
//
// Every mbarrier wait is bounded.  The two cluster barriers are reached by
// every thread on every path (a role that gives up leaves its loop and
// falls through), so a CTA that timed out cannot leave its peers waiting.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"
#include "gemm_skinny.cuh"

namespace gemm_tn_dev {

constexpr int kClusterMaxCs = 8;  // portable cluster size limit

// K depth of a stage of the cluster kernel, in 64-deep sub-blocks: four
// (256 of K) up to MMA width 16, three up to 64, two up to 128, one above --
// deeper than the split kernel's, since a GB300 SM streams larger TMA boxes
// faster and this kernel may run on fewer SMs than there are.
__host__ __device__ constexpr int cluster_sub(int mp) {
  return mp <= 16 ? 4 : (mp <= 64 ? 3 : (mp <= 128 ? 2 : 1));
}
// Ring depth: 3 stages (4 for MMA width 96, 5 for 192, 4 for 256).
__host__ __device__ constexpr int cluster_stages(int mp) {
  return mp <= 64 ? 3 : (mp <= 96 ? 4 : (mp <= 128 ? 3 : (mp <= 192 ? 5 : 4)));
}

// Shared memory of the cluster kernel: STAGES x (B sub-blocks, then A
// sub-blocks), each 64-deep sub-block 1024-aligned, then the barriers.
template <int STAGES, int MP>
struct ClusterSmem {
  static constexpr int kSub = cluster_sub(MP);
  static constexpr uint32_t kBSub = kSkinnyBN * kSkinnyBK * 2;  // 16 KiB
  static constexpr uint32_t kASub = MP * kSkinnyBK * 2;
  static constexpr uint32_t kBBytes = kSub * kBSub;
  static constexpr uint32_t kABytes = kSub * kASub;
  static constexpr uint32_t kStageBytes = kBBytes + kABytes;
  static constexpr uint32_t kBarOffset = STAGES * kStageBytes;
  static constexpr uint32_t kNumBars = 2 * STAGES + 2;
  static constexpr uint32_t kCtlOffset = kBarOffset + kNumBars * 8;
  static constexpr uint32_t kBytes = kCtlOffset + 16;
  static constexpr uint32_t kDynamicBytes = kBytes + 1024;
  static_assert(kDynamicBytes <= 232448, "over the 227 KiB of shared memory per CTA");
  static_assert(kASub % 1024 == 0 || MP % 8 == 0, "A sub-blocks keep the swizzle atoms aligned");
};

struct SkinnyClusterArgs {
  int M, N, K;
  int tiles;         // ceil(N / 128): one cluster per tile
  int cs;            // CTAs per cluster (K splits per tile): 1, 2, 4 or 8
  int k_blocks;      // K blocks of 64 * cluster_sub(MP)
  int ko;            // operands through K-chunk maps {64, rows, K / 64}
  uint64_t timeout_ns;
  int test_stall;
  int trace;
};

// Load of one fp32 word from shared memory of CTA `rank` of the cluster, at
// the offset of the local shared address `addr`.
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr, uint32_t rank) {
  float v;
  const uint32_t a = mapa_shared(addr, rank);
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

// Cluster-wide barrier with release / acquire semantics (all threads of all
// CTAs of the cluster).
__device__ __forceinline__ void cluster_barrier() {
  __syncwarp();
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// CTA `rank` of a cluster of CS finishes rows [r0, r1) of tile `tile`: per
// output (m, n) the CS partials P_q[m][row] in rank order q = 0..CS-1, then
// D = alpha * sum + beta * C (see EpiArgs).  Each thread keeps kOuts outputs
// in flight (their C values and partials loaded before any is used);
// consecutive threads take consecutive rows, so C / D accesses and the
// partial reads are contiguous.
template <int CS>
__device__ __forceinline__ void skinny_cluster_reduce(const SkinnyClusterArgs& p, const EpiArgs& e,
                                                      int tile, uint32_t rank, uint32_t part_u32) {
  constexpr int kOuts = 8;
  const int r0 = static_cast<int>(rank) * kSkinnyBN / CS;
  const int nrows = kSkinnyBN / CS;
  const int total = nrows * p.M;
  for (int base = static_cast<int>(threadIdx.x); base < total; base += kSkinnyThreads * kOuts) {
    float part_v[kOuts][CS];
    __half cv[kOuts];
    int64_t d_off[kOuts];
#pragma unroll
    for (int j = 0; j < kOuts; ++j) {
      const int idx = base + j * kSkinnyThreads;
      const int m = idx / nrows, row = r0 + (idx - m * nrows);
      const int n = tile * kSkinnyBN + row;
      const bool valid = idx < total && n < p.N;
      d_off[j] = valid ? static_cast<int64_t>(m) * e.ldD + n : -1;
      cv[j] = (valid && e.read_c) ? e.C[static_cast<int64_t>(m) * e.ldC + n] : __ushort_as_half(0);
      const uint32_t addr = part_u32 + 4u * static_cast<uint32_t>(m * kSkinnyBN + row);
#pragma unroll
      for (int q = 0; q < CS; ++q)
        part_v[j][q] = valid ? ld_dsmem_f32(addr, static_cast<uint32_t>(q)) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kOuts; ++j) {
      if (d_off[j] < 0) continue;
      float sum = 0.f;
#pragma unroll
      for (int q = 0; q < CS; ++q) sum += part_v[j][q];
      e.D[d_off[j]] = epi_one(e, false, __float_as_uint(sum), cv[j]);
    }
  }
}

template <int STAGES, int MP>
__global__ void __launch_bounds__(kSkinnyThreads, 1)
    gemm_tn_skinny_cluster_kernel(const __grid_constant__ CUtensorMap tmA,
                                  const __grid_constant__ CUtensorMap tmB,
                                  const SkinnyClusterArgs p, const EpiArgs e) {
  using L = ClusterSmem<STAGES, MP>;
  static_assert(kSkinnyBN * MP * 4 <= STAGES * L::kStageBytes,
                "the partial sums are parked in the operand ring");
  constexpr uint32_t kTmemCols = MP <= 32 ? 32 : (MP <= 64 ? 64 : (MP <= 128 ? 128 : 256));
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kCtlOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kCtlOffset + 4);
  // partial sum P[m][r] (m < MP, r < 128), fp32, over the ring once idle
  float* part = reinterpret_cast<float*>(smem);

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + STAGES);
  const uint32_t tfull = smem_u32(bars + 2 * STAGES);
  const uint32_t drain = smem_u32(bars + 2 * STAGES + 1);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const int tile = static_cast<int>(blockIdx.x) / p.cs;
  const int kb0 = static_cast<int>(static_cast<int64_t>(rank) * p.k_blocks / p.cs);
  const int kb1 = static_cast<int>(static_cast<int64_t>(rank + 1) * p.k_blocks / p.cs);
  // The next kernel in the stream may become resident now; it waits for
  // this grid's completion before it touches memory.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    trace_entry(p.trace);
    trace_value(p.trace, kTrSm, sm_id());
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The kernel before this one in the stream (which may write A, B or C)
  // must be complete before any global memory is touched.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) trace_mark(p.trace, kTrReady);

  bool acc_ok = false;  // the accumulator holds this CTA's partial sum
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();     // A: read by every cluster
      const uint64_t stream = l2_policy_evict_first();  // B: read once
      uint32_t stage = 0, phase = 0, issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int kb = kb0; ok && kb < kb1; ++kb) {
        if (!wait_bounded(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.timeout_ns,
                          timeout_code(kRoleProducer, stage))) {
          ok = false;
          break;
        }
        if (!(p.test_stall && kb == kb0)) {
          const uint32_t fb = full0 + 8 * stage;
          const uint32_t b_dst = smem_u32(smem + stage * L::kStageBytes);
          const uint32_t a_dst = b_dst + L::kBBytes;
          mbar_arrive_expect_tx(fb, L::kStageBytes);
          if (p.ko) {
            // K chunks sub * kb .. + sub - 1 (past K: zero-filled)
            tma_load_4d_hint(b_dst, &tmB, fb, 0, tile * kSkinnyBN, kb * L::kSub, 0, stream);
            tma_load_4d_hint(a_dst, &tmA, fb, 0, 0, kb * L::kSub, 0, keep);
          } else {
#pragma unroll
            for (int sub = 0; sub < L::kSub; ++sub) {
              const int k0 = (kb * L::kSub + sub) * kSkinnyBK;
              tma_load_2d_hint(b_dst + sub * L::kBSub, &tmB, fb, k0, tile * kSkinnyBN, stream);
              tma_load_2d_hint(a_dst + sub * L::kASub, &tmA, fb, k0, 0, keep);
            }
          }
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok || *abort_flag) {
        for (int s = 0; s < STAGES; ++s)
          if (issued_mask >> s & 1u)
            wait_bounded(full0 + 8 * s, issued_parity >> s & 1u, abort_flag, p.timeout_ns,
                         timeout_code(kRoleProducer, 0x100 + s), false);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc_f16(kSkinnyBN, MP, true, 0, 0);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_bounded(full0 + 8 * stage, phase, abort_flag, p.timeout_ns,
                          timeout_code(kRoleMma, stage))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (kb == kb0) trace_mark(p.trace, kTrFirstStage);
        const uint32_t b_base = smem_u32(smem + stage * L::kStageBytes);
        const uint32_t a_base = b_base + L::kBBytes;
#pragma unroll
        for (int k = 0; k < L::kSub * kSkinnyBK / 16; ++k) {
          // MMA A operand = tile of B (128 x 16), MMA B operand = A (MP x 16)
          const int sub = k >> 2, kk = k & 3;
          const uint64_t bd = make_sw128_desc(b_base + sub * L::kBSub + kk * 32, 16, 1024);
          const uint64_t ad = make_sw128_desc(a_base + sub * L::kASub + kk * 32, 16, 1024);
          mma_f16(tmem_base, bd, ad, idesc, (kb != kb0) || (k != 0));
        }
        mma_commit(empty0 + 8 * stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // accumulator complete (or, after a failure, every issued MMA done)
      mma_commit(ok ? tfull : drain);
      if (!ok) wait_bounded(drain, 0, abort_flag, p.timeout_ns, timeout_code(kRoleMma, 0x300), false);
      trace_mark(p.trace, kTrLastMma);
      trace_value(p.trace, kTrUnits, static_cast<uint64_t>(kb1 - kb0));
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Park this CTA's partial sum: lane = row of the B tile, 16 columns
    // (values of m) per TMEM load, stored as P[m][row] (consecutive lanes,
    // consecutive words).  An empty K range (never chosen by the host)
    // parks zeros.
    const uint32_t quad = static_cast<uint32_t>(warp & 3);
    const int row = static_cast<int>(quad * 32 + lane);
    if (kb1 > kb0) {
      if (wait_bounded(tfull, 0, abort_flag, p.timeout_ns, timeout_code(kRoleEpilogue, 0))) {
        tc_fence_after();
        if (warp == 2 && lane == 0) trace_mark(p.trace, kTrFirstAcc);
        acc_ok = true;
        const uint32_t t_row = tmem_base + ((quad * 32) << 16);
#pragma unroll
        for (int c = 0; c < MP / 16; ++c) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(t_row + c * 16, r);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) part[(c * 16 + j) * kSkinnyBN + row] = __uint_as_float(r[j]);
        }
      }
    } else {
      acc_ok = true;
      for (int m = 0; m < MP; ++m) part[m * kSkinnyBN + row] = 0.f;
    }
  }

  // Every CTA's partial parked (or its failure recorded) before any is read.
  tc_fence_before();
  __syncthreads();
  cluster_barrier();

  // ---------------------------------------------------------------- reduce
  switch (p.cs) {
    case 1: skinny_cluster_reduce<1>(p, e, tile, rank, smem_u32(part)); break;
    case 2: skinny_cluster_reduce<2>(p, e, tile, rank, smem_u32(part)); break;
    case 4: skinny_cluster_reduce<4>(p, e, tile, rank, smem_u32(part)); break;
    default: skinny_cluster_reduce<8>(p, e, tile, rank, smem_u32(part)); break;
  }
  if (threadIdx.x == 64 && acc_ok) trace_mark(p.trace, kTrLastChunk);

  // No CTA leaves (or frees its shared memory) while a peer may still read it.
  __syncthreads();
  cluster_barrier();
  if (threadIdx.x == 0) trace_exit(p.trace);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace gemm_tn_dev
