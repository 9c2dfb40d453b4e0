// gemm_skinny.cuh -- HBM-streaming path for skinny M (M <= 256), sm_103a.
//
// With M this small the work is one pass over B (N x K fp16), so the kernel
// is bound by HBM, not by the tensor cores.  The roles of the operands are
// swapped so that B fills the 128-row side of tcgen05.mma:
//
//     D^T(n,m) = sum_k B(n,k) * A(m,k)      (MMA M = 128 rows of B,
//                                            MMA N = M rounded up to 16)
//
// which is the same TN product read with A and B exchanged ("Reading CuTe's
// make_tiled_mma", section "Fix the matrices and directions first": D is
// symmetric in the roles of A and B up to a transpose).
//
// N/128 output tiles are far fewer than the SMs, so the K loop is split.
// The (tile, K-block) units are laid out tile-major and cut into contiguous
// ranges of equal length, one per CTA (persistent, one CTA per SM).  A range
// covers whole or partial K loops of one or more tiles; each maximal piece
// inside one tile is a segment whose fp32 partial sum (128 x MP) goes to the
// workspace.  A second kernel adds, for every output, the partials of the
// CTAs that touched its tile in increasing CTA order and then C, exactly
// once, and rounds to fp16 -- the rule for K split across workers in the
// same page's section "Thread groups along K, and the loop along K": the
// partial sums must be reduced and the initial C added only once.  The fixed
// order makes the result deterministic.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace gemm_tn_dev {

constexpr int kSkinnyBN = 128;  // rows of B per tile (the MMA's M)
constexpr int kSkinnyBK = 64;
constexpr int kSkinnyThreads = 192;

struct SkinnyArgs {
  int M, N, K;
  int mp;            // M rounded up to 16 (the MMA's N)
  int tiles, k_blocks;
  int64_t units;     // tiles * k_blocks
  int64_t per;       // units per CTA: CTA c owns [c*per, min((c+1)*per, units))
  int max_segs;      // segments one CTA can produce
  int grid;          // CTAs of the split kernel (ceil(units / per))
  float* ws;         // [grid * max_segs][mp/4][128] float4 partials (see skinny_partial)
  uint64_t timeout_ns;
  int test_stall;
  int trace;         // phase trace on (see trace_mark)
};

// 64-deep K sub-blocks per pipeline stage (and per unit of the K split):
// two for MMA widths up to 128 -- 256 contiguous bytes of each B row per
// stage -- and one above, where A's share of a stage would leave too few
// stages.
__host__ __device__ constexpr int skinny_sub(int mp) { return mp <= 128 ? 2 : 1; }

template <int STAGES, int MP>
struct SkinnySmem {
  static constexpr int kSub = skinny_sub(MP);
  static constexpr uint32_t kBSub = kSkinnyBN * kSkinnyBK * 2;  // 16 KiB per sub-block
  static constexpr uint32_t kASub = MP * kSkinnyBK * 2;         // MP rows of 128 B
  static constexpr uint32_t kBBytes = kSub * kBSub;
  static constexpr uint32_t kABytes = kSub * kASub;
  static constexpr uint32_t kStageBytes = kBBytes + kABytes;
  static constexpr uint32_t kBarOffset = STAGES * kStageBytes;
  static constexpr uint32_t kNumBars = 2 * STAGES + 5;
  static constexpr uint32_t kCtlOffset = kBarOffset + kNumBars * 8;
  static constexpr uint32_t kBytes = kCtlOffset + 16;
  static constexpr uint32_t kDynamicBytes = kBytes + 1024;
  // two accumulators of MP fp32 columns, rounded up to a power of two
  static constexpr uint32_t kTmemCols =
      MP <= 16 ? 32 : (MP <= 32 ? 64 : (MP <= 64 ? 128 : (MP <= 128 ? 256 : 512)));
};

// Partial sums of one segment slot: 128 rows (n) x MP columns (m) of fp32,
// stored column-quad-major -- float4 q of row r at (slot * MP/4 + q) * 128 + r
// -- so that 32 consecutive rows' quad is 512 contiguous bytes: the epilogue
// warps store and the reduction reads whole lines.
template <int MP>
__device__ __forceinline__ int64_t skinny_partial(int64_t slot, int q, int row) {
  return (slot * (MP / 4) + q) * kSkinnyBN + row;
}

// Segments of CTA `cta`: consecutive pieces of [begin, end) that stay inside
// one tile.  seg j covers [max(begin, (first_tile + j) * kb), min(end, ...)).
struct SegIter {
  int64_t begin, end;
  int kb;
  __device__ SegIter(int64_t units, int cta, int64_t per, int k_blocks)
      : begin(unit_begin(units, cta, per)), end(unit_begin(units, cta + 1, per)),
        kb(k_blocks) {}
  __device__ int first_tile() const { return static_cast<int>(div_nonneg(begin, kb)); }
  __device__ int count() const {
    if (end <= begin) return 0;
    return static_cast<int>(div_nonneg(end - 1, kb)) - first_tile() + 1;
  }
  __device__ void seg(int j, int& tile, int& kb0, int& kb1) const {
    tile = first_tile() + j;
    const int64_t lo = max(begin, static_cast<int64_t>(tile) * kb);
    const int64_t hi = min(end, static_cast<int64_t>(tile + 1) * kb);
    kb0 = static_cast<int>(lo - static_cast<int64_t>(tile) * kb);
    kb1 = static_cast<int>(hi - static_cast<int64_t>(tile) * kb);
  }
};

template <int STAGES, int MP>
__global__ void __launch_bounds__(kSkinnyThreads, 1)
    gemm_tn_skinny_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB, const SkinnyArgs p) {
  using L = SkinnySmem<STAGES, MP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // stage s: B box at s*kStageBytes (16 KiB, 1024-aligned), A box right after
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kCtlOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kCtlOffset + 4);

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + STAGES);
  const uint32_t tfull0 = smem_u32(bars + 2 * STAGES);
  const uint32_t tempty0 = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t drain = smem_u32(bars + 2 * STAGES + 4);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const SegIter segs(p.units, blockIdx.x, p.per, p.k_blocks);
  // The reduction kernel may be scheduled now; it waits for this grid's
  // completion before it reads anything.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int nseg = segs.count();

  if (threadIdx.x == 0) {
    trace_entry(p.trace);
    trace_value(p.trace, kTrSm, sm_id());
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
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
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Launched as a programmatic dependent: the kernel before this one in the
  // stream (which may write A, B or C, or read the workspace) must be
  // complete before any global memory is touched.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) trace_mark(p.trace, kTrReady);

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();   // A: re-read by every CTA
      const uint64_t stream = l2_policy_evict_first();  // B: read once
      uint32_t stage = 0, phase = 0, issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int j = 0; ok && j < nseg; ++j) {
        int tile, kb0, kb1;
        segs.seg(j, tile, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bounded(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.timeout_ns,
                            timeout_code(kRoleProducer, stage))) {
            ok = false;
            break;
          }
          if (!(p.test_stall && j == 0 && kb == kb0)) {
            const uint32_t fb = full0 + 8 * stage;
            const uint32_t b_dst = smem_u32(smem + stage * L::kStageBytes);
            const uint32_t a_dst = b_dst + L::kBBytes;
            mbar_arrive_expect_tx(fb, L::kStageBytes);
#pragma unroll
            for (int sub = 0; sub < L::kSub; ++sub) {
              // a sub-block past K is zero-filled (and still counted)
              const int k0 = (kb * L::kSub + sub) * kSkinnyBK;
              tma_load_2d_hint(b_dst + sub * L::kBSub, &tmB, fb, k0, tile * kSkinnyBN, stream);
              tma_load_2d_hint(a_dst + sub * L::kASub, &tmA, fb, k0, 0, keep);
            }
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
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
    if (lane == 0) {
      const uint32_t idesc = make_idesc_f16(kSkinnyBN, MP, true, 0, 0);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, first_stage = true;
      for (int j = 0; ok && j < nseg; ++j) {
        int tile, kb0, kb1;
        segs.seg(j, tile, kb0, kb1);
        if (!wait_bounded(tempty0 + 8 * acc, acc_phase ^ 1u, abort_flag, p.timeout_ns,
                          timeout_code(kRoleMma, 0x200 + acc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * MP;
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
          const uint32_t b_base = smem_u32(smem + stage * L::kStageBytes);
          const uint32_t a_base = b_base + L::kBBytes;
#pragma unroll
          for (int k = 0; k < L::kSub * kSkinnyBK / 16; ++k) {
            // MMA A operand = tile of B (128 x 16), MMA B operand = A (MP x 16);
            // 16-deep step k is step k % 4 of sub-block k / 4
            const int sub = k >> 2, kk = k & 3;
            const uint64_t bd = make_sw128_desc(b_base + sub * L::kBSub + kk * 32, 16, 1024);
            const uint64_t ad = make_sw128_desc(a_base + sub * L::kASub + kk * 32, 16, 1024);
            mma_f16(d_tmem, bd, ad, idesc, (kb != kb0) || (k != 0));
          }
          mma_commit(empty0 + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * acc);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      trace_mark(p.trace, kTrLastMma);
      trace_value(p.trace, kTrUnits, static_cast<uint64_t>(nseg));
      if (!ok || *abort_flag) {
        mma_commit(drain);
        wait_bounded(drain, 0, abort_flag, p.timeout_ns, timeout_code(kRoleMma, 0x300), false);
      }
    }
  } else {
    const uint32_t quad = static_cast<uint32_t>(warp & 3);
    const int row = static_cast<int>(quad * 32 + lane);  // row of the B tile = n offset
    uint32_t acc = 0, acc_phase = 0;
    for (int j = 0; j < nseg; ++j) {
      if (!wait_bounded(tfull0 + 8 * acc, acc_phase, abort_flag, p.timeout_ns,
                        timeout_code(kRoleEpilogue, acc)))
        break;
      tc_fence_after();
      if (warp == 2 && lane == 0 && j == 0) trace_mark(p.trace, kTrFirstAcc);
      const int64_t slot = static_cast<int64_t>(blockIdx.x) * p.max_segs + j;
      float4* dst = reinterpret_cast<float4*>(p.ws) + skinny_partial<MP>(slot, 0, row);
      const uint32_t t_row = tmem_base + ((quad * 32) << 16) + acc * MP;
#pragma unroll
      for (int c = 0; c < MP / 16; ++c) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(t_row + c * 16, r);
        tmem_wait_ld();
#pragma unroll
        for (int v = 0; v < 4; ++v)
          dst[(4 * c + v) * kSkinnyBN] =
              make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                          __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (warp == 2 && lane == 0) trace_mark(p.trace, kTrLastChunk);
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) trace_exit(p.trace);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::kTmemCols);
  }
}

// D(m,n) = fp16( alpha * (sum over the CTAs that touched tile n/128, in CTA
// order, of their partial (n%128, m))  +  beta * C(m,n) ) -- see EpiArgs;
// with alpha = beta = 1 the sum plus C.  Block (tile, y) has 512 threads;
// thread (g, r) owns column n = 128*tile + r and rows 4g..4g+3 with
// g = 4y + threadIdx.x/128, reads one 16-byte vector of partials per
// contributing CTA (a warp reads 512 contiguous bytes), and adds C once.  The kernel is
// launched as a programmatic dependent of the split-K kernel: its blocks
// become resident while the split-K kernel runs and wait for its completion
// (and the visibility of its partial sums) in griddepcontrol.wait.
constexpr int kReduceThreads = 4 * kSkinnyBN;  // four 4-row groups per block

template <int MP>
__global__ void __launch_bounds__(kReduceThreads)
    gemm_tn_splitk_reduce_kernel(const SkinnyArgs p, const EpiArgs e) {
  // The next call's kernels may become resident now (they wait for this
  // grid's completion before touching memory).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int tile = static_cast<int>(blockIdx.x);
  const int r = static_cast<int>(threadIdx.x) % kSkinnyBN;
  const int g = 4 * static_cast<int>(blockIdx.y) + static_cast<int>(threadIdx.x) / kSkinnyBN;
  const int n = tile * kSkinnyBN + r;
  if (n >= p.N || 4 * g >= p.M) return;
  const int64_t u0 = static_cast<int64_t>(tile) * p.k_blocks;
  const int c_first = cta_of_unit(u0, p.per);
  const int c_last = cta_of_unit(u0 + p.k_blocks - 1, p.per);
  const float4* ws = reinterpret_cast<const float4*>(p.ws);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  // every CTA from c_first to c_last has a non-empty range inside this tile
  for (int c = c_first; c <= c_last; ++c) {
    const int64_t b = static_cast<int64_t>(c) * p.per;
    const int j = tile - static_cast<int>(div_nonneg(b, p.k_blocks));
    const int64_t slot = static_cast<int64_t>(c) * p.max_segs + j;
    const float4 x = ws[skinny_partial<MP>(slot, g, r)];
    acc.x += x.x;
    acc.y += x.y;
    acc.z += x.z;
    acc.w += x.w;
  }
  const float v[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int m = 4 * g + j;
    if (m < p.M) {
      const __half c = e.read_c ? e.C[static_cast<int64_t>(m) * e.ldC + n] : __ushort_as_half(0);
      e.D[static_cast<int64_t>(m) * e.ldD + n] = epi_one(e, false, __float_as_uint(v[j]), c);
    }
  }
}

}  // namespace gemm_tn_dev
