// gemm_strided.cuh -- the TN GEMM for operand views TMA cannot describe.
//
// The layout page (sections 1-2) lets an operand be any shape:stride view;
// the tile kernels need one stride-1 mode, 16-byte aligned rows and 16-byte
// aligned leading dimensions for TMA.  This kernel takes arbitrary element
// strides for A (M,K), B (N,K) and C/D (M,N) and keeps everything after the
// copy the same:
//
//   warps 0-11  copy producer: each thread gathers 16-byte K-chunks (8 fp16
//               along K) of A and B rows through the strides, six chunks in
//               flight at a time -- a contiguous chunk from the one or two
//               aligned 16-byte words under it (shift_window), else eight
//               2-byte loads -- and writes them to the 128B-swizzled K-major
//               layout the TMA unit would produce (row r, chunk j at byte
//               r*128 + 16*(j ^ (r%8))), zero outside the matrix; then
//               fence.proxy.async and one arrival per thread on `full`.
//   warp 12     TMEM allocation and the single MMA-issuing thread
//               (tcgen05.mma M=128, N=256, K=16, always K-major descriptors).
//   warps 13-16 epilogue: tcgen05.ld, + C, round, D.  A row-major C/D view
//               goes through a per-warp 32 x 32 transpose in shared memory,
//               so that C is read and D written a row segment per
//               instruction; any other view element by element with one row
//               per lane (coalesced when the M mode has stride 1).
//
// 128 x 256 tiles, 4 stages of 48 KiB, two TMEM accumulators, persistent
// grid, bounded waits; no asynchronous copies, so an abort only has to drain
// the MMAs.
//
// Row-class variant (kTma, both operands with a stride-1 K mode): the rows
// of a view with any leading dimension ld fall into eight classes r % 8,
// and the rows of one class are 16 * ld bytes apart -- a stride TMA
// accepts.  One tensor map per class and operand, on the class's first row
// rounded down to 16 bytes (the row then starts delta = 0..7 elements into
// the map's rows), brings a K block in as one 128B-swizzled box per class
// (32 rows of A or of B) straight into the stage the MMA reads.  Warps:
//   0-15   one stage row per thread, shifted left in place by its delta,
//          the last delta elements taken from the same row of the next K
//          block's box (after a tile's last K block, read from the row);
//   16     TMEM allocation and the MMA thread: 256 x 256 tiles as two
//          M = 128 MMAs per step into the two halves of the tensor memory;
//   17-20  epilogue, as above, over both halves;
//   21     lanes 0-15 issue the sixteen boxes of each stage as soon as the
//          MMA has released it.
// Three stages of 64 KiB.  A stage holds the tile's rows in class order
// (stage row s of A is tile row s / 32 + 8 (s % 32), likewise for B's tile
// columns); the MMA does not mind, and the epilogue reads the accumulator
// back in tile order.  Rows past M / N and K past the end arrive as zeros
// from the tensor maps' bounds.  The TMA loads of the class boxes set the
// route's pace: with nothing to shift it is only ~20 % faster.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"
#include "shift.cuh"

namespace gemm_tn_dev {

constexpr int kStrBM = 128;
constexpr int kStrBN = 256;
constexpr int kStrBK = 64;
constexpr int kStrStages = 4;
// Twelve producer warps: with the MMA and four epilogue warps, 17 warps put
// at most five on an SM sub-partition, which leaves 96 registers a thread
// (sixteen producer warps would cap it at 80 and spill in the shift pass).
constexpr int kStrProducers = 384;
constexpr int kStrThreads = 544;    // 12 producer warps, MMA warp, 4 epilogue warps
// The row-class variant has sixteen producer warps (one stage row each)
// and a warp that issues the boxes: 22 warps, six on some SM
// sub-partitions, so at most 80 registers a thread (its launch bounds are
// declared for 768 threads to make the compiler keep to that).
template <bool kTma>
__host__ __device__ constexpr int str_producers() { return kTma ? 512 : kStrProducers; }
template <bool kTma>
__host__ __device__ constexpr int str_threads() { return str_producers<kTma>() + (kTma ? 6 : 5) * 32; }
template <bool kTma>
__host__ __device__ constexpr int str_bound_threads() { return kTma ? 768 : kStrThreads; }

struct StridedArgs {
  int M, N, K;
  // row-class variant: byte offset of a row of class c in its map row, in
  // bits 4c..4c+3 (a register-held word: indexing an array of the kernel's
  // parameters by the class would read it through memory on every chunk)
  uint32_t a_shifts, b_shifts;
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

// Tensor maps of the row-class variant: class c of A (rows c, c + 8, ...)
// and of B.
struct StridedMaps {
  CUtensorMap a[8];
  CUtensorMap b[8];
};

// Tile rows: the row-class variant takes 256 x 256 tiles (two M = 128 MMAs
// per step into the two halves of the tensor memory), so that each of its
// sixteen boxes per K block feeds twice the MMA work.
template <bool kTma>
__host__ __device__ constexpr int str_bm() { return kTma ? 2 * kStrBM : kStrBM; }

template <bool kTma>
struct StridedSmem {
  // swizzled stages the MMA reads (the row-class variant's boxes land in
  // them and are shifted in place)
  static constexpr int kStages = kTma ? 3 : kStrStages;
  static constexpr int kAccs = kTma ? 1 : 2;  // accumulator sets (512 TMEM columns in all)
  static constexpr uint32_t kABytes = str_bm<kTma>() * kStrBK * 2;  // 32 / 16 KiB
  static constexpr uint32_t kBBytes = kStrBN * kStrBK * 2;          // 32 KiB
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  // per epilogue warp a 32 x 33 word transpose buffer
  static constexpr uint32_t kXposeOffset = kStages * kStageBytes;
  static constexpr uint32_t kXposeBytes = 32 * 33 * 4;
  static constexpr uint32_t kBarOffset = kXposeOffset + 4 * kXposeBytes;
  // full and empty per stage, two tfull, two tempty, drain; row-class
  // variant: `landed` per stage (the stage's boxes are in)
  static constexpr uint32_t kNumBars = 2 * kStages + 5 + (kTma ? kStages : 0);
  static constexpr uint32_t kCtlOffset = kBarOffset + kNumBars * 8;
  static constexpr uint32_t kBytes = kCtlOffset + 16;
  static constexpr uint32_t kDynamicBytes = kBytes + 1024;
};

// Eight consecutive-k elements X(row, k0..k0+7) of a (rows, K) view with
// strides (s_row, s_k); zeros outside the matrix.
__device__ __forceinline__ uint4 gather_chunk(const __half* X, int64_t s_row, int64_t s_k,
                                              int rows, int K, int row, int k0) {
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (row >= rows || k0 >= K) return v;
  const __half* src = X + static_cast<int64_t>(row) * s_row + static_cast<int64_t>(k0) * s_k;
  if (s_k == 1 && k0 + 8 <= K) {
    // the one or two aligned 16-byte words holding the chunk's bytes
    const uintptr_t a = reinterpret_cast<uintptr_t>(src);
    const uintptr_t w = a & ~static_cast<uintptr_t>(15);
    const int sh = static_cast<int>(a & 15u);
    const uint4 lo = __ldg(reinterpret_cast<const uint4*>(w));
    if (sh == 0) return lo;
    return shift_window(lo, __ldg(reinterpret_cast<const uint4*>(w + 16)), sh);
  }
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

// Chunk q of one operand's stage (rows x 64 of K): row and 16-byte K-chunk.
// When K is the contiguous mode consecutive q walk along K (eight chunks per
// row), else along the rows, so that neighbouring threads read neighbouring
// elements.
__device__ __forceinline__ void chunk_coords(bool k_fast, int rows, int q, int& r, int& j) {
  r = k_fast ? q >> 3 : q % rows;
  j = k_fast ? q & 7 : q / rows;
}

// Fill one stage: A's kStrBM x 64 and B's kStrBN x 64 of K in the K-major
// 128B-swizzled layout.  The stage's chunks (A's first, then B's) are dealt
// round-robin to the producer threads and gathered kBatch at a time, all
// their loads issued before the first store, so that enough bytes are in
// flight per SM.
__device__ __forceinline__ void fill_stage(uint8_t* dst_a, uint8_t* dst_b, const StridedArgs& p,
                                           int m0, int n0, int k0, int tid) {
  const bool a_kfast = (p.sAk == 1) || (p.sAm != 1 && p.sAk <= p.sAm);
  const bool b_kfast = (p.sBk == 1) || (p.sBn != 1 && p.sBk <= p.sBn);
  constexpr int kA = kStrBM * 8, kTotal = (kStrBM + kStrBN) * 8;
  constexpr int kBatch = 6;
  for (int q0 = tid; q0 < kTotal; q0 += kBatch * kStrProducers) {
    uint4 v[kBatch];
    uint8_t* dst[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int q = q0 + b * kStrProducers;
      dst[b] = nullptr;
      v[b] = make_uint4(0u, 0u, 0u, 0u);
      if (q < kTotal) {
        int r, j;
        if (q < kA) {
          chunk_coords(a_kfast, kStrBM, q, r, j);
          v[b] = gather_chunk(p.A, p.sAm, p.sAk, p.M, p.K, m0 + r, k0 + 8 * j);
          dst[b] = dst_a + r * 128 + 16 * (j ^ (r & 7));
        } else {
          chunk_coords(b_kfast, kStrBN, q - kA, r, j);
          v[b] = gather_chunk(p.B, p.sBn, p.sBk, p.N, p.K, n0 + r, k0 + 8 * j);
          dst[b] = dst_b + r * 128 + 16 * (j ^ (r & 7));
        }
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b)
      if (dst[b]) *reinterpret_cast<uint4*>(dst[b]) = v[b];
  }
}

// wait_bounded for a wait that normally lasts a whole tile's main loop: the
// waiting warp sleeps between probes instead of spinning, so that it does not
// take issue slots from the producer warps that share its SM sub-partitions.
__device__ __forceinline__ bool wait_bounded_sleeping(uint32_t bar, uint32_t parity,
                                                      volatile uint32_t* abort_flag,
                                                      uint64_t limit_ns, uint32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    __nanosleep(500);
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicCAS(&g_error_word, 0u, code);
      *abort_flag = 1u;
      return false;
    }
  }
}

// Row-class variant.  A class box (32 rows of A or B, 64 elements of K)
// lands as consecutive rows of a stage, so stage row s of the A part holds
// tile row (s / 32) + 8 (s % 32), and stage row s of the B part tile column
// (s / 32) + 8 (s % 32).  The MMA multiplies the rows in that order; the
// epilogue reads accumulator lanes and columns back as those tile rows and
// columns.
__device__ __forceinline__ int class_row(int s) { return (s >> 5) + 8 * (s & 31); }

// A box row starts `sh` bytes (even, 0..14) before the row's K block: the
// row, 128B-swizzled at stage row s (16-byte chunk j at 16 (j ^ (s % 8))),
// is shifted left in place by sh bytes, its last sh bytes taken from `next`
// (the first 16 bytes of the same row of the following K block).
__device__ __forceinline__ void shift_row_in_place(uint8_t* row, uint32_t sw, int sh,
                                                   const uint4& next) {
  uint4 w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = *reinterpret_cast<const uint4*>(row + 16 * (j ^ sw));
#pragma unroll
  for (int j = 0; j < 8; ++j)
    *reinterpret_cast<uint4*>(row + 16 * (j ^ sw)) = shift_window(w[j], j < 7 ? w[j + 1] : next, sh);
}

// The 16 bytes after the last K block of a row that starts sh bytes into its
// box: elements k0 - sh/2 .. k0 - 1 of the row (k0 = the blocks' end), those
// below K, in bytes [0, sh); zeros elsewhere.  Plain 2-byte loads inside
// the row (the next box would start past the blocks' end).
__device__ __forceinline__ uint4 row_tail(const __half* row, int K, int k0, int sh) {
  uint32_t v[4] = {0u, 0u, 0u, 0u};
  const int d = sh >> 1;
#pragma unroll
  for (int e = 0; e < 7; ++e) {
    const int k = k0 - d + e;
    if (e < d && k < K) {
      const uint32_t h = __ldg(reinterpret_cast<const unsigned short*>(row + k));
      v[e >> 1] |= h << (16 * (e & 1));
    }
  }
  return make_uint4(v[0], v[1], v[2], v[3]);
}

// tcgen05.ld of 4 consecutive accumulator columns for the warp's 32 lanes.
__device__ __forceinline__ void tmem_ld_32x32b_x4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
}

template <bool kTma>
__global__ void __launch_bounds__(str_bound_threads<kTma>(), 1)
    gemm_tn_strided_kernel(const __grid_constant__ StridedMaps maps, const StridedArgs p) {
  using L = StridedSmem<kTma>;
  constexpr int kStages = L::kStages;
  constexpr int kProducers = str_producers<kTma>();  // producer threads
  constexpr int kMmaWarp = kProducers / 32;          // then 4 epilogue warps
  constexpr int kIssueWarp = kMmaWarp + 5;           // row-class variant only
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
  const uint32_t land0 = smem_u32(bars + 2 * kStages + 5);  // row-class variant only

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, kProducers);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 4);
    }
    mbar_init(drain, 1);
    if (kTma)
      for (int s = 0; s < kStages; ++s) mbar_init(land0 + 8 * s, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (kTma && threadIdx.x == 32) {
    for (int c = 0; c < 8; ++c) {
      tma_prefetch_desc(&maps.a[c]);
      tma_prefetch_desc(&maps.b[c]);
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 2 * kStrBN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp < kMmaWarp && kTma) {
    // ------------------------------------------------ row-class TMA producer
    // A stage has 2 * 256 rows (A's, then B's); thread tid owns row tid (and
    // tid + kProducers, were there fewer threads than rows) in every stage
    // and shifts it in place once the row's box and the following K block's
    // box have landed.
    // No other thread touches those rows, so the next block's first 16 bytes
    // are read before this thread shifts that block.
    constexpr int kBM = str_bm<kTma>();
    const int tid = static_cast<int>(threadIdx.x);
    const int n_own = tid + kProducers < kBM + kStrBN ? 2 : 1;
    const int my_tiles = p.num_tiles > static_cast<int>(blockIdx.x)
                             ? (p.num_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                             : 0;
    const int units = my_tiles * p.k_blocks;  // (tile, K block) pairs of this CTA, in order
    bool ok = true;
    for (int u = 0; ok && u < units; ++u) {
      const int slot = u % kStages;
      const int kb = u % p.k_blocks;
      const bool last = kb == p.k_blocks - 1;
      const int nslot = (u + 1) % kStages;
      if (!wait_bounded(land0 + 8 * slot, static_cast<uint32_t>(u / kStages) & 1u, abort_flag,
                        p.timeout_ns, timeout_code(kRoleProducer, 0x500 + slot)) ||
          (!last && !wait_bounded(land0 + 8 * nslot, static_cast<uint32_t>((u + 1) / kStages) & 1u,
                                  abort_flag, p.timeout_ns,
                                  timeout_code(kRoleProducer, 0x500 + nslot)))) {
        ok = false;
        break;
      }
#pragma unroll
      for (int o = 0; o < 2; ++o) {
        if (o >= n_own) continue;
        const int row = tid + o * kProducers;  // of the stage's A rows, then B rows
        const bool is_b = row >= kBM;
        const int s = is_b ? row - kBM : row;
        const int sh = static_cast<int>(((is_b ? p.b_shifts : p.a_shifts) >> (4 * (s >> 5))) & 15u);
        if (sh == 0) continue;
        uint8_t* const at = (is_b ? sB : sA) + s * 128;  // the row in stage 0
        const uint32_t step = is_b ? L::kBBytes : L::kABytes;
        const uint32_t sw = static_cast<uint32_t>(s & 7);
        uint4 next;
        if (!last) {
          next = *reinterpret_cast<const uint4*>(at + nslot * step + 16 * sw);
        } else {
          const int t = static_cast<int>(blockIdx.x) + (u / p.k_blocks) * static_cast<int>(gridDim.x);
          int tm, tn;
          tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
          const int grow = (is_b ? tn * kStrBN : tm * kBM) + class_row(s);
          next = grow < (is_b ? p.N : p.M)
                     ? row_tail((is_b ? p.B : p.A) + static_cast<int64_t>(grow) * (is_b ? p.sBn : p.sAm),
                                p.K, p.k_blocks * kStrBK, sh)
                     : make_uint4(0u, 0u, 0u, 0u);
        }
        shift_row_in_place(at + slot * step, sw, sh, next);
      }
      fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
      mbar_arrive(full0 + 8 * slot);
    }
    (void)ok;
  } else if (kTma && warp == kIssueWarp) {
    // ------------------------------------------------ row-class box issue
    // Lanes 0-15 load unit v into stage v % kStages as soon as the MMA has
    // released the stage: lane i issues box i (A classes 0-7, then B
    // classes 0-7, 32 rows each) after lane 0 has armed `landed` with the
    // stage's bytes (a copy that lands before the arming drives the byte
    // count below zero; the phase still needs the arrival).  With a warp of
    // their own the loads run two stages ahead of the shift; issued by the
    // shifting threads after their own rows, every shift waited a whole
    // round trip for the next block's boxes.
    if (lane < 16) {
      constexpr int kBM = str_bm<kTma>();
      const int i = static_cast<int>(lane);
      const int my_tiles = p.num_tiles > static_cast<int>(blockIdx.x)
                               ? (p.num_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                               : 0;
      const int units = my_tiles * p.k_blocks;
      uint32_t issued_mask = 0, issued_parity = 0;  // stages with copies in flight
      bool ok = true;
      for (int v = 0; ok && v < units; ++v) {
        const int slot = v % kStages;
        const uint32_t use = static_cast<uint32_t>(v / kStages);
        if (!wait_bounded(empty0 + 8 * slot, (use & 1u) ^ 1u, abort_flag, p.timeout_ns,
                          timeout_code(kRoleProducer, 0x400 + slot))) {
          ok = false;
          break;
        }
        const int t = static_cast<int>(blockIdx.x) + (v / p.k_blocks) * static_cast<int>(gridDim.x);
        const int kb = v % p.k_blocks;
        int tm, tn;
        tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
        const uint32_t lb = land0 + 8 * slot;
        if (i == 0) mbar_arrive_expect_tx(lb, L::kStageBytes);
        const int c = i & 7;
        if (i < 8)
          tma_load_2d(smem_u32(sA + slot * L::kABytes + c * (kBM / 8) * 128), &maps.a[c], lb,
                      kb * kStrBK, tm * (kBM / 8));
        else
          tma_load_2d(smem_u32(sB + slot * L::kBBytes + c * (kStrBN / 8) * 128), &maps.b[c], lb,
                      kb * kStrBK, tn * (kStrBN / 8));
        issued_mask |= 1u << slot;
        issued_parity = (issued_parity & ~(1u << slot)) | ((use & 1u) << slot);
      }
      if (!ok || *abort_flag) {
        // every copy this lane issued lands before the CTA can leave
        for (int q = 0; q < kStages; ++q)
          if (issued_mask >> q & 1u)
            wait_bounded(land0 + 8 * q, issued_parity >> q & 1u, abort_flag, p.timeout_ns,
                         timeout_code(kRoleProducer, 0x600 + q), false);
      }
    }
  } else if (warp < kMmaWarp) {
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
        fill_stage(sA + stage * L::kABytes, sB + stage * L::kBBytes, p, tm * kStrBM,
                   tn * kStrBN, kb * kStrBK, tid);
        fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
        mbar_arrive(full0 + 8 * stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == kMmaWarp) {
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
          for (int k = 0; k < kStrBK / 16; ++k) {
            const uint64_t bd = make_sw128_desc(b_base + k * 32, 16, 1024);
            mma_f16(d_tmem, make_sw128_desc(a_base + k * 32, 16, 1024), bd, idesc, (kb | k) != 0);
            // row-class tiles: stage rows 128..255 into accumulator columns 256..511
            if (kTma)
              mma_f16(d_tmem + kStrBN, make_sw128_desc(a_base + kStrBM * 128 + k * 32, 16, 1024),
                      bd, idesc, (kb | k) != 0);
          }
          mma_commit(empty0 + 8 * stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * acc);
        if (++acc == L::kAccs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok || *abort_flag) {
        mma_commit(drain);
        wait_bounded(drain, 0, abort_flag, p.timeout_ns, timeout_code(kRoleMma, 0x300), false);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    constexpr int kBM = str_bm<kTma>();
    constexpr int kHalves = kBM / 128;  // accumulator halves (stage rows 128h ..)
    const uint32_t quad = static_cast<uint32_t>(warp & 3);  // TMEM lanes of this warp
    // 32 x 33 words: row `lane` of a 32 x 32 accumulator block, read back by column
    uint32_t* xp = reinterpret_cast<uint32_t*>(smem + L::kXposeOffset +
                                               (warp - kMmaWarp - 1) * L::kXposeBytes);
    uint32_t acc = 0, acc_phase = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int tm, tn;
      tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
      if (!wait_bounded_sleeping(tfull0 + 8 * acc, acc_phase, abort_flag, p.timeout_ns,
                        timeout_code(kRoleEpilogue, acc)))
        break;
      tc_fence_after();
#pragma unroll 1
      for (int h = 0; h < kHalves; ++h) {
      // accumulator lane quad * 32 + lane of half h is stage row 128 h + that
      // lane: its tile row (rows come in class order in the row-class variant)
      const int first_lane = 128 * h + static_cast<int>(quad * 32);
      const int m = tm * kBM + (kTma ? class_row(first_lane + static_cast<int>(lane))
                                     : first_lane + static_cast<int>(lane));
      const uint32_t t_row = tmem_base + ((quad * 32) << 16) + acc * kStrBN + h * kStrBN;
#pragma unroll 1
      for (int c = 0; c < kStrBN / 32; ++c) {
        uint32_t r[32];
        if (kTma) {
          // tile columns 32c .. 32c + 31: column 32c + q + 8i (class q, i < 4)
          // is accumulator column 32q + 4c + i
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            uint32_t r4[4];
            tmem_ld_32x32b_x4(t_row + 32 * q + 4 * c, r4);
#pragma unroll
            for (int i = 0; i < 4; ++i) r[q + 8 * i] = r4[i];
          }
        } else {
          tmem_ld_32x32b_x32(t_row + c * 32, r);
        }
        tmem_wait_ld();
        if (p.sCn == 1) {
          // row-major C/D: transpose the block through shared memory, then
          // row i of the block is read and written by the 32 lanes at once
#pragma unroll
          for (int j = 0; j < 32; ++j) xp[lane * 33 + j] = r[j];
          __syncwarp();
          const int n = tn * kStrBN + c * 32 + static_cast<int>(lane);
#pragma unroll 1
          for (int i0 = 0; i0 < 32; i0 += 8) {
            __half cv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int li = first_lane + i0 + i;
              const int mi = tm * kBM + (kTma ? class_row(li) : li);
              cv[i] = (mi < p.M && n < p.N) ? p.CD[static_cast<int64_t>(mi) * p.sCm + n]
                                            : __ushort_as_half(0);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int li = first_lane + i0 + i;
              const int mi = tm * kBM + (kTma ? class_row(li) : li);
              if (mi < p.M && n < p.N) {
                const uint32_t a = xp[(i0 + i) * 33 + static_cast<int>(lane)];
                p.CD[static_cast<int64_t>(mi) * p.sCm + n] =
                    p.acc_f16 ? __hadd(__ushort_as_half(static_cast<unsigned short>(a)), cv[i])
                              : __float2half_rn(__uint_as_float(a) + __half2float(cv[i]));
              }
            }
          }
          __syncwarp();  // the block is read before the next one is written
        } else if (m < p.M) {
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
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      if (++acc == L::kAccs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * kStrBN);
  }
}

}  // namespace gemm_tn_dev
