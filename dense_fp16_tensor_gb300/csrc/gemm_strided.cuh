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
// the map's rows), brings a K block in as boxes 72 elements wide (the block
// plus the offset) into a raw ring; warps 0-11 then cut each 8-element chunk
// out of the two raw 16-byte words under it (shift_window) into the
// swizzled stage the MMA reads.  Rows past M / N and K past the end arrive
// as zeros from the tensor maps' bounds.
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
constexpr int kStrMmaWarp = kStrProducers / 32;

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

constexpr int kStrRawK = kStrBK + 8;        // elements per raw row (the block plus the offset)
constexpr int kStrRawRowBytes = kStrRawK * 2;  // 144

template <bool kTma>
struct StridedSmem {
  static constexpr int kStages = kTma ? 2 : kStrStages;  // swizzled stages the MMA reads
  static constexpr int kRawStages = kTma ? 2 : 0;
  static constexpr uint32_t kABytes = kStrBM * kStrBK * 2;  // 16 KiB
  static constexpr uint32_t kBBytes = kStrBN * kStrBK * 2;  // 32 KiB
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  // raw ring: per class 16 rows of A and 32 rows of B, 144 bytes each
  static constexpr uint32_t kRawABytes = kStrBM * kStrRawRowBytes;  // 18 KiB
  static constexpr uint32_t kRawBBytes = kStrBN * kStrRawRowBytes;  // 36 KiB
  static constexpr uint32_t kRawStageBytes = kRawABytes + kRawBBytes;
  static constexpr uint32_t kRawOffset = kStages * kStageBytes;
  // per epilogue warp a 32 x 33 word transpose buffer
  static constexpr uint32_t kXposeOffset = kRawOffset + kRawStages * kRawStageBytes;
  static constexpr uint32_t kXposeBytes = 32 * 33 * 4;
  static constexpr uint32_t kBarOffset = kXposeOffset + 4 * kXposeBytes;
  static constexpr uint32_t kNumBars = 2 * kStages + 5 + 2 * kRawStages;
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

// Row-class variant: this thread's chunks of a stage, kStrChunks of them (A's
// 1024 chunks first, then B's 2048, dealt round-robin to the producer
// threads).  Chunks are numbered class by class (row j of class c is tile
// row c + 8j), so the 32 chunks of one warp instruction share a class and
// its shift: the shift's branch is uniform across the warp.  The offsets do
// not depend on the K block, so they are worked out once.
constexpr int kStrChunks = (kStrBM + kStrBN) * 8 / kStrProducers;
static_assert(kStrChunks * kStrProducers == (kStrBM + kStrBN) * 8, "whole chunks per thread");
static_assert(kStrBM * 8 % 32 == 0, "A's chunks end on a warp boundary");

struct RowChunks {
  // per chunk: bits 0-15 its first aligned word in the raw stage (< 64 KiB),
  // bits 16-30 its 16 bytes in the A or B part of the swizzled stage, bit 31
  // set for B (the same in a whole warp: A's chunks end on a warp boundary)
  uint32_t off[kStrChunks];
  uint32_t shifts;  // bits 4i..4i+3: byte offset of chunk i in its first word
};

template <typename L>
__device__ __forceinline__ RowChunks row_chunks(uint32_t a_shifts, uint32_t b_shifts, int tid) {
  static_assert(kStrBM == 128 && kStrBN == 256, "class sizes below");
  constexpr int kA = kStrBM * 8;
  static_assert(L::kRawStageBytes <= 65536 && kStrBN * 128 <= 32768, "packed offsets");
  RowChunks rc;
  uint32_t shifts = 0;
#pragma unroll
  for (int i = 0; i < kStrChunks; ++i) {
    const int q = tid + i * kStrProducers;
    const bool is_a = q < kA;
    const int qq = is_a ? q : q - kA;
    const int c = is_a ? qq >> 7 : qq >> 8, within = is_a ? qq & 127 : qq & 255;
    const int j = within >> 3, k8 = within & 7, r = c + 8 * j;
    const uint32_t raw_off = (is_a ? (c * (kStrBM / 8) + j) * kStrRawRowBytes
                                    : L::kRawABytes + (c * (kStrBN / 8) + j) * kStrRawRowBytes) +
                             16 * k8;
    const uint32_t dst_off = r * 128 + 16 * (k8 ^ (r & 7));
    rc.off[i] = raw_off | (dst_off << 16) | (is_a ? 0u : 0x80000000u);
    shifts |= (((is_a ? a_shifts : b_shifts) >> (4 * c)) & 15u) << (4 * i);
  }
  rc.shifts = shifts;
  return rc;
}

// Cut one stage of the swizzled ring out of a raw stage.
__device__ __forceinline__ void rows_to_stage(const uint8_t* raw, uint8_t* dst_a, uint8_t* dst_b,
                                              const RowChunks& rc) {
  // four chunks at a time: their loads in flight together, within the
  // registers the block's size leaves a thread
  constexpr int kBatch = 4;
  static_assert(kStrChunks % kBatch == 0, "whole batches");
#pragma unroll
  for (int b = 0; b < kStrChunks; b += kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const uint32_t off = rc.off[b + i];
      const uint4* w = reinterpret_cast<const uint4*>(raw + (off & 0xFFFFu));
      const int sh = static_cast<int>((rc.shifts >> (4 * (b + i))) & 15u);
      v[i] = sh ? shift_window(w[0], w[1], sh) : w[0];
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const uint32_t off = rc.off[b + i];
      *reinterpret_cast<uint4*>(((off >> 31) ? dst_b : dst_a) + ((off >> 16) & 0x7FFFu)) = v[i];
    }
  }
}

template <bool kTma>
__global__ void __launch_bounds__(kStrThreads, 1)
    gemm_tn_strided_kernel(const __grid_constant__ StridedMaps maps, const StridedArgs p) {
  using L = StridedSmem<kTma>;
  constexpr int kStages = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;                             // stage s at s * kABytes
  uint8_t* sB = smem + kStages * L::kABytes;      // stage s at s * kBBytes
  uint8_t* raw0 = smem + L::kRawOffset;           // raw stage s at s * kRawStageBytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kCtlOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kCtlOffset + 4);

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + kStages);
  const uint32_t tfull0 = smem_u32(bars + 2 * kStages);
  const uint32_t tempty0 = smem_u32(bars + 2 * kStages + 2);
  const uint32_t drain = smem_u32(bars + 2 * kStages + 4);
  const uint32_t raw_full0 = smem_u32(bars + 2 * kStages + 5);
  const uint32_t raw_empty0 = raw_full0 + 8 * L::kRawStages;

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, kStrProducers);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 4);
    }
    mbar_init(drain, 1);
    for (int s = 0; s < L::kRawStages; ++s) {
      mbar_init(raw_full0 + 8 * s, 1);
      mbar_init(raw_empty0 + 8 * s, kStrProducers);
    }
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (kTma && threadIdx.x == 32) {
    for (int c = 0; c < 8; ++c) {
      tma_prefetch_desc(&maps.a[c]);
      tma_prefetch_desc(&maps.b[c]);
    }
  }
  if (warp == kStrMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 2 * kStrBN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp < kStrMmaWarp && kTma) {
    // ------------------------------------------------ row-class TMA producer
    const int tid = static_cast<int>(threadIdx.x);
    const int my_tiles = p.num_tiles > static_cast<int>(blockIdx.x)
                             ? (p.num_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                             : 0;
    const int units = my_tiles * p.k_blocks;  // (tile, K block) pairs of this CTA, in order
    uint32_t issued_mask = 0, issued_parity = 0;  // thread 0: raw stages with copies in flight
    // thread 0 loads unit u into raw stage u % 2 once the stage's previous
    // unit has been cut out by every producer thread
    auto issue = [&](int u) -> bool {
      const int slot = u % L::kRawStages;
      const uint32_t use = static_cast<uint32_t>(u / L::kRawStages);
      if (!wait_bounded(raw_empty0 + 8 * slot, (use & 1u) ^ 1u, abort_flag, p.timeout_ns,
                        timeout_code(kRoleProducer, 0x400 + slot)))
        return false;
      const int t = static_cast<int>(blockIdx.x) + (u / p.k_blocks) * static_cast<int>(gridDim.x);
      const int kb = u % p.k_blocks;
      int tm, tn;
      tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
      const uint32_t fb = raw_full0 + 8 * slot;
      const uint32_t dst = smem_u32(raw0 + slot * L::kRawStageBytes);
      mbar_arrive_expect_tx(fb, L::kRawStageBytes);
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        tma_load_2d(dst + c * (kStrBM / 8) * kStrRawRowBytes, &maps.a[c], fb, kb * kStrBK,
                    tm * (kStrBM / 8));
        tma_load_2d(dst + L::kRawABytes + c * (kStrBN / 8) * kStrRawRowBytes, &maps.b[c], fb,
                    kb * kStrBK, tn * (kStrBN / 8));
      }
      issued_mask |= 1u << slot;
      issued_parity = (issued_parity & ~(1u << slot)) | ((use & 1u) << slot);
      return true;
    };
    bool ok = true;
    const RowChunks rc = row_chunks<L>(p.a_shifts, p.b_shifts, tid);
    if (tid == 0) {
      for (int u = 0; ok && u < min(units, L::kRawStages); ++u) ok = issue(u);
    }
    for (int u = 0; ok && u < units; ++u) {
      const int slot = u % L::kRawStages;
      const int ss = u % kStages;
      if (!wait_bounded(raw_full0 + 8 * slot, static_cast<uint32_t>(u / L::kRawStages) & 1u,
                        abort_flag, p.timeout_ns, timeout_code(kRoleProducer, 0x500 + slot)) ||
          !wait_bounded(empty0 + 8 * ss, (static_cast<uint32_t>(u / kStages) & 1u) ^ 1u,
                        abort_flag, p.timeout_ns, timeout_code(kRoleProducer, ss))) {
        ok = false;
        break;
      }
      rows_to_stage(raw0 + slot * L::kRawStageBytes, sA + ss * L::kABytes,
                    sB + ss * L::kBBytes, rc);
      fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
      mbar_arrive(full0 + 8 * ss);
      mbar_arrive(raw_empty0 + 8 * slot);
      if (tid == 0 && u + L::kRawStages < units) ok = issue(u + L::kRawStages);
    }
    if (tid == 0 && (!ok || *abort_flag)) {
      // every copy this thread issued lands before the CTA can leave
      for (int s = 0; s < L::kRawStages; ++s)
        if (issued_mask >> s & 1u)
          wait_bounded(raw_full0 + 8 * s, issued_parity >> s & 1u, abort_flag, p.timeout_ns,
                       timeout_code(kRoleProducer, 0x600 + s), false);
    }
  } else if (warp < kStrMmaWarp) {
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
  } else if (warp == kStrMmaWarp) {
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
          if (++stage == kStages) {
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
    const uint32_t quad = static_cast<uint32_t>(warp & 3);  // TMEM lanes of this warp
    const int row_in_tile = static_cast<int>(quad * 32 + lane);
    // 32 x 33 words: row `lane` of a 32 x 32 accumulator block, read back by column
    uint32_t* xp = reinterpret_cast<uint32_t*>(smem + L::kXposeOffset +
                                               (warp - kStrMmaWarp - 1) * L::kXposeBytes);
    uint32_t acc = 0, acc_phase = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int tm, tn;
      tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
      if (!wait_bounded_sleeping(tfull0 + 8 * acc, acc_phase, abort_flag, p.timeout_ns,
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
        if (p.sCn == 1) {
          // row-major C/D: transpose the block through shared memory, then
          // row i of the block is read and written by the 32 lanes at once
#pragma unroll
          for (int j = 0; j < 32; ++j) xp[lane * 33 + j] = r[j];
          __syncwarp();
          const int n = tn * kStrBN + c * 32 + static_cast<int>(lane);
          const int mrow0 = tm * kStrBM + static_cast<int>(quad * 32);
#pragma unroll 1
          for (int i0 = 0; i0 < 32; i0 += 8) {
            __half cv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int mi = mrow0 + i0 + i;
              cv[i] = (mi < p.M && n < p.N) ? p.CD[static_cast<int64_t>(mi) * p.sCm + n]
                                            : __ushort_as_half(0);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int mi = mrow0 + i0 + i;
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
  if (warp == kStrMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * kStrBN);
  }
}

}  // namespace gemm_tn_dev
