// common.cuh -- pieces shared by the GEMM kernels: the sticky device error
// word, bounded mbarrier waits and the tile raster.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

#include "ptx.cuh"

namespace gemm_tn_dev {

// Sticky error word: the first wait that gives up records who it was.
//   bits 24-31: 0xE1 (marks a timeout), bits 16-23: role, bits 0-15: stage
// (The library is one translation unit, so the definition lives here.)
__device__ uint32_t g_error_word = 0u;

enum : uint32_t { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3 };

__device__ __forceinline__ uint32_t timeout_code(uint32_t role, uint32_t stage) {
  return 0xE1000000u | (role << 16) | (stage & 0xFFFFu);
}

// Wait for the phase of `bar` with parity `parity`, giving up after
// `limit_ns` of wall time.  On giving up, record `code` in the error word,
// raise the CTA's abort flag (and the peer CTA's, when peer_abort is a
// shared::cluster address) and return false.  With honour_abort, also return
// false (without recording) as soon as another role raised the flag.
// kCluster selects cluster-scope acquire, for barriers other CTAs arrive on.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile uint32_t* abort_flag, uint64_t limit_ns,
                                             uint32_t code, bool honour_abort = true,
                                             uint32_t peer_abort = 0u) {
  auto probe = [&]() {
    return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (probe()) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (probe()) return true;
    if ((i & 15u) == 0) {
      if (honour_abort && *abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        atomicCAS(&g_error_word, 0u, code);
        *abort_flag = 1u;
        if (peer_abort) st_shared_cluster_u32(peer_abort, 1u);
        return false;
      }
    }
  }
}

// Epilogue operands and scalars, shared by every kernel:
//   D(l,m,n) = fp16( alpha * acc(l,m,n) + beta * C(l,m,n) )
// for batch l (the simple_gemm page's cuBLAS comparison, section 8.1, uses
// this alpha / beta form).  With scaled == 0 (alpha = beta = 1) the sum is
// acc + C in the accumulator's precision (fp32, or fp16 for fp16
// accumulation); otherwise it is formed in fp32 as fma(alpha, acc, beta * C)
// and rounded once.  With read_c == 0 (beta == 0) the C term is left out:
// D = alpha * acc, C is not read, and NaN or Inf stored there cannot reach
// D (an absent term is not added as +0, so a lone -0 stays -0).
struct EpiArgs {
  const __half* C;
  int64_t ldC, sC;  // row and batch strides of C (elements)
  __half* D;
  int64_t ldD, sD;  // row and batch strides of D
  float alpha, beta;
  int scaled;       // (alpha, beta) != (1, 1)
  int read_c;       // beta != 0
};

// Two outputs from fp32 accumulator values and two C values.
__device__ __forceinline__ __half2 epi_f32x2(const EpiArgs& e, float a0, float a1, __half2 c) {
  const float2 cf = __half22float2(c);
  if (!e.scaled) return __floats2half2_rn(a0 + cf.x, a1 + cf.y);
  if (!e.read_c) return __floats2half2_rn(e.alpha * a0, e.alpha * a1);
  return __floats2half2_rn(fmaf(e.alpha, a0, e.beta * cf.x), fmaf(e.alpha, a1, e.beta * cf.y));
}

// Two outputs from an fp16 accumulator pair and two C values.
__device__ __forceinline__ __half2 epi_f16x2(const EpiArgs& e, __half2 acc, __half2 c) {
  if (!e.scaled) return __hadd2(acc, c);
  const float2 af = __half22float2(acc), cf = __half22float2(c);
  if (!e.read_c) return __floats2half2_rn(e.alpha * af.x, e.alpha * af.y);
  return __floats2half2_rn(fmaf(e.alpha, af.x, e.beta * cf.x), fmaf(e.alpha, af.y, e.beta * cf.y));
}

// One output from one accumulator word (fp32, or fp16 in the low half).
__device__ __forceinline__ __half epi_one(const EpiArgs& e, bool acc_f16, uint32_t a, __half c) {
  if (acc_f16) {
    const __half ah = __ushort_as_half(static_cast<unsigned short>(a));
    if (!e.scaled) return __hadd(ah, c);
    if (!e.read_c) return __float2half_rn(e.alpha * __half2float(ah));
    return __float2half_rn(fmaf(e.alpha, __half2float(ah), e.beta * __half2float(c)));
  }
  const float af = __uint_as_float(a);
  if (!e.scaled) return __float2half_rn(af + __half2float(c));
  if (!e.read_c) return __float2half_rn(e.alpha * af);
  return __float2half_rn(fmaf(e.alpha, af, e.beta * __half2float(c)));
}

// Phase trace (gemm_tn_options.trace): when a launch has tracing on, one
// thread per role stamps %globaltimer into g_trace at fixed points, per CTA,
// so that a launch's time can be split into set-up, first data, main loop,
// drain and exit.  Slot layout per CTA (kTraceSlots 64-bit words):
//   0 entry               kernel start (thread 0)
//   1 ready               after griddepcontrol.wait (producer)
//   2 first stage         first pipeline stage complete (MMA issuer)
//   3 last MMA            last accumulator committed (MMA issuer)
//   4 first accumulator   first accumulator ready (first epilogue warp)
//   5 last chunk          last output chunk handed to the copy engine
//   6 stores done         the CTA's last stores performed (first epilogue warp)
//   7 exit                before tensor memory is freed (thread 0)
//   8 SM id, 9 work units of this CTA
//   10, 11 the SM's cycle counter at entry and at exit (with slots 0 and 7:
//          the clock the CTA ran at)
// CTAs past kTraceCtas are not recorded.
constexpr int kTraceSlots = 12;
constexpr int kTraceCtas = 512;
enum : int {
  kTrEntry = 0, kTrReady, kTrFirstStage, kTrLastMma, kTrFirstAcc, kTrLastChunk,
  kTrStoresDone, kTrExit, kTrSm, kTrUnits, kTrCyclesEntry, kTrCyclesExit
};

// (One translation unit: the definition lives here, like g_error_word.)
__device__ __align__(256) uint64_t g_trace[kTraceCtas * kTraceSlots];

__device__ __forceinline__ void trace_mark(int on, int slot) {
  if (on && blockIdx.x < kTraceCtas) g_trace[blockIdx.x * kTraceSlots + slot] = globaltimer_ns();
}

__device__ __forceinline__ void trace_value(int on, int slot, uint64_t v) {
  if (on && blockIdx.x < kTraceCtas) g_trace[blockIdx.x * kTraceSlots + slot] = v;
}

// Entry / exit stamps with the SM's cycle counter beside the global time.
__device__ __forceinline__ void trace_entry(int on) {
  if (on && blockIdx.x < kTraceCtas) {
    g_trace[blockIdx.x * kTraceSlots + kTrCyclesEntry] = static_cast<uint64_t>(clock64());
    g_trace[blockIdx.x * kTraceSlots + kTrEntry] = globaltimer_ns();
  }
}

__device__ __forceinline__ void trace_exit(int on) {
  if (on && blockIdx.x < kTraceCtas) {
    g_trace[blockIdx.x * kTraceSlots + kTrExit] = globaltimer_ns();
    g_trace[blockIdx.x * kTraceSlots + kTrCyclesExit] = static_cast<uint64_t>(clock64());
  }
}

__device__ __forceinline__ uint32_t sm_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}

// Grouped raster over output tiles: runs of `group_m` tile-rows are walked
// column by column, so CTAs that run at the same time share A row-panels and
// B column-panels in L2.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group_m,
                                            int& tm, int& tn) {
  const int per_group = group_m * tiles_n;
  const int g = t / per_group;
  const int first_m = g * group_m;
  const int rows = min(tiles_m - first_m, group_m);
  const int r = t - g * per_group;
  tm = first_m + r % rows;
  tn = r / rows;
}

// Quotient of two non-negative 64-bit values, in 32-bit arithmetic when both
// fit (a 64-bit division is a long software routine; the unit indices of a
// real problem are far below 2^31).
__device__ __forceinline__ int64_t div_nonneg(int64_t a, int64_t b) {
  if ((static_cast<uint64_t>(a) | static_cast<uint64_t>(b)) >> 31 == 0)
    return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
  return a / b;
}

// Contiguous split of `units` work units into ranges of `per` units: CTA c
// owns [c*per, min((c+1)*per, units)); the last non-empty range may be
// shorter, and the grid has ceil(units/per) CTAs.
__device__ __forceinline__ int64_t unit_begin(int64_t units, int cta, int64_t per) {
  return min(static_cast<int64_t>(cta) * per, units);
}

// CTA whose unit range holds unit u.
__device__ __forceinline__ int cta_of_unit(int64_t u, int64_t per) {
  return static_cast<int>(div_nonneg(u, per));
}

}  // namespace gemm_tn_dev
