// common.cuh -- pieces shared by the GEMM kernels: the sticky device error
// word, bounded mbarrier waits and the tile raster.
#pragma once

#include <cstdint>

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

// Contiguous split of `units` work units over `grid` CTAs: CTA c owns
// [unit_begin(c), unit_begin(c+1)).
__device__ __forceinline__ int64_t unit_begin(int64_t units, int cta, int grid) {
  return units * cta / grid;
}

// CTA whose unit range holds unit u (ranges from unit_begin are monotone).
__device__ __forceinline__ int cta_of_unit(int64_t u, int64_t units, int grid) {
  int c = static_cast<int>(u * grid / units);
  while (c + 1 < grid && unit_begin(units, c + 1, grid) <= u) ++c;
  while (c > 0 && unit_begin(units, c, grid) > u) --c;
  return c;
}

}  // namespace gemm_tn_dev
