// shift.cuh -- a 16-byte window at any even byte offset of two consecutive
// aligned 16-byte words: how the row copy and the strided kernel's producer
// read rows that are not on the 16-byte grid with aligned vector loads only.
#pragma once

#include <cstdint>

namespace gemm_tn_dev {

// Bytes [sh, sh + 16) of the 32-byte concatenation lo:hi (sh even, 0..14):
// words of the window shifted by whole words (q = sh / 4) and, for sh % 4
// == 2, by a further half word.
__device__ __forceinline__ uint4 shift_window(const uint4& lo, const uint4& hi, int sh) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint32_t o[4];
  const bool half = (sh & 3) != 0;
  switch (sh >> 2) {
#define GEMM_TN_SHIFT_CASE(Q)                                                        \
  case Q:                                                                            \
    _Pragma("unroll") for (int i = 0; i < 4; ++i) o[i] =                             \
        half ? __funnelshift_r(w[Q + i], w[Q + i + 1], 16) : w[Q + i];               \
    break;
    GEMM_TN_SHIFT_CASE(0)
    GEMM_TN_SHIFT_CASE(1)
    GEMM_TN_SHIFT_CASE(2)
    default:
      _Pragma("unroll") for (int i = 0; i < 3; ++i) o[i] =
          half ? __funnelshift_r(w[3 + i], w[4 + i], 16) : w[3 + i];
      o[3] = half ? __funnelshift_r(w[6], w[7], 16) : w[6];
      break;
#undef GEMM_TN_SHIFT_CASE
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace gemm_tn_dev
