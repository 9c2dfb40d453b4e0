// gemm_tn.cu -- host side of the C ABI in include/gemm_tn.h: argument
// checks, path choice, TMA descriptor construction and kernel launches.
//
// The operation, the operand views and the status codes are specified in the
// header.  This file owns:
//   * validation (sizes, leading dimensions, alignment, aliasing) before any
//     work is enqueued;
//   * tensor maps for A, B and D (128-byte swizzle, zero fill out of range,
//     a batch coordinate), built with cuTensorMapEncodeTiled from the
//     driver entry point;
//   * the choice of path (tile kernels, skinny split-K, scale-only) and of
//     tile kernel, K splits and stream-K, and the grid sizes (one CTA per
//     SM, persistent);
//   * stream-ordered workspaces from a library-owned memory pool (split-K
//     partials, stream-K partials, repacked strided operands).
// Every entry point describes its call as one Problem (a batch of
// D = alpha * A.B^T + beta * C); gemm_tn itself is the case batch 1,
// alpha = beta = 1, D = C in place.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>

#include "../../include/gemm_tn.h"
#include "gemm_large.cuh"
#include "gemm_large2.cuh"
#include "gemm_wide.cuh"
#include "gemm_skinny.cuh"
#include "gemm_skinny_cluster.cuh"
#include "gemm_strided.cuh"
#include "repack.cuh"
#include "scale.cuh"

namespace {

using namespace gemm_tn_dev;

constexpr int kMaxDevices = 64;
constexpr int kSkinnyMaxM = 256;  // the skinny kernel serves M <= 256
// The automatic choice takes the skinny path for M <= 192 and, for M up to
// 256, while N is at most this: 56 CTA-pair tiles of 256 columns, under 3/4
// of the pairs a GB300 runs at once.  Wider N keeps the pair kernel busy
// enough to stream B faster than the skinny kernel's 4-stage ring at MMA
// width 256.
constexpr int64_t kSkinnyWideMaxN = 56 * 256;
// ... and only from this K on: shorter K loops finish sooner on the tile
// kernels (one launch, no partial sums; 128 x 128 tiles with their own K
// split when they leave SMs idle).  Crossovers measured one call at a time
// with a cold L2: K ~ 2048 for M = 16, ~4096-8192 for M = 64, ~8192 for
// M = 128 and 256 (tile / skinny at K = 512: 14 / 17-24 us).
constexpr int64_t skinny_min_k(int64_t M) { return M <= 32 ? 2048 : M <= 64 ? 4096 : 8192; }
constexpr int kNoallocMaxM = 64;   // the allocation-free entry point's limit
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;  // 1 s per wait

thread_local int t_last_launches = 0;
thread_local const char* t_last_kernels = "";

struct DeviceState {
  bool probed = false;
  bool supported = false;
  int num_sms = 0;
  bool attrs_set = false;
  int max_pairs = 0;  // CTA pairs of gemm_tn_large2_kernel that fit at once
  cudaMemPool_t pool = nullptr;  // library-owned stream-ordered workspace pool
  uint64_t* trace = nullptr;     // device address of g_trace on this device
};

// Workspaces come from a pool owned by the library (one per device) that
// keeps up to this much memory cached between calls, so a call's workspace
// is normally served without new physical allocation.
constexpr uint64_t kPoolKeepBytes = 1ull << 30;

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int resolve_encoder() {
  if (g_encode) return GEMM_TN_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
    return GEMM_TN_ERR_CUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return GEMM_TN_OK;
}

template <int STAGES, int MP>
cudaError_t set_skinny_attr() {
  cudaError_t e = cudaFuncSetAttribute(gemm_tn_skinny_kernel<STAGES, MP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SkinnySmem<STAGES, MP>::kDynamicBytes);
  constexpr int CS = cluster_stages(MP);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_tn_skinny_cluster_kernel<CS, MP>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             ClusterSmem<CS, MP>::kDynamicBytes);
  return e;
}

// Ring depth of the skinny kernel: stages of two 64-deep sub-blocks up to
// MP = 128 -- 5 of 36-40 KiB up to MP = 32, 4 of 44-56 KiB up to 96, 3 of
// 64 KiB at 128 -- and of one sub-block above: 5 at 192 (40 KiB) and 4 at
// 256 (48 KiB).
constexpr int skinny_stages(int mp) {
  return mp <= 32 ? 5 : (mp <= 64 ? 4 : (mp <= 96 ? 4 : (mp <= 128 ? 3 : (mp <= 192 ? 5 : 4))));
}

// MMA width for M rows of A: M rounded up to 16 up to 64, then 96, 128, 192
// or 256.
int skinny_mp(int64_t M) {
  if (M <= 64) return static_cast<int>((M + 15) / 16 * 16);
  return M <= 96 ? 96 : (M <= 128 ? 128 : (M <= 192 ? 192 : 256));
}

}  // namespace

// Phase-trace records (g_trace, common.cuh) of the last traced launch on
// each device (gemm_tn_options.trace).
static_assert(GEMM_TN_TRACE_CTAS == kTraceCtas && GEMM_TN_TRACE_SLOTS == kTraceSlots,
              "trace layout of the header and the kernels");

namespace {

// Per-device set-up (under g_mu): capability check, SM count, kernel
// attributes.  Returns a status.
int device_setup(int dev, DeviceState*& st) {
  if (dev < 0 || dev >= kMaxDevices) return GEMM_TN_ERR_UNSUPPORTED;
  st = &g_dev[dev];
  if (!st->probed) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return GEMM_TN_ERR_CUDA;
    st->probed = true;
    st->supported = (major == 10 && minor == 3);
    st->num_sms = sms;
  }
  if (!st->supported) return GEMM_TN_ERR_UNSUPPORTED;
  if (!st->attrs_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tn_large_kernel<256>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         LargeSmem<256>::kDynamicBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_tn_large_kernel<64>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               LargeSmem<64>::kDynamicBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_tn_large_kernel<64, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               LargeSmem<64, true>::kDynamicBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_tn_large_kernel<128>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               LargeSmem<128>::kDynamicBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_tn_large_kernel<128, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               LargeSmem<128, true>::kDynamicBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_tn_large2_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               PairSmem<false>::kDynamicBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_tn_large2_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               PairSmem<true>::kDynamicBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_tn_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               WideSmem::kDynamicBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_tn_strided_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               StridedSmem<false>::kDynamicBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_tn_strided_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               StridedSmem<true>::kDynamicBytes);
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg;
      std::memset(&cfg, 0, sizeof cfg);
      cfg.gridDim = dim3(2 * static_cast<unsigned>(st->num_sms / 2), 1, 1);
      cfg.blockDim = dim3(kPairThreads, 1, 1);
      static_assert(PairSmem<false>::kDynamicBytes >= PairSmem<true>::kDynamicBytes,
                    "pair occupancy is taken from the larger layout");
      cfg.dynamicSmemBytes = PairSmem<false>::kDynamicBytes;
      int clusters = 0;
      e = cudaOccupancyMaxActiveClusters(&clusters, gemm_tn_large2_kernel<false>, &cfg);
      st->max_pairs = clusters;
    }
    if (e == cudaSuccess) e = set_skinny_attr<skinny_stages(16), 16>();
    if (e == cudaSuccess) e = set_skinny_attr<skinny_stages(32), 32>();
    if (e == cudaSuccess) e = set_skinny_attr<skinny_stages(48), 48>();
    if (e == cudaSuccess) e = set_skinny_attr<skinny_stages(64), 64>();
    if (e == cudaSuccess) e = set_skinny_attr<skinny_stages(96), 96>();
    if (e == cudaSuccess) e = set_skinny_attr<skinny_stages(128), 128>();
    if (e == cudaSuccess) e = set_skinny_attr<skinny_stages(192), 192>();
    if (e == cudaSuccess) e = set_skinny_attr<skinny_stages(256), 256>();
    if (e != cudaSuccess) return GEMM_TN_ERR_CUDA;
    st->attrs_set = true;
  }
  if (resolve_encoder() != GEMM_TN_OK) return GEMM_TN_ERR_CUDA;
  if (st->trace == nullptr) {
    void* t = nullptr;
    if (cudaGetSymbolAddress(&t, gemm_tn_dev::g_trace) != cudaSuccess || t == nullptr) {
      cudaGetLastError();
      return GEMM_TN_ERR_CUDA;
    }
    st->trace = static_cast<uint64_t*>(t);
  }
  return GEMM_TN_OK;
}

// Whether this call's kernel traces (the buffer is cleared on the stream
// first).
int trace_for(const gemm_tn_options& o, const DeviceState& st, cudaStream_t stream) {
  if (!o.trace) return 0;
  if (cudaMemsetAsync(st.trace, 0, sizeof(uint64_t) * kTraceCtas * kTraceSlots, stream) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return 1;
}

// The device's workspace pool (under g_mu), created on the first call of an
// entry point that may need a workspace.  The allocation-free entry point
// never calls this.
int pool_setup(int dev, DeviceState* st) {
  if (st->pool != nullptr) return GEMM_TN_OK;
  cudaMemPoolProps props;
  std::memset(&props, 0, sizeof props);
  props.allocType = cudaMemAllocationTypePinned;
  props.location.type = cudaMemLocationTypeDevice;
  props.location.id = dev;
  cudaMemPool_t pool = nullptr;
  if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return GEMM_TN_ERR_CUDA;
  uint64_t keep = kPoolKeepBytes;
  if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
    cudaMemPoolDestroy(pool);
    return GEMM_TN_ERR_CUDA;
  }
  st->pool = pool;
  return GEMM_TN_OK;
}

// Stream-ordered workspace from the device's library pool.  With the
// test-only `test_fail_alloc` option the request fails as an exhausted pool
// would, before anything is enqueued.
cudaError_t ws_alloc(void** p, size_t bytes, const DeviceState& st, cudaStream_t stream,
                     const gemm_tn_options& o) {
  if (o.test_fail_alloc) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMallocFromPoolAsync(p, bytes, st.pool, stream);
}

// Tensor map over a (rows, K) operand.  K-major: dims {K, rows}, box
// {64, box_rows}.  MN-major: dims {rows, K}, box {64, 64}.  128-byte
// swizzle; out-of-range elements read as zero.
int encode_operand(CUtensorMap* map, const void* ptr, int64_t rows, int64_t K, int64_t ld,
                   int mn_major, uint32_t box_rows) {
  cuuint64_t dims[2], strides[1];
  cuuint32_t box[2], estr[2] = {1, 1};
  if (!mn_major) {
    dims[0] = static_cast<cuuint64_t>(K);
    dims[1] = static_cast<cuuint64_t>(rows);
    box[0] = 64;
    box[1] = box_rows;
  } else {
    dims[0] = static_cast<cuuint64_t>(rows);
    dims[1] = static_cast<cuuint64_t>(K);
    box[0] = 64;
    box[1] = 64;
  }
  strides[0] = static_cast<cuuint64_t>(ld) * 2;
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_TN_OK : GEMM_TN_ERR_CUDA;
}

// The same over a batch: dims {inner, outer, L} with batch stride `bstride`
// elements.  A shared operand (bstride 0) or a single problem gets a batch
// extent of 1 (its coordinate is always 0) and a nominal stride.
int encode_operand_batched(CUtensorMap* map, const void* ptr, int64_t rows, int64_t K,
                           int64_t ld, int64_t bstride, int64_t L, int mn_major,
                           uint32_t box_rows) {
  const int64_t inner = mn_major ? rows : K, outer = mn_major ? K : rows;
  const bool batched = L > 1 && bstride != 0;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer),
                        static_cast<cuuint64_t>(batched ? L : 1)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2,
                           static_cast<cuuint64_t>(batched ? bstride : outer * ld) * 2};
  cuuint32_t box[3] = {64, mn_major ? 64u : box_rows, 1}, estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_TN_OK : GEMM_TN_ERR_CUDA;
}

// K-major operand as K chunks: dims {64, rows, K/64, L}, the third stepping
// K by 64 elements (128 bytes), box {64, box_rows, depth, 1}: one box brings
// 64 * depth of K for box_rows rows, as `depth` consecutive 128B-swizzled
// blocks.  Needs K
// a multiple of 64 (the inner dimension is never clipped, so a partial last
// chunk would read past K); the chunk past the last one is zero-filled.
int encode_operand_ko(CUtensorMap* map, const void* ptr, int64_t rows, int64_t K, int64_t ld,
                      int64_t bstride, int64_t L, uint32_t box_rows, uint32_t depth = 2) {
  const bool batched = L > 1 && bstride != 0;
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(K / 64),
                        static_cast<cuuint64_t>(batched ? L : 1)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(ld) * 2, 128,
                           static_cast<cuuint64_t>(batched ? bstride : rows * ld) * 2};
  cuuint32_t box[4] = {64, box_rows, depth, 1}, estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_TN_OK : GEMM_TN_ERR_CUDA;
}

// Tensor map over D, a batch of (M,N):(ldD,1) views sD elements apart, for
// 32-row x 64-column epilogue boxes with the 128-byte swizzle (the staging
// layout); out-of-range rows and columns of a stored box are not written.
int encode_d(CUtensorMap* map, void* ptr, int64_t M, int64_t N, int64_t ldD, int64_t sD,
             int64_t L) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M),
                        static_cast<cuuint64_t>(L > 1 ? L : 1)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldD) * 2,
                           static_cast<cuuint64_t>(L > 1 ? sD : M * ldD) * 2};
  cuuint32_t box[3] = {64, 32, 1}, estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_TN_OK : GEMM_TN_ERR_CUDA;
}

// One call: a batch of L problems D = alpha * A.B^T + beta * C, operand l's
// view starting l * stride elements after the base pointer.
struct Problem {
  int64_t M, N, K, L;
  float alpha, beta;
  const void* A;
  int64_t ldA, sA;
  int a_major;
  const void* B;
  int64_t ldB, sB;
  int b_major;
  const void* C;
  int64_t ldC, sC;
  void* D;
  int64_t ldD, sD;
  int accum;
  bool use_ab() const { return alpha != 0.f && K > 0; }
  bool read_c() const { return beta != 0.f; }
  bool in_place() const {
    return C == D && ldC == ldD && (L <= 1 || sC == sD);
  }
};

EpiArgs epi_of(const Problem& q) {
  EpiArgs e;
  std::memset(&e, 0, sizeof e);
  e.read_c = q.read_c() ? 1 : 0;
  e.C = e.read_c ? static_cast<const __half*>(q.C) : nullptr;
  e.ldC = q.ldC;
  e.sC = q.L > 1 ? q.sC : 0;
  e.D = static_cast<__half*>(q.D);
  e.ldD = q.ldD;
  e.sD = q.L > 1 ? q.sD : 0;
  e.alpha = q.alpha;
  e.beta = q.beta;
  e.scaled = (q.alpha != 1.f || q.beta != 1.f) ? 1 : 0;
  return e;
}

// Byte range [lo, hi) touched by a (rows, cols) view with the given major.
void extent(const void* p, int64_t rows, int64_t cols, int64_t ld, int mn_major, uintptr_t& lo,
            uintptr_t& hi) {
  const int64_t inner = mn_major ? rows : cols;
  const int64_t outer = mn_major ? cols : rows;
  lo = reinterpret_cast<uintptr_t>(p);
  hi = lo + static_cast<uintptr_t>(((outer - 1) * ld + inner) * 2);
}

// Byte range [lo, hi) touched by L views of (rows, cols) `stride` elements apart.
void extent_batched(const void* p, int64_t rows, int64_t cols, int64_t ld, int mn_major,
                    int64_t stride, int64_t L, uintptr_t& lo, uintptr_t& hi) {
  extent(p, rows, cols, ld, mn_major, lo, hi);
  if (L > 1) hi += static_cast<uintptr_t>((L - 1) * stride * 2);
}

bool overlap(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

// A batch stride whose last view starts at most 2^61 elements (2^62 bytes)
// in, so that the byte extents below stay inside 64-bit arithmetic (no
// allocation comes near that).
bool stride_in_range(int64_t stride, int64_t L) {
  return stride >= 0 && (L <= 1 || stride <= (int64_t{1} << 61) / (L - 1));
}

int validate(const Problem& q) {
  const int64_t kMax = 0x7FFFFFFF;
  if (q.M < 0 || q.N < 0 || q.K < 0 || q.L < 0 || q.M > kMax || q.N > kMax || q.K > kMax ||
      q.L > kMax)
    return GEMM_TN_ERR_INVALID_ARG;
  if ((q.a_major != GEMM_TN_MAJOR_K && q.a_major != GEMM_TN_MAJOR_MN) ||
      (q.b_major != GEMM_TN_MAJOR_K && q.b_major != GEMM_TN_MAJOR_MN))
    return GEMM_TN_ERR_INVALID_ARG;
  if (q.accum != GEMM_TN_ACC_F32 && q.accum != GEMM_TN_ACC_F16) return GEMM_TN_ERR_INVALID_ARG;
  if (q.M == 0 || q.N == 0 || q.L == 0) return GEMM_TN_OK;
  const bool batched = q.L > 1;
  // D: written; batches may not overlap one another
  if (q.D == nullptr || q.ldD < q.N || q.ldD > kMax) return GEMM_TN_ERR_INVALID_ARG;
  if (batched && (q.sD < q.M * q.ldD || !stride_in_range(q.sD, q.L)))
    return GEMM_TN_ERR_INVALID_ARG;
  uintptr_t d0, d1;
  extent_batched(q.D, q.M, q.N, q.ldD, 0, q.sD, q.L, d0, d1);
  if (q.read_c()) {
    if (q.C == nullptr || q.ldC < q.N || q.ldC > kMax || (batched && !stride_in_range(q.sC, q.L)))
      return GEMM_TN_ERR_INVALID_ARG;
    if (!q.in_place()) {
      uintptr_t c0, c1;
      extent_batched(q.C, q.M, q.N, q.ldC, 0, q.sC, q.L, c0, c1);
      if (overlap(c0, c1, d0, d1)) return GEMM_TN_ERR_INVALID_ARG;
    }
  }
  if (q.use_ab()) {
    if (q.A == nullptr || q.B == nullptr) return GEMM_TN_ERR_INVALID_ARG;
    const int64_t a_outer = q.a_major ? q.K : q.M, b_outer = q.b_major ? q.K : q.N;
    if (q.ldA < (q.a_major ? q.M : q.K) || q.ldB < (q.b_major ? q.N : q.K) || q.ldA > kMax ||
        q.ldB > kMax)
      return GEMM_TN_ERR_INVALID_ARG;
    // batch strides: 0 (one operand for every problem) or whole views apart
    if (batched && ((q.sA != 0 && q.sA < a_outer * q.ldA) || (q.sB != 0 && q.sB < b_outer * q.ldB) ||
                    !stride_in_range(q.sA, q.L) || !stride_in_range(q.sB, q.L)))
      return GEMM_TN_ERR_INVALID_ARG;
    uintptr_t a0, a1, b0, b1;
    extent_batched(q.A, q.M, q.K, q.ldA, q.a_major, q.sA, q.L, a0, a1);
    extent_batched(q.B, q.N, q.K, q.ldB, q.b_major, q.sB, q.L, b0, b1);
    if (overlap(d0, d1, a0, a1) || overlap(d0, d1, b0, b1)) return GEMM_TN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q.A) | reinterpret_cast<uintptr_t>(q.B)) & 15u)
      return GEMM_TN_ERR_ALIGNMENT;
    if ((q.ldA | q.ldB) & 7) return GEMM_TN_ERR_ALIGNMENT;
    if (batched && ((q.sA | q.sB) & 7)) return GEMM_TN_ERR_ALIGNMENT;
  }
  if ((reinterpret_cast<uintptr_t>(q.D) & 15u) || (q.ldD & 7) || (batched && (q.sD & 7)))
    return GEMM_TN_ERR_ALIGNMENT;
  if (q.read_c() && ((reinterpret_cast<uintptr_t>(q.C) & 15u) || (q.ldC & 7) ||
                     (batched && (q.sC & 7))))
    return GEMM_TN_ERR_ALIGNMENT;
  return GEMM_TN_OK;
}

// The legacy in-place description: one problem, D = C + A.B^T in CD.
Problem in_place_problem(int64_t M, int64_t N, int64_t K, const void* A, int64_t ldA,
                         int a_major, const void* B, int64_t ldB, int b_major, void* CD,
                         int64_t ldC, int accum) {
  Problem q;
  std::memset(&q, 0, sizeof q);
  q.M = M; q.N = N; q.K = K; q.L = 1;
  q.alpha = 1.f; q.beta = 1.f;
  q.A = A; q.ldA = ldA; q.a_major = a_major;
  q.B = B; q.ldB = ldB; q.b_major = b_major;
  q.C = CD; q.ldC = ldC;
  q.D = CD; q.ldD = ldC;
  q.accum = accum;
  return q;
}

// Argument checks of the in-place form (the allocation-free entry point
// uses them too).
int validate(int64_t M, int64_t N, int64_t K, const void* A, int64_t ldA, int a_major,
             const void* B, int64_t ldB, int b_major, void* CD, int64_t ldC, int accum) {
  return validate(in_place_problem(M, N, K, A, ldA, a_major, B, ldB, b_major, CD, ldC, accum));
}

int plan(int64_t M, int64_t N, int64_t K, int a_major, int b_major, int accum, int requested,
         int64_t L = 1) {
  const bool skinny_ok = M <= kSkinnyMaxM && a_major == GEMM_TN_MAJOR_K &&
                         b_major == GEMM_TN_MAJOR_K && accum == GEMM_TN_ACC_F32 && L <= 1;
  if (requested == GEMM_TN_PATH_SKINNY) return skinny_ok ? GEMM_TN_PATH_SKINNY : -1;
  if (requested == GEMM_TN_PATH_LARGE) return GEMM_TN_PATH_LARGE;
  const bool auto_ok = (M <= 192 || N <= kSkinnyWideMaxN) && K >= skinny_min_k(M);
  return skinny_ok && auto_ok ? GEMM_TN_PATH_SKINNY : GEMM_TN_PATH_LARGE;
}

// Every kernel of the library is a programmatic dependent launch: it may
// become resident while the kernel before it in the stream finishes, sets
// up its barriers and tensor memory, and waits in griddepcontrol.wait before
// it touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Automatic K split of the CTA-pair kernel for problems with few 256 x 256
// tiles and long K loops: s splits of at least 4096 of K each, as many as
// keep the units within the pairs, taken only when the units then fill at
// least half the pairs (fp32 accumulation, M and N above 128).  Measured
// with an L2 flush per call, against the automatic choice before it
// (128-row tiles, with their own K split when few): 1024^2 x 16384 51.2 ->
// 42.8 us, 512 x 2048 x 16384 52.3 -> 45.1, 1024 x 2048 x 8192 42.6 ->
// 40.0, 512 x 4096 x 8192 45.1 -> 43.1; with shorter K per split, or fewer
// units, the 128-row kernel stayed ahead (512^2 x 8192: 20.5 against 22.6
// at best).  Returns 1 for no split.
int pair_split_count(int64_t M, int64_t N, int64_t K, int64_t pair_tiles, int accum,
                     const DeviceState& st) {
  if (accum != GEMM_TN_ACC_F32 || M <= kLargeBM || N <= 128 || st.max_pairs <= 0 ||
      pair_tiles <= 0)
    return 1;
  const int64_t s = std::min<int64_t>(st.max_pairs / pair_tiles, K / 4096);
  if (s < 2 || 2 * pair_tiles * s < st.max_pairs) return 1;
  return static_cast<int>(s);
}

// Tile width of the CTA-pair kernel (unsplit): the width whose waves of
// tiles over the pairs take the least time.  A tile's time per 16-deep K
// step is the MMA's bn / 2 clocks, or, when longer, the time each SM needs
// to take in its 128 + bn / 2 rows of A and B (32 bytes each) at about 75
// bytes per clock (the TMA ingress rate measured on GB300).  Narrower tiles
// are taken only when at least 3 % faster; with an M/N-major B only widths
// that are whole 64-element boxes per CTA (256, 128).  Ragged 4000 x 3000
// tiles this way as 16 x 14 tiles of 256 x 224 (2.95 waves over 76 pairs)
// instead of 16 x 12 of 256 x 256 (2.53 waves, i.e. 3).
bool p_acc_f16(int accum) { return accum == GEMM_TN_ACC_F16; }

// The last-wave split (see launch_large) counts for 256-wide tiles: the
// partial last round then takes 1/s of a tile's time, plus ~0.1 of a tile
// for the partial sums and their reduction.
int last_wave_splits(int64_t tiles, int max_pairs, int k_blocks) {
  if (max_pairs <= 0 || tiles < max_pairs) return 0;
  const int64_t rem = tiles % max_pairs;
  if (rem == 0) return 0;
  const int s = static_cast<int>(std::min<int64_t>(std::min<int64_t>(max_pairs / rem, 4), k_blocks / 8));
  return s >= 2 ? s : 0;
}

int pair_tile_n(int64_t M, int64_t N, int64_t L, int b_major, int max_pairs, bool split_ok,
                int k_blocks) {
  int best = 256;
  double best_cost = -1.0;
  for (int bn = 256; bn >= 128; bn -= 32) {
    if (b_major == GEMM_TN_MAJOR_MN && bn % 128 != 0) continue;
    const int64_t tiles = ((M + 255) / 256) * ((N + bn - 1) / bn) * L;
    const int64_t waves = (tiles + max_pairs - 1) / max_pairs;
    const double step = std::max(bn / 2.0, (4096.0 + 16.0 * bn) / 75.0);
    double cost = static_cast<double>(waves) * step;
    const int s = bn == 256 && split_ok ? last_wave_splits(tiles, max_pairs, k_blocks) : 0;
    if (s) cost = (static_cast<double>(tiles / max_pairs) + 1.0 / s + 0.1) * step;
    if (best_cost < 0.0 || cost < 0.97 * best_cost) {
      best = bn;
      best_cost = cost;
    }
  }
  return best;
}

int launch_large(const Problem& q, cudaStream_t stream, const gemm_tn_options& o,
                 const DeviceState& st) {
  const int64_t M = q.M, N = q.N, K = q.K;
  const int a_major = q.a_major, b_major = q.b_major, accum = q.accum;
  // Kernel choice: 256 x 256 single-CTA tiles (fewest operand bytes per
  // flop per SM) unless the problem is too small to fill them or the caller
  // asked for another tile kernel.
  int kind = o.tile_kernel;
  int tile_n = o.tile_n;
  if (kind == 0) {
    // The CTA pair (256 x BN per two SMs, double-buffered accumulators,
    // 128-deep stages) for every problem with both sides above 128: at
    // 8192^3 it runs 1785-1787 TFLOP/s over 20 calls and 1621-1624 over 400
    // (power-limited) against 1751-1763 and 1619-1620 for 256 x 256 tiles
    // on one CTA, whose single accumulator stalls the MMA for each drain
    // (16384^2 x 2048: 1317 against 1639).  128-row tiles when a side is too
    // short for 256, and 128 x 128 tiles when even 128 x 256 tiles would
    // leave half the SMs idle.
    const int64_t tiles_128x256 = ((M + 127) / 128) * ((N + 255) / 256) * q.L;
    const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256) * q.L;
    if (pair_split_count(M, N, K, pair_tiles, accum, st) > 1) {
      kind = 2;  // few pair tiles with long K loops: the pair kernel with a K split
    } else if (2 * tiles_128x256 <= st.num_sms) {
      kind = 1;
      // 128 x 64 tiles when even 128 x 128 tiles would leave more than half
      // the SMs idle and no K split will spread the work instead (fp16
      // accumulation is never split; fp32 only from K = 2048 on)
      const int64_t tiles_128x128 = ((M + 127) / 128) * ((N + 127) / 128) * q.L;
      const bool no_split = accum == GEMM_TN_ACC_F16 || K < 2048;
      if (tile_n == 0) tile_n = (2 * tiles_128x128 <= st.num_sms && no_split) ? 64 : 128;
    } else if (M > kLargeBM && N > 128) {
      kind = st.max_pairs > 0 ? 2 : 3;
    } else {
      kind = 1;
      if (tile_n == 0 && N <= 128) tile_n = 128;  // a 256-wide tile would be half empty
    }
  }
  if (kind == 2 && st.max_pairs <= 0) return GEMM_TN_ERR_UNSUPPORTED;
  const bool pair = kind == 2, wide = kind == 3;
  // The pair's K split runs 256-wide tiles; an unsplit pair kernel takes the
  // width that balances its waves (tile_n, when given, is a request: 128 or
  // 256).
  const int auto_pair_splits =
      pair && o.tile_kernel == 0 && o.split_k == 0
          ? pair_split_count(M, N, K, ((M + 255) / 256) * ((N + 255) / 256) * q.L, accum, st)
          : 1;
  const bool pair_split = pair && !p_acc_f16(accum) &&
                          ((o.tile_kernel == 2 && o.split_k > 0) || auto_pair_splits > 1);
  const bool pair_width_asked = pair && o.tile_kernel == 2 && o.tile_n != 0;
  if (pair_width_asked && (pair_split || o.tile_n < 128 ||
                           (b_major == GEMM_TN_MAJOR_MN && o.tile_n % 128 != 0)))
    return GEMM_TN_ERR_INVALID_ARG;
  if (kind == 1 && tile_n != 0 && tile_n != 64 && tile_n != 128 && tile_n != 256)
    return GEMM_TN_ERR_INVALID_ARG;
  const int bn = wide ? 256
               : pair ? (pair_split ? 256
                         : pair_width_asked
                             ? o.tile_n
                             : pair_tile_n(M, N, q.L, b_major, st.max_pairs,
                                           accum == GEMM_TN_ACC_F32 && o.split_k == 0 &&
                                               o.stream_k != -1,
                                           static_cast<int>((K + (K >= 1024 ? 127 : 63)) /
                                                            (K >= 1024 ? 128 : 64))))
               : (tile_n == 64 || tile_n == 128) ? tile_n : 256;
  const int bm = (pair || wide) ? 256 : kLargeBM;
  // K-chunk boxes (stages of 128 of K) for 128 x 128 tiles when both
  // operands are K-major and K is a multiple of 64, from K = 1024 on
  // (shorter K loops fill and drain the 3-stage ring too often: 6-8 % slower
  // at K = 512).  The CTA pair takes 128-deep stages of plain 64-deep boxes
  // from K = 1024 on (1-2 % faster than K-chunk boxes from K = 2048 on, even
  // at K = 1024, and 5-17 % faster than 64-deep stages at 8192^3 with an
  // M-major A), unless a K-major operand's rows are not 128-byte aligned
  // (3-5 % slower there than 64-deep stages).
  const bool ko = kind == 1 && bn <= 128 && a_major == GEMM_TN_MAJOR_K &&
                  b_major == GEMM_TN_MAJOR_K && K % 64 == 0 && K >= 1024;
  // The pair's 128-deep stages from K = 1024 on, also when a K-major
  // operand's rows are off the 128-byte grid (ragged 4000 x 3000 x 2500 with
  // B's ld 2504: 43.8 against 48.4 us back to back, 53.3 against 55.2 us
  // alone after an L2 flush; equal within noise on 8192^3 and 4096 x 3072 x
  // 2560 with off-grid rows).
  const bool deep_auto = K >= 1024;
  const bool deep = ko || (pair && (o.k_stage ? o.k_stage == 128 : deep_auto));
  CUtensorMap tmA, tmB;
  int s;
  if (ko) {
    s = encode_operand_ko(&tmA, q.A, M, K, q.ldA, q.sA, q.L, 128);
    if (s == GEMM_TN_OK)
      s = encode_operand_ko(&tmB, q.B, N, K, q.ldB, q.sB, q.L, static_cast<uint32_t>(bn));
  } else {
    s = encode_operand_batched(&tmA, q.A, M, K, q.ldA, q.sA, q.L, a_major, wide ? 256 : kLargeBM);
    if (s == GEMM_TN_OK)
      s = encode_operand_batched(&tmB, q.B, N, K, q.ldB, q.sB, q.L, b_major,
                                 static_cast<uint32_t>(pair ? bn / 2 : bn));
  }
  if (s != GEMM_TN_OK) return s;
  LargeArgs p;
  std::memset(&p, 0, sizeof p);
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.e = epi_of(q);
  p.acc_f16 = accum == GEMM_TN_ACC_F16;
  p.a_mn = a_major;
  p.b_mn = b_major;
  p.bn = bn;
  p.tiles_m = static_cast<int>((M + bm - 1) / bm);
  p.tiles_n = static_cast<int>((N + bn - 1) / bn);
  const int64_t per_batch = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
  if (per_batch * q.L > 0x7FFFFFFF) return GEMM_TN_ERR_UNSUPPORTED;
  p.batch = static_cast<int>(q.L);
  p.tiles_per_batch = static_cast<int>(per_batch);
  p.a_batched = q.L > 1 && q.sA != 0;
  p.b_batched = q.L > 1 && q.sB != 0;
  p.num_tiles = static_cast<int>(per_batch * q.L);
  // K blocks of the kernel's stage depth: 128 with K-chunk boxes or the
  // pair's deep stages, else 64
  const int64_t bk = deep ? 128 : kLargeBK;
  p.k_blocks = static_cast<int>((K + bk - 1) / bk);
  const int64_t kb64 = (K + kLargeBK - 1) / kLargeBK;
  p.group_m = (pair || wide) ? 8 : 16;
  p.timeout_ns = o.timeout_ns ? o.timeout_ns : kDefaultTimeoutNs;
  p.test_stall = o.test_stall;
  p.trace = trace_for(o, st, stream);
  p.sk_tile0 = p.num_tiles;  // no split tiles unless stream-K is set up below
  p.ks_splits = 1;           // no K split of the 128-row kernel unless set up below
  p.ks_kb_per = p.k_blocks;
  void* sk_ws = nullptr;
  CUtensorMap tmD;
  s = encode_d(&tmD, q.D, M, N, q.ldD, q.sD, q.L);
  if (s != GEMM_TN_OK) return s;
  if (wide) {
    int grid = std::min(p.num_tiles, st.num_sms);
    // Stream-K for the last, partial wave, on request only (fp32
    // accumulation only: a split fp16 accumulation would round at different
    // places).
    const int G = st.num_sms;
    const int full = p.num_tiles / G, rem = p.num_tiles - full * G;
    const int64_t units = static_cast<int64_t>(rem) * p.k_blocks;
    const int64_t per = (units + G - 1) / G;
    const bool want = !p.acc_f16 && rem > 0 && p.k_blocks >= 2 &&
                      per * (G + 1) < (int64_t{1} << 31) && o.stream_k == 1;
    if (want) {
      const int max_segs = static_cast<int>(per / p.k_blocks + 2);
      const size_t part_bytes = static_cast<size_t>(G) * max_segs * kWideBM * kWideBN * 4;
      const size_t cnt_bytes = static_cast<size_t>(rem) * 8 * sizeof(int);
      if (ws_alloc(&sk_ws, part_bytes + cnt_bytes, st, stream, o) == cudaSuccess) {
        int* counters = reinterpret_cast<int*>(static_cast<char*>(sk_ws) + part_bytes);
        if (cudaMemsetAsync(counters, 0, cnt_bytes, stream) == cudaSuccess) {
          p.sk_tile0 = full * G;
          p.sk_units = static_cast<int>(units);
          p.sk_per = static_cast<int>(per);
          p.sk_max_segs = max_segs;
          p.sk_partials = static_cast<float*>(sk_ws);
          p.sk_counters = counters;
          grid = G;
        } else {
          cudaGetLastError();
          cudaFreeAsync(sk_ws, stream);
          sk_ws = nullptr;
        }
      } else {
        cudaGetLastError();  // no workspace: run unsplit
        sk_ws = nullptr;
      }
    }
    const cudaError_t le = launch_pdl(gemm_tn_wide_kernel, dim3(grid), dim3(kWideThreads),
                                      WideSmem::kDynamicBytes, stream, tmA, tmB, tmD, p);
    if (sk_ws) cudaFreeAsync(sk_ws, stream);
    if (le != cudaSuccess) {
      cudaGetLastError();
      return GEMM_TN_ERR_CUDA;
    }
  } else if (pair) {
    // K split of the pair tiles (fp32 accumulation only): on request
    // (split_k with tile_kernel 2), or chosen by pair_split_count when the
    // kernel was chosen automatically.  Each unit stores its CTAs' fp32 partial
    // rows as two 128-row tiles; gemm_tn_tile_reduce_kernel adds the splits
    // in order and applies the epilogue.
    // A split the caller asked for fails with GEMM_TN_ERR_NO_MEMORY when its
    // workspace cannot be had; one the library chose by itself falls back
    // to the unsplit kernel.
    int splits = 1;
    const bool asked = !p.acc_f16 && o.tile_kernel == 2 && o.split_k > 0;
    if (asked)
      splits = o.split_k;
    else
      splits = auto_pair_splits;  // counted on 256-wide tiles (bn is 256 when > 1)
    splits = std::max(1, std::min(splits, p.k_blocks));
    void* ks_ws = nullptr;
    if (splits > 1) {
      const int kb_per = (p.k_blocks + splits - 1) / splits;
      const int nsplit = (p.k_blocks + kb_per - 1) / kb_per;  // no empty split
      const size_t bytes = static_cast<size_t>(p.num_tiles) * 2 * nsplit * kLargeBM * kPairBN * 4;
      if (static_cast<int64_t>(p.num_tiles) * 2 * nsplit > 0x7FFFFFFF ||
          ws_alloc(&ks_ws, bytes, st, stream, o) != cudaSuccess) {
        cudaGetLastError();
        ks_ws = nullptr;
        if (asked) return GEMM_TN_ERR_NO_MEMORY;
      } else {
        p.ks_kb_per = kb_per;
        p.ks_splits = nsplit;
        p.ks_ws = static_cast<float*>(ks_ws);
      }
    } else {
      // The last, partial wave of 256-wide tiles split along K over the
      // pairs the whole tiles leave idle: after `full` rounds of whole tiles
      // the rem tiles left run as s splits each in one more round, which
      // then takes 1/s of a tile's time (s <= 4 and at least 8 K blocks per
      // split).  fp32 accumulation; off with stream_k = -1; dropped when
      // the pool cannot serve the partial sums.
      const int P = st.max_pairs;
      const int full = P > 0 ? p.num_tiles / P : 0;
      const int rem = p.num_tiles - full * P;
      int s = last_wave_splits(p.num_tiles, P, p.k_blocks);
      if (!p.acc_f16 && bn == 256 && o.split_k == 0 && o.stream_k != -1 && s >= 2) {
        const int kb_per = (p.k_blocks + s - 1) / s;
        s = (p.k_blocks + kb_per - 1) / kb_per;
        const size_t bytes = static_cast<size_t>(rem) * 2 * s * kLargeBM * kPairBN * 4;
        if (ws_alloc(&ks_ws, bytes, st, stream, o) == cudaSuccess) {
          p.ks_tile0 = full * P;
          p.ks_kb_per = kb_per;
          p.ks_splits = s;
          p.ks_ws = static_cast<float*>(ks_ws);
        } else {
          cudaGetLastError();
          ks_ws = nullptr;
        }
      }
    }
    const int64_t units = p.ks_splits > 1
                              ? p.ks_tile0 + static_cast<int64_t>(p.num_tiles - p.ks_tile0) * p.ks_splits
                              : p.num_tiles;
    const int pairs = static_cast<int>(std::min<int64_t>(units, st.max_pairs));
    cudaError_t le =
        deep ? launch_pdl(gemm_tn_large2_kernel<true>, dim3(2 * pairs), dim3(kPairThreads),
                          PairSmem<true>::kDynamicBytes, stream, tmA, tmB, tmD, p)
             : launch_pdl(gemm_tn_large2_kernel<false>, dim3(2 * pairs), dim3(kPairThreads),
                          PairSmem<false>::kDynamicBytes, stream, tmA, tmB, tmD, p);
    if (ks_ws) {
      if (le == cudaSuccess) {
        // The reduction sees pair tile t as 128-row tiles 2t and 2t+1: twice
        // the row tiles and twice the raster group, which keeps that
        // numbering (tile_coords maps 2t + r to rows 2 tm + r of column tn).
        LargeArgs pr = p;
        pr.tiles_m = 2 * p.tiles_m;
        pr.group_m = 2 * p.group_m;
        pr.tiles_per_batch = 2 * p.tiles_per_batch;
        pr.num_tiles = 2 * p.num_tiles;
        pr.ks_tile0 = 2 * p.ks_tile0;  // split pair tiles only
        const dim3 rgrid(static_cast<unsigned>(4 * (kPairBN / 64)),
                         static_cast<unsigned>(2 * (p.num_tiles - p.ks_tile0)));
        le = launch_pdl(gemm_tn_tile_reduce_kernel<kPairBN>, rgrid, dim3(kTileReduceThreads), 0,
                        stream, pr);
      }
      const cudaError_t f = cudaFreeAsync(ks_ws, stream);
      if (le != cudaSuccess || f != cudaSuccess) {
        cudaGetLastError();
        return GEMM_TN_ERR_CUDA;
      }
      t_last_launches = 2;
      t_last_kernels = deep ? "gemm_tn_large2_kernel<deep>+gemm_tn_tile_reduce_kernel"
                            : "gemm_tn_large2_kernel+gemm_tn_tile_reduce_kernel";
      return GEMM_TN_OK;
    }
    if (le != cudaSuccess) {
      cudaGetLastError();
      return GEMM_TN_ERR_CUDA;
    }
  } else {
    // K split over several CTAs per tile (fp32 accumulation only: a split
    // fp16 accumulation would round at different places): on request
    // (split_k with tile_kernel 1), or automatically when the kernel was
    // chosen automatically, its tiles leave more than half the SMs idle and
    // K is long enough (>= 2048, >= 512 per split) to pay for the partials
    // and the reduction.
    // As for the pair kernel: a requested split needs its workspace, an
    // automatic one falls back to the unsplit kernel without it.
    int splits = 1;
    const bool asked = !p.acc_f16 && o.tile_kernel == 1 && o.split_k > 0;
    if (!p.acc_f16) {
      if (asked)
        splits = o.split_k;
      else if (o.tile_kernel == 0 && o.split_k == 0 && 2 * p.num_tiles <= st.num_sms &&
               kb64 >= 32)
        splits = static_cast<int>(std::min<int64_t>(st.num_sms / p.num_tiles, kb64 / 8));
      splits = std::max(1, std::min(splits, p.k_blocks));
    }
    void* ks_ws = nullptr;
    if (splits > 1) {
      const int kb_per = (p.k_blocks + splits - 1) / splits;
      const int nsplit = (p.k_blocks + kb_per - 1) / kb_per;  // no empty split
      const size_t bytes = static_cast<size_t>(p.num_tiles) * nsplit * kLargeBM * bn * 4;
      if (static_cast<int64_t>(p.num_tiles) * nsplit > 0x7FFFFFFF ||
          ws_alloc(&ks_ws, bytes, st, stream, o) != cudaSuccess) {
        cudaGetLastError();
        ks_ws = nullptr;
        if (asked) return GEMM_TN_ERR_NO_MEMORY;
      } else {
        p.ks_kb_per = kb_per;
        p.ks_splits = nsplit;
        p.ks_ws = static_cast<float*>(ks_ws);
      }
    }
    const int grid = static_cast<int>(
        std::min<int64_t>(static_cast<int64_t>(p.num_tiles) * p.ks_splits, st.num_sms));
    cudaError_t le;
    if (bn == 256)
      le = launch_pdl(gemm_tn_large_kernel<256>, dim3(grid), dim3(kLargeThreads),
                      LargeSmem<256>::kDynamicBytes, stream, tmA, tmB, tmD, p);
    else if (bn == 128 && ko)
      le = launch_pdl(gemm_tn_large_kernel<128, true>, dim3(grid), dim3(kLargeThreads),
                      LargeSmem<128, true>::kDynamicBytes, stream, tmA, tmB, tmD, p);
    else if (bn == 128)
      le = launch_pdl(gemm_tn_large_kernel<128>, dim3(grid), dim3(kLargeThreads),
                      LargeSmem<128>::kDynamicBytes, stream, tmA, tmB, tmD, p);
    else if (ko)
      le = launch_pdl(gemm_tn_large_kernel<64, true>, dim3(grid), dim3(kLargeThreads),
                      LargeSmem<64, true>::kDynamicBytes, stream, tmA, tmB, tmD, p);
    else
      le = launch_pdl(gemm_tn_large_kernel<64>, dim3(grid), dim3(kLargeThreads),
                      LargeSmem<64>::kDynamicBytes, stream, tmA, tmB, tmD, p);
    if (le != cudaSuccess && !ks_ws) {
      cudaGetLastError();
      return GEMM_TN_ERR_CUDA;
    }
    if (ks_ws) {
      cudaError_t e = le;
      if (e == cudaSuccess) {
        // the reduction: resident early, it waits in griddepcontrol.wait for
        // the split kernel's partials
        const dim3 rgrid(static_cast<unsigned>(4 * (bn / 64)), static_cast<unsigned>(p.num_tiles));
        e = bn == 256   ? launch_pdl(gemm_tn_tile_reduce_kernel<256>, rgrid,
                                     dim3(kTileReduceThreads), 0, stream, p)
            : bn == 128 ? launch_pdl(gemm_tn_tile_reduce_kernel<128>, rgrid,
                                     dim3(kTileReduceThreads), 0, stream, p)
                        : launch_pdl(gemm_tn_tile_reduce_kernel<64>, rgrid,
                                     dim3(kTileReduceThreads), 0, stream, p);
      }
      const cudaError_t f = cudaFreeAsync(ks_ws, stream);
      if (e != cudaSuccess || f != cudaSuccess) {
        cudaGetLastError();
        return GEMM_TN_ERR_CUDA;
      }
      t_last_launches = 2;
      t_last_kernels = bn == 256   ? "gemm_tn_large_kernel<256>+gemm_tn_tile_reduce_kernel"
                       : bn == 128 ? "gemm_tn_large_kernel<128>+gemm_tn_tile_reduce_kernel"
                                   : "gemm_tn_large_kernel<64>+gemm_tn_tile_reduce_kernel";
      return GEMM_TN_OK;
    }
  }
  if (cudaGetLastError() != cudaSuccess) return GEMM_TN_ERR_CUDA;
  t_last_launches = sk_ws ? 2 : 1;  // the counters' memset counts as a launch
  t_last_kernels = wide ? (sk_ws ? "memset+gemm_tn_wide_kernel" : "gemm_tn_wide_kernel")
                 : pair ? (deep ? "gemm_tn_large2_kernel<deep>" : "gemm_tn_large2_kernel")
                        : (bn == 256   ? "gemm_tn_large_kernel<256>"
                           : bn == 128 ? "gemm_tn_large_kernel<128>"
                                       : "gemm_tn_large_kernel<64>");
  return GEMM_TN_OK;
}

// Split-K kernel and its reduction for one MMA width MP.
template <int MP>
cudaError_t launch_skinny_mp(int grid, const CUtensorMap& tmA, const CUtensorMap& tmB,
                             const SkinnyArgs& p, const EpiArgs& ep, cudaStream_t stream) {
  cudaError_t e = launch_pdl(gemm_tn_skinny_kernel<skinny_stages(MP), MP>, dim3(grid),
                             dim3(kSkinnyThreads),
                             SkinnySmem<skinny_stages(MP), MP>::kDynamicBytes, stream, tmA, tmB,
                             p);
  if (e != cudaSuccess) return e;
  e = launch_pdl(gemm_tn_splitk_reduce_kernel<MP>, dim3(static_cast<unsigned>(p.tiles), MP / 16),
                 dim3(kReduceThreads), 0, stream, p, ep);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_skinny_kernels(int grid, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                  const SkinnyArgs& p, const EpiArgs& ep,
                                  cudaStream_t stream) {
  switch (p.mp) {
    case 16: return launch_skinny_mp<16>(grid, tmA, tmB, p, ep, stream);
    case 32: return launch_skinny_mp<32>(grid, tmA, tmB, p, ep, stream);
    case 48: return launch_skinny_mp<48>(grid, tmA, tmB, p, ep, stream);
    case 64: return launch_skinny_mp<64>(grid, tmA, tmB, p, ep, stream);
    case 96: return launch_skinny_mp<96>(grid, tmA, tmB, p, ep, stream);
    case 128: return launch_skinny_mp<128>(grid, tmA, tmB, p, ep, stream);
    case 192: return launch_skinny_mp<192>(grid, tmA, tmB, p, ep, stream);
    default: return launch_skinny_mp<256>(grid, tmA, tmB, p, ep, stream);
  }
}

// The cluster-reduced skinny kernel for MMA width MP: a cluster of p.cs CTAs
// per 128-row tile of B, a programmatic dependent launch.
template <int MP>
cudaError_t launch_skinny_cluster_mp(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                     const SkinnyClusterArgs& p, const EpiArgs& ep,
                                     cudaStream_t stream) {
  constexpr int S = cluster_stages(MP);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(p.cs);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>(p.tiles * p.cs));
  cfg.blockDim = dim3(kSkinnyThreads);
  cfg.dynamicSmemBytes = ClusterSmem<S, MP>::kDynamicBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_tn_skinny_cluster_kernel<S, MP>, tmA, tmB, p, ep);
}

cudaError_t launch_skinny_cluster(int mp, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                  const SkinnyClusterArgs& p, const EpiArgs& ep,
                                  cudaStream_t stream) {
  switch (mp) {
    case 16: return launch_skinny_cluster_mp<16>(tmA, tmB, p, ep, stream);
    case 32: return launch_skinny_cluster_mp<32>(tmA, tmB, p, ep, stream);
    case 48: return launch_skinny_cluster_mp<48>(tmA, tmB, p, ep, stream);
    case 64: return launch_skinny_cluster_mp<64>(tmA, tmB, p, ep, stream);
    case 96: return launch_skinny_cluster_mp<96>(tmA, tmB, p, ep, stream);
    case 128: return launch_skinny_cluster_mp<128>(tmA, tmB, p, ep, stream);
    case 192: return launch_skinny_cluster_mp<192>(tmA, tmB, p, ep, stream);
    default: return launch_skinny_cluster_mp<256>(tmA, tmB, p, ep, stream);
  }
}

// Cluster size of the cluster-reduced skinny kernel: the largest power of
// two up to 8 with tiles * cs within the SMs and at least one K block per
// split.  It is used for MMA widths up to 64 and at least two CTAs per tile
// (returns 0 otherwise: the contiguous split over one CTA per SM takes
// those).  Measured back to back (us, cluster / split): M=16, N=K=8192
// 24.5 / 26.4; 16 x 4096 x 16384 23.9 / 26.7; 64 x 8192^2 27.5 / 29.3.  One
// CTA per tile leaves SMs idle, and an SM streams B from HBM at only about
// 47 GB/s, so the split wins there (16 x 16384^2: 90 / 83; 32 x 16384 x
// 8192: 46.6 / 45.4); so it does at widths 128 and up, where more of each
// stage is MMA work (128 x 8192^2: 31.4 / 30.3; 256 x 8192^2 42.5 / 39.1).
int skinny_cluster_size(int M, int tiles, int k_blocks, const DeviceState& st) {
  if (skinny_mp(M) > 64 || tiles <= 0 || 2 * tiles > st.num_sms) return 0;
  int cs = 1;
  while (cs < kClusterMaxCs && tiles * cs * 2 <= st.num_sms && cs * 2 <= k_blocks) cs *= 2;
  return cs >= 2 ? cs : 0;
}

// The skinny path with the K split reduced in a cluster: one kernel, no
// workspace.
int launch_skinny_cluster_path(const Problem& q, int cs, cudaStream_t stream,
                               const gemm_tn_options& o, const DeviceState& st) {
  const int mp = skinny_mp(q.M);
  SkinnyClusterArgs p;
  std::memset(&p, 0, sizeof p);
  p.M = static_cast<int>(q.M);
  p.N = static_cast<int>(q.N);
  p.K = static_cast<int>(q.K);
  p.tiles = static_cast<int>((q.N + kSkinnyBN - 1) / kSkinnyBN);
  p.cs = cs;
  const int sub = cluster_sub(mp);
  p.k_blocks = static_cast<int>((q.K + kSkinnyBK * sub - 1) / (kSkinnyBK * sub));
  p.ko = q.K % 64 == 0 ? 1 : 0;
  p.timeout_ns = o.timeout_ns ? o.timeout_ns : kDefaultTimeoutNs;
  p.test_stall = o.test_stall;
  CUtensorMap tmA, tmB;
  int s;
  if (p.ko) {
    s = encode_operand_ko(&tmA, q.A, q.M, q.K, q.ldA, 0, 1, static_cast<uint32_t>(mp),
                          static_cast<uint32_t>(sub));
    if (s == GEMM_TN_OK)
      s = encode_operand_ko(&tmB, q.B, q.N, q.K, q.ldB, 0, 1, kSkinnyBN,
                            static_cast<uint32_t>(sub));
  } else {
    s = encode_operand(&tmA, q.A, q.M, q.K, q.ldA, 0, static_cast<uint32_t>(mp));
    if (s == GEMM_TN_OK) s = encode_operand(&tmB, q.B, q.N, q.K, q.ldB, 0, kSkinnyBN);
  }
  if (s != GEMM_TN_OK) return s;
  p.trace = trace_for(o, st, stream);
  if (launch_skinny_cluster(mp, tmA, tmB, p, epi_of(q), stream) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_TN_ERR_CUDA;
  }
  t_last_launches = 1;
  t_last_kernels = "gemm_tn_skinny_cluster_kernel";
  return GEMM_TN_OK;
}

int launch_skinny(const Problem& q, cudaStream_t stream, const gemm_tn_options& o,
                  const DeviceState& st) {
  // Without an explicit split count, the cluster-reduced kernel whenever one
  // wave of clusters covers the tiles.
  if (o.split_k == 0) {
    const int mp = skinny_mp(q.M), sub = cluster_sub(mp);
    const int tiles = static_cast<int>((q.N + kSkinnyBN - 1) / kSkinnyBN);
    const int k_blocks = static_cast<int>((q.K + kSkinnyBK * sub - 1) / (kSkinnyBK * sub));
    const int cs = skinny_cluster_size(static_cast<int>(q.M), tiles, k_blocks, st);
    if (cs > 0) return launch_skinny_cluster_path(q, cs, stream, o, st);
  }
  const int64_t M = q.M, N = q.N, K = q.K, ldA = q.ldA, ldB = q.ldB;
  const void *A = q.A, *B = q.B;
  SkinnyArgs p;
  std::memset(&p, 0, sizeof p);
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.mp = skinny_mp(M);
  p.tiles = static_cast<int>((N + kSkinnyBN - 1) / kSkinnyBN);
  p.k_blocks = static_cast<int>((K + kSkinnyBK * skinny_sub(p.mp) - 1) /
                                 (kSkinnyBK * skinny_sub(p.mp)));
  p.units = static_cast<int64_t>(p.tiles) * p.k_blocks;
  // Ranges of ceil(units / CTAs) units; a range spans at most per / k_blocks
  // + 2 tiles.  Recomputing the grid from per drops CTAs left without work.
  const int64_t want = std::min<int64_t>(o.split_k > 0 ? o.split_k : st.num_sms, p.units);
  const int64_t per = (p.units + want - 1) / want;
  const int grid = static_cast<int>((p.units + per - 1) / per);
  p.per = per;
  p.grid = grid;
  p.max_segs = static_cast<int>(per / p.k_blocks + 2);
  p.timeout_ns = o.timeout_ns ? o.timeout_ns : kDefaultTimeoutNs;
  p.test_stall = o.test_stall;

  const size_t need = static_cast<size_t>(grid) * p.max_segs * kSkinnyBN * p.mp * sizeof(float);

  CUtensorMap tmA, tmB;
  int s = encode_operand(&tmA, A, M, K, ldA, 0, static_cast<uint32_t>(p.mp));
  if (s == GEMM_TN_OK) s = encode_operand(&tmB, B, N, K, ldB, 0, kSkinnyBN);
  if (s != GEMM_TN_OK) return s;

  // Stream-ordered workspace: concurrent calls on different streams never
  // share it, and the pool keeps the memory for the next call.
  void* ws = nullptr;
  if (ws_alloc(&ws, need, st, stream, o) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_TN_ERR_NO_MEMORY;
  }
  p.ws = static_cast<float*>(ws);
  p.trace = trace_for(o, st, stream);
  const cudaError_t e = launch_skinny_kernels(grid, tmA, tmB, p, epi_of(q), stream);
  const cudaError_t f = cudaFreeAsync(ws, stream);
  if (e != cudaSuccess || f != cudaSuccess) {
    cudaGetLastError();
    return GEMM_TN_ERR_CUDA;
  }
  t_last_launches = 2;
  t_last_kernels = "gemm_tn_skinny_kernel+gemm_tn_splitk_reduce_kernel";
  return GEMM_TN_OK;
}

// D = beta * C (or zero) when the product term is absent.
int launch_scale(const Problem& q, cudaStream_t stream, const DeviceState& st) {
  const int64_t groups = (q.N + 7) / 8;
  const int64_t total = q.L * q.M * groups;
  const int64_t want = (total + kScaleThreads - 1) / kScaleThreads;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, 8LL * st.num_sms)));
  gemm_tn_scale_kernel<<<grid, kScaleThreads, 0, stream>>>(
      static_cast<int>(q.M), static_cast<int>(q.N), static_cast<int>(q.L), epi_of(q));
  if (cudaGetLastError() != cudaSuccess) return GEMM_TN_ERR_CUDA;
  t_last_launches = 1;
  t_last_kernels = "gemm_tn_scale_kernel";
  return GEMM_TN_OK;
}

// Tile widths any tile kernel can run (0 = the library's choice).
bool tile_n_ok(int n) {
  return n == 0 || n == 64 || n == 128 || n == 160 || n == 192 || n == 224 || n == 256;
}

bool options_ok(const gemm_tn_options& o) {
  return !(o.path < GEMM_TN_PATH_AUTO || o.path > GEMM_TN_PATH_SKINNY || o.split_k < 0 ||
           !tile_n_ok(o.tile_n) ||
           o.tile_kernel < 0 || (o.k_stage != 0 && o.k_stage != 64 && o.k_stage != 128) ||
           o.tile_kernel > 3);
}

int device_state(DeviceState*& st) {
  int dev = 0;
  // The current device of this host thread; cudaSetDevice makes its primary
  // context current here too, which the driver calls below (tensor-map
  // encoding) need on a thread that has not used CUDA yet.
  if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess)
    return GEMM_TN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  const int s = device_setup(dev, st);
  return s == GEMM_TN_OK ? pool_setup(dev, st) : s;
}

// Every entry point but the strided and allocation-free ones ends here.
int run_problem(const Problem& q, void* stream, const gemm_tn_options* opts) {
  t_last_launches = 0;
  t_last_kernels = "";
  gemm_tn_options o;
  std::memset(&o, 0, sizeof o);
  if (opts) o = *opts;
  if (!options_ok(o)) return GEMM_TN_ERR_INVALID_ARG;
  int s = validate(q);
  if (s != GEMM_TN_OK) return s;
  if (q.M == 0 || q.N == 0 || q.L == 0) return GEMM_TN_OK;
  // D = beta * C: nothing to do in place with beta == 1
  if (!q.use_ab() && q.beta == 1.f && q.in_place()) return GEMM_TN_OK;

  const int path = plan(q.M, q.N, q.K, q.a_major, q.b_major, q.accum, o.path, q.L);
  if (path < 0) return GEMM_TN_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  s = device_state(st);
  if (s != GEMM_TN_OK) return s;

  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (!q.use_ab())
    s = launch_scale(q, cs, *st);
  else if (path == GEMM_TN_PATH_SKINNY)
    s = launch_skinny(q, cs, o, *st);
  else
    s = launch_large(q, cs, o, *st);
  if (s != GEMM_TN_OK) return s;
  if (o.sync_check) return gemm_tn_check_device_error(stream, nullptr);
  return GEMM_TN_OK;
}

}  // namespace

extern "C" {

GEMM_TN_API int gemm_tn_check_device_error(void* stream, uint32_t* detail) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return GEMM_TN_ERR_CUDA;
  uint32_t word = 0, zero = 0;
  if (cudaMemcpyFromSymbolAsync(&word, gemm_tn_dev::g_error_word, sizeof word, 0,
                                cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GEMM_TN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GEMM_TN_ERR_CUDA;
  if (word != 0u) {
    if (cudaMemcpyToSymbolAsync(gemm_tn_dev::g_error_word, &zero, sizeof zero, 0,
                                cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return GEMM_TN_ERR_CUDA;
  }
  if (detail) *detail = word;
  return word ? GEMM_TN_ERR_DEVICE_TIMEOUT : GEMM_TN_OK;
}

GEMM_TN_API int gemm_tn_trace_read(void* stream, uint64_t* out, int max_ctas, int* recorded) {
  if (out == nullptr || max_ctas < 0) return GEMM_TN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return GEMM_TN_ERR_CUDA;
  const int n = std::min(max_ctas, kTraceCtas);
  if (n > 0 && (cudaMemcpyFromSymbolAsync(out, gemm_tn_dev::g_trace, sizeof(uint64_t) * kTraceSlots * n, 0,
                                          cudaMemcpyDeviceToHost, s) != cudaSuccess ||
                cudaStreamSynchronize(s) != cudaSuccess)) {
    cudaGetLastError();
    return GEMM_TN_ERR_CUDA;
  }
  if (recorded) {
    int r = 0;
    for (int c = 0; c < n; ++c) r += out[c * kTraceSlots + kTrEntry] != 0;
    *recorded = r;
  }
  return GEMM_TN_OK;
}

GEMM_TN_API int gemm_tn_ex(int64_t M, int64_t N, int64_t K, const void* A, int64_t ldA,
                           int a_major, const void* B, int64_t ldB, int b_major, void* CD,
                           int64_t ldC, int accum_dtype, void* stream,
                           const gemm_tn_options* opts) {
  return run_problem(
      in_place_problem(M, N, K, A, ldA, a_major, B, ldB, b_major, CD, ldC, accum_dtype), stream,
      opts);
}

GEMM_TN_API int gemm_tn_batched_ex(int64_t M, int64_t N, int64_t K, int64_t batch, float alpha,
                                   const void* A, int64_t ldA, int64_t strideA, int a_major,
                                   const void* B, int64_t ldB, int64_t strideB, int b_major,
                                   float beta, const void* C, int64_t ldC, int64_t strideC,
                                   void* D, int64_t ldD, int64_t strideD, int accum_dtype,
                                   void* stream, const gemm_tn_options* opts) {
  Problem q;
  std::memset(&q, 0, sizeof q);
  q.M = M; q.N = N; q.K = K; q.L = batch;
  q.alpha = alpha; q.beta = beta;
  q.A = A; q.ldA = ldA; q.sA = strideA; q.a_major = a_major;
  q.B = B; q.ldB = ldB; q.sB = strideB; q.b_major = b_major;
  q.C = C; q.ldC = ldC; q.sC = strideC;
  q.D = D; q.ldD = ldD; q.sD = strideD;
  q.accum = accum_dtype;
  return run_problem(q, stream, opts);
}

GEMM_TN_API int gemm_tn_batched(int64_t M, int64_t N, int64_t K, int64_t batch, float alpha,
                                const void* A, int64_t ldA, int64_t strideA, int a_major,
                                const void* B, int64_t ldB, int64_t strideB, int b_major,
                                float beta, const void* C, int64_t ldC, int64_t strideC, void* D,
                                int64_t ldD, int64_t strideD, int accum_dtype, void* stream) {
  return gemm_tn_batched_ex(M, N, K, batch, alpha, A, ldA, strideA, a_major, B, ldB, strideB,
                            b_major, beta, C, ldC, strideC, D, ldD, strideD, accum_dtype, stream,
                            nullptr);
}

GEMM_TN_API int gemm_tn_scaled(int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                               int64_t ldA, int a_major, const void* B, int64_t ldB, int b_major,
                               float beta, const void* C, int64_t ldC, void* D, int64_t ldD,
                               int accum_dtype, void* stream) {
  return gemm_tn_batched_ex(M, N, K, 1, alpha, A, ldA, 0, a_major, B, ldB, 0, b_major, beta, C,
                            ldC, 0, D, ldD, 0, accum_dtype, stream, nullptr);
}

GEMM_TN_API int gemm_tn(int64_t M, int64_t N, int64_t K, const void* A, int64_t ldA,
                        int a_major, const void* B, int64_t ldB, int b_major, void* CD,
                        int64_t ldC, int accum_dtype, void* stream) {
  return gemm_tn_ex(M, N, K, A, ldA, a_major, B, ldB, b_major, CD, ldC, accum_dtype, stream,
                    nullptr);
}

GEMM_TN_API int gemm_tn_plan_path(int64_t M, int64_t N, int64_t K, int a_major, int b_major) {
  return plan(M, N, K, a_major, b_major, GEMM_TN_ACC_F32, GEMM_TN_PATH_AUTO);
}

GEMM_TN_API int gemm_tn_last_launch_count(void) { return t_last_launches; }

GEMM_TN_API const char* gemm_tn_last_kernels(void) { return t_last_kernels; }

GEMM_TN_API const char* gemm_tn_status_string(int status) {
  switch (status) {
    case GEMM_TN_OK: return "GEMM_TN_OK";
    case GEMM_TN_ERR_INVALID_ARG: return "GEMM_TN_ERR_INVALID_ARG";
    case GEMM_TN_ERR_ALIGNMENT: return "GEMM_TN_ERR_ALIGNMENT";
    case GEMM_TN_ERR_UNSUPPORTED: return "GEMM_TN_ERR_UNSUPPORTED";
    case GEMM_TN_ERR_CUDA: return "GEMM_TN_ERR_CUDA";
    case GEMM_TN_ERR_DEVICE_TIMEOUT: return "GEMM_TN_ERR_DEVICE_TIMEOUT";
    case GEMM_TN_ERR_NO_MEMORY: return "GEMM_TN_ERR_NO_MEMORY";
    default: return "GEMM_TN_ERR_UNKNOWN";
  }
}

}  // extern "C"

// ---------------------------------------------------------------------------
// gemm_tn_skinny_noalloc: the skinny path with its partial sums in a fixed
// array compiled into the library, so that callers that cannot have device
// memory allocated for them (see the header) can still use it.  Nothing here
// calls cudaMalloc, cudaFree or any other allocating routine, and it does not
// create the workspace pool (device_setup only probes the device and sets
// kernel attributes; pool_setup is left to the other entry points).

static __device__ __align__(256) float
    g_noalloc_scratch[GEMM_TN_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {

// Device address of g_noalloc_scratch per device.  In host code the array's
// name is only a host-side stand-in, so the address is looked up once per
// device, with that device current, and passed to the kernels.
float* g_noalloc_ptr[kMaxDevices] = {};

int noalloc_scratch(int dev, float** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return GEMM_TN_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return GEMM_TN_OK;
}

}  // namespace

extern "C" GEMM_TN_API int gemm_tn_skinny_noalloc(int64_t M, int64_t N, int64_t K,
                                                  const void* A, int64_t ldA, int a_major,
                                                  const void* B, int64_t ldB, int b_major,
                                                  void* CD, int64_t ldC, int accum_dtype,
                                                  void* stream) {
  t_last_launches = 0;
  t_last_kernels = "";
  int s = validate(M, N, K, A, ldA, a_major, B, ldB, b_major, CD, ldC, accum_dtype);
  if (s != GEMM_TN_OK) return s;
  if (M > kNoallocMaxM || a_major != GEMM_TN_MAJOR_K || b_major != GEMM_TN_MAJOR_K ||
      accum_dtype != GEMM_TN_ACC_F32)
    return GEMM_TN_ERR_INVALID_ARG;
  if (M == 0 || N == 0 || K == 0) return GEMM_TN_OK;  // D = C: nothing to do

  int dev = 0;
  // The current device of this host thread; cudaSetDevice makes its primary
  // context current here too, which the driver calls below (tensor-map
  // encoding) need on a thread that has not used CUDA yet.
  if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess)
    return GEMM_TN_ERR_CUDA;
  DeviceState* st = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    s = device_setup(dev, st);
  }
  if (s != GEMM_TN_OK) return s;

  // Same split as the skinny path of gemm_tn: one CTA per SM.
  SkinnyArgs p;
  std::memset(&p, 0, sizeof p);
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.mp = skinny_mp(M);
  p.tiles = static_cast<int>((N + kSkinnyBN - 1) / kSkinnyBN);
  p.k_blocks = static_cast<int>((K + kSkinnyBK * skinny_sub(p.mp) - 1) /
                                 (kSkinnyBK * skinny_sub(p.mp)));
  p.units = static_cast<int64_t>(p.tiles) * p.k_blocks;
  const int64_t want = std::min<int64_t>(st->num_sms, p.units);
  const int64_t per = (p.units + want - 1) / want;
  const int grid = static_cast<int>((p.units + per - 1) / per);
  p.per = per;
  p.grid = grid;
  p.max_segs = static_cast<int>(per / p.k_blocks + 2);
  p.timeout_ns = kDefaultTimeoutNs;
  const uint64_t need =
      static_cast<uint64_t>(grid) * p.max_segs * kSkinnyBN * p.mp * sizeof(float);
  if (need > GEMM_TN_NOALLOC_SCRATCH_BYTES) return GEMM_TN_ERR_INVALID_ARG;

  s = noalloc_scratch(dev, &p.ws);
  if (s != GEMM_TN_OK) return s;

  CUtensorMap tmA, tmB;
  s = encode_operand(&tmA, A, M, K, ldA, 0, static_cast<uint32_t>(p.mp));
  if (s == GEMM_TN_OK) s = encode_operand(&tmB, B, N, K, ldB, 0, kSkinnyBN);
  if (s != GEMM_TN_OK) return s;

  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const EpiArgs ep =
      epi_of(in_place_problem(M, N, K, A, ldA, 0, B, ldB, 0, CD, ldC, GEMM_TN_ACC_F32));
  if (launch_skinny_kernels(grid, tmA, tmB, p, ep, cs) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_TN_ERR_CUDA;
  }
  t_last_launches = 2;
  t_last_kernels = "gemm_tn_skinny_kernel+gemm_tn_splitk_reduce_kernel";
  return GEMM_TN_OK;
}

// ---------------------------------------------------------------------------
// General element strides (copy-producer kernel).

namespace {

// Byte range touched by a (rows, cols) view with element strides (s_r, s_c).
void extent_strided(const void* p, int64_t rows, int64_t cols, int64_t s_r, int64_t s_c,
                    uintptr_t& lo, uintptr_t& hi) {
  lo = reinterpret_cast<uintptr_t>(p);
  hi = lo + static_cast<uintptr_t>(((rows - 1) * s_r + (cols - 1) * s_c + 1) * 2);
}

// Strides small enough that the view's byte extent stays inside 64-bit
// arithmetic (its last element at most 2^61 elements in).
bool strides_in_range(int64_t rows, int64_t cols, int64_t s_r, int64_t s_c) {
  const int64_t lim = int64_t{1} << 60;
  return (rows <= 1 || s_r <= lim / (rows - 1)) && (cols <= 1 || s_c <= lim / (cols - 1));
}

// No two coordinates of the (rows, cols) view share an element.
bool injective2(int64_t rows, int64_t cols, int64_t s_r, int64_t s_c) {
  if (rows <= 1 && cols <= 1) return true;
  if (rows <= 1) return s_c >= 1;
  if (cols <= 1) return s_r >= 1;
  if (s_r < 1 || s_c < 1) return false;
  return s_r >= s_c * cols || s_c >= s_r * rows;
}

}  // namespace

namespace {

cudaError_t repack2d(const void* src, int64_t s_sr, int64_t s_sc, void* dst, int64_t s_dr,
                     int64_t s_dc, int64_t rows, int64_t cols, cudaStream_t stream) {
  if (s_sc == 1 && s_dc == 1 && rows <= 65535) {
    const int64_t words = (cols + 7) / 8 + 1;  // 16-byte words a row can touch
    const int64_t span = static_cast<int64_t>(kRepackThreads) * kRowWords;
    const dim3 grid(static_cast<unsigned>(std::min<int64_t>((words + span - 1) / span, 64)),
                    static_cast<unsigned>(rows), 1);
    return launch_pdl(repack_rows_kernel, grid, dim3(kRepackThreads), 0, stream,
                      static_cast<const __half*>(src), s_sr, static_cast<__half*>(dst), s_dr,
                      static_cast<int>(rows), static_cast<int>(cols));
  }
  const dim3 grid(static_cast<unsigned>((cols + kRepackTile - 1) / kRepackTile),
                  static_cast<unsigned>((rows + kRepackTile - 1) / kRepackTile), 1);
  return launch_pdl(repack2d_kernel, grid, dim3(kRepackThreads), 0, stream,
                    static_cast<const __half*>(src), s_sr, s_sc, static_cast<__half*>(dst), s_dr,
                    s_dc, static_cast<int>(rows), static_cast<int>(cols));
}

int64_t round8(int64_t x) { return (x + 7) / 8 * 8; }
int64_t round64(int64_t x) { return (x + 63) / 64 * 64; }

// A (rows, K) view that TMA can read directly: (major, ld) or false.
bool tma_view(const void* p, int64_t rows, int64_t K, int64_t s_r, int64_t s_k, int& major,
              int64_t& ld) {
  if (reinterpret_cast<uintptr_t>(p) & 15u) return false;
  if (s_k == 1 && (rows == 1 || (s_r % 8 == 0 && s_r >= K))) {
    major = GEMM_TN_MAJOR_K;
    ld = rows == 1 ? round8(K) : s_r;
    return true;
  }
  if (s_r == 1 && (K == 1 || (s_k % 8 == 0 && s_k >= rows))) {
    major = GEMM_TN_MAJOR_MN;
    ld = K == 1 ? round8(rows) : s_k;
    return true;
  }
  return false;
}

// Tensor map of row class c (rows c, c + 8, ...) of a (rows, K) operand with
// a stride-1 K mode and row stride ld elements: base rounded down to 16
// bytes, the class's rows 16 * ld bytes apart, dims {K + delta, class rows},
// box {K block, tile rows / 8}, 128B swizzle.  Returns the byte offset of
// the rows in the map's rows (2 * delta) or -1.
int encode_row_class(CUtensorMap* map, const void* X, int64_t rows, int64_t K, int64_t ld, int c,
                     uint32_t box_rows) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(X) + 2 * static_cast<uintptr_t>(c) *
                                                          static_cast<uintptr_t>(ld);
  const uintptr_t base = a & ~static_cast<uintptr_t>(15);
  const int shift = static_cast<int>(a - base);
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K + shift / 2),
                        static_cast<cuuint64_t>((rows - c + 7) / 8)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 16};
  // one K block per box, 128B-swizzled as the MMA reads it (the producer
  // then shifts each row in place by the row's start within the box)
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kStrBK), box_rows}, estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, reinterpret_cast<void*>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? shift : -1;
}

int strided_copy_path(const StridedArgs& base, const DeviceState& st, cudaStream_t stream) {
  StridedArgs p = base;
  // The row-class TMA variant when both operands have a stride-1 K mode,
  // rows that do not overlap (ld >= K) and at least one row of every class
  // (M, N >= 8); otherwise every chunk is gathered by the producer threads.
  StridedMaps maps;
  std::memset(&maps, 0, sizeof maps);
  const int64_t kMaxLd = int64_t{1} << 35;  // class strides of 16 * ld bytes stay below 2^40
  bool tma = p.sAk == 1 && p.sBk == 1 && p.M >= 8 && p.N >= 8 && p.K >= 1 && p.sAm >= p.K &&
             p.sBn >= p.K && p.sAm < kMaxLd && p.sBn < kMaxLd;
  for (int c = 0; tma && c < 8; ++c) {
    const int sa = encode_row_class(&maps.a[c], p.A, p.M, p.K, p.sAm, c, str_bm<true>() / 8);
    const int sb = encode_row_class(&maps.b[c], p.B, p.N, p.K, p.sBn, c, kStrBN / 8);
    tma = sa >= 0 && sb >= 0;
    if (tma) {
      p.a_shifts |= static_cast<uint32_t>(sa) << (4 * c);
      p.b_shifts |= static_cast<uint32_t>(sb) << (4 * c);
    }
  }
  if (tma) {
    // 256 x 256 tiles in this variant
    p.tiles_m = (p.M + str_bm<true>() - 1) / str_bm<true>();
    p.num_tiles = p.tiles_m * p.tiles_n;
    const int grid = std::min(p.num_tiles, st.num_sms);
    gemm_tn_strided_kernel<true><<<grid, str_threads<true>(), StridedSmem<true>::kDynamicBytes,
                                   stream>>>(maps, p);
  } else {
    const int grid = std::min(p.num_tiles, st.num_sms);
    gemm_tn_strided_kernel<false><<<grid, kStrThreads, StridedSmem<false>::kDynamicBytes,
                                    stream>>>(maps, p);
  }
  if (cudaGetLastError() != cudaSuccess) return GEMM_TN_ERR_CUDA;
  t_last_launches = 1;
  t_last_kernels = tma ? "gemm_tn_strided_kernel<rows>" : "gemm_tn_strided_kernel";
  return GEMM_TN_OK;
}

// Repack the views TMA cannot read into row-major buffers from the stream's
// memory pool, run the tile kernels, scatter D back if needed.  Returns
// GEMM_TN_ERR_NO_MEMORY (nothing enqueued) when the pool cannot serve it.
int strided_repack_path(int64_t M, int64_t N, int64_t K, const void* A, int64_t sAm,
                        int64_t sAk, const void* B, int64_t sBn, int64_t sBk, void* CD,
                        int64_t sCm, int64_t sCn, int accum, const DeviceState& st,
                        cudaStream_t stream, const gemm_tn_options& caller) {
  int a_major = 0, b_major = 0, c_major = 0;
  int64_t ldA = 0, ldB = 0, ldC = 0;
  const bool a_direct = tma_view(A, M, K, sAm, sAk, a_major, ldA);
  const bool b_direct = tma_view(B, N, K, sBn, sBk, b_major, ldB);
  // C/D must be row-major for the tile kernels: (M,N):(ldC,1)
  const bool c_direct = tma_view(CD, M, N, sCm, sCn, c_major, ldC) && c_major == GEMM_TN_MAJOR_K;
  // repacked rows start on 128-byte boundaries (ld a multiple of 64
  // elements): TMA reads of unaligned rows fetch a fifth more sectors and
  // ran 17-21 % slower
  const int64_t Kp = round64(K), Np = round64(N);
  const size_t a_elems = a_direct ? 0 : static_cast<size_t>(M) * Kp;
  const size_t b_elems = b_direct ? 0 : static_cast<size_t>(N) * Kp;
  const size_t c_elems = c_direct ? 0 : static_cast<size_t>(M) * Np;
  const size_t total = (a_elems + b_elems + c_elems) * 2;
  void* ws = nullptr;
  if (total > 0 && ws_alloc(&ws, total, st, stream, caller) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_TN_ERR_NO_MEMORY;
  }
  __half* wa = static_cast<__half*>(ws);
  __half* wb = wa + a_elems;
  __half* wc = wb + b_elems;
  int launches = 0;
  cudaError_t e = cudaSuccess;
  const void* Ause = A;
  const void* Buse = B;
  void* Cuse = CD;
  if (!a_direct) {
    e = repack2d(A, sAm, sAk, wa, Kp, 1, M, K, stream);
    Ause = wa, a_major = GEMM_TN_MAJOR_K, ldA = Kp, ++launches;
  }
  if (e == cudaSuccess && !b_direct) {
    e = repack2d(B, sBn, sBk, wb, Kp, 1, N, K, stream);
    Buse = wb, b_major = GEMM_TN_MAJOR_K, ldB = Kp, ++launches;
  }
  if (e == cudaSuccess && !c_direct) {
    e = repack2d(CD, sCm, sCn, wc, Np, 1, M, N, stream);
    Cuse = wc, ldC = Np, ++launches;
  }
  int s = GEMM_TN_OK;
  const char* gemm_kernels = "";
  if (e == cudaSuccess) {
    gemm_tn_options o;
    std::memset(&o, 0, sizeof o);
    o.timeout_ns = caller.timeout_ns;
    o.test_fail_alloc = caller.test_fail_alloc;
    const int path = plan(M, N, K, a_major, b_major, accum, GEMM_TN_PATH_AUTO);
    const Problem q =
        in_place_problem(M, N, K, Ause, ldA, a_major, Buse, ldB, b_major, Cuse, ldC, accum);
    s = path == GEMM_TN_PATH_SKINNY ? launch_skinny(q, stream, o, st)
                                    : launch_large(q, stream, o, st);
    launches += t_last_launches;
    gemm_kernels = t_last_kernels;
  } else {
    s = GEMM_TN_ERR_CUDA;
  }
  if (s == GEMM_TN_OK && !c_direct) {
    e = repack2d(wc, Np, 1, CD, sCm, sCn, M, N, stream);
    if (e != cudaSuccess) s = GEMM_TN_ERR_CUDA;
    ++launches;
  }
  if (ws && cudaFreeAsync(ws, stream) != cudaSuccess && s == GEMM_TN_OK) s = GEMM_TN_ERR_CUDA;
  if (s != GEMM_TN_OK) {
    cudaGetLastError();
    t_last_launches = 0;
    t_last_kernels = "";
    return s;
  }
  t_last_launches = launches;
  // the repack kernels run around the tile kernel(s) named here
  static thread_local char names[160];
  std::snprintf(names, sizeof names, "%s%s", (a_direct && b_direct && c_direct) ? "" : "repack2d_kernel+",
                gemm_kernels);
  t_last_kernels = names;
  return GEMM_TN_OK;
}

}  // namespace

extern "C" GEMM_TN_API int gemm_tn_strided_ex(int64_t M, int64_t N, int64_t K, const void* A,
                                              int64_t sAm, int64_t sAk, const void* B,
                                              int64_t sBn, int64_t sBk, void* CD, int64_t sCm,
                                              int64_t sCn, int accum_dtype, void* stream,
                                              const gemm_tn_options* opts) {
  t_last_launches = 0;
  t_last_kernels = "";
  const int64_t kMax = 0x7FFFFFFF;
  const int route = opts ? opts->path : GEMM_TN_PATH_AUTO;
  if (route != GEMM_TN_PATH_AUTO && route != GEMM_TN_PATH_STRIDED_COPY &&
      route != GEMM_TN_PATH_STRIDED_REPACK)
    return GEMM_TN_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || M > kMax || N > kMax || K > kMax) return GEMM_TN_ERR_INVALID_ARG;
  if (sAm < 0 || sAk < 0 || sBn < 0 || sBk < 0 || sCm < 0 || sCn < 0)
    return GEMM_TN_ERR_INVALID_ARG;
  if (!strides_in_range(M, K, sAm, sAk) || !strides_in_range(N, K, sBn, sBk) ||
      !strides_in_range(M, N, sCm, sCn))
    return GEMM_TN_ERR_INVALID_ARG;
  if (accum_dtype != GEMM_TN_ACC_F32 && accum_dtype != GEMM_TN_ACC_F16)
    return GEMM_TN_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_TN_OK;
  if (CD == nullptr || !injective2(M, N, sCm, sCn)) return GEMM_TN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(CD) & 1u) return GEMM_TN_ERR_ALIGNMENT;
  if (K == 0) return GEMM_TN_OK;  // D = C
  if (A == nullptr || B == nullptr) return GEMM_TN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 1u)
    return GEMM_TN_ERR_ALIGNMENT;
  uintptr_t a0, a1, b0, b1, c0, c1;
  extent_strided(A, M, K, sAm, sAk, a0, a1);
  extent_strided(B, N, K, sBn, sBk, b0, b1);
  extent_strided(CD, M, N, sCm, sCn, c0, c1);
  if ((c0 < a1 && a0 < c1) || (c0 < b1 && b0 < c1)) return GEMM_TN_ERR_INVALID_ARG;

  int dev = 0;
  // The current device of this host thread; cudaSetDevice makes its primary
  // context current here too, which the driver calls below (tensor-map
  // encoding) need on a thread that has not used CUDA yet.
  if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess)
    return GEMM_TN_ERR_CUDA;
  DeviceState* st = nullptr;
  int s;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    s = device_setup(dev, st);
    if (s == GEMM_TN_OK) s = pool_setup(dev, st);
  }
  if (s != GEMM_TN_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);

  // Repacking costs two extra passes over the operands and an allocation;
  // below ~2^24 multiply-adds the copy-producer kernel is as fast.
  const bool big = static_cast<double>(M) * N * K >= 16777216.0;
  if (route == GEMM_TN_PATH_STRIDED_REPACK || (route == GEMM_TN_PATH_AUTO && big)) {
    gemm_tn_options o;
    std::memset(&o, 0, sizeof o);
    if (opts) o = *opts;
    s = strided_repack_path(M, N, K, A, sAm, sAk, B, sBn, sBk, CD, sCm, sCn, accum_dtype, *st,
                            cs, o);
    if (s != GEMM_TN_ERR_NO_MEMORY || route == GEMM_TN_PATH_STRIDED_REPACK) return s;
    // pool exhausted: the copy producer needs no workspace
  }

  StridedArgs p;
  std::memset(&p, 0, sizeof p);
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.A = static_cast<const __half*>(A);
  p.sAm = sAm;
  p.sAk = sAk;
  p.B = static_cast<const __half*>(B);
  p.sBn = sBn;
  p.sBk = sBk;
  p.CD = static_cast<__half*>(CD);
  p.sCm = sCm;
  p.sCn = sCn;
  p.acc_f16 = accum_dtype == GEMM_TN_ACC_F16;
  p.tiles_m = static_cast<int>((M + kStrBM - 1) / kStrBM);
  p.tiles_n = static_cast<int>((N + kStrBN - 1) / kStrBN);
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.k_blocks = static_cast<int>((K + kStrBK - 1) / kStrBK);
  p.group_m = 16;
  p.timeout_ns = (opts && opts->timeout_ns) ? opts->timeout_ns : kDefaultTimeoutNs;
  return strided_copy_path(p, *st, cs);
}

extern "C" GEMM_TN_API int gemm_tn_strided(int64_t M, int64_t N, int64_t K, const void* A,
                                           int64_t sAm, int64_t sAk, const void* B, int64_t sBn,
                                           int64_t sBk, void* CD, int64_t sCm, int64_t sCn,
                                           int accum_dtype, void* stream) {
  return gemm_tn_strided_ex(M, N, K, A, sAm, sAk, B, sBn, sBk, CD, sCm, sCn, accum_dtype, stream,
                            nullptr);
}

// ---------------------------------------------------------------------------
// Host-buffer entry point: B copied once, then panels of M rows of A and C
// copied in on a copy stream, each panel's GEMM on the caller's stream as
// soon as its rows have arrived, and its D rows copied out on a second copy
// stream, so that copies in both directions and the GEMMs overlap.

namespace {

constexpr int kHostMaxPanels = 64;
constexpr int kHostRing = 3;  // device slots for A and C/D panels

struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr;
  // Two device workspaces used by alternate calls, each with the event that
  // marks the end of its last call's use (recorded on that call's stream).
  // They are the pipeline's own (not the pool's): a pool block freed on one
  // stream and taken on the copy-in stream would make the copies wait for
  // the freeing call to finish, and consecutive calls could not overlap.
  void* ws[2] = {nullptr, nullptr};
  size_t ws_bytes[2] = {0, 0};
  cudaEvent_t ws_free[2] = {nullptr, nullptr};
  unsigned calls = 0;
  cudaEvent_t in_done[kHostMaxPanels];
  cudaEvent_t gemm_done[kHostMaxPanels];
  cudaEvent_t out_done[kHostMaxPanels];
};

std::mutex g_host_mu;  // held while a gemm_tn_host call enqueues (streams and events are shared)
HostPipe g_pipe[kMaxDevices];

// The device's copy streams and events, created on first use (under g_host_mu).
int host_pipe(int dev, HostPipe*& hp) {
  if (dev < 0 || dev >= kMaxDevices) return GEMM_TN_ERR_UNSUPPORTED;
  hp = &g_pipe[dev];
  if (hp->ready) return GEMM_TN_OK;
  bool ok = cudaStreamCreateWithFlags(&hp->in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&hp->out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&hp->start, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&hp->ws_free[0], cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&hp->ws_free[1], cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < kHostMaxPanels; ++i)
    ok = cudaEventCreateWithFlags(&hp->in_done[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&hp->gemm_done[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&hp->out_done[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return GEMM_TN_ERR_CUDA;  // (what was created stays for the next attempt to leak; rare)
  }
  hp->ready = true;
  return GEMM_TN_OK;
}

// Rows of M per panel: the caller's (rounded up to 8), else all of M up to
// 1024 rows, else ceil(M / 8) rounded up to 256 and at least 512; never more
// than kHostMaxPanels panels.
int64_t host_panel_rows(int64_t M, int requested) {
  int64_t P;
  if (requested > 0)
    P = (static_cast<int64_t>(requested) + 7) / 8 * 8;
  else if (M <= 1024)
    P = M;
  else
    P = std::max<int64_t>(512, ((M + 7) / 8 + 255) / 256 * 256);
  if ((M + P - 1) / P > kHostMaxPanels) P = ((M + kHostMaxPanels - 1) / kHostMaxPanels + 7) / 8 * 8;
  return std::max<int64_t>(P, 1);
}

// Row counts of the panels: P rows each; with the library's choice
// (tapered) the last P or fewer rows are cut into a half and two quarters
// (multiples of 8), so that the GEMM and copy-out left after the last
// copy-in are short.  Returns the number of panels.
int host_panels(int64_t M, int64_t P, bool tapered, int64_t (&rows)[kHostMaxPanels]) {
  int n = 0;
  int64_t left = M;
  while (left > P && n < kHostMaxPanels - 3) {
    rows[n++] = P;
    left -= P;
  }
  if (tapered && left >= 64 && left <= P) {
    const int64_t q = (left / 4 + 7) / 8 * 8;
    rows[n++] = left - 2 * q;
    rows[n++] = q;
    rows[n++] = q;
  } else {
    while (left > 0) {  // (only when more than kHostMaxPanels - 3 panels of P were cut)
      const int64_t r = std::min(left, P);
      rows[n++] = r;
      left -= r;
    }
  }
  return n;
}

// height rows of width elements: host (pitch spitch elements) -> device
// (pitch dpitch elements), or back.
cudaError_t copy2d(void* dst, int64_t dpitch, const void* src, int64_t spitch, int64_t width,
                   int64_t height, cudaMemcpyKind kind, cudaStream_t s) {
  if (width <= 0 || height <= 0) return cudaSuccess;
  if (height == 1 || (dpitch == width && spitch == width))  // one contiguous range
    return cudaMemcpyAsync(dst, src, static_cast<size_t>(width) * 2 * static_cast<size_t>(height),
                           kind, s);
  return cudaMemcpy2DAsync(dst, static_cast<size_t>(dpitch) * 2, src, static_cast<size_t>(spitch) * 2,
                           static_cast<size_t>(width) * 2, static_cast<size_t>(height), kind, s);
}

// Byte range of a host (rows, cols) view with row pitch ld.
void host_extent(const void* p, int64_t rows, int64_t cols, int64_t ld, uintptr_t& lo,
                 uintptr_t& hi) {
  lo = reinterpret_cast<uintptr_t>(p);
  hi = lo + static_cast<uintptr_t>(((rows - 1) * ld + cols) * 2);
}

}  // namespace

extern "C" GEMM_TN_API int gemm_tn_host(int64_t M, int64_t N, int64_t K, float alpha,
                                        const void* A, int64_t ldA, int a_major, const void* B,
                                        int64_t ldB, int b_major, float beta, const void* C,
                                        int64_t ldC, void* D, int64_t ldD, int accum_dtype,
                                        void* stream, const gemm_tn_options* opts) {
  t_last_launches = 0;
  t_last_kernels = "";
  gemm_tn_options o;
  std::memset(&o, 0, sizeof o);
  if (opts) o = *opts;
  if (!options_ok(o) || o.host_panel_rows < 0) return GEMM_TN_ERR_INVALID_ARG;
  const int64_t kMax = 0x7FFFFFFF;
  if (M < 0 || N < 0 || K < 0 || M > kMax || N > kMax || K > kMax) return GEMM_TN_ERR_INVALID_ARG;
  if ((a_major != GEMM_TN_MAJOR_K && a_major != GEMM_TN_MAJOR_MN) ||
      (b_major != GEMM_TN_MAJOR_K && b_major != GEMM_TN_MAJOR_MN) ||
      (accum_dtype != GEMM_TN_ACC_F32 && accum_dtype != GEMM_TN_ACC_F16))
    return GEMM_TN_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_TN_OK;
  const bool use_ab = alpha != 0.f && K > 0;
  const bool read_c = beta != 0.f;
  // A (M,K) and B (N,K) rows of their stride-1 mode, C and D rows of N
  const int64_t a_rows = a_major == GEMM_TN_MAJOR_K ? M : K, a_cols = a_major == GEMM_TN_MAJOR_K ? K : M;
  const int64_t b_rows = b_major == GEMM_TN_MAJOR_K ? N : K, b_cols = b_major == GEMM_TN_MAJOR_K ? K : N;
  if (D == nullptr || ldD < N || (read_c && (C == nullptr || ldC < N))) return GEMM_TN_ERR_INVALID_ARG;
  if (use_ab && (A == nullptr || B == nullptr || ldA < a_cols || ldB < b_cols))
    return GEMM_TN_ERR_INVALID_ARG;
  uintptr_t d0, d1;
  host_extent(D, M, N, ldD, d0, d1);
  if (read_c && C != D) {
    uintptr_t c0, c1;
    host_extent(C, M, N, ldC, c0, c1);
    if (overlap(c0, c1, d0, d1)) return GEMM_TN_ERR_INVALID_ARG;
  }
  if (read_c && C == D && ldC != ldD) return GEMM_TN_ERR_INVALID_ARG;
  if (use_ab) {
    uintptr_t a0, a1, b0, b1;
    host_extent(A, a_rows, a_cols, ldA, a0, a1);
    host_extent(B, b_rows, b_cols, ldB, b0, b1);
    if (overlap(a0, a1, d0, d1) || overlap(b0, b1, d0, d1)) return GEMM_TN_ERR_INVALID_ARG;
  }

  DeviceState* st = nullptr;
  int s = device_state(st);
  if (s != GEMM_TN_OK) return s;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_TN_ERR_CUDA;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);

  const int64_t P = host_panel_rows(M, o.host_panel_rows);
  int64_t prow[kHostMaxPanels];
  // (tapered only for calls that do not overlap their neighbours: with
  // host_inputs_ready the next call's copies fill the tail instead, and the
  // extra copies of the small panels cost more than they save)
  const int panels =
      host_panels(M, P, o.host_panel_rows == 0 && M > 1024 && o.host_inputs_ready == 0, prow);
  const int ring = std::min(kHostRing, panels);
  const int64_t Kp = round64(std::max<int64_t>(K, 1)), Np = round64(N), Pp = round64(P);
  // device layouts: B and A panels keep their major (rows on 128-byte
  // boundaries), C/D panels are row-major with ld Np
  const size_t b_elems = use_ab ? static_cast<size_t>(b_major == GEMM_TN_MAJOR_K ? N * Kp : K * Np) : 0;
  const size_t a_slot = use_ab ? static_cast<size_t>(a_major == GEMM_TN_MAJOR_K ? P * Kp : K * Pp) : 0;
  const size_t c_slot = static_cast<size_t>(P * Np);
  const size_t bytes = 2 * (b_elems + ring * (a_slot + c_slot));

  std::lock_guard<std::mutex> lk(g_host_mu);
  HostPipe* hp = nullptr;
  s = host_pipe(dev, hp);
  if (s != GEMM_TN_OK) return s;
  // With host_inputs_ready the copies in wait only for the copies in of
  // earlier calls (the copy-in stream is FIFO) and for the end of the call
  // before last, which used the same workspace, so that a call's copies in
  // overlap the previous call's last GEMMs and copies out.
  // Under stream capture the workspace comes from the pool in `stream`'s
  // order instead (a graph memory node), and the copies in follow `stream`.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(cs, &cap) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_TN_ERR_CUDA;
  }
  const bool captured = cap != cudaStreamCaptureStatusNone;
  const bool eager = o.host_inputs_ready != 0 && !captured;
  const int wsi = static_cast<int>(hp->calls & 1u);
  void* ws = nullptr;
  if (captured) {
    if (ws_alloc(&ws, bytes, *st, cs, o) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_TN_ERR_NO_MEMORY;
    }
  } else {
    if (o.test_fail_alloc) return GEMM_TN_ERR_NO_MEMORY;
    if (hp->ws_bytes[0] < bytes) {
      // grow both workspaces once their last calls are done with them (a
      // host wait; only when a call needs more than any earlier one)
      for (int j = 0; j < 2; ++j) {
        if (hp->ws[j] != nullptr &&
            (cudaEventSynchronize(hp->ws_free[j]) != cudaSuccess || cudaFree(hp->ws[j]) != cudaSuccess)) {
          cudaGetLastError();
          return GEMM_TN_ERR_CUDA;
        }
        hp->ws[j] = nullptr;
        hp->ws_bytes[j] = 0;
      }
      for (int j = 0; j < 2; ++j) {
        if (cudaMalloc(&hp->ws[j], bytes) != cudaSuccess) {
          cudaGetLastError();
          for (int i = 0; i < 2; ++i) {
            if (hp->ws[i]) cudaFree(hp->ws[i]);
            hp->ws[i] = nullptr;
            hp->ws_bytes[i] = 0;
          }
          return GEMM_TN_ERR_NO_MEMORY;
        }
        hp->ws_bytes[j] = bytes;
      }
    }
    ++hp->calls;
    ws = hp->ws[wsi];
    if (cudaStreamWaitEvent(hp->in, hp->ws_free[wsi], 0) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_TN_ERR_CUDA;
    }
  }
  __half* wB = static_cast<__half*>(ws);
  __half* wA = wB + b_elems;
  __half* wC = wA + ring * a_slot;
  const __half* hA = static_cast<const __half*>(A);
  const __half* hC = static_cast<const __half*>(C);
  __half* hD = static_cast<__half*>(D);

  gemm_tn_options og = o;
  og.sync_check = 0;
  og.host_panel_rows = 0;
  og.host_inputs_ready = 0;
  int launches = 0;
  const char* kernels = "";
  int last_in = -1, last_out = -1;  // last recorded events of the copy streams
  auto done = [&](int status) {
    // join the copy streams back into `stream` and release the workspace
    cudaEventRecord(hp->start, hp->in);
    cudaStreamWaitEvent(cs, hp->start, 0);
    if (last_out >= 0) cudaStreamWaitEvent(cs, hp->out_done[last_out], 0);
    // the workspace is free again once `stream` has passed this point
    const cudaError_t e = captured ? cudaFreeAsync(ws, cs) : cudaEventRecord(hp->ws_free[wsi], cs);
    if (e != cudaSuccess && status == GEMM_TN_OK) status = GEMM_TN_ERR_CUDA;
    if (status != GEMM_TN_OK) cudaGetLastError();
    return status;
  };
  // D is written only after everything enqueued on `stream` before the call
  // (which may still read it); A, B and C are read after it too unless the
  // caller declared them ready
  if (cudaEventRecord(hp->start, cs) != cudaSuccess ||
      (!eager && cudaStreamWaitEvent(hp->in, hp->start, 0) != cudaSuccess) ||
      cudaStreamWaitEvent(hp->out, hp->start, 0) != cudaSuccess)
    return done(GEMM_TN_ERR_CUDA);
  if (use_ab && copy2d(wB, b_major == GEMM_TN_MAJOR_K ? Kp : Np, B, ldB, b_cols, b_rows,
                       cudaMemcpyHostToDevice, hp->in) != cudaSuccess)
    return done(GEMM_TN_ERR_CUDA);
  int64_t m0 = 0;
  for (int i = 0; i < panels; m0 += prow[i], ++i) {
    const int64_t rows = prow[i];
    const int slot = i % ring;
    __half* a_i = wA + slot * a_slot;
    __half* c_i = wC + slot * c_slot;
    // the slot's previous panel has been copied out (so its GEMM is done too)
    if (i >= ring && cudaStreamWaitEvent(hp->in, hp->out_done[i - ring], 0) != cudaSuccess)
      return done(GEMM_TN_ERR_CUDA);
    cudaError_t e = cudaSuccess;
    if (use_ab)
      e = a_major == GEMM_TN_MAJOR_K
              ? copy2d(a_i, Kp, hA + m0 * ldA, ldA, K, rows, cudaMemcpyHostToDevice, hp->in)
              : copy2d(a_i, Pp, hA + m0, ldA, rows, K, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess && read_c)
      e = copy2d(c_i, Np, hC + m0 * ldC, ldC, N, rows, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess) e = cudaEventRecord(hp->in_done[i], hp->in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, hp->in_done[i], 0);
    if (e != cudaSuccess) return done(GEMM_TN_ERR_CUDA);
    last_in = i;
    Problem q;
    std::memset(&q, 0, sizeof q);
    q.M = rows; q.N = N; q.K = K; q.L = 1;
    q.alpha = alpha; q.beta = beta;
    q.A = a_i; q.ldA = a_major == GEMM_TN_MAJOR_K ? Kp : Pp; q.a_major = a_major;
    q.B = wB; q.ldB = b_major == GEMM_TN_MAJOR_K ? Kp : Np; q.b_major = b_major;
    q.C = c_i; q.ldC = Np;
    q.D = c_i; q.ldD = Np;
    q.accum = accum_dtype;
    s = run_problem(q, cs, &og);
    if (s != GEMM_TN_OK) return done(s);
    launches += t_last_launches;
    if (i == 0) kernels = t_last_kernels;
    e = cudaEventRecord(hp->gemm_done[i], cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->gemm_done[i], 0);
    if (e == cudaSuccess)
      e = copy2d(hD + m0 * ldD, ldD, c_i, Np, N, rows, cudaMemcpyDeviceToHost, hp->out);
    if (e == cudaSuccess) e = cudaEventRecord(hp->out_done[i], hp->out);
    if (e != cudaSuccess) return done(GEMM_TN_ERR_CUDA);
    last_out = i;
  }
  (void)last_in;
  s = done(GEMM_TN_OK);
  if (s != GEMM_TN_OK) return s;
  t_last_launches = launches;
  t_last_kernels = kernels;
  if (o.sync_check) return gemm_tn_check_device_error(stream, nullptr);
  return GEMM_TN_OK;
}
