// Spherical k-means assignment on the tensor cores: for every indexable key
// i of segment s, a(i) = argmax_j k_i . mu_j over the segment's centroids, the
// lowest j among equal maxima ("RetroInfer: A Vector Storage Engine for
// Scalable Long-Context LLM Inference", technical summary (es) §2.A.2
// spherical-k-means clustering index and §3 segmented clustering).
//
// The dot products of a 128-key tile with all (<= 512) centroids of its
// segment are one dense contraction (M = 128, N = k, K = 128) issued as
// tcgen05.mma kind::f16 (bf16 operands from shared memory, f32 accumulators in
// tensor memory: 512 columns hold the whole 128 x 512 tile).  Operands arrive
// by TMA with 128-byte swizzling.  The epilogue reads each thread's row back
// with tcgen05.ld and keeps a running argmax, so the dot-product matrix never
// leaves the SM.  Persistent CTAs walk a contiguous range of (segment, tile)
// work items; a segment's centroids are loaded once per CTA visit.
#include <cuda.h>

#include "wi_device.cuh"
#include "wi_internal.h"

namespace wi {

namespace {

constexpr int kTcThreads = 128;  // 4 warps: one TMEM lane quarter each
constexpr int kTileM = 128;
constexpr uint32_t kAHalf = 128u * 128u;   // 128 rows x 64 bf16 (one 128-byte swizzle span)
constexpr uint32_t kAStage = 2u * kAHalf;  // both K halves of a key tile: 32 KB
constexpr uint32_t kBHalf = 256u * 128u;   // 256 centroids x 64 bf16
constexpr uint32_t kBChunk = 2u * kBHalf;  // 256 centroids x 128: 64 KB
constexpr uint32_t kSmemB = 0;
constexpr uint32_t kSmemA = 2u * kBChunk;            // after up to 512 centroids
constexpr uint32_t kSmemBar = kSmemA + 2u * kAStage;  // two key-tile stages
constexpr uint32_t kSmemUsed = kSmemBar + 64u;
constexpr size_t kTcDynSmem = kSmemUsed + 1024u;  // slack to align the base to 1024 B
constexpr uint32_t kTmemCols = 512;

__global__ void __launch_bounds__(kTcThreads, 1)
    assign_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     BuildArgs a, int tiles_per_unit, int n_units, int n_chunks) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* sm = smem_raw + (base - raw);
  const uint32_t sB = base + kSmemB, sA = base + kSmemA;
  const uint32_t bar_a[2] = {base + kSmemBar, base + kSmemBar + 8};
  const uint32_t bar_b = base + kSmemBar + 16, bar_mma = base + kSmemBar + 24;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sm + kSmemBar + 32);
  volatile int* fail_flag = reinterpret_cast<volatile int*>(sm + kSmemBar + 40);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long total = (long long)n_units * tiles_per_unit;
  const int t_begin = (int)(total * blockIdx.x / gridDim.x);
  const int t_end = (int)(total * (blockIdx.x + 1) / gridDim.x);
  if (t_begin >= t_end) return;

  if (tid == 0) {
    mbar_init(bar_a[0], 1);
    mbar_init(bar_a[1], 1);
    mbar_init(bar_b, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
    *fail_flag = 0;
  }
  if (warp == 0) {
    tmem_alloc(base + kSmemBar + 32, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto a_row = [&](int t) -> int {
    const int u = t / tiles_per_unit, tl = t - u * tiles_per_unit;
    const int bg = u / a.n_seg, s = u - bg * a.n_seg;
    return bg * a.N + a.seg_lo(s) + tl * kTileM;
  };
  // producer bookkeeping (thread 0): loads/commits issued vs. waited for
  int a_issued[2] = {0, 0}, a_waited[2] = {0, 0}, b_issued = 0, b_waited = 0;
  int mma_issued = 0, mma_waited = 0;
  auto issue_a = [&](int t, int stage) {
    const uint32_t dst = sA + (uint32_t)stage * kAStage;
    const int y = a_row(t);
    mbar_arrive_expect_tx(bar_a[stage], kAStage);
    tma_load_2d(dst, &tmA, 0, y, bar_a[stage]);
    tma_load_2d(dst + kAHalf, &tmA, 64, y, bar_a[stage]);
    ++a_issued[stage];
  };
  auto issue_b = [&](int u) {
    const int bg = u / a.n_seg, s = u - bg * a.n_seg;
    const int y = bg * a.C + s * a.k;
    mbar_arrive_expect_tx(bar_b, (uint32_t)n_chunks * kBChunk);
    for (int nc = 0; nc < n_chunks; ++nc) {
      tma_load_2d(sB + (uint32_t)nc * kBChunk, &tmB, 0, y + nc * 256, bar_b);
      tma_load_2d(sB + (uint32_t)nc * kBChunk + kBHalf, &tmB, 64, y + nc * 256, bar_b);
    }
    ++b_issued;
  };

  if (tid == 0) issue_a(t_begin, 0);
  int cur_unit = -1;
  bool ok = true;
  for (int t = t_begin; t < t_end; ++t) {
    const int i = t - t_begin, stage = i & 1;
    const int u = t / tiles_per_unit;
    const bool new_unit = (u != cur_unit);
    if (tid == 0) {
      // The previous tile's MMAs have completed (waited below), so both the
      // centroid buffer and the other key stage are free to be overwritten.
      if (new_unit) issue_b(u);
      if (t + 1 < t_end) issue_a(t + 1, stage ^ 1);
      bool good = mbar_wait(bar_a[stage], (uint32_t)(a_waited[stage] & 1), a.status);
      if (good) ++a_waited[stage];
      if (good && b_waited < b_issued) {
        good = mbar_wait(bar_b, (uint32_t)(b_waited & 1), a.status);
        if (good) ++b_waited;
      }
      if (good) {
        tc_fence_after();
        for (int nc = 0; nc < n_chunks; ++nc) {
          const int ncols = min(256, a.k - nc * 256);
          const uint32_t idesc = idesc_bf16_f32(kTileM, (ncols + 15) & ~15);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ka = (uint32_t)(kk >> 2) * kAHalf + (uint32_t)(kk & 3) * 32u;
            const uint32_t kb = (uint32_t)(kk >> 2) * kBHalf + (uint32_t)(kk & 3) * 32u;
            tc_mma_bf16(tmem + (uint32_t)nc * 256u,
                        smem_desc_k_sw128(sA + (uint32_t)stage * kAStage + ka),
                        smem_desc_k_sw128(sB + (uint32_t)nc * kBChunk + kb), idesc,
                        kk > 0 ? 1u : 0u);
          }
        }
        tc_commit(bar_mma);
        ++mma_issued;
      } else {
        *fail_flag = 1;
      }
    }
    if (new_unit) cur_unit = u;
    __syncthreads();
    if (*fail_flag) {
      ok = false;
      break;
    }
    const bool done = mbar_wait(bar_mma, (uint32_t)(i & 1), a.status);
    if (!__syncthreads_and(done)) {
      ok = false;
      break;
    }
    if (tid == 0) ++mma_waited;
    tc_fence_after();

    // epilogue: thread (warp, lane) owns TMEM lane 32*warp + lane = tile row
    const int bg = u / a.n_seg, s = u - bg * a.n_seg, tl = t - u * tiles_per_unit;
    const int row = a.seg_lo(s) + tl * kTileM + warp * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
    float best = -INFINITY;
    int bj = 0;
    for (int c0 = 0; c0 < a.k; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(lane_addr + (uint32_t)c0, v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float x = __uint_as_float(v[j]);
        if (c0 + j < a.k && x > best) {
          best = x;
          bj = c0 + j;
        }
      }
    }
    if (row < a.seg_hi(s)) a.assign[(size_t)bg * a.N + row] = s * a.k + bj;
    tc_fence_before();
    __syncthreads();
  }
  if (!ok && tid == 0) {
    // a bounded wait ran out: let every copy and MMA already issued finish
    // (each wait bounded again) before the tensor memory is released
    for (int st = 0; st < 2; ++st)
      while (a_waited[st] < a_issued[st] &&
             mbar_wait(bar_a[st], (uint32_t)(a_waited[st] & 1), a.status))
        ++a_waited[st];
    while (b_waited < b_issued && mbar_wait(bar_b, (uint32_t)(b_waited & 1), a.status)) ++b_waited;
    while (mma_waited < mma_issued &&
           mbar_wait(bar_mma, (uint32_t)(mma_waited & 1), a.status))
      ++mma_waited;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D view [rows, 128] of a bf16 row-major array, boxes of 64 x box_rows
// elements, 128-byte swizzle, zero fill outside the array.
bool make_map(CUtensorMap* m, const void* base, unsigned long long rows, unsigned box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_kmeans_assign(const BuildArgs& a, cudaStream_t st) {
  if (a.N_idx == 0) return cudaSuccess;
  const long long rows_a = (long long)a.B * a.Hkv * a.N;
  const long long rows_b = (long long)a.B * a.Hkv * a.C;
  if (rows_a >= (1LL << 31) || rows_b >= (1LL << 31) || a.k > 2 * 256)
    return cudaErrorInvalidValue;
  CUtensorMap tmA, tmB;
  if (!make_map(&tmA, a.K, (unsigned long long)rows_a, kTileM) ||
      !make_map(&tmB, a.mu, (unsigned long long)rows_b, 256))
    return cudaErrorNotSupported;
  const int tiles_per_unit = (min(a.L, a.N_idx) + kTileM - 1) / kTileM;
  const int n_units = a.B * a.Hkv * a.n_seg;
  const int n_chunks = (a.k + 255) / 256;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  static bool attr_set = false;
  if (!attr_set) {
    e = cudaFuncSetAttribute(assign_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kTcDynSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const long long total = (long long)n_units * tiles_per_unit;
  const int grid = (int)(total < sms ? total : sms);
  assign_tc_kernel<<<grid, kTcThreads, kTcDynSmem, st>>>(tmA, tmB, a, tiles_per_unit, n_units,
                                                         n_chunks);
  return cudaGetLastError();
}

}  // namespace wi
