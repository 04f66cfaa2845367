// Spherical k-means assignment, a(i) = argmax_j k_i . mu_j over the
// centroids of the token's segment, lowest j among equal maxima
// ("RetroInfer: A Vector Storage Engine for Scalable Long-Context LLM
// Inference", technical summary (es) §2.A.2 and §3).
#include "wi_device.cuh"
#include "wi_internal.h"

namespace wi {

namespace {

constexpr int kAsgThreads = 128;

// One thread per key; the segment's centroids sit in shared memory and are
// read as broadcasts.  f32 dot products of the bf16 operands.
__global__ void __launch_bounds__(kAsgThreads) assign_simt_kernel(BuildArgs a, int tiles_per_seg) {
  extern __shared__ __align__(16) uint4 smu[];
  const int tile = blockIdx.x % tiles_per_seg;
  const int sg = blockIdx.x / tiles_per_seg;
  const int s = sg % a.n_seg;
  const int bg = sg / a.n_seg;
  const int lo = a.seg_lo(s), hi = a.seg_hi(s);
  if (lo + tile * kAsgThreads >= hi) return;
  const uint4* mu = reinterpret_cast<const uint4*>(a.mu + ((size_t)bg * a.C + (size_t)s * a.k) * kD);
  for (int i = threadIdx.x; i < a.k * (kD / 8); i += kAsgThreads) smu[i] = mu[i];
  __syncthreads();
  const int p = lo + tile * kAsgThreads + threadIdx.x;
  if (p >= hi) return;
  uint4 kr[kD / 8];
  const uint4* krow = reinterpret_cast<const uint4*>(a.K + ((size_t)bg * a.N + p) * kD);
#pragma unroll
  for (int w = 0; w < kD / 8; ++w) kr[w] = krow[w];
  float best = -INFINITY;
  int bj = 0;
  for (int j = 0; j < a.k; ++j) {
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kD / 8; ++w) {
      const uint4 m = smu[j * (kD / 8) + w];
      acc += bf_lo(kr[w].x) * bf_lo(m.x) + bf_hi(kr[w].x) * bf_hi(m.x) +
             bf_lo(kr[w].y) * bf_lo(m.y) + bf_hi(kr[w].y) * bf_hi(m.y) +
             bf_lo(kr[w].z) * bf_lo(m.z) + bf_hi(kr[w].z) * bf_hi(m.z) +
             bf_lo(kr[w].w) * bf_lo(m.w) + bf_hi(kr[w].w) * bf_hi(m.w);
    }
    if (acc > best) {
      best = acc;
      bj = j;
    }
  }
  a.assign[(size_t)bg * a.N + p] = s * a.k + bj;
}

}  // namespace

cudaError_t launch_kmeans_assign(const BuildArgs& a, cudaStream_t st) {
  const int tiles_per_seg = (a.L + kAsgThreads - 1) / kAsgThreads;
  const size_t smem = (size_t)a.k * kD * 2;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(assign_simt_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)((size_t)WI_MAX_K_PER_SEG * kD * 2));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  assign_simt_kernel<<<a.B * a.Hkv * a.n_seg * tiles_per_seg, kAsgThreads, smem, st>>>(a,
                                                                                       tiles_per_seg);
  return cudaGetLastError();
}

}  // namespace wi
