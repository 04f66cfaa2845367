// Host-side plumbing shared by the libwi translation units: kernel argument
// blocks and launcher prototypes.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "wi.h"

namespace wi {

// Segment s covers absolute positions [s*L, (s+1)*L) minus the steady zone:
// [seg_lo(s), seg_hi(s)) with both ends clamped into [sink, N - window].
__host__ __device__ inline int clamp_pos(long long x, int sink, int N, int window) {
  const long long lo = sink, hi = (long long)N - window;
  return (int)(x < lo ? lo : (x > hi ? hi : x));
}

struct BuildArgs {
  int B, Hkv, N, sink, window, L, k, n_seg, C, N_idx;
  const uint16_t* K;  // bf16 [B,Hkv,N,128]
  const uint16_t* V;
  float* norms;       // f32 [B,Hkv,N] (workspace)
  float* kbar;        // f32 [B,Hkv,C,128]
  uint16_t* mu;       // bf16 [B,Hkv,C,128]
  float* vsum;        // f32 [B,Hkv,C,128]
  int* size;          // [B,Hkv,C]
  int* offset;        // [B,Hkv,C+1]
  int* perm;          // [B,Hkv,N_idx]
  int* assign;        // [B,Hkv,N]
  uint16_t* ksorted;  // bf16 [B,Hkv,N_idx,128]
  uint16_t* vsorted;
  int* status;
  __host__ __device__ int seg_lo(int s) const { return clamp_pos((long long)s * L, sink, N, window); }
  __host__ __device__ int seg_hi(int s) const {
    return clamp_pos((long long)(s + 1) * L, sink, N, window);
  }
};

struct DecodeArgs {
  int B, Hq, Hkv, G, N, sink, window, r, C, N_idx;
  float scale;
  const uint16_t* q;        // bf16 [B,Hq,128]
  const uint16_t* K;        // bf16 [B,Hkv,N,128]
  const uint16_t* V;
  const float* kbar;        // f32 [B,Hkv,C,128]
  const float* vsum;        // f32 [B,Hkv,C,128]
  const int* size;          // [B,Hkv,C]
  const int* offset;        // [B,Hkv,C+1]
  const uint16_t* ksorted;  // bf16 [B,Hkv,N_idx,128]
  const uint16_t* vsorted;
  // workspace regions
  int* status;
  float* scores;        // [B,Hq,C]
  float* head_max;      // [B,Hq]
  int* sel_ids;         // [B,Hq,r]   (r >= 1 slots)
  int* sel_prefix;      // [B,Hq,r+1]
  int* counters;        // [B,Hq]  arrival counters of the attention blocks
  float* att_part;      // [B,Hq,att_splits,2,2+128]  (exact; minus retrieved estimate)
  float* est_part;      // [B,Hq,est_chunks,2+128]
  int att_splits, est_chunks, est_chunk_clusters;
  int inject;           // test hook: block 0 skips its first staging copy
  // outputs
  int* topk_out;        // [B,Hq,r] or null
  float* out;           // [B,Hq,128]
  float* lse;           // [B,Hq] or null
};

constexpr int kPartStride = 2 + 128;  // (m, l, o[128]) per partial

// decode launchers (wi_decode.cu)
cudaError_t launch_decode_score(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_decode_select(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_decode_attend(const DecodeArgs& a, cudaStream_t st);
constexpr int kEstChunk = 256;  // clusters per estimation block

// build launchers (wi_build.cu)
cudaError_t launch_build_init(const BuildArgs& a, cudaStream_t st);
cudaError_t launch_kmeans_assign(const BuildArgs& a, cudaStream_t st);
cudaError_t launch_cluster_sort(const BuildArgs& a, cudaStream_t st);
cudaError_t launch_centroid_update(const BuildArgs& a, cudaStream_t st);
cudaError_t launch_finalize_stats(const BuildArgs& a, cudaStream_t st);

}  // namespace wi
