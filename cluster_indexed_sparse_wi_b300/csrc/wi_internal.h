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

// Most blocks one decode launch uses (one per SM); partial buffers are sized
// for this many so that the workspace layout does not depend on the device.
constexpr int kMaxBlocks = 256;
constexpr int kPartStride = 2 + 128;  // (m, l, o[128]) per partial
constexpr int kDecodeTile = 64;       // index rows / tokens per staging tile

// Which decode stages one launch runs (wi_decode_attention runs all three,
// with grid-wide barriers between them).
enum : int { kStageScore = 1, kStageSelect = 2, kStageAttend = 4 };

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
  // per-launch progress counters, zero at the start of every launch (the last
  // block to finish resets them)
  unsigned* end_cnt;    // blocks finished
  unsigned* mq_tail;    // heads queued for merging (in completion order)
  unsigned* mq_head;    // merge-queue slots claimed
  unsigned* grp_cnt;    // [B*Hkv] scored (index tile, warp) pairs of each KV group
  unsigned* est_cnt;    // [B*Hkv] estimate pieces written for each KV group
  unsigned* head_cnt;   // [B*Hq]  exact-attention units finished for each head
  unsigned* sel_ready;  // [B*Hq]  1 once the head's selection is written
  unsigned* neg_ready;  // [B*Hq]  1 once the estimate of its selection is written
  int* mq_bh;           // [B*Hq]  merge queue: the head of each slot
  unsigned* mq_ready;   // [B*Hq]  1 once the slot's head is written
  int counter_words;    // words from grp_cnt to the end of mq_ready (contiguous)
  float* scores;        // [B,Hq,C]
  float* head_max;      // [B,Hq]
  int* sel_ids;         // [B,Hq,rs]  retrieved ids ascending, -1 padding (rs = max(r,1))
  int* sel_rows;        // [B,Hq,rs]  first sorted row of each retrieved cluster
  int* sel_cnts;        // [B,Hq,rs]  members of each retrieved cluster (0 = padding)
  float* est_part;      // [kMaxBlocks + B*Hkv][G][kPartStride]
  float* std_part;      // [kMaxBlocks + B*Hq][kPartStride]
  float* ret_part;      // [kMaxBlocks + B*Hq][kPartStride]
  float* neg_part;      // [B*Hq][kPartStride]
  // schedule (identical in every block)
  int nb;               // grid size
  int nsel;             // blocks [0, nsel) select; the others score
  int stages;           // kStage* mask
  int fused;            // the stages run in one launch and wait on each other
  int tpg;              // index tiles per KV group: ceil(C / 64)
  int tph;              // steady tiles per query head: ceil((sink + window) / 64)
  int inject;           // test hook: every block skips the copies of its first tile
  // outputs
  int* topk_out;        // [B,Hq,r] or null
  float* out;           // [B,Hq,128]
  float* lse;           // [B,Hq] or null
};

// decode launcher (wi_decode.cu): one persistent launch of the stages in
// a.stages on a.nb blocks.
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st);
// blocks a decode launch uses on the current device
cudaError_t decode_blocks(int* nb);

// build launchers (wi_build.cu)
cudaError_t launch_build_init(const BuildArgs& a, cudaStream_t st);
cudaError_t launch_kmeans_assign(const BuildArgs& a, cudaStream_t st);
cudaError_t launch_cluster_sort(const BuildArgs& a, cudaStream_t st);
cudaError_t launch_centroid_update(const BuildArgs& a, cudaStream_t st);
cudaError_t launch_finalize_stats(const BuildArgs& a, cudaStream_t st);

}  // namespace wi
