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
constexpr int kChunkMax = 16;         // index tiles per chunk
// Static work per block is counted in units of 4 KB of streamed bytes, i.e.
// 8 tokens of K and V (512 bytes per token).
constexpr int kTokPerUnit = 8;

// Which decode stages one launch runs (wi_decode_attention runs all three in
// one launch whose blocks wait on each other's results).
enum : int { kStageScore = 1, kStageSelect = 2, kStageAttend = 4 };

struct DecodeArgs {
  int B, Hq, Hkv, G, N, sink, window, r, C, N_idx;
  float scale;
  const uint16_t* q;        // bf16 [B,Hq,128]
  const uint16_t* K;        // bf16 [B,Hkv,N,128]
  const uint16_t* V;
  const float* kbar;        // f32 [B,Hkv,C,128]
  const float* vsum;        // f32 [B,Hkv,C,128]
  const uint16_t* kbar16;   // bf16 copies of kbar / vsum [B,Hkv,C,128], or null (f32 index)
  const uint16_t* vsum16;
  const int* size;          // [B,Hkv,C]
  const int* offset;        // [B,Hkv,C+1]
  const uint16_t* ksorted;  // bf16 [B,Hkv,N_idx,128]
  const uint16_t* vsorted;
  // workspace regions
  int* status;
  // per-launch progress counters: zero when a launch starts; the last block
  // to finish clears them again
  unsigned* end_cnt;    // blocks finished
  unsigned* sel_done;   // heads whose selection is published
  unsigned* grp_cnt;    // [B*Hkv] index tiles scored per KV group
  unsigned* head_cnt;   // [B*Hq]  partials published per query head
  unsigned* sel_flag;   // [B*Hq]  the head's selection is published
  int counter_words;    // words from grp_cnt to the end of sel_flag (contiguous)
  float* scores;        // [B,Hq,C]   s_c (f32), -inf for empty clusters
  float* head_max;      // [B,Hq]
  int* sel_ids;         // [B,Hq,rs]  retrieved ids ascending, -1 padding (rs = max(r,1))
  int* sel_rows;        // [B,Hq,rs]  first sorted row of each retrieved cluster
  int* sel_cnts;        // [B,Hq,rs]  members of each (0 = padding)
  int* sel_pre;         // [B,Hq,rs]  members of the clusters before it (token offset)
  float* sel_sc;        // [B,Hq,rs]  its score s_c
  int* head_tok;        // [B,Hq]     retrieved tokens of the head
  float* grp_vals;      // [B,Hkv,C]  shared selection: summed ranking keys
  float* est_part;      // [(nchunks + B*Hkv) * G][kPartStride]
  float* std_part;      // [B*Hkv*tph * G][kPartStride]
  float* ret_part;      // [(nb + B*Hq)][kPartStride]
  // schedule (identical in every block)
  int nb;               // grid size
  int stages;           // kStage* mask
  int fused;            // the stages run in one launch and wait on each other
  int tpg;              // index tiles per KV group: ceil(C / 64)
  int tph;              // steady tiles per KV group: ceil((sink + window) / 64)
  int nt;               // index tiles: B * Hkv * tpg
  int Q;                // index tiles per chunk (<= kChunkMax)
  int nchunks;          // ceil(nt / Q); chunk j is taken by block j % nb in round j / nb
  int rounds;           // ceil(nchunks / nb)
  int kbar_first;       // every round's centroid-key tiles before any selection
  int ret_per_head;     // retrieval by fixed per-head block ranges (few heads), each
                        // started once its head's selection is published
  int inject;           // test hook: every block skips the copies of its first tile
  // selection options
  int rank_mass;        // rank clusters by s_c + ln n_c instead of s_c
  int share;            // one retrieval set per KV group (summed ranking keys)
  float tau;            // reuse threshold on the group's smallest query cosine
  const uint16_t* prev_q;  // bf16 [B,Hq,128] previous step's queries, or null (no reuse)
  const int* prev_topk;    // [B,Hq,r] previous step's retrieved ids (ascending, -1 padding)
  int* reused;             // [B,Hkv] 1 where the group reused, or null
  long long static_units;         // sum of static_w
  unsigned static_w[kMaxBlocks];  // static work of each block, 4 KB units
  // outputs
  int* topk_out;        // [B,Hq,r] or null
  float* out;           // [B,Hq,128]
  float* lse;           // [B,Hq] or null
};

// ---- the static schedule, shared by the host (work estimates) and the kernel
// Chunk j holds index tiles [j*Q, min((j+1)*Q, nt)).
__host__ __device__ inline int chunk_tiles(const DecodeArgs& a, int j) {
  const int lo = j * a.Q, hi = lo + a.Q < a.nt ? lo + a.Q : a.nt;
  return hi > lo ? hi - lo : 0;
}
// (nt = B * Hkv * tpg < 2^31 is checked on the host: 32-bit arithmetic)
__host__ __device__ inline int first_chunk(const DecodeArgs& a, int bg) {
  return bg * a.tpg / a.Q;
}
__host__ __device__ inline int last_chunk(const DecodeArgs& a, int bg) {
  return (bg * a.tpg + a.tpg - 1) / a.Q;
}
// Head bh (b*Hq + h) of KV group bg = bh / G is selected by block
// (last_chunk(bg) - bh % G) mod nb, after that block's centroid-key tiles of
// round last_chunk(bg) / nb: a selection only waits on chunks of its own or
// earlier rounds.
__host__ __device__ inline int sel_block(const DecodeArgs& a, int bh) {
  const int x = (last_chunk(a, bh / a.G) - bh % a.G) % a.nb;
  return x < 0 ? x + a.nb : x;
}
__host__ __device__ inline int sel_round(const DecodeArgs& a, int bh) {
  return last_chunk(a, bh / a.G) / a.nb;
}
// Steady tile t (of B*Hkv*tph) is taken by block nb - 1 - t % nb.
__host__ __device__ inline int steady_block(const DecodeArgs& a, int t) {
  return a.nb - 1 - t % a.nb;
}
// With a.ret_per_head, head bh's retrieved tokens are split evenly over the
// blocks [ret_first(bh), ret_first(bh + 1)).
__host__ __device__ inline int ret_first(const DecodeArgs& a, int bh) {
  const int H = a.B * a.Hq;
  return (int)(((long long)bh * a.nb + H - 1) / H);
}
// Head bh is merged by block bh % nb.
__host__ __device__ inline int merge_block(const DecodeArgs& a, int bh) { return bh % a.nb; }

// Host checks of a decode call that need no workspace (parameters, index,
// pointers, device); wi_api.cu.
int decode_precheck(const wi_decode_params* p, const void* q, const void* K, const void* V,
                    const wi_index* ix, const float* out);

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
// Index maintenance: the context grew from N0 to N1 positions; positions
// [N0 - window, N1 - window) join the index (wi_build.cu).
struct ExtendArgs {
  int B, Hkv, N0, N1, sink, window, L, k, C_old, C_new, s_last;
  const uint16_t* K;         // bf16 [B,Hkv,N1,128]
  const uint16_t* mu_old;    // bf16 [B,Hkv,C_old,128]
  const int* assign_old;     // [B,Hkv,N0]
  uint16_t* mu_new;          // bf16 [B,Hkv,C_new,128]
  int* assign_new;           // [B,Hkv,N1]
};
cudaError_t launch_extend(const ExtendArgs& e, cudaStream_t st);

// dst[i] = bf16(src[i]) for i < n (n a multiple of 4; 16-byte aligned arrays)
cudaError_t launch_round_bf16(const float* src, uint16_t* dst, size_t n, cudaStream_t st);

}  // namespace wi
