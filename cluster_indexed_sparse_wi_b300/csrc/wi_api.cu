// C ABI of libwi (declared in include/wi.h): argument validation, workspace
// layout, and kernel enqueueing on the caller's stream.  No device memory is
// allocated here and nothing synchronises except wi_sync_status.
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "wi.h"
#include "wi_internal.h"

using wi::BuildArgs;
using wi::DecodeArgs;

namespace {

constexpr size_t kStatusBytes = 256;  // status word + reserved
constexpr size_t kSyncBytes = 256;    // launch-wide words (blocks finished, selections published) at the start of the counters region
std::atomic<int> g_inject{0};         // wi_debug_inject request

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

int device_ok() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return WI_ERR_LAUNCH;
  static int checked[64] = {0};  // 0 unknown, 1 ok, 2 unsupported
  if (dev >= 0 && dev < 64 && checked[dev] != 0) return checked[dev] == 1 ? WI_OK : WI_ERR_UNSUPPORTED;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return WI_ERR_LAUNCH;
  const bool ok = (major == 10 && minor == 3);
  if (dev >= 0 && dev < 64) checked[dev] = ok ? 1 : 2;
  return ok ? WI_OK : WI_ERR_UNSUPPORTED;
}

int check_build(const wi_build_params* p) {
  if (p == nullptr) return WI_ERR_INVALID_ARG;
  if (p->B < 1 || p->Hkv < 1 || p->N < 1 || p->sink < 0 || p->window < 0 || p->iters < 1 ||
      p->seg_len < 1 || p->k_per_seg < 1)
    return WI_ERR_INVALID_ARG;
  if ((long long)p->sink + p->window > p->N) return WI_ERR_INVALID_ARG;
  if (p->d != WI_HEAD_DIM) return WI_ERR_UNSUPPORTED;
  if (p->seg_len > WI_MAX_SEG_LEN || p->k_per_seg > WI_MAX_K_PER_SEG) return WI_ERR_UNSUPPORTED;
  if (p->N > (1 << 30)) return WI_ERR_UNSUPPORTED;
  const long long n_seg = ((long long)p->N + p->seg_len - 1) / p->seg_len;
  if (n_seg * p->k_per_seg > WI_MAX_CLUSTERS) return WI_ERR_UNSUPPORTED;
  return WI_OK;
}

int n_clusters_of(const wi_build_params* p) {
  return (int)(((long long)p->N + p->seg_len - 1) / p->seg_len) * p->k_per_seg;
}

size_t build_ws_bytes(const wi_build_params* p) {
  return kStatusBytes + align256((size_t)p->B * p->Hkv * p->N * sizeof(float));
}

int fill_build_args(const wi_build_params* p, const void* K, const void* V, wi_index* ix,
                    void* ws, size_t ws_bytes, BuildArgs* a) {
  int st = check_build(p);
  if (st != WI_OK) return st;
  if (ix == nullptr || ws == nullptr || K == nullptr) return WI_ERR_INVALID_ARG;
  if (ws_bytes < build_ws_bytes(p)) return WI_ERR_WORKSPACE;
  if (!aligned(ws, 256) || !aligned(K, 16) || (V != nullptr && !aligned(V, 16)))
    return WI_ERR_ALIGNMENT;
  memset(a, 0, sizeof(*a));
  a->B = p->B;
  a->Hkv = p->Hkv;
  a->N = p->N;
  a->sink = p->sink;
  a->window = p->window;
  a->L = p->seg_len;
  a->k = p->k_per_seg;
  a->n_seg = (int)(((long long)p->N + p->seg_len - 1) / p->seg_len);
  a->C = a->n_seg * a->k;
  a->N_idx = p->N - p->sink - p->window;
  a->K = static_cast<const uint16_t*>(K);
  a->V = static_cast<const uint16_t*>(V);
  a->status = static_cast<int*>(ws);
  a->norms = reinterpret_cast<float*>(static_cast<char*>(ws) + kStatusBytes);
  a->kbar = ix->centroid_key;
  a->mu = static_cast<uint16_t*>(ix->unit_centroid);
  a->vsum = ix->value_sum;
  a->size = ix->size;
  a->offset = ix->offset;
  a->perm = ix->perm;
  a->assign = ix->assign;
  a->ksorted = static_cast<uint16_t*>(ix->k_sorted);
  a->vsorted = static_cast<uint16_t*>(ix->v_sorted);
  return WI_OK;
}

// Pointers a build step needs, by step.
enum Need { kNeedInit = 1, kNeedAssign = 2, kNeedUpdate = 4, kNeedFinal = 8 };

int check_index_ptrs(const BuildArgs& a, int need) {
  const void* req[9] = {nullptr};
  int n = 0;
  req[n++] = a.mu;
  req[n++] = a.assign;
  if (need & (kNeedUpdate | kNeedFinal)) {
    req[n++] = a.size;
    req[n++] = a.offset;
    req[n++] = a.perm;
  }
  if (need & kNeedFinal) {
    req[n++] = a.kbar;
    req[n++] = a.vsum;
    req[n++] = a.ksorted;
    req[n++] = a.vsorted;
  }
  for (int i = 0; i < n; ++i) {
    // arrays with N_idx rows (perm, k_sorted, v_sorted) may be NULL when N_idx == 0
    const bool may_be_null = a.N_idx == 0 && (req[i] == a.perm || req[i] == a.ksorted ||
                                              req[i] == a.vsorted);
    if (req[i] == nullptr && !may_be_null) return WI_ERR_INVALID_ARG;
    if (!aligned(req[i], 16)) return WI_ERR_ALIGNMENT;
  }
  if ((need & kNeedFinal) && a.V == nullptr) return WI_ERR_INVALID_ARG;
  return WI_OK;
}

int check_recorded(const wi_build_params* p, const wi_index* ix) {
  const int C = n_clusters_of(p);
  if (ix->B != p->B || ix->Hkv != p->Hkv || ix->N != p->N || ix->d != p->d ||
      ix->sink != p->sink || ix->window != p->window || ix->seg_len != p->seg_len ||
      ix->k_per_seg != p->k_per_seg || ix->n_clusters != C)
    return WI_ERR_INDEX_MISMATCH;
  return WI_OK;
}

void record(const wi_build_params* p, wi_index* ix) {
  ix->B = p->B;
  ix->Hkv = p->Hkv;
  ix->N = p->N;
  ix->d = p->d;
  ix->sink = p->sink;
  ix->window = p->window;
  ix->seg_len = p->seg_len;
  ix->k_per_seg = p->k_per_seg;
  ix->n_clusters = n_clusters_of(p);
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? WI_OK : WI_ERR_LAUNCH; }

// ---------------------------------------------------------------- decode
int check_decode(const wi_decode_params* p, int C) {
  if (p == nullptr) return WI_ERR_INVALID_ARG;
  if (p->B < 1 || p->Hq < 1 || p->Hkv < 1 || p->N < 1 || p->sink < 0 || p->window < 0 ||
      p->r < 0 || C < 1)
    return WI_ERR_INVALID_ARG;
  if ((long long)p->sink + p->window > p->N || p->r > C) return WI_ERR_INVALID_ARG;
  if (p->Hq % p->Hkv != 0) return WI_ERR_INVALID_ARG;
  const int G = p->Hq / p->Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return WI_ERR_UNSUPPORTED;
  if (p->d != WI_HEAD_DIM || C > WI_MAX_CLUSTERS || p->N > (1 << 30)) return WI_ERR_UNSUPPORTED;
  if (!(p->scale == p->scale)) return WI_ERR_INVALID_ARG;
  return WI_OK;
}

// Index tiles, steady tiles and chunking of a decode over C clusters on nb
// blocks (the kernel's static schedule).
struct DecodeShape {
  int tpg, tph, nt, Q, nchunks, rounds;
};
DecodeShape decode_shape(const wi_decode_params* p, int C, int nb) {
  DecodeShape d;
  d.tpg = (C + wi::kDecodeTile - 1) / wi::kDecodeTile;
  d.tph = (p->sink + p->window + wi::kDecodeTile - 1) / wi::kDecodeTile;
  d.nt = p->B * p->Hkv * d.tpg;
  // chunks of at most kChunkMax tiles, about equal, in whole rounds of nb
  const long long per_round = (long long)nb * wi::kChunkMax;
  int rounds = (int)((d.nt + per_round - 1) / per_round);
  if (rounds < 1) rounds = 1;
  d.Q = (int)((d.nt + (long long)nb * rounds - 1) / ((long long)nb * rounds));
  if (d.Q < 1) d.Q = 1;
  d.nchunks = (d.nt + d.Q - 1) / d.Q;
  d.rounds = (d.nchunks + nb - 1) / nb;
  return d;
}

// Chunks are at most kChunkMax tiles and number at most nb per round, so
// nchunks <= nt / kChunkMax + nb: a bound that does not depend on the device.
size_t est_slots(const wi_decode_params* p, int C) {
  const size_t tpg = (size_t)(C + wi::kDecodeTile - 1) / wi::kDecodeTile;
  const size_t nt = (size_t)p->B * p->Hkv * tpg;
  size_t nch = nt / wi::kChunkMax + wi::kMaxBlocks + 1;
  if (nch > nt) nch = nt;
  return nch + (size_t)p->B * p->Hkv;
}

int decode_layout(const wi_decode_params* p, int C, wi_decode_layout* L) {
  const int st = check_decode(p, C);
  if (st != WI_OK) return st;
  memset(L, 0, sizeof(*L));
  const size_t heads = (size_t)p->B * p->Hq;
  const size_t groups = (size_t)p->B * p->Hkv;
  const size_t G = (size_t)(p->Hq / p->Hkv);
  const size_t rs = p->r > 0 ? (size_t)p->r : 1;
  const size_t part = (size_t)wi::kPartStride * 4;
  const size_t tph = (size_t)(p->sink + p->window + wi::kDecodeTile - 1) / wi::kDecodeTile;
  size_t off = kStatusBytes;
  L->counters = off;
  L->counter_bytes = (int)align256(kSyncBytes + (groups + 2 * heads) * 4);
  off += (size_t)L->counter_bytes;
  L->scores = off;
  off += align256(heads * (size_t)C * 4);
  L->head_max = off;
  off += align256(heads * 4);
  L->selected = off;
  off += align256(heads * rs * 4);
  L->sel_rows = off;
  off += align256(heads * rs * 4);
  L->sel_counts = off;
  off += align256(heads * rs * 4);
  L->sel_prefix = off;
  off += align256(heads * rs * 4);
  L->sel_scores = off;
  off += align256(heads * rs * 4);
  L->head_tokens = off;
  off += align256(heads * 4);
  L->group_values = off;
  off += align256(groups * (size_t)C * 4);
  L->partials = off;
  off += align256(est_slots(p, C) * G * part);         // estimate pieces
  off += align256(groups * tph * G * part);            // steady pieces
  off += align256((wi::kMaxBlocks + heads) * part);    // retrieval pieces
  L->total = off;
  L->max_blocks = wi::kMaxBlocks;
  return WI_OK;
}

// Streamed-work equivalent of one per-head selection, in 4 KB units (the
// scores and sizes it reads and the passes over them).
unsigned selection_units(int C) { return 24u + (unsigned)(C / 96); }

}  // namespace

namespace wi {

int decode_precheck(const wi_decode_params* p, const void* q, const void* K, const void* V,
                    const wi_index* ix, const float* out) {
  if (p == nullptr || ix == nullptr) return WI_ERR_INVALID_ARG;
  int st = check_decode(p, ix->n_clusters);
  if (st != WI_OK) return st;
  if (ix->B != p->B || ix->Hkv != p->Hkv || ix->N != p->N || ix->d != p->d ||
      ix->sink != p->sink || ix->window != p->window)
    return WI_ERR_INDEX_MISMATCH;
  const bool no_idx = p->N - p->sink - p->window == 0;  // sorted arrays may be NULL then
  const void* req[] = {ix->centroid_key, ix->value_sum, ix->size, ix->offset,
                       ix->k_sorted, ix->v_sorted};
  for (int i = 0; i < 6; ++i) {
    if (req[i] == nullptr && !(no_idx && i >= 4)) return WI_ERR_INVALID_ARG;
    if (!aligned(req[i], 16)) return WI_ERR_ALIGNMENT;
  }
  if (q == nullptr || K == nullptr || V == nullptr || out == nullptr) return WI_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(K, 16) || !aligned(V, 16)) return WI_ERR_ALIGNMENT;
  const long long n_tiles = (long long)p->B * p->Hkv *
                            ((ix->n_clusters + wi::kDecodeTile - 1) / wi::kDecodeTile);
  if (n_tiles >= (1LL << 31) || (long long)p->B * p->Hq >= (1LL << 31)) return WI_ERR_UNSUPPORTED;
  return device_ok();
}

}  // namespace wi

namespace {

int fill_decode_args(const wi_decode_params* p, const void* q, const void* K, const void* V,
                     const wi_index* ix, void* ws, size_t ws_bytes, DecodeArgs* a,
                     bool need_q, bool need_kv, const wi_decode_options* opt) {
  if (p == nullptr || ix == nullptr || ws == nullptr) return WI_ERR_INVALID_ARG;
  wi_decode_layout L;
  int st = decode_layout(p, ix->n_clusters, &L);
  if (st != WI_OK) return st;
  if (ix->B != p->B || ix->Hkv != p->Hkv || ix->N != p->N || ix->d != p->d ||
      ix->sink != p->sink || ix->window != p->window)
    return WI_ERR_INDEX_MISMATCH;
  if (ws_bytes < L.total) return WI_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return WI_ERR_ALIGNMENT;
  const bool no_idx = p->N - p->sink - p->window == 0;  // sorted arrays may be NULL then
  const void* req[] = {ix->centroid_key, ix->value_sum, ix->size, ix->offset,
                       ix->k_sorted, ix->v_sorted};
  for (int i = 0; i < 6; ++i) {
    if (req[i] == nullptr && !(no_idx && i >= 4)) return WI_ERR_INVALID_ARG;
    if (!aligned(req[i], 16)) return WI_ERR_ALIGNMENT;
  }
  if (need_q) {
    if (q == nullptr) return WI_ERR_INVALID_ARG;
    if (!aligned(q, 16)) return WI_ERR_ALIGNMENT;
  }
  if (need_kv) {
    if (K == nullptr || V == nullptr) return WI_ERR_INVALID_ARG;
    if (!aligned(K, 16) || !aligned(V, 16)) return WI_ERR_ALIGNMENT;
  }
  const int C = ix->n_clusters;
  const long long n_tiles = (long long)p->B * p->Hkv * ((C + wi::kDecodeTile - 1) / wi::kDecodeTile);
  if (n_tiles >= (1LL << 31) || (long long)p->B * p->Hq >= (1LL << 31)) return WI_ERR_UNSUPPORTED;
  if ((long long)p->B * p->Hkv * ((p->sink + p->window + wi::kDecodeTile - 1) / wi::kDecodeTile) >=
      (1LL << 31))
    return WI_ERR_UNSUPPORTED;
  if ((st = device_ok()) != WI_OK) return st;
  int nb = 0;
  if (wi::decode_blocks(&nb) != cudaSuccess || nb < 2) return WI_ERR_LAUNCH;
  memset(a, 0, sizeof(*a));
  char* w = static_cast<char*>(ws);
  a->B = p->B;
  a->Hq = p->Hq;
  a->Hkv = p->Hkv;
  a->G = p->Hq / p->Hkv;
  a->N = p->N;
  a->sink = p->sink;
  a->window = p->window;
  a->r = p->r;
  a->C = C;
  a->N_idx = p->N - p->sink - p->window;
  a->scale = p->scale;
  a->q = static_cast<const uint16_t*>(q);
  a->K = static_cast<const uint16_t*>(K);
  a->V = static_cast<const uint16_t*>(V);
  a->kbar = ix->centroid_key;
  a->vsum = ix->value_sum;
  if (opt != nullptr && opt->centroid_key_bf16 != nullptr) {
    a->kbar16 = static_cast<const uint16_t*>(opt->centroid_key_bf16);
    a->vsum16 = static_cast<const uint16_t*>(opt->value_sum_bf16);
  }
  a->size = ix->size;
  a->offset = ix->offset;
  a->ksorted = static_cast<const uint16_t*>(ix->k_sorted);
  a->vsorted = static_cast<const uint16_t*>(ix->v_sorted);
  a->status = reinterpret_cast<int*>(w);
  const size_t heads = (size_t)p->B * p->Hq, groups = (size_t)p->B * p->Hkv;
  {
    unsigned* c = reinterpret_cast<unsigned*>(w + L.counters);
    a->end_cnt = c;
    a->sel_done = c + 1;
    a->grp_cnt = c + kSyncBytes / 4;
    a->head_cnt = a->grp_cnt + groups;
    a->sel_flag = a->head_cnt + heads;
    a->counter_words = (int)(groups + 2 * heads);
  }
  a->scores = reinterpret_cast<float*>(w + L.scores);
  a->head_max = reinterpret_cast<float*>(w + L.head_max);
  a->sel_ids = reinterpret_cast<int*>(w + L.selected);
  a->sel_rows = reinterpret_cast<int*>(w + L.sel_rows);
  a->sel_cnts = reinterpret_cast<int*>(w + L.sel_counts);
  a->sel_pre = reinterpret_cast<int*>(w + L.sel_prefix);
  a->sel_sc = reinterpret_cast<float*>(w + L.sel_scores);
  a->head_tok = reinterpret_cast<int*>(w + L.head_tokens);
  a->grp_vals = reinterpret_cast<float*>(w + L.group_values);
  const size_t part = (size_t)wi::kPartStride * 4;
  const DecodeShape d = decode_shape(p, C, nb);
  size_t off = L.partials;
  a->est_part = reinterpret_cast<float*>(w + off);
  off += align256(est_slots(p, C) * (size_t)a->G * part);
  a->std_part = reinterpret_cast<float*>(w + off);
  off += align256(groups * (size_t)d.tph * (size_t)a->G * part);
  a->ret_part = reinterpret_cast<float*>(w + off);
  a->nb = nb;
  a->tpg = d.tpg;
  a->tph = d.tph;
  a->nt = d.nt;
  a->Q = d.Q;
  a->nchunks = d.nchunks;
  a->rounds = d.rounds;
  // With few heads, the selections of the groups scored in the last round
  // would start only near the end of the index stream: score every round
  // first and select in one wave.  With many heads, selections round by
  // round keep the index stream busy on the other blocks meanwhile.
  a->kbar_first = (d.rounds > 1 && (long long)p->B * p->Hq <= nb) ? 1 : 0;
  // static work of every block (4 KB units): its index tiles (centroid keys
  // and value sums, 64 KB per tile), steady tiles (32 KB) and selections
  const unsigned su = selection_units(C);
  for (int b = 0; b < nb; ++b) a->static_w[b] = 0u;
  const unsigned tile_units = a->kbar16 ? 8u : 16u;  // both passes of one index tile
  for (int j = 0; j < a->nchunks; ++j)
    a->static_w[j % nb] += tile_units * (unsigned)wi::chunk_tiles(*a, j);
  const int nst = (int)groups * d.tph;
  for (int t = 0; t < nst; ++t) a->static_w[wi::steady_block(*a, t)] += 8u;
  for (size_t bh = 0; bh < heads; ++bh) a->static_w[wi::sel_block(*a, (int)bh)] += su;
  // Retrieval starts once every selection is published: after the centroid-
  // key tiles of every round (and, round by round, the value-sum tiles of
  // the earlier rounds) and one selection.  Work a block finishes before
  // then does not delay its retrieval share, so only the rest counts.
  const unsigned wait = tile_units / 2u * (unsigned)d.Q *
                           (a->kbar_first ? (unsigned)d.rounds : 2u * (unsigned)d.rounds - 1u) +
                       su;
  for (int b = 0; b < nb; ++b) a->static_w[b] = a->static_w[b] > wait ? a->static_w[b] - wait : 0u;
  a->static_units = 0;
  for (int b = 0; b < nb; ++b) a->static_units += a->static_w[b];
  return WI_OK;
}

// Host checks of the selection options (only the fused call takes them).
int check_options(const wi_decode_options* o, const wi_decode_params* p) {
  if (o == nullptr) return WI_OK;
  if (o->rank != WI_RANK_SCORE && o->rank != WI_RANK_MASS) return WI_ERR_INVALID_ARG;
  if (o->share != WI_SHARE_HEAD && o->share != WI_SHARE_GROUP) return WI_ERR_INVALID_ARG;
  if (o->prev_q != nullptr && p != nullptr && p->r > 0) {
    if (o->prev_topk == nullptr || !(o->tau == o->tau)) return WI_ERR_INVALID_ARG;
    if (!aligned(o->prev_q, 16) || !aligned(o->prev_topk, 4)) return WI_ERR_ALIGNMENT;
  }
  if (!aligned(o->reused, 4)) return WI_ERR_ALIGNMENT;
  if ((o->centroid_key_bf16 == nullptr) != (o->value_sum_bf16 == nullptr)) return WI_ERR_INVALID_ARG;
  if (!aligned(o->centroid_key_bf16, 16) || !aligned(o->value_sum_bf16, 16)) return WI_ERR_ALIGNMENT;
  return WI_OK;
}

int run_decode(const wi_decode_params* p, const void* q, const void* K, const void* V,
               const wi_index* index, float* out, float* lse, int32_t* topk_ids, void* workspace,
               size_t workspace_bytes, wi_stream_t stream, int stages, bool need_q, bool need_kv,
               const wi_decode_options* opt = nullptr) {
  if ((stages & wi::kStageAttend) && out == nullptr) return WI_ERR_INVALID_ARG;
  DecodeArgs a;
  int st = check_options(opt, p);
  if (st != WI_OK) return st;
  st = fill_decode_args(p, q, K, V, index, workspace, workspace_bytes, &a, need_q, need_kv, opt);
  if (st != WI_OK) return st;
  if (opt != nullptr) {
    a.rank_mass = opt->rank == WI_RANK_MASS ? 1 : 0;
    // (the static work estimates keep one selection per head: a group's
    // selection costs about as much as its heads' would have together)
    a.share = opt->share == WI_SHARE_GROUP ? 1 : 0;
    if (opt->prev_q != nullptr && p->r > 0) {
      a.prev_q = static_cast<const uint16_t*>(opt->prev_q);
      a.prev_topk = opt->prev_topk;
      a.tau = opt->tau;
    }
    a.reused = opt->reused;
  }
  a.stages = stages;
  a.fused = stages == (wi::kStageScore | wi::kStageSelect | wi::kStageAttend) ? 1 : 0;
  a.out = out;
  a.lse = lse;
  a.topk_out = topk_ids;
  if (stages & wi::kStageAttend) a.inject = g_inject.exchange(0);
  // few heads with short retrieval lists (about r N_idx / C <= 4096 tokens a
  // head): each head's retrieval on its own block range, started as soon as
  // that head is selected (no wait for every selection, no partition).  With
  // longer lists the token-balanced split over all heads wins.  The stage
  // calls split the same way, so they compose to the fused call.
  const long long est_tokens = a.C > 0 ? (long long)a.r * a.N_idx / a.C : 0;
  a.ret_per_head = (!a.share && a.r > 0 && (long long)a.B * a.Hq * 4 <= a.nb &&
                    est_tokens <= 4096) ? 1 : 0;
  return cuda_status(wi::launch_decode(a, (cudaStream_t)stream));
}

}  // namespace

extern "C" {

int wi_index_sizes(const wi_build_params* p, size_t* bytes_out) {
  const int st = check_build(p);
  if (st != WI_OK) return st;
  if (bytes_out == nullptr) return WI_ERR_INVALID_ARG;
  const size_t heads = (size_t)p->B * p->Hkv;
  const size_t C = (size_t)n_clusters_of(p);
  const size_t n_idx = (size_t)(p->N - p->sink - p->window);
  bytes_out[WI_FIELD_CENTROID_KEY] = heads * C * WI_HEAD_DIM * 4;
  bytes_out[WI_FIELD_UNIT_CENTROID] = heads * C * WI_HEAD_DIM * 2;
  bytes_out[WI_FIELD_VALUE_SUM] = heads * C * WI_HEAD_DIM * 4;
  bytes_out[WI_FIELD_SIZE] = heads * C * 4;
  bytes_out[WI_FIELD_OFFSET] = heads * (C + 1) * 4;
  bytes_out[WI_FIELD_PERM] = heads * n_idx * 4;
  bytes_out[WI_FIELD_ASSIGN] = heads * (size_t)p->N * 4;
  bytes_out[WI_FIELD_K_SORTED] = heads * n_idx * WI_HEAD_DIM * 2;
  bytes_out[WI_FIELD_V_SORTED] = heads * n_idx * WI_HEAD_DIM * 2;
  return WI_OK;
}

size_t wi_build_workspace_bytes(const wi_build_params* p) {
  return check_build(p) == WI_OK ? build_ws_bytes(p) : 0;
}

int wi_build_init(const wi_build_params* p, const void* K, wi_index* index, void* workspace,
                  size_t workspace_bytes, wi_stream_t stream) {
  BuildArgs a;
  int st = fill_build_args(p, K, nullptr, index, workspace, workspace_bytes, &a);
  if (st != WI_OK) return st;
  if ((st = check_index_ptrs(a, kNeedInit)) != WI_OK) return st;
  if ((st = device_ok()) != WI_OK) return st;
  record(p, index);
  return cuda_status(wi::launch_build_init(a, (cudaStream_t)stream));
}

int wi_kmeans_assign(const wi_build_params* p, const void* K, wi_index* index, void* workspace,
                     size_t workspace_bytes, wi_stream_t stream) {
  BuildArgs a;
  int st = fill_build_args(p, K, nullptr, index, workspace, workspace_bytes, &a);
  if (st != WI_OK) return st;
  if ((st = check_index_ptrs(a, kNeedAssign)) != WI_OK) return st;
  if ((st = check_recorded(p, index)) != WI_OK) return st;
  if ((st = device_ok()) != WI_OK) return st;
  return cuda_status(wi::launch_kmeans_assign(a, (cudaStream_t)stream));
}

int wi_kmeans_update(const wi_build_params* p, const void* K, wi_index* index, void* workspace,
                     size_t workspace_bytes, wi_stream_t stream) {
  BuildArgs a;
  int st = fill_build_args(p, K, nullptr, index, workspace, workspace_bytes, &a);
  if (st != WI_OK) return st;
  if ((st = check_index_ptrs(a, kNeedUpdate)) != WI_OK) return st;
  if ((st = check_recorded(p, index)) != WI_OK) return st;
  if ((st = device_ok()) != WI_OK) return st;
  const cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = wi::launch_cluster_sort(a, s);
  if (e == cudaSuccess) e = wi::launch_centroid_update(a, s);
  return cuda_status(e);
}

int wi_build_finalize(const wi_build_params* p, const void* K, const void* V, wi_index* index,
                      void* workspace, size_t workspace_bytes, wi_stream_t stream) {
  BuildArgs a;
  int st = fill_build_args(p, K, V, index, workspace, workspace_bytes, &a);
  if (st != WI_OK) return st;
  if ((st = check_index_ptrs(a, kNeedFinal)) != WI_OK) return st;
  if ((st = check_recorded(p, index)) != WI_OK) return st;
  if ((st = device_ok()) != WI_OK) return st;
  const cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = wi::launch_cluster_sort(a, s);
  if (e == cudaSuccess) e = wi::launch_finalize_stats(a, s);
  return cuda_status(e);
}

int wi_index_extend(const wi_build_params* p, const void* K, const void* V,
                    const wi_index* old_index, wi_index* index, void* workspace,
                    size_t workspace_bytes, wi_stream_t stream) {
  if (old_index == nullptr) return WI_ERR_INVALID_ARG;
  BuildArgs a;
  int st = fill_build_args(p, K, V, index, workspace, workspace_bytes, &a);
  if (st != WI_OK) return st;
  if ((st = check_index_ptrs(a, kNeedInit | kNeedAssign | kNeedUpdate | kNeedFinal)) != WI_OK)
    return st;
  const wi_index* o = old_index;
  if (o->B != p->B || o->Hkv != p->Hkv || o->d != p->d || o->sink != p->sink ||
      o->window != p->window || o->seg_len != p->seg_len || o->k_per_seg != p->k_per_seg ||
      o->N > p->N || o->n_clusters <= 0)
    return WI_ERR_INDEX_MISMATCH;
  if (o->unit_centroid == nullptr || o->assign == nullptr) return WI_ERR_INVALID_ARG;
  if (!aligned(o->unit_centroid, 16) || !aligned(o->assign, 16)) return WI_ERR_ALIGNMENT;
  // the joining positions must lie in segments the earlier index clustered
  const int hi_old = o->N - o->window;
  if (hi_old <= o->sink) return WI_ERR_UNSUPPORTED;
  const int s_last = (hi_old - 1) / p->seg_len;
  if ((long long)p->N - p->window > (long long)(s_last + 1) * p->seg_len) return WI_ERR_UNSUPPORTED;
  if ((st = device_ok()) != WI_OK) return st;
  wi::ExtendArgs e;
  e.B = p->B;
  e.Hkv = p->Hkv;
  e.N0 = o->N;
  e.N1 = p->N;
  e.sink = p->sink;
  e.window = p->window;
  e.L = p->seg_len;
  e.k = p->k_per_seg;
  e.C_old = o->n_clusters;
  e.C_new = a.C;
  e.s_last = s_last;
  e.K = a.K;
  e.mu_old = static_cast<const uint16_t*>(o->unit_centroid);
  e.assign_old = o->assign;
  e.mu_new = a.mu;
  e.assign_new = a.assign;
  record(p, index);
  const cudaStream_t s = (cudaStream_t)stream;
  cudaError_t err = wi::launch_extend(e, s);
  if (err == cudaSuccess) err = wi::launch_cluster_sort(a, s);
  if (err == cudaSuccess) err = wi::launch_finalize_stats(a, s);
  return cuda_status(err);
}

int wi_build_index(const wi_build_params* p, const void* K, const void* V, wi_index* index,
                   void* workspace, size_t workspace_bytes, wi_stream_t stream) {
  BuildArgs a;
  int st = fill_build_args(p, K, V, index, workspace, workspace_bytes, &a);
  if (st != WI_OK) return st;
  if ((st = check_index_ptrs(a, kNeedInit | kNeedAssign | kNeedUpdate | kNeedFinal)) != WI_OK)
    return st;
  if ((st = device_ok()) != WI_OK) return st;
  record(p, index);
  const cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = wi::launch_build_init(a, s);
  for (int it = 0; it < p->iters && e == cudaSuccess; ++it) {
    e = wi::launch_kmeans_assign(a, s);
    if (e == cudaSuccess) e = wi::launch_cluster_sort(a, s);
    if (e == cudaSuccess) e = wi::launch_centroid_update(a, s);
  }
  // the last update sorted the final assignment: size/offset/perm are current
  if (e == cudaSuccess) e = wi::launch_finalize_stats(a, s);
  return cuda_status(e);
}

size_t wi_decode_workspace_bytes(const wi_decode_params* p, int n_clusters) {
  wi_decode_layout L;
  return decode_layout(p, n_clusters, &L) == WI_OK ? L.total : 0;
}

int wi_decode_workspace_layout(const wi_decode_params* p, int n_clusters,
                               wi_decode_layout* layout_out) {
  if (layout_out == nullptr) return WI_ERR_INVALID_ARG;
  return decode_layout(p, n_clusters, layout_out);
}

int wi_decode_score(const wi_decode_params* p, const void* q, const wi_index* index,
                    void* workspace, size_t workspace_bytes, wi_stream_t stream) {
  return run_decode(p, q, nullptr, nullptr, index, nullptr, nullptr, nullptr, workspace,
                    workspace_bytes, stream, wi::kStageScore, true, false);
}

int wi_decode_select(const wi_decode_params* p, const wi_index* index, int32_t* topk_ids,
                     void* workspace, size_t workspace_bytes, wi_stream_t stream) {
  return run_decode(p, nullptr, nullptr, nullptr, index, nullptr, nullptr, topk_ids, workspace,
                    workspace_bytes, stream, wi::kStageSelect, false, false);
}

int wi_decode_attend(const wi_decode_params* p, const void* q, const void* K, const void* V,
                     const wi_index* index, float* out, float* lse, void* workspace,
                     size_t workspace_bytes, wi_stream_t stream) {
  return run_decode(p, q, K, V, index, out, lse, nullptr, workspace, workspace_bytes, stream,
                    wi::kStageAttend, true, true);
}

int wi_decode_attention(const wi_decode_params* p, const void* q, const void* K, const void* V,
                        const wi_index* index, float* out, float* lse, int32_t* topk_ids,
                        void* workspace, size_t workspace_bytes, wi_stream_t stream) {
  return run_decode(p, q, K, V, index, out, lse, topk_ids, workspace, workspace_bytes, stream,
                    wi::kStageScore | wi::kStageSelect | wi::kStageAttend, true, true);
}

int wi_index_round_bf16(const wi_index* index, void* centroid_key_bf16, void* value_sum_bf16,
                        wi_stream_t stream) {
  if (index == nullptr || centroid_key_bf16 == nullptr || value_sum_bf16 == nullptr ||
      index->centroid_key == nullptr || index->value_sum == nullptr)
    return WI_ERR_INVALID_ARG;
  if (index->B <= 0 || index->Hkv <= 0 || index->n_clusters <= 0 || index->d != WI_HEAD_DIM)
    return WI_ERR_INVALID_ARG;
  if (!aligned(centroid_key_bf16, 16) || !aligned(value_sum_bf16, 16) ||
      !aligned(index->centroid_key, 16) || !aligned(index->value_sum, 16))
    return WI_ERR_ALIGNMENT;
  int st = device_ok();
  if (st != WI_OK) return st;
  const size_t n = (size_t)index->B * index->Hkv * index->n_clusters * WI_HEAD_DIM;
  const cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = wi::launch_round_bf16(index->centroid_key, static_cast<uint16_t*>(centroid_key_bf16), n, s);
  if (e == cudaSuccess)
    e = wi::launch_round_bf16(index->value_sum, static_cast<uint16_t*>(value_sum_bf16), n, s);
  return cuda_status(e);
}

int wi_decode_attention_ex(const wi_decode_params* p, const wi_decode_options* options,
                           const void* q, const void* K, const void* V, const wi_index* index,
                           float* out, float* lse, int32_t* topk_ids, void* workspace,
                           size_t workspace_bytes, wi_stream_t stream) {
  return run_decode(p, q, K, V, index, out, lse, topk_ids, workspace, workspace_bytes, stream,
                    wi::kStageScore | wi::kStageSelect | wi::kStageAttend, true, true, options);
}

int wi_sync_status(void* workspace, wi_stream_t stream, int* device_status) {
  if (workspace == nullptr || device_status == nullptr) return WI_ERR_INVALID_ARG;
  const cudaStream_t s = (cudaStream_t)stream;
  int host = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&host, workspace, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    *device_status = WI_ERR_CUDA;
    return WI_ERR_CUDA;
  }
  *device_status = host;
  return WI_OK;
}

const char* wi_status_string(int status) {
  switch (status) {
    case WI_OK: return "ok";
    case WI_ERR_INVALID_ARG: return "invalid argument";
    case WI_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case WI_ERR_LAUNCH: return "kernel launch failed";
    case WI_ERR_INDEX_MISMATCH: return "parameters do not match the index";
    case WI_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case WI_ERR_WORKSPACE: return "workspace too small";
    case WI_ERR_ALIGNMENT: return "pointer not aligned";
    case WI_ERR_CUDA: return "CUDA error on the stream";
    default: return "unknown status";
  }
}

int wi_debug_inject(int flags) {
  g_inject.store(flags & 1);
  return WI_OK;
}

const char* wi_version(void) { return "0.1.0"; }

}  // extern "C"
