// Decode kernel of the wave-index tripartite attention ("RetroInfer: A Vector
// Storage Engine for Scalable Long-Context LLM Inference", technical summary
// (es) §2.A: steady zone, retrieval zone, estimation zone; technical summary
// (ar) §2.a: estimation from the centroids and the value sum, §2.b: retrieved
// KV laid out contiguously for the attention kernel).
//
// One persistent launch, one block per SM.  Each block has 16 consumer warps,
// one producer warp and one signaling warp.  The producer streams every byte
// the block reads through a 4-stage ring of 32 KB shared-memory stages with
// the bulk-copy (TMA) engine; each consumer warp waits on a stage's mbarrier
// itself, copies its 4 rows into registers, releases the stage and computes,
// so no block-wide barrier sits inside a streaming loop.
//
// Work of block b, in order:
//   1. for each round: its chunk of index tiles (64 clusters of one KV group
//      per tile, consecutive tiles, chunk j = round * nb + b):
//        a. centroid-key tiles: s[b,h,c] = scale q_h . kbar_c (-inf if empty)
//           for the group's G query heads -> scores (global) and a copy of
//           the block's own scores in shared memory;
//        b. the selections assigned to this block and round: once the head's
//           KV group is fully scored, the r largest ranking keys (ties to the
//           lower id), their clusters' sorted rows, sizes, token offsets and
//           scores;
//        c. value-sum tiles of the same clusters: the estimate of every
//           non-empty cluster from the block's own scores,
//           (m, l = sum n_c e^{s_c - m}, o = sum e^{s_c - m} vsum_c), one
//           partial per (chunk, KV group, query head);
//      with few heads over several rounds (a.kbar_first) the centroid-key
//      tiles of every round come first, then every selection, then the
//      value-sum tiles (last round first; earlier rounds' scores are read
//      back from global memory);
//   2. its steady-zone tiles (sink and local-window K/V rows of one KV group,
//      the group's G query heads at once), exact attention, one partial per
//      (tile, head);
//   3. its share of the retrieved tokens: once every selection is published,
//      all heads' retrieved tokens, in head order and within a head in
//      cluster-id order, are split into contiguous ranges, one per block,
//      weighted so that each block's total streamed bytes are about equal.
//      A retrieved token i of cluster c enters with the weight
//      e^{l_i} - e^{s_c}: its exact term minus its share of the cluster's
//      estimate, so that "estimate of every cluster" + "retrieved tokens" is
//      the estimate of the clusters outside the retrieval set plus the exact
//      attention of its members.  Every warp keeps its own softmax state; at
//      the end of a head's range the last warp to finish combines the 16
//      states into one partial;
//   4. the merges of heads b, b + nb, ...: once every partial of the head is
//      published, the log-sum-exp combine of all of them into out and lse.
//
// There is no grid-wide barrier: a consumer of another block's results waits
// (bounded) on a counter of exactly what it reads -- a KV group's scored
// tiles, the number of published selections, a head's published partials.
// The signaling warp publishes the block's results (one gpu-scope fence per
// batch, then the counter atomics) off the consumers' path.  Every wait is
// bounded (kWaitLimitNs) and reports WI_ERR_DEVICE_TIMEOUT; a block that gives
// up lets its issued copies land before it exits.  Block-wide barriers occur
// only at points fixed by the static schedule, which every consumer warp
// passes whether or not a wait of it gave up.
//
// Every staged byte is read once per call, so the copies carry an L2
// evict-first policy.  Softmax quantities are kept in log2 units (logits
// scaled by log2 e) so that every exponential is an exp2.
//
// Options (wi_decode_options): the ranking key may be the attention mass
// s_c + ln n_c; a KV group may reuse the previous step's sets while its
// queries stay within cosine tau of the previous ones; one set may be
// shared by a group (chosen on the summed keys); the index statistics may be
// read as bf16 (two tiles per stage).
#include <float.h>
#include <limits.h>
#include <stddef.h>

#include "wi_device.cuh"
#include "wi_internal.h"

namespace wi {

namespace {

constexpr int kCW = 16;                        // consumer warps
constexpr int kCT = kCW * 32;                  // consumer threads
constexpr int kThreads = kCT + 64;             // + producer warp + signaling warp
constexpr int kStages = 4;
constexpr int kTile = kDecodeTile;             // index rows or tokens per tile
constexpr uint32_t kStageBytes = kTile * 512;  // 64 f32 rows, or 64 K + 64 V bf16 rows
constexpr int kQSlotBytes = 8 * kD * 2;        // up to 8 bf16 query rows
constexpr int kSlots = kStages + 1;            // retrieval pieces in flight (see consumers)
constexpr int kBins = 1024;                    // selection histogram
constexpr int kCand = 256;                     // selection candidates ranked exactly
constexpr int kSelChunk = kCT * 16;            // keys per register chunk (16 per thread)
constexpr int kPubSlots = 32;
static_assert(kSlots >= kStages + 1, "a warp may run kStages tiles ahead of the slowest");

enum : int { kTileRet = 1, kTileEnd = 2 };

// With a bf16 index a stage carries tiles i and i + 1 of chunk j (n tiles)
// when both exist and belong to one KV group; producer and consumers pair
// tiles by this rule.
__device__ __forceinline__ bool pair_tiles(const DecodeArgs& a, int j, int i, int n) {
  return a.kbar16 != nullptr && i + 1 < n && (j * a.Q + i + 1) % a.tpg != 0;
}

// Retrieval tile description, written by the producer with the tile.
struct TileInfo {
  int kind;
  int bh;     // query head (b*Hq + h)
  int ntok;   // tokens staged
  int last;   // the block's range of this head ends with this tile
};

// One warp's softmax state of a retrieval piece.
struct WarpPart {
  float m, l;
  float pad[2];
  float o[kD];
};

// A request to the signaling warp: after a gpu-scope fence covering every
// write made before the request was queued, add `val` to the n counters
// cnt[0..n).
struct PubReq {
  unsigned* cnt;
  unsigned val;
  int n;
  int ready;  // sequence number + 1 once the entry is written
  int pad;
};

struct __align__(128) DecSmem {
  unsigned char ring[kStages][kStageBytes];  // bulk-copy destinations
  unsigned char qs[kStages][kQSlotBytes];    // query rows staged with a tile
  union __align__(16) {
    int n[2 * kTile];  // index tiles: cluster sizes (two tiles per stage with a bf16 index)
    float s[kTile];    // retrieval tiles: the cluster score of each token (log2 units)
  } side[kStages];
  union __align__(16) {
    struct {
      float sc[kChunkMax][kCW][32];  // the block's scores of its chunk, per warp and lane
      int n[kChunkMax][kCW][4];      // sizes of the warp's rows
    } chunk;
    WarpPart slot[kSlots][kCW];      // retrieval pieces: per-warp states
  } a;
  union __align__(16) {
    struct {
      float o[kCW][4][kD];
      float m[kCW][4];
      float l[kCW][4];
    } comb;
    struct {
      uint32_t key[16][kCT];  // keys of the first 8192 clusters: id 16 t + j at [j][t]
      int hist[kBins];
      unsigned long long cand[kCand];
      int ncand;
      int res[4];
      float cosv[8];  // query cosines of the group (speculative reuse)
    } sel;
    struct {
      int rb[kMaxBlocks];  // blocks holding a retrieval piece of the head
      float w[32];
      float wl[4];
      int cnt[kCW];
      float red[3 * kD];
    } merge;
  } u;
  unsigned long long full[kStages];
  unsigned long long empty[kStages];
  TileInfo info[kStages];
  int bnd[kMaxBlocks + 1];  // token start of every block's retrieval range
  unsigned static_w[kMaxBlocks];  // copy of the blocks' static work
  unsigned slot_cnt[kSlots];
  int2 scan[2][kCW];
  uint32_t red_u[6][kCW];
  float red_f[2][kCW];
  int abort;      // some wait of this block gave up
  int issued;     // tiles whose copies the producer issued
  int flag;
  PubReq pub[kPubSlots];
  int pub_claim;  // requests claimed (consumers)
  int pub_done;   // requests published (signaling warp)
  int cons_done;  // the consumers queue no more requests
  int sig_done;   // the signaling warp has finished
};
static_assert(offsetof(DecSmem, qs) % 16 == 0, "bulk-copy alignment");
static_assert(offsetof(DecSmem, side) % 16 == 0, "bulk-copy alignment");
static_assert(offsetof(DecSmem, a) % 16 == 0, "float4 alignment");
static_assert(offsetof(DecSmem, u) % 16 == 0, "float4 alignment");
static_assert(offsetof(DecSmem, full) % 8 == 0, "mbarrier alignment");
static_assert(sizeof(WarpPart) % 16 == 0, "float4 alignment");
static_assert(sizeof(DecSmem) <= 227 * 1024, "dynamic shared memory per block");

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Named barrier 1 over the 512 consumer threads.
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
// Named barrier 1 with an OR-reduction of a predicate over the consumers.
__device__ __forceinline__ bool cany(bool x) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 512, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)x)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ uint2 lds2(const void* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ float4 bf4(uint2 w) {
  return make_float4(bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y));
}
__device__ __forceinline__ uint32_t score_key(float s) {
  return (s == -INFINITY) ? 0u : float_key(s);  // 0 <=> empty cluster
}

__device__ __forceinline__ void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void st_release_cta(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_cta(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}
__device__ __forceinline__ unsigned atom_add_release_cta(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.release.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(smem_addr(p)), "r"(v)
               : "memory");
  return old;
}
__device__ __forceinline__ void fence_acq_cta() { asm volatile("fence.acq_rel.cta;" ::: "memory"); }
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Bounded wait until *cnt >= target; gives up early once *abort is set.
__device__ __noinline__ bool count_wait(const unsigned* cnt, unsigned target, int* status,
                                        const int* abort) {
  if (ld_acquire(cnt) >= target) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    __nanosleep(64);
    if (ld_acquire(cnt) >= target) return true;
    if (*(volatile const int*)abort) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      report(status, WI_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}
// Bounded wait of one warp (every lane polls) for a ring stage's phase; gives
// up early once *abort is set.  Warp-uniform result.
__device__ __forceinline__ bool stage_wait(uint32_t bar, uint32_t parity, int* status, int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*(volatile int*)abort) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      report(status, WI_ERR_DEVICE_TIMEOUT);
      *(volatile int*)abort = 1;
      return false;
    }
  }
}

// Reduce-scatter of V = 4G per-lane values: afterwards lane L holds the sum
// over all 32 lanes of value index (L mod V).
template <int V>
__device__ __forceinline__ float reduce_scatter(float (&v)[V], int lane) {
#pragma unroll
  for (int off = V / 2; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, off);
    }
  }
  float x = v[0];
#pragma unroll
  for (int off = V; off < 32; off <<= 1) x += __shfl_xor_sync(kFull, x, off);
  return x;
}

// Exclusive scan of an int2 over the 512 consumers; *total gets the sum.  One
// named barrier: the two halves of S.scan alternate between calls (`buf`),
// and every call's barrier separates a half's reads from its next write.
__device__ int2 cscan2(int2 v, DecSmem& S, int2* total, int& buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int2 incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(kFull, incl.x, o);
    const int y = __shfl_up_sync(kFull, incl.y, o);
    if (lane >= o) {
      incl.x += x;
      incl.y += y;
    }
  }
  int2* sh = S.scan[buf];
  buf ^= 1;
  if (lane == 31) sh[warp] = incl;
  csync();
  int2 base = make_int2(0, 0), tot = make_int2(0, 0);
#pragma unroll
  for (int w = 0; w < kCW; ++w) {
    const int2 t = sh[w];
    if (w < warp) {
      base.x += t.x;
      base.y += t.y;
    }
    tot.x += t.x;
    tot.y += t.y;
  }
  *total = tot;
  return make_int2(base.x + incl.x - v.x, base.y + incl.y - v.y);
}

// Queue a request to the signaling warp (any consumer thread).  The writes it
// publishes must be ordered before the call: by a barrier, or by this thread.
__device__ void publish(DecSmem& S, const DecodeArgs& a, unsigned* cnt, unsigned val, int n) {
  const int t = (int)atomicAdd(reinterpret_cast<unsigned*>(&S.pub_claim), 1u);
  if (t - ld_acquire_cta(&S.pub_done) >= kPubSlots) {  // ring full: wait (bounded)
    const unsigned long long t0 = global_ns();
    while (t - ld_acquire_cta(&S.pub_done) >= kPubSlots) {
      if (global_ns() - t0 > kWaitLimitNs) {
        report(a.status, WI_ERR_DEVICE_TIMEOUT);
        *(volatile int*)&S.abort = 1;
        return;  // the entry stays unwritten; the signaling warp gives up on it
      }
      __nanosleep(32);
    }
  }
  PubReq& q = S.pub[t % kPubSlots];
  q.cnt = cnt;
  q.val = val;
  q.n = n;
  st_release_cta(&q.ready, t + 1);
}

// Combine the 16 consumer warps' states of nh <= 4 heads into partials:
// dst(h)[0] = m (log2 units), dst(h)[1] = l, dst(h)[2..] = o.  m[h] is
// warp-uniform, l[h] valid in every lane, o[h] this lane's 4 dimensions.
// Two barriers; afterwards the partials may be published.
template <int NH>
__device__ void combine_write(DecSmem& S, const float (&m)[NH], const float (&l)[NH],
                              const float4 (&o)[NH], float* const (&dst)[NH]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  static_assert(NH <= 4, "four heads per pass");
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    if (lane == 0) {
      S.u.comb.m[warp][h] = m[h];
      S.u.comb.l[warp][h] = l[h];
    }
    reinterpret_cast<float4*>(S.u.comb.o[warp][h])[lane] = o[h];
  }
  csync();
  if (tid < NH * kD) {
    const int h = tid / kD, d = tid % kD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCW; ++w) M = fmaxf(M, S.u.comb.m[w][h]);
    float L = 0.f, O = 0.f;
    if (M > -INFINITY) {
#pragma unroll
      for (int w = 0; w < kCW; ++w) {
        const float mw = S.u.comb.m[w][h];
        const float f = mw > -INFINITY ? exp2f(mw - M) : 0.f;
        L += S.u.comb.l[w][h] * f;
        O += S.u.comb.o[w][h][d] * f;
      }
    }
    float* p = dst[0];
#pragma unroll
    for (int hh = 1; hh < NH; ++hh)
      if (h == hh) p = dst[hh];
    if (d == 0) {
      p[0] = M;
      p[1] = L;
    }
    p[2 + d] = O;
  }
  csync();
}

// ---------------------------------------------------------------------------
// selection of one query head, common case (all 512 consumers)
// ---------------------------------------------------------------------------
// The same set as the general path below, in three passes over the ranking
// values v (the score, or s_c + ln n_c; -inf = empty cluster).  Thread t holds
// the values of ids 16 t .. 16 t + 15 of the first 8192 clusters in
// registers; further clusters are re-read at every pass.
//   A. count, smallest and largest value (and the largest score);
//   B. a histogram of kBins bins linear in v between them (monotone in v);
//      a scan from the top gives the bin b* holding the r_eff-th largest;
//   C. ids in bins above b* are marked in a bitmap of the ids; b*'s values
//      are ranked exactly by (v desc, id asc) and the best `need` marked;
//   then the bitmap, read in id order, gives the ids in ascending order.
// Returns the number selected, or -1 (nothing written) when b* holds more
// than kCand values or the ids do not fit the bitmap: the general path then
// takes over.
__device__ int select_fast(const DecodeArgs& a, DecSmem& S, const float* sc, const int* sz,
                           bool mass, float* hm_out, int* ids, int* topk) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = a.C, r = a.r;
  const int nch = (C + kSelChunk - 1) / kSelChunk;
  const int nwords = (C + 31) / 32;
  if (nwords > 16 * kCT) return -1;  // the bitmap lives in S.u.sel.key
  uint32_t* bits = &S.u.sel.key[0][0];
  const bool vec = (C & 3) == 0;
  float smx = -INFINITY;  // largest score (differs from the largest v when ranking by mass)
  auto mval = [](float s, int n) { return n > 0 ? s + logf((float)n) : -INFINITY; };
  // values of chunk ch for this thread
  auto load = [&](int ch, float (&x)[16]) {
    const int c0 = ch * kSelChunk + tid * 16;
    if (vec && c0 + 16 <= C) {
      const float4* p = reinterpret_cast<const float4*>(sc + c0);
      float4 f[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) f[j] = __ldcg(p + j);
      if (mass) {
        const int4* pn = reinterpret_cast<const int4*>(sz + c0);
        int4 n[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) n[j] = __ldg(pn + j);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          smx = fmaxf(smx, fmaxf(fmaxf(f[j].x, f[j].y), fmaxf(f[j].z, f[j].w)));
          x[4 * j] = mval(f[j].x, n[j].x);
          x[4 * j + 1] = mval(f[j].y, n[j].y);
          x[4 * j + 2] = mval(f[j].z, n[j].z);
          x[4 * j + 3] = mval(f[j].w, n[j].w);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          x[4 * j] = f[j].x;
          x[4 * j + 1] = f[j].y;
          x[4 * j + 2] = f[j].z;
          x[4 * j + 3] = f[j].w;
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        x[j] = -INFINITY;
        if (c0 + j < C) {
          const float s = __ldcg(sc + c0 + j);
          smx = fmaxf(smx, s);
          x[j] = mass ? mval(s, __ldg(sz + c0 + j)) : s;
        }
      }
    }
  };
  // lean block scan: exclusive prefix and total of x over the 512 consumers
  auto bscan = [&](int x, int2* sh, int& total) {
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sh[warp].x = incl;
    csync();
    const int wt = sh[lane & (kCW - 1)].x;
    int wincl = wt;
#pragma unroll
    for (int o = 1; o < kCW; o <<= 1) {
      const int y = __shfl_up_sync(kFull, wincl, o);
      if ((lane & (kCW - 1)) >= o) wincl += y;
    }
    total = __shfl_sync(kFull, wincl, kCW - 1);
    return __shfl_sync(kFull, wincl - wt, warp) + incl - x;
  };

  // A. count and range; the histogram and the bitmap are cleared meanwhile
  float v[16];
  load(0, v);
  int cnt = 0;
  float vmax = -INFINITY, vmin = INFINITY;
  auto tally = [&](const float (&x)[16]) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const bool ok = x[j] > -INFINITY;
      cnt += (int)ok;
      vmax = ok ? fmaxf(vmax, x[j]) : vmax;
      vmin = ok ? fminf(vmin, x[j]) : vmin;
    }
  };
  tally(v);
  for (int ch = 1; ch < nch; ++ch) {
    float x[16];
    load(ch, x);
    tally(x);
  }
  if (!mass) smx = vmax;
  for (int i = tid; i < kBins; i += kCT) S.u.sel.hist[i] = 0;
  for (int i = tid; i < nwords; i += kCT) bits[i] = 0u;
  if (tid == 0) S.u.sel.ncand = 0;
  {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      cnt += __shfl_xor_sync(kFull, cnt, o);
      vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, o));
      vmin = fminf(vmin, __shfl_xor_sync(kFull, vmin, o));
      smx = fmaxf(smx, __shfl_xor_sync(kFull, smx, o));
    }
    if (lane == 0) {
      S.red_u[0][warp] = (uint32_t)cnt;
      S.red_u[1][warp] = __float_as_uint(vmax);
      S.red_u[2][warp] = __float_as_uint(vmin);
      S.red_u[3][warp] = __float_as_uint(smx);
    }
    csync();
    const int w = lane & (kCW - 1);
    cnt = (int)S.red_u[0][w];
    vmax = __uint_as_float(S.red_u[1][w]);
    vmin = __uint_as_float(S.red_u[2][w]);
    smx = __uint_as_float(S.red_u[3][w]);
#pragma unroll
    for (int o = kCW / 2; o > 0; o >>= 1) {
      cnt += __shfl_xor_sync(kFull, cnt, o);
      vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, o));
      vmin = fminf(vmin, __shfl_xor_sync(kFull, vmin, o));
      smx = fmaxf(smx, __shfl_xor_sync(kFull, smx, o));
    }
  }
  const int r_eff = min(r, cnt);
  if (tid == 0 && hm_out) *hm_out = cnt > 0 ? smx : -INFINITY;
  if (r_eff == 0) return 0;

  // B. histogram and boundary bin (skipped when every valid id is taken)
  const float inv = (vmax > vmin) ? (float)kBins / (vmax - vmin) : 0.f;
  auto binf = [&](float x) { return min((int)((x - vmin) * inv), kBins - 1); };
  int bstar = -1, need = 0;
  if (r_eff < cnt) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (v[j] > -INFINITY) atomicAdd(&S.u.sel.hist[binf(v[j])], 1);
    for (int ch = 1; ch < nch; ++ch) {
      float x[16];
      load(ch, x);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (x[j] > -INFINITY) atomicAdd(&S.u.sel.hist[binf(x[j])], 1);
    }
    csync();
    // thread t owns bins kBins-1-2t and kBins-2-2t (counted from the top)
    const int b_hi = kBins - 1 - 2 * tid;
    const int c1 = S.u.sel.hist[b_hi], c2 = S.u.sel.hist[b_hi - 1];
    int tot;
    const int above = bscan(c1 + c2, S.scan[0], tot);
    if (above < r_eff && r_eff <= above + c1) {
      S.u.sel.res[0] = b_hi;
      S.u.sel.res[1] = r_eff - above;
      S.u.sel.res[2] = c1;
    } else if (above + c1 < r_eff && r_eff <= above + c1 + c2) {
      S.u.sel.res[0] = b_hi - 1;
      S.u.sel.res[1] = r_eff - above - c1;
      S.u.sel.res[2] = c2;
    }
    csync();
    bstar = S.u.sel.res[0];
    need = S.u.sel.res[1];
    if (S.u.sel.res[2] > kCand) return -1;  // crowded bin: the general path
  }

  // C. mark the ids above b*, collect b*'s values (every valid id when bstar < 0)
  auto mark = [&](int ch, const float (&x)[16]) {
    uint32_t m = 0u;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (!(x[j] > -INFINITY)) continue;
      const int b = bstar < 0 ? kBins : binf(x[j]);
      if (b > bstar) {
        m |= 1u << j;
      } else if (b == bstar) {
        const int p = atomicAdd(&S.u.sel.ncand, 1);  // p < kCand: the bin holds <= kCand
        const uint32_t id = (uint32_t)(ch * kSelChunk + tid * 16 + j);
        S.u.sel.cand[p] = ((unsigned long long)score_key(x[j]) << 32) |
                          (unsigned long long)(0xffffffffu - id);
      }
    }
    if (m) atomicOr(&bits[ch * (kSelChunk / 32) + (tid >> 1)], m << ((tid & 1) * 16));
  };
  mark(0, v);
  for (int ch = 1; ch < nch; ++ch) {
    float x[16];
    load(ch, x);
    mark(ch, x);
  }
  csync();
  if (bstar >= 0) {
    // the best `need` of b*'s values: ranked by (value desc, id asc)
    const int nc = S.u.sel.ncand;
    if (tid < nc) {
      const unsigned long long mine = S.u.sel.cand[tid];
      int rank = 0;
      for (int j = 0; j < nc; ++j) rank += (int)(S.u.sel.cand[j] > mine);
      if (rank < need) {
        const uint32_t id = 0xffffffffu - (uint32_t)mine;
        atomicOr(&bits[id >> 5], 1u << (id & 31));
      }
    }
    csync();
  }

  // the marked ids in ascending order: thread t reads words [t k, t k + k)
  const int kw = (nwords + kCT - 1) / kCT;
  const int w0 = tid * kw, w1 = min(w0 + kw, nwords);
  int n = 0;
  for (int w = w0; w < w1; ++w) n += __popc(bits[w]);
  int tot;
  int pos = bscan(n, S.scan[1], tot);
  for (int w = w0; w < w1; ++w) {
    uint32_t m = bits[w];
    while (m) {
      const int id = w * 32 + __ffs(m) - 1;
      m &= m - 1;
      if (pos < r) {
        ids[pos] = id;
        if (topk) topk[pos] = id;
      }
      ++pos;
    }
  }
  return min(tot, r);  // == r_eff
}

// ---------------------------------------------------------------------------
// selection of one query head (all 512 consumers)
// ---------------------------------------------------------------------------
// T = the r_eff = min(r, non-empty) largest ranking keys, ties to the lower
// id.  The ranking key is the score s_c, or with a.rank_mass the estimated
// attention mass n_c e^{s_c}, compared as s_c + ln n_c (the attention-aware
// index of technical summary (ar) §2.a).  Keys are order-preserving images of
// these values (0 = empty cluster).  The keys of the first 8192 clusters are
// kept in shared memory (thread t holds ids 16 t .. 16 t + 15); the rest are
// re-read from the scores at every pass.
//   0. speculative reuse (FreeKV technical summary §2.A): with a.prev_q set,
//      the group's smallest cosine between a query and its previous query;
//      if it is at least a.tau, T is the previous step's set for this head
//      (a.prev_topk row) and steps 1-3 are skipped;
//   1. count, smallest and largest key;
//   2. a histogram of 1024 bins linear in the score between the smallest and
//      largest score (monotone in the score, so few keys share a bin) gives
//      the bin holding the r_eff-th largest key;
//   3. that bin's keys (normally a few) are ranked exactly by (key desc, id
//      asc); the r_eff-th overall gives the threshold (Kb, cb): a cluster is
//      selected iff its key k and id c satisfy k > Kb, or k == Kb and c <= cb.
//      A bin of more than 256 keys is narrowed by histograms of its key range
//      until it holds at most 256 keys, or a single key value whose lowest
//      ids are then taken;
//   4. the selected ids are written in id order; then every selected
//      cluster's size, first sorted row and score are loaded in one round and
//      a scan of the sizes gives the token offsets.
// Steps 1-3 and the marking of step 4 run only when select_fast gives up.
// Returns the number selected.
__device__ int select_head(const DecodeArgs& a, DecSmem& S, int bh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bg = bh / a.G;
  const int C = a.C, r = a.r, rs = r > 0 ? r : 1;
  // shared selection: bh is the group's first head and the set is chosen on
  // the group's summed ranking keys (written to a.grp_vals below), then
  // recorded for every head of the group
  const bool shared = a.share != 0;
  const int nh = shared ? a.G : 1;
  const float* sc = shared ? a.grp_vals + (size_t)bg * C : a.scores + (size_t)bh * C;
  const int* sz = a.size + (size_t)bg * C;
  const int* off = a.offset + (size_t)bg * (C + 1);
  const int nch = (C + kSelChunk - 1) / kSelChunk;
  const bool vec = (C & 3) == 0;  // rows of scores and sizes start on 16-byte boundaries
  const bool mass = a.rank_mass != 0 && !shared;  // the group row holds the mass keys already
  int buf = 0;

  // ranking key of the mass order: s_c + ln n_c (0 for an empty cluster)
  auto mass_key = [](float sv, int n) { return n > 0 ? score_key(sv + logf((float)n)) : 0u; };
  // keys of chunk ch for this thread, in groups of four: f(key, id)
  auto chunk_keys = [&](int ch, auto&& f) {
    const int c0 = ch * kSelChunk + tid * 16;
    if (vec && c0 + 16 <= C) {
      const float4* p = reinterpret_cast<const float4*>(sc + c0);
      float4 v[4];  // all four loads in flight before any key is used
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = __ldcg(p + j);
      if (mass) {
        const int4* pn = reinterpret_cast<const int4*>(sz + c0);
        int4 n[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) n[j] = __ldg(pn + j);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          f(mass_key(v[j].x, n[j].x), c0 + 4 * j);
          f(mass_key(v[j].y, n[j].y), c0 + 4 * j + 1);
          f(mass_key(v[j].z, n[j].z), c0 + 4 * j + 2);
          f(mass_key(v[j].w, n[j].w), c0 + 4 * j + 3);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          f(score_key(v[j].x), c0 + 4 * j);
          f(score_key(v[j].y), c0 + 4 * j + 1);
          f(score_key(v[j].z), c0 + 4 * j + 2);
          f(score_key(v[j].w), c0 + 4 * j + 3);
        }
      }
    } else {
#pragma unroll 4
      for (int j = 0; j < 16; ++j) {
        uint32_t k = 0u;
        if (c0 + j < C) {
          const float sv = __ldcg(sc + c0 + j);
          k = mass ? mass_key(sv, __ldg(sz + c0 + j)) : score_key(sv);
        }
        f(k, c0 + j);
      }
    }
  };
  // f(key, id) over every key: chunk 0 from shared memory
  auto visit = [&](auto&& f) {
#pragma unroll 4
    for (int j = 0; j < 16; ++j) f(S.u.sel.key[j][tid], tid * 16 + j);
    for (int ch = 1; ch < nch; ++ch) chunk_keys(ch, f);
  };
  // block sum, key extrema and a second maximum (one barrier)
  auto block_count_range = [&](int& cnt, uint32_t& kmx, uint32_t& kmn, uint32_t& mx2) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      cnt += __shfl_xor_sync(kFull, cnt, o);
      kmx = max(kmx, __shfl_xor_sync(kFull, kmx, o));
      kmn = min(kmn, __shfl_xor_sync(kFull, kmn, o));
      mx2 = max(mx2, __shfl_xor_sync(kFull, mx2, o));
    }
    int2* sh = S.scan[buf];
    uint32_t(*ru)[kCW] = buf ? &S.red_u[3] : &S.red_u[0];
    buf ^= 1;
    if (lane == 0) {
      sh[warp] = make_int2(cnt, 0);
      ru[0][warp] = kmx;
      ru[1][warp] = kmn;
      ru[2][warp] = mx2;
    }
    csync();
    cnt = 0;
    kmx = 0u;
    kmn = 0xffffffffu;
    mx2 = 0u;
#pragma unroll
    for (int w = 0; w < kCW; ++w) {
      cnt += sh[w].x;
      kmx = max(kmx, ru[0][w]);
      kmn = min(kmn, ru[1][w]);
      mx2 = max(mx2, ru[2][w]);
    }
  };

  const int rsel0 = bh * rs;
  int* ids = a.sel_ids + rsel0;

  // 0. speculative reuse: the group's smallest query cosine against tau
  bool reuse = false;
  int n_reuse = 0;
  if (a.prev_q != nullptr && r > 0) {
    if (warp < a.G) {
      const size_t row = ((size_t)bg * a.G + warp) * kD + lane * 4;
      const float4 x = bf4(__ldg(reinterpret_cast<const uint2*>(a.q + row)));
      const float4 y = bf4(__ldg(reinterpret_cast<const uint2*>(a.prev_q + row)));
      float dot = x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
      float xx = x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
      float yy = y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        dot += __shfl_xor_sync(kFull, dot, o);
        xx += __shfl_xor_sync(kFull, xx, o);
        yy += __shfl_xor_sync(kFull, yy, o);
      }
      if (lane == 0)
        S.u.sel.cosv[warp] = (xx > 0.f && yy > 0.f) ? dot / (sqrtf(xx) * sqrtf(yy)) : 0.f;
    }
    csync();
    float cmin = S.u.sel.cosv[0];
    for (int h = 1; h < a.G; ++h) cmin = fminf(cmin, S.u.sel.cosv[h]);
    if (cmin >= a.tau) {
      // the previous row: strictly ascending ids in [0, C), then -1 padding
      const int* prv = a.prev_topk + (size_t)bh * r;
      int n = 0, bad = 0;
      for (int i = tid; i < r; i += kCT) {
        const int x = __ldcg(prv + i);
        if (x >= 0) {
          const int y = i > 0 ? __ldcg(prv + i - 1) : -1;
          bad |= (int)(x >= C || (i > 0 && (y < 0 || y >= x)));
          ids[i] = x;
          ++n;
        } else {
          bad |= (int)(x != -1);
        }
      }
      int2 tot;
      cscan2(make_int2(n, bad), S, &tot, buf);
      if (tot.y != 0) {
        if (tid == 0) report(a.status, WI_ERR_INVALID_ARG);  // not a retrieval set: select
      } else {
        reuse = true;
        n_reuse = tot.x;
      }
    }
  }
  if (tid < nh && a.reused != nullptr) a.reused[bh + tid] = reuse ? 1 : 0;
  if (shared) {
    // the group row v_c = sum_h key_h(c) and every head's largest score
    const float* s0 = a.scores + (size_t)bh * C;
    float hm[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) hm[h] = -INFINITY;
    for (int c = tid; c < C; c += kCT) {
      const int n = __ldg(sz + c);
      const float lg = (a.rank_mass && n > 0) ? logf((float)n) : 0.f;
      float v = 0.f;
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        if (h < nh) {
          const float sv = __ldcg(s0 + (size_t)h * C + c);
          hm[h] = fmaxf(hm[h], sv);
          v += sv + lg;
        }
      }
      a.grp_vals[(size_t)bg * C + c] = n > 0 ? v : -INFINITY;
    }
    float* red = reinterpret_cast<float*>(S.u.sel.hist);  // [8][kCW] partial maxima
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      float x = hm[h];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, o));
      if (lane == 0) red[h * kCW + warp] = x;
    }
    csync();
    if (tid < nh) {
      float x = -INFINITY;
      for (int w = 0; w < kCW; ++w) x = fmaxf(x, red[tid * kCW + w]);
      a.head_max[bh + tid] = x;
    }
    csync();  // the group row is written; the partial maxima are read
  }
  int* topk = (a.topk_out && !shared) ? a.topk_out + (size_t)bh * r : nullptr;
  const int n_fast =
      reuse ? -1 : select_fast(a, S, sc, sz, mass, shared ? nullptr : a.head_max + bh, ids, topk);
  const bool general = !reuse && n_fast < 0;

  // 1. keys of the first chunk into shared memory; count and key range; the
  // largest score (the head's maximum) separately when the keys are not the
  // scores or are not visited
  int valid = 0;
  uint32_t kmax = 0u, kmin = 0xffffffffu, smax = 0u;
  auto tally = [&](uint32_t k, int) {
    valid += (int)(k != 0u);
    kmax = max(kmax, k);
    kmin = min(kmin, k != 0u ? k : 0xffffffffu);
  };
  if (!shared && (reuse || (general && mass))) {
    for (int c = tid; c < C; c += kCT) smax = max(smax, score_key(__ldcg(sc + c)));
  }
  if (general) {
    chunk_keys(0, [&](uint32_t k, int id) {
      S.u.sel.key[id - tid * 16][tid] = k;
      tally(k, id);
    });
    for (int ch = 1; ch < nch; ++ch) chunk_keys(ch, tally);
    if (!mass) smax = kmax;
  }
  if (reuse || general) {
    block_count_range(valid, kmax, kmin, smax);
    if (tid == 0 && !shared) a.head_max[bh] = smax != 0u ? key_float(smax) : -INFINITY;
  }
  const int r_eff = reuse ? n_reuse : (general ? min(r, valid) : n_fast);

  // threshold (Kb, cb): selected iff k > Kb, or k == Kb and id <= cb
  uint32_t Kb = 0xffffffffu;
  int cb = -1;
  if (!general) {
    // T is the previous set, or select_fast's, already in ids
  } else if (r_eff > 0 && r_eff == valid) {
    Kb = 0u;  // every non-empty cluster
    cb = INT_MAX;
  } else if (r_eff > 0) {
    // 2. score-linear histogram: the bin of the r_eff-th largest key
    const float smin = key_float(kmin), smax = key_float(kmax);
    const float inv = (smax > smin) ? (float)kBins / (smax - smin) : 0.f;
    auto bin_of = [&](uint32_t k) {
      const float x = (key_float(k) - smin) * inv;
      return x < (float)(kBins - 1) ? (int)x : kBins - 1;
    };
    for (int i = tid; i < kBins; i += kCT) S.u.sel.hist[i] = 0;
    if (tid == 0) S.u.sel.ncand = 0;
    csync();
    visit([&](uint32_t k, int) {
      if (k != 0u) atomicAdd(&S.u.sel.hist[bin_of(k)], 1);
    });
    csync();
    // boundary bin: thread t owns the 2 bins kBins-2t-2 .. kBins-2t-1 (from the top)
    auto boundary = [&](int need_in) {
      const int b_hi = kBins - 2 * tid;
      const int c1 = S.u.sel.hist[b_hi - 1], c2 = S.u.sel.hist[b_hi - 2];
      int2 tot;
      const int above0 = cscan2(make_int2(c1 + c2, 0), S, &tot, buf).x;
      if (above0 < need_in && need_in <= above0 + c1) {
        S.u.sel.res[0] = b_hi - 1;
        S.u.sel.res[1] = above0;
        S.u.sel.res[2] = c1;
      } else if (above0 + c1 < need_in && need_in <= above0 + c1 + c2) {
        S.u.sel.res[0] = b_hi - 2;
        S.u.sel.res[1] = above0 + c1;
        S.u.sel.res[2] = c2;
      }
      csync();
    };
    boundary(r_eff);
    const int bstar = S.u.sel.res[0];
    int need = r_eff - S.u.sel.res[1];
    const int nbin = S.u.sel.res[2];
    // rank the keys of a narrow range exactly: composite (key << 32 | ~id),
    // larger first; the need-th is the threshold
    auto rank_exact = [&](auto&& in_range) {
      visit([&](uint32_t k, int id) {
        if (k != 0u && in_range(k)) {
          const int p = atomicAdd(&S.u.sel.ncand, 1);
          if (p < kCand)
            S.u.sel.cand[p] =
                ((unsigned long long)k << 32) | (unsigned long long)(0xffffffffu - (uint32_t)id);
        }
      });
      csync();
      const int nc = min(S.u.sel.ncand, kCand);
      if (tid < nc) {
        const unsigned long long mine = S.u.sel.cand[tid];
        int rank = 0;
        for (int j = 0; j < nc; ++j) rank += (int)(S.u.sel.cand[j] > mine);
        if (rank == need - 1) {
          S.u.sel.res[0] = (int)(uint32_t)(mine >> 32);
          S.u.sel.res[1] = (int)(0xffffffffu - (uint32_t)mine);
        }
      }
      csync();
      Kb = (uint32_t)S.u.sel.res[0];
      cb = S.u.sel.res[1];
    };
    if (nbin <= kCand) {
      rank_exact([&](uint32_t k) { return bin_of(k) == bstar; });
    } else {
      // 3'. a crowded bin (ties or a pathological spread): its key range, then
      // histograms of that range, kBins equal bins at a time
      int nb2 = 0;
      uint32_t lo = 0xffffffffu, hi = 0u, unused = 0u;
      visit([&](uint32_t k, int) {
        if (k != 0u && bin_of(k) == bstar) {
          lo = min(lo, k);
          hi = max(hi, k);
        }
      });
      block_count_range(nb2, hi, lo, unused);
      uint32_t span = hi - lo;
      for (int iter = 0; iter < 8; ++iter) {
        int shift = 0;
        while ((span >> shift) >= (uint32_t)kBins) ++shift;
        for (int i = tid; i < kBins; i += kCT) S.u.sel.hist[i] = 0;
        if (tid == 0) S.u.sel.ncand = 0;
        csync();
        {
          const uint32_t l0 = lo, sp = span;
          const int sh = shift;
          visit([&](uint32_t k, int) {
            if (k != 0u && k - l0 <= sp) atomicAdd(&S.u.sel.hist[(k - l0) >> sh], 1);
          });
        }
        csync();
        boundary(need);
        const int bs = S.u.sel.res[0], above = S.u.sel.res[1], nbn = S.u.sel.res[2];
        need -= above;
        const uint32_t bin_lo = lo + ((uint32_t)bs << shift);
        const uint32_t bin_span = min(span - ((uint32_t)bs << shift), (1u << shift) - 1u);
        if (nbn <= kCand) {
          const uint32_t l0 = bin_lo, sp = bin_span;
          rank_exact([&](uint32_t k) { return k - l0 <= sp; });
          break;
        }
        if (shift == 0 || bin_span == 0u) {
          // one key value: the `need` lowest ids holding it
          Kb = bin_lo;
          int eq_base = 0;
          for (int ch = 0; ch < nch; ++ch) {
            int ne = 0;
            auto cnt_eq = [&](uint32_t k, int) { ne += (k == bin_lo); };
            if (ch == 0) {
#pragma unroll 4
              for (int j = 0; j < 16; ++j) cnt_eq(S.u.sel.key[j][tid], 0);
            } else {
              chunk_keys(ch, cnt_eq);
            }
            int2 t2;
            const int before = eq_base + cscan2(make_int2(ne, 0), S, &t2, buf).x;
            eq_base += t2.x;
            if (before < need && need <= before + ne) {
              int x = before;
              auto find = [&](uint32_t k, int id) {
                if (k == bin_lo && ++x == need) S.u.sel.res[3] = id;
              };
              if (ch == 0) {
                for (int j = 0; j < 16; ++j) find(S.u.sel.key[j][tid], tid * 16 + j);
              } else {
                chunk_keys(ch, find);
              }
            }
          }
          csync();
          cb = S.u.sel.res[3];
          break;
        }
        lo = bin_lo;  // narrow to the boundary bin
        span = bin_span;
      }
    }
  }

  // 4. ids in ascending order, then each selected cluster's size, row, score
  int sel_base = 0;
  if (r_eff > 0 && general) {
    for (int ch = 0; ch < nch; ++ch) {
      uint32_t mask = 0u;
      int nsel = 0;
      auto mark = [&](uint32_t k, int id) {
        if (k != 0u && (k > Kb || (k == Kb && id <= cb))) {
          mask |= 1u << (id & 15);
          ++nsel;
        }
      };
      if (ch == 0) {
#pragma unroll 4
        for (int j = 0; j < 16; ++j) mark(S.u.sel.key[j][tid], tid * 16 + j);
      } else {
        chunk_keys(ch, mark);
      }
      int2 tot;
      int pos = sel_base + cscan2(make_int2(nsel, 0), S, &tot, buf).x;
      sel_base += tot.x;
      const int c0 = ch * kSelChunk + tid * 16;
      while (mask) {
        const int j = __ffs(mask) - 1;
        mask &= mask - 1;
        if (pos < r) {
          ids[pos] = c0 + j;
          if (topk) topk[pos] = c0 + j;
        }
        ++pos;
      }
    }
  }
  const int nsel_tot = general ? min(sel_base, r) : r_eff;  // == r_eff
  csync();  // the ids are written (and visible to the block)
  // every head of the set (one, or the group's nh when shared): the same ids,
  // rows, sizes and token offsets, and the head's own scores
  const bool topk_here = a.topk_out != nullptr && (reuse || shared);
  const float* s_own = a.scores + (size_t)bh * C;
  int tok_base = 0;
  for (int i0 = 0; i0 < nsel_tot; i0 += kCT) {
    const int i = i0 + tid;
    int n = 0, row = 0, c = -1;
    float sv = -INFINITY;
    if (i < nsel_tot) {
      c = ids[i];
      n = __ldg(sz + c);
      row = __ldg(off + c);
      sv = __ldcg(s_own + c);
      if (n < 0 || row < 0 || (long long)row + n > a.N_idx) {
        report(a.status, WI_ERR_INDEX_MISMATCH);  // inconsistent index: stage nothing
        n = 0;
        row = 0;
      }
    }
    int2 tot;
    const int ex = cscan2(make_int2(n, 0), S, &tot, buf).x;
    if (i < nsel_tot) {
      for (int h = 0; h < nh; ++h) {
        const size_t o = (size_t)(bh + h) * rs + i;
        a.sel_ids[o] = c;
        a.sel_rows[o] = row;
        a.sel_cnts[o] = n;
        a.sel_pre[o] = tok_base + ex;
        a.sel_sc[o] = h == 0 ? sv : __ldcg(s_own + (size_t)h * C + c);
        if (topk_here) a.topk_out[(size_t)(bh + h) * r + i] = c;
      }
    }
    tok_base += tot.x;
  }
  for (int h = 0; h < nh; ++h) {
    for (int i = nsel_tot + tid; i < rs; i += kCT) {
      const size_t o = (size_t)(bh + h) * rs + i;
      a.sel_ids[o] = -1;
      a.sel_rows[o] = 0;
      a.sel_cnts[o] = 0;
      a.sel_pre[o] = tok_base;
      a.sel_sc[o] = -INFINITY;
      if (a.topk_out && i < r) a.topk_out[(size_t)(bh + h) * r + i] = -1;
    }
  }
  if (tid < nh) a.head_tok[bh + tid] = tok_base;
  csync();  // the selection is complete after this barrier
  return nsel_tot;
}

// ---------------------------------------------------------------------------
// merge of one query head (all 512 consumers)
// ---------------------------------------------------------------------------
// Partials: the estimate pieces of its KV group (every non-empty cluster),
// its steady pieces and its retrieval pieces (exact tokens minus their
// clusters' estimate).  out = O / L, lse = (M + log2 L) ln 2.  The partials
// are loaded in rounds of 32 independent loads per thread.
__device__ void merge_head(const DecodeArgs& a, DecSmem& S, int bh, int n_est, int e_lo,
                           int n_ret) {
  constexpr int kPerThread = 8;  // partials per thread and round: 32 per round
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bg = bh / a.G, hl = bh % a.G;
  const int nstd = a.tph;
  const int P = n_est + nstd + n_ret;
  // partial i: estimate pieces, steady pieces, then the retrieval pieces of
  // the blocks listed in S.u.merge.rb
  auto part = [&](int i) -> const float* {
    if (i < n_est) return a.est_part + ((size_t)(e_lo + i + bg) * a.G + hl) * kPartStride;
    i -= n_est;
    if (i < nstd) return a.std_part + ((size_t)((long long)bg * a.tph + i) * a.G + hl) * kPartStride;
    return a.ret_part + (size_t)(S.u.merge.rb[i - nstd] + bh) * kPartStride;
  };
  float* wm = S.u.merge.w;
  float* wl = S.u.merge.wl;
  const int dim = tid & (kD - 1), qq = tid >> 7;
  float M = -INFINITY, L = 0.f, O = 0.f;
  for (int base = 0; base < P; base += 4 * kPerThread) {
    const int np = min(4 * kPerThread, P - base);
    float mi = -INFINITY, li = 0.f;
    if (tid < np) {
      const float* p = part(base + tid);
      mi = __ldcg(p);
      li = __ldcg(p + 1);
    }
    float ov[kPerThread];
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
      const int i = qq + 4 * u;
      ov[u] = i < np ? __ldcg(part(base + i) + 2 + dim) : 0.f;
    }
    if (warp == 0) {
      const float mc = fmaxf(M, warp_max(mi));
      const float f = (mi > -INFINITY) ? exp2f(mi - mc) : 0.f;
      const float corr = (M > -INFINITY) ? exp2f(M - mc) : 0.f;
      const float lr = warp_sum(f * li);
      wm[lane] = f;
      if (lane == 0) {
        wl[0] = mc;
        wl[1] = corr;
        wl[2] = lr;
      }
    }
    csync();
    const float Mn = wl[0], corr = wl[1];
    if (Mn > -INFINITY) {
      L = L * corr + wl[2];
      O *= corr;
#pragma unroll
      for (int u = 0; u < kPerThread; ++u) {
        const int i = qq + 4 * u;
        if (i < np) O += wm[i] * ov[u];
      }
      M = Mn;
    }
    csync();
  }
  float* red = S.u.merge.red;
  if (qq > 0) red[(qq - 1) * kD + dim] = O;
  csync();
  if (qq == 0) {
    O += red[dim] + red[kD + dim] + red[2 * kD + dim];
    a.out[(size_t)bh * kD + dim] = (L > 0.f) ? O / L : 0.f;
    if (a.lse != nullptr && dim == 0) a.lse[bh] = (L > 0.f) ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
  csync();
}

// ---------------------------------------------------------------------------
// retrieval partition (identical in every block)
// ---------------------------------------------------------------------------
// Block b's share of the retrieved tokens is [bnd[b], bnd[b+1]) of the list of
// every head's retrieved tokens (heads in order).  Shares are proportional to
// w_b = max(0, avg - static_b), where static_b is the block's other streamed
// work and avg the mean total work per block, and start on 64-token
// boundaries.  Computed by the producer warp into S.bnd.
__device__ void partition(const DecodeArgs& a, DecSmem& S, long long Ttot) {
  const int lane = threadIdx.x & 31;
  // in tokens, scaled by nb: w_b * nb = max(0, total - nb * static_b)
  const long long total = a.static_units * kTokPerUnit + Ttot;
  long long wsum = 0;
  for (int b0 = 0; b0 < a.nb; b0 += 32) {
    const int b = b0 + lane;
    long long w = b < a.nb ? total - (long long)a.nb * S.static_w[b] * kTokPerUnit : 0;
    w = w > 0 ? w : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(kFull, w, o);
    wsum += w;
  }
  // shares proportional to w (float ratios: the same operations in every
  // block give the same, monotone boundaries)
  const float scale = wsum > 0 ? (float)Ttot / (float)wsum : 0.f;
  long long carry = 0;
  for (int b0 = 0; b0 < a.nb; b0 += 32) {
    const int b = b0 + lane;
    long long w = b < a.nb ? total - (long long)a.nb * S.static_w[b] * kTokPerUnit : 0;
    w = w > 0 ? w : 0;
    long long incl = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    const long long excl = carry + incl - w;
    if (b < a.nb) {
      long long t = (long long)((float)excl * scale);
      t = (t / kTile) * kTile;
      S.bnd[b] = (int)(t < Ttot ? t : Ttot);
    }
    carry += __shfl_sync(kFull, incl, 31);
  }
  if (lane == 0) S.bnd[a.nb] = (int)Ttot;
  __syncwarp();
}

// ---------------------------------------------------------------------------
// producer warp
// ---------------------------------------------------------------------------
template <int G>
__device__ void producer(const DecodeArgs& a, DecSmem& S) {
  const int lane = threadIdx.x & 31;
  uint32_t seq = 0;
  bool inject = a.inject != 0, skipped = false;
  const int ns = a.sink + a.window;
  const uint64_t stream_policy = l2_evict_first();  // every staged byte is read once per call
  const long long H = (long long)a.B * a.Hq;

  // claim the next ring slot (warp-uniform); false once this block aborted
  auto slot = [&](int& stage) -> bool {
    stage = (int)(seq % kStages);
    int good = 1;
    if (lane == 0) {
      if (*(volatile int*)&S.abort) {
        good = 0;
      } else if (seq >= (uint32_t)kStages) {
        good = stage_wait(smem_addr(&S.empty[stage]), ((seq / kStages) - 1u) & 1u, a.status,
                          &S.abort);
      }
      if (good) fence_proxy_async_smem();
    }
    return __shfl_sync(kFull, good, 0) != 0;
  };
  // lane 0 posts the expected bytes (after every lane's side-data writes)
  auto post = [&](int stage, uint32_t bytes) {
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(smem_addr(&S.full[stage]), bytes);
    __syncwarp();
  };
  auto commit = [&]() {
    if (__any_sync(kFull, skipped)) inject = false;
    __syncwarp();
    if (lane == 0) S.issued = (int)(seq + 1);
    ++seq;
  };
  auto copy_to = [&](void* dst, const void* src, uint32_t bytes, int stage) {
    if (inject) skipped = true;
    else bulk_g2s_hint(smem_addr(dst), src, bytes, smem_addr(&S.full[stage]), stream_policy);
  };

  // 1-2. index and steady tiles: lane 0 alone, addresses advanced
  // incrementally, one bulk copy per operand; the other lanes wait
  if (lane == 0) {
    bool inj = inject;
    // next ring slot; false once this block aborted
    auto wait_slot = [&](int& stage) -> bool {
      stage = (int)(seq % kStages);
      if (*(volatile int*)&S.abort) return false;
      if (seq >= (uint32_t)kStages &&
          !stage_wait(smem_addr(&S.empty[stage]), ((seq / kStages) - 1u) & 1u, a.status, &S.abort))
        return false;
      fence_proxy_async_smem();
      return true;
    };
    auto issue = [&](void* dst, const void* src, uint32_t bytes, int stage) {
      if (!inj) bulk_g2s_hint(smem_addr(dst), src, bytes, smem_addr(&S.full[stage]), stream_policy);
    };
    auto done_tile = [&]() {
      inj = false;  // the test hook drops the copies of the first tile only
      S.issued = (int)(++seq);
    };
    bool ok = true;
    const bool side_bulk = (a.C & 3) == 0;  // rows of sizes start 16-byte aligned
    if (a.stages & kStageScore) {
      // round by round, centroid-key tiles then value-sum tiles; or, with
      // a.kbar_first, every round's centroid-key tiles, then every round's
      // value-sum tiles in reverse round order (the consumers still hold the
      // last round's scores in shared memory)
      {
        for (int step = 0; step < 2 * a.rounds && ok; ++step) {
          const int pass = a.kbar_first ? step / a.rounds : step & 1;
          const int rd = !a.kbar_first ? step >> 1
                         : (pass == 0 ? step : 2 * a.rounds - 1 - step);
          const int j = rd * a.nb + (int)blockIdx.x;
          if (j >= a.nchunks) continue;
          const int n = chunk_tiles(a, j);
          // f32 rows (512 B), or bf16 rows (256 B) with two tiles of one group per stage
          const bool h16 = a.kbar16 != nullptr;
          const unsigned char* src =
              h16 ? reinterpret_cast<const unsigned char*>(pass == 0 ? a.kbar16 : a.vsum16)
                  : reinterpret_cast<const unsigned char*>(pass == 0 ? a.kbar : a.vsum);
          const uint32_t rowb = h16 ? 256u : 512u;
          int bg = (j * a.Q) / a.tpg, c0 = (j * a.Q - bg * a.tpg) * kTile;
          int q_bg = -1;  // the group whose query rows were staged last
          for (int i = 0; i < n;) {
            const int nsub = pair_tiles(a, j, i, n) ? 2 : 1;
            const int nrows = min(nsub * kTile, a.C - c0);
            int stage;
            if (!wait_slot(stage)) {
              ok = false;
              break;
            }
            const size_t row0 = (size_t)bg * a.C + c0;
            uint32_t bytes = (uint32_t)nrows * rowb;
            const bool bulk_n = side_bulk && (nrows & 3) == 0;
            const bool with_q = pass == 0 && bg != q_bg;
            if (pass == 0) {
              if (with_q) bytes += (uint32_t)G * kD * 2;
              if (bulk_n) {
                bytes += (uint32_t)nrows * 4u;
              } else {  // ragged rows of sizes: plain loads before the tile is posted
                for (int c = 0; c < nsub * kTile; ++c)
                  S.side[stage].n[c] = c < nrows ? __ldg(a.size + row0 + c) : 0;
              }
            }
            mbar_arrive_expect_tx(smem_addr(&S.full[stage]), bytes);
            issue(S.ring[stage], src + row0 * rowb, (uint32_t)nrows * rowb, stage);
            if (with_q) {  // the consumers read the query rows with a group's first tile
              const int b = bg / a.Hkv, g = bg - b * a.Hkv;
              issue(S.qs[stage], a.q + ((size_t)b * a.Hq + (size_t)g * G) * kD,
                    (uint32_t)G * kD * 2, stage);
              q_bg = bg;
            }
            if (pass == 0 && bulk_n)
              issue(S.side[stage].n, a.size + row0, (uint32_t)nrows * 4u, stage);
            done_tile();
            i += nsub;
            c0 += nsub * kTile;
            if (c0 >= a.C) {
              c0 = 0;
              ++bg;
            }
          }
        }
      }
    }
    // steady tiles: K/V rows of one KV group, with the group's query rows;
    // steady index u < sink is position u, the rest are N - window + (u - sink)
    if (ok && (a.stages & kStageAttend)) {
      const int nst = a.B * a.Hkv * a.tph;
      for (int t = a.nb - 1 - (int)blockIdx.x; t < nst; t += a.nb) {
        int stage;
        if (!wait_slot(stage)) break;
        const int bg = t / a.tph, i = t - bg * a.tph;
        const int u0 = i * kTile, u1 = min(ns, u0 + kTile), n = u1 - u0;
        const int b = bg / a.Hkv, g = bg - b * a.Hkv;
        mbar_arrive_expect_tx(smem_addr(&S.full[stage]), (uint32_t)n * 512u + (uint32_t)G * kD * 2u);
        const int a1 = min(u1, a.sink);
        if (u0 < a1) {
          const size_t r0 = (size_t)bg * a.N + u0;
          issue(S.ring[stage], a.K + r0 * kD, (uint32_t)(a1 - u0) * 256u, stage);
          issue(S.ring[stage] + kStageBytes / 2, a.V + r0 * kD, (uint32_t)(a1 - u0) * 256u, stage);
        }
        const int b0 = max(u0, a.sink);
        if (b0 < u1) {
          const size_t r0 = (size_t)bg * a.N + (a.N - a.window + (b0 - a.sink));
          const uint32_t d = (uint32_t)(b0 - u0) * 256u;
          issue(S.ring[stage] + d, a.K + r0 * kD, (uint32_t)(u1 - b0) * 256u, stage);
          issue(S.ring[stage] + kStageBytes / 2 + d, a.V + r0 * kD, (uint32_t)(u1 - b0) * 256u,
                stage);
        }
        issue(S.qs[stage], a.q + ((size_t)b * a.Hq + (size_t)g * G) * kD, (uint32_t)G * kD * 2,
              stage);
        done_tile();
      }
    }
    inject = inj;
  }
  __syncwarp();
  seq = __shfl_sync(kFull, seq, 0);
  inject = __shfl_sync(kFull, (int)inject, 0) != 0;
  if (*(volatile int*)&S.abort || !(a.stages & kStageAttend)) return;

  // retrieval tiles of tokens [x0, x1) of head bh (its clusters in id
  // order, 64 tokens per tile); false once this block aborted
  auto stream_piece = [&](int bh, int x0, int x1) -> bool {
    const int rs = a.r;
    const int b = bh / a.Hq, g = (bh - b * a.Hq) / G;
    const size_t head = (size_t)b * a.Hkv + g;
    const uint16_t* Ks = a.ksorted + head * (size_t)a.N_idx * kD;
    const uint16_t* Vs = a.vsorted + head * (size_t)a.N_idx * kD;
    const int* rows_g = a.sel_rows + (size_t)bh * rs;
    const int* cnts_g = a.sel_cnts + (size_t)bh * rs;
    const int* pre_g = a.sel_pre + (size_t)bh * rs;
    const float* ss_g = a.sel_sc + (size_t)bh * rs;
    // first cluster: the last j with pre_j <= x0 (32-ary search)
    int jlo = 0, jhi = rs;  // answer in [jlo, jhi)
    while (jhi - jlo > 1) {
      const int step = (jhi - jlo + 31) / 32;
      const int jj = jlo + lane * step;
      const int pj = jj < jhi ? __ldcg(pre_g + jj) : INT_MAX;
      const unsigned le = __ballot_sync(kFull, jj < jhi && pj <= x0);
      const int k = 31 - __clz(le);  // lanes 0..k hold pre <= x0 (pre ascending)
      jlo = jlo + k * step;
      jhi = min(jhi, jlo + step);
    }
    // clusters in two windows of 32 (A current, B prefetched): lane i of a
    // window holds cluster jA + i (or jA + 32 + i): first sorted row,
    // count, first token (piece-relative to the head) and score
    int jA = jlo;
    auto load_win = [&](int jbase, int& row, int& cnt, int& st, float& s2) {
      const int j = jbase + lane;
      row = 0;
      cnt = 0;
      st = INT_MAX;
      s2 = 0.f;
      if (j < rs) {
        row = __ldcg(rows_g + j);
        cnt = __ldcg(cnts_g + j);
        st = __ldcg(pre_g + j);
        s2 = __ldcg(ss_g + j) * kLog2e;
        if (cnt < 0 || row < 0 || (long long)row + cnt > a.N_idx) {
          report(a.status, WI_ERR_INDEX_MISMATCH);
          cnt = 0;
          row = 0;
        }
      }
    };
    int rowA, cntA, stA, rowB, cntB, stB;
    float sA, sB;
    load_win(jA, rowA, cntA, stA, sA);
    load_win(jA + 32, rowB, cntB, stB, sB);
    auto shift = [&]() {  // A <- B, B <- the next 32 clusters
      rowA = rowB;
      cntA = cntB;
      stA = stB;
      sA = sB;
      jA += 32;
      load_win(jA + 32, rowB, cntB, stB, sB);
    };
    // end (exclusive) of window A's last cluster
    auto endA = [&]() {
      const int st = __shfl_sync(kFull, stA, 31), cnt = __shfl_sync(kFull, cntA, 31);
      return st == INT_MAX ? INT_MAX : st + cnt;
    };
    for (int x = x0; x < x1; x += kTile) {
      const int e = min(x + kTile, x1), n = e - x;
      while (endA() <= x && jA + 32 < rs) shift();  // A fully used before this tile
      int stage;
      if (!slot(stage)) return false;
      // every cluster meeting [x, e): the score of its token slots (side
      // data) and the copies of its K and V rows
      uint32_t bytes = 0;
      for (;;) {
        const int y0 = max(x, stA), y1 = min(e, stA == INT_MAX ? stA : stA + cntA);
        if (y0 < y1) {
          for (int y = y0; y < y1; ++y) S.side[stage].s[y - x] = sA;
          const size_t srow = (size_t)rowA + (y0 - stA);
          const uint32_t d = (uint32_t)(y0 - x) * 256u, nb2 = (uint32_t)(y1 - y0) * 256u;
          copy_to(S.ring[stage] + d, Ks + srow * kD, nb2, stage);
          copy_to(S.ring[stage] + kStageBytes / 2 + d, Vs + srow * kD, nb2, stage);
          bytes += 2u * nb2;
        }
        if (endA() >= e || jA + 32 >= rs) break;
        shift();  // the tile runs past window A
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(kFull, bytes, o);
      if (lane == 0) {
        TileInfo ti;
        ti.kind = kTileRet;
        ti.bh = bh;
        ti.ntok = n;
        ti.last = (e == x1);
        S.info[stage] = ti;
        copy_to(S.qs[stage], a.q + (size_t)bh * kD, kD * 2, stage);
      }
      post(stage, bytes + kD * 2u);
      commit();
    }
    return true;
  };
  // 3. retrieval tiles of the block's share of the retrieved tokens
  if (a.r > 0 && a.ret_per_head) {
    // part p of P of one head: its tokens [T p / P, T (p + 1) / P), once that
    // head's selection is published
    const int bh = (int)(((long long)blockIdx.x * H) / a.nb);
    const int b0 = ret_first(a, bh), P = ret_first(a, bh + 1) - b0;
    int good = 1;
    if (lane == 0 && a.fused) {
      good = !*(volatile int*)&S.abort && count_wait(a.sel_flag + bh, 1u, a.status, &S.abort);
      if (!good) *(volatile int*)&S.abort = 1;
    }
    if (!__shfl_sync(kFull, good, 0)) return;
    __syncwarp();
    const long long T = __ldcg(a.head_tok + bh), p = (long long)blockIdx.x - b0;
    const int x0 = (int)(T * p / P), x1 = (int)(T * (p + 1) / P);
    if (x0 < x1 && !stream_piece(bh, x0, x1)) return;
  } else if (a.r > 0) {
    if (a.fused) {
      int good = 1;
      if (lane == 0) {
        good = !*(volatile int*)&S.abort &&
               count_wait(a.sel_done, (unsigned)H, a.status, &S.abort);
        if (!good) *(volatile int*)&S.abort = 1;
      }
      if (!__shfl_sync(kFull, good, 0)) return;
      __syncwarp();
    }
    // total retrieved tokens, and the block's share
    long long Ttot = 0;
    for (long long h0 = 0; h0 < H; h0 += 32) {
      long long x = (h0 + lane < H) ? (long long)__ldcg(a.head_tok + h0 + lane) : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
      Ttot += x;
    }
    partition(a, S, Ttot);
    const long long t0 = S.bnd[blockIdx.x], t1 = S.bnd[blockIdx.x + 1];
    // walk the heads that meet [t0, t1)
    long long P = 0;  // first token of the current head window
    for (long long h0 = 0; h0 < H && P < t1; h0 += 32) {
      const int th = (h0 + lane < H) ? __ldcg(a.head_tok + h0 + lane) : 0;
      int incl = th;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += x;
      }
      const long long lo_l = P + incl - th, hi_l = P + incl;  // this lane's head: [lo_l, hi_l)
      unsigned meet = __ballot_sync(kFull, th > 0 && hi_l > t0 && lo_l < t1);
      while (meet) {
        const int src = __ffs(meet) - 1;
        meet &= meet - 1;
        const int bh = (int)h0 + src;
        const long long hlo = __shfl_sync(kFull, lo_l, src);
        const int Th = __shfl_sync(kFull, th, src);
        const int x0 = (int)max(0ll, t0 - hlo), x1 = (int)min((long long)Th, t1 - hlo);
        if (!stream_piece(bh, x0, x1)) return;
      }
      P += __shfl_sync(kFull, incl, 31);
    }
  }
  // end marker
  int stage;
  if (!slot(stage)) return;
  if (lane == 0) {
    TileInfo ti;
    ti.kind = kTileEnd;
    ti.bh = 0;
    ti.ntok = 0;
    ti.last = 0;
    S.info[stage] = ti;
  }
  post(stage, 0u);
  commit();
}

// ---------------------------------------------------------------------------
// consumer tiles
// ---------------------------------------------------------------------------
// Lane L < 4G of warp w works on row (or token) 4w + L / G and head L mod G.
template <int G>
__device__ __forceinline__ int lane_row(int lane) {
  return (lane & (4 * G - 1)) / G;
}
template <int G>
__device__ __forceinline__ int lane_head(int lane) {
  return (lane & (4 * G - 1)) % G;
}

// G-head online-softmax state of one warp (steady tiles).
template <int G>
struct HeadsState {
  float m[G];   // running max (log2 units), warp-uniform
  float4 o[G];  // this lane's 4 dimensions
  float l;      // lane L < 4G: running sum for head L mod G
};
template <int G>
__device__ __forceinline__ void heads_reset(HeadsState<G>& e) {
#pragma unroll
  for (int h = 0; h < G; ++h) {
    e.m[h] = -INFINITY;
    e.o[h] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  e.l = 0.f;
}
// Add the weights of 4 rows for G heads: lane L < 4G holds x (log2 units,
// -inf = absent) of row L / G and head L mod G and its multiplicity n;
// v[j] are this lane's 4 dimensions of row j.
template <int G>
__device__ __forceinline__ void heads_add(HeadsState<G>& e, float x, float n, const float4 (&v)[4],
                                          int lane) {
  const int hL = lane_head<G>(lane);
  float mt = lane < 4 * G ? x : -INFINITY;
#pragma unroll
  for (int o = G; o < 4 * G; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, o));
  float mL = -INFINITY, corrL = 1.f;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float th = __shfl_sync(kFull, mt, h);
    if (th > e.m[h]) {
      const float corr = (e.m[h] > -INFINITY) ? exp2f(e.m[h] - th) : 0.f;
      e.o[h].x *= corr;
      e.o[h].y *= corr;
      e.o[h].z *= corr;
      e.o[h].w *= corr;
      if (hL == h) corrL = corr;
      e.m[h] = th;
    }
    if (hL == h) mL = e.m[h];
  }
  e.l *= corrL;
  const float p = (lane < 4 * G && x > -INFINITY) ? exp2f(x - mL) : 0.f;
  e.l += p * n;
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float pj = __shfl_sync(kFull, p, jj * G + h);
      e.o[h].x += pj * v[jj].x;
      e.o[h].y += pj * v[jj].y;
      e.o[h].z += pj * v[jj].z;
      e.o[h].w += pj * v[jj].w;
    }
  }
}
// Write the G heads' partials of one piece (dst(h) = base + h * kPartStride)
// through combine_write, four heads per pass.
template <int G>
__device__ void heads_flush(DecSmem& S, HeadsState<G>& e, float* base, int lane) {
  float lh[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float x = (lane < 4 * G && lane_head<G>(lane) == h) ? e.l : 0.f;
    lh[h] = warp_sum(x);
  }
  constexpr int NH = G < 4 ? G : 4;
#pragma unroll
  for (int h0 = 0; h0 < G; h0 += NH) {
    float m[NH], l[NH];
    float4 o[NH];
    float* dst[NH];
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      m[h] = e.m[h0 + h];
      l[h] = lh[h0 + h];
      o[h] = e.o[h0 + h];
      dst[h] = base + (size_t)(h0 + h) * kPartStride;
    }
    combine_write<NH>(S, m, l, o, dst);
  }
  heads_reset(e);
}

// heads_flush of a copy of the state, out of line (keeps the callers' loops
// free of the combine's registers).
template <int G>
__device__ __noinline__ void heads_flush_nv(DecSmem& S, HeadsState<G> e, float* base) {
  heads_flush<G>(S, e, base, threadIdx.x & 31);
}

// ---------------------------------------------------------------------------
// consumer warps
// ---------------------------------------------------------------------------
// Per-warp position in the ring.  A warp whose wait gave up turns hollow: it
// waits for nothing more and computes nothing, but it still passes every
// block-wide barrier of the static schedule.
struct Ring {
  uint32_t seq;
  bool hollow;
};
__device__ __forceinline__ bool acquire(const DecodeArgs& a, DecSmem& S, Ring& rg, int& stage) {
  stage = (int)(rg.seq % kStages);
  if (rg.hollow) return false;
  if (!stage_wait(smem_addr(&S.full[stage]), (rg.seq / kStages) & 1u, a.status, &S.abort)) {
    rg.hollow = true;
    return false;
  }
  return true;
}
__device__ __forceinline__ void release(DecSmem& S, Ring& rg, int stage) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(smem_addr(&S.empty[stage]));
  ++rg.seq;
}
// Collective bounded wait until *cnt >= target (thread 0 waits; one barrier
// makes the answer uniform).
__device__ bool wait_count_all(const DecodeArgs& a, DecSmem& S, const unsigned* cnt,
                               unsigned target) {
  int ok = 1;
  if (threadIdx.x == 0) {
    ok = !*(volatile int*)&S.abort && count_wait(cnt, target, a.status, &S.abort);
    if (!ok) *(volatile int*)&S.abort = 1;
  }
  return !cany(!ok);
}

// Centroid-key tiles of chunk j (n tiles): scores of the group's G heads,
// into the workspace and the block's chunk copy; then the groups' scored-tile
// counts are published.
template <int G, bool H16>
__device__ __forceinline__ void kbar_tiles(const DecodeArgs& a, DecSmem& S, Ring& rg, int j, int n) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L4 = 4 * G;
  const int jr = lane_row<G>(lane), hr = lane_head<G>(lane);
  const int C = a.C;
  // tile i of the chunk: KV group bg, first cluster c0 (advanced per tile)
  int bg = (j * a.Q) / a.tpg, c0 = (j * a.Q - bg * a.tpg) * kTile;
  int cur_bg = -1;
  float4 qs[G];           // this lane's 4 dimensions of the group's query rows, scaled
  float* srow = nullptr;  // scores row of this lane's head
#pragma unroll
  for (int h = 0; h < G; ++h) qs[h] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = 0; i < n;) {
    const int nsub = (H16 && pair_tiles(a, j, i, n)) ? 2 : 1;
    int stage;
    const bool got = acquire(a, S, rg, stage);
    if (got && bg != cur_bg) {  // the group's query rows come with its first tile
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float4 qf = bf4(lds2(S.qs[stage] + h * kD * 2 + lane * 8));
        qs[h] = make_float4(qf.x * a.scale, qf.y * a.scale, qf.z * a.scale, qf.w * a.scale);
      }
      cur_bg = bg;
      const int b = bg / a.Hkv, g = bg - b * a.Hkv;
      srow = a.scores + ((size_t)b * a.Hq + (size_t)g * G + hr) * C;
    }
    for (int sub = 0; sub < nsub; ++sub) {  // the tiles of the stage (one group)
      const int nrows = min(kTile, C - c0);
      const int ii = i + sub;
      if (got) {
        float4 k[4];
#pragma unroll
        for (int r4 = 0; r4 < 4; ++r4) {
          const int row = warp * 4 + r4;
          if (H16) {
            const uint16_t* kb = reinterpret_cast<const uint16_t*>(S.ring[stage]) + sub * kTile * kD;
            k[r4] = row < nrows ? bf4(lds2(kb + row * kD + lane * 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
          } else {
            const float* kb = reinterpret_cast<const float*>(S.ring[stage]);
            k[r4] = row < nrows ? lds4(kb + row * kD + lane * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        const int nsz = S.side[stage].n[sub * kTile + warp * 4 + jr];
        if (sub == nsub - 1) release(S, rg, stage);
        float v[4 * G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
          for (int r4 = 0; r4 < 4; ++r4)
            v[r4 * G + h] = k[r4].x * qs[h].x + k[r4].y * qs[h].y + k[r4].z * qs[h].z + k[r4].w * qs[h].w;
        }
        const float tot = reduce_scatter<4 * G>(v, lane);
        const int row = warp * 4 + jr;
        const float s = (row < nrows && nsz > 0) ? tot : -INFINITY;
        if (lane < L4) {
          if (row < nrows) srow[c0 + row] = s;
          S.a.chunk.sc[ii][warp][lane] = s;
          if (hr == 0) S.a.chunk.n[ii][warp][jr] = row < nrows ? nsz : 0;
        }
      } else if (lane < L4) {
        S.a.chunk.sc[ii][warp][lane] = -INFINITY;
        if (hr == 0) S.a.chunk.n[ii][warp][jr] = 0;
      }
      c0 += kTile;
      if (c0 >= C) {
        c0 = 0;
        ++bg;
      }
    }
    i += nsub;
  }
  if (n > 0) {
    csync();  // every warp's scores of the chunk are written
    if (a.fused && tid < 32) {
      // one request per KV group met by the chunk: its scored tiles
      const int T0 = j * a.Q, T1 = T0 + n;
      const int g0 = T0 / a.tpg, g1 = (T1 - 1) / a.tpg;
      for (int bg = g0 + tid; bg <= g1; bg += 32) {
        const int lo = max(T0, bg * a.tpg), hi = min(T1, (bg + 1) * a.tpg);
        publish(S, a, a.grp_cnt + bg, (unsigned)(hi - lo), 1);
      }
    }
  }
}

// The selections assigned to this block in round rd (heads in order): each
// once its KV group is fully scored.
template <int G>
__device__ __forceinline__ void selections(const DecodeArgs& a, DecSmem& S, const Ring& rg, int rd) {
  const int tid = threadIdx.x;
  const int blk = (int)blockIdx.x;
  // b. selections assigned to this block and round (heads in order)
  if (a.stages & kStageSelect) {
    // groups whose last chunk falls in round rd
    const int nbg = a.B * a.Hkv;
    int g_lo = 0, g_hi = nbg;  // first group with last_chunk >= rd*nb, first with >= (rd+1)*nb
    {
      int lo = 0, hi = nbg;
      while (lo < hi) {
        const int mid = (lo + hi) / 2;
        if (last_chunk(a, mid) >= rd * a.nb) hi = mid;
        else lo = mid + 1;
      }
      g_lo = lo;
      lo = g_lo;
      hi = nbg;
      while (lo < hi) {
        const int mid = (lo + hi) / 2;
        if (last_chunk(a, mid) >= (rd + 1) * a.nb) hi = mid;
        else lo = mid + 1;
      }
      g_hi = lo;
    }
    for (int bg = g_lo; bg < g_hi; ++bg) {
      const int lc = last_chunk(a, bg);
      int hl = (lc - blk) % a.nb;
      if (hl < 0) hl += a.nb;
      if (hl >= (a.share ? 1 : G)) continue;
      const int bh = bg * G + hl;
      const bool ok = a.fused ? wait_count_all(a, S, a.grp_cnt + bg, (unsigned)a.tpg) : !cany(rg.hollow);
      if (!ok) continue;
      select_head(a, S, bh);
      if (a.fused && tid == 0) {
        publish(S, a, a.sel_done, a.share ? (unsigned)G : 1u, 1);
        if (a.ret_per_head) publish(S, a, a.sel_flag + bh, 1u, 1);
      }
    }
  }
}

// Value-sum tiles of chunk j: the estimate of every cluster of the chunk,
// against the warp's own maximum score of each KV group (a fixed reference:
// no rescaling), one partial per (chunk, KV group, query head).
template <int G, bool H16>
__device__ __forceinline__ void vsum_tiles(const DecodeArgs& a, DecSmem& S, Ring& rg, int j, int n,
                                           bool refill) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L4 = 4 * G;
  const int jr = lane_row<G>(lane), hr = lane_head<G>(lane);
  if (refill) {
    // the chunk's scores and sizes back into this warp's shared-memory slots,
    // as its centroid-key pass left them (-inf / 0 past the group's last row)
    if (lane < L4) {
      for (int i = 0; i < n; ++i) {
        const int t = j * a.Q + i, bg = t / a.tpg;
        const int c0 = (t - bg * a.tpg) * kTile, row = warp * 4 + jr;
        const bool in = c0 + row < a.C;
        const int b = bg / a.Hkv, g = bg - b * a.Hkv;
        const float* srow = a.scores + ((size_t)b * a.Hq + (size_t)g * G + hr) * a.C;
        S.a.chunk.sc[i][warp][lane] = in ? __ldcg(srow + c0 + row) : -INFINITY;
        if (hr == 0) S.a.chunk.n[i][warp][jr] = in ? __ldg(a.size + (size_t)bg * a.C + c0 + row) : 0;
      }
    }
    __syncwarp();
  }
  // one KV group at a time: tiles [i0, i1) of the chunk
  for (int i0 = 0; i0 < n;) {
    const int bg = (j * a.Q + i0) / a.tpg;
    const int i1 = min(n, (bg + 1) * a.tpg - j * a.Q);
    // the warp's maximum score per head over its rows of this group: the
    // fixed reference of its estimate (every weight is at most 1)
    float m[G];
    float4 o[G];
    float lacc = 0.f;
    {
      float mx = -INFINITY;
      if (lane < L4)
        for (int ii = i0; ii < i1; ++ii) mx = fmaxf(mx, S.a.chunk.sc[ii][warp][lane]);
#pragma unroll
      for (int o2 = G; o2 < 32; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o2));
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mh = __shfl_sync(kFull, mx, h);
        m[h] = mh > -INFINITY ? mh * kLog2e : -INFINITY;
        o[h] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float mL = m[0];
#pragma unroll
    for (int h = 1; h < G; ++h)
      if (hr == h) mL = m[h];
    for (int i = i0; i < i1;) {
      const int nsub = (H16 && pair_tiles(a, j, i, n)) ? 2 : 1;
      int stage;
      if (!acquire(a, S, rg, stage)) {
        i += nsub;
        continue;
      }
      for (int sub = 0; sub < nsub; ++sub, ++i) {  // the tiles of the stage (one group)
        const int c0 = (j * a.Q + i - bg * a.tpg) * kTile;
        const int nrows = min(kTile, a.C - c0);
        float4 v[4];
#pragma unroll
        for (int r4 = 0; r4 < 4; ++r4) {
          const int row = warp * 4 + r4;
          if (H16) {
            const uint16_t* vs = reinterpret_cast<const uint16_t*>(S.ring[stage]) + sub * kTile * kD;
            v[r4] = row < nrows ? bf4(lds2(vs + row * kD + lane * 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
          } else {
            const float* vs = reinterpret_cast<const float*>(S.ring[stage]);
            v[r4] = row < nrows ? lds4(vs + row * kD + lane * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        if (sub == nsub - 1) release(S, rg, stage);
        const float s = lane < L4 ? S.a.chunk.sc[i][warp][lane] : -INFINITY;
        const int nn = lane < L4 ? S.a.chunk.n[i][warp][jr] : 0;
        const float p = (s > -INFINITY && nn > 0) ? exp2f(s * kLog2e - mL) : 0.f;
        lacc += p * (float)nn;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float pj = __shfl_sync(kFull, p, jj * G + h);
            o[h].x += pj * v[jj].x;
            o[h].y += pj * v[jj].y;
            o[h].z += pj * v[jj].z;
            o[h].w += pj * v[jj].w;
          }
        }
      }
    }
    // est partial slot of (chunk j, group bg): (j + bg) * G + h
    HeadsState<G> e;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      e.m[h] = m[h];
      e.o[h] = o[h];
    }
    e.l = lacc;
    heads_flush_nv<G>(S, e, a.est_part + (size_t)(j + bg) * G * kPartStride);
    if (a.fused && tid == 0) {
      const int b = bg / a.Hkv, g = bg - b * a.Hkv;
      publish(S, a, a.head_cnt + (size_t)b * a.Hq + (size_t)g * G, 1u, G);
    }
    i0 = i1;
  }
}

// Steady tiles of this block: the sink and local-window K/V rows of one KV
// group, its G heads at once; one partial per (tile, head).
template <int G>
__device__ __forceinline__ void steady_tiles(const DecodeArgs& a, DecSmem& S, Ring& rg) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int blk = (int)blockIdx.x;
  const int jr = lane_row<G>(lane);
  // ---- 2. steady tiles: the group's G heads at once
  const long long nst = (long long)a.B * a.Hkv * a.tph;
  const float qs = a.scale * kLog2e;
  for (long long t = a.nb - 1 - (long long)blk; t < nst; t += a.nb) {
    const int bg = (int)(t / a.tph), i = (int)(t - (long long)bg * a.tph);
    const int u0 = i * kTile, ntok = min(a.sink + a.window, u0 + kTile) - u0;
    HeadsState<G> e;
    heads_reset(e);
    int stage;
    if (acquire(a, S, rg, stage)) {
      const uint16_t* kt = reinterpret_cast<const uint16_t*>(S.ring[stage]);
      const uint16_t* vt = kt + kTile * kD;
      uint2 kk[4], vv[4], q[G];
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4) {
        const int tk = warp * 4 + r4;
        kk[r4] = tk < ntok ? lds2(kt + tk * kD + lane * 4) : make_uint2(0u, 0u);
        vv[r4] = tk < ntok ? lds2(vt + tk * kD + lane * 4) : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int h = 0; h < G; ++h) q[h] = lds2(S.qs[stage] + h * kD * 2 + lane * 8);
      release(S, rg, stage);
      float v[4 * G];
      float4 vf[4];
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4) vf[r4] = bf4(vv[r4]);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float4 qf = bf4(q[h]);
#pragma unroll
        for (int r4 = 0; r4 < 4; ++r4) {
          const float4 kf = bf4(kk[r4]);
          v[r4 * G + h] = (kf.x * qf.x + kf.y * qf.y + kf.z * qf.z + kf.w * qf.w) * qs;
        }
      }
      const float lg = reduce_scatter<4 * G>(v, lane);
      const float x = (warp * 4 + jr < ntok) ? lg : -INFINITY;
      heads_add<G>(e, x, 1.f, vf, lane);
    }
    heads_flush<G>(S, e, a.std_part + (size_t)t * G * kPartStride, lane);
    if (tid == 0) {
      const int b = bg / a.Hkv, g = bg - b * a.Hkv;
      publish(S, a, a.head_cnt + (size_t)b * a.Hq + (size_t)g * G, 1u, G);
    }
  }

}

// Retrieval tiles of this block's share, one head per tile, until the end
// marker.  Every warp keeps its own softmax state; at the end of a head's
// range the last warp to finish combines the 16 states into the piece's
// partial (slot block + head) and publishes it.
__device__ __forceinline__ void retrieval_tiles(const DecodeArgs& a, DecSmem& S, Ring& rg) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int blk = (int)blockIdx.x;
  // ---- 3. retrieval tiles: one head per tile; every warp keeps its own state
  {
    float m = -INFINITY, l = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    int piece = 0;
    const float qsc = a.scale * kLog2e;
    for (;;) {
      int stage;
      if (!acquire(a, S, rg, stage)) break;
      const TileInfo ti = S.info[stage];
      if (ti.kind == kTileEnd) {
        release(S, rg, stage);
        break;
      }
      const uint16_t* kt = reinterpret_cast<const uint16_t*>(S.ring[stage]);
      const uint16_t* vt = kt + kTile * kD;
      uint2 kk[4], vv[4];
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4) {
        const int tk = warp * 4 + r4;
        kk[r4] = tk < ti.ntok ? lds2(kt + tk * kD + lane * 4) : make_uint2(0u, 0u);
        vv[r4] = tk < ti.ntok ? lds2(vt + tk * kD + lane * 4) : make_uint2(0u, 0u);
      }
      const uint2 q = lds2(S.qs[stage] + lane * 8);
      const float sc = (lane < 4 && warp * 4 + lane < ti.ntok) ? S.side[stage].s[warp * 4 + lane]
                                                               : -INFINITY;
      release(S, rg, stage);
      if (warp * 4 < ti.ntok) {
        const float4 qf = bf4(q);
        float v[4];
#pragma unroll
        for (int r4 = 0; r4 < 4; ++r4) {
          const float4 kf = bf4(kk[r4]);
          v[r4] = (kf.x * qf.x + kf.y * qf.y + kf.z * qf.z + kf.w * qf.w) * qsc;
        }
        const float lg0 = reduce_scatter<4>(v, lane);  // lane L: token L mod 4
        const bool ok = (lane & 3) + warp * 4 < ti.ntok;
        const float lg = ok ? lg0 : -INFINITY;
        const float s2 = __shfl_sync(kFull, sc, lane & 3);  // token's cluster score
        float mt = fmaxf(lg, ok ? s2 : -INFINITY);
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 1));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 2));
        const float mn = fmaxf(m, mt);
        const float corr = (m > -INFINITY) ? exp2f(m - mn) : 0.f;
        // weight of token (lane mod 4): exact term minus its estimate share
        const float p = ok ? exp2f(lg - mn) - (s2 > -INFINITY ? exp2f(s2 - mn) : 0.f) : 0.f;
        float ps = p;
        ps += __shfl_xor_sync(kFull, ps, 1);
        ps += __shfl_xor_sync(kFull, ps, 2);
        l = l * corr + ps;
        o.x *= corr;
        o.y *= corr;
        o.z *= corr;
        o.w *= corr;
#pragma unroll
        for (int r4 = 0; r4 < 4; ++r4) {
          const float pj = __shfl_sync(kFull, p, r4);
          const float4 vf = bf4(vv[r4]);
          o.x += pj * vf.x;
          o.y += pj * vf.y;
          o.z += pj * vf.z;
          o.w += pj * vf.w;
        }
        m = mn;
      }
      if (ti.last) {
        // this warp's state into the piece's slot; the last warp combines
        const int sl = piece % kSlots;
        WarpPart& wp = S.a.slot[sl][warp];
        if (lane == 0) {
          wp.m = m;
          wp.l = l;
        }
        reinterpret_cast<float4*>(wp.o)[lane] = o;
        __syncwarp();
        unsigned old = 0;
        if (lane == 0) old = atom_add_release_cta(&S.slot_cnt[sl], 1u);
        old = __shfl_sync(kFull, old, 0);
        const unsigned target = (unsigned)kCW * (unsigned)(piece / kSlots + 1);
        if (old + 1u == target) {
          fence_acq_cta();
          float Mx = -INFINITY;
#pragma unroll
          for (int w = 0; w < kCW; ++w) Mx = fmaxf(Mx, S.a.slot[sl][w].m);
          float Lx = 0.f;
          float4 Ox = make_float4(0.f, 0.f, 0.f, 0.f);
          if (Mx > -INFINITY) {
#pragma unroll 4
            for (int w = 0; w < kCW; ++w) {
              const float mw = S.a.slot[sl][w].m;
              const float f = mw > -INFINITY ? exp2f(mw - Mx) : 0.f;
              Lx += S.a.slot[sl][w].l * f;
              const float4 ow = reinterpret_cast<const float4*>(S.a.slot[sl][w].o)[lane];
              Ox.x += ow.x * f;
              Ox.y += ow.y * f;
              Ox.z += ow.z * f;
              Ox.w += ow.w * f;
            }
          }
          float* dst = a.ret_part + (size_t)(blk + ti.bh) * kPartStride;
          if (lane == 0) {
            dst[0] = Mx;
            dst[1] = Lx;
          }
          // partials are 130 floats: their o is only 8-byte aligned
          dst[2 + 4 * lane] = Ox.x;
          dst[3 + 4 * lane] = Ox.y;
          dst[4 + 4 * lane] = Ox.z;
          dst[5 + 4 * lane] = Ox.w;
          __syncwarp();
          if (lane == 0) publish(S, a, a.head_cnt + ti.bh, 1u, 1);
        }
        m = -INFINITY;
        l = 0.f;
        o = make_float4(0.f, 0.f, 0.f, 0.f);
        ++piece;
      }
    }
  }
}

// Merges of heads blk, blk + nb, ...: once every partial of the head is
// published, the log-sum-exp combine into out and lse.
__device__ __forceinline__ void merges(const DecodeArgs& a, DecSmem& S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int blk = (int)blockIdx.x;
  const int H = a.B * a.Hq;
  for (int bh = blk; bh < H; bh += a.nb) {
    const int bg = bh / a.G;
    // with per-head ranges this block need not have waited for the head's
    // selection: its token count is read only once it is published
    if (a.ret_per_head && a.fused && !wait_count_all(a, S, a.sel_flag + bh, 1u)) break;
    // this head's retrieval pieces: blocks whose share meets its tokens
    int P_lo = 0;
    {
      int part = 0;
      for (int h2 = tid; h2 < bh; h2 += kCT) part += __ldcg(a.head_tok + h2);
      part = __reduce_add_sync(kFull, part);
      if (lane == 0) S.u.merge.cnt[warp] = part;
      csync();
      for (int w = 0; w < kCW; ++w) P_lo += S.u.merge.cnt[w];
      csync();
    }
    const int Th = a.r > 0 ? __ldcg(a.head_tok + bh) : 0;
    // blocks whose share is non-empty and meets [P_lo, P_lo + Th), in order;
    // with per-head ranges, the blocks of the head's range with a non-empty part
    if (tid == 0) {
      int n = 0;
      if (Th > 0 && a.ret_per_head) {
        const int b0 = ret_first(a, bh), P = ret_first(a, bh + 1) - b0;
        for (int p = 0; p < P; ++p)
          if ((long long)Th * (p + 1) / P > (long long)Th * p / P) S.u.merge.rb[n++] = b0 + p;
      } else if (Th > 0) {
        for (int b = 0; b < a.nb; ++b)
          if (S.bnd[b] < S.bnd[b + 1] && S.bnd[b + 1] > P_lo && S.bnd[b] < P_lo + Th)
            S.u.merge.rb[n++] = b;
      }
      S.u.merge.cnt[0] = n;
    }
    csync();
    const int n_ret = S.u.merge.cnt[0];
    const int e_lo = first_chunk(a, bg), e_hi = last_chunk(a, bg);
    const int n_est = e_hi - e_lo + 1;
    // estimate pieces are counted only when this launch wrote them
    const unsigned target = (unsigned)((a.fused ? n_est : 0) + a.tph + n_ret);
    if (!wait_count_all(a, S, a.head_cnt + bh, target)) break;
    merge_head(a, S, bh, n_est, e_lo, n_ret);
    csync();  // S.u.merge.cnt is rewritten by the next head
  }
}

template <int G>
__device__ void consumers(const DecodeArgs& a, DecSmem& S) {
  const int tid = threadIdx.x;
  const int blk = (int)blockIdx.x;
  Ring rg;
  rg.seq = 0;
  rg.hollow = false;
  // 1. the centroid-key tiles of every round, the selections, then the
  // value-sum tiles of every round, last round first (its scores are still
  // in shared memory; earlier rounds' are read back)
  auto chunk_n = [&](int rd) {
    const int j = rd * a.nb + blk;
    return (j < a.nchunks && (a.stages & kStageScore)) ? chunk_tiles(a, j) : 0;
  };
  // steps: (centroid-key tiles, selections, value-sum tiles) of round 0, of
  // round 1, ...; or with a.kbar_first every round's centroid-key tiles,
  // every round's selections, every round's value-sum tiles (last round
  // first)
  int last_rd = -1;
  for (int step = 0; step < 3 * a.rounds; ++step) {
    int kind, rd;
    if (a.kbar_first) {
      kind = step / a.rounds;
      rd = step - kind * a.rounds;
      if (kind == 2) rd = a.rounds - 1 - rd;
    } else {
      rd = step / 3;
      kind = step - rd * 3;
    }
    if (kind == 1) {
      if (a.stages & kStageSelect) selections<G>(a, S, rg, rd);
      continue;
    }
    const int n = chunk_n(rd);
    if (n == 0) continue;
    if (kind == 0) {
      if (a.kbar16)
        kbar_tiles<G, true>(a, S, rg, rd * a.nb + blk, n);
      else
        kbar_tiles<G, false>(a, S, rg, rd * a.nb + blk, n);
      last_rd = rd;
    } else {
      if (a.kbar16)
        vsum_tiles<G, true>(a, S, rg, rd * a.nb + blk, n, a.kbar_first && rd != last_rd);
      else
        vsum_tiles<G, false>(a, S, rg, rd * a.nb + blk, n, a.kbar_first && rd != last_rd);
    }
  }
  if (a.stages & kStageAttend) {
    steady_tiles<G>(a, S, rg);  // 2.
    // the retrieval pieces' per-warp states share shared memory with the
    // value-sum tiles' scores: no warp may start on them while another still
    // reads those scores
    csync();
    retrieval_tiles(a, S, rg);  // 3.
  }
  // 4. merges
  csync();
  if ((a.stages & kStageAttend) && !cany(rg.hollow)) merges(a, S);
  // no more requests; wait for the signaling warp to publish the last batch
  if (tid == 0) {
    st_release_cta(&S.cons_done, 1);
    const unsigned long long t0 = global_ns();
    while (!ld_acquire_cta(&S.sig_done)) {
      if (global_ns() - t0 > kWaitLimitNs) {
        report(a.status, WI_ERR_DEVICE_TIMEOUT);
        *(volatile int*)&S.abort = 1;
        break;
      }
      __nanosleep(64);
    }
  }
}


// ---------------------------------------------------------------------------
// signaling warp: publishes the consumers' queued requests with one gpu-scope
// fence per batch, off the consumers' path.
// ---------------------------------------------------------------------------
__device__ void signaler(const DecodeArgs& a, DecSmem& S) {
  const int lane = threadIdx.x & 31;
  int done = 0;
  for (;;) {
    int upto = done, fin = 0;
    if (lane == 0) {
      const unsigned long long t0 = global_ns();
      for (;;) {
        fin = ld_acquire_cta(&S.cons_done);  // first: requests queued before it are seen below
        upto = done;
        while (upto - done < kPubSlots && ld_acquire_cta(&S.pub[upto % kPubSlots].ready) == upto + 1)
          ++upto;
        if (upto > done) break;
        if (fin) {
          // every claimed request must be written before the consumers finish
          const int claimed = ld_acquire_cta(&S.pub_claim);
          if (claimed == done) break;
        }
        if (*(volatile int*)&S.abort || global_ns() - t0 > kWaitLimitNs) {
          upto = -1;  // the consumers gave up (and reported why)
          break;
        }
        __nanosleep(32);
      }
    }
    upto = __shfl_sync(kFull, upto, 0);
    fin = __shfl_sync(kFull, fin, 0);
    if (upto < 0) break;
    if (upto == done) break;  // finished and nothing pending
    fence_gpu();  // every write the consumers made before these requests
    for (int i = done; i < upto; ++i) {
      const PubReq q = S.pub[i % kPubSlots];
      for (int c = lane; c < q.n; c += 32) atomicAdd(q.cnt + c, q.val);
    }
    __syncwarp();
    if (lane == 0) st_release_cta(&S.pub_done, upto);
    done = upto;
  }
  if (lane == 0) st_release_cta(&S.sig_done, 1);
}

template <int G>
// 96 registers: 18 warps, up to 5 per SM sub-partition, fit its 16K registers.
// (A per-kernel register limit instead of launch bounds: the same limit
// without the spills the launch-bounds heuristics leave.)
__global__ void __maxnreg__(96) decode_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  DecSmem& S = *reinterpret_cast<DecSmem*>(smem_raw);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&S.full[s]), 1);
      mbar_init(smem_addr(&S.empty[s]), kCW);
    }
    fence_mbar_init();
    S.abort = 0;
    S.issued = 0;
    S.flag = 0;
    S.pub_claim = S.pub_done = 0;
    S.cons_done = S.sig_done = 0;
  }
  if (tid < kPubSlots) S.pub[tid].ready = 0;
  if (tid < kSlots) S.slot_cnt[tid] = 0u;
  for (int b = tid; b < a.nb; b += kThreads) S.static_w[b] = a.static_w[b];
  __syncthreads();
  if (tid >= kCT + 32) signaler(a, S);
  else if (tid >= kCT) producer<G>(a, S);
  else consumers<G>(a, S);
  __syncthreads();
  if (tid == 0) {
    // let every copy still in flight land before the block exits: the phases
    // of the last kStages issued tiles
    const int is = S.issued;
    for (int q = is - kStages > 0 ? is - kStages : 0; q < is; ++q)
      mbar_wait(smem_addr(&S.full[q % kStages]), (uint32_t)(q / kStages) & 1u, a.status);
    // the last block to finish clears the progress counters for the next launch
    fence_gpu();
    S.flag = atomicAdd(a.end_cnt, 1u) == (unsigned)(a.nb - 1);
    if (S.flag) fence_gpu();
  }
  __syncthreads();
  if (S.flag) {
    for (int i = tid; i < a.counter_words; i += kThreads) a.grp_cnt[i] = 0u;
    if (tid == 0) {
      *a.sel_done = 0u;
      *a.end_cnt = 0u;
    }
  }
}

}  // namespace

cudaError_t decode_blocks(int* nb) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  *nb = sms < kMaxBlocks ? sms : kMaxBlocks;
  return cudaSuccess;
}

template <int G>
static cudaError_t launch_g(const DecodeArgs& a, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(DecSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.nb);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(DecSmem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<G>, a);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  switch (a.G) {
    case 1: return launch_g<1>(a, st);
    case 2: return launch_g<2>(a, st);
    case 4: return launch_g<4>(a, st);
    case 8: return launch_g<8>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace wi
