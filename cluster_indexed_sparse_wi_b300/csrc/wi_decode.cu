// Decode kernel of the wave-index tripartite attention ("RetroInfer: A Vector
// Storage Engine for Scalable Long-Context LLM Inference", technical summary
// (es) §2.A: steady zone, retrieval zone, estimation zone; technical summary
// (ar) §2.a: estimation from the centroids and the value sum, §2.b: retrieved
// KV laid out contiguously for the attention kernel).
//
// One persistent launch, one block per SM.  Each block has 16 consumer warps
// and one producer warp.  The producer streams every byte the block needs
// through a 4-stage shared-memory ring with the TMA bulk-copy engine
// (cp.async.bulk + mbarrier complete_tx); the consumers compute on the staged
// tiles.  Blocks [0, nsel) are selection blocks, the others scoring blocks.
//
//   stage 1  (all blocks) centroid-key tiles (64 rows of kbar, f32) with
//            the group's query rows, in KV-group order, dealt round robin:
//              s[b,h,c] = scale q_h . kbar_c (-inf if n_c = 0)   -> scores
//            every warp counts its finished tiles on the group's counter;
//   stage 2  (selection blocks) once a head's group is fully scored: radix
//            select of the r largest scores (score desc, id asc), the selected
//            clusters' sorted rows and sizes; afterwards the estimate of the
//            selected clusters with a negative sign (all-minus-retrieved is the
//            estimation zone);
//            (scoring blocks) value-sum tiles of a contiguous share of the
//            clusters: the estimate of EVERY non-empty cluster, (m, l = sum n_c
//            e^{s_c-m}, o = sum e^{s_c-m} vsum_c), one partial per (block, KV
//            group, query head);
//   stage 3  (all blocks) steady-zone tiles (K/V rows of the sink and the local
//            window) and retrieved-cluster tiles (K/V rows of the
//            cluster-sorted copies, streamed once the head's selection is
//            published), exact attention with an online softmax; every
//            finished piece adds itself to its head's arrival counter, and a
//            completed head joins a merge queue from which blocks that have
//            finished their tiles take heads and merge all of their partials
//            (log-sum-exp) into out and lse.
//
// There is no grid-wide barrier: each consumer of another block's results
// waits on a counter of exactly what it reads (a KV group's scores, a head's
// selection, a group's estimate pieces, a head's negative estimate), so the
// selections of early groups overlap the scoring of later ones and the
// streaming of value sums and steady rows.  The counters start at zero; the
// last block to finish a launch clears them again.  Every wait is bounded
// (kWaitLimitNs) and reports WI_ERR_DEVICE_TIMEOUT; a block that gives up lets
// its issued copies land before it exits.
//
// Softmax quantities are kept in log2 units (logits scaled by log2 e) so that
// every exponential is an exp2.
#include <float.h>
#include <limits.h>
#include <stddef.h>

#include "wi_device.cuh"
#include "wi_internal.h"

namespace wi {

namespace {

constexpr int kCW = 16;                       // consumer warps
constexpr int kCT = kCW * 32;                 // consumer threads
constexpr int kThreads = kCT + 64;            // + one producer warp + one signaling warp
constexpr int kStages = 4;
constexpr int kTile = kDecodeTile;            // index rows or tokens per tile
constexpr int kRowsPerWarp = kTile / kCW;     // 4
constexpr uint32_t kStageBytes = kTile * 512; // 64 f32 rows, or 64 K + 64 V bf16 rows
constexpr int kQSlotBytes = 8 * kD * 2;       // up to 8 bf16 query rows
constexpr int kBins = 4096;                   // radix-select histogram (12-bit digits)
constexpr int kCand = 1024;                   // selected clusters kept in shared memory
constexpr int kSelChunk = kCT * 16;           // keys per register chunk (16 per thread)
// candidate windows below the largest key, in 12-bit key digits (8 per octave)
constexpr int kNumWindows = 8;
__host__ __device__ constexpr uint32_t window_digits(int w) { return 2u * (w + 1); }  // 2, 4, ..., 16
static_assert(kRowsPerWarp == 4, "tile layout");

enum : int { kTileEnd = 0, kTileSteady = 1, kTileRet = 2, kTileIndex = 3 };

// Written by the producer for every staged tile, so that the consumers do no
// index arithmetic of their own.
struct TileInfo {
  int kind;
  int bh;     // exact tiles: query head (b*Hq + h); index tiles: KV group (b*Hkv + g)
  int ntok;   // rows (index tiles) or tokens (exact tiles) staged
  int last;   // exact tiles: the piece ends with this tile
  int units;  // exact tiles: units the piece adds to its head's arrival counter
  int c0;     // index tiles: first cluster of the tile
  int h0;     // index tiles: first query head of the group (b*Hq + g*G)
  int pad;
};

struct Cand {
  int c[kCand];
  float s[kCand];
  int n[kCand];
  int row[kCand];
};

// Side data of one staged index tile: the sizes of its clusters and (value-sum
// tiles) the scores of the group's query heads, staged with the tile.
struct __align__(16) StageSide {
  int n[kTile];
  float s[8][kTile];
};

// A request to the signaling warp: after a gpu-scope fence (covering every
// write the consumers made before queueing it), add val to *cnt (kPubAdd),
// set *cnt = val (kPubSet), or add val to head bh's arrival counter and queue
// the head for merging in this block if that completes it (kPubPiece).
enum : int { kPubAdd = 0, kPubSet = 1, kPubPiece = 2 };
struct PubReq {
  unsigned* cnt;
  unsigned val;
  int op, bh, pad;
};
constexpr int kPubSlots = 16;

struct __align__(128) DecSmem {
  unsigned char ring[kStages][kStageBytes];  // bulk-copy destinations (16-byte aligned)
  StageSide sd[kStages];
  unsigned char qs[kStages][kQSlotBytes];
  float red_o[kCW][kD];
  float red_m[kCW];
  float red_l[kCW];
  union __align__(16) {
    int hist[kBins];
    Cand cand;
    float w[kBins];
    struct {                       // a fast-path selection (ids ascending)
      unsigned long long comp[kCT];  // candidate composites, then free
      int c[kCT];                  // cluster ids
      float s[kCT];                // scores
      int n[kCT];                  // sizes
    } kept;
  } u;
  unsigned long long full[kStages];
  unsigned long long empty[kStages];
  TileInfo info[kStages];
  int2 scan[2][kCW];
  int sel_i[4];
  uint32_t red_u[2][kCW];
  uint32_t win_sum[2][kCW][kNumWindows / 2];
  int abort;              // some wait of this block gave up
  int issued;             // tiles whose copies the producer issued
  int confirmed;          // tiles whose full barrier the consumers saw complete
  int flag;
  int scored;             // stage-1 tiles whose scores every consumer warp has stored
  PubReq pub[kPubSlots];  // requests to the signaling warp (ring)
  int pub_tail;           // requests queued (consumer thread 0)
  int pub_head;           // requests done (signaling warp)
  int cons_done;          // the consumers queue no more requests
  int sig_done;           // the signaling warp has finished
};
static_assert(offsetof(DecSmem, qs) % 16 == 0, "bulk-copy alignment");
static_assert(offsetof(DecSmem, sd) % 16 == 0, "bulk-copy alignment");
static_assert(offsetof(DecSmem, red_o) % 16 == 0, "float4 alignment");
static_assert(offsetof(DecSmem, full) % 8 == 0, "mbarrier alignment");
static_assert(offsetof(DecSmem, u) % 16 == 0, "scratch union alignment");

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Named barrier 1 over the 512 consumer threads (the producer warp never
// takes part).
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
__device__ __forceinline__ uint32_t score_key(float s) {
  return (s == -INFINITY) ? 0u : float_key(s);  // 0 <=> empty cluster
}

// Progress counters: a count that only grows within a launch.  Writers make
// their results visible (every writing thread fences, then a barrier) before
// one thread adds to the count; a reader waits (acquire) until the count
// reaches what it needs.
__device__ __forceinline__ void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void st_release_cta(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_cta(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}
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
    __nanosleep(128);
    if (ld_acquire(cnt) >= target) return true;
    if (*(volatile const int*)abort) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      report(status, WI_ERR_DEVICE_TIMEOUT);
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

// Block-range helpers for the uniform partitions: block b of nb owns
// [b*len/nb, (b+1)*len/nb).
__device__ __forceinline__ long long part_lo(long long b, long long len, int nb) {
  return b * len / nb;
}
__device__ __forceinline__ int part_owner(long long p, long long len, int nb) {
  return (int)(((p + 1) * nb - 1) / len);
}

struct Sched {
  bool sel;                    // a selection block
  int sel0, sel_step;          // its heads sel0, sel0 + sel_step, ... < B*Hq
  int k0, kstep, n1;           // centroid-key tiles k0 + i*kstep, i < n1 (every block)
  int kj, nk;                  // scoring block kj of nk ...
  int v0, v1;                  // ... and its value-sum tiles [v0, v1)
  long long s0, s1;            // steady tiles
  long long r0, r1;            // retrieved slots
};

__device__ Sched schedule(const DecodeArgs& a, int b) {
  Sched s;
  const long long nt = (long long)a.B * a.Hkv * a.tpg;
  s.sel = b < a.nsel;
  s.sel0 = b;
  s.sel_step = a.nsel;
  s.nk = a.nb - a.nsel;
  s.kj = b - a.nsel;
  // centroid-key tiles are dealt round robin over all blocks in KV-group
  // order (the selection blocks have nothing else to do until a group is done)
  s.k0 = b;
  s.kstep = a.nb;
  s.n1 = b < nt ? (int)((nt - b + a.nb - 1) / a.nb) : 0;
  s.v0 = s.v1 = 0;
  if (!s.sel) {
    s.v0 = (int)part_lo(s.kj, nt, s.nk);
    s.v1 = (int)part_lo(s.kj + 1, nt, s.nk);
  }
  const long long nst = (long long)a.B * a.Hq * a.tph;
  s.s0 = part_lo(b, nst, a.nb);
  s.s1 = part_lo(b + 1, nst, a.nb);
  const long long nr = (long long)a.B * a.Hq * a.r;
  s.r0 = part_lo(b, nr, a.nb);
  s.r1 = part_lo(b + 1, nr, a.nb);
  return s;
}

// Combine the 16 consumer warps' (m, l, o) into one partial at dst:
// dst[0] = m (log2 units), dst[1] = sign * l, dst[2..] = sign * o.
// m and l are warp-uniform; o holds this lane's 4 dimensions.  Ends with a
// consumer barrier, after which the partial may be published.
__device__ void combine_write(DecSmem& S, float m, float l, float4 o, float* dst, float sign) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (lane == 0) {
    S.red_m[warp] = m;
    S.red_l[warp] = l;
  }
  reinterpret_cast<float4*>(S.red_o[warp])[lane] = o;
  csync();
  if (tid < kD) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCW; ++w) M = fmaxf(M, S.red_m[w]);
    float L = 0.f, O = 0.f;
    if (M > -INFINITY) {
#pragma unroll
      for (int w = 0; w < kCW; ++w) {
        const float mw = S.red_m[w];
        const float f = mw > -INFINITY ? exp2f(mw - M) : 0.f;
        L += S.red_l[w] * f;
        O += S.red_o[w][tid] * f;
      }
    }
    if (tid == 0) {
      dst[0] = (L > 0.f) ? M : -INFINITY;
      dst[1] = sign * L;
    }
    dst[2 + tid] = sign * O;
  }
  csync();
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

// ---------------------------------------------------------------------------
// selection of one query head (all 512 consumers)
// ---------------------------------------------------------------------------
// T = the r_eff = min(r, non-empty) largest scores, ties to the lower id.
// Keys (order-preserving images of the scores, 0 = empty cluster) are held in
// registers, 16 consecutive ids per thread.
//   Up to 8192 clusters: after one barrier for the count and range of the
//   keys, one pass counts the keys of 8 windows below the largest (2, 4, ...,
//   16 digits of the top 12 key bits) and one block scan of those counts
//   gives every thread its place in each window.  The smallest window holding
//   at least r_eff keys is gathered in id order (at most 512 candidates) and
//   each candidate counts the candidates ranked above it by (key desc, id
//   asc): it is selected iff fewer than r_eff are.  A last scan writes the
//   selected ids ascending with their clusters' sizes and first sorted rows,
//   loaded while the ranks are counted.
//   Otherwise (more clusters, or no window small enough): an exact radix
//   select over the keys, 12 bits per pass, gives a threshold (Kb, cb) -- a
//   cluster is selected iff k > Kb, or k == Kb and its id <= cb -- and a
//   compaction pass over all keys writes the selection.
template <int G>
__device__ int select_head(const DecodeArgs& a, DecSmem& S, int bh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = bh / a.Hq, h = bh - b * a.Hq, g = h / G;
  const size_t bg = (size_t)b * a.Hkv + g;
  const int C = a.C, r = a.r, rs = r > 0 ? r : 1;
  const float* sc = a.scores + (size_t)bh * C;
  const int* sz = a.size + bg * C;
  const int* off = a.offset + bg * (C + 1);
  const int nch = (C + kSelChunk - 1) / kSelChunk;
  const bool vec = (C & 3) == 0;  // rows of scores start on 16-byte boundaries
  int buf = 0;

  auto load16 = [&](int ch, uint32_t(&k)[16]) {
    const int c0 = ch * kSelChunk + tid * 16;
    if (vec && c0 + 16 <= C) {
      const float4* p = reinterpret_cast<const float4*>(sc + c0);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 f = __ldcg(p + j);
        k[4 * j] = score_key(f.x);
        k[4 * j + 1] = score_key(f.y);
        k[4 * j + 2] = score_key(f.z);
        k[4 * j + 3] = score_key(f.w);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) k[j] = (c0 + j < C) ? score_key(__ldcg(sc + c0 + j)) : 0u;
    }
  };
  uint32_t k0[16];
  load16(0, k0);
  // f(key, id) over this thread's keys
  auto visit = [&](auto&& f) {
#pragma unroll
    for (int j = 0; j < 16; ++j) f(k0[j], tid * 16 + j);
    for (int ch = 1; ch < nch; ++ch) {
      uint32_t kk[16];
      load16(ch, kk);
#pragma unroll
      for (int j = 0; j < 16; ++j) f(kk[j], ch * kSelChunk + tid * 16 + j);
    }
  };

  // non-empty count and key range
  int valid = 0;
  uint32_t kmax = 0u, kmin = 0xffffffffu;
  visit([&](uint32_t k, int) {  // branch-free: selects, no divergent jumps
    valid += (int)(k != 0u);
    kmax = max(kmax, k);
    kmin = min(kmin, k != 0u ? k : 0xffffffffu);
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    valid += __shfl_xor_sync(kFull, valid, o);
    kmax = max(kmax, __shfl_xor_sync(kFull, kmax, o));
    kmin = min(kmin, __shfl_xor_sync(kFull, kmin, o));
  }
  {
    int2* sh = S.scan[buf];
    buf ^= 1;
    if (lane == 0) {
      sh[warp] = make_int2(valid, 0);
      S.red_u[0][warp] = kmax;
      S.red_u[1][warp] = kmin;
    }
    csync();
    valid = 0;
    kmax = 0u;
    kmin = 0xffffffffu;
#pragma unroll
    for (int w = 0; w < kCW; ++w) {
      valid += sh[w].x;
      kmax = max(kmax, S.red_u[0][w]);
      kmin = min(kmin, S.red_u[1][w]);
    }
  }
  const int r_eff = min(r, valid);
  if (tid == 0) a.head_max[bh] = valid > 0 ? key_float(kmax) : -INFINITY;

  // threshold (Kb, cb); the default selects nothing
  uint32_t Kb = 0xffffffffu;
  int cb = -1;
  if (r_eff > 0 && r_eff == valid) {
    Kb = 0u;  // every non-empty cluster
  } else if (r_eff > 0) {
    bool done = false;
    if (nch == 1) {
      // Candidates: keys whose top 12 bits (d = k >> 20) lie within w digits
      // of the largest key's, d_max - d <= w, for the smallest w of 2, 4, ..., 16
      // that holds at least r_eff keys.  One pass counts every window and one
      // block scan of the counts gives each thread its gather position in all
      // of them.
      const uint32_t dmax = kmax >> 20;
      // per-thread counts of the windows, one byte each (at most 16 keys): a
      // key o digits below the largest is in windows w >= w0(o)
      unsigned long long cw64 = 0ull;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t k = k0[j];
        const uint32_t o = dmax - (k >> 20);
        const uint32_t w0 = o <= 2u ? 0u : min((o - 1u) >> 1, 8u);  // 8: in no window
        const unsigned long long inc = w0 < 8u ? (0x0101010101010101ull << (8u * w0)) : 0ull;
        cw64 += k != 0u ? inc : 0ull;
      }
      // windows 2x and 2x+1 as two 16-bit fields of word x (block totals <= 8192)
      uint32_t own[4], incl[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const uint32_t c = (uint32_t)(cw64 >> (16 * x));
        own[x] = (c & 0xffu) | ((c >> 8 & 0xffu) << 16);
        incl[x] = own[x];
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const uint32_t t = __shfl_up_sync(kFull, incl[x], o);
          if (lane >= o) incl[x] += t;
        }
      }
      uint32_t(*wsum)[kNumWindows / 2] =
          reinterpret_cast<uint32_t(*)[kNumWindows / 2]>(S.win_sum[buf]);
      buf ^= 1;
      if (lane == 31) {
#pragma unroll
        for (int x = 0; x < 4; ++x) wsum[warp][x] = incl[x];
      }
      csync();
      uint32_t base[4] = {0u, 0u, 0u, 0u}, tot[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int y = 0; y < kCW; ++y) {
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const uint32_t t = wsum[y][x];
          if (y < warp) base[x] += t;
          tot[x] += t;
        }
      }
      int win = -1, n_cand = 0;
#pragma unroll
      for (int w = kNumWindows - 1; w >= 0; --w) {
        const int t = (int)((tot[w / 2] >> (16 * (w % 2))) & 0xffffu);
        if (t >= r_eff) {
          win = w;
          n_cand = t;
        }
      }
      if (win >= 0 && n_cand <= kCT) {
        // gather the candidates in id order as composites (key << 32 | ~id):
        // a larger composite is selected first; unique since the ids are
        uint32_t pos = 0u;
#pragma unroll
        for (int w = 0; w < kNumWindows; ++w)
          if (w == win)
            pos = ((base[w / 2] + incl[w / 2] - own[w / 2]) >> (16 * (w % 2))) & 0xffffu;
        const uint32_t wsel = window_digits(win);
        unsigned long long* cand = S.u.kept.comp;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t k = k0[j];
          if (k != 0u && dmax - (k >> 20) <= wsel)
            cand[pos++] = ((unsigned long long)k << 32) | (unsigned long long)(0xffffffffu - (uint32_t)(tid * 16 + j));
        }
        csync();
        // Thread t < n_cand ranks candidate t against all of them; its
        // cluster's size and first sorted row are loaded meanwhile.
        const bool has = tid < n_cand;
        const unsigned long long mine = has ? cand[tid] : 0ull;
        const int cid = (int)(0xffffffffu - (uint32_t)mine);
        int nj = 0, rowj = 0;
        if (has) {
          nj = __ldg(sz + cid);
          rowj = __ldg(off + cid);
        }
        int rank = 0;
        if (has) {
          const ulonglong2* c2 = reinterpret_cast<const ulonglong2*>(cand);
          const int half = n_cand >> 1;
#pragma unroll 4
          for (int j = 0; j < half; ++j) {
            const ulonglong2 v = c2[j];
            rank += (int)(v.x > mine) + (int)(v.y > mine);
          }
          if (n_cand & 1) rank += (int)(cand[n_cand - 1] > mine);
        }
        const bool take = has && rank < r_eff;
        int2 ptot;
        const int p = cscan2(make_int2(take ? 1 : 0, 0), S, &ptot, buf).x;  // ids ascending
        int* ids = a.sel_ids + (size_t)bh * rs;
        int* rows = a.sel_rows + (size_t)bh * rs;
        int* cnts = a.sel_cnts + (size_t)bh * rs;
        int* topk = a.topk_out ? a.topk_out + (size_t)bh * r : nullptr;
        if (take) {
          if (nj < 0 || rowj < 0 || (long long)rowj + nj > a.N_idx) {
            report(a.status, WI_ERR_INDEX_MISMATCH);  // inconsistent index: stage nothing
            nj = 0;
            rowj = 0;
          }
          ids[p] = cid;
          rows[p] = rowj;
          cnts[p] = nj;
          if (topk) topk[p] = cid;
          // kept for the estimate of the selection (estimate_kept)
          S.u.kept.c[p] = cid;
          S.u.kept.s[p] = key_float((uint32_t)(mine >> 32));
          S.u.kept.n[p] = nj;
        }
        for (int i = r_eff + tid; i < rs; i += kCT) {
          ids[i] = -1;
          rows[i] = 0;
          cnts[i] = 0;
          if (topk && i < r) topk[i] = -1;
        }
        csync();  // the selection is published after this barrier
        return r_eff;
      }
    }
    if (!done) {
      // exact radix select over the keys, 12 bits per pass from the highest
      // bit in which they differ
      int remaining = r_eff;
      uint32_t prefix = 0u, mask = 0u;
      bool tie = false;
      if (kmax == kmin) {
        prefix = kmax;
        mask = 0xffffffffu;
        tie = true;
      } else {
        int bit = 31 - __clz(kmax ^ kmin);
        mask = (bit == 31) ? 0u : (0xffffffffu << (bit + 1));
        prefix = kmax & mask;
        for (int pass = 0;; ++pass) {
          const int width = min(12, bit + 1), shift = bit + 1 - width;
          const uint32_t dmask = (1u << width) - 1u;
          const int nbins = 1 << width;
          for (int i = tid; i < nbins; i += kCT) S.u.hist[i] = 0;
          csync();
          const uint32_t pf = prefix, mk = mask;
          visit([&](uint32_t k, int) {
            if (k != 0u && (k & mk) == pf) atomicAdd(&S.u.hist[(k >> shift) & dmask], 1);
          });
          csync();
          const int bhi = nbins - 8 * tid, blo = max(0, bhi - 8);
          int own = 0;
          if (bhi > 0)
            for (int i = blo; i < bhi; ++i) own += S.u.hist[i];
          int2 tot;
          const int excl = cscan2(make_int2(own, 0), S, &tot, buf).x;
          uint32_t* hand = S.red_u[pass & 1];
          if (own > 0 && excl < remaining && remaining <= excl + own) {
            int acc = excl;
            for (int i = bhi - 1; i >= blo; --i) {
              const int cnt = S.u.hist[i];
              if (acc + cnt >= remaining) {
                hand[0] = (uint32_t)i;
                hand[1] = (uint32_t)acc;
                hand[2] = (uint32_t)cnt;
                break;
              }
              acc += cnt;
            }
          }
          csync();
          const int D = (int)hand[0], above = (int)hand[1], cntD = (int)hand[2];
          remaining -= above;
          prefix |= (uint32_t)D << shift;
          mask |= dmask << shift;
          if (cntD == remaining) break;  // the boundary bin is taken whole
          if (shift == 0) {              // equal full keys straddle the boundary
            tie = true;
            break;
          }
          bit = shift - 1;
        }
      }
      if (!tie) {
        // (k & mask) >= prefix  <=>  k >= prefix
        Kb = prefix > 0u ? prefix - 1u : 0u;
        cb = -1;
      } else {
        // k > prefix, plus the `remaining` lowest ids with k == prefix
        Kb = prefix;
        int eq_base = 0;
        for (int ch = 0; ch < nch; ++ch) {
          uint32_t kk[16];
          if (ch == 0) {
#pragma unroll
            for (int j = 0; j < 16; ++j) kk[j] = k0[j];
          } else {
            load16(ch, kk);
          }
          int ne = 0;
#pragma unroll
          for (int j = 0; j < 16; ++j) ne += (kk[j] == prefix);
          int2 tot;
          const int before = eq_base + cscan2(make_int2(ne, 0), S, &tot, buf).x;
          eq_base += tot.x;
          if (before < remaining && remaining <= before + ne) {
            int x = before;
            for (int j = 0; j < 16; ++j) {
              if (kk[j] == prefix && ++x == remaining) {
                S.red_u[1][2] = (uint32_t)(ch * kSelChunk + tid * 16 + j);
                break;
              }
            }
          }
        }
        csync();
        cb = (int)S.red_u[1][2];
      }
    }
  }

  // ordered compaction (ids ascending) into shared memory and the id outputs
  int* ids = a.sel_ids + (size_t)bh * rs;
  int* rows = a.sel_rows + (size_t)bh * rs;
  int* cnts = a.sel_cnts + (size_t)bh * rs;
  int* topk = a.topk_out ? a.topk_out + (size_t)bh * r : nullptr;
  int sel_base = 0;
  if (r_eff > 0) {
    for (int ch = 0; ch < nch; ++ch) {
      uint32_t kk[16];
      if (ch == 0) {
#pragma unroll
        for (int j = 0; j < 16; ++j) kk[j] = k0[j];
      } else {
        load16(ch, kk);
      }
      const int c0 = ch * kSelChunk + tid * 16;
      uint32_t selmask = 0u;
      int nsel = 0;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t k = kk[j];
        if (k != 0u && (k > Kb || (k == Kb && c0 + j <= cb))) {
          selmask |= 1u << j;
          ++nsel;
        }
      }
      int2 tot;
      int pos = sel_base + cscan2(make_int2(nsel, 0), S, &tot, buf).x;
      sel_base += tot.x;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if ((selmask & (1u << j)) && pos < r) {
          const int c = c0 + j;
          ids[pos] = c;
          if (topk) topk[pos] = c;
          if (pos < kCand) {
            S.u.cand.c[pos] = c;
            S.u.cand.s[pos] = key_float(kk[j]);
          }
          ++pos;
        }
      }
    }
  }
  const int nsel_tot = min(sel_base, r);  // == r_eff
  for (int i = nsel_tot + tid; i < rs; i += kCT) {
    ids[i] = -1;
    rows[i] = 0;
    cnts[i] = 0;
    if (topk && i < r) topk[i] = -1;
  }
  csync();

  // the selected clusters' sizes and first sorted rows (one round of
  // independent loads, 16 clusters per warp)
  for (int j0 = warp * 32; j0 < nsel_tot; j0 += kCW * 32) {
    const int j = j0 + lane;
    if (j < nsel_tot) {
      const int cj = j < kCand ? S.u.cand.c[j] : ids[j];
      int nj = __ldg(sz + cj), rowj = __ldg(off + cj);
      if (nj < 0 || rowj < 0 || (long long)rowj + nj > a.N_idx) {
        report(a.status, WI_ERR_INDEX_MISMATCH);  // inconsistent index: stage nothing
        nj = 0;
        rowj = 0;
      }
      rows[j] = rowj;
      cnts[j] = nj;
    }
  }
  csync();  // the selection is published after this barrier
  return -1;
}

// The estimate of one head's selected clusters (kept with a negative sign):
// (m, l = sum n_c e^{s_c - m}, o = sum e^{s_c - m} vsum_c) over T.  It reads
// the selection outputs back (written by this block) and runs after the block
// has published its selections.
template <int G>
__device__ void estimate_selected(const DecodeArgs& a, DecSmem& S, int bh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = bh / a.Hq, h = bh - b * a.Hq, g = h / G;
  const size_t bg = (size_t)b * a.Hkv + g;
  const int r = a.r, rs = r > 0 ? r : 1;
  const int* ids = a.sel_ids + (size_t)bh * rs;
  const int* cnts = a.sel_cnts + (size_t)bh * rs;
  const float* sc = a.scores + (size_t)bh * a.C;
  const float4* vs = reinterpret_cast<const float4*>(a.vsum + bg * (size_t)a.C * kD);
  float m = -INFINITY, l = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = warp * 8; j0 < r; j0 += kCW * 8) {
    const int j = j0 + (lane & 7);
    int cj = -1, nj = 0;
    float sj = -INFINITY;
    if (lane < 8 && j < r) {
      cj = __ldcg(ids + j);
      nj = __ldcg(cnts + j);
      if (cj >= 0 && cj < a.C && nj > 0) sj = __ldcg(sc + cj) * kLog2e;
      else nj = 0;
    }
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int cu = __shfl_sync(kFull, cj, u);
      v[u] = (cu >= 0 && cu < a.C) ? __ldg(vs + (size_t)cu * (kD / 4) + lane)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float mt = sj;
#pragma unroll
    for (int o2 = 4; o2 > 0; o2 >>= 1) mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, o2));
    mt = __shfl_sync(kFull, mt, 0);
    if (mt > -INFINITY) {
      const float mn = fmaxf(m, mt);
      const float corr = (m > -INFINITY) ? exp2f(m - mn) : 0.f;
      const float p = (sj > -INFINITY) ? exp2f(sj - mn) : 0.f;
      l *= corr;
      o.x *= corr;
      o.y *= corr;
      o.z *= corr;
      o.w *= corr;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float pu = __shfl_sync(kFull, p, u);
        const float nu = (float)__shfl_sync(kFull, nj, u);
        l += pu * nu;
        o.x += pu * v[u].x;
        o.y += pu * v[u].y;
        o.z += pu * v[u].z;
        o.w += pu * v[u].w;
      }
      m = mn;
    }
  }
  combine_write(S, m, l, o, a.neg_part + (size_t)bh * kPartStride, -1.f);
}

// The same estimate for a fast-path selection, from the ids, scores and sizes
// select_head kept in shared memory: every value-sum row of the selection is
// loaded in one round (warp w takes the selected j = w, w + 16, ...).
template <int G>
__device__ void estimate_kept(const DecodeArgs& a, DecSmem& S, int bh, int n_sel) {
  constexpr int kRows = 10;  // rows per warp per round: 160 per round
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = bh / a.Hq, g = (bh - b * a.Hq) / G;
  const size_t bg = (size_t)b * a.Hkv + g;
  const float4* vs = reinterpret_cast<const float4*>(a.vsum + bg * (size_t)a.C * kD);
  float m = -INFINITY, l = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = warp; j0 < n_sel; j0 += kCW * kRows) {
    float4 v[kRows];
    float x[kRows];
    int n[kRows];
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      const int j = j0 + u * kCW;
      n[u] = 0;
      x[u] = -INFINITY;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < n_sel) {
        n[u] = S.u.kept.n[j];
        x[u] = S.u.kept.s[j] * kLog2e;
        v[u] = __ldg(vs + (size_t)S.u.kept.c[j] * (kD / 4) + lane);
      }
    }
    float mt = -INFINITY;
#pragma unroll
    for (int u = 0; u < kRows; ++u)
      if (n[u] > 0) mt = fmaxf(mt, x[u]);
    if (mt > -INFINITY) {
      const float mn = fmaxf(m, mt);
      const float corr = (m > -INFINITY) ? exp2f(m - mn) : 0.f;
      l *= corr;
      o.x *= corr;
      o.y *= corr;
      o.z *= corr;
      o.w *= corr;
#pragma unroll
      for (int u = 0; u < kRows; ++u) {
        if (n[u] > 0) {
          const float pu = exp2f(x[u] - mn);
          l += pu * (float)n[u];
          o.x += pu * v[u].x;
          o.y += pu * v[u].y;
          o.z += pu * v[u].z;
          o.w += pu * v[u].w;
        }
      }
      m = mn;
    }
  }
  combine_write(S, m, l, o, a.neg_part + (size_t)bh * kPartStride, -1.f);
}

// ---------------------------------------------------------------------------
// merge of one query head (all 512 consumers)
// ---------------------------------------------------------------------------
// Partials: steady pieces, retrieved pieces (exact, +), the KV group's
// estimate pieces (every non-empty cluster, +) and the selected clusters'
// estimate (-).  out = O / L, lse = (M + log2 L) ln 2.  Every partial is
// loaded in one round of independent loads (thread (q, d) holds element d of
// the partials q, q + 4, ...), so the merge costs one global round trip.
template <int G>
__device__ void merge_head(const DecodeArgs& a, DecSmem& S, int bh) {
  constexpr int kPerThread = 8;  // partials per thread and round: 32 per round
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = bh / a.Hq, h = bh - b * a.Hq, g = h / G, hl = h - g * G;
  const int bg = b * a.Hkv + g;
  const long long H = (long long)a.B * a.Hq;
  // piece owners (a block with an empty range wrote no piece)
  const long long nst = H * a.tph, nr = H * a.r;
  int s_lo = 0, s_hi = -1, r_lo = 0, r_hi = -1;
  if (a.tph > 0) {
    s_lo = part_owner((long long)bh * a.tph, nst, a.nb);
    s_hi = part_owner((long long)bh * a.tph + a.tph - 1, nst, a.nb);
  }
  if (a.r > 0) {
    r_lo = part_owner((long long)bh * a.r, nr, a.nb);
    r_hi = part_owner((long long)bh * a.r + a.r - 1, nr, a.nb);
  }
  // estimate pieces: the scoring blocks whose value-sum share meets the group
  const int nk = a.nb - a.nsel;
  const long long nt = (long long)a.B * a.Hkv * a.tpg;
  const int e_lo = part_owner((long long)bg * a.tpg, nt, nk);
  const int e_hi = part_owner((long long)bg * a.tpg + a.tpg - 1, nt, nk);
  const int ns_ = s_hi - s_lo + 1, nr_ = r_hi - r_lo + 1, ne_ = e_hi - e_lo + 1;
  const int P = ns_ + nr_ + ne_ + 1;
  // pointer of partial i, or null when that block wrote none
  // (with at least nb units every block owns some, and no division is needed)
  auto part = [&](int i) -> const float* {
    if (i < ns_) {
      const int o = s_lo + i;
      if (nst < a.nb && part_lo(o, nst, a.nb) == part_lo(o + 1, nst, a.nb)) return nullptr;
      return a.std_part + (size_t)(o + bh) * kPartStride;
    }
    i -= ns_;
    if (i < nr_) {
      const int o = r_lo + i;
      if (nr < a.nb && part_lo(o, nr, a.nb) == part_lo(o + 1, nr, a.nb)) return nullptr;
      return a.ret_part + (size_t)(o + bh) * kPartStride;
    }
    i -= nr_;
    if (i < ne_) {
      const int o = e_lo + i;
      if (nt < nk && part_lo(o, nt, nk) == part_lo(o + 1, nt, nk)) return nullptr;
      return a.est_part + ((size_t)(a.nsel + o + bg) * G + hl) * kPartStride;
    }
    return a.neg_part + (size_t)bh * kPartStride;
  };
  // partial pointers, computed once (thread i: partial i)
  const float** ptrs = reinterpret_cast<const float**>(S.u.w);     // [P]
  float* wm = S.u.w + 2 * 1024;                                     // [32] m, then weight
  float* wl = wm + 64;                                              // [32] l
  for (int i = tid; i < P; i += kCT) ptrs[i] = part(i);
  csync();
  const int dim = tid & (kD - 1), qq = tid >> 7;
  float M = -INFINITY, L = 0.f, O = 0.f;
  for (int base = 0; base < P; base += 4 * kPerThread) {
    const int np = min(4 * kPerThread, P - base);
    // one round of independent loads: (m, l) by threads < np, element dim of
    // partials base + qq + 4u by thread (qq, dim)
    float mi = -INFINITY, li = 0.f;
    if (tid < np) {
      const float* p = ptrs[base + tid];
      if (p) {
        mi = __ldcg(p);
        li = __ldcg(p + 1);
      }
    }
    float ov[kPerThread];
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
      const int i = qq + 4 * u;
      const float* p = i < np ? ptrs[base + i] : nullptr;
      ov[u] = p ? __ldcg(p + 2 + dim) : 0.f;
    }
    // warp 0: new running max, weights of this round's partials, L
    if (warp == 0) {
      float mc = fmaxf(M, warp_max(mi));
      const float f = (mi > -INFINITY) ? exp2f(mi - mc) : 0.f;
      const float corr = (M > -INFINITY) ? exp2f(M - mc) : 0.f;
      const float lr = warp_sum(f * li);
      if (lane < 32) wm[lane] = f;
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
  float* red = &S.red_o[0][0];
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
// producer warp
// ---------------------------------------------------------------------------
template <int G>
__device__ void producer(const DecodeArgs& a, DecSmem& S, const Sched& sc) {
  const int lane = threadIdx.x & 31;
  uint32_t seq = 0;
  // test hook: the first tile with copies in every block loses them
  bool inject = a.inject != 0, skipped = false;
  const int ns = a.sink + a.window;

  // claim the next ring slot (warp-uniform); false once this block aborted
  auto slot = [&](int& stage) -> bool {
    stage = (int)(seq % kStages);
    int good = 1;
    if (lane == 0) {
      if (*(volatile int*)&S.abort) {
        good = 0;
      } else if (seq >= (uint32_t)kStages) {
        good = mbar_wait(smem_addr(&S.empty[stage]), ((seq / kStages) - 1u) & 1u, a.status);
      }
      if (good) fence_proxy_async_smem();
      else S.abort = 1;
    }
    return __shfl_sync(kFull, good, 0) != 0;
  };
  // lane 0: tile description + expected bytes; then lanes issue the copies
  auto post = [&](int stage, int kind, int bh, int ntok, int last, int units, uint32_t bytes,
                  int c0 = 0, int h0 = 0) {
    if (lane == 0) {
      TileInfo t;
      t.kind = kind;
      t.bh = bh;
      t.ntok = ntok;
      t.last = last;
      t.units = units;
      t.c0 = c0;
      t.h0 = h0;
      t.pad = 0;
      S.info[stage] = t;
      mbar_arrive_expect_tx(smem_addr(&S.full[stage]), bytes);
    }
    __syncwarp();
  };
  auto commit = [&]() {
    if (__any_sync(kFull, skipped)) inject = false;
    __syncwarp();
    if (lane == 0) S.issued = (int)(seq + 1);
    ++seq;
  };
  auto copy = [&](int stage, uint32_t dst_off, const void* src, uint32_t bytes) {
    if (inject) skipped = true;
    else bulk_g2s(smem_addr(S.ring[stage]) + dst_off, src, bytes, smem_addr(&S.full[stage]));
  };
  auto copy_q = [&](int stage, const void* src, uint32_t bytes) {
    if (inject) skipped = true;
    else bulk_g2s(smem_addr(S.qs[stage]), src, bytes, smem_addr(&S.full[stage]));
  };
  auto copy_to = [&](void* dst, const void* src, uint32_t bytes, int stage) {
    if (inject) skipped = true;
    else bulk_g2s(smem_addr(dst), src, bytes, smem_addr(&S.full[stage]));
  };

  // stage 1 (every block): centroid-key tiles k0, k0 + kstep, ...
  // with the group's query rows and the clusters' sizes; then (scoring
  // blocks) the value-sum tiles [v0, v1) with the sizes and the group's
  // scores (each group's once every score of it is written)
  const bool side_bulk = (a.C & 3) == 0;  // rows of sizes and scores start 16-byte aligned
  for (int pass = 0; pass < 2; ++pass) {
    if ((pass == 1 && sc.sel) || !(a.stages & (pass == 0 ? kStageScore : kStageSelect))) continue;
    const float* src = pass == 0 ? a.kbar : a.vsum;
    const int n = pass == 0 ? sc.n1 : sc.v1 - sc.v0;
    int ready_bg = -1;
    for (int i = 0; i < n; ++i) {
      const int T = pass == 0 ? sc.k0 + i * sc.kstep : sc.v0 + i;
      const int bg = T / a.tpg, c0 = (T - bg * a.tpg) * kTile;
      const int nrows = min(kTile, a.C - c0);
      const int b = bg / a.Hkv, g = bg - b * a.Hkv;
      const int h0 = b * a.Hq + g * G;
      const float* srow = a.scores + (size_t)h0 * a.C + c0;  // scores[b, g*G, c0]
      if (pass == 1 && bg != ready_bg && a.fused) {
        int good = 1;
        if (lane == 0) {
          good = !*(volatile int*)&S.abort &&
                 count_wait(a.grp_cnt + bg, (unsigned)(a.tpg * kCW), a.status, &S.abort);
          if (good) fence_proxy_async_global();  // the scores, read by the copy engine
          else S.abort = 1;
        }
        if (!__shfl_sync(kFull, good, 0)) return;
        ready_bg = bg;
      }
      int stage;
      if (!slot(stage)) return;
      const bool bulk = side_bulk && (nrows & 3) == 0;
      const int nside = pass == 0 ? 1 : 1 + G;  // rows of side data (sizes, scores)
      StageSide& sd = S.sd[stage];
      if (!bulk) {  // ragged: plain loads, stored before the stage is posted
        for (int k = lane; k < nside * kTile; k += 32) {
          const int row = k / kTile, c = k - row * kTile;
          if (row == 0) sd.n[c] = c < nrows ? __ldg(a.size + (size_t)bg * a.C + c0 + c) : 0;
          else sd.s[row - 1][c] = c < nrows ? __ldcg(srow + (size_t)(row - 1) * a.C + c) : -INFINITY;
        }
        __syncwarp();
      }
      const uint32_t qbytes = pass == 0 ? (uint32_t)G * kD * 2 : 0u;
      const uint32_t sbytes = bulk ? (uint32_t)(nside * nrows * 4) : 0u;
      post(stage, kTileIndex, bg, nrows, 0, 0, (uint32_t)nrows * 512u + qbytes + sbytes, c0, h0);
      if (lane == 0) copy(stage, 0, src + ((size_t)bg * a.C + c0) * kD, (uint32_t)nrows * 512u);
      if (lane == 1 && pass == 0)
        copy_q(stage, a.q + ((size_t)b * a.Hq + (size_t)g * G) * kD, qbytes);
      if (bulk && lane == 2) copy_to(sd.n, a.size + (size_t)bg * a.C + c0, (uint32_t)nrows * 4u, stage);
      if (bulk && pass == 1 && lane >= 3 && lane < 3 + G)
        copy_to(sd.s[lane - 3], srow + (size_t)(lane - 3) * a.C, (uint32_t)nrows * 4u, stage);
      commit();
    }
  }
  if (!(a.stages & kStageAttend)) return;

  // stage 3a: steady tiles
  for (long long T = sc.s0; T < sc.s1; ++T) {
    int stage;
    if (!slot(stage)) return;
    const int bh = (int)(T / a.tph), j = (int)(T - (long long)bh * a.tph);
    const int u0 = j * kTile, u1 = min(ns, u0 + kTile), n = u1 - u0;
    const int b = bh / a.Hq, g = (bh - b * a.Hq) / G;
    const size_t head = (size_t)b * a.Hkv + g;
    const bool last = (j == a.tph - 1) || (T == sc.s1 - 1);
    // units: steady tiles of this head inside the block's range
    const long long first = max(sc.s0, (long long)bh * a.tph);
    post(stage, kTileSteady, bh, n, last, last ? (int)(T - first + 1) : 0,
         (uint32_t)n * 512u + kD * 2u);
    // rows: [u0, min(u1, sink)) are positions u; the rest are N - window + (u - sink)
    const int a1 = min(u1, a.sink);
    if (lane < 2 && u0 < a1) {
      const uint16_t* base = (lane == 0 ? a.K : a.V) + (head * a.N + u0) * kD;
      copy(stage, lane == 0 ? 0u : kStageBytes / 2, base, (uint32_t)(a1 - u0) * 256u);
    }
    const int b0 = max(u0, a.sink);
    if (lane >= 2 && lane < 4 && b0 < u1) {
      const int row = a.N - a.window + (b0 - a.sink);
      const uint16_t* base = (lane == 2 ? a.K : a.V) + (head * a.N + row) * kD;
      const uint32_t dst = (uint32_t)(b0 - u0) * 256u + (lane == 2 ? 0u : kStageBytes / 2);
      copy(stage, dst, base, (uint32_t)(u1 - b0) * 256u);
    }
    if (lane == 4) copy_q(stage, a.q + (size_t)bh * kD, kD * 2);
    commit();
  }

  // stage 3b: retrieved tiles, each head's once its selection is published
  if (sc.r0 < sc.r1) {
    const int r = a.r, rs = r > 0 ? r : 1;
    long long slot0 = sc.r0;
    while (slot0 < sc.r1) {
      const int bh = (int)(slot0 / r);
      const int j_lo = (int)(slot0 - (long long)bh * r);
      const int j_hi = (int)min((long long)r, sc.r1 - (long long)bh * r);
      slot0 = (long long)bh * r + j_hi;
      if (a.fused) {
        int good = 1;
        if (lane == 0) {
          good = !*(volatile int*)&S.abort && count_wait(a.sel_ready + bh, 1u, a.status, &S.abort);
          if (!good) S.abort = 1;
        }
        if (!__shfl_sync(kFull, good, 0)) return;
        __syncwarp();  // the other lanes' loads come after lane 0's acquire
      }
      const int b = bh / a.Hq, g = (bh - b * a.Hq) / G;
      const size_t head = (size_t)b * a.Hkv + g;
      const uint16_t* Ks = a.ksorted + head * (size_t)a.N_idx * kD;
      const uint16_t* Vs = a.vsorted + head * (size_t)a.N_idx * kD;
      const int* rows_g = a.sel_rows + (size_t)bh * rs;
      const int* cnts_g = a.sel_cnts + (size_t)bh * rs;
      // two windows of 32 clusters in registers: (row, count, piece-relative start)
      auto load_win = [&](int j, int& row, int& cnt) {
        row = 0;
        cnt = 0;
        if (j < j_hi) {
          row = __ldcg(rows_g + j);
          cnt = __ldcg(cnts_g + j);
          if (cnt < 0 || row < 0 || (long long)row + cnt > a.N_idx) {
            report(a.status, WI_ERR_INDEX_MISMATCH);
            cnt = 0;
            row = 0;
          }
        }
      };
      int rowA, cntA, rowB, cntB;
      load_win(j_lo + lane, rowA, cntA);
      load_win(j_lo + 32 + lane, rowB, cntB);
      // exclusive prefix of counts over a window + its total
      auto wscan = [&](int cnt, int& total) {
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += t;
        }
        total = __shfl_sync(kFull, incl, 31);
        return incl - cnt;
      };
      // window A = slots [jA, jA + 32), window B = the next 32; starts are
      // piece-relative token positions
      int jA = j_lo, totA, totB;
      int stA = wscan(cntA, totA);
      int stB = totA + wscan(cntB, totB);
      int baseA = 0, cur = 0;
      bool posted_last = false;
      for (;;) {
        const int avail = baseA + totA + totB - cur;
        const bool more = jA + 64 < j_hi;
        if (avail > 0) {
          const int n = min(kTile, avail);
          const bool last = (n == avail) && !more;
          int stage;
          if (!slot(stage)) return;
          post(stage, kTileRet, bh, n, last, last ? j_hi - j_lo : 0,
               (uint32_t)n * 512u + kD * 2u);
          const int t0 = cur, t1 = cur + n;
#pragma unroll
          for (int w2 = 0; w2 < 2; ++w2) {
            const int ca = baseA + (w2 == 0 ? stA : stB), cnt = w2 == 0 ? cntA : cntB;
            const int row = w2 == 0 ? rowA : rowB;
            const int x0 = max(t0, ca), x1 = min(t1, ca + cnt);
            if (x0 < x1) {
              const size_t srow = (size_t)row + (x0 - ca);
              const uint32_t d = (uint32_t)(x0 - t0) * 256u, nb = (uint32_t)(x1 - x0) * 256u;
              copy(stage, d, Ks + srow * kD, nb);
              copy(stage, kStageBytes / 2 + d, Vs + srow * kD, nb);
            }
          }
          if (lane == 0) copy_q(stage, a.q + (size_t)bh * kD, kD * 2);
          commit();
          cur = t1;
          if (last) {
            posted_last = true;
            break;
          }
        } else if (!more) {
          break;
        }
        // window A used up: B becomes A, the next 32 slots are loaded into B
        if (cur >= baseA + totA && jA + 32 < j_hi) {
          baseA += totA;
          rowA = rowB;
          cntA = cntB;
          stA = stB - totA;
          totA = totB;
          jA += 32;
          load_win(jA + 32 + lane, rowB, cntB);
          stB = totA + wscan(cntB, totB);
        }
      }
      if (!posted_last) {  // the piece's slots must be reported even without tokens
        int stage;
        if (!slot(stage)) return;
        post(stage, kTileRet, bh, 0, 1, j_hi - j_lo, 0u);
        commit();
      }
    }
  }
  // end marker
  int stage;
  if (!slot(stage)) return;
  post(stage, kTileEnd, 0, 0, 0, 0, 0u);
  commit();
}

// ---------------------------------------------------------------------------
// consumer tiles
// ---------------------------------------------------------------------------
// Consumers copy their share of a staged tile (rows, query rows, side data)
// into registers and release the stage at once, so that the ring refills while
// they compute.  For index tiles lane L < 4G of warp w works on row 4w + L / G
// and query head L mod G of the group.

// Centroid-key tile: warp w scores rows 4w..4w+3 for the G heads of the group.
template <int G>
struct KbarRegs {
  float4 k[4];
  uint2 q[G];
};
template <int G>
__device__ __forceinline__ void kbar_load(const DecSmem& S, int stage, int nrows, KbarRegs<G>& t,
                                          int lane, int warp) {
  const float* kb = reinterpret_cast<const float*>(S.ring[stage]);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int row = warp * 4 + j;
    t.k[j] = row < nrows ? lds4(kb + row * kD + lane * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int h = 0; h < G; ++h) t.q[h] = lds2(S.qs[stage] + h * kD * 2 + lane * 8);
}
// Lane L < 4G gets the score of row 4w + L / G for head L mod G.
template <int G>
__device__ __forceinline__ float kbar_dot(const DecodeArgs& a, const KbarRegs<G>& t, int lane) {
  float v[4 * G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float q0 = bf_lo(t.q[h].x) * a.scale, q1 = bf_hi(t.q[h].x) * a.scale;
    const float q2 = bf_lo(t.q[h].y) * a.scale, q3 = bf_hi(t.q[h].y) * a.scale;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      v[j * G + h] = t.k[j].x * q0 + t.k[j].y * q1 + t.k[j].z * q2 + t.k[j].w * q3;
  }
  return reduce_scatter<4 * G>(v, lane);
}
// This lane's row and head of an index tile (lane L < 4G).
template <int G>
__device__ __forceinline__ int lane_row(int lane, int warp) {
  return warp * 4 + (lane & (4 * G - 1)) / G;
}
template <int G>
__device__ __forceinline__ int lane_head(int lane) {
  return (lane & (4 * G - 1)) % G;
}
// n = the size of this lane's row (read from the stage before its release).
template <int G>
__device__ __forceinline__ void kbar_store(const DecodeArgs& a, float tot, const TileInfo& ti, int n,
                                           int lane, int warp) {
  const int row = lane_row<G>(lane, warp);
  if (lane < 4 * G && row < ti.ntok)
    a.scores[(size_t)(ti.h0 + lane_head<G>(lane)) * a.C + ti.c0 + row] = n > 0 ? tot : -INFINITY;
}

// Per-warp estimate state for the G heads of one KV group.
template <int G>
struct EstState {
  float m[G];      // running max (log2 units), warp-uniform
  float4 o[G];     // this lane's 4 dimensions
  float lacc;      // lane L < 4G: running sum n e^{s-m} for head L mod G
};

template <int G>
__device__ __forceinline__ void est_reset(EstState<G>& e) {
#pragma unroll
  for (int h = 0; h < G; ++h) {
    e.m[h] = -INFINITY;
    e.o[h] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  e.lacc = 0.f;
}

__device__ __forceinline__ void vsum_load(const DecSmem& S, int stage, int nrows, float4 (&v)[4],
                                          int lane, int warp) {
  const float* vs = reinterpret_cast<const float*>(S.ring[stage]);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int row = warp * 4 + j;
    v[j] = row < nrows ? lds4(vs + row * kD + lane * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Value-sum tile: warp w accumulates rows 4w..4w+3.  Lane L < 4G holds sj,
// the score of its (row, head), and n, the row's size.
template <int G>
__device__ __forceinline__ void vsum_compute(const float4 (&v)[4], int nrows, float sj, int n,
                                             EstState<G>& e, int lane, int warp) {
  const int L = lane & (4 * G - 1), hL = L % G;
  const int row = lane_row<G>(lane, warp);
  const float x = (lane < 4 * G && row < nrows && n > 0 && sj > -INFINITY) ? sj * kLog2e
                                                                            : -INFINITY;
  float mt = x;
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
  e.lacc *= corrL;
  const float p = (x > -INFINITY) ? exp2f(x - mL) : 0.f;
  e.lacc += p * (float)n;
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

// Writes the block's estimate piece of group bg (ntiles of its tiles); the
// caller publishes it.
template <int G>
__device__ void est_flush(const DecodeArgs& a, DecSmem& S, EstState<G>& e, int bg, int lane) {
  const int L = lane & (4 * G - 1);
  const int hL = L % G;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float lh = warp_sum((lane < 4 * G && hL == h) ? e.lacc : 0.f);
    float* dst = a.est_part + ((size_t)(blockIdx.x + bg) * G + h) * kPartStride;
    combine_write(S, e.m[h], lh, e.o[h], dst, 1.f);
  }
  est_reset(e);
}

// Exact-attention tile (steady or retrieved rows): warp w takes tokens
// 4w..4w+3; online softmax in log2 units.
struct AttState {
  float m, l;
  float4 o;
};
struct AttRegs {
  uint2 k[4], v[4], q;
};

__device__ __forceinline__ void att_load(const DecSmem& S, int stage, int ntok, AttRegs& t,
                                         int lane, int warp) {
  const uint16_t* kt = reinterpret_cast<const uint16_t*>(S.ring[stage]);
  const uint16_t* vt = kt + kTile * kD;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int tk = warp * 4 + i;
    t.k[i] = tk < ntok ? lds2(kt + tk * kD + lane * 4) : make_uint2(0u, 0u);
    t.v[i] = tk < ntok ? lds2(vt + tk * kD + lane * 4) : make_uint2(0u, 0u);
  }
  t.q = lds2(S.qs[stage] + lane * 8);
}

__device__ __forceinline__ void att_compute(const DecodeArgs& a, const AttRegs& t, int ntok,
                                            AttState& st, int lane, int warp) {
  if (warp * kRowsPerWarp >= ntok) return;
  const float qs = a.scale * kLog2e;
  const float q0 = bf_lo(t.q.x) * qs, q1 = bf_hi(t.q.x) * qs, q2 = bf_lo(t.q.y) * qs,
              q3 = bf_hi(t.q.y) * qs;
  float v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    v[i] = bf_lo(t.k[i].x) * q0 + bf_hi(t.k[i].x) * q1 + bf_lo(t.k[i].y) * q2 +
           bf_hi(t.k[i].y) * q3;
  const float mine = reduce_scatter<4>(v, lane);
  float lg[4];
  float mt = -INFINITY;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    lg[i] = __shfl_sync(kFull, mine, i);
    if (warp * 4 + i >= ntok) lg[i] = -INFINITY;
    mt = fmaxf(mt, lg[i]);
  }
  const float mn = fmaxf(st.m, mt);
  const float corr = (st.m > -INFINITY) ? exp2f(st.m - mn) : 0.f;
  st.l *= corr;
  st.o.x *= corr;
  st.o.y *= corr;
  st.o.z *= corr;
  st.o.w *= corr;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (warp * 4 + i < ntok) {
      const float p = exp2f(lg[i] - mn);
      st.l += p;
      st.o.x += p * bf_lo(t.v[i].x);
      st.o.y += p * bf_hi(t.v[i].x);
      st.o.z += p * bf_lo(t.v[i].y);
      st.o.w += p * bf_hi(t.v[i].y);
    }
  }
  st.m = mn;
}

// ---------------------------------------------------------------------------
// consumer warps
// ---------------------------------------------------------------------------
template <int G>
__device__ void consumers(const DecodeArgs& a, DecSmem& S, const Sched& sc) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t seq = 0;
  bool bad = false;  // uniform over the consumers
  const long long H = (long long)a.B * a.Hq;
  const unsigned grp_target = (unsigned)(a.tpg * kCW);  // (tile, warp) pairs of a group

  // wait for the next tile; collective: every consumer gets the same answer
  auto acquire = [&](int& stage) -> bool {
    stage = (int)(seq % kStages);
    int ok = 1;
    if (tid == 0) {
      ok = !*(volatile int*)&S.abort &&
           mbar_wait(smem_addr(&S.full[stage]), (seq / kStages) & 1u, a.status);
      if (ok) S.confirmed = (int)(seq + 1);
      else S.abort = 1;
    }
    bad = cany(!ok);
    return !bad;
  };
  // Queue a request to the signaling warp (thread 0; every consumer calls it
  // after the barrier that follows the writes it publishes).
  auto publish = [&](unsigned* cnt, unsigned val, int op, int bh) {
    if (tid == 0) {
      const int t = S.pub_tail;
      if (t - ld_acquire_cta(&S.pub_head) >= kPubSlots) {  // ring full: wait (bounded)
        const unsigned long long t0 = global_ns();
        while (t - ld_acquire_cta(&S.pub_head) >= kPubSlots) {
          if (*(volatile int*)&S.abort) break;
          if (global_ns() - t0 > kWaitLimitNs) {
            report(a.status, WI_ERR_DEVICE_TIMEOUT);
            S.abort = 1;
            break;
          }
          __nanosleep(64);
        }
      }
      PubReq& q = S.pub[t % kPubSlots];
      q.cnt = cnt;
      q.val = val;
      q.op = op;
      q.bh = bh;
      st_release_cta(&S.pub_tail, t + 1);
    }
  };
  // release a stage whose data this warp has copied to registers
  auto release = [&](int stage) {
    __syncwarp();
    if (lane == 31) mbar_arrive(smem_addr(&S.empty[stage]));
    ++seq;
  };
  // collective bounded wait until *cnt >= target (one launch running every
  // stage; stage-only launches find their inputs complete)
  auto wait_count = [&](const unsigned* cnt, unsigned target) -> bool {
    if (!a.fused) return !bad;
    int ok = 1;
    if (tid == 0) {
      ok = !*(volatile int*)&S.abort && count_wait(cnt, target, a.status, &S.abort);
      if (!ok) S.abort = 1;
    }
    bad = cany(!ok) || bad;
    return !bad;
  };
  // a head merges once its group's estimate pieces and its negative estimate
  // are written
  auto merge_ready = [&](int bh) -> bool {
    const int b = bh / a.Hq, g = (bh - b * a.Hq) / G;
    return wait_count(a.est_cnt + (size_t)b * a.Hkv + g, (unsigned)a.tpg) &&
           wait_count(a.neg_ready + bh, 1u);
  };
  // this lane's size (and, for value-sum tiles, score) of a staged index tile
  auto side_of = [&](int stage, int& n, float& sj) {
    const int row = lane_row<G>(lane, warp);
    n = S.sd[stage].n[row];
    sj = S.sd[stage].s[lane_head<G>(lane)][row];
  };

  // ---- stage 1 (every block): scores
  if (a.stages & kStageScore) {
    // Every warp stores its scores of tile i - 1 before the barrier of tile
    // i's acquire; thread 0 then hands the count of stored tiles to the
    // signaling warp, which publishes them on the groups' counters.
    for (int i = 0; i < sc.n1; ++i) {
      int stage;
      if (!acquire(stage)) break;
      if (tid == 0 && i > 0) st_release_cta(&S.scored, i);
      const TileInfo ti = S.info[stage];
      KbarRegs<G> t;
      kbar_load<G>(S, stage, ti.ntok, t, lane, warp);
      int n;
      float unused;
      side_of(stage, n, unused);
      release(stage);
      const float tot = kbar_dot<G>(a, t, lane);
      kbar_store<G>(a, tot, ti, n, lane, warp);
    }
    if (!bad && sc.n1 > 0) {
      csync();
      if (tid == 0) st_release_cta(&S.scored, sc.n1);
    }
  }

  // ---- stage 2: selections (selection blocks); estimate of every cluster
  // (scoring blocks)
  if ((a.stages & kStageSelect) && !bad) {
    if (sc.sel) {
      for (int bh = sc.sel0; bh < H; bh += sc.sel_step) {
        const int b = bh / a.Hq, g = (bh - b * a.Hq) / G;
        if (!wait_count(a.grp_cnt + (size_t)b * a.Hkv + g, grp_target)) break;
        const int kept = select_head<G>(a, S, bh);
        publish(a.sel_ready + bh, 1u, kPubSet, bh);
        // the estimate of the selection (kept with a negative sign)
        if (kept >= 0) estimate_kept<G>(a, S, bh, kept);
        else estimate_selected<G>(a, S, bh);
        publish(a.neg_ready + bh, 1u, kPubSet, bh);
      }
    } else if (sc.v0 < sc.v1) {
      // (the producer stages a group's tiles once all of its scores are written)
      EstState<G> e;
      est_reset(e);
      int cur_bg = sc.v0 / a.tpg, cur_n = 0, bg_end = (cur_bg + 1) * a.tpg;
      for (int T = sc.v0; T < sc.v1; ++T) {
        if (T == bg_end) {  // same tiles in every warp: a uniform barrier
          est_flush<G>(a, S, e, cur_bg, lane);
          publish(a.est_cnt + cur_bg, (unsigned)cur_n, kPubAdd, 0);
          ++cur_bg;
          cur_n = 0;
          bg_end += a.tpg;
        }
        ++cur_n;
        int stage;
        if (!acquire(stage)) break;
        float4 v[4];
        vsum_load(S, stage, S.info[stage].ntok, v, lane, warp);
        const int nrows = S.info[stage].ntok;
        int n;
        float sj;
        side_of(stage, n, sj);
        release(stage);
        vsum_compute<G>(v, nrows, sj, n, e, lane, warp);
      }
      if (!bad) {
        est_flush<G>(a, S, e, cur_bg, lane);
        publish(a.est_cnt + cur_bg, (unsigned)cur_n, kPubAdd, 0);
      }
    }
  }

  // ---- stage 3: exact attention over steady and retrieved rows, merges
  if ((a.stages & kStageAttend) && !bad) {
    AttState st = {-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
    const int per_head = a.tph + a.r;
    for (;;) {
      int stage;
      if (!acquire(stage)) break;
      const TileInfo t = S.info[stage];
      if (t.kind == kTileEnd) {
        release(stage);
        break;
      }
      AttRegs ar;
      att_load(S, stage, t.ntok, ar, lane, warp);
      release(stage);
      att_compute(a, ar, t.ntok, st, lane, warp);
      if (t.last) {
        float* dst = (t.kind == kTileSteady ? a.std_part : a.ret_part) +
                     (size_t)(blockIdx.x + t.bh) * kPartStride;
        combine_write(S, st.m, st.l, st.o, dst, 1.f);
        st.m = -INFINITY;
        st.l = 0.f;
        st.o = make_float4(0.f, 0.f, 0.f, 0.f);
        publish(a.head_cnt + t.bh, (unsigned)t.units, kPubPiece, t.bh);
      }
    }
    // heads with no steady tile and no retrieval budget: one designated block
    if (per_head == 0 && !bad) {
      for (long long bh = blockIdx.x; bh < H && !bad; bh += a.nb)
        if (merge_ready((int)bh)) merge_head<G>(a, S, (int)bh);
    }
  }
  // No more requests; wait for the signaling warp to publish the last batch.
  if (tid == 0) {
    st_release_cta(&S.cons_done, 1);
    const unsigned long long t0 = global_ns();
    while (!ld_acquire_cta(&S.sig_done)) {
      if (global_ns() - t0 > kWaitLimitNs) {
        report(a.status, WI_ERR_DEVICE_TIMEOUT);
        S.abort = 1;
        break;
      }
      __nanosleep(64);
    }
  }
  csync();
  // Merges: a block that has finished its tiles claims slots of the merge
  // queue, where the signaling warps put every head as its last piece is
  // published (completion order), and merges them; no block with tiles left
  // spends time merging.
  if ((a.stages & kStageAttend) && a.tph + a.r > 0) {
    const unsigned H = (unsigned)(a.B * a.Hq);
    for (;;) {
      if (tid == 0) {
        int bh = -1;
        const unsigned slot = *(volatile int*)&S.abort ? H : atomicAdd(a.mq_head, 1u);
        if (slot < H) {
          if (count_wait(a.mq_ready + slot, 1u, a.status, &S.abort)) bh = __ldcg(a.mq_bh + slot);
          else S.abort = 1;
        }
        S.flag = bh;
      }
      csync();
      const int bh = S.flag;
      if (bh < 0) break;
      if (merge_ready(bh)) merge_head<G>(a, S, bh);  // barriers inside: S.flag is read by then
      if (bad) break;
    }
  }
}

// ---------------------------------------------------------------------------
// signaling warp: publishes the block's results on the grid's counters -- the
// scored index tiles on the KV groups' counters and the consumers' queued
// requests -- with one gpu-scope fence per batch, off the consumers' path.
// A piece that completes its head puts the head on the launch's merge queue.
// ---------------------------------------------------------------------------
__device__ void signaler(const DecodeArgs& a, DecSmem& S, const Sched& sc) {
  const int lane = threadIdx.x & 31;
  const int n1 = (a.stages & kStageScore) ? sc.n1 : 0;
  const unsigned per_head = (unsigned)(a.tph + a.r);
  int done1 = 0, ph = 0;
  for (;;) {
    int c1 = done1, pt = ph, fin = 0;
    if (lane == 0) {
      const unsigned long long t0 = global_ns();
      for (;;) {
        fin = ld_acquire_cta(&S.cons_done);  // first: what was queued before it is seen below
        c1 = n1 > 0 ? ld_acquire_cta(&S.scored) : 0;
        pt = ld_acquire_cta(&S.pub_tail);
        if (c1 > done1 || pt > ph || fin) break;
        if (*(volatile int*)&S.abort || global_ns() - t0 > kWaitLimitNs) {
          c1 = -1;  // the consumers gave up (and reported why)
          break;
        }
        __nanosleep(64);
      }
    }
    c1 = __shfl_sync(kFull, c1, 0);
    pt = __shfl_sync(kFull, pt, 0);
    fin = __shfl_sync(kFull, fin, 0);
    if (c1 < 0) break;
    __syncwarp();
    if (c1 == done1 && pt == ph) break;  // fin: nothing more will come
    fence_gpu();  // every write the consumers made before these requests
    for (int j = done1 + lane; j < c1; j += 32)
      atomicAdd(a.grp_cnt + (sc.k0 + j * sc.kstep) / a.tpg, (unsigned)kCW);
    if (lane == 0) {
      for (int i = ph; i < pt; ++i) {
        const PubReq q = S.pub[i % kPubSlots];
        if (q.op == kPubSet) {
          atomicExch(q.cnt, q.val);
        } else {
          const unsigned old = atomicAdd(q.cnt, q.val);
          if (q.op == kPubPiece && old + q.val == per_head) {
            // the head is complete: queue it for a merging block (the fence
            // orders every block's pieces, seen through the counter, first)
            fence_gpu();
            const unsigned slot = atomicAdd(a.mq_tail, 1u);
            a.mq_bh[slot] = q.bh;
            fence_gpu();
            atomicExch(a.mq_ready + slot, 1u);
          }
        }
      }
      st_release_cta(&S.pub_head, pt);
    }
    __syncwarp();
    done1 = c1;
    ph = pt;
  }
  if (lane == 0) st_release_cta(&S.sig_done, 1);
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ DecodeArgs a) {
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
    S.confirmed = 0;
    S.flag = 0;
    S.scored = 0;
    S.pub_tail = S.pub_head = 0;
    S.cons_done = S.sig_done = 0;
  }
  __syncthreads();
  const Sched sc = schedule(a, blockIdx.x);
  if (tid >= kCT + 32) signaler(a, S, sc);
  else if (tid >= kCT) producer<G>(a, S, sc);
  else consumers<G>(a, S, sc);
  __syncthreads();
  if (tid == 0) {
    // let every copy still in flight land before the block exits
    for (int q = S.confirmed; q < S.issued; ++q)
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
      *a.mq_tail = 0u;
      *a.mq_head = 0u;
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
