// Decode kernels of the wave-index tripartite attention ("RetroInfer: A Vector
// Storage Engine for Scalable Long-Context LLM Inference", technical summary
// (es) §2.A: steady zone, retrieval zone, estimation zone; technical summary
// (ar) §2.a: estimation from centroids and the value sum, §2.b: retrieved KV
// laid out contiguously).  Three launches, chained with programmatic
// dependent launch:
//
//   score_kernel   s[b,h,c] = scale q_h . kbar_c (-inf if empty): one pass over
//                  the f32 centroid keys, one warp per 512-byte row, 128-bit
//                  loads, all query heads of a KV group per pass.
//   select_kernel  two block roles in one launch, so that the selection's
//                  latency hides under the value-sum stream:
//                  (a) per query head, radix select of the r largest scores
//                      (order: score desc, id asc): ids ascending + token prefix;
//                  (b) per chunk of clusters of one KV head, the estimate of
//                      EVERY non-empty cluster: (m, l = sum n_c e^{s_c-m},
//                      o = sum e^{s_c-m} vsum_c).
//   attend_kernel  per (query head, split of its token list): exact attention
//                  over the steady zone and the retrieved clusters, rows staged
//                  into shared memory by the TMA bulk-copy engine (cp.async.bulk
//                  + mbarrier, double buffered); the same block emits the
//                  retrieved clusters' estimates with a negative sign, so that
//                  all-minus-retrieved is the estimation zone; the last block of
//                  a head merges every partial (log-sum-exp) into out and lse.
// Softmax quantities are kept in log2 units (logits scaled by log2 e) so that
// every exponential is an exp2.
#include <float.h>
#include <limits.h>
#include <stddef.h>

#include "wi_device.cuh"
#include "wi_internal.h"

namespace wi {

namespace {

template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t st, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// --------------------------------------------------------------------------
// K1: centroid scoring
// --------------------------------------------------------------------------
constexpr int kScoreThreads = 256;
constexpr int kScoreWarps = kScoreThreads / 32;

template <int G>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(DecodeArgs a, int rows_per_block,
                                                              int blocks_per_head) {
  grid_dep_launch();
  grid_dep_wait();
  constexpr int ROWS = 32 / G;  // rows per transpose-reduce batch
  constexpr int NB = ROWS >= 16 ? 1 : 2;  // batches in flight: 8-32 rows per warp
  const int bg = blockIdx.x / blocks_per_head;
  const int chunk = blockIdx.x - bg * blocks_per_head;
  const int b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  float4 qv[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint2 w =
        reinterpret_cast<const uint2*>(a.q + ((size_t)b * a.Hq + g * G + h) * kD)[lane];
    qv[h] = make_float4(bf_lo(w.x) * a.scale, bf_hi(w.x) * a.scale, bf_lo(w.y) * a.scale,
                        bf_hi(w.y) * a.scale);
  }
  const float4* kb = reinterpret_cast<const float4*>(a.kbar + (size_t)bg * a.C * kD);
  const int* sz = a.size + (size_t)bg * a.C;
  const int c_begin = chunk * rows_per_block;
  const int c_end = min(a.C, c_begin + rows_per_block);
  for (int c0 = c_begin + warp * NB * ROWS; c0 < c_end; c0 += kScoreWarps * NB * ROWS) {
    float4 kv[NB * ROWS];
#pragma unroll
    for (int r = 0; r < NB * ROWS; ++r) {
      const int c = c0 + r;
      kv[r] = (c < c_end) ? __ldg(kb + (size_t)c * (kD / 4) + lane)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      float v[32];
#pragma unroll
      for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 k4 = kv[nb * ROWS + r];
          v[r * G + h] = k4.x * qv[h].x + k4.y * qv[h].y + k4.z * qv[h].z + k4.w * qv[h].w;
        }
      const float tot = warp_transpose_sum32(v, lane);
      const int r = lane / G, h = lane - (lane / G) * G;
      const int c = c0 + nb * ROWS + r;
      if (c < c_end) {
        const int n = __ldg(sz + c);
        a.scores[((size_t)b * a.Hq + g * G + h) * a.C + c] = n > 0 ? tot : -INFINITY;
      }
    }
  }
}

// --------------------------------------------------------------------------
// K2: selection (role a) and estimation over all clusters (role b)
// --------------------------------------------------------------------------
constexpr int kK2Threads = 512;
constexpr int kK2Warps = kK2Threads / 32;
constexpr int kSelCacheMax = 16384;              // keys kept in shared memory up to this C
constexpr int kEstBatch = kEstChunk / kK2Warps;  // clusters per warp: 16
static_assert(kEstBatch == 16, "estimation batch layout");

__device__ __forceinline__ uint32_t score_key(float s) {
  return (s == -INFINITY) ? 0u : float_key(s);  // 0 <=> empty cluster
}

// Exclusive scan of an int pair over the block; returns the prefix and the
// block total in *total.  sh must hold 33 entries.
__device__ __forceinline__ int2 block_scan2(int2 v, int2* sh, int2* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
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
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int2 w = lane < nwarps ? sh[lane] : make_int2(0, 0);
    int2 wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(kFull, wi.x, o);
      const int y = __shfl_up_sync(kFull, wi.y, o);
      if (lane >= o) {
        wi.x += x;
        wi.y += y;
      }
    }
    sh[lane] = make_int2(wi.x - w.x, wi.y - w.y);
    if (lane == 31) sh[32] = wi;
  }
  __syncthreads();
  const int2 base = sh[warp];
  *total = sh[32];
  const int2 res = make_int2(base.x + incl.x - v.x, base.y + incl.y - v.y);
  __syncthreads();  // sh may be reused by the caller
  return res;
}

struct SelShared {
  int hist[256];
  int2 scan[33];
  int i[8];
  uint32_t u[32];
};

// Role (a): the r_eff = min(r, non-empty) largest scores of one query head.
// Radix select on order-preserving keys, 8 bits per pass, histograms built
// with warp-aggregated shared atomics; stops as soon as the boundary bin is
// taken whole.  Equal keys at the boundary keep the lowest ids.
__device__ void select_head(const DecodeArgs& a, int bh, uint32_t* skey, SelShared& S,
                            int cached) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = bh / a.Hq, h = bh - b * a.Hq, g = h / a.G;
  const int C = a.C;
  const float* sc = a.scores + (size_t)bh * C;
  const int* sz = a.size + ((size_t)b * a.Hkv + g) * C;
  auto key = [&](int c) -> uint32_t { return cached ? skey[c] : score_key(__ldcg(sc + c)); };

  int valid = 0;
  uint32_t kmax = 0;
  for (int c = tid; c < C; c += kK2Threads) {
    const uint32_t k = score_key(__ldcg(sc + c));
    if (cached) skey[c] = k;
    valid += (k != 0);
    kmax = max(kmax, k);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    valid += __shfl_xor_sync(kFull, valid, o);
    kmax = max(kmax, __shfl_xor_sync(kFull, kmax, o));
  }
  if (lane == 0) {
    S.scan[warp].x = valid;
    S.u[warp] = kmax;
  }
  __syncthreads();
  if (warp == 0) {
    int v = lane < kK2Warps ? S.scan[lane].x : 0;
    uint32_t m = lane < kK2Warps ? S.u[lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      v += __shfl_xor_sync(kFull, v, o);
      m = max(m, __shfl_xor_sync(kFull, m, o));
    }
    if (lane == 0) {
      S.i[0] = v;
      S.i[5] = (int)m;
    }
  }
  __syncthreads();
  valid = S.i[0];
  kmax = (uint32_t)S.i[5];
  const int r = a.r;
  const int r_eff = min(r, valid);
  if (tid == 0) a.head_max[bh] = valid > 0 ? key_float(kmax) : -INFINITY;

  uint32_t prefix = 0, mask = 0;
  int remaining = r_eff, count = 0;
  if (r_eff > 0) {
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (tid < 256) S.hist[tid] = 0;
      __syncthreads();
      for (int base = 0; base < C; base += kK2Threads) {
        const int c = base + tid;
        const uint32_t k = c < C ? key(c) : 0u;
        const bool in = k != 0u && (k & mask) == prefix;
        const int d = in ? (int)((k >> shift) & 0xffu) : 256 + lane;
        const unsigned peers = __match_any_sync(kFull, d);
        if (in && lane == __ffs(peers) - 1) atomicAdd(&S.hist[d], __popc(peers));
      }
      __syncthreads();
      if (warp == 0) {
        int cnt[8];
        int tot = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          cnt[j] = S.hist[255 - 8 * lane - j];
          tot += cnt[j];
        }
        int incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += t;
        }
        const int excl = incl - tot;
        if (excl < remaining && remaining <= incl) {
          int acc = excl;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (acc + cnt[j] >= remaining) {
              S.i[1] = 255 - 8 * lane - j;
              S.i[2] = acc;
              S.i[3] = cnt[j];
              break;
            }
            acc += cnt[j];
          }
        }
      }
      __syncthreads();
      remaining -= S.i[2];
      count = S.i[3];
      prefix |= (uint32_t)S.i[1] << shift;
      mask |= 0xffu << shift;
      if (count == remaining) break;  // the whole boundary bin is selected
    }
  }
  const bool any = r_eff > 0;
  const bool tie_cut = any && remaining < count;  // equal full keys at the boundary
  int c_cut = INT_MAX;
  const int per = (C + kK2Threads - 1) / kK2Threads;
  const int my0 = min(C, tid * per), my1 = min(C, my0 + per);
  if (tie_cut) {
    int ne = 0;
    for (int c = my0; c < my1; ++c) ne += (key(c) == prefix);
    int2 tot;
    const int before = block_scan2(make_int2(ne, 0), S.scan, &tot).x;
    if (before < remaining && remaining <= before + ne) {
      int cnt = before;
      for (int c = my0; c < my1; ++c) {
        if (key(c) == prefix && ++cnt == remaining) {
          S.i[4] = c;
          break;
        }
      }
    }
    __syncthreads();
    c_cut = S.i[4];
  }
  auto is_sel = [&](uint32_t k, int c) {
    return any && k != 0u &&
           ((k & mask) > prefix || ((k & mask) == prefix && (!tie_cut || c <= c_cut)));
  };
  // ordered compaction: ids ascending, exclusive prefix of member counts
  int nsel = 0, ntok = 0;
  for (int c = my0; c < my1; ++c) {
    if (is_sel(key(c), c)) {
      ++nsel;
      ntok += __ldg(sz + c);
    }
  }
  int2 total;
  const int2 ex = block_scan2(make_int2(nsel, ntok), S.scan, &total);
  int* ids = a.sel_ids + (size_t)bh * r;
  int* pre = a.sel_prefix + (size_t)bh * (r + 1);
  int* topk = a.topk_out ? a.topk_out + (size_t)bh * r : nullptr;
  int pos = ex.x, tok = ex.y;
  for (int c = my0; c < my1; ++c) {
    if (is_sel(key(c), c)) {
      ids[pos] = c;
      pre[pos] = tok;
      if (topk) topk[pos] = c;
      ++pos;
      tok += __ldg(sz + c);
    }
  }
  for (int i = total.x + tid; i <= r; i += kK2Threads) {
    pre[i] = total.y;
    if (i < r) {
      ids[i] = -1;
      if (topk) topk[i] = -1;
    }
  }
}

// Role (b): estimate of every non-empty cluster of a 256-cluster chunk of one
// KV head, for each of its G query heads.  Warp w takes 16 consecutive
// clusters: lane i < 16 computes e^{s - m_warp} for cluster i (m_warp = the
// warp's max score), then the 16 value-sum rows are streamed with 128-bit
// loads and accumulated with the broadcast weights.
template <int G>
__device__ void estimate_all(const DecodeArgs& a, int bg, int chunk, float* red) {
  float(*red_o)[G][kD] = reinterpret_cast<float(*)[G][kD]>(red);
  float* red_m = red + kK2Warps * G * kD;
  float* red_l = red_m + kK2Warps * G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int c_end = min(a.C, (chunk + 1) * kEstChunk);
  const int base = chunk * kEstChunk + warp * kEstBatch;
  const int c = base + (lane & 15);
  const bool valid = c < c_end;
  const int n = valid ? __ldg(a.size + (size_t)bg * a.C + c) : 0;
  float p[G], mw[G], lw[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const size_t bh = (size_t)b * a.Hq + g * G + h;
    const float s = (n > 0) ? __ldcg(a.scores + bh * a.C + c) * kLog2e : -INFINITY;
    float m = s;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    mw[h] = m;
    p[h] = (s > -INFINITY) ? exp2f(s - m) : 0.f;
    lw[h] = lane < 16 ? p[h] * (float)n : 0.f;
  }
  const float4* vs = reinterpret_cast<const float4*>(a.vsum + ((size_t)bg * a.C) * kD);
  float4 v[kEstBatch];
#pragma unroll
  for (int j = 0; j < kEstBatch; ++j)
    v[j] = (base + j < c_end) ? __ldg(vs + (size_t)(base + j) * (kD / 4) + lane)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll
    for (int j = 0; j < kEstBatch; ++j) {
      const float pj = __shfl_sync(kFull, p[h], j);
      acc0 += pj * v[j].x;
      acc1 += pj * v[j].y;
      acc2 += pj * v[j].z;
      acc3 += pj * v[j].w;
    }
    lw[h] = warp_sum(lw[h]);
    reinterpret_cast<float4*>(red_o[warp][h])[lane] = make_float4(acc0, acc1, acc2, acc3);
    if (lane == 0) {
      red_m[warp * G + h] = mw[h];
      red_l[warp * G + h] = lw[h];
    }
  }
  __syncthreads();
  for (int idx = tid; idx < G * kD; idx += kK2Threads) {
    const int h = idx / kD, dim = idx - h * kD;
    float M = -INFINITY;
    for (int w = 0; w < kK2Warps; ++w) M = fmaxf(M, red_m[w * G + h]);
    float L = 0.f, O = 0.f;
    if (M > -INFINITY) {
      for (int w = 0; w < kK2Warps; ++w) {
        const float mwh = red_m[w * G + h];
        const float f = mwh > -INFINITY ? exp2f(mwh - M) : 0.f;
        L += red_l[w * G + h] * f;
        O += red_o[w][h][dim] * f;
      }
    }
    const size_t bh = (size_t)b * a.Hq + g * G + h;
    float* P = a.est_part + (bh * a.est_chunks + chunk) * kPartStride;
    if (dim == 0) {
      P[0] = (L > 0.f) ? M : -INFINITY;
      P[1] = L;
    }
    P[2 + dim] = O;
  }
}

template <int G>
__global__ void __launch_bounds__(kK2Threads) select_kernel(DecodeArgs a, int n_sel, int cached) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ SelShared S;
  grid_dep_launch();
  grid_dep_wait();
  if ((int)blockIdx.x < n_sel) {
    select_head(a, blockIdx.x, reinterpret_cast<uint32_t*>(smem), S, cached);
  } else {
    const int idx = blockIdx.x - n_sel;
    const int bg = idx / a.est_chunks;
    estimate_all<G>(a, bg, idx - bg * a.est_chunks, reinterpret_cast<float*>(smem));
  }
}

// --------------------------------------------------------------------------
// K3: exact attention + retrieved-estimate subtraction + merge
// --------------------------------------------------------------------------
constexpr int kAttThreads = 256;
constexpr int kAttWarps = kAttThreads / 32;
constexpr int kTile = 64;      // tokens per pipeline stage (8 per warp)
constexpr int kStages = 2;
constexpr int kWinCap = 512;   // retrieved clusters staged per window

struct __align__(128) AttSmem {
  uint16_t k[kStages][kTile * kD];  // bulk-copy destinations: 16-byte aligned
  uint16_t v[kStages][kTile * kD];
  float red_o[2][kAttWarps][kD];    // written as float4: 16-byte aligned
  float red_m[2][kAttWarps];
  float red_l[2][kAttWarps];
  unsigned long long bar[kStages];  // mbarriers: 8-byte aligned
  int win_prefix[kWinCap + 1];
  int win_row[kWinCap];
  int win_cid[kWinCap];
  int last;
};
static_assert(offsetof(AttSmem, v) % 128 == 0, "staging buffer alignment");
static_assert(offsetof(AttSmem, red_o) % 16 == 0, "float4 reduction buffer alignment");
static_assert(offsetof(AttSmem, bar) % 8 == 0, "mbarrier alignment");
// the merge reuses the staging buffers (K and V, all stages) for per-partial weights
constexpr int kMergeMaxPartials = (int)(2 * sizeof(uint16_t) * kStages * kTile * kD / sizeof(float));

__device__ void combine_warps(AttSmem& S, int slot, float m_run, float l_run, float o0, float o1,
                              float o2, float o3, float sign, float* P, bool ok) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (lane == 0) {
    S.red_m[slot][warp] = m_run;
    S.red_l[slot][warp] = l_run;
  }
  reinterpret_cast<float4*>(S.red_o[slot][warp])[lane] = make_float4(o0, o1, o2, o3);
  __syncthreads();
  if (tid < kD) {
    float M = -INFINITY;
    for (int w = 0; w < kAttWarps; ++w) M = fmaxf(M, S.red_m[slot][w]);
    float L = 0.f, O = 0.f;
    if (ok && M > -INFINITY) {
      for (int w = 0; w < kAttWarps; ++w) {
        const float mw = S.red_m[slot][w];
        const float f = mw > -INFINITY ? exp2f(mw - M) : 0.f;
        L += S.red_l[slot][w] * f;
        O += S.red_o[slot][w][tid] * f;
      }
    } else {
      M = -INFINITY;
    }
    if (tid == 0) {
      P[0] = M;
      P[1] = sign * L;
    }
    P[2 + tid] = sign * O;
  }
}

__device__ void attend_tokens(const DecodeArgs& a, int bh, int sp, AttSmem& S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = bh / a.Hq, h = bh - b * a.Hq, g = h / a.G;
  const size_t head = (size_t)b * a.Hkv + g;
  const uint16_t* Kh = a.K + head * (size_t)a.N * kD;
  const uint16_t* Vh = a.V + head * (size_t)a.N * kD;
  const uint16_t* Ksh = a.ksorted + head * (size_t)a.N_idx * kD;
  const uint16_t* Vsh = a.vsorted + head * (size_t)a.N_idx * kD;
  const float4* vsum = reinterpret_cast<const float4*>(a.vsum + head * (size_t)a.C * kD);
  const float* sc = a.scores + (size_t)bh * a.C;
  const int* off = a.offset + head * (size_t)(a.C + 1);
  const int* ids = a.sel_ids + (size_t)bh * a.r;
  const int* pre = a.sel_prefix + (size_t)bh * (a.r + 1);
  const int ns = a.sink + a.window;
  const int T_h = ns + pre[a.r];
  const int lo = (int)((long long)T_h * sp / a.att_splits);
  const int hi = (int)((long long)T_h * (sp + 1) / a.att_splits);

  const float qs = a.scale * kLog2e;
  const uint2 qw = reinterpret_cast<const uint2*>(a.q + (size_t)bh * kD)[lane];
  const float q0 = bf_lo(qw.x) * qs, q1 = bf_hi(qw.x) * qs;
  const float q2 = bf_lo(qw.y) * qs, q3 = bf_hi(qw.y) * qs;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_addr(&S.bar[s]), 1);
    fence_mbar_init();
  }
  __syncthreads();

  float m_run = -INFINITY, l_run = 0.f, o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
  // estimates of the retrieved clusters whose first token lies in this block
  float m_neg = -INFINITY, l_neg = 0.f, n0 = 0.f, n1 = 0.f, n2 = 0.f, n3 = 0.f;
  uint32_t phase = 0;
  bool ok = true;
  int round_lo = lo;
  while (ok && round_lo < hi) {
    int round_hi = hi;
    int n_cl = 0;
    if (hi > ns) {
      // window of retrieved clusters overlapping [round_lo, hi)
      const int lo_u = max(round_lo - ns, 0), hi_u = hi - ns;
      int cnt_le = 0, cnt_lt = 0;
      for (int base = 0; base < a.r; base += kAttThreads) {
        const int j = base + tid;
        const int p = (j < a.r) ? pre[j] : INT_MAX;
        cnt_le += __syncthreads_count(p <= lo_u);
        cnt_lt += __syncthreads_count(p < hi_u);
      }
      const int i0 = cnt_le - 1;
      n_cl = cnt_lt - i0;
      if (n_cl > kWinCap) {
        n_cl = kWinCap;
        round_hi = ns + pre[i0 + kWinCap];
      }
      for (int j = tid; j <= n_cl; j += kAttThreads) S.win_prefix[j] = pre[i0 + j];
      for (int j = tid; j < n_cl; j += kAttThreads) {
        const int c = ids[i0 + j];
        S.win_cid[j] = c;
        S.win_row[j] = off[c];
      }
      __syncthreads();
    }
    const int ntiles = (round_hi - round_lo + kTile - 1) / kTile;
    int ci = 0;  // producer's cursor into the window
    auto issue = [&](int t, int stage) {
      const int t0 = round_lo + t * kTile;
      const int t1 = min(t0 + kTile, round_hi);
      const uint32_t bar = smem_addr(&S.bar[stage]);
      mbar_arrive_expect_tx(bar, (uint32_t)(t1 - t0) * (2u * kD * 2u));
      const uint32_t dk = smem_addr(S.k[stage]), dv = smem_addr(S.v[stage]);
      uint32_t drow = 0;
      for (int tt = t0; tt < t1;) {
        const uint16_t *ks, *vs;
        int cnt;
        if (tt < a.sink) {
          cnt = min(t1, a.sink) - tt;
          ks = Kh + (size_t)tt * kD;
          vs = Vh + (size_t)tt * kD;
        } else if (tt < ns) {
          const int row = a.N - a.window + (tt - a.sink);
          cnt = min(t1, ns) - tt;
          ks = Kh + (size_t)row * kD;
          vs = Vh + (size_t)row * kD;
        } else {
          const int u = tt - ns;
          while (S.win_prefix[ci + 1] <= u) ++ci;
          const int row = S.win_row[ci] + (u - S.win_prefix[ci]);
          cnt = min(t1 - tt, S.win_prefix[ci + 1] - u);
          if (row < 0 || row + cnt > a.N_idx) {
            // inconsistent index (offset/size beyond the sorted arrays): report
            // it and stage steady row 0 instead, keeping the byte count
            report(a.status, WI_ERR_INDEX_MISMATCH);
            for (int e = 0; e < cnt; ++e) {
              bulk_g2s(dk + (drow + e) * (kD * 2), Kh, kD * 2, bar);
              bulk_g2s(dv + (drow + e) * (kD * 2), Vh, kD * 2, bar);
            }
            tt += cnt;
            drow += cnt;
            continue;
          }
          ks = Ksh + (size_t)row * kD;
          vs = Vsh + (size_t)row * kD;
        }
        bulk_g2s(dk + drow * (kD * 2), ks, (uint32_t)cnt * (kD * 2), bar);
        bulk_g2s(dv + drow * (kD * 2), vs, (uint32_t)cnt * (kD * 2), bar);
        tt += cnt;
        drow += cnt;
      }
    };
    const bool skip_first = a.inject != 0 && blockIdx.x == 0 && round_lo == lo;
    if (tid == 0)
      for (int t = 0; t < min(kStages, ntiles); ++t)
        if (!(skip_first && t == 0)) issue(t, t);

    // while the first copies are in flight: the estimates to subtract, one
    // warp per cluster (clusters that start inside this round)
    for (int j = warp; j < n_cl; j += kAttWarps) {
      const int start = ns + S.win_prefix[j];
      if (start < round_lo || start >= round_hi) continue;
      const int c = S.win_cid[j];
      const float s = __ldcg(sc + c) * kLog2e;
      const float n = (float)(S.win_prefix[j + 1] - S.win_prefix[j]);
      const float4 vv = __ldg(vsum + (size_t)c * (kD / 4) + lane);
      const float m_new = fmaxf(m_neg, s);
      const float corr = exp2f(m_neg - m_new);
      const float p = exp2f(s - m_new);
      l_neg = l_neg * corr + p * n;
      n0 = n0 * corr + p * vv.x;
      n1 = n1 * corr + p * vv.y;
      n2 = n2 * corr + p * vv.z;
      n3 = n3 * corr + p * vv.w;
      m_neg = m_new;
    }

    for (int t = 0; t < ntiles; ++t) {
      const int stage = t % kStages;
      const int ntok = min(kTile, round_hi - (round_lo + t * kTile));
      const bool waited = mbar_wait(smem_addr(&S.bar[stage]), (phase >> stage) & 1u, a.status);
      phase ^= 1u << stage;
      if (!__syncthreads_and(waited)) {
        // give up: first let the copies already issued for later tiles land
        for (int u = t + 1; u < min(ntiles, t + kStages); ++u) {
          const int s2 = u % kStages;
          mbar_wait(smem_addr(&S.bar[s2]), (phase >> s2) & 1u, a.status);
          phase ^= 1u << s2;
        }
        ok = false;
        break;
      }
      const uint2* kt = reinterpret_cast<const uint2*>(S.k[stage]);
      const uint2* vt = reinterpret_cast<const uint2*>(S.v[stage]);
      constexpr int U = kTile / kAttWarps;  // tokens per warp per tile
      float lg[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint2 kw = kt[(warp * U + u) * (kD / 4) + lane];
        lg[u] = bf_lo(kw.x) * q0 + bf_hi(kw.x) * q1 + bf_lo(kw.y) * q2 + bf_hi(kw.y) * q3;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int u = 0; u < U; ++u) lg[u] += __shfl_xor_sync(kFull, lg[u], o);
      float mt = -INFINITY;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (warp * U + u >= ntok) lg[u] = -INFINITY;
        mt = fmaxf(mt, lg[u]);
      }
      if (mt > -INFINITY) {
        const float m_new = fmaxf(m_run, mt);
        const float corr = exp2f(m_run - m_new);
        l_run *= corr;
        o0 *= corr;
        o1 *= corr;
        o2 *= corr;
        o3 *= corr;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (warp * U + u < ntok) {
            const float p = exp2f(lg[u] - m_new);
            const uint2 vw = vt[(warp * U + u) * (kD / 4) + lane];
            l_run += p;
            o0 += p * bf_lo(vw.x);
            o1 += p * bf_hi(vw.x);
            o2 += p * bf_lo(vw.y);
            o3 += p * bf_hi(vw.y);
          }
        }
        m_run = m_new;
      }
      __syncthreads();
      if (tid == 0 && t + kStages < ntiles) {
        fence_proxy_async_smem();
        issue(t + kStages, stage);
      }
    }
    round_lo = round_hi;
    __syncthreads();
  }
  float* P = a.att_part + ((size_t)bh * a.att_splits + sp) * 2 * kPartStride;
  combine_warps(S, 0, m_run, l_run, o0, o1, o2, o3, 1.f, P, ok);
  combine_warps(S, 1, m_neg, l_neg, n0, n1, n2, n3, -1.f, P + kPartStride, ok);
}

// Log-sum-exp merge of every partial of one query head: exact (+), retrieved
// estimates (-) and estimation chunks (+).
__device__ void merge_head(const DecodeArgs& a, int bh, AttSmem& S) {
  const int tid = threadIdx.x;
  float* w = reinterpret_cast<float*>(S.k);  // per-partial weight (reuses staging)
  __shared__ float sh_red[kAttWarps];
  const int n_att = 2 * a.att_splits;
  const int P = n_att + a.est_chunks;
  const float* PA = a.att_part + (size_t)bh * n_att * kPartStride;
  const float* PE = a.est_part + (size_t)bh * a.est_chunks * kPartStride;
  auto part = [&](int i) {
    return i < n_att ? PA + (size_t)i * kPartStride : PE + (size_t)(i - n_att) * kPartStride;
  };
  float M = -INFINITY;
  for (int i = tid; i < P; i += kAttThreads) {
    const float m = __ldcg(part(i));
    w[i] = m;
    M = fmaxf(M, m);
  }
  M = warp_max(M);
  if ((tid & 31) == 0) sh_red[tid >> 5] = M;
  __syncthreads();
  M = -INFINITY;
  for (int i = 0; i < kAttWarps; ++i) M = fmaxf(M, sh_red[i]);
  __syncthreads();
  float L = 0.f;
  for (int i = tid; i < P; i += kAttThreads) {
    const float m = w[i];
    const float f = (M > -INFINITY && m > -INFINITY) ? exp2f(m - M) : 0.f;
    w[i] = f;
    L += f * __ldcg(part(i) + 1);
  }
  L = warp_sum(L);
  if ((tid & 31) == 0) sh_red[tid >> 5] = L;
  __syncthreads();
  L = 0.f;
  for (int i = 0; i < kAttWarps; ++i) L += sh_red[i];
  // two threads per output dimension, each over half of the partials
  const int dim = tid & (kD - 1), half = tid >> 7;
  float O = 0.f;
#pragma unroll 4
  for (int i = half; i < P; i += 2) O += w[i] * __ldcg(part(i) + 2 + dim);
  float* red = reinterpret_cast<float*>(S.red_o);
  __syncthreads();
  if (half == 1) red[dim] = O;
  __syncthreads();
  if (half == 0) {
    O += red[dim];
    a.out[(size_t)bh * kD + dim] = (L > 0.f) ? O / L : 0.f;
    if (a.lse != nullptr && dim == 0) a.lse[bh] = (L > 0.f) ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
}

__global__ void __launch_bounds__(kAttThreads) attend_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  AttSmem& S = *reinterpret_cast<AttSmem*>(smem);
  grid_dep_launch();
  grid_dep_wait();
  const int bh = blockIdx.x / a.att_splits;
  const int sp = blockIdx.x - bh * a.att_splits;
  attend_tokens(a, bh, sp, S);
  // the last block of this head to finish merges all of its partials
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) S.last = (atomicAdd(&a.counters[bh], 1) == a.att_splits - 1);
  __syncthreads();
  if (S.last) {
    __threadfence();
    merge_head(a, bh, S);
    if (threadIdx.x == 0) a.counters[bh] = 0;  // ready for the next call
  }
}

template <typename F>
cudaError_t set_smem(F* f, size_t bytes) {
  return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

// --------------------------------------------------------------------------
// launchers
// --------------------------------------------------------------------------
cudaError_t launch_decode_score(const DecodeArgs& a, cudaStream_t st) {
  const int rows = 32 / a.G;
  const int rows_per_sweep = kScoreWarps * (rows >= 16 ? rows : 2 * rows);
  const long long target_blocks = 148LL * 4;
  const long long rows_total = (long long)a.C * a.B * a.Hkv;
  long long rpb = (rows_total + target_blocks - 1) / target_blocks;
  rpb = ((rpb + rows_per_sweep - 1) / rows_per_sweep) * rows_per_sweep;
  const int rows_per_block = (int)rpb;
  const int blocks_per_head = (a.C + rows_per_block - 1) / rows_per_block;
  const dim3 grid((unsigned)(blocks_per_head * a.B * a.Hkv));
  switch (a.G) {
    case 1: return launch_ex(score_kernel<1>, grid, dim3(kScoreThreads), 0, st, false, a, rows_per_block, blocks_per_head);
    case 2: return launch_ex(score_kernel<2>, grid, dim3(kScoreThreads), 0, st, false, a, rows_per_block, blocks_per_head);
    case 4: return launch_ex(score_kernel<4>, grid, dim3(kScoreThreads), 0, st, false, a, rows_per_block, blocks_per_head);
    case 8: return launch_ex(score_kernel<8>, grid, dim3(kScoreThreads), 0, st, false, a, rows_per_block, blocks_per_head);
    default: return cudaErrorInvalidValue;
  }
}

template <int G>
static cudaError_t launch_select_g(const DecodeArgs& a, cudaStream_t st) {
  const int cached = a.C <= kSelCacheMax ? 1 : 0;
  const size_t sel_smem = cached ? (size_t)a.C * sizeof(uint32_t) : 0;
  const size_t est_smem = sizeof(float) * (size_t)kK2Warps * G * (kD + 2);
  const size_t smem = sel_smem > est_smem ? sel_smem : est_smem;
  static bool attr_set = false;
  if (!attr_set) {
    const size_t mx = (size_t)kSelCacheMax * sizeof(uint32_t) > est_smem
                          ? (size_t)kSelCacheMax * sizeof(uint32_t)
                          : est_smem;
    cudaError_t e = set_smem(select_kernel<G>, mx);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int n_sel = a.B * a.Hq;
  const int n_est = a.B * a.Hkv * a.est_chunks;
  return launch_ex(select_kernel<G>, dim3((unsigned)(n_sel + n_est)), dim3(kK2Threads), smem, st,
                   true, a, n_sel, cached);
}

cudaError_t launch_decode_select(const DecodeArgs& a, cudaStream_t st) {
  switch (a.G) {
    case 1: return launch_select_g<1>(a, st);
    case 2: return launch_select_g<2>(a, st);
    case 4: return launch_select_g<4>(a, st);
    case 8: return launch_select_g<8>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_attend(const DecodeArgs& a, cudaStream_t st) {
  if (a.est_chunks + 2 * a.att_splits > kMergeMaxPartials) return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = set_smem(attend_kernel, sizeof(AttSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(attend_kernel, dim3((unsigned)(a.B * a.Hq * a.att_splits)), dim3(kAttThreads),
                   sizeof(AttSmem), st, true, a);
}

}  // namespace wi
