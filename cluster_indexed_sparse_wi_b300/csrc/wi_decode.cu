// Decode kernels of the wave-index tripartite attention ("RetroInfer: A Vector
// Storage Engine for Scalable Long-Context LLM Inference", technical summary
// §2.A: steady zone, retrieval zone, estimation zone; (ar) §2.a: estimation
// from centroids and the value sum; (ar) §2.b: contiguous retrieved KV).
//
//   score_kernel   : s[b,h,c] = scale q_h . kbar_c (-inf if empty); one pass
//                    over the f32 centroid keys, one warp per 512-byte row,
//                    128-bit loads, all query heads of a KV group per pass.
//   select_kernel  : per query head, radix select of the r largest scores
//                    (composite order: score desc, id asc), selected ids in
//                    ascending order, their token prefix and a bit mask.
//   attend_kernel  : one launch, two block roles.
//                    (a) exact attention over the steady zone and the
//                        retrieved clusters: token-balanced splits, rows
//                        staged into shared memory by the TMA bulk-copy engine
//                        (cp.async.bulk + mbarrier, double buffered), warp
//                        shuffle dot products, online softmax -> (m, l, o).
//                    (b) estimation zone over cluster chunks of one KV head:
//                        every non-retrieved non-empty cluster adds
//                        n_c e^{s_c - m} to l and e^{s_c - m} vsum_c to o.
//   merge_kernel   : log-sum-exp merge of all partials -> out, lse.
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

template <int G>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(DecodeArgs a, int rows_per_block,
                                                              int blocks_per_head) {
  grid_dep_launch();
  grid_dep_wait();
  constexpr int ROWS = 32 / G;
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
  constexpr int kWarps = kScoreThreads / 32;
  for (int c0 = c_begin + warp * ROWS; c0 < c_end; c0 += kWarps * ROWS) {
    float4 kv[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      const int c = c0 + r;
      kv[r] = (c < c_end) ? __ldg(kb + (size_t)c * (kD / 4) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float v[32];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
      for (int h = 0; h < G; ++h)
        v[r * G + h] = kv[r].x * qv[h].x + kv[r].y * qv[h].y + kv[r].z * qv[h].z + kv[r].w * qv[h].w;
    const float tot = warp_transpose_sum32(v, lane);
    const int r = lane / G, h = lane - (lane / G) * G;
    const int c = c0 + r;
    if (c < c_end) {
      const int n = __ldg(sz + c);
      a.scores[((size_t)b * a.Hq + g * G + h) * a.C + c] = n > 0 ? tot : -INFINITY;
    }
  }
}

// --------------------------------------------------------------------------
// K2: per-head top-r radix select
// --------------------------------------------------------------------------
constexpr int kSelThreads = 1024;
constexpr int kSelCacheMax = 32768;  // keys kept in shared memory up to this C

__device__ __forceinline__ uint32_t score_key(float s) {
  return (s == -INFINITY) ? 0u : float_key(s);  // 0 <=> empty cluster
}

// Exclusive scan of an int pair over the block; returns the prefix, and the
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

__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(DecodeArgs a, int cached) {
  extern __shared__ __align__(16) uint32_t skey[];
  __shared__ int hist[256];
  __shared__ int2 sh_scan[33];
  __shared__ int sh_i[8];
  __shared__ uint32_t sh_u[32];
  grid_dep_launch();
  grid_dep_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bh = blockIdx.x, b = bh / a.Hq, h = bh - b * a.Hq, g = h / a.G;
  const int C = a.C;
  const float* sc = a.scores + (size_t)bh * C;
  const int* sz = a.size + ((size_t)b * a.Hkv + g) * C;
  auto key = [&](int c) -> uint32_t { return cached ? skey[c] : score_key(sc[c]); };

  // pass 0: keys, number of non-empty clusters, maximum
  int valid = 0;
  uint32_t kmax = 0;
  for (int c = tid; c < C; c += kSelThreads) {
    const uint32_t k = score_key(sc[c]);
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
    sh_scan[warp].x = valid;
    sh_u[warp] = kmax;
  }
  __syncthreads();
  if (warp == 0) {
    int v = sh_scan[lane].x;
    uint32_t m = sh_u[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      v += __shfl_xor_sync(kFull, v, o);
      m = max(m, __shfl_xor_sync(kFull, m, o));
    }
    if (lane == 0) {
      sh_i[0] = v;
      sh_i[5] = (int)m;
    }
  }
  __syncthreads();
  valid = sh_i[0];
  kmax = (uint32_t)sh_i[5];
  const int r = a.r;
  const int r_eff = min(r, valid);
  if (tid == 0) a.head_max[bh] = valid > 0 ? key_float(kmax) : -INFINITY;

  // radix select of the r_eff-th largest key, 8 bits per pass
  uint32_t prefix = 0, mask = 0;
  int remaining = r_eff, count_eq = 0;
  if (r_eff > 0) {
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (tid < 256) hist[tid] = 0;
      __syncthreads();
      for (int c = tid; c < C; c += kSelThreads) {
        const uint32_t k = key(c);
        if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 0xffu], 1);
      }
      __syncthreads();
      if (warp == 0) {
        int cnt[8];
        int tot = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          cnt[j] = hist[255 - 8 * lane - j];
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
              sh_i[1] = 255 - 8 * lane - j;
              sh_i[2] = acc;
              sh_i[3] = cnt[j];
              break;
            }
            acc += cnt[j];
          }
        }
      }
      __syncthreads();
      remaining -= sh_i[2];
      count_eq = sh_i[3];
      prefix |= (uint32_t)sh_i[1] << shift;
      mask |= 0xffu << shift;
    }
  }
  const bool any = r_eff > 0;
  const uint32_t T = prefix;  // the r_eff-th largest key
  // equal keys at the threshold: keep the `remaining` lowest ids
  int c_cut = INT_MAX;
  const int per = (C + kSelThreads - 1) / kSelThreads;
  const int my0 = min(C, tid * per), my1 = min(C, my0 + per);
  if (any && remaining < count_eq) {
    int ne = 0;
    for (int c = my0; c < my1; ++c) ne += (key(c) == T);
    int2 tot;
    const int before = block_scan2(make_int2(ne, 0), sh_scan, &tot).x;
    if (before < remaining && remaining <= before + ne) {
      int cnt = before;
      for (int c = my0; c < my1; ++c) {
        if (key(c) == T && ++cnt == remaining) {
          sh_i[4] = c;
          break;
        }
      }
    }
    __syncthreads();
    c_cut = sh_i[4];
  }
  auto is_sel = [&](uint32_t k, int c) { return any && (k > T || (k == T && c <= c_cut)); };

  // ordered compaction: ids ascending, exclusive prefix of member counts
  int nsel = 0, ntok = 0;
  for (int c = my0; c < my1; ++c) {
    if (is_sel(key(c), c)) {
      ++nsel;
      ntok += sz[c];
    }
  }
  int2 total;
  const int2 ex = block_scan2(make_int2(nsel, ntok), sh_scan, &total);
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
      tok += sz[c];
    }
  }
  for (int i = total.x + tid; i <= r; i += kSelThreads) {
    pre[i] = total.y;
    if (i < r) {
      ids[i] = -1;
      if (topk) topk[i] = -1;
    }
  }
  uint32_t* mk = a.sel_mask + (size_t)bh * a.n_words;
  for (int w = tid; w < a.n_words; w += kSelThreads) {
    uint32_t bits = 0;
    for (int j = 0; j < 32; ++j) {
      const int c = 32 * w + j;
      if (c < C && is_sel(key(c), c)) bits |= 1u << j;
    }
    mk[w] = bits;
  }
}

// --------------------------------------------------------------------------
// K3 + K4: exact attention (steady + retrieved) and estimation, one launch
// --------------------------------------------------------------------------
constexpr int kAttThreads = 256;
constexpr int kAttWarps = kAttThreads / 32;
constexpr int kTile = 64;      // tokens per pipeline stage (8 per warp)
constexpr int kStages = 2;
constexpr int kWinCap = 512;   // retrieved clusters staged per window

struct __align__(128) AttSmem {
  uint16_t k[kStages][kTile * kD];  // bulk-copy destinations: 16-byte aligned
  uint16_t v[kStages][kTile * kD];
  float red_o[kAttWarps][kD];       // written as float4: 16-byte aligned
  float red_m[kAttWarps];
  float red_l[kAttWarps];
  unsigned long long bar[kStages];  // mbarriers: 8-byte aligned
  int win_prefix[kWinCap + 1];
  int win_row[kWinCap];
};
static_assert(offsetof(AttSmem, v) % 128 == 0, "staging buffer alignment");
static_assert(offsetof(AttSmem, red_o) % 16 == 0, "float4 reduction buffer alignment");
static_assert(offsetof(AttSmem, bar) % 8 == 0, "mbarrier alignment");

template <int G>
struct EstSmem {
  float red_o[kAttWarps][G][kD];  // offset 0, written as float4
  float red_l[kAttWarps][G];
};

__device__ void attend_tokens(const DecodeArgs& a, int bh, int sp, AttSmem& S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = bh / a.Hq, h = bh - b * a.Hq, g = h / a.G;
  const size_t head = (size_t)b * a.Hkv + g;
  const uint16_t* Kh = a.K + head * (size_t)a.N * kD;
  const uint16_t* Vh = a.V + head * (size_t)a.N * kD;
  const uint16_t* Ksh = a.ksorted + head * (size_t)a.N_idx * kD;
  const uint16_t* Vsh = a.vsorted + head * (size_t)a.N_idx * kD;
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
  uint32_t phase = 0;
  bool ok = true;
  int round_lo = lo;
  while (ok && round_lo < hi) {
    int round_hi = hi;
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
      int n_cl = cnt_lt - i0;
      if (n_cl > kWinCap) {
        n_cl = kWinCap;
        round_hi = ns + pre[i0 + kWinCap];
      }
      for (int j = tid; j <= n_cl; j += kAttThreads) S.win_prefix[j] = pre[i0 + j];
      for (int j = tid; j < n_cl; j += kAttThreads) S.win_row[j] = off[ids[i0 + j]];
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
  // combine the warps
  if (lane == 0) {
    S.red_m[warp] = m_run;
    S.red_l[warp] = l_run;
  }
  reinterpret_cast<float4*>(S.red_o[warp])[lane] = make_float4(o0, o1, o2, o3);
  __syncthreads();
  if (tid < kD) {
    float M = -INFINITY;
    for (int w = 0; w < kAttWarps; ++w) M = fmaxf(M, S.red_m[w]);
    float L = 0.f, O = 0.f;
    if (ok && M > -INFINITY) {
      for (int w = 0; w < kAttWarps; ++w) {
        const float f = exp2f(S.red_m[w] - M);
        L += S.red_l[w] * f;
        O += S.red_o[w][tid] * f;
      }
    } else {
      M = -INFINITY;
    }
    float* P = a.att_part + ((size_t)bh * a.att_splits + sp) * kPartStride;
    if (tid == 0) {
      P[0] = M;
      P[1] = L;
    }
    P[2 + tid] = O;
  }
}

template <int G>
__device__ void estimate_clusters(const DecodeArgs& a, int bg, int chunk, EstSmem<G>& S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int c_begin = chunk * a.est_chunk_clusters;
  const int c_end = min(a.C, c_begin + a.est_chunk_clusters);
  const float4* vs = reinterpret_cast<const float4*>(a.vsum + (size_t)bg * a.C * kD);
  const int* sz = a.size + (size_t)bg * a.C;
  float hm[G];
  const float* sc[G];
  const uint32_t* mk[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const size_t bh = (size_t)b * a.Hq + g * G + h;
    hm[h] = a.head_max[bh] * kLog2e;
    sc[h] = a.scores + bh * a.C;
    mk[h] = a.sel_mask + bh * a.n_words;
  }
  float acc[G][4];
  float lsum[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    lsum[h] = 0.f;
    acc[h][0] = acc[h][1] = acc[h][2] = acc[h][3] = 0.f;
  }
  for (int base = c_begin + warp * 32; base < c_end; base += kAttWarps * 32) {
    const int c = base + lane;
    const bool valid = c < c_end;
    const int n = valid ? __ldg(sz + c) : 0;
    float p[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const bool sel = valid && ((__ldg(mk[h] + (c >> 5)) >> (c & 31)) & 1u);
      p[h] = (n > 0 && !sel) ? exp2f(__ldg(sc[h] + c) * kLog2e - hm[h]) : 0.f;
      lsum[h] += p[h] * (float)n;
    }
    const int cnt = min(32, c_end - base);
#pragma unroll 1
    for (int j0 = 0; j0 < cnt; j0 += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u;
        v[u] = (j < cnt) ? __ldg(vs + (size_t)(base + j) * (kD / 4) + lane)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float pj = __shfl_sync(kFull, p[h], j0 + u);
          acc[h][0] += pj * v[u].x;
          acc[h][1] += pj * v[u].y;
          acc[h][2] += pj * v[u].z;
          acc[h][3] += pj * v[u].w;
        }
      }
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    lsum[h] = warp_sum(lsum[h]);
    reinterpret_cast<float4*>(S.red_o[warp][h])[lane] =
        make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
    if (lane == 0) S.red_l[warp][h] = lsum[h];
  }
  __syncthreads();
  for (int idx = tid; idx < G * kD; idx += kAttThreads) {
    const int h = idx / kD, dim = idx - h * kD;
    float O = 0.f, L = 0.f;
    for (int w = 0; w < kAttWarps; ++w) {
      O += S.red_o[w][h][dim];
      L += S.red_l[w][h];
    }
    const size_t bh = (size_t)b * a.Hq + g * G + h;
    float* P = a.est_part + (bh * a.est_chunks + chunk) * kPartStride;
    if (dim == 0) {
      P[0] = (L > 0.f) ? a.head_max[bh] * kLog2e : -INFINITY;
      P[1] = L;
    }
    P[2 + dim] = O;
  }
}

template <int G>
__global__ void __launch_bounds__(kAttThreads) attend_kernel(DecodeArgs a, int n_att_blocks) {
  extern __shared__ __align__(128) unsigned char smem[];
  grid_dep_launch();
  grid_dep_wait();
  if ((int)blockIdx.x < n_att_blocks) {
    const int bh = blockIdx.x / a.att_splits;
    const int sp = blockIdx.x - bh * a.att_splits;
    attend_tokens(a, bh, sp, *reinterpret_cast<AttSmem*>(smem));
  } else {
    const int idx = blockIdx.x - n_att_blocks;
    const int bg = idx / a.est_chunks;
    const int chunk = idx - bg * a.est_chunks;
    estimate_clusters<G>(a, bg, chunk, *reinterpret_cast<EstSmem<G>*>(smem));
  }
}

// --------------------------------------------------------------------------
// K5: log-sum-exp merge
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(kD) merge_kernel(DecodeArgs a) {
  __shared__ float sh_m[kD / 32];
  grid_dep_launch();
  grid_dep_wait();
  const int bh = blockIdx.x, tid = threadIdx.x;
  const float* PA = a.att_part + (size_t)bh * a.att_splits * kPartStride;
  const float* PE = a.est_part + (size_t)bh * a.est_chunks * kPartStride;
  const int P = a.att_splits + a.est_chunks;
  auto part = [&](int i) {
    return i < a.att_splits ? PA + (size_t)i * kPartStride
                            : PE + (size_t)(i - a.att_splits) * kPartStride;
  };
  float M = -INFINITY;
  for (int i = tid; i < P; i += kD) M = fmaxf(M, part(i)[0]);
  M = warp_max(M);
  if ((tid & 31) == 0) sh_m[tid >> 5] = M;
  __syncthreads();
  M = fmaxf(fmaxf(sh_m[0], sh_m[1]), fmaxf(sh_m[2], sh_m[3]));
  float L = 0.f, O = 0.f;
  if (M > -INFINITY) {
#pragma unroll 4
    for (int i = 0; i < P; ++i) {
      const float* p = part(i);
      const float m = p[0];
      if (m > -INFINITY) {
        const float f = exp2f(m - M);
        L += p[1] * f;
        O += p[2 + tid] * f;
      }
    }
  }
  a.out[(size_t)bh * kD + tid] = (L > 0.f) ? O / L : 0.f;
  if (a.lse != nullptr && tid == 0) a.lse[bh] = (L > 0.f) ? (M + log2f(L)) * kLn2 : -INFINITY;
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
  const int rows_per_sweep = (kScoreThreads / 32) * (32 / a.G);
  const long long target_blocks = 148LL * 8;
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

cudaError_t launch_decode_select(const DecodeArgs& a, cudaStream_t st) {
  const int cached = a.C <= kSelCacheMax ? 1 : 0;
  const size_t smem = cached ? (size_t)a.C * sizeof(uint32_t) : 0;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = set_smem(select_kernel, (size_t)kSelCacheMax * sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(select_kernel, dim3((unsigned)(a.B * a.Hq)), dim3(kSelThreads), smem, st, true,
                   a, cached);
}

template <int G>
static cudaError_t launch_attend_g(const DecodeArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(AttSmem) > sizeof(EstSmem<G>) ? sizeof(AttSmem) : sizeof(EstSmem<G>);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = set_smem(attend_kernel<G>, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int n_att = a.B * a.Hq * a.att_splits;
  const int n_est = a.B * a.Hkv * a.est_chunks;
  return launch_ex(attend_kernel<G>, dim3((unsigned)(n_att + n_est)), dim3(kAttThreads), smem, st,
                   true, a, n_att);
}

cudaError_t launch_decode_attend(const DecodeArgs& a, cudaStream_t st) {
  switch (a.G) {
    case 1: return launch_attend_g<1>(a, st);
    case 2: return launch_attend_g<2>(a, st);
    case 4: return launch_attend_g<4>(a, st);
    case 8: return launch_attend_g<8>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_merge(const DecodeArgs& a, cudaStream_t st) {
  return launch_ex(merge_kernel, dim3((unsigned)(a.B * a.Hq)), dim3(kD), 0, st, true, a);
}

}  // namespace wi
