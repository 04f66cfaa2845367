// Index-build kernels: segmented spherical k-means over each KV head's keys
// ("RetroInfer: A Vector Storage Engine for Scalable Long-Context LLM
// Inference", technical summary (es) §2.A.2 clustering index and §3 segmented
// clustering; (ar) §2.a centroids and value sums, §2.b contiguous KV layout).
//
//   init_norms_kernel     : ||k_i|| in f32 for every position; assign = -1 on
//                           the steady zone.
//   init_centroids_kernel : strided seeding, mu_j = bf16(k_p / ||k_p||).
//   assign (wi_assign.cu) : argmax_j k_i . mu_j on the tensor cores.
//   cluster_sort_kernel   : per segment, stable counting sort of the
//                           assignment (per-warp histograms, no atomics):
//                           size, offset, perm.
//   centroid_update_kernel: mu_j = bf16(normalize(sum k_i / ||k_i||)) over the
//                           sorted members, f32, in position order.
//   finalize_kernel       : mean key, value sum, cluster-sorted K/V copies.
//   round_bf16_kernel     : bf16 copies of the mean keys and value sums (the
//                           leaner index decode may stream instead).
//   extend_copy_kernel /  : index maintenance as the local window slides:
//   extend_assign_kernel    earlier assignments and centroids carried over,
//                           each joining position to its segment's nearest
//                           unit centroid (then the sort and statistics
//                           kernels above on the new assignment).
#include "wi_device.cuh"
#include "wi_internal.h"

namespace wi {

namespace {

constexpr int kRowThreads = 256;

__global__ void __launch_bounds__(kRowThreads) init_norms_kernel(BuildArgs a) {
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)a.B * a.Hkv * a.N;
  const long long warps = (long long)gridDim.x * (kRowThreads / 32);
  for (long long row = (long long)blockIdx.x * (kRowThreads / 32) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const uint2 w = reinterpret_cast<const uint2*>(a.K + row * kD)[lane];
    const float x0 = bf_lo(w.x), x1 = bf_hi(w.x), x2 = bf_lo(w.y), x3 = bf_hi(w.y);
    const float ss = warp_sum(x0 * x0 + x1 * x1 + x2 * x2 + x3 * x3);
    if (lane == 0) {
      a.norms[row] = sqrtf(ss);
      const int pos = (int)(row % a.N);
      if (pos < a.sink || pos >= a.N - a.window) a.assign[row] = -1;
    }
  }
}

__global__ void __launch_bounds__(kRowThreads) init_centroids_kernel(BuildArgs a) {
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)a.B * a.Hkv * a.C;
  const long long warps = (long long)gridDim.x * (kRowThreads / 32);
  for (long long row = (long long)blockIdx.x * (kRowThreads / 32) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const long long bg = row / a.C;
    const int c = (int)(row - bg * a.C);
    const int s = c / a.k, j = c - s * a.k;
    const int lo = a.seg_lo(s), hi = a.seg_hi(s);
    const int m = hi - lo;
    uint2 out = make_uint2(0u, 0u);
    if (m > 0) {
      const int p = lo + (int)(((long long)j * m) / a.k);
      const uint2 w = reinterpret_cast<const uint2*>(a.K + (bg * a.N + p) * kD)[lane];
      const float x0 = bf_lo(w.x), x1 = bf_hi(w.x), x2 = bf_lo(w.y), x3 = bf_hi(w.y);
      const float nrm = sqrtf(warp_sum(x0 * x0 + x1 * x1 + x2 * x2 + x3 * x3));
      if (nrm > 0.f) out = make_uint2(pack_bf2(x0 / nrm, x1 / nrm), pack_bf2(x2 / nrm, x3 / nrm));
    }
    reinterpret_cast<uint2*>(a.mu + row * kD)[lane] = out;
  }
}

// Stable counting sort of one segment's assignment.  Warp w owns a contiguous
// run of the segment's positions and counts them in rounds of 32 with
// __match_any_sync; a scan over (bucket, warp) gives every warp its base per
// bucket; the scatter repeats the rounds.  Order within a bucket = position.
constexpr int kSortThreads = 1024;
constexpr int kSortWarps = kSortThreads / 32;

__global__ void __launch_bounds__(kSortThreads, 1) cluster_sort_kernel(BuildArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint16_t* loc = reinterpret_cast<uint16_t*>(smem_raw);                   // [WI_MAX_SEG_LEN]
  uint16_t* wh = loc + WI_MAX_SEG_LEN;                                      // [kSortWarps][k]
  int* bstart = reinterpret_cast<int*>(wh + kSortWarps * WI_MAX_K_PER_SEG);  // [k]
  __shared__ int sh_w[33];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bg = blockIdx.x / a.n_seg, s = blockIdx.x - (blockIdx.x / a.n_seg) * a.n_seg;
  const int lo = a.seg_lo(s), hi = a.seg_hi(s), m = hi - lo;
  const int k = a.k;
  const int slot0 = lo - a.sink;  // first sorted slot of this segment
  const int* asg = a.assign + (size_t)bg * a.N + lo;
  for (int e = tid; e < m; e += kSortThreads) {
    int lj = asg[e] - s * k;
    if ((unsigned)lj >= (unsigned)k) {  // not an id of this segment: keep memory safe
      report(a.status, WI_ERR_INDEX_MISMATCH);
      lj = 0;
    }
    loc[e] = (uint16_t)lj;
  }
  for (int i = tid; i < kSortWarps * k; i += kSortThreads) wh[i] = 0;
  __syncthreads();

  const int E = (m + kSortWarps - 1) / kSortWarps;
  const int e_begin = warp * E, e_end = min(m, e_begin + E);
  const unsigned lt_mask = (1u << lane) - 1u;
  // counting rounds
  for (int e0 = e_begin; e0 < e_end; e0 += 32) {
    const int e = e0 + lane;
    const bool valid = e < e_end;
    const unsigned bucket = valid ? loc[e] : 0xffffu;
    const unsigned peers = __match_any_sync(kFull, bucket);
    const int leader = __ffs(peers) - 1;
    if (valid && lane == leader) wh[warp * k + bucket] += (uint16_t)__popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // bucket totals, exclusive scan over buckets, per-(bucket, warp) bases
  int tot = 0;
  if (tid < k) {
    for (int w = 0; w < kSortWarps; ++w) tot += wh[w * k + tid];
  }
  int incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sh_w[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = sh_w[lane];
    int vi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, vi, o);
      if (lane >= o) vi += t;
    }
    sh_w[lane] = vi - v;
  }
  __syncthreads();
  if (tid < k) {
    const int start = sh_w[warp] + incl - tot;
    bstart[tid] = start;
    int run = start;
    for (int w = 0; w < kSortWarps; ++w) {
      const int t = wh[w * k + tid];
      wh[w * k + tid] = (uint16_t)run;
      run += t;
    }
    const size_t c = (size_t)bg * a.C + (size_t)s * k + tid;
    a.size[c] = tot;
    a.offset[(size_t)bg * (a.C + 1) + (size_t)s * k + tid] = slot0 + start;
  }
  if (tid == 0 && s == a.n_seg - 1) a.offset[(size_t)bg * (a.C + 1) + a.C] = a.N_idx;
  __syncthreads();
  // scatter rounds
  int* perm = a.perm + (size_t)bg * a.N_idx + slot0;
  for (int e0 = e_begin; e0 < e_end; e0 += 32) {
    const int e = e0 + lane;
    const bool valid = e < e_end;
    const unsigned bucket = valid ? loc[e] : 0xffffu;
    const unsigned peers = __match_any_sync(kFull, bucket);
    const int leader = __ffs(peers) - 1;
    const int rank = __popc(peers & lt_mask);
    int base = 0;
    if (valid) base = wh[warp * k + bucket];
    __syncwarp();
    if (valid) {
      perm[base + rank] = lo + e;
      if (lane == leader) wh[warp * k + bucket] = (uint16_t)(base + __popc(peers));
    }
    __syncwarp();
  }
}

// One warp per cluster; members are contiguous in perm.  Members are summed
// in position order (the sorted order), 8 rows in flight per warp.
constexpr int kClusterThreads = 256;
constexpr int kClustersPerBlock = 64;

template <bool kFinalize>
__global__ void __launch_bounds__(kClusterThreads) cluster_reduce_kernel(BuildArgs a,
                                                                         int blocks_per_head) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int bg = blockIdx.x / blocks_per_head;
  const int cb = (blockIdx.x - bg * blocks_per_head) * kClustersPerBlock;
  const uint16_t* Kh = a.K + (size_t)bg * a.N * kD;
  const uint16_t* Vh = a.V + (size_t)bg * a.N * kD;
  const float* nrm = a.norms + (size_t)bg * a.N;
  const int* perm = a.perm + (size_t)bg * a.N_idx;
  for (int c = cb + warp; c < min(a.C, cb + kClustersPerBlock); c += kClusterThreads / 32) {
    const size_t cg = (size_t)bg * a.C + c;
    const int n = a.size[cg];
    const int o = a.offset[(size_t)bg * (a.C + 1) + c];
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;  // keys (unit or raw)
    float t0 = 0.f, t1 = 0.f, t2 = 0.f, t3 = 0.f;  // values
    for (int m0 = 0; m0 < n; m0 += 32) {
      const int cnt = min(32, n - m0);
      const int mypos = lane < cnt ? perm[o + m0 + lane] : 0;
      for (int u0 = 0; u0 < cnt; u0 += 8) {
        uint2 kw[8], vw[8];
        float nk[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int pos = __shfl_sync(kFull, mypos, (u0 + u) & 31);
          if (u0 + u < cnt) {
            kw[u] = reinterpret_cast<const uint2*>(Kh + (size_t)pos * kD)[lane];
            if (kFinalize) {
              vw[u] = reinterpret_cast<const uint2*>(Vh + (size_t)pos * kD)[lane];
            } else {
              nk[u] = nrm[pos];
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (u0 + u < cnt) {
            const float x0 = bf_lo(kw[u].x), x1 = bf_hi(kw[u].x);
            const float x2 = bf_lo(kw[u].y), x3 = bf_hi(kw[u].y);
            if (kFinalize) {
              s0 += x0; s1 += x1; s2 += x2; s3 += x3;
              t0 += bf_lo(vw[u].x); t1 += bf_hi(vw[u].x);
              t2 += bf_lo(vw[u].y); t3 += bf_hi(vw[u].y);
              const size_t slot = (size_t)bg * a.N_idx + o + m0 + u0 + u;
              reinterpret_cast<uint2*>(a.ksorted + slot * kD)[lane] = kw[u];
              reinterpret_cast<uint2*>(a.vsorted + slot * kD)[lane] = vw[u];
            } else if (nk[u] > 0.f) {
              s0 += x0 / nk[u]; s1 += x1 / nk[u]; s2 += x2 / nk[u]; s3 += x3 / nk[u];
            }
          }
        }
      }
    }
    if (kFinalize) {
      const float fn = (float)n;
      const float4 kb = n > 0 ? make_float4(s0 / fn, s1 / fn, s2 / fn, s3 / fn)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
      reinterpret_cast<float4*>(a.kbar + cg * kD)[lane] = kb;
      reinterpret_cast<float4*>(a.vsum + cg * kD)[lane] = make_float4(t0, t1, t2, t3);
    } else {
      const float ss = warp_sum(s0 * s0 + s1 * s1 + s2 * s2 + s3 * s3);
      if (n > 0 && ss > 0.f) {
        const float nr = sqrtf(ss);
        reinterpret_cast<uint2*>(a.mu + cg * kD)[lane] =
            make_uint2(pack_bf2(s0 / nr, s1 / nr), pack_bf2(s2 / nr, s3 / nr));
      }
    }
  }
}

int grid_rows(long long rows) {
  const long long warps_per_block = kRowThreads / 32;
  long long blocks = (rows + warps_per_block - 1) / warps_per_block;
  const long long cap = 148LL * 16;
  return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_build_init(const BuildArgs& a, cudaStream_t st) {
  init_norms_kernel<<<grid_rows((long long)a.B * a.Hkv * a.N), kRowThreads, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  init_centroids_kernel<<<grid_rows((long long)a.B * a.Hkv * a.C), kRowThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_cluster_sort(const BuildArgs& a, cudaStream_t st) {
  const size_t smem = (size_t)WI_MAX_SEG_LEN * 2 + (size_t)kSortWarps * WI_MAX_K_PER_SEG * 2 +
                      (size_t)WI_MAX_K_PER_SEG * 4;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(cluster_sort_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cluster_sort_kernel<<<a.B * a.Hkv * a.n_seg, kSortThreads, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_centroid_update(const BuildArgs& a, cudaStream_t st) {
  const int bph = (a.C + kClustersPerBlock - 1) / kClustersPerBlock;
  cluster_reduce_kernel<false><<<a.B * a.Hkv * bph, kClusterThreads, 0, st>>>(a, bph);
  return cudaGetLastError();
}

// dst[i] = bf16(src[i]) (round to nearest even), 4 values per thread step
__global__ void round_bf16_kernel(const float4* __restrict__ src, uint2* __restrict__ dst,
                                  size_t n4) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 v = src[i];
    dst[i] = make_uint2((uint32_t)f2bf(v.x) | ((uint32_t)f2bf(v.y) << 16),
                        (uint32_t)f2bf(v.z) | ((uint32_t)f2bf(v.w) << 16));
  }
}

// Carried-over state of one (sequence, KV head): unit centroids (zero for
// clusters new to the index), assignments of the earlier indexable positions,
// -1 on the steady zone.  Joining positions are left to extend_assign_kernel.
__global__ void extend_copy_kernel(ExtendArgs e) {
  const int bh = blockIdx.y;
  const size_t mu_words = (size_t)e.C_new * kD / 2;  // bf16 pairs
  const uint32_t* src = reinterpret_cast<const uint32_t*>(e.mu_old) + (size_t)bh * e.C_old * kD / 2;
  uint32_t* dst = reinterpret_cast<uint32_t*>(e.mu_new) + (size_t)bh * mu_words;
  const size_t old_words = (size_t)e.C_old * kD / 2;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < mu_words;
       i += (size_t)gridDim.x * blockDim.x)
    dst[i] = i < old_words ? src[i] : 0u;
  const int hi_old = e.N0 - e.window, hi = e.N1 - e.window;
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < e.N1; p += gridDim.x * blockDim.x) {
    if (p >= hi_old && p < hi && p >= e.sink) continue;  // joining: extend_assign_kernel
    const bool idx = p >= e.sink && p < hi_old;
    e.assign_new[(size_t)bh * e.N1 + p] = idx ? e.assign_old[(size_t)bh * e.N0 + p] : -1;
  }
}

// One warp per joining position: a(p) = t k + argmax_j k_p . mu_{t k + j}
// (f32 sums of bf16 products, the lowest j among equal maxima), t = p / L,
// the position's segment (clustered before: the host checks it).
__global__ void __launch_bounds__(256) extend_assign_kernel(ExtendArgs e, int n_join) {
  __shared__ float keys[8][kD];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const long long gw = (long long)blockIdx.x * 8 + w;
  const int bh = (int)(gw / n_join);
  if (bh >= e.B * e.Hkv) return;
  const int p = max(e.N0 - e.window, e.sink) + (int)(gw - (long long)bh * n_join);
  const uint2 kw = *reinterpret_cast<const uint2*>(e.K + ((size_t)bh * e.N1 + p) * kD + lane * 4);
  keys[w][lane * 4] = bf_lo(kw.x);
  keys[w][lane * 4 + 1] = bf_hi(kw.x);
  keys[w][lane * 4 + 2] = bf_lo(kw.y);
  keys[w][lane * 4 + 3] = bf_hi(kw.y);
  __syncwarp();
  const int t = p / e.L;
  const uint16_t* mu = e.mu_old + ((size_t)bh * e.C_old + (size_t)t * e.k) * kD;
  float best = -INFINITY;
  int arg = 0x7fffffff;
  for (int j = lane; j < e.k; j += 32) {
    const uint2* row = reinterpret_cast<const uint2*>(mu + (size_t)j * kD);
    float acc = 0.f;
#pragma unroll 8
    for (int q = 0; q < kD / 4; ++q) {
      const uint2 m = row[q];
      acc = fmaf(keys[w][4 * q], bf_lo(m.x), acc);
      acc = fmaf(keys[w][4 * q + 1], bf_hi(m.x), acc);
      acc = fmaf(keys[w][4 * q + 2], bf_lo(m.y), acc);
      acc = fmaf(keys[w][4 * q + 3], bf_hi(m.y), acc);
    }
    if (acc > best) {  // j ascends within the lane: the first maximum is kept
      best = acc;
      arg = j;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(kFull, best, o);
    const int oa = __shfl_xor_sync(kFull, arg, o);
    if (ob > best || (ob == best && oa < arg)) {
      best = ob;
      arg = oa;
    }
  }
  if (lane == 0) e.assign_new[(size_t)bh * e.N1 + p] = t * e.k + (arg < e.k ? arg : 0);
}

cudaError_t launch_extend(const ExtendArgs& e, cudaStream_t st) {
  extend_copy_kernel<<<dim3(16, e.B * e.Hkv), 256, 0, st>>>(e);
  cudaError_t err = cudaGetLastError();
  const int n_join = (e.N1 - e.window) - max(e.N0 - e.window, e.sink);
  if (err != cudaSuccess || n_join <= 0) return err;
  const long long warps = (long long)e.B * e.Hkv * n_join;
  extend_assign_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(e, n_join);
  return cudaGetLastError();
}

cudaError_t launch_round_bf16(const float* src, uint16_t* dst, size_t n, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const size_t n4 = n / 4;  // n is a multiple of 128
  round_bf16_kernel<<<sms * 4, 256, 0, st>>>(reinterpret_cast<const float4*>(src),
                                             reinterpret_cast<uint2*>(dst), n4);
  return cudaGetLastError();
}

cudaError_t launch_finalize_stats(const BuildArgs& a, cudaStream_t st) {
  const int bph = (a.C + kClustersPerBlock - 1) / kClustersPerBlock;
  cluster_reduce_kernel<true><<<a.B * a.Hkv * bph, kClusterThreads, 0, st>>>(a, bph);
  return cudaGetLastError();
}

}  // namespace wi
