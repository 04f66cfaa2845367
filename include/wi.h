/*
 * wi.h -- C ABI of libwi: wave-index tripartite decode attention and its
 * segmented spherical-k-means index build, for one NVIDIA B300 (sm_103a).
 *
 * Method: "RetroInfer: A Vector Storage Engine for Scalable Long-Context LLM
 * Inference".  Technical summary (es) §2.A "Wave Index": a tripartite attention
 * approximation -- §2.A.1 steady zone (sink tokens and the local window,
 * attended exactly), §2.A.2 retrieval zone (a spherical-k-means clustering
 * index; the clusters most similar to the query are attended exactly),
 * §2.A.3 estimation zone (cluster centroids estimate the remaining tokens);
 * §3 segmented clustering (k-means on short segments of the sequence, to cut
 * index-build time at prefill).  Technical summary (ar) §2.a: the estimation
 * zone uses the cluster centroids and the sum of the value vectors; §2.b the
 * execution buffer lays retrieved KV out contiguously for FlashAttention-class
 * kernels.  The pages print no formulas; the exact arithmetic of every call is
 * stated beside it below.
 *
 * Conventions (all calls):
 *  - Every pointer argument is a DEVICE pointer, allocated and owned by the
 *    caller, unless its comment says "host".  The library never allocates or
 *    frees memory and never synchronises, except wi_sync_status.
 *  - Every call is asynchronous on the given stream (NULL = legacy default
 *    stream) and returns a wi_status.  Argument errors are found on the host
 *    before anything is enqueued.  Errors found on the device (an exhausted
 *    bounded wait) are recorded in the status word at the start of the
 *    caller's workspace; wi_sync_status reads and clears it.
 *  - bf16 tensors are IEEE bfloat16 bit patterns (uint16).  K and V use the
 *    head-major layout [B, Hkv, N, d], contiguous, d = 128; query head h reads
 *    KV head h / (Hq / Hkv) (grouped-query attention).
 *  - Pointers must be 16-byte aligned (256-byte aligned for workspaces).
 *  - Calls that share a workspace must not overlap on the GPU: they race.
 *  - Workspaces must be zero-filled once before their first use; the library
 *    leaves their status word and counters at zero after every call that does
 *    not fail.
 */
#ifndef WI_H_
#define WI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols keep default visibility; everything else is hidden. */
#if defined(__GNUC__)
#define WI_API __attribute__((visibility("default")))
#else
#define WI_API
#endif

/* cudaStream_t without including the CUDA headers. */
typedef struct CUstream_st *wi_stream_t;

typedef enum {
  WI_OK = 0,
  WI_ERR_INVALID_ARG = 1,     /* NULL pointer, bad size, bad combination      */
  WI_ERR_UNSUPPORTED = 2,     /* d != 128, group size not in {1,2,4,8}, limit */
  WI_ERR_LAUNCH = 3,          /* a CUDA launch or query failed                */
  WI_ERR_INDEX_MISMATCH = 4,  /* decode params disagree with the index        */
  WI_ERR_DEVICE_TIMEOUT = 5,  /* a device-side bounded wait ran out           */
  WI_ERR_WORKSPACE = 6,       /* workspace too small                          */
  WI_ERR_ALIGNMENT = 7,       /* a pointer is not suitably aligned            */
  WI_ERR_CUDA = 8             /* wi_sync_status: the stream reported an error */
} wi_status;

/* Limits of this library. */
#define WI_HEAD_DIM 128
#define WI_MAX_K_PER_SEG 512
#define WI_MAX_SEG_LEN 16384
#define WI_MAX_CLUSTERS (1 << 20)

/* Index-build parameters.
 *  B, Hkv, N, d   : sequences, KV heads, context length, head dim (128).
 *  sink, window   : steady zone = positions [0, sink) and [N - window, N);
 *                   sink + window <= N.  The index covers the other N_idx =
 *                   N - sink - window positions.
 *  seg_len        : segment length; segment s covers absolute positions
 *                   [s * seg_len, (s + 1) * seg_len) minus the steady zone;
 *                   n_seg = ceil(N / seg_len), 1 <= seg_len <= WI_MAX_SEG_LEN.
 *  k_per_seg      : clusters per segment (1..WI_MAX_K_PER_SEG);
 *                   cluster j of segment s has id c = s * k_per_seg + j and
 *                   C = n_seg * k_per_seg <= WI_MAX_CLUSTERS.
 *  iters          : (assign, update) rounds of spherical k-means, >= 1. */
typedef struct {
  int B, Hkv, N, d, sink, window, seg_len, k_per_seg, iters;
} wi_build_params;

/* Decode parameters.
 *  r     : retrieval budget, clusters per query head, 0 <= r <= C.
 *  scale : logit scale, normally 1/sqrt(d).
 *  sink, window must equal the index's. */
typedef struct {
  int B, Hq, Hkv, N, d, sink, window, r;
  float scale;
} wi_decode_params;

/* The wave index of every (sequence b, KV head g).  The caller allocates
 * every array (sizes from wi_index_sizes) and fills the pointers; the build
 * writes the arrays and the scalar fields after the pointers.
 *   centroid_key  f32  [B,Hkv,C,d]   mean raw key of each cluster (0 if empty)
 *   unit_centroid bf16 [B,Hkv,C,d]   spherical k-means centroid (unit length)
 *   value_sum     f32  [B,Hkv,C,d]   sum of the cluster's value vectors
 *   size          i32  [B,Hkv,C]     members per cluster, n_c
 *   offset        i32  [B,Hkv,C+1]   start of cluster c in the sorted arrays
 *   perm          i32  [B,Hkv,N_idx] sorted slot -> absolute position, sorted
 *                                    by (cluster, position)
 *   assign        i32  [B,Hkv,N]     position -> cluster id, -1 = steady zone
 *   k_sorted      bf16 [B,Hkv,N_idx,d]  K rows in perm order
 *   v_sorted      bf16 [B,Hkv,N_idx,d]  V rows in perm order */
typedef struct {
  float *centroid_key;
  void *unit_centroid;
  float *value_sum;
  int32_t *size;
  int32_t *offset;
  int32_t *perm;
  int32_t *assign;
  void *k_sorted;
  void *v_sorted;
  /* recorded by wi_build_index / wi_build_init */
  int B, Hkv, N, d, sink, window, seg_len, k_per_seg, n_clusters;
} wi_index;

enum {
  WI_FIELD_CENTROID_KEY = 0,
  WI_FIELD_UNIT_CENTROID,
  WI_FIELD_VALUE_SUM,
  WI_FIELD_SIZE,
  WI_FIELD_OFFSET,
  WI_FIELD_PERM,
  WI_FIELD_ASSIGN,
  WI_FIELD_K_SORTED,
  WI_FIELD_V_SORTED,
  WI_NUM_FIELDS
};

/* Bytes of every index array, in WI_FIELD_* order, into host array
 * bytes_out[WI_NUM_FIELDS].  No device work. */
WI_API int wi_index_sizes(const wi_build_params *p, size_t *bytes_out);

/* Workspace bytes needed by the build calls (status word + per-token key
 * norms).  0 on invalid parameters.  No device work. */
WI_API size_t wi_build_workspace_bytes(const wi_build_params *p);

/* Full index build (technical summary (es) §2.A.2 and §3; (ar) §2.a, §2.b):
 * wi_build_init, then iters x (wi_kmeans_assign, wi_kmeans_update), then
 * wi_build_finalize on the last assignment.  K, V: bf16 [B,Hkv,N,d]. */
WI_API int wi_build_index(const wi_build_params *p, const void *K, const void *V, wi_index *index,
                   void *workspace, size_t workspace_bytes, wi_stream_t stream);

/* Index maintenance as the local window slides (technical summary (es)
 * §2.A.1; the pages give no maintenance rule, this is the reading): the
 * context grew from old_index->N to p->N positions, so positions
 * [old N - window, p->N - window) leave the steady zone and join the index
 * without re-clustering.  Earlier positions keep their clusters and the unit
 * centroids are carried over (clusters of segments new to the index start
 * empty with zero centroids); a joining position p takes the nearest unit
 * centroid of its segment, argmax_j k_p . mu_j (f32 sums, the lowest j among
 * equal maxima); then size / offset / perm, mean keys, value sums and the
 * sorted copies are those of the new assignment (as wi_build_finalize).
 * p: the build parameters of the grown context (same B, Hkv, sink, window,
 * seg_len, k_per_seg as old_index; iters unused).  K, V: bf16 [B,Hkv,p->N,d].
 * index: arrays sized by wi_index_sizes(p), not shared with old_index.
 * workspace: wi_build_workspace_bytes(p).  WI_ERR_INDEX_MISMATCH when the
 * shapes differ or the context shrank; WI_ERR_UNSUPPORTED when a joining
 * position falls in a segment the earlier index did not cluster (or it
 * clustered none): a rebuild opens that segment. */
WI_API int wi_index_extend(const wi_build_params *p, const void *K, const void *V,
                    const wi_index *old_index, wi_index *index, void *workspace,
                    size_t workspace_bytes, wi_stream_t stream);

/* Build step 1: key norms ||k_i|| (f32, into the workspace), assign = -1 on
 * the steady zone, and the initial centroids: with the m_s indexable keys of
 * segment s in position order, centroid j = bf16(k_p / ||k_p||) for
 * p = floor(j * m_s / k_per_seg) (zero when m_s = 0).  Records the index's
 * scalar fields. */
WI_API int wi_build_init(const wi_build_params *p, const void *K, wi_index *index, void *workspace,
                  size_t workspace_bytes, wi_stream_t stream);

/* Build step 2 (one spherical k-means assignment): for every indexable
 * position i of segment s, assign[i] = s * k_per_seg + argmax_j k_i . mu_j
 * over the segment's centroids, the lowest j among equal maxima.  The dot
 * products run on the tensor cores (bf16 operands, f32 accumulation). */
WI_API int wi_kmeans_assign(const wi_build_params *p, const void *K, wi_index *index, void *workspace,
                     size_t workspace_bytes, wi_stream_t stream);

/* Build step 3 (one spherical k-means update): a stable counting sort of the
 * current assignment writes size, offset and perm; then every non-empty
 * cluster gets mu_j = bf16(normalize(sum over members of k_i / ||k_i||)),
 * summed in f32 in position order without atomics.  Empty clusters, and
 * clusters whose member directions sum to zero, keep their centroid. */
WI_API int wi_kmeans_update(const wi_build_params *p, const void *K, wi_index *index, void *workspace,
                     size_t workspace_bytes, wi_stream_t stream);

/* Build step 4: from the current assignment, size / offset / perm (stable
 * counting sort), centroid_key = (sum of member keys) / n_c and value_sum =
 * sum of member values (f32 sums in position order), and the cluster-sorted
 * copies k_sorted / v_sorted. */
WI_API int wi_build_finalize(const wi_build_params *p, const void *K, const void *V, wi_index *index,
                      void *workspace, size_t workspace_bytes, wi_stream_t stream);

/* Workspace bytes of wi_decode_attention and its stage calls; 0 on invalid
 * parameters.  n_clusters is the index's C.  No device work. */
WI_API size_t wi_decode_workspace_bytes(const wi_decode_params *p, int n_clusters);

/* Byte offsets of the decode workspace regions (host struct), for
 * inspection of intermediate results.  No device work.  Partials are
 * (m, l, o[d]) triples in log2 units (m is a log2-scaled logit). */
typedef struct {
  size_t counters;      /* per-call progress counters: launch-wide words
                           (blocks finished, selections published; 256 B),
                           then u32 [B*Hkv] scored index tiles, u32 [B*Hq]
                           published partials and u32 [B*Hq] published
                           selections; zero before the first call; every
                           call leaves them at zero                        */
  size_t scores;        /* f32 [B,Hq,C]   s_c = scale q.kbar_c, -inf if empty */
  size_t head_max;      /* f32 [B,Hq]     max_c s_c                           */
  size_t selected;      /* i32 [B,Hq,max(r,1)]  retrieved ids ascending, -1 pad */
  size_t sel_rows;      /* i32 [B,Hq,max(r,1)]  first k_sorted row of each      */
  size_t sel_counts;    /* i32 [B,Hq,max(r,1)]  its size n_c (0 for padding)     */
  size_t sel_prefix;    /* i32 [B,Hq,max(r,1)]  retrieved tokens before it       */
  size_t sel_scores;    /* f32 [B,Hq,max(r,1)]  its score s_c (-inf padding)     */
  size_t head_tokens;   /* i32 [B,Hq]     retrieved tokens of the head           */
  size_t group_values;  /* f32 [B,Hkv,C]  shared selection: the group's summed
                           ranking keys (-inf if empty)                      */
  size_t partials;      /* f32 partials: estimate pieces (per chunk of index
                           tiles and query head), steady pieces (per steady
                           tile and query head), retrieval pieces            */
  size_t total;
  int counter_bytes;    /* bytes of the counters region                        */
  int max_blocks;       /* blocks the partial buffers are sized for            */
  int reserved0, reserved1;
} wi_decode_layout;
WI_API int wi_decode_workspace_layout(const wi_decode_params *p, int n_clusters,
                               wi_decode_layout *layout_out);

/* Tripartite decode attention for one query per (sequence, query head)
 * (technical summary (es) §2.A; (ar) §2.a):
 *   s_c  = scale q.centroid_key_c for n_c > 0, -inf otherwise;
 *   T    = the r largest s_c over non-empty clusters, ties to the lower id;
 *   S    = steady positions + members of T, logits l_i = scale q.k_i
 *          (members read from k_sorted / v_sorted, the steady zone from K / V);
 *   E    = non-empty clusters outside T;
 *   M    = max(max_S l_i, max_E s_c),
 *   L    = sum_S e^{l_i - M} + sum_E n_c e^{s_c - M},
 *   out  = (sum_S e^{l_i - M} v_i + sum_E e^{s_c - M} value_sum_c) / L,
 *   lse  = M + ln L  (log-sum-exp merge of the three zones).
 * The E sums are formed as (all non-empty clusters) minus (clusters in T), in
 * f32: every member i of a cluster c in T enters with the weight
 * e^{l_i} - e^{s_c}; this reorders the arithmetic only.
 * q: bf16 [B,Hq,d]; out: f32 [B,Hq,d]; lse: f32 [B,Hq] or NULL;
 * topk_ids: i32 [B,Hq,r] (ascending ids, -1 padding) or NULL.
 * One persistent cooperative launch of one block per SM runs the three
 * stages below as one pipeline: blocks wait on per-call counters for exactly
 * the results they read (a KV group's scores, the published selections, a
 * head's partials), with no grid-wide barrier.  The blocks must be
 * co-resident: the launch fails with WI_ERR_LAUNCH otherwise.  Equivalent to
 * wi_decode_score, wi_decode_select, wi_decode_attend in order. */
WI_API int wi_decode_attention(const wi_decode_params *p, const void *q, const void *K, const void *V,
                        const wi_index *index, float *out, float *lse, int32_t *topk_ids,
                        void *workspace, size_t workspace_bytes, wi_stream_t stream);

/* Ranking keys of the retrieval zone (wi_decode_options.rank). */
enum { WI_RANK_SCORE = 0, WI_RANK_MASS = 1 };
/* Granularity of the retrieval zone (wi_decode_options.share). */
enum { WI_SHARE_HEAD = 0, WI_SHARE_GROUP = 1 };

/* Options of wi_decode_attention_ex.  All-zero options (rank WI_RANK_SCORE,
 * prev_q NULL, reused NULL) give wi_decode_attention. */
typedef struct {
  /* WI_RANK_SCORE: T = the r largest s_c (ties to the lower id).
   * WI_RANK_MASS: T = the r largest estimated attention masses n_c e^{s_c},
   * compared as s_c + ln n_c in f32 (ties to the lower id); the attention-
   * aware ranking of technical summary (ar) §2.a.  Everything after the
   * selection is unchanged. */
  int rank;
  /* Speculative reuse with correction (FreeKV technical summary §2.A).  With
   * prev_q set, for each KV group (b, g) the smallest cosine
   * cos(q[b,h], prev_q[b,h]) over its query heads h (0 where either query is
   * zero; f32) is compared with tau: if it is >= tau, every head of the group
   * takes as T the ids of its row of prev_topk instead of selecting; else
   * the group selects afresh.  The decision is an f32 comparison: a cosine
   * within rounding of tau may go either way.  A prev_topk row must hold
   * strictly ascending ids in [0, C) followed by -1 padding (what topk_ids
   * returns); a row that does not is reported as WI_ERR_INVALID_ARG in the
   * device status and that head selects afresh.  topk_ids may be the same
   * array as prev_topk: each row is read before it is rewritten.  Ignored
   * when r = 0. */
  float tau;
  const void *prev_q;        /* bf16 [B,Hq,d] device, 16-byte aligned, or NULL   */
  const int32_t *prev_topk;  /* i32 [B,Hq,r] device (required with prev_q)      */
  int32_t *reused;           /* i32 [B,Hq] device or NULL: 1 where the head took
                                its previous set, else 0                         */
  /* WI_SHARE_HEAD: every query head selects its own set.  WI_SHARE_GROUP:
   * one set per KV group, the r largest summed ranking keys
   * sum_h key_h(c) over the group's query heads (ties to the lower id);
   * every head of the group attends over it with its own logits and scores
   * (the selection granularity is left open by technical summary (es)
   * §2.A.2).  With reuse, a group takes its first head's previous set. */
  int share;
  /* Leaner index: bf16 copies of index->centroid_key and index->value_sum
   * (bf16 [B,Hkv,C,d] device, 16-byte aligned, as wi_index_round_bf16
   * writes them), both or neither.  When set, decode streams these instead of
   * the f32 arrays (half the index bytes); scores and estimates use the
   * rounded values. */
  const void *centroid_key_bf16;
  const void *value_sum_bf16;
} wi_decode_options;

/* The bf16 copies of a built index's mean keys and value sums used by
 * wi_decode_options.centroid_key_bf16 / value_sum_bf16: each element is the
 * f32 value rounded to nearest even.  Output arrays bf16 [B,Hkv,C,d] (device,
 * 16-byte aligned, caller-owned).  WI_ERR_INVALID_ARG for null pointers or an
 * index without recorded shape. */
WI_API int wi_index_round_bf16(const wi_index *index, void *centroid_key_bf16, void *value_sum_bf16,
                        wi_stream_t stream);

/* wi_decode_attention with selection options (options may be NULL).
 * Returns WI_ERR_INVALID_ARG for an unknown rank or share, prev_q without
 * prev_topk, a NaN tau or only one of the bf16 index arrays, and WI_ERR_ALIGNMENT for misaligned option pointers, before
 * anything is enqueued. */
WI_API int wi_decode_attention_ex(const wi_decode_params *p, const wi_decode_options *options,
                           const void *q, const void *K, const void *V,
                           const wi_index *index, float *out, float *lse, int32_t *topk_ids,
                           void *workspace, size_t workspace_bytes, wi_stream_t stream);

/* Decode stage 1: one stream over the centroid keys and the value sums:
 * the cluster scores s into the workspace, and the estimate of every
 * non-empty cluster, (m, l = sum n_c e^{s_c - m}, o = sum e^{s_c - m}
 * value_sum_c), as partials. */
WI_API int wi_decode_score(const wi_decode_params *p, const void *q, const wi_index *index,
                    void *workspace, size_t workspace_bytes, wi_stream_t stream);

/* Decode stage 2: per query head, the retrieval set T (the r largest scores,
 * ties to the lower id) with the clusters' sorted rows, sizes, token offsets
 * and scores, and the head's maximum score.  topk_ids may be NULL. */
WI_API int wi_decode_select(const wi_decode_params *p, const wi_index *index, int32_t *topk_ids,
                     void *workspace, size_t workspace_bytes, wi_stream_t stream);

/* Decode stage 3: exact attention over the steady zone and over the members
 * of T, each member i of cluster c weighted e^{l_i} - e^{s_c} (its exact term
 * minus its share of the cluster's estimate), and the log-sum-exp merge of
 * every partial into out and lse (lse may be NULL). */
WI_API int wi_decode_attend(const wi_decode_params *p, const void *q, const void *K, const void *V,
                     const wi_index *index, float *out, float *lse, void *workspace,
                     size_t workspace_bytes, wi_stream_t stream);

/* Size of the fixed device scratch used by wi_decode_attention_static. */
#define WI_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

/* Decode for callers that cannot allocate device memory.  The paper has no
 * counterpart: this is a packaging of wi_decode_attention for hosts that give
 * a library no allocator (runtimes that hand a plugin only pre-planned
 * buffers, or whose device-memory budget is fixed before the plugin runs).
 * Same arguments and results as wi_decode_attention, minus the workspace:
 * the call uses a scratch array of WI_STATIC_SCRATCH_BYTES that every GPU
 * loading this library holds from module load until process exit.  It calls
 * no allocator.
 *  - Returns WI_ERR_WORKSPACE when the decode needs more scratch than
 *    WI_STATIC_SCRATCH_BYTES (wi_decode_workspace_bytes tells how much).
 *  - The first call on a device looks the scratch's address up on that device
 *    (the device must be current); make that first call before any stream
 *    capture.
 *  - Every call, from any thread or stream, shares the one array: calls that
 *    overlap on the GPU race and corrupt each other's results.  Each call
 *    clears the parts that must start at zero; the rest keeps the previous
 *    call's contents.
 *  - Argument errors are found before anything is enqueued.  Device-side
 *    errors (a bounded wait that ran out) are recorded in the scratch's status
 *    word, which keeps the first error until wi_decode_static_status reads
 *    and clears it. */
WI_API int wi_decode_attention_static(const wi_decode_params *p, const void *q, const void *K,
                               const void *V, const wi_index *index, float *out, float *lse,
                               int32_t *topk_ids, wi_stream_t stream);

/* The device status of wi_decode_attention_static on the current device:
 * synchronise `stream`, then read and clear the status word of the fixed
 * scratch into *device_status (host), as wi_sync_status does for a
 * workspace.  Like the decode, its first call on a device looks the
 * scratch's address up there. */
WI_API int wi_decode_static_status(wi_stream_t stream, int *device_status);

/* Synchronise `stream`, then read and clear the device status word at the
 * start of `workspace` into *device_status (host).  Returns WI_OK, or
 * WI_ERR_CUDA if the stream reported an error (then *device_status is
 * WI_ERR_CUDA as well). */
WI_API int wi_sync_status(void *workspace, wi_stream_t stream, int *device_status);

/* Static description of a status code. */
WI_API const char *wi_status_string(int status);

/* Test hook for the device-side error path (no GPU fault involved): when bit 0
 * of `flags` is set, the next wi_decode_attention or wi_decode_attend call
 * makes every block skip the copies of its first staging tile.  The blocks'
 * bounded waits then run out after about one second, they return without
 * output, and wi_sync_status reports WI_ERR_DEVICE_TIMEOUT.
 * The request is consumed by that one call.  Returns WI_OK. */
WI_API int wi_debug_inject(int flags);

/* Library version, "major.minor.patch". */
WI_API const char *wi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* WI_H_ */
