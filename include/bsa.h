/*
 * bsa.h — C ABI of libbsa.so: dynamic block-sparse attention with a mean-pooled
 * block router, for one NVIDIA GB300 (sm_103a).
 *
 * The method is the coarse-grained dynamic selection of
 * "2.1 · 粗粒度选择: 从内容分组到动态稀疏块" (PaperTrace, sparse-attention 2-1),
 * cited below as [P2], with the worklist / kernel rules of PaperTrace
 * sparse-attention 5-1 ("从索引输出到工作表", "稀疏 softmax 仍要保持数值一致"),
 * cited as [P3].
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every pointer argument is a DEVICE pointer owned by the caller, unless it
 *    is a pointer to one of the descriptor structs below (host memory, read
 *    during the call only).  The library never frees, retains or reallocates a
 *    caller buffer and keeps no pointer after the call returns.
 *  - Every call enqueues its kernels on `stream` and returns without
 *    synchronising.  Outputs are valid once the caller's stream has passed them.
 *  - Scratch memory comes from the caller through `ws` / `ws_bytes`, sized by the
 *    matching *_workspace_size() query; the library itself never allocates
 *    device memory.
 *  - Host-detectable errors (null pointers, unsupported sizes, a workspace that
 *    is too small) return a non-zero status BEFORE anything is enqueued.
 *  - Device-detected errors (malformed index rows, a bounded wait that ran out)
 *    are written to the caller's `int32_t *dev_status` (set it to 0 first);
 *    the first error wins.  The caller reads it after its own synchronisation.
 *    The outputs of a failing row are then unspecified.  No kernel traps.
 *  - Layouts are head-major and packed: Q and O are [H, T, d], K and V are
 *    [H_kv, T, d] with T = sum of the sequence lengths; sequence i owns tokens
 *    cu_seqlens[i] .. cu_seqlens[i+1]-1.  [P2] section 1 states the same tensors
 *    as B x H x n x d_h; a fixed-length batch is the case cu_seqlens[i] = i n.
 *  - Block ids in J, col_idx and sel are sequence-relative logical ids ([P2]
 *    §2.1 on packed sequences; §3.1 on logical ids mapped by a block table).
 */
#ifndef BSA_H_
#define BSA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BSA_VERSION 8

typedef enum {
  BSA_OK = 0,
  BSA_ERR_INVALID_ARG = 1,   /* null pointer, inconsistent sizes          (host) */
  BSA_ERR_UNSUPPORTED = 2,   /* head_dim / block / dtype / k_max not built (host) */
  BSA_ERR_WORKSPACE = 3,     /* ws_bytes below the *_workspace_size value  (host) */
  BSA_ERR_LAUNCH = 4,        /* a kernel launch returned an error          (host) */
  BSA_ERR_INDEX_RANGE = 16,  /* a J entry outside [0, r]                 (device) */
  BSA_ERR_INDEX_ORDER = 17,  /* a J row not strictly increasing          (device) */
  BSA_ERR_COUNT = 18,        /* counts[row] outside [0, k_max]           (device) */
  BSA_ERR_TIMEOUT = 19,      /* a bounded barrier wait ran out           (device) */
  BSA_ERR_CACHE = 20         /* chunk prefix off the page grid, context past the
                                block table, or a physical page id outside
                                [0, num_phys_pages)                      (device) */
} bsa_status_t;

typedef enum { BSA_BF16 = 0, BSA_FP32 = 1 } bsa_dtype_t;

enum { BSA_ROUTE_TOPK = 0, BSA_ROUTE_THRESHOLD = 1 };

/* Number of capacity buckets of the work list (4, 8, 16, 32, 64, 128, 256). */
#define BSA_NUM_BUCKETS 7
/* Largest supported row capacity k_max. */
#define BSA_MAX_K 256
/* Longest global block list of union routing (bsa_route_params_t.global_blocks). */
#define BSA_MAX_GLOBAL 32

/* Shape of a packed prefill batch ([P2] section 1, problem statement). */
typedef struct {
  int32_t num_seqs;          /* B                                              */
  int32_t total_tokens;      /* T = cu_seqlens[B] >= 1 (a batch without tokens
                                is rejected: BSA_ERR_INVALID_ARG); single
                                sequences may be empty (n_i = 0)             */
  int32_t max_seqlen;        /* max_i n_i >= 1                                 */
  int32_t num_heads;         /* H query heads                                  */
  int32_t num_kv_heads;      /* H_kv; H % H_kv == 0, G = H / H_kv (GQA)        */
  int32_t head_dim;          /* d_h: 64 or 128                                 */
  int32_t block;             /* b = b_q = b_k: 64 or 128                       */
  int32_t max_blocks;        /* N_q = ceil(max_seqlen / block)                 */
  bsa_dtype_t dtype;         /* element type of Q, K, V, O                     */
  const int32_t *cu_seqlens; /* device [B + 1], non-decreasing, cu[0] = 0      */
} bsa_shape_t;

/* Router parameters ([P2] §2.1 "top-k, threshold and capacity", eq.(7); union
 * routing N_u = L_u ∪ G ∪ I_u of [P2] §3.2 with the representations of §3.1: an
 * implicit local window, one short global list, and the dynamic top-k or
 * threshold choice over the history blocks neither of them keeps).
 * Row r keeps F_r = {r-window+1 .. r} ∪ {g in global_blocks : g <= r} (∪ {0} with
 * force_sink), each block once, plus the dynamic picks; k_max counts F_r, so the
 * call is rejected (BSA_ERR_INVALID_ARG) unless
 * max(1, window) + num_global + (force_sink != 0) <= k_max. */
typedef struct {
  int32_t mode;       /* BSA_ROUTE_TOPK or BSA_ROUTE_THRESHOLD                      */
  int32_t k_max;      /* row capacity of J, forced blocks included; 1 .. BSA_MAX_K  */
  int32_t k_min;      /* threshold mode: lower clamp of eq.(7)                      */
  float tau_delta;    /* threshold mode: tau_r = (max candidate score) - tau_delta   */
  int32_t force_sink; /* non-zero: block 0 is always kept (a global sink block)      */
  int32_t window;     /* local window in blocks, diagonal included; <= 1: diagonal  */
  int32_t num_global; /* entries of global_blocks, 0 .. BSA_MAX_GLOBAL               */
  const int32_t *global_blocks; /* device [num_global] sequence-relative block ids
                                   (>= 0; ids past a row are ignored by that row);
                                   NULL when num_global == 0; read during the call */
  int32_t screen;     /* BF16 scores without a score matrix (no effect on the result,
                         only on the work): the tensor cores compute q . (c_hi + c_mid)
                         of the three-part bf16 split of each fp32 summary, every score
                         carries a rigorous error bound, and only the candidates whose
                         bound meets the selection boundary are rescored exactly.
                         0 = automatic: on when a row pools G * block >= 512 query
                         rows, where the saved third of the score products outweighs
                         the per-row bound work; 1 = always; -1 = never (three parts).
                         A call that passes `scores` always computes them exactly. */
} bsa_route_params_t;

/* Paged decode shape ([P2] §2.2 decode; §3.1 paged KV cache and block table). */
typedef struct {
  int32_t num_reqs;          /* R requests, one query token each                 */
  int32_t num_heads;         /* H <= 256                                         */
  int32_t num_kv_heads;      /* H_kv, H / H_kv in {1, 2, 4, 8}                   */
  int32_t head_dim;          /* 128                                              */
  int32_t page_size;         /* tokens per page = routing block: 64              */
  int32_t max_pages_per_req; /* columns of block_table                           */
  int32_t num_phys_pages;    /* P, rows of the caches and of page_summ           */
  int32_t top_k;             /* dynamic pages per (request, KV head), 1 .. 64    */
} bsa_decode_shape_t;

/* ---------------------------------------------------------------------------
 * a1. Block summaries — [P2] §2.1 eq.(6), mean-pooled key summary
 *     c_j = (1 / r_j) sum of the keys of block j, where r_j is the number of
 *     keys the block holds (eq.(11)): a partial tail block averages its valid
 *     keys only, padding never enters ([P2] §4.1).
 *   K : [H_kv, T, d] of shape->dtype.
 *   C : [B, H_kv, N_q, d] fp32, written for every block j < ceil(n_i / b);
 *       entries of blocks past a sequence's end are set to 0.
 * ------------------------------------------------------------------------- */
bsa_status_t bsa_block_summaries(const bsa_shape_t *shape, const void *K, float *C,
                                 cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * a2 + a3. Router — [P2] §2.1 eq.(6) scores, eq.(7) selection.
 *   score g[i,h,r,j] = max over the G query heads of KV head h and over the
 *   valid query tokens t of block r of  Q[hq, t] . C[i, h, j],  for j < r
 *   (unscaled; GQA candidates are shared per KV head, [P2] §4).
 *   Forced blocks: the diagonal r always (the triangle branch of [P2] §2.1),
 *   block 0 too when force_sink; they are not dynamic candidates.
 *   TOPK: keep the forced blocks plus the best k_max - |forced| candidates.
 *   THRESHOLD: tau_r = max candidate score - tau_delta; with A the candidates
 *   scoring >= tau_r, k_r = min(k_max, max(k_min, |forced| + |A|),
 *   |forced| + |candidates|); keep forced plus the best k_r - |forced|.
 *   Ranking is (score descending, block index ascending).  Each row of J is
 *   deduplicated and sorted ascending ([P2] §1.2 eq.(1) address order).
 *   Q      : [H, T, d] of shape->dtype.     C : [B, H_kv, N_q, d] fp32.
 *   J      : [B, H_kv, N_q, k_max] int32, -1 past counts.
 *   counts : [B, H_kv, N_q] int32; 0 for rows r >= ceil(n_i / b).
 *   scores : nullable; if given, [B, H_kv, N_q, N_q] fp32 receives g for j < r
 *            (other entries unspecified) — a debugging output.
 *   ws     : at least bsa_route_workspace_size() bytes, 256-byte aligned.
 *   dev_status : see conventions.
 * ------------------------------------------------------------------------- */
size_t bsa_route_workspace_size(const bsa_shape_t *shape, const bsa_route_params_t *params);
bsa_status_t bsa_route(const bsa_shape_t *shape, const bsa_route_params_t *params,
                       const void *Q, const float *C, int32_t *J, int32_t *counts,
                       float *scores, int32_t *dev_status, void *ws, size_t ws_bytes,
                       cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * a4. Worklist — [P2] §3.1 index representations (fixed J -> CSR row_ptr /
 *     col_idx); [P3] "从索引输出到工作表" (length buckets, persistent kernel).
 *   Validates every row r < ceil(n_i / b): counts in [0, k_max]
 *   (BSA_ERR_COUNT), entries in [0, r] (BSA_ERR_INDEX_RANGE), strictly
 *   increasing (BSA_ERR_INDEX_ORDER, which also rejects duplicates: a block
 *   may enter the softmax only once, [P2] §1.2).  An empty row is replaced by
 *   its diagonal block {r} ([P3] sparse-softmax section: empty rows fall back to
 *   the self block).
 *   row_ptr    : [B * H_kv * N_q + 1] int32, CSR offsets; rows past a
 *                sequence's end are empty.
 *   col_idx    : [B * H_kv * N_q * k_max] int32 capacity, CSR block ids.
 *   work       : [B * H_kv * N_q] int32 capacity: flattened row ids
 *                (i * H_kv + h) * N_q + r of the non-empty rows: rows longer
 *                than 32 blocks first, longest first (lengths above 256 count
 *                as 256), then the others by capacity bucket, largest first;
 *                row-id order among rows of equal key.  So grouped by
 *                capacity bucket, largest first.
 *   bucket_off : [BSA_NUM_BUCKETS + 1] int32: rows of capacity 256 >> s occupy
 *                work[bucket_off[s] .. bucket_off[s+1]); bucket_off[7] is the
 *                number of rows.  A row's capacity is max(4, next power of 2
 *                of its length).
 * ------------------------------------------------------------------------- */
size_t bsa_worklist_workspace_size(const bsa_shape_t *shape, int32_t k_max);
bsa_status_t bsa_build_worklist(const bsa_shape_t *shape, int32_t k_max, const int32_t *J,
                                const int32_t *counts, int32_t *row_ptr, int32_t *col_idx,
                                int32_t *work, int32_t *bucket_off, int32_t *dev_status,
                                void *ws, size_t ws_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Worklist builder that allocates nothing.  The pages have no counterpart:
 * this is a packaging of bsa_build_worklist for callers that cannot hand the
 * library any scratch memory — for example a serving runtime that plans every
 * GPU buffer up front and only owns its inputs and outputs, or code running
 * where a cudaMalloc would synchronise the device or is not permitted.
 *
 * Arguments, results, validation and device-side errors are exactly those of
 * bsa_build_worklist, without ws / ws_bytes.  The scratch it needs (one int32
 * per row) lives in a fixed device array inside the library,
 * BSA_WORKLIST_NOALLOC_MAX_ROWS entries (1 MiB), which every GPU that loads
 * the library keeps until the process exits.
 *  - Shapes with B * H_kv * N_q > BSA_WORKLIST_NOALLOC_MAX_ROWS are rejected
 *    with BSA_ERR_UNSUPPORTED before anything is enqueued.
 *  - The first call on a device looks up that array's device address, with
 *    the caller's current device; make this first call before any stream
 *    capture.  The address is kept per device together with the CUDA context
 *    it belongs to: a call from another context of that device (after a
 *    cudaDeviceReset, or with a context of the caller's own made current)
 *    looks it up again, so such a call too must come before any capture.
 *  - Every call uses the same array.  Calls ordered on one stream are safe;
 *    calls whose kernels may overlap on the GPU (different streams, or host
 *    threads issuing to one device without ordering) race on it and may all
 *    produce wrong worklists.  Each call rewrites every entry it reads, so
 *    nothing left by an earlier call needs clearing.
 *  - It never calls cudaMalloc, cudaFree or any other allocating routine.
 * ------------------------------------------------------------------------- */
#define BSA_WORKLIST_NOALLOC_MAX_ROWS (1 << 18)
bsa_status_t bsa_build_worklist_noalloc(const bsa_shape_t *shape, int32_t k_max,
                                        const int32_t *J, const int32_t *counts,
                                        int32_t *row_ptr, int32_t *col_idx, int32_t *work,
                                        int32_t *bucket_off, int32_t *dev_status,
                                        cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * a5. Sparse attention forward — [P2] §1.2 eqs.(1)-(5): for each row listed
 *   in `work` and every query head of its group, exact S = Q_r K_j^T * scale
 *   on the selected tiles only (eq.(2)), the causal mask s <= t inside the
 *   diagonal tile and the tail mask s < n_i applied before the softmax, tiles
 *   merged with the online-softmax recurrences (3)-(5), O = u / l.
 *   BF16 runs on the tensor cores (tcgen05, TMEM accumulators); FP32 is a
 *   SIMT correctness path.
 *   softmax_scale : <= 0 selects 1 / sqrt(d).
 *   O   : [H, T, d] of shape->dtype; rows of valid query tokens are written.
 *   lse : [H, T] fp32 natural-log logsumexp of the scaled scores (nullable).
 *   row_ptr / col_idx / work / bucket_off : as produced by bsa_build_worklist.
 * ------------------------------------------------------------------------- */
bsa_status_t bsa_attention_fwd(const bsa_shape_t *shape, const void *Q, const void *K,
                               const void *V, const int32_t *row_ptr, const int32_t *col_idx,
                               const int32_t *work, const int32_t *bucket_off,
                               float softmax_scale, void *O, float *lse, int32_t *dev_status,
                               cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Page summaries for decode — [P2] §3.1 "block summaries are cache state",
 *   eq.(11): the mean of the keys each page holds.  For request rho and logical
 *   page p < ceil(len / page_size), page_summ[block_table[rho][p], h, :] =
 *   mean of the valid keys of that page.  Pages no request references are
 *   left untouched.
 *   k_cache     : [P, H_kv, page_size, d] bf16.
 *   block_table : [R, max_pages_per_req] int32 physical page ids; an id outside
 *                 [0, P) is skipped (nothing is read or written through it).
 *   context_lens: [R] int32, 1 .. max_pages_per_req * page_size (pages past the
 *                 block table are not summarised; 0 skips a request).
 *   page_summ   : [P, H_kv, d] fp32.
 * ------------------------------------------------------------------------- */
bsa_status_t bsa_page_summaries(const bsa_decode_shape_t *shape, const void *k_cache,
                                const int32_t *block_table, const int32_t *context_lens,
                                float *page_summ, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Streaming page summaries — [P2] §3.1 eq.(11): the summary of the block still
 *   being filled is cache state kept as a vector sum and a count,
 *   s <- s + k_t, c = s / r.  Call after every request appended one key (already
 *   written to k_cache at position context_lens[rho] - 1): the page holding it
 *   gets s <- s + k (s <- k when the key opens the page, r = 1) and
 *   c = s / r, r = the page's key count.  Other pages are untouched.
 *   page_sum  : [P, H_kv, d] fp32 running sums (the state; a page's sum must be
 *               valid for its keys before the append, e.g. built by appending
 *               from an empty page);
 *   page_summ : [P, H_kv, d] fp32 means, as bsa_page_summaries writes them.
 *   context_lens : [R] int32, counts after the append (>= 1; 0 skips a request,
 *               and so does a count past max_pages_per_req * page_size or a page id
 *               outside [0, P)).
 * ------------------------------------------------------------------------- */
bsa_status_t bsa_page_summaries_append(const bsa_decode_shape_t *shape, const void *k_cache,
                                       const int32_t *block_table, const int32_t *context_lens,
                                       float *page_sum, float *page_summ, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * a6. Paged sparse decode — [P2] §2.2 (decode reads the summaries, O(N_k d_r),
 *   then only the selected K/V) and §3.1 (the router emits logical page ids
 *   that the block table maps to physical pages at attention time).
 *   For request rho (L = ceil(len / page_size) logical pages) and KV head h:
 *   pages 0 .. L-2 are scored by max over the group's query heads of
 *   q . page_summ[phys(p), h]; the best top_k (score desc, index asc) plus the
 *   last page L-1 are kept, ascending, in sel; the softmax (scale, default
 *   1/sqrt(d)) runs over the valid tokens of the kept pages.
 *   q        : [R, H, d] bf16.          k_cache, v_cache : [P, H_kv, page, d] bf16;
 *              slots of a request's last page past its length must hold finite
 *              values (zeros, as bsa_chunk_append leaves them): they are masked
 *              out of the softmax but still meet P = 0 in the P.V product, where a
 *              NaN or Inf would reach the output.
 *   page_summ: [P, H_kv, d] fp32.       block_table, context_lens as above.
 *   o        : [R, H, d] bf16.          lse : [R, H] fp32 (nullable).
 *   sel      : [R, H_kv, top_k + 1] int32 logical pages, -1 padded.
 *   sel_counts : [R, H_kv] int32.
 *   ws       : at least bsa_decode_workspace_size() bytes, 256-byte aligned.
 *   num_reqs <= 65535 (else BSA_ERR_UNSUPPORTED).
 *   Lengths and page ids are checked on the device before they index anything:
 *   - context_lens[rho] == 0 is an idle slot (a padded batch): sel row all -1,
 *     count 0, o = 0, lse = -inf, no error.
 *   - a length < 0 or > max_pages_per_req * page_size gives the same empty result
 *     and sets BSA_ERR_CACHE in dev_status (nullable: then not reported).
 *   - a block_table entry outside [0, num_phys_pages) sets BSA_ERR_CACHE; that
 *     page scores -inf, and where it is still kept (a request with at most top_k
 *     scored pages) the attention reads zeros in its place.  Other requests are
 *     unaffected.
 * ------------------------------------------------------------------------- */
size_t bsa_decode_workspace_size(const bsa_decode_shape_t *shape);
bsa_status_t bsa_decode_paged(const bsa_decode_shape_t *shape, const void *q,
                              const void *k_cache, const void *v_cache,
                              const float *page_summ, const int32_t *block_table,
                              const int32_t *context_lens, float softmax_scale, void *o,
                              float *lse, int32_t *sel, int32_t *sel_counts,
                              int32_t *dev_status, void *ws, size_t ws_bytes,
                              cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Backward of the sparse attention, for training ([P2] §2.2 training paragraph:
 *   keep the index and the softmax statistics; [P3] verification of forward output
 *   and gradients against the dense-then-mask reference).  Given the forward's
 *   worklist (same J), its output O and lse, and the upstream gradient dO, returns
 *   dQ, dK, dV of the forward of bsa_attention_fwd (same masks, same scale: <= 0
 *   means 1/sqrt(d)).  P is recomputed from lse; nothing is re-routed.  dK and dV
 *   sum the contributions of every query row and query head that selected a key
 *   block (GQA).
 *   BF16 with head_dim 128 runs on the tensor cores (tcgen05, fp32 accumulators in
 *   TMEM): a query-major pass for dQ over the worklist and a key-major pass for dK
 *   and dV over its transpose (built in the workspace), each gradient element
 *   written once, a key block's rows summed in ascending order (the result does
 *   not change between runs).  Other shapes (fp32, head_dim 64) run an FP32 SIMT
 *   path, whose dK / dV are summed with fp32 atomics.
 *   Q, dQ, O, dO : [H, T, d];  K, V, dK, dV : [H_kv, T, d];  element type shape->dtype.
 *   lse          : [H, T] fp32 from the forward.
 *   dev_status   : see conventions (a bounded wait that ran out).
 *   ws           : at least bsa_attention_bwd_workspace_size() bytes, 256-aligned;
 *                  contents are overwritten.
 * ------------------------------------------------------------------------- */
size_t bsa_attention_bwd_workspace_size(const bsa_shape_t *shape);
bsa_status_t bsa_attention_bwd(const bsa_shape_t *shape, const void *Q, const void *K,
                               const void *V, const void *O, const void *dO, const float *lse,
                               const int32_t *row_ptr, const int32_t *col_idx,
                               const int32_t *work, const int32_t *bucket_off,
                               float softmax_scale, void *dQ, void *dK, void *dV,
                               int32_t *dev_status, void *ws, size_t ws_bytes,
                               cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Density-1 worklist — every causal block: row r of a sequence holds blocks
 *   0 .. r ([P2] §3.1 validation, the dense side of the second layer; §2.2 the
 *   dense causal baseline).  Same outputs as bsa_build_worklist, fed to
 *   bsa_attention_fwd it computes dense causal attention with the same kernel:
 *   the reference for the coverage below and for density-1 timing.  No J and no
 *   row-length limit (rows longer than BSA_MAX_K go to the longest bucket).
 *   col_idx  : at least bsa_causal_worklist_capacity() int32 entries (an upper
 *              bound: B * H_kv * N_q (N_q + 1) / 2); larger than INT32_MAX entries:
 *              BSA_ERR_UNSUPPORTED.
 *   ws       : at least bsa_worklist_workspace_size(shape, 1) bytes.
 * ------------------------------------------------------------------------- */
size_t bsa_causal_worklist_capacity(const bsa_shape_t *shape);
bsa_status_t bsa_build_causal_worklist(const bsa_shape_t *shape, int32_t *row_ptr,
                                       int32_t *col_idx, int32_t *work, int32_t *bucket_off,
                                       void *ws, size_t ws_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Coverage C_i of [P2] §3.1 eq.(10): the dense softmax mass that the selected
 *   blocks hold, per query head and token, computed as
 *   C = exp(lse_sparse - lse_dense) from the lse of bsa_attention_fwd on the
 *   routed worklist and on the density-1 worklist (same scale).
 *   lse_sparse, lse_dense : [H, T] fp32;   C : [H, T] fp32, in (0, 1] up to rounding.
 * ------------------------------------------------------------------------- */
bsa_status_t bsa_coverage(const bsa_shape_t *shape, const float *lse_sparse,
                          const float *lse_dense, float *C, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Token recall against the dense top-t teacher — [P2] §1.1, the paragraph on
 *   recall@k: with G_i the dense attention's top-t keys of query i and N(i) its
 *   candidate keys, token recall = |G_i ∩ N(i)| / |G_i|, to be reported beside
 *   the physical tile budget.  For query token t (sequence position) of query head
 *   hq: G_i = the min(t_top, t + 1) visible keys s <= t of the same sequence with
 *   the largest unscaled score Q[hq].K[hq / G, s], ranked by (score descending,
 *   index ascending), scores in fp32 from the stored elements; N(i) = the visible
 *   keys whose block is in the J row (i, hq / G, t / block), an empty row keeping
 *   its diagonal.  A measurement of the router (fp32 SIMT, several passes over
 *   each query's keys), not part of the hot path.
 *   Queries are taken in tiles of 64 consecutive sequence positions of one query
 *   head: tile id (i * H + hq) * bsa_recall_tiles_per_seq(shape) + c covers
 *   positions 64 c .. 64 c + 63 of sequence i.
 *   tiles     : device [num_tiles] tile ids, or NULL for every tile of the batch
 *               (num_tiles then 0); an id outside the batch sets
 *               BSA_ERR_INDEX_RANGE; tiles past a sequence's end are skipped.
 *   J, counts : as bsa_route writes them (k_max = row capacity).
 *   hits      : [H, T] int32; |G_i ∩ N(i)| written for the queries of the listed
 *               tiles, other entries untouched.  |G_i| = min(t_top, t + 1).
 *   Needs max_blocks <= 65536.
 * ------------------------------------------------------------------------- */
int32_t bsa_recall_tiles_per_seq(const bsa_shape_t *shape);
bsa_status_t bsa_token_recall(const bsa_shape_t *shape, int32_t t_top, const void *Q,
                              const void *K, const int32_t *J, const int32_t *counts,
                              int32_t k_max, const int32_t *tiles, int32_t num_tiles,
                              int32_t *hits, int32_t *dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Chunked prefill over a paged KV cache — [P2] §3.1 (block summaries are cache
 *   state kept beside the KV cache and updated as keys arrive, eq.(11); the
 *   router emits logical block ids that a block table maps to physical pages)
 *   and §2.2 (routing a query block needs only the summaries of its history).
 *   A prompt is processed chunk by chunk: each chunk's keys and values are
 *   appended to the cache with their page summaries (bsa_chunk_append), its query
 *   blocks are routed against the summaries of every earlier block, cached or in
 *   the chunk (bsa_route_chunk), and the selected pages are attended
 *   (bsa_build_worklist_chunk, bsa_attention_chunk).  For every token of the
 *   chunk the result is that of a single-pass prefill of the whole prompt.
 *
 *   Conventions of the calls below:
 *   - `shape` describes the CHUNK: cu_seqlens over the chunk's packed tokens,
 *     n_i = tokens sequence i adds (0 allowed), max_blocks = ceil(max n_i / 64);
 *     dtype BSA_BF16, block 64 (the page size), head_dim 64 or 128.
 *   - prefix_i = cache->prefix_lens[i] tokens are already cached.  When n_i > 0
 *     it must be a multiple of 64, so chunk query block q of sequence i is
 *     logical block r = prefix_i / 64 + q, and ceil((prefix_i + n_i) / 64) <=
 *     max_context_blocks; a sequence breaking either rule contributes no rows
 *     and sets BSA_ERR_CACHE in dev_status.  A sequence with n_i = 0 is idle
 *     (its prefix may end anywhere, e.g. a finished prompt).
 *   - J, counts, row_ptr and work are indexed by (i, h, q) like a prefill of the
 *     chunk; J holds logical block ids 0 .. r (routing, forced blocks and union
 *     parameters exactly as bsa_route with r the logical block).
 *   - Page slots past a sequence's context must hold finite values; the append
 *     zeroes them in the pages it writes (see bsa_decode_paged on why).
 * ------------------------------------------------------------------------- */
typedef struct {
  void *k_cache;               /* [P, H_kv, 64, d] bf16                                */
  void *v_cache;               /* [P, H_kv, 64, d] bf16                                */
  float *page_summ;            /* [P, H_kv, d] fp32 page means c = s / r_p (eq.(11))   */
  float *page_sum;             /* nullable; [P, H_kv, d] fp32 running sums s (eq.(11)),
                                  the state bsa_page_summaries_append continues from   */
  const int32_t *block_table;  /* [B, max_pages_per_req] physical page of each logical
                                  block of each sequence                              */
  const int32_t *prefix_lens;  /* [B] tokens cached before this chunk                 */
  int32_t max_pages_per_req;   /* columns of block_table                              */
  int32_t num_phys_pages;      /* P                                                   */
  int32_t max_context_blocks;  /* N_k: >= max_i ceil((prefix_i + n_i) / 64), and
                                  max_blocks <= N_k <= max_pages_per_req              */
} bsa_kv_cache_t;

/* Append the chunk's keys and values to their pages and summarise those pages:
 *   key/value t of sequence i goes to page block_table[i][(prefix_i + t) / 64],
 *   slot t % 64; slots of the chunk's last page past its end are zeroed.  For
 *   every page the chunk wrote, page_summ = mean of its keys (and page_sum = their
 *   sum, when given).  Physical ids outside [0, P) are skipped (BSA_ERR_CACHE).
 *   K, V : [H_kv, T, d] bf16, the chunk packed as in a prefill.               */
bsa_status_t bsa_chunk_append(const bsa_shape_t *shape, const bsa_kv_cache_t *cache,
                              const void *K, const void *V, int32_t *dev_status,
                              cudaStream_t stream);

/* Route the chunk's query blocks against the cached page summaries (eq.(6),
 *   eq.(7)): score g[i,h,q,j] = max over the group's query heads and the valid
 *   tokens of chunk block q of Q . page_summ[block_table[i][j], h] for j < r.
 *   Q      : [H, T, d] bf16 (the chunk).  J, counts : as bsa_route, rows (i, h, q).
 *   scores : nullable; [B, H_kv, N_q, N_k] fp32 receives g for j < r.
 *   ws     : bsa_route_chunk_workspace_size() bytes, 256-byte aligned.        */
size_t bsa_route_chunk_workspace_size(const bsa_shape_t *shape, const bsa_kv_cache_t *cache,
                                      const bsa_route_params_t *params);
bsa_status_t bsa_route_chunk(const bsa_shape_t *shape, const bsa_kv_cache_t *cache,
                             const bsa_route_params_t *params, const void *Q, int32_t *J,
                             int32_t *counts, float *scores, int32_t *dev_status, void *ws,
                             size_t ws_bytes, cudaStream_t stream);

/* Worklist of a chunk: bsa_build_worklist with row (i, h, q) validated against
 *   its logical block r (entries in [0, r]; an empty row becomes {r}).
 *   ws : bsa_worklist_workspace_size(shape, k_max) bytes.                     */
bsa_status_t bsa_build_worklist_chunk(const bsa_shape_t *shape, const bsa_kv_cache_t *cache,
                                      int32_t k_max, const int32_t *J, const int32_t *counts,
                                      int32_t *row_ptr, int32_t *col_idx, int32_t *work,
                                      int32_t *bucket_off, int32_t *dev_status, void *ws,
                                      size_t ws_bytes, cudaStream_t stream);

/* Sparse attention of the chunk's queries over the selected pages (eqs.(1)-(5)
 *   as bsa_attention_fwd; the causal mask inside the diagonal block r).  K and V
 *   tiles are read from the cache pages the block table names.
 *   Q, O : [H, T, d] bf16 (the chunk);  lse : [H, T] fp32 (nullable).         */
bsa_status_t bsa_attention_chunk(const bsa_shape_t *shape, const bsa_kv_cache_t *cache,
                                 const void *Q, const int32_t *row_ptr, const int32_t *col_idx,
                                 const int32_t *work, const int32_t *bucket_off,
                                 float softmax_scale, void *O, float *lse, int32_t *dev_status,
                                 cudaStream_t stream);

/* Self-test of the failure path: one small kernel waits, with the kernels' own
 * bounded barrier wait and a budget of about 10 ms, on a barrier that nothing
 * arrives at.  After the caller's synchronisation *dev_status holds
 * BSA_ERR_TIMEOUT (if it was 0) and the context remains usable.  Touches no other
 * state. */
bsa_status_t bsa_selftest_wait_timeout(int32_t *dev_status, cudaStream_t stream);

/* Human-readable name of a status code (static storage). */
const char *bsa_status_string(bsa_status_t status);

/* BSA_VERSION of the built library. */
int32_t bsa_version(void);

/* 1 in the bounds-checked build (libbsa_bounds.so, compiled with
 * -DBSA_BOUNDS_CHECK=1), 0 in the default build.  The bounds-checked build
 * range-checks, on the device, every index its kernels read from a caller-visible
 * table before using it to address memory: worklist col_idx entries against
 * [0, r] of their row (bsa_attention_fwd, bsa_attention_bwd, bsa_attention_chunk),
 * chunk block-table entries against [0, num_phys_pages), and decode selections
 * against [0, max_pages_per_req).  An index outside its range sets
 * BSA_ERR_INDEX_RANGE in dev_status and is clamped into the range, so the call
 * completes without touching memory outside its buffers (its outputs are then
 * meaningless).  The default build trusts these tables, which the library's own
 * validated kernels produce.  Same ABI and results otherwise. */
int32_t bsa_bounds_checked(void);

#ifdef __cplusplus
}
#endif
#endif /* BSA_H_ */
