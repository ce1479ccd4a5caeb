// C ABI of libbsa.so: argument checks, workspace sizing and dispatch to the
// launchers.  Every entry point validates its arguments before anything is
// enqueued; nothing here allocates, copies or synchronises.
#include <climits>
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace bsa {

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  static int cache[64] = {0};
  if (dev < 0 || dev >= 64) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

}  // namespace bsa

namespace {

bool shape_ok(const bsa_shape_t *s) {
  if (s == nullptr || s->cu_seqlens == nullptr) return false;
  if (s->num_seqs < 1 || s->total_tokens < 1 || s->max_seqlen < 1) return false;
  if (s->num_heads < 1 || s->num_kv_heads < 1 || s->num_heads % s->num_kv_heads != 0) return false;
  if (s->block < 1) return false;
  if (s->max_blocks != (s->max_seqlen + s->block - 1) / s->block) return false;
  const long long rows = (long long)s->num_seqs * s->num_kv_heads * s->max_blocks;
  if (rows > (1LL << 30)) return false;
  return true;
}

bool shape_supported(const bsa_shape_t *s) {
  return (s->head_dim == 64 || s->head_dim == 128) && (s->block == 64 || s->block == 128) &&
         (s->dtype == BSA_BF16 || s->dtype == BSA_FP32);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bsa_status_t launched(cudaError_t e) { return e == cudaSuccess ? BSA_OK : BSA_ERR_LAUNCH; }

// Router parameters: BSA_OK or the status the call returns.
bsa_status_t route_params_status(const bsa_route_params_t &p) {
  if (p.mode != BSA_ROUTE_TOPK && p.mode != BSA_ROUTE_THRESHOLD) return BSA_ERR_INVALID_ARG;
  if (p.k_max < 1 || p.k_max > BSA_MAX_K) return BSA_ERR_UNSUPPORTED;
  if (p.mode == BSA_ROUTE_THRESHOLD &&
      (p.k_min < 0 || !(p.tau_delta >= 0.f) || !isfinite(p.tau_delta)))
    return BSA_ERR_INVALID_ARG;
  if (p.num_global < 0 || p.num_global > BSA_MAX_GLOBAL ||
      (p.num_global > 0 && p.global_blocks == nullptr))
    return BSA_ERR_INVALID_ARG;
  if (p.window > p.k_max ||
      (p.window > 1 ? p.window : 1) + p.num_global + (p.force_sink ? 1 : 0) > p.k_max)
    return BSA_ERR_INVALID_ARG;
  return BSA_OK;
}

// A chunk over a paged cache: BSA_OK or the status the call returns.  The page
// is the routing block (64 tokens); a page's first row, (phys * H_kv + h) * 64,
// must fit in int32; a score row of N_k entries must fit the select kernel's
// shared memory.
bsa_status_t chunk_status(const bsa_shape_t *s, const bsa_kv_cache_t *c) {
  if (!shape_ok(s) || c == nullptr || c->k_cache == nullptr || c->v_cache == nullptr ||
      c->page_summ == nullptr || c->block_table == nullptr || c->prefix_lens == nullptr)
    return BSA_ERR_INVALID_ARG;
  if (s->dtype != BSA_BF16 || s->block != 64 || (s->head_dim != 64 && s->head_dim != 128))
    return BSA_ERR_UNSUPPORTED;
  if (c->max_pages_per_req < 1 || c->num_phys_pages < 1 || c->max_context_blocks < s->max_blocks ||
      c->max_context_blocks > c->max_pages_per_req)
    return BSA_ERR_INVALID_ARG;
  if ((long long)c->num_phys_pages * s->num_kv_heads * 64 > INT32_MAX ||
      (long long)s->num_seqs * s->num_kv_heads * c->max_context_blocks > (1LL << 30) ||
      !bsa::route_select_fits(c->max_context_blocks, s->head_dim))
    return BSA_ERR_UNSUPPORTED;
  if (!aligned16(c->k_cache) || !aligned16(c->v_cache) || !aligned16(c->page_summ) ||
      (c->page_sum != nullptr && !aligned16(c->page_sum)))
    return BSA_ERR_INVALID_ARG;
  return BSA_OK;
}

bool decode_ok(const bsa_decode_shape_t *s) {
  return s != nullptr && s->num_reqs >= 1 && s->num_heads >= 1 && s->num_kv_heads >= 1 &&
         s->num_heads % s->num_kv_heads == 0 && s->max_pages_per_req >= 1 &&
         s->num_phys_pages >= 1;
}

bool decode_supported(const bsa_decode_shape_t *s) {
  const int G = s->num_heads / s->num_kv_heads;
  return s->head_dim == 128 && s->page_size == 64 && s->top_k >= 1 && s->top_k <= 64 &&
         (G == 1 || G == 2 || G == 4 || G == 8) && s->num_heads <= 256 && s->num_reqs <= 65535 &&
         s->max_pages_per_req <= 16384 &&
         (long long)s->num_phys_pages * s->num_kv_heads < INT32_MAX;
}

}  // namespace

extern "C" {

int32_t bsa_version(void) { return BSA_VERSION; }

int32_t bsa_bounds_checked(void) { return BSA_BOUNDS_CHECK ? 1 : 0; }

const char *bsa_status_string(bsa_status_t s) {
  switch (s) {
    case BSA_OK: return "ok";
    case BSA_ERR_INVALID_ARG: return "invalid argument";
    case BSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case BSA_ERR_WORKSPACE: return "workspace too small";
    case BSA_ERR_LAUNCH: return "kernel launch failed";
    case BSA_ERR_INDEX_RANGE: return "index row entry outside [0, r]";
    case BSA_ERR_INDEX_ORDER: return "index row not strictly increasing";
    case BSA_ERR_COUNT: return "row count outside [0, k_max]";
    case BSA_ERR_TIMEOUT: return "bounded barrier wait timed out";
    case BSA_ERR_CACHE: return "chunk prefix off the page grid, or page outside the cache";
  }
  return "unknown status";
}

bsa_status_t bsa_selftest_wait_timeout(int32_t *dev_status, cudaStream_t stream) {
  if (dev_status == nullptr) return BSA_ERR_INVALID_ARG;
  return launched(bsa::launch_wait_timeout_selftest(dev_status, stream));
}

bsa_status_t bsa_block_summaries(const bsa_shape_t *shape, const void *K, float *C,
                                 cudaStream_t stream) {
  if (!shape_ok(shape) || K == nullptr || C == nullptr) return BSA_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return BSA_ERR_UNSUPPORTED;
  if (!aligned16(K) || !aligned16(C)) return BSA_ERR_INVALID_ARG;
  return launched(bsa::launch_block_summaries(*shape, K, C, stream));
}

size_t bsa_route_workspace_size(const bsa_shape_t *shape, const bsa_route_params_t *params) {
  if (!shape_ok(shape) || params == nullptr) return 0;
  return bsa::route_workspace_bytes(*shape, *params);
}

bsa_status_t bsa_route(const bsa_shape_t *shape, const bsa_route_params_t *params,
                       const void *Q, const float *C, int32_t *J, int32_t *counts,
                       float *scores, int32_t *dev_status, void *ws, size_t ws_bytes,
                       cudaStream_t stream) {
  if (!shape_ok(shape) || params == nullptr || Q == nullptr || C == nullptr || J == nullptr ||
      counts == nullptr)
    return BSA_ERR_INVALID_ARG;
  if (!shape_supported(shape) || !bsa::route_select_fits(shape->max_blocks, shape->head_dim))
    return BSA_ERR_UNSUPPORTED;
  const bsa_status_t ps = route_params_status(*params);
  if (ps != BSA_OK) return ps;
  if (!aligned16(Q) || !aligned16(C)) return BSA_ERR_INVALID_ARG;
  const size_t need = bsa::route_workspace_bytes(*shape, *params);
  if (ws == nullptr || ws_bytes < need) return BSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return BSA_ERR_INVALID_ARG;
  return launched(bsa::launch_route(*shape, *params, Q, C, nullptr, J, counts, scores,
                                    dev_status, ws, stream));
}

size_t bsa_worklist_workspace_size(const bsa_shape_t *shape, int32_t k_max) {
  if (!shape_ok(shape)) return 0;
  return bsa::worklist_workspace_bytes(*shape, k_max);
}

bsa_status_t bsa_build_worklist(const bsa_shape_t *shape, int32_t k_max, const int32_t *J,
                                const int32_t *counts, int32_t *row_ptr, int32_t *col_idx,
                                int32_t *work, int32_t *bucket_off, int32_t *dev_status,
                                void *ws, size_t ws_bytes, cudaStream_t stream) {
  if (!shape_ok(shape) || J == nullptr || counts == nullptr || row_ptr == nullptr ||
      col_idx == nullptr || work == nullptr || bucket_off == nullptr || dev_status == nullptr)
    return BSA_ERR_INVALID_ARG;
  if (k_max < 1 || k_max > BSA_MAX_K) return BSA_ERR_UNSUPPORTED;
  if (ws == nullptr || ws_bytes < bsa::worklist_workspace_bytes(*shape, k_max))
    return BSA_ERR_WORKSPACE;
  return launched(bsa::launch_worklist(*shape, k_max, J, counts, row_ptr, col_idx, work,
                                       bucket_off, dev_status, ws, stream));
}

bsa_status_t bsa_build_worklist_noalloc(const bsa_shape_t *shape, int32_t k_max,
                                        const int32_t *J, const int32_t *counts,
                                        int32_t *row_ptr, int32_t *col_idx, int32_t *work,
                                        int32_t *bucket_off, int32_t *dev_status,
                                        cudaStream_t stream) {
  if (!shape_ok(shape) || J == nullptr || counts == nullptr || row_ptr == nullptr ||
      col_idx == nullptr || work == nullptr || bucket_off == nullptr || dev_status == nullptr)
    return BSA_ERR_INVALID_ARG;
  if (k_max < 1 || k_max > BSA_MAX_K) return BSA_ERR_UNSUPPORTED;
  const long long rows = (long long)shape->num_seqs * shape->num_kv_heads * shape->max_blocks;
  if (rows > BSA_WORKLIST_NOALLOC_MAX_ROWS) return BSA_ERR_UNSUPPORTED;
  int32_t *scratch = nullptr;
  if (bsa::worklist_noalloc_scratch(&scratch) != cudaSuccess) return BSA_ERR_LAUNCH;
  return launched(bsa::launch_worklist(*shape, k_max, J, counts, row_ptr, col_idx, work,
                                       bucket_off, dev_status, scratch, stream));
}

size_t bsa_attention_bwd_workspace_size(const bsa_shape_t *shape) {
  if (!shape_ok(shape)) return 0;
  return bsa::attention_bwd_workspace_bytes(*shape);
}

bsa_status_t bsa_attention_bwd(const bsa_shape_t *shape, const void *Q, const void *K,
                               const void *V, const void *O, const void *dO, const float *lse,
                               const int32_t *row_ptr, const int32_t *col_idx,
                               const int32_t *work, const int32_t *bucket_off,
                               float softmax_scale, void *dQ, void *dK, void *dV,
                               int32_t *dev_status, void *ws, size_t ws_bytes,
                               cudaStream_t stream) {
  if (!shape_ok(shape) || Q == nullptr || K == nullptr || V == nullptr || O == nullptr ||
      dO == nullptr || lse == nullptr || row_ptr == nullptr || col_idx == nullptr ||
      work == nullptr || bucket_off == nullptr || dQ == nullptr || dK == nullptr ||
      dV == nullptr || dev_status == nullptr)
    return BSA_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return BSA_ERR_UNSUPPORTED;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(dO) || !aligned16(dQ))
    return BSA_ERR_INVALID_ARG;
  if (bsa::attention_bwd_tc_supported(*shape) &&
      bsa::causal_worklist_capacity(*shape) > (size_t)INT32_MAX)
    return BSA_ERR_UNSUPPORTED;
  if (ws == nullptr || ws_bytes < bsa::attention_bwd_workspace_bytes(*shape))
    return BSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return BSA_ERR_INVALID_ARG;
  const float scale =
      softmax_scale > 0.f ? softmax_scale : 1.f / sqrtf((float)shape->head_dim);
  return launched(bsa::launch_attention_bwd(*shape, Q, K, V, O, dO, lse, row_ptr, col_idx, work,
                                            bucket_off, scale, dQ, dK, dV, ws, dev_status,
                                            stream));
}

size_t bsa_causal_worklist_capacity(const bsa_shape_t *shape) {
  if (!shape_ok(shape)) return 0;
  return bsa::causal_worklist_capacity(*shape);
}

bsa_status_t bsa_build_causal_worklist(const bsa_shape_t *shape, int32_t *row_ptr,
                                       int32_t *col_idx, int32_t *work, int32_t *bucket_off,
                                       void *ws, size_t ws_bytes, cudaStream_t stream) {
  if (!shape_ok(shape) || row_ptr == nullptr || col_idx == nullptr || work == nullptr ||
      bucket_off == nullptr)
    return BSA_ERR_INVALID_ARG;
  if (bsa::causal_worklist_capacity(*shape) > (size_t)INT32_MAX) return BSA_ERR_UNSUPPORTED;
  if (ws == nullptr || ws_bytes < bsa::worklist_workspace_bytes(*shape, 1))
    return BSA_ERR_WORKSPACE;
  return launched(
      bsa::launch_causal_worklist(*shape, row_ptr, col_idx, work, bucket_off, ws, stream));
}

bsa_status_t bsa_coverage(const bsa_shape_t *shape, const float *lse_sparse,
                          const float *lse_dense, float *C, cudaStream_t stream) {
  if (!shape_ok(shape) || lse_sparse == nullptr || lse_dense == nullptr || C == nullptr)
    return BSA_ERR_INVALID_ARG;
  return launched(bsa::launch_coverage(*shape, lse_sparse, lse_dense, C, stream));
}

int32_t bsa_recall_tiles_per_seq(const bsa_shape_t *shape) {
  if (!shape_ok(shape)) return 0;
  return bsa::recall_tiles_per_seq(*shape);
}

bsa_status_t bsa_token_recall(const bsa_shape_t *shape, int32_t t_top, const void *Q,
                              const void *K, const int32_t *J, const int32_t *counts,
                              int32_t k_max, const int32_t *tiles, int32_t num_tiles,
                              int32_t *hits, int32_t *dev_status, cudaStream_t stream) {
  if (!shape_ok(shape) || Q == nullptr || K == nullptr || J == nullptr || counts == nullptr ||
      hits == nullptr || dev_status == nullptr || t_top < 1 || num_tiles < 0 ||
      (tiles == nullptr && num_tiles != 0))
    return BSA_ERR_INVALID_ARG;
  if (!shape_supported(shape) || k_max < 1 || k_max > BSA_MAX_K || shape->max_blocks > 65536 ||
      (long long)shape->num_seqs * shape->num_heads * bsa::recall_tiles_per_seq(*shape) >
          INT32_MAX)
    return BSA_ERR_UNSUPPORTED;
  if (!aligned16(Q) || !aligned16(K)) return BSA_ERR_INVALID_ARG;
  return launched(bsa::launch_token_recall(*shape, t_top, Q, K, J, counts, k_max, tiles,
                                           num_tiles, hits, dev_status, stream));
}

bsa_status_t bsa_chunk_append(const bsa_shape_t *shape, const bsa_kv_cache_t *cache,
                              const void *K, const void *V, int32_t *dev_status,
                              cudaStream_t stream) {
  const bsa_status_t cs = chunk_status(shape, cache);
  if (cs != BSA_OK) return cs;
  if (K == nullptr || V == nullptr || dev_status == nullptr) return BSA_ERR_INVALID_ARG;
  if (!aligned16(K) || !aligned16(V)) return BSA_ERR_INVALID_ARG;
  return launched(bsa::launch_chunk_append(*shape, *cache, K, V, dev_status, stream));
}

size_t bsa_route_chunk_workspace_size(const bsa_shape_t *shape, const bsa_kv_cache_t *cache,
                                      const bsa_route_params_t *params) {
  if (chunk_status(shape, cache) != BSA_OK || params == nullptr) return 0;
  return bsa::route_workspace_bytes(*shape, *params, cache);
}

bsa_status_t bsa_route_chunk(const bsa_shape_t *shape, const bsa_kv_cache_t *cache,
                             const bsa_route_params_t *params, const void *Q, int32_t *J,
                             int32_t *counts, float *scores, int32_t *dev_status, void *ws,
                             size_t ws_bytes, cudaStream_t stream) {
  const bsa_status_t cs = chunk_status(shape, cache);
  if (cs != BSA_OK) return cs;
  if (params == nullptr || Q == nullptr || J == nullptr || counts == nullptr ||
      dev_status == nullptr)
    return BSA_ERR_INVALID_ARG;
  const bsa_status_t ps = route_params_status(*params);
  if (ps != BSA_OK) return ps;
  if (!aligned16(Q)) return BSA_ERR_INVALID_ARG;
  const size_t need = bsa::route_workspace_bytes(*shape, *params, cache);
  if (ws == nullptr || ws_bytes < need) return BSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return BSA_ERR_INVALID_ARG;
  return launched(bsa::launch_route(*shape, *params, Q, nullptr, cache, J, counts, scores,
                                    dev_status, ws, stream));
}

bsa_status_t bsa_build_worklist_chunk(const bsa_shape_t *shape, const bsa_kv_cache_t *cache,
                                      int32_t k_max, const int32_t *J, const int32_t *counts,
                                      int32_t *row_ptr, int32_t *col_idx, int32_t *work,
                                      int32_t *bucket_off, int32_t *dev_status, void *ws,
                                      size_t ws_bytes, cudaStream_t stream) {
  const bsa_status_t cs = chunk_status(shape, cache);
  if (cs != BSA_OK) return cs;
  if (J == nullptr || counts == nullptr || row_ptr == nullptr || col_idx == nullptr ||
      work == nullptr || bucket_off == nullptr || dev_status == nullptr)
    return BSA_ERR_INVALID_ARG;
  if (k_max < 1 || k_max > BSA_MAX_K) return BSA_ERR_UNSUPPORTED;
  if (ws == nullptr || ws_bytes < bsa::worklist_workspace_bytes(*shape, k_max))
    return BSA_ERR_WORKSPACE;
  return launched(bsa::launch_worklist(*shape, k_max, J, counts, row_ptr, col_idx, work,
                                       bucket_off, dev_status, ws, stream, cache));
}

bsa_status_t bsa_attention_chunk(const bsa_shape_t *shape, const bsa_kv_cache_t *cache,
                                 const void *Q, const int32_t *row_ptr, const int32_t *col_idx,
                                 const int32_t *work, const int32_t *bucket_off,
                                 float softmax_scale, void *O, float *lse, int32_t *dev_status,
                                 cudaStream_t stream) {
  const bsa_status_t cs = chunk_status(shape, cache);
  if (cs != BSA_OK) return cs;
  if (Q == nullptr || row_ptr == nullptr || col_idx == nullptr || work == nullptr ||
      bucket_off == nullptr || O == nullptr || dev_status == nullptr)
    return BSA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(O)) return BSA_ERR_INVALID_ARG;
  if (!isfinite(softmax_scale)) return BSA_ERR_INVALID_ARG;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.f / sqrtf((float)shape->head_dim);
  return launched(bsa::launch_attention_chunk(*shape, *cache, Q, row_ptr, col_idx, work,
                                              bucket_off, scale, O, lse, dev_status, stream));
}

bsa_status_t bsa_attention_fwd(const bsa_shape_t *shape, const void *Q, const void *K,
                               const void *V, const int32_t *row_ptr, const int32_t *col_idx,
                               const int32_t *work, const int32_t *bucket_off,
                               float softmax_scale, void *O, float *lse, int32_t *dev_status,
                               cudaStream_t stream) {
  if (!shape_ok(shape) || Q == nullptr || K == nullptr || V == nullptr || row_ptr == nullptr ||
      col_idx == nullptr || work == nullptr || bucket_off == nullptr || O == nullptr ||
      dev_status == nullptr)
    return BSA_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return BSA_ERR_UNSUPPORTED;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O))
    return BSA_ERR_INVALID_ARG;
  if (!isfinite(softmax_scale)) return BSA_ERR_INVALID_ARG;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.f / sqrtf((float)shape->head_dim);
  if (shape->dtype == BSA_BF16)
    return launched(bsa::launch_attention_tc(*shape, Q, K, V, row_ptr, col_idx, work, bucket_off,
                                             scale, O, lse, dev_status, stream));
  return launched(bsa::launch_attention_simt_f32(*shape, Q, K, V, row_ptr, col_idx, work,
                                                 bucket_off, scale, O, lse, dev_status, stream));
}

bsa_status_t bsa_page_summaries(const bsa_decode_shape_t *shape, const void *k_cache,
                                const int32_t *block_table, const int32_t *context_lens,
                                float *page_summ, cudaStream_t stream) {
  if (!decode_ok(shape) || k_cache == nullptr || block_table == nullptr ||
      context_lens == nullptr || page_summ == nullptr)
    return BSA_ERR_INVALID_ARG;
  if (!decode_supported(shape)) return BSA_ERR_UNSUPPORTED;
  if (!aligned16(k_cache) || !aligned16(page_summ)) return BSA_ERR_INVALID_ARG;
  return launched(bsa::launch_page_summaries(*shape, k_cache, block_table, context_lens,
                                             page_summ, stream));
}

bsa_status_t bsa_page_summaries_append(const bsa_decode_shape_t *shape, const void *k_cache,
                                       const int32_t *block_table, const int32_t *context_lens,
                                       float *page_sum, float *page_summ, cudaStream_t stream) {
  if (!decode_ok(shape) || k_cache == nullptr || block_table == nullptr ||
      context_lens == nullptr || page_sum == nullptr || page_summ == nullptr)
    return BSA_ERR_INVALID_ARG;
  if (!decode_supported(shape)) return BSA_ERR_UNSUPPORTED;
  return launched(bsa::launch_page_summaries_append(*shape, k_cache, block_table, context_lens,
                                                    page_sum, page_summ, stream));
}

size_t bsa_decode_workspace_size(const bsa_decode_shape_t *shape) {
  if (!decode_ok(shape)) return 0;
  return bsa::decode_workspace_bytes(*shape);
}

bsa_status_t bsa_decode_paged(const bsa_decode_shape_t *shape, const void *q,
                              const void *k_cache, const void *v_cache,
                              const float *page_summ, const int32_t *block_table,
                              const int32_t *context_lens, float softmax_scale, void *o,
                              float *lse, int32_t *sel, int32_t *sel_counts,
                              int32_t *dev_status, void *ws, size_t ws_bytes,
                              cudaStream_t stream) {
  if (!decode_ok(shape) || q == nullptr || k_cache == nullptr || v_cache == nullptr ||
      page_summ == nullptr || block_table == nullptr || context_lens == nullptr ||
      o == nullptr || sel == nullptr || sel_counts == nullptr)
    return BSA_ERR_INVALID_ARG;
  if (!decode_supported(shape)) return BSA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(page_summ))
    return BSA_ERR_INVALID_ARG;
  if (!isfinite(softmax_scale)) return BSA_ERR_INVALID_ARG;
  if (ws == nullptr || ws_bytes < bsa::decode_workspace_bytes(*shape)) return BSA_ERR_WORKSPACE;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.f / sqrtf((float)shape->head_dim);
  return launched(bsa::launch_decode(*shape, q, k_cache, v_cache, page_summ, block_table,
                                     context_lens, scale, o, lse, sel, sel_counts, dev_status, ws,
                                     stream));
}

}  // extern "C"
