// Host-side launchers implemented in the kernel translation units and called by
// the argument-checking entry points in api.cu.  Every launcher enqueues on the
// given stream and returns the launch error, if any.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/bsa.h"

namespace bsa {

int num_sms();

// Launch `kernel` with programmatic stream serialization: it may begin while the
// previous kernel on the stream is still running, and must call grid_dep_wait()
// before reading that kernel's outputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// 3-D bf16 TMA descriptor (dims d0 innermost .. d2, dense strides) with a
// 128-byte swizzle and box b0 x b1 x b2 (tmap.cu).
bool make_tmap_3d_bf16(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint32_t b0, uint32_t b1, uint32_t b2);

// a2 on the tensor cores (route_tc.cu): fp32 scores from bf16 Q and the three-way
// bf16 split of the fp32 summaries; writes S[row][j] for j < r.  screen: two of the
// three parts (q . (c_hi + c_mid)), and the norms that bound the rest.
// cache != nullptr: a chunked prefill, summaries gathered from the paged cache.
size_t route_tc_workspace_bytes(const bsa_shape_t &s, const bsa_kv_cache_t *cache);
cudaError_t launch_route_scores_tc(const bsa_shape_t &s, const void *Q, const float *C,
                                   const bsa_kv_cache_t *cache, float *S, bool screen, void *ws,
                                   int32_t *qlen, int32_t *dev_status, cudaStream_t st);
// Where the screen's inputs live in the route workspace: the split planes
// [3, c3_rows, d] bf16, |c| and |c - c_hi - c_mid| per summary row, and the largest
// query norm of each router row.
struct RouteScreen {
  const uint16_t *C3;
  const float *cn, *rn, *Qn;
  size_t c3_rows;
};
RouteScreen route_tc_screen(const bsa_shape_t &s, const bsa_kv_cache_t *cache, void *ws);

// a1 and the decode page summaries (summaries.cu)
cudaError_t launch_block_summaries(const bsa_shape_t &s, const void *K, float *C,
                                   cudaStream_t st);
cudaError_t launch_page_summaries_append(const bsa_decode_shape_t &s, const void *k_cache,
                                         const int32_t *block_table,
                                         const int32_t *context_lens, float *page_sum,
                                         float *page_summ, cudaStream_t st);
cudaError_t launch_page_summaries(const bsa_decode_shape_t &s, const void *k_cache,
                                  const int32_t *block_table, const int32_t *context_lens,
                                  float *page_summ, cudaStream_t st);
cudaError_t launch_chunk_append(const bsa_shape_t &s, const bsa_kv_cache_t &cache, const void *K,
                                const void *V, int32_t *dev_status, cudaStream_t st);

// a2 + a3 (route.cu)
// cache != nullptr: a chunked prefill (C unused, summaries from the cache).
size_t route_workspace_bytes(const bsa_shape_t &s, const bsa_route_params_t &p,
                             const bsa_kv_cache_t *cache = nullptr);
// Whether a score row of Nk entries fits the selection kernel's shared memory.
bool route_select_fits(int Nk, int d);
cudaError_t launch_route(const bsa_shape_t &s, const bsa_route_params_t &p, const void *Q,
                         const float *C, const bsa_kv_cache_t *cache, int32_t *J,
                         int32_t *counts, float *scores, int32_t *dev_status, void *ws,
                         cudaStream_t st);

// a4 (worklist.cu)
size_t worklist_workspace_bytes(const bsa_shape_t &s, int32_t k_max);
cudaError_t launch_worklist(const bsa_shape_t &s, int32_t k_max, const int32_t *J,
                            const int32_t *counts, int32_t *row_ptr, int32_t *col_idx,
                            int32_t *work, int32_t *bucket_off, int32_t *dev_status, void *ws,
                            cudaStream_t st, const bsa_kv_cache_t *cache = nullptr);
// Row lengths (>= 0; a negative entry counts as 1) -> CSR offsets, and the rows of
// non-zero length, those above 128 in exact order of length, the others grouped by
// capacity bucket, longest first (worklist.cu).
cudaError_t launch_length_scan(const int32_t *len, int32_t *row_ptr, int32_t *work,
                               int32_t *bucket_off, int nrows, cudaStream_t st);
// Tensor-core backward, BF16 with head_dim 128 (attn_bwd_tc.cu): workspace of
// its key-major index, and the launch given D = rowsum(dO * O) [H, T].
bool attention_bwd_tc_supported(const bsa_shape_t &s);
size_t attention_bwd_tc_index_bytes(const bsa_shape_t &s);
cudaError_t launch_attention_bwd_tc(const bsa_shape_t &s, const void *Q, const void *K,
                                    const void *V, const void *dO, const float *lse,
                                    const float *Dv, const int32_t *row_ptr,
                                    const int32_t *col_idx, const int32_t *work,
                                    const int32_t *bucket_off, float scale, void *dQ, void *dK,
                                    void *dV, void *ws, int32_t *dev_status, cudaStream_t st);
// Bounded-wait self-test (selftest.cu).
cudaError_t launch_wait_timeout_selftest(int32_t *dev_status, cudaStream_t st);
// Backward of the sparse attention (attn_bwd.cu).
size_t attention_bwd_workspace_bytes(const bsa_shape_t &s);
cudaError_t launch_attention_bwd(const bsa_shape_t &s, const void *Q, const void *K,
                                 const void *V, const void *O, const void *dO, const float *lse,
                                 const int32_t *row_ptr, const int32_t *col_idx,
                                 const int32_t *work, const int32_t *bucket_off, float scale,
                                 void *dQ, void *dK, void *dV, void *ws, int32_t *dev_status,
                                 cudaStream_t st);

// Density-1 worklist (every causal block) and coverage of eq.(10) (worklist.cu).
size_t causal_worklist_capacity(const bsa_shape_t &s);
cudaError_t launch_causal_worklist(const bsa_shape_t &s, int32_t *row_ptr, int32_t *col_idx,
                                   int32_t *work, int32_t *bucket_off, void *ws, cudaStream_t st);
cudaError_t launch_coverage(const bsa_shape_t &s, const float *lse_sparse, const float *lse_dense,
                            float *C, cudaStream_t st);
// Device address of the fixed scratch array used by bsa_build_worklist_noalloc.
cudaError_t worklist_noalloc_scratch(int32_t **out);

// Token recall against the dense top-t teacher (recall.cu).
int recall_tiles_per_seq(const bsa_shape_t &s);
cudaError_t launch_token_recall(const bsa_shape_t &s, int32_t t_top, const void *Q,
                                const void *K, const int32_t *J, const int32_t *counts,
                                int32_t k_max, const int32_t *tiles, int32_t num_tiles,
                                int32_t *hits, int32_t *dev_status, cudaStream_t st);

// a5, tensor-core BF16 path (attn_tc.cu) and SIMT FP32 path (attn_simt.cu)
cudaError_t launch_attention_tc(const bsa_shape_t &s, const void *Q, const void *K,
                                const void *V, const int32_t *row_ptr, const int32_t *col_idx,
                                const int32_t *work, const int32_t *bucket_off, float scale,
                                void *O, float *lse, int32_t *dev_status, cudaStream_t st);
// Chunked prefill: the chunk's queries over the selected pages of the cache.
cudaError_t launch_attention_chunk(const bsa_shape_t &s, const bsa_kv_cache_t &cache,
                                   const void *Q, const int32_t *row_ptr, const int32_t *col_idx,
                                   const int32_t *work, const int32_t *bucket_off, float scale,
                                   void *O, float *lse, int32_t *dev_status, cudaStream_t st);
cudaError_t launch_attention_simt_f32(const bsa_shape_t &s, const void *Q, const void *K,
                                      const void *V, const int32_t *row_ptr,
                                      const int32_t *col_idx, const int32_t *work,
                                      const int32_t *bucket_off, float scale, void *O,
                                      float *lse, int32_t *status, cudaStream_t st);

// a6 (decode.cu)
size_t decode_workspace_bytes(const bsa_decode_shape_t &s);
cudaError_t launch_decode(const bsa_decode_shape_t &s, const void *q, const void *k_cache,
                          const void *v_cache, const float *page_summ,
                          const int32_t *block_table, const int32_t *context_lens, float scale,
                          void *o, float *lse, int32_t *sel, int32_t *sel_counts,
                          int32_t *dev_status, void *ws, cudaStream_t st);

}  // namespace bsa
