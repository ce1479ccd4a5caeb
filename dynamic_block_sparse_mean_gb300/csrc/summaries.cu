// a1: mean-pooled block summaries ("2.1 · 粗粒度选择" §2.1 eq.(6), with the
// valid-key divisor r_j of eq.(11)), and the same mean over the pages of a paged
// KV cache.  Both are HBM-bound: every key is read once with 16-byte loads and
// each CTA writes one d-vector of fp32.
#include "common.cuh"
#include "kernels.h"

namespace bsa {
namespace {

constexpr int kThreads = 256;

template <typename T>
struct Vec16;
template <>
struct Vec16<uint16_t> {  // 8 bf16
  static constexpr int kElems = 8;
  BSA_DEV static void add(const uint4 &v, float *acc) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc[2 * e] += __uint_as_float(w[e] << 16);
      acc[2 * e + 1] += __uint_as_float(w[e] & 0xFFFF0000u);
    }
  }
};
template <>
struct Vec16<float> {  // 4 fp32
  static constexpr int kElems = 4;
  BSA_DEV static void add(const uint4 &v, float *acc) {
    acc[0] += __uint_as_float(v.x);
    acc[1] += __uint_as_float(v.y);
    acc[2] += __uint_as_float(v.z);
    acc[3] += __uint_as_float(v.w);
  }
};

// Mean over `nrows` rows (row stride `stride` elements) of a d-wide slab; the
// CTA's threads split rows x 16-byte vectors, then reduce through shared memory.
template <typename T>
BSA_DEV void block_mean(const T *__restrict__ base, int nrows, long long stride, int d,
                        float *__restrict__ out, float *red) {
  constexpr int E = Vec16<T>::kElems;
  const int vecs = d / E;             // 16-byte vectors per row
  const int rgroups = kThreads / vecs;
  const int vec = threadIdx.x % vecs;
  const int rg = threadIdx.x / vecs;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int row = rg; row < nrows; row += rgroups) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(base + row * stride) + vec);
    Vec16<T>::add(v, acc);
  }
#pragma unroll
  for (int e = 0; e < E; ++e) red[rg * d + vec * E + e] = acc[e];
  __syncthreads();
  for (int c = threadIdx.x; c < d; c += kThreads) {
    float s = 0.f;
    for (int g = 0; g < rgroups; ++g) s += red[g * d + c];
    out[c] = nrows > 0 ? s / (float)nrows : 0.f;
  }
}

// grid (N_q, B, H_kv): one CTA per (block j, sequence i, KV head h).
template <typename T>
__global__ void __launch_bounds__(kThreads) block_summaries_kernel(
    const T *__restrict__ K, const int32_t *__restrict__ cu, float *__restrict__ C, int T_tok,
    int Nq, int Hk, int d, int b) {
  extern __shared__ float red[];
  grid_dep_wait();  // K may come from the previous launch
  const int j = blockIdx.x, i = blockIdx.y, h = blockIdx.z;
  const int s0 = cu[i], n = cu[i + 1] - s0;
  const int lo = j * b;
  const int nrows = max(0, min(b, n - lo));
  float *out = C + (((size_t)i * Hk + h) * Nq + j) * d;
  const T *base = K + ((size_t)h * T_tok + s0 + lo) * d;
  block_mean<T>(base, nrows, d, d, out, red);
  grid_dep_launch();
}

// grid (max_pages_per_req, R, H_kv): one CTA per (logical page p, request, KV head).
// A page id outside [0, P) is skipped (nothing is read or written through it).
__global__ void __launch_bounds__(kThreads) page_summaries_kernel(
    const uint16_t *__restrict__ kc, const int32_t *__restrict__ bt,
    const int32_t *__restrict__ lens, float *__restrict__ ps, int max_pages, int Hk, int page,
    int d, int P) {
  extern __shared__ float red[];
  const int p = blockIdx.x, rho = blockIdx.y, h = blockIdx.z;
  const int n = lens[rho];
  const int lo = p * page;
  if (lo >= n) return;
  const int nrows = min(page, n - lo);
  const int phys = bt[(size_t)rho * max_pages + p];
  if (phys < 0 || phys >= P) return;
  const uint16_t *base = kc + (((size_t)phys * Hk + h) * page) * d;
  block_mean<uint16_t>(base, nrows, d, d, ps + ((size_t)phys * Hk + h) * d, red);
}

// grid (R, H_kv), d threads: eq.(11) for the key each request just appended.  A
// length past the block table, or a page id outside [0, P), skips the request.
__global__ void page_summaries_append_kernel(const uint16_t *__restrict__ kc,
                                             const int32_t *__restrict__ bt,
                                             const int32_t *__restrict__ lens,
                                             float *__restrict__ psum, float *__restrict__ ps,
                                             int max_pages, int Hk, int page, int d, int P) {
  const int rho = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  const int n = lens[rho];  // keys after the append; the new one sits at n - 1
  if (n < 1 || n > max_pages * page || c >= d) return;
  const int p = (n - 1) / page, slot = (n - 1) % page;
  const int phys = bt[(size_t)rho * max_pages + p];
  if (phys < 0 || phys >= P) return;
  const size_t row = (size_t)phys * Hk + h;
  const float k = bf16_to_f32(kc[(row * page + slot) * d + c]);
  const float sum = slot == 0 ? k : psum[row * d + c] + k;  // s <- s + k_t (a new page starts at k)
  psum[row * d + c] = sum;
  ps[row * d + c] = sum / (float)(slot + 1);                 // c = s / r
}

// Chunked prefill, grid (N_q, B, H_kv): one CTA per (chunk block q, sequence i,
// KV head h) copies the block's keys and values into its page — block q of the
// chunk is logical block prefix_i / 64 + q — zeroing the page slots past the
// chunk's end, and writes the page's key mean and sum ("2.1 · 粗粒度选择" §3.1,
// eq.(11): a summary is the running sum of the page's keys over their count).
__global__ void __launch_bounds__(kThreads) chunk_append_kernel(
    const uint16_t *__restrict__ K, const uint16_t *__restrict__ V,
    const int32_t *__restrict__ cu, const int32_t *__restrict__ prefix,
    const int32_t *__restrict__ bt, uint16_t *__restrict__ kc, uint16_t *__restrict__ vc,
    float *__restrict__ ps, float *__restrict__ psum, int32_t *status, int T_tok, int Hk, int d,
    int maxp, int P, int Nk) {
  extern __shared__ float red[];
  grid_dep_wait();  // K and V may come from the previous launch
  const int q = blockIdx.x, i = blockIdx.y, h = blockIdx.z;
  const int s0 = cu[i], n = cu[i + 1] - s0;
  const int lo = q * 64;
  if (lo >= n) return;
  const int pre = prefix[i];
  const int phys = chunk_ok(pre, n, 64, Nk) ? bt[(size_t)i * maxp + pre / 64 + q] : -1;
  if (phys < 0 || phys >= P) {
    if (threadIdx.x == 0) set_status(status, BSA_ERR_CACHE);
    return;
  }
  const int nrows = min(64, n - lo);
  const size_t src = ((size_t)h * T_tok + s0 + lo) * d;
  const size_t dst = ((size_t)phys * Hk + h) * 64 * d;
  const int vecs = d / 8, rgroups = kThreads / vecs;
  const int vec = threadIdx.x % vecs, rg = threadIdx.x / vecs;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  // this thread's rows (d / 32 of them, at most 4): every load goes out before the
  // first store, so a thread keeps all of its copies in flight
  uint4 kv[4], vv[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int row = rg + t * rgroups;
    kv[t] = vv[t] = make_uint4(0u, 0u, 0u, 0u);
    if (row < nrows) {
      kv[t] = __ldg(reinterpret_cast<const uint4 *>(K + src + (size_t)row * d) + vec);
      vv[t] = __ldg(reinterpret_cast<const uint4 *>(V + src + (size_t)row * d) + vec);
    }
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int row = rg + t * rgroups;
    if (row < 64) {
      if (row < nrows) Vec16<uint16_t>::add(kv[t], acc);
      reinterpret_cast<uint4 *>(kc + dst + (size_t)row * d)[vec] = kv[t];
      reinterpret_cast<uint4 *>(vc + dst + (size_t)row * d)[vec] = vv[t];
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) red[rg * d + vec * 8 + e] = acc[e];
  __syncthreads();
  float *out = ps + ((size_t)phys * Hk + h) * d;
  for (int c = threadIdx.x; c < d; c += kThreads) {
    float sum = 0.f;
    for (int g = 0; g < rgroups; ++g) sum += red[g * d + c];
    out[c] = sum / (float)nrows;
    if (psum != nullptr) psum[((size_t)phys * Hk + h) * d + c] = sum;
  }
  grid_dep_launch();
}

}  // namespace

cudaError_t launch_chunk_append(const bsa_shape_t &s, const bsa_kv_cache_t &c, const void *K,
                                const void *V, int32_t *dev_status, cudaStream_t st) {
  const dim3 grid(s.max_blocks, s.num_seqs, s.num_kv_heads);
  const size_t sm = (size_t)(kThreads / (s.head_dim / 8)) * s.head_dim * sizeof(float);
  return launch_dependent(chunk_append_kernel, grid, dim3(kThreads), sm, st,
                          static_cast<const uint16_t *>(K), static_cast<const uint16_t *>(V),
                          s.cu_seqlens, c.prefix_lens, c.block_table,
                          static_cast<uint16_t *>(c.k_cache), static_cast<uint16_t *>(c.v_cache),
                          c.page_summ, c.page_sum, dev_status, s.total_tokens, s.num_kv_heads,
                          s.head_dim, c.max_pages_per_req, c.num_phys_pages,
                          c.max_context_blocks);
}

cudaError_t launch_page_summaries_append(const bsa_decode_shape_t &s, const void *k_cache,
                                         const int32_t *block_table,
                                         const int32_t *context_lens, float *page_sum,
                                         float *page_summ, cudaStream_t st) {
  page_summaries_append_kernel<<<dim3(s.num_reqs, s.num_kv_heads), s.head_dim, 0, st>>>(
      static_cast<const uint16_t *>(k_cache), block_table, context_lens, page_sum, page_summ,
      s.max_pages_per_req, s.num_kv_heads, s.page_size, s.head_dim, s.num_phys_pages);
  return cudaGetLastError();
}

cudaError_t launch_block_summaries(const bsa_shape_t &s, const void *K, float *C,
                                   cudaStream_t st) {
  const dim3 grid(s.max_blocks, s.num_seqs, s.num_kv_heads);
  if (s.dtype == BSA_BF16) {
    const size_t sm = (size_t)(kThreads / (s.head_dim / 8)) * s.head_dim * sizeof(float);
    return launch_dependent(block_summaries_kernel<uint16_t>, grid, dim3(kThreads), sm, st,
                            static_cast<const uint16_t *>(K), s.cu_seqlens, C, s.total_tokens,
                            s.max_blocks, s.num_kv_heads, s.head_dim, s.block);
  } else {
    const size_t sm = (size_t)(kThreads / (s.head_dim / 4)) * s.head_dim * sizeof(float);
    block_summaries_kernel<float><<<grid, kThreads, sm, st>>>(
        static_cast<const float *>(K), s.cu_seqlens, C, s.total_tokens, s.max_blocks,
        s.num_kv_heads, s.head_dim, s.block);
  }
  return cudaGetLastError();
}

cudaError_t launch_page_summaries(const bsa_decode_shape_t &s, const void *k_cache,
                                  const int32_t *block_table, const int32_t *context_lens,
                                  float *page_summ, cudaStream_t st) {
  const dim3 grid(s.max_pages_per_req, s.num_reqs, s.num_kv_heads);
  const size_t sm = (size_t)(kThreads / (s.head_dim / 8)) * s.head_dim * sizeof(float);
  page_summaries_kernel<<<grid, kThreads, sm, st>>>(
      static_cast<const uint16_t *>(k_cache), block_table, context_lens, page_summ,
      s.max_pages_per_req, s.num_kv_heads, s.page_size, s.head_dim, s.num_phys_pages);
  return cudaGetLastError();
}

}  // namespace bsa
