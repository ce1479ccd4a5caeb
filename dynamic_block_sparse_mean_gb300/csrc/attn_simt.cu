// a5, FP32 correctness path: the same sparse attention as the tensor-core kernel
// ("2.1 · 粗粒度选择" §1.2 eqs.(1)-(5)) on fp32 inputs with SIMT FFMA.  One CTA
// per (work row, query head); each warp owns b/8 query rows and walks the row's
// selected blocks 32 keys at a time, merging chunks with eqs.(3)-(5).
#include "common.cuh"
#include "kernels.h"

namespace bsa {
namespace {

constexpr int kWarps = 8;
constexpr int kChunk = 32;

template <int D, int B>
__global__ void __launch_bounds__(kWarps * 32) attn_simt_kernel(
    const float *__restrict__ Q, const float *__restrict__ K, const float *__restrict__ V,
    const int32_t *__restrict__ cu, const int32_t *__restrict__ row_ptr,
    const int32_t *__restrict__ col_idx, const int32_t *__restrict__ work,
    const int32_t *__restrict__ bucket_off, float scale, float *__restrict__ O,
    float *__restrict__ lse, int T_tok, int Nq, int Hk, int G, int32_t *__restrict__ status) {
  constexpr int RPW = B / kWarps;  // query rows per warp
  constexpr int DL = D / 32;       // output columns per lane
  extern __shared__ float smem[];
  float *Qs = smem;                        // [B][D]
  float *Ks = Qs + B * D;                  // [kChunk][D + 1]
  float *Vs = Ks + kChunk * (D + 1);       // [kChunk][D]
  const int unit = blockIdx.x;
  const int nrows = bucket_off[BSA_NUM_BUCKETS];
  if (unit >= nrows * G) return;
  const int row = work[unit / G];
  const int hq_local = unit % G;
  const int r = row % Nq, h = (row / Nq) % Hk, i = row / (Nq * Hk);
  const int hq = h * G + hq_local;
  const int s0 = cu[i], n = cu[i + 1] - s0;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  for (int e = threadIdx.x; e < B * D; e += blockDim.x) {
    const int t = r * B + e / D;
    Qs[e] = t < n ? Q[((size_t)hq * T_tok + s0 + t) * D + e % D] : 0.f;
  }
  float o[RPW][DL], m[RPW], l[RPW];
#pragma unroll
  for (int a = 0; a < RPW; ++a) {
    m[a] = -INFINITY;
    l[a] = 0.f;
#pragma unroll
    for (int c = 0; c < DL; ++c) o[a][c] = 0.f;
  }
  const int kb0 = row_ptr[row], nkv = row_ptr[row + 1] - kb0;
  for (int jj = 0; jj < nkv; ++jj) {
    const int kb = checked_index(col_idx[kb0 + jj], 0, r, status);
    for (int c0 = 0; c0 < B; c0 += kChunk) {
      __syncthreads();
      for (int e = threadIdx.x; e < kChunk * D; e += blockDim.x) {
        const int s = kb * B + c0 + e / D;
        const size_t g = ((size_t)h * T_tok + s0 + s) * D + e % D;
        const bool ok = s < n;
        Ks[(e / D) * (D + 1) + e % D] = ok ? K[g] : 0.f;
        Vs[e] = ok ? V[g] : 0.f;
      }
      __syncthreads();
      const int s = kb * B + c0 + lane;  // this lane's key
#pragma unroll
      for (int a = 0; a < RPW; ++a) {
        const int qi = warp + a * kWarps;
        const int t = r * B + qi;
        float dot = 0.f;
#pragma unroll 8
        for (int e = 0; e < D; ++e) dot = fmaf(Qs[qi * D + e], Ks[lane * (D + 1) + e], dot);
        const bool ok = s < n && s <= t;
        const float sv = ok ? dot * scale : -INFINITY;
        float mx = sv;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m[a], mx);
        if (m_new == -INFINITY) continue;  // nothing visible yet in this chunk
        const float alpha = expf(m[a] - m_new);
        const float p = ok ? expf(sv - m_new) : 0.f;
        float ps = p;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        l[a] = l[a] * alpha + ps;
#pragma unroll
        for (int c = 0; c < DL; ++c) o[a][c] *= alpha;
        for (int k = 0; k < kChunk; ++k) {
          const float pk = __shfl_sync(0xffffffffu, p, k);
#pragma unroll
          for (int c = 0; c < DL; ++c) o[a][c] = fmaf(pk, Vs[k * D + lane + 32 * c], o[a][c]);
        }
        m[a] = m_new;
      }
    }
  }
#pragma unroll
  for (int a = 0; a < RPW; ++a) {
    const int t = r * B + warp + a * kWarps;
    if (t >= n) continue;
    const float inv = 1.f / l[a];
#pragma unroll
    for (int c = 0; c < DL; ++c) O[((size_t)hq * T_tok + s0 + t) * D + lane + 32 * c] = o[a][c] * inv;
    if (lse != nullptr && lane == 0) lse[(size_t)hq * T_tok + s0 + t] = m[a] + logf(l[a]);
  }
}

template <int D, int B>
cudaError_t launch_simt(const bsa_shape_t &s, const void *Q, const void *K, const void *V,
                        const int32_t *row_ptr, const int32_t *col_idx, const int32_t *work,
                        const int32_t *bucket_off, float scale, void *O, float *lse,
                        int32_t *status, cudaStream_t st) {
  const size_t sm = (size_t)(B * D + kChunk * (D + 1) + kChunk * D) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel<D, B>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const int G = s.num_heads / s.num_kv_heads;
  const long long units = (long long)s.num_seqs * s.num_kv_heads * s.max_blocks * G;
  attn_simt_kernel<D, B><<<(unsigned)units, kWarps * 32, sm, st>>>(
      static_cast<const float *>(Q), static_cast<const float *>(K), static_cast<const float *>(V),
      s.cu_seqlens, row_ptr, col_idx, work, bucket_off, scale, static_cast<float *>(O), lse,
      s.total_tokens, s.max_blocks, s.num_kv_heads, G, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_simt_f32(const bsa_shape_t &s, const void *Q, const void *K,
                                      const void *V, const int32_t *row_ptr,
                                      const int32_t *col_idx, const int32_t *work,
                                      const int32_t *bucket_off, float scale, void *O,
                                      float *lse, int32_t *status, cudaStream_t st) {
  if (s.head_dim == 64 && s.block == 64)
    return launch_simt<64, 64>(s, Q, K, V, row_ptr, col_idx, work, bucket_off, scale, O, lse, status,
                               st);
  if (s.head_dim == 64 && s.block == 128)
    return launch_simt<64, 128>(s, Q, K, V, row_ptr, col_idx, work, bucket_off, scale, O, lse, status,
                                st);
  if (s.head_dim == 128 && s.block == 64)
    return launch_simt<128, 64>(s, Q, K, V, row_ptr, col_idx, work, bucket_off, scale, O, lse, status,
                                st);
  return launch_simt<128, 128>(s, Q, K, V, row_ptr, col_idx, work, bucket_off, scale, O, lse,
                               status, st);
}

}  // namespace bsa
