// Backward of the sparse attention on the selected tiles: dQ, dK, dV for an
// upstream gradient dO, reusing the forward's worklist (the router's J) and its
// saved lse, so nothing is re-routed ("2.1 · 粗粒度选择" §2.2: training keeps the
// index and the softmax statistics; the forward of §1.2 eqs.(1)-(5)).  For every
// allowed (query t, key s) pair of a row's tiles:
//   P = exp(S - lse_t),  S = q_t . k_s * scale         (recomputed, not stored)
//   dV_s += P dO_t,  dP = dO_t . v_s,  dS = P (dP - D_t),  D_t = dO_t . O_t
//   dQ_t += dS k_s * scale,  dK_s += dS q_t * scale
// The same masks as the forward: keys past the query (diagonal tile) or past the
// sequence end are excluded.
//
// FP32 arithmetic on the SIMT pipes (bf16 or fp32 inputs and outputs).  One CTA
// per (work row, query head): the row's queries and dO stay in shared memory, the
// selected key blocks stream through it 32 keys at a time, dQ accumulates in
// registers and is written once; dK and dV of a key chunk are summed over the
// block's queries in the CTA and added to fp32 accumulators in global memory with
// atomics (rows of several query blocks and heads share key blocks), then
// converted to the output type by a last launch.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace bsa {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kKC = 32;  // keys per chunk

template <typename T>
BSA_DEV float ldf(const T *p, size_t i);
template <>
BSA_DEV float ldf<float>(const float *p, size_t i) {
  return p[i];
}
template <>
BSA_DEV float ldf<uint16_t>(const uint16_t *p, size_t i) {
  return bf16_to_f32(p[i]);
}

template <typename T>
BSA_DEV void stf(T *p, size_t i, float v);
template <>
BSA_DEV void stf<float>(float *p, size_t i, float v) {
  p[i] = v;
}
template <>
BSA_DEV void stf<uint16_t>(uint16_t *p, size_t i, float v) {
  const __nv_bfloat16 b = __float2bfloat16_rn(v);
  p[i] = *reinterpret_cast<const uint16_t *>(&b);
}

// D[row] = dO[row] . O[row] over the head dimension; one warp per (head, token) row.
template <typename T>
__global__ void bwd_dot_kernel(const T *__restrict__ O, const T *__restrict__ dO,
                               float *__restrict__ Dv, size_t rows, int D) {
  const int lane = threadIdx.x % 32;
  for (size_t row = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) / 32; row < rows;
       row += (size_t)gridDim.x * blockDim.x / 32) {
    float acc = 0.f;
    for (int c = lane; c < D; c += 32) acc = fmaf(ldf(dO, row * D + c), ldf(O, row * D + c), acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) Dv[row] = acc;
  }
}

// The same for bf16 rows of 128: 16 lanes per row, 8 elements (16 bytes) each.
__global__ void bwd_dot_bf16_d128_kernel(const uint16_t *__restrict__ O,
                                         const uint16_t *__restrict__ dO, float *__restrict__ Dv,
                                         size_t rows) {
  const int sub = threadIdx.x % 16;
  for (size_t row = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) / 16; row < rows;
       row += (size_t)gridDim.x * blockDim.x / 16) {
    const uint4 a = __ldg(reinterpret_cast<const uint4 *>(O + row * 128) + sub);
    const uint4 g = __ldg(reinterpret_cast<const uint4 *>(dO + row * 128) + sub);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, gv[4] = {g.x, g.y, g.z, g.w};
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(__uint_as_float(av[e] << 16), __uint_as_float(gv[e] << 16), acc);
      acc = fmaf(__uint_as_float(av[e] & 0xFFFF0000u), __uint_as_float(gv[e] & 0xFFFF0000u), acc);
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (sub == 0) Dv[row] = acc;
  }
}

__global__ void bwd_zero_kernel(float *__restrict__ a, size_t n) {
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x)
    a[e] = 0.f;
}

template <typename T>
__global__ void bwd_convert_kernel(const float *__restrict__ a, T *__restrict__ out, size_t n) {
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x)
    stf(out, e, a[e]);
}

template <typename T, int D, int B>
__global__ void __launch_bounds__(kBwdThreads) attn_bwd_kernel(
    const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
    const T *__restrict__ dO, const float *__restrict__ lse, const float *__restrict__ Dv,
    const int32_t *__restrict__ cu, const int32_t *__restrict__ row_ptr,
    const int32_t *__restrict__ col_idx, const int32_t *__restrict__ work,
    const int32_t *__restrict__ bucket_off, float scale, T *__restrict__ dQ,
    float *__restrict__ dK32, float *__restrict__ dV32, int T_tok, int Nq, int Hk, int G,
    int32_t *__restrict__ status) {
  constexpr int DP = D + 1;                  // padded shared rows (conflict-free columns)
  constexpr int KP = kKC + 1;
  constexpr int EQ = B * D / kBwdThreads;    // dQ elements per thread
  constexpr int EK = kKC * D / kBwdThreads;  // dK / dV chunk elements per thread
  constexpr int EP = B * kKC / kBwdThreads;  // (query, key) pairs per thread
  extern __shared__ float smem[];
  float *Qs = smem;                 // [B][DP]
  float *dOs = Qs + B * DP;         // [B][DP]
  float *Ks = dOs + B * DP;         // [kKC][DP]
  float *Vs = Ks + kKC * DP;        // [kKC][DP]
  float *Ps = Vs + kKC * DP;        // [B][KP]
  float *dSs = Ps + B * KP;         // [B][KP]  (dS * scale)
  float *Ls = dSs + B * KP;         // [B]
  float *Dd = Ls + B;               // [B]
  const int unit = blockIdx.x;
  const int nrows = bucket_off[BSA_NUM_BUCKETS];
  if (unit >= nrows * G) return;
  const int row = work[unit / G];
  const int hq_local = unit % G;
  const int r = row % Nq, h = (row / Nq) % Hk, i = row / (Nq * Hk);
  const int hq = h * G + hq_local;
  const int s0 = cu[i], n = cu[i + 1] - s0;
  const int tid = threadIdx.x;

  for (int e = tid; e < B * D; e += kBwdThreads) {
    const int t = r * B + e / D;
    const size_t g = ((size_t)hq * T_tok + s0 + t) * D + e % D;
    Qs[(e / D) * DP + e % D] = t < n ? ldf(Q, g) : 0.f;
    dOs[(e / D) * DP + e % D] = t < n ? ldf(dO, g) : 0.f;
  }
  for (int t = tid; t < B; t += kBwdThreads) {
    const int tq = r * B + t;
    Ls[t] = tq < n ? lse[(size_t)hq * T_tok + s0 + tq] : 0.f;
    Dd[t] = tq < n ? Dv[(size_t)hq * T_tok + s0 + tq] : 0.f;
  }
  float dq[EQ];
#pragma unroll
  for (int m = 0; m < EQ; ++m) dq[m] = 0.f;

  const int kb0 = row_ptr[row], nkv = row_ptr[row + 1] - kb0;
  for (int jj = 0; jj < nkv; ++jj) {
    const int kb = checked_index(col_idx[kb0 + jj], 0, r, status);
    for (int c0 = 0; c0 < B; c0 += kKC) {
      __syncthreads();
      for (int e = tid; e < kKC * D; e += kBwdThreads) {
        const int s = kb * B + c0 + e / D;
        const size_t g = ((size_t)h * T_tok + s0 + s) * D + e % D;
        const bool ok = s < n;
        Ks[(e / D) * DP + e % D] = ok ? ldf(K, g) : 0.f;
        Vs[(e / D) * DP + e % D] = ok ? ldf(V, g) : 0.f;
      }
      __syncthreads();
      // P and dS of every (query, key) pair of the chunk
#pragma unroll
      for (int m = 0; m < EP; ++m) {
        const int pr = tid + kBwdThreads * m;
        const int t = pr / kKC, kk = pr % kKC;
        const int tq = r * B + t, sk = kb * B + c0 + kk;
        float p = 0.f, ds = 0.f;
        if (tq < n && sk < n && sk <= tq) {
          float sdot = 0.f, pdot = 0.f;
#pragma unroll 8
          for (int e = 0; e < D; ++e) {
            sdot = fmaf(Qs[t * DP + e], Ks[kk * DP + e], sdot);
            pdot = fmaf(dOs[t * DP + e], Vs[kk * DP + e], pdot);
          }
          p = expf(sdot * scale - Ls[t]);
          ds = p * (pdot - Dd[t]);
        }
        Ps[t * KP + kk] = p;
        dSs[t * KP + kk] = ds * scale;
      }
      __syncthreads();
      // dQ += dS K
#pragma unroll
      for (int m = 0; m < EQ; ++m) {
        const int e = tid + kBwdThreads * m;
        const int t = e / D, d = e % D;
        float acc = 0.f;
#pragma unroll 8
        for (int kk = 0; kk < kKC; ++kk) acc = fmaf(dSs[t * KP + kk], Ks[kk * DP + d], acc);
        dq[m] += acc;
      }
      // dK and dV of the chunk, summed over the block's queries
#pragma unroll
      for (int m = 0; m < EK; ++m) {
        const int f = tid + kBwdThreads * m;
        const int kk = f / D, d = f % D;
        const int sk = kb * B + c0 + kk;
        if (sk >= n) continue;
        float dk = 0.f, dv = 0.f;
#pragma unroll 8
        for (int t = 0; t < B; ++t) {
          dk = fmaf(dSs[t * KP + kk], Qs[t * DP + d], dk);
          dv = fmaf(Ps[t * KP + kk], dOs[t * DP + d], dv);
        }
        const size_t g = ((size_t)h * T_tok + s0 + sk) * D + d;
        atomicAdd(dK32 + g, dk);
        atomicAdd(dV32 + g, dv);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < EQ; ++m) {
    const int e = tid + kBwdThreads * m;
    const int t = e / D, d = e % D;
    const int tq = r * B + t;
    if (tq < n) stf(dQ, ((size_t)hq * T_tok + s0 + tq) * D + d, dq[m]);
  }
}

template <typename T, int D, int B>
cudaError_t launch_bwd(const bsa_shape_t &s, const void *Q, const void *K, const void *V,
                       const void *dO, const float *lse, const float *Dv,
                       const int32_t *row_ptr, const int32_t *col_idx, const int32_t *work,
                       const int32_t *bucket_off, float scale, void *dQ, float *dK32,
                       float *dV32, int32_t *status, cudaStream_t st) {
  const size_t sm =
      (size_t)(2 * B * (D + 1) + 2 * kKC * (D + 1) + 2 * B * (kKC + 1) + 2 * B) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<T, D, B>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const int G = s.num_heads / s.num_kv_heads;
  const long long units = (long long)s.num_seqs * s.num_kv_heads * s.max_blocks * G;
  attn_bwd_kernel<T, D, B><<<(unsigned)units, kBwdThreads, sm, st>>>(
      static_cast<const T *>(Q), static_cast<const T *>(K), static_cast<const T *>(V),
      static_cast<const T *>(dO), lse, Dv, s.cu_seqlens, row_ptr, col_idx, work, bucket_off,
      scale, static_cast<T *>(dQ), dK32, dV32, s.total_tokens, s.max_blocks, s.num_kv_heads, G,
      status);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd_typed(const bsa_shape_t &s, const void *Q, const void *K, const void *V,
                             const void *O, const void *dO, const float *lse,
                             const int32_t *row_ptr, const int32_t *col_idx, const int32_t *work,
                             const int32_t *bucket_off, float scale, void *dQ, void *dK, void *dV,
                             void *ws, int32_t *status, cudaStream_t st) {
  const size_t hrows = (size_t)s.num_heads * s.total_tokens;
  const size_t kv = (size_t)s.num_kv_heads * s.total_tokens * s.head_dim;
  char *w = static_cast<char *>(ws);
  float *Dv = reinterpret_cast<float *>(w);
  w += (hrows * sizeof(float) + 255) & ~(size_t)255;
  float *dK32 = reinterpret_cast<float *>(w);
  w += (kv * sizeof(float) + 255) & ~(size_t)255;
  float *dV32 = reinterpret_cast<float *>(w);
  const int grid = std::max(1, std::min(8 * num_sms(), (int)((hrows * 32 + 255) / 256)));
  bwd_dot_kernel<T><<<grid, 256, 0, st>>>(static_cast<const T *>(O), static_cast<const T *>(dO),
                                           Dv, hrows, s.head_dim);
  const int zgrid = std::max(1, std::min(8 * num_sms(), (int)((kv + 255) / 256)));
  bwd_zero_kernel<<<zgrid, 256, 0, st>>>(dK32, kv);
  bwd_zero_kernel<<<zgrid, 256, 0, st>>>(dV32, kv);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (s.head_dim == 64 && s.block == 64)
    e = launch_bwd<T, 64, 64>(s, Q, K, V, dO, lse, Dv, row_ptr, col_idx, work, bucket_off, scale,
                              dQ, dK32, dV32, status, st);
  else if (s.head_dim == 64 && s.block == 128)
    e = launch_bwd<T, 64, 128>(s, Q, K, V, dO, lse, Dv, row_ptr, col_idx, work, bucket_off, scale,
                               dQ, dK32, dV32, status, st);
  else if (s.head_dim == 128 && s.block == 64)
    e = launch_bwd<T, 128, 64>(s, Q, K, V, dO, lse, Dv, row_ptr, col_idx, work, bucket_off, scale,
                               dQ, dK32, dV32, status, st);
  else
    e = launch_bwd<T, 128, 128>(s, Q, K, V, dO, lse, Dv, row_ptr, col_idx, work, bucket_off,
                                scale, dQ, dK32, dV32, status, st);
  if (e != cudaSuccess) return e;
  bwd_convert_kernel<T><<<zgrid, 256, 0, st>>>(dK32, static_cast<T *>(dK), kv);
  bwd_convert_kernel<T><<<zgrid, 256, 0, st>>>(dV32, static_cast<T *>(dV), kv);
  return cudaGetLastError();
}

}  // namespace

// Workspace: D = rowsum(dO * O) [H, T] fp32, then the tensor-core path's key-major
// index (BF16, head_dim 128) or the SIMT path's fp32 dK / dV accumulators.
size_t attention_bwd_workspace_bytes(const bsa_shape_t &s) {
  const size_t hrows = (size_t)s.num_heads * s.total_tokens;
  const size_t kv = (size_t)s.num_kv_heads * s.total_tokens * s.head_dim;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  if (attention_bwd_tc_supported(s))
    return up(hrows * sizeof(float)) + attention_bwd_tc_index_bytes(s);
  return up(hrows * sizeof(float)) + 2 * up(kv * sizeof(float));
}

cudaError_t launch_attention_bwd(const bsa_shape_t &s, const void *Q, const void *K,
                                 const void *V, const void *O, const void *dO, const float *lse,
                                 const int32_t *row_ptr, const int32_t *col_idx,
                                 const int32_t *work, const int32_t *bucket_off, float scale,
                                 void *dQ, void *dK, void *dV, void *ws, int32_t *dev_status,
                                 cudaStream_t st) {
  if (attention_bwd_tc_supported(s)) {
    const size_t hrows = (size_t)s.num_heads * s.total_tokens;
    float *Dv = static_cast<float *>(ws);
    const int grid = std::max(1, std::min(8 * num_sms(), (int)((hrows * 16 + 255) / 256)));
    bwd_dot_bf16_d128_kernel<<<grid, 256, 0, st>>>(static_cast<const uint16_t *>(O),
                                                   static_cast<const uint16_t *>(dO), Dv, hrows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    void *index_ws = static_cast<char *>(ws) + ((hrows * sizeof(float) + 255) & ~(size_t)255);
    return launch_attention_bwd_tc(s, Q, K, V, dO, lse, Dv, row_ptr, col_idx, work, bucket_off,
                                   scale, dQ, dK, dV, index_ws, dev_status, st);
  }
  if (s.dtype == BSA_BF16)
    return launch_bwd_typed<uint16_t>(s, Q, K, V, O, dO, lse, row_ptr, col_idx, work, bucket_off,
                                      scale, dQ, dK, dV, ws, dev_status, st);
  return launch_bwd_typed<float>(s, Q, K, V, O, dO, lse, row_ptr, col_idx, work, bucket_off,
                                 scale, dQ, dK, dV, ws, dev_status, st);
}

}  // namespace bsa
