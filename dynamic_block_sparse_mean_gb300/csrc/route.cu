// a2 + a3: the block router of "2.1 · 粗粒度选择" §2.1.
//   scores  g[i,h,r,j] = max over the group's query heads and the valid tokens
//           of block r of q . c_j, j < r (eq.(6), pool = max; unscaled)
//   select  forced diagonal (+ sink), then top-k or the clamped threshold of
//           eq.(7); ranking (score desc, index asc); rows deduplicated and
//           sorted ascending (eq.(1) address order).
// Scores are fp32 FFMA dot products (fp32-accurate: the selection is compared
// bit-exactly, up to a 1e-5 tie band, with a float64 oracle).
#include "common.cuh"
#include "kernels.h"

namespace bsa {
namespace {

constexpr int kTile = 64;     // query rows x summaries per CTA tile
constexpr int kKc = 32;       // d chunk
constexpr int kThreads = 256;  // 16 x 16 threads, 4 x 4 outputs each

template <typename T>
BSA_DEV void load8(const T *p, float *v);
template <>
BSA_DEV void load8<uint16_t>(const uint16_t *p, float *v) {
  const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[2 * e] = __uint_as_float(w[e] << 16);
    v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}
template <>
BSA_DEV void load8<float>(const float *p, float *v) {
  const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
  const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// grid (N_q, H_kv, B): one CTA per router row (i, h, r); writes g[r][0 .. r-1].
template <typename T>
__global__ void __launch_bounds__(kThreads) route_scores_kernel(
    const T *__restrict__ Q, const float *__restrict__ C, const int32_t *__restrict__ cu,
    float *__restrict__ S, int T_tok, int Nq, int Hk, int G, int d, int b) {
  __shared__ float Qs[kKc][kTile + 4];
  __shared__ float Cs[kKc][kTile + 4];
  __shared__ float red[16][kTile];
  const int r = blockIdx.x, h = blockIdx.y, i = blockIdx.z;
  const int s0 = cu[i], n = cu[i + 1] - s0;
  const int nb = (n + b - 1) / b;
  if (r >= nb || r == 0) return;
  const int nvalid = min(b, n - r * b);       // valid query tokens of block r
  const int nrows = G * nvalid;                // pooled query rows
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const float *Crow = C + (((size_t)i * Hk + h) * Nq) * d;
  float *Srow = S + (((size_t)i * Hk + h) * Nq + r) * Nq;
  // loader mapping: 256 threads x 8 elements = 64 rows x 32 columns
  const int lrow = threadIdx.x / 4, lk = (threadIdx.x % 4) * 8;

  for (int j0 = 0; j0 < r; j0 += kTile) {
    float runmax[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    for (int q0 = 0; q0 < nrows; q0 += kTile) {
      float acc[4][4] = {};
      for (int k0 = 0; k0 < d; k0 += kKc) {
        {
          float v[8];
          const int rho = q0 + lrow;
          if (rho < nrows) {
            const int hq = h * G + rho / nvalid, t = r * b + rho % nvalid;
            load8<T>(Q + ((size_t)hq * T_tok + s0 + t) * d + k0 + lk, v);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.f;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) Qs[lk + e][lrow] = v[e];
          const int j = j0 + lrow;
          if (j < r) {
            const float4 *cp = reinterpret_cast<const float4 *>(Crow + (size_t)j * d + k0 + lk);
            const float4 a = __ldg(cp), c = __ldg(cp + 1);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.f;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) Cs[lk + e][lrow] = v[e];
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < kKc; ++k) {
          const float4 qa = *reinterpret_cast<const float4 *>(&Qs[k][ty * 4]);
          const float4 ca = *reinterpret_cast<const float4 *>(&Cs[k][tx * 4]);
          const float qv[4] = {qa.x, qa.y, qa.z, qa.w};
          const float cv[4] = {ca.x, ca.y, ca.z, ca.w};
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(qv[a], cv[c], acc[a][c]);
        }
        __syncthreads();
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
        if (q0 + ty * 4 + a < nrows)
#pragma unroll
          for (int c = 0; c < 4; ++c) runmax[c] = fmaxf(runmax[c], acc[a][c]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) red[ty][tx * 4 + c] = runmax[c];
    __syncthreads();
    if (threadIdx.x < kTile) {
      float m = -INFINITY;
#pragma unroll
      for (int y = 0; y < 16; ++y) m = fmaxf(m, red[y][threadIdx.x]);
      const int j = j0 + threadIdx.x;
      if (j < r) Srow[j] = m;
    }
    __syncthreads();
  }
}

// Order-preserving map of a float score onto uint32 (larger score, larger key;
// -0 and +0 map alike, as they compare equal).
BSA_DEV uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp per router row: forced blocks, then top-k / eq.(7) threshold, then the
// row in ascending order.  The dynamic picks are the k_dyn largest candidates under
// (score desc, index asc), found by a radix select on order-preserving keys (8 bits
// per pass from the top; it stops once the bin of the k-th key holds exactly the
// keys still needed), then written with the forced blocks in one ordered pass.
// Row (i, h, qb) selects for logical block r = qb, or in a chunked prefill
// qb + the blocks cached before the chunk (qoff: cached tokens per sequence);
// S rows hold Nk scores.
// Dynamic shared memory: Nk floats of scores, a 256-bin histogram, Nk flag bytes.
__global__ void __launch_bounds__(32) route_select_kernel(
    const float *__restrict__ S, const int32_t *__restrict__ cu,
    const int32_t *__restrict__ qoff, int32_t *__restrict__ J, int32_t *__restrict__ counts,
    int Nq, int Nk, int Hk, int b, int mode, int k_max, int k_min, float tau_delta,
    int force_sink, int window, int num_global, const int32_t *__restrict__ global_blocks) {
  extern __shared__ uint8_t sm[];
  float *sc = reinterpret_cast<float *>(sm);
  int32_t *hist = reinterpret_cast<int32_t *>(sm + (size_t)Nk * 4);
  uint8_t *taken = sm + (size_t)Nk * 4 + 256 * 4;
  const int lane = threadIdx.x;
  const int row = blockIdx.x;
  const int qb = row % Nq, i = row / (Nq * Hk);
  grid_dep_wait();  // the scores come from the previous launch
  const int n = cu[i + 1] - cu[i];
  const int nb = (n + b - 1) / b;
  int r = qb;
  bool ok = true;
  if (qoff != nullptr) {
    const int pre = qoff[i];
    ok = chunk_ok(pre, n, b, Nk);
    if (ok) r += pre / b;
  }
  int32_t *Jrow = J + (size_t)row * k_max;
  if (!ok || qb >= nb) {
    for (int e = lane; e < k_max; e += 32) Jrow[e] = -1;
    if (lane == 0) counts[row] = 0;
    return;
  }
  const float *Srow = S + (size_t)row * Nk;
  // Forced blocks F_r (union routing: local window, global list, sink, diagonal)
  // are marked `taken` so the dynamic choice never spends budget on them; a block
  // named by several branches is kept once.
  const int wlo = max(0, r - max(1, window) + 1);
  for (int j = lane; j < r; j += 32) {
    sc[j] = Srow[j];
    taken[j] = (j >= wlo || (force_sink && j == 0)) ? 1 : 0;
  }
  __syncwarp();
  if (lane < num_global) {
    const int gb = global_blocks[lane];
    if (gb >= 0 && gb < r) taken[gb] = 1;
  }
  __syncwarp();
  int nhist = 0;  // forced history blocks (j < r)
  for (int j = lane; j < r; j += 32) nhist += taken[j] ? 1 : 0;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) nhist += __shfl_xor_sync(0xffffffffu, nhist, off);
  const int nforced = nhist + 1;  // + the diagonal
  const int ncand = r - nhist;

  int k_dyn;
  if (mode == BSA_ROUTE_TOPK) {
    k_dyn = k_max - nforced;
  } else {
    float mx = -INFINITY;
    for (int j = lane; j < r; j += 32)
      if (!taken[j]) mx = fmaxf(mx, sc[j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float tau = mx - tau_delta;
    int a = 0;
    for (int j = lane; j < r; j += 32)
      if (!taken[j] && sc[j] >= tau) ++a;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
    const int k_r = min(k_max, min(max(k_min, nforced + a), nforced + ncand));
    k_dyn = k_r - nforced;
  }
  k_dyn = max(0, min(k_dyn, ncand));

  uint32_t prefix = 0, mask = 0;
  int remaining = k_dyn;  // dynamic picks still to place at or below the current bin
  if (k_dyn > 0 && k_dyn < ncand) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int e = lane; e < 256; e += 32) hist[e] = 0;
      __syncwarp();
      for (int j = lane; j < r; j += 32)
        if (!taken[j]) {
          const uint32_t kk = order_key(sc[j]);
          if ((kk & mask) == prefix) atomicAdd(&hist[(kk >> shift) & 255u], 1);
        }
      __syncwarp();
      // lane l owns bins 255 - 8l .. 248 - 8l (descending); counts from the top
      int loc[8], tot = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        loc[q] = hist[255 - 8 * lane - q];
        tot += loc[q];
      }
      int incl = tot;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const int excl = incl - tot;
      int bin = -1, above = 0, inbin = 0;
      if (excl < remaining && incl >= remaining) {
        int acc = excl;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (bin < 0 && acc + loc[q] >= remaining) {
            bin = 255 - 8 * lane - q;
            above = acc;
            inbin = loc[q];
          }
          acc += loc[q];
        }
      }
      const int src = __ffs(__ballot_sync(0xffffffffu, bin >= 0)) - 1;
      bin = __shfl_sync(0xffffffffu, bin, src);
      above = __shfl_sync(0xffffffffu, above, src);
      inbin = __shfl_sync(0xffffffffu, inbin, src);
      remaining -= above;
      prefix |= (uint32_t)bin << shift;
      mask |= 0xFFu << shift;
      __syncwarp();  // every lane has read hist before the next pass clears it
      // the k-th key's bin holds exactly the keys still needed: all are picked
      if (inbin == remaining) break;
    }
  }
  // One ordered pass: forced blocks, candidates above the k-th key's bin, and the
  // first `remaining` candidates inside it (ties to the lower block index).
  int w = 0, eq_seen = 0;
  for (int j0 = 0; j0 <= r; j0 += 32) {
    const int j = j0 + lane;
    bool keep = false, eq = false;
    if (j < r) {
      if (taken[j]) {
        keep = true;
      } else if (k_dyn >= ncand) {
        keep = k_dyn > 0;
      } else if (k_dyn > 0) {
        const uint32_t kk = order_key(sc[j]) & mask;
        keep = kk > prefix;
        eq = kk == prefix;
      }
    } else if (j == r) {
      keep = true;  // the diagonal
    }
    const unsigned em = __ballot_sync(0xffffffffu, eq);
    if (eq) keep = eq_seen + __popc(em & ((1u << lane) - 1u)) < remaining;
    eq_seen += __popc(em);
    const unsigned km = __ballot_sync(0xffffffffu, keep);
    if (keep) Jrow[w + __popc(km & ((1u << lane) - 1u))] = j;
    w += __popc(km);
  }
  for (int e = w + lane; e < k_max; e += 32) Jrow[e] = -1;
  if (lane == 0) counts[row] = w;
  grid_dep_launch();
}

}  // namespace

// Workspace: [bf16 split of C, BF16 path only][score matrix, unless the caller
// passes its own `scores` buffer].  With a cache (chunked prefill) the summaries
// come from its pages and score rows hold N_k entries.
size_t route_workspace_bytes(const bsa_shape_t &s, const bsa_route_params_t &,
                             const bsa_kv_cache_t *cache) {
  const size_t split = s.dtype == BSA_BF16 ? route_tc_workspace_bytes(s, cache) : 0;
  const size_t Nk = cache != nullptr ? cache->max_context_blocks : s.max_blocks;
  return split + (size_t)s.num_seqs * s.num_kv_heads * s.max_blocks * Nk * sizeof(float);
}

cudaError_t launch_route(const bsa_shape_t &s, const bsa_route_params_t &p, const void *Q,
                         const float *C, const bsa_kv_cache_t *cache, int32_t *J,
                         int32_t *counts, float *scores, int32_t *dev_status, void *ws,
                         cudaStream_t st) {
  const size_t split = s.dtype == BSA_BF16 ? route_tc_workspace_bytes(s, cache) : 0;
  float *S = scores != nullptr ? scores
                               : reinterpret_cast<float *>(static_cast<char *>(ws) + split);
  const int G = s.num_heads / s.num_kv_heads;
  const int Nk = cache != nullptr ? cache->max_context_blocks : s.max_blocks;
  const dim3 grid(s.max_blocks, s.num_kv_heads, s.num_seqs);
  cudaError_t e;
  if (s.dtype == BSA_BF16) {
    e = launch_route_scores_tc(s, Q, C, cache, S, ws, dev_status, st);
    if (e != cudaSuccess) return e;
  } else {
    route_scores_kernel<float><<<grid, kThreads, 0, st>>>(
        static_cast<const float *>(Q), C, s.cu_seqlens, S, s.total_tokens, s.max_blocks,
        s.num_kv_heads, G, s.head_dim, s.block);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int rows = s.num_seqs * s.num_kv_heads * s.max_blocks;
  const size_t sm = (size_t)Nk * 5 + 256 * 4 + 16;
  if (sm > 48 * 1024) {
    e = cudaFuncSetAttribute(route_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm);
    if (e != cudaSuccess) return e;
  }
  return launch_dependent(route_select_kernel, dim3(rows), dim3(32), sm, st, S, s.cu_seqlens,
                          cache != nullptr ? cache->prefix_lens : nullptr, J, counts,
                          s.max_blocks, Nk, s.num_kv_heads, s.block, p.mode, p.k_max, p.k_min,
                          p.tau_delta, p.force_sink, p.window, p.num_global, p.global_blocks);
}

}  // namespace bsa
