// Router quality: token recall against the dense top-t teacher ("2.1 · 粗粒度选择"
// §1.1, the paragraph on recall@k: G_i = the dense attention's top-t keys of query
// i, N(i) = its candidate keys, recall = |G_i ∩ N(i)| / |G_i|).  A measurement of
// the router, run outside the hot path.
//
// One CTA per tile of 64 consecutive query tokens of one query head (all in one
// router row, since b >= 64).  The sequence's visible keys stream through shared
// memory in 64-key chunks; every pass recomputes the 64 x 64 fp32 scores q . k of a
// chunk (a register-tiled SIMT product, 4 x 4 per thread) and:
//   radix passes  histogram the next 8 bits of the order-preserving score key of
//                 the keys still tied with the t-th largest, per query, until the
//                 t-th largest key is resolved (or its bin holds exactly the keys
//                 still needed);
//   final pass    counts, per query, the teacher keys inside the row's selected
//                 blocks: keys above the resolved prefix, plus the first
//                 `remaining` keys equal to it in index order (the teacher's
//                 (score desc, index asc) rule), found with a segmented scan over
//                 the 16 threads that hold a query's 64 chunk keys in order.
// Shared memory: the tile's queries and the chunk's keys as transposed fp32 panels,
// a 64 x 256 histogram, per-query state and a bitmap of the row's selected blocks.
#include "common.cuh"
#include "kernels.h"

namespace bsa {
namespace {

constexpr int kRT = 256;   // threads: 16 x 16, each 4 queries x 4 keys
constexpr int kRQ = 64;    // queries per tile
constexpr int kRK = 64;    // keys per chunk
constexpr int kPad = 68;   // row stride (floats) of the transposed panels

BSA_DEV uint32_t okey(float v) {  // monotone map of floats onto uint32 (-0 = +0)
  const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <typename T>
struct Elem;
template <>
struct Elem<uint16_t> {
  static constexpr int kPerVec = 8;
  BSA_DEV static void unpack(const uint4 &v, float *f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[2 * e] = __uint_as_float(w[e] << 16);
      f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
  }
};
template <>
struct Elem<float> {
  static constexpr int kPerVec = 4;
  BSA_DEV static void unpack(const uint4 &v, float *f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};

// rows [row0, row0 + 64) of a [rows, D] matrix -> panel[kk][row] (fp32); rows at or
// past `nvalid` are zero.
template <typename T, int D>
BSA_DEV void load_panel(const T *__restrict__ base, int nvalid, float *panel) {
  constexpr int E = Elem<T>::kPerVec;
  constexpr int kVecs = kRQ * D / E;
  for (int v = threadIdx.x; v < kVecs; v += kRT) {
    // consecutive threads take consecutive rows: conflict-free transposed stores
    const int row = v % kRQ, col = (v / kRQ) * E;
    float f[E];
    if (row < nvalid) {
      Elem<T>::unpack(__ldg(reinterpret_cast<const uint4 *>(base + (size_t)row * D + col)), f);
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) f[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) panel[(col + e) * kPad + row] = f[e];
  }
}

template <int D>
BSA_DEV void chunk_scores(const float *Qs, const float *Ks, int ty, int tx, float (&acc)[4][4]) {
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
#pragma unroll 8
  for (int kk = 0; kk < D; ++kk) {
    const float4 qa = *reinterpret_cast<const float4 *>(Qs + kk * kPad + 4 * ty);
    const float4 kb = *reinterpret_cast<const float4 *>(Ks + kk * kPad + 4 * tx);
    const float qv[4] = {qa.x, qa.y, qa.z, qa.w}, kv[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(qv[a], kv[c], acc[a][c]);
  }
}

struct RecallParams {
  const int32_t *cu, *J, *counts, *tiles;
  int32_t *hits, *status;
  int T, H, Hk, G, Nq, k_max, b, t_top, tiles_per_seq, num_tiles_all, bitmap_words;
};

template <typename T, int D>
__global__ void __launch_bounds__(kRT, 1)
    token_recall_kernel(const T *__restrict__ Q, const T *__restrict__ K, const RecallParams p) {
  extern __shared__ __align__(16) float rsm[];
  float *Qs = rsm;                       // [D][kPad]
  float *Ks = Qs + D * kPad;             // [D][kPad]
  int *hist = reinterpret_cast<int *>(Ks + D * kPad);   // [64][256]
  uint32_t *s_prefix = reinterpret_cast<uint32_t *>(hist + kRQ * 256);
  uint32_t *s_mask = s_prefix + kRQ;
  int *s_rem = reinterpret_cast<int *>(s_mask + kRQ);
  int *s_done = s_rem + kRQ;
  int *s_t = s_done + kRQ;               // sequence position of each query, -1 if none
  int *s_eq = s_t + kRQ;                 // equal keys seen so far (final pass)
  int *s_hits = s_eq + kRQ;
  uint32_t *s_bits = reinterpret_cast<uint32_t *>(s_hits + kRQ);  // selected blocks
  __shared__ int s_all_done;

  const int tile = p.tiles != nullptr ? p.tiles[blockIdx.x] : (int)blockIdx.x;
  if (tile < 0 || tile >= p.num_tiles_all) {  // a listed tile id outside the batch
    if (threadIdx.x == 0) set_status(p.status, BSA_ERR_INDEX_RANGE);
    return;
  }
  const int per_seq = p.tiles_per_seq;
  const int c = tile % per_seq, ih = tile / per_seq;
  const int hq = ih % p.H, i = ih / p.H;
  const int s0 = p.cu[i], n = p.cu[i + 1] - s0;
  const int t0 = c * kRQ;
  if (t0 >= n) return;  // a tile past the sequence's end
  const int h = hq / p.G, r = t0 / p.b;
  const int kend = min(n, t0 + kRQ);     // keys 0 .. kend-1 are visible to some query

  // the row's selected blocks as a bitmap (an empty row keeps its diagonal)
  for (int w = threadIdx.x; w < p.bitmap_words; w += kRT) s_bits[w] = 0u;
  __syncthreads();
  const size_t row = ((size_t)i * p.Hk + h) * p.Nq + r;
  const int cnt = min(max(p.counts[row], 0), p.k_max);
  for (int e = threadIdx.x; e < cnt; e += kRT) {
    const int j = p.J[row * p.k_max + e];
    if (j >= 0 && j < p.Nq) atomicOr(&s_bits[j >> 5], 1u << (j & 31));
  }
  if (cnt == 0 && threadIdx.x == 0) atomicOr(&s_bits[r >> 5], 1u << (r & 31));
  if (threadIdx.x < kRQ) {
    const int q = threadIdx.x, t = t0 + q;
    const bool valid = t < n;
    const int vis = t + 1;
    s_t[q] = valid ? t : -1;
    s_prefix[q] = 0u;
    s_mask[q] = 0u;
    // a teacher as large as the visible set is the whole set: resolved at once
    s_rem[q] = valid ? (vis <= p.t_top ? vis : p.t_top) : 0;
    s_done[q] = valid ? (vis <= p.t_top ? 1 : 0) : 1;
    s_eq[q] = 0;
    s_hits[q] = 0;
  }
  load_panel<T, D>(Q + ((size_t)hq * p.T + s0 + t0) * D, kend - t0, Qs);
  __syncthreads();

  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  const T *Kh = K + ((size_t)h * p.T + s0) * D;
  float acc[4][4];

  // ---- radix passes over the order-preserving score keys
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (threadIdx.x == 0) {
      int all = 1;
      for (int q = 0; q < kRQ; ++q) all &= s_done[q];
      s_all_done = all;
    }
    for (int e = threadIdx.x; e < kRQ * 256; e += kRT) hist[e] = 0;
    __syncthreads();
    if (s_all_done) break;
    for (int cs = 0; cs < kend; cs += kRK) {
      load_panel<T, D>(Kh + (size_t)cs * D, kend - cs, Ks);
      __syncthreads();
      chunk_scores<D>(Qs, Ks, ty, tx, acc);
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int q = 4 * ty + a;
        if (s_done[q]) continue;
        const uint32_t pm = s_prefix[q], mk = s_mask[q];
        const int t = s_t[q];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int s = cs + 4 * tx + cc;
          const uint32_t k = okey(acc[a][cc]);
          if (s <= t && (k & mk) == pm) atomicAdd(&hist[q * 256 + ((k >> shift) & 255)], 1);
        }
      }
      __syncthreads();
    }
    if (threadIdx.x < kRQ && !s_done[threadIdx.x]) {
      const int q = threadIdx.x;
      int rem = s_rem[q], above = 0, bin = -1;
      for (int bb = 255; bb >= 0; --bb) {
        const int hc = hist[q * 256 + bb];
        if (above + hc >= rem) {
          bin = bb;
          break;
        }
        above += hc;
      }
      if (bin < 0) {  // cannot happen: the keys matching the prefix always suffice
        set_status(p.status, BSA_ERR_COUNT);
        s_done[q] = 1;
      } else {
        rem -= above;
        s_rem[q] = rem;
        s_prefix[q] |= (uint32_t)bin << shift;
        s_mask[q] |= 0xFFu << shift;
        if (hist[q * 256 + bin] == rem || shift == 0) s_done[q] = 1;
      }
    }
    __syncthreads();
  }

  // ---- final pass: teacher keys inside the selected blocks
  int mine[4] = {0, 0, 0, 0};
  for (int cs = 0; cs < kend; cs += kRK) {
    const int blk = cs / p.b;  // a 64-key chunk lies inside one block (b >= 64)
    const bool in_set = (s_bits[blk >> 5] >> (blk & 31)) & 1u;
    load_panel<T, D>(Kh + (size_t)cs * D, kend - cs, Ks);
    __syncthreads();
    chunk_scores<D>(Qs, Ks, ty, tx, acc);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int q = 4 * ty + a;
      const uint32_t pm = s_prefix[q], mk = s_mask[q];
      const int t = s_t[q], rem = s_rem[q];
      int eq_local = 0, strict = 0;
      bool eqf[4];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int s = cs + 4 * tx + cc;
        const uint32_t k = okey(acc[a][cc]) & mk;
        const bool valid = s <= t;
        eqf[cc] = valid && k == pm;
        eq_local += eqf[cc] ? 1 : 0;
        strict += (valid && k > pm && in_set) ? 1 : 0;
      }
      // order of this thread's equal keys among the query's equal keys so far:
      // the 16 threads of a half-warp hold keys 4 tx .. 4 tx + 3 of this chunk
      int incl = eq_local;
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off, 16);
        if (tx >= off) incl += y;
      }
      const int chunk_eq = __shfl_sync(0xffffffffu, incl, 15, 16);
      int before = s_eq[q] + incl - eq_local;
      int take = 0;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
        if (eqf[cc]) {
          take += (before < rem && in_set) ? 1 : 0;
          ++before;
        }
      mine[a] += strict + take;
      __syncwarp();
      if (tx == 0) s_eq[q] += chunk_eq;
    }
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    int v = mine[a];
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off, 16);
    if (tx == 0) s_hits[4 * ty + a] = v;
  }
  __syncthreads();
  if (threadIdx.x < kRQ && s_t[threadIdx.x] >= 0)
    p.hits[(size_t)hq * p.T + s0 + s_t[threadIdx.x]] = s_hits[threadIdx.x];
}

template <int D>
size_t recall_smem(const RecallParams &p) {
  return (size_t)2 * D * kPad * sizeof(float) + (size_t)kRQ * 256 * sizeof(int) +
         (size_t)8 * kRQ * sizeof(int) + (size_t)p.bitmap_words * sizeof(uint32_t);
}

template <typename T, int D>
cudaError_t launch_recall_t(const void *Q, const void *K, const RecallParams &p, int grid,
                            cudaStream_t st) {
  const size_t sm = recall_smem<D>(p);
  cudaError_t e = cudaFuncSetAttribute(token_recall_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  token_recall_kernel<T, D><<<grid, kRT, sm, st>>>(static_cast<const T *>(Q),
                                                    static_cast<const T *>(K), p);
  return cudaGetLastError();
}

}  // namespace

int recall_tiles_per_seq(const bsa_shape_t &s) { return (s.max_seqlen + kRQ - 1) / kRQ; }

cudaError_t launch_token_recall(const bsa_shape_t &s, int32_t t_top, const void *Q,
                                const void *K, const int32_t *J, const int32_t *counts,
                                int32_t k_max, const int32_t *tiles, int32_t num_tiles,
                                int32_t *hits, int32_t *dev_status, cudaStream_t st) {
  RecallParams p;
  p.cu = s.cu_seqlens;
  p.J = J;
  p.counts = counts;
  p.tiles = tiles;
  p.hits = hits;
  p.status = dev_status;
  p.T = s.total_tokens;
  p.H = s.num_heads;
  p.Hk = s.num_kv_heads;
  p.G = s.num_heads / s.num_kv_heads;
  p.Nq = s.max_blocks;
  p.k_max = k_max;
  p.b = s.block;
  p.t_top = t_top;
  p.tiles_per_seq = recall_tiles_per_seq(s);
  p.bitmap_words = (s.max_blocks + 31) / 32;
  const long long all = (long long)s.num_seqs * s.num_heads * p.tiles_per_seq;
  p.num_tiles_all = (int)all;
  const int grid = tiles != nullptr ? num_tiles : (int)all;
  if (grid == 0) return cudaSuccess;
  const bool bf16 = s.dtype == BSA_BF16;
  if (s.head_dim == 128)
    return bf16 ? launch_recall_t<uint16_t, 128>(Q, K, p, grid, st)
                : launch_recall_t<float, 128>(Q, K, p, grid, st);
  return bf16 ? launch_recall_t<uint16_t, 64>(Q, K, p, grid, st)
              : launch_recall_t<float, 64>(Q, K, p, grid, st);
}

}  // namespace bsa
