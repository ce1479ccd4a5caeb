// a6: paged sparse decode ("2.1 · 粗粒度选择" §2.2: decode reads the block
// summaries, O(N_k d_r), then only the selected K/V; §3.1: the router emits
// logical page ids, the block table maps them to physical pages when the
// attention runs).  Four launches, all HBM-bound:
//   score   q . page summary for the complete pages 0 .. L-2 of each
//           (request, KV head), max over the group's query heads
//   select  exact top-k by (score desc, index asc) via a 4-pass radix select,
//           plus the last page L-1, written in ascending order
//   attn    split-KV: each CTA merges a few selected pages per warp with the
//           online-softmax recurrences (eqs.(3)-(5)) in the log2 domain
//   merge   combines the splits into o and lse
#include "common.cuh"
#include "kernels.h"

namespace bsa {
namespace {

constexpr int kD = 128;          // decode head_dim
constexpr int kMaxG = 8;         // query heads per KV head supported (1, 2, 4 or 8)
constexpr int kPagesPerSplit = 4;
constexpr int kScoreThreads = 256;
constexpr int kSelThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- score
// grid (ceil(max_pages / 64), H_kv, R): 64 logical pages per CTA, 8 per warp.
__global__ void __launch_bounds__(kScoreThreads) dec_score_kernel(
    const uint16_t *__restrict__ q, const float *__restrict__ ps, const int32_t *__restrict__ bt,
    const int32_t *__restrict__ lens, float *__restrict__ scores, int H, int Hk, int max_pages) {
  __shared__ float qs[kMaxG][kD];
  const int rho = blockIdx.z, h = blockIdx.y;
  const int G = H / Hk;
  const int L = (lens[rho] + 63) / 64;  // page_size 64
  const int p_begin = blockIdx.x * 64;
  if (p_begin >= L - 1) return;
  for (int e = threadIdx.x; e < G * kD; e += blockDim.x)
    qs[e / kD][e % kD] = bf16_to_f32(q[((size_t)rho * H + h * G + e / kD) * kD + e % kD]);
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int p_end = min(L - 1, p_begin + 64);
  for (int p = p_begin + warp; p < p_end; p += kScoreThreads / 32) {
    const int phys = bt[(size_t)rho * max_pages + p];
    const float4 c = __ldg(reinterpret_cast<const float4 *>(ps + ((size_t)phys * Hk + h) * kD) + lane);
    float best = -INFINITY;
    for (int g = 0; g < G; ++g) {
      float s = qs[g][4 * lane] * c.x + qs[g][4 * lane + 1] * c.y + qs[g][4 * lane + 2] * c.z +
                qs[g][4 * lane + 3] * c.w;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      best = fmaxf(best, s);
    }
    if (lane == 0) scores[((size_t)rho * Hk + h) * max_pages + p] = best;
  }
}

// ---------------------------------------------------------------- select

BSA_DEV uint32_t order_key(float v) {  // monotone map of floats onto uint32
  uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block-wide scan of one int per thread; returns (exclusive, total).
BSA_DEV int2 block_scan(int v, int *buf) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32, nw = blockDim.x / 32;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) buf[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? buf[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    if (lane < nw) buf[lane] = w;
  }
  __syncthreads();
  const int before = warp > 0 ? buf[warp - 1] : 0;
  const int total = buf[nw - 1];
  __syncthreads();
  return make_int2(before + x - v, total);
}

// grid (H_kv, R), one CTA per (request, KV head).
__global__ void __launch_bounds__(kSelThreads) dec_select_kernel(
    const float *__restrict__ scores, const int32_t *__restrict__ lens, int32_t *__restrict__ sel,
    int32_t *__restrict__ sel_counts, int Hk, int max_pages, int top_k) {
  extern __shared__ uint32_t keys[];  // max_pages
  __shared__ int hist[256];
  __shared__ int scan_buf[32];
  __shared__ int s_bin, s_above;
  const int rho = blockIdx.y, h = blockIdx.x;
  const int L = (lens[rho] + 63) / 64;
  const int N = L - 1;  // scored pages
  const float *sc = scores + ((size_t)rho * Hk + h) * max_pages;
  int32_t *out = sel + ((size_t)rho * Hk + h) * (top_k + 1);
  const int k = min(top_k, N);
  for (int e = threadIdx.x; e < N; e += blockDim.x) keys[e] = order_key(sc[e]);
  __syncthreads();

  uint32_t prefix = 0, mask = 0;
  int remaining = k;  // how many of the best are still to be located
  if (k < N) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int e = threadIdx.x; e < 256; e += blockDim.x) hist[e] = 0;
      __syncthreads();
      for (int e = threadIdx.x; e < N; e += blockDim.x)
        if ((keys[e] & mask) == prefix) atomicAdd(&hist[(keys[e] >> shift) & 255], 1);
      __syncthreads();
      if (threadIdx.x < 32) {
        // lane l owns bins 255 - 8l .. 248 - 8l (descending); suffix counts from the top.
        const int lane = threadIdx.x;
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
        if (excl < remaining && incl >= remaining) {
          int acc = excl;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (acc < remaining && acc + loc[q] >= remaining) {
              s_bin = 255 - 8 * lane - q;
              s_above = acc;
            }
            acc += loc[q];
          }
        }
      }
      __syncthreads();
      remaining -= s_above;
      prefix |= (uint32_t)s_bin << shift;
      mask |= 0xFFu << shift;
      __syncthreads();
    }
  }
  // Compact in index order: keys above the k-th key, then the first `remaining`
  // keys equal to it (ties go to the lower page index).
  const int per = (N + blockDim.x - 1) / blockDim.x;
  const int lo = min(N, (int)threadIdx.x * per), hi = min(N, lo + per);
  int n_eq = 0;
  for (int e = lo; e < hi; ++e) n_eq += (k < N && keys[e] == prefix) ? 1 : 0;
  const int2 eq = block_scan(n_eq, scan_buf);
  int taken = 0, eq_seen = eq.x;
  for (int e = lo; e < hi; ++e) {
    bool s;
    if (k >= N) {
      s = true;
    } else if (keys[e] > prefix) {
      s = true;
    } else if (keys[e] == prefix) {
      s = eq_seen < remaining;
      ++eq_seen;
    } else {
      s = false;
    }
    taken += s ? 1 : 0;
  }
  const int2 pos = block_scan(taken, scan_buf);
  int w = pos.x;
  eq_seen = eq.x;
  for (int e = lo; e < hi; ++e) {
    bool s;
    if (k >= N) {
      s = true;
    } else if (keys[e] > prefix) {
      s = true;
    } else if (keys[e] == prefix) {
      s = eq_seen < remaining;
      ++eq_seen;
    } else {
      s = false;
    }
    if (s) out[w++] = e;
  }
  if (threadIdx.x == 0) {
    out[k] = L - 1;  // the last logical page is always kept
    for (int e = k + 1; e <= top_k; ++e) out[e] = -1;
    sel_counts[(size_t)rho * Hk + h] = k + 1;
  }
}

// ---------------------------------------------------------------- attention
// grid (nsplit, H_kv, R), 4 warps; warp w of split s handles selected page
// s * 4 + w.  Lane = 8 * tk + dl: token group tk (4 tokens per step), d-slice dl
// of 16 elements; K and V rows are read as two 16-byte vectors per lane.
template <int G>
__global__ void __launch_bounds__(kPagesPerSplit * 32) dec_attn_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ kc,
    const uint16_t *__restrict__ vc, const int32_t *__restrict__ bt,
    const int32_t *__restrict__ lens, const int32_t *__restrict__ sel,
    const int32_t *__restrict__ sel_counts, float scale_log2, float *__restrict__ part_ml,
    float *__restrict__ part_o, int H, int Hk, int max_pages, int top_k, int nsplit) {
  __shared__ float qs[G][kD];
  __shared__ float wm[kPagesPerSplit][G], wl[kPagesPerSplit][G];
  __shared__ float wo[kPagesPerSplit][G][kD];
  const int rho = blockIdx.z, h = blockIdx.y, split = blockIdx.x;
  const int n = lens[rho];
  const int cnt = sel_counts[(size_t)rho * Hk + h];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int tk = lane / 8, dl = lane % 8;
  for (int e = threadIdx.x; e < G * kD; e += blockDim.x)
    qs[e / kD][e % kD] = bf16_to_f32(q[((size_t)rho * H + h * G + e / kD) * kD + e % kD]) * scale_log2;
  __syncthreads();

  float m[G], l[G], o[G][16];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) o[g][e] = 0.f;
  }
  const int pi = split * kPagesPerSplit + warp;
  if (pi < cnt) {
    const int lp = sel[((size_t)rho * Hk + h) * (top_k + 1) + pi];
    const int phys = bt[(size_t)rho * max_pages + lp];
    const int valid = min(64, n - lp * 64);
    const uint16_t *kp = kc + ((size_t)phys * Hk + h) * 64 * kD;
    const uint16_t *vp = vc + ((size_t)phys * Hk + h) * 64 * kD;
    float s[16][G];
#pragma unroll
    for (int it = 0; it < 16; ++it) {
      const int tok = it * 4 + tk;
      const uint4 *kr = reinterpret_cast<const uint4 *>(kp + (size_t)tok * kD + dl * 16);
      const uint4 a = __ldg(kr), b = __ldg(kr + 1);
      float kv[16];
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        kv[2 * e] = __uint_as_float(w[e] << 16);
        kv[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (g < G) {
          float acc = 0.f;
#pragma unroll
          for (int e = 0; e < 16; ++e) acc = fmaf(qs[g][dl * 16 + e], kv[e], acc);
          acc += __shfl_xor_sync(0xffffffffu, acc, 1);
          acc += __shfl_xor_sync(0xffffffffu, acc, 2);
          acc += __shfl_xor_sync(0xffffffffu, acc, 4);
          s[it][g] = tok < valid ? acc : -INFINITY;
        }
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (g < G) {
        float mx = -INFINITY;
#pragma unroll
        for (int it = 0; it < 16; ++it) mx = fmaxf(mx, s[it][g]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        m[g] = mx;  // one page per warp: the first tile sets the running max
        float sum = 0.f;
#pragma unroll
        for (int it = 0; it < 16; ++it) {
          s[it][g] = fast_exp2(s[it][g] - mx);
          sum += s[it][g];
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 8);
        sum += __shfl_xor_sync(0xffffffffu, sum, 16);
        l[g] = sum;
      }
    }
#pragma unroll
    for (int it = 0; it < 16; ++it) {
      const int tok = it * 4 + tk;
      const uint4 *vr = reinterpret_cast<const uint4 *>(vp + (size_t)tok * kD + dl * 16);
      const uint4 a = __ldg(vr), b = __ldg(vr + 1);
      float vv[16];
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        vv[2 * e] = __uint_as_float(w[e] << 16);
        vv[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
      }
#pragma unroll
      for (int g = 0; g < G; ++g)
        if (g < G)
#pragma unroll
          for (int e = 0; e < 16; ++e) o[g][e] = fmaf(s[it][g], vv[e], o[g][e]);
    }
    // sum the four token groups
#pragma unroll
    for (int g = 0; g < G; ++g)
      if (g < G)
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], 8);
          o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], 16);
        }
  }
  // Combine the warps of this split (eqs.(3)-(5)) through shared memory.
  if (lane == 0)
    for (int g = 0; g < G; ++g) {
      wm[warp][g] = m[g];
      wl[warp][g] = l[g];
    }
  if (tk == 0)
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < 16; ++e) wo[warp][g][dl * 16 + e] = o[g][e];
  __syncthreads();
  const size_t base = (((size_t)rho * Hk + h) * nsplit + split) * G;
  for (int idx = threadIdx.x; idx < G * kD; idx += blockDim.x) {
    const int g = idx / kD, c = idx % kD;
    float M = -INFINITY;
    for (int w = 0; w < kPagesPerSplit; ++w) M = fmaxf(M, wm[w][g]);
    float Lsum = 0.f, acc = 0.f;
    if (M != -INFINITY)
      for (int w = 0; w < kPagesPerSplit; ++w) {
        if (wm[w][g] == -INFINITY) continue;
        const float f = fast_exp2(wm[w][g] - M);
        Lsum += f * wl[w][g];
        acc += f * wo[w][g][c];
      }
    part_o[(base + g) * kD + c] = acc;
    if (c == 0) {
      part_ml[(base + g) * 2] = M;
      part_ml[(base + g) * 2 + 1] = Lsum;
    }
  }
}

// grid (H_kv, R), 128 threads: combine the splits of every query head of the group.
__global__ void __launch_bounds__(128) dec_merge_kernel(
    const float *__restrict__ part_ml, const float *__restrict__ part_o, uint16_t *__restrict__ o,
    float *__restrict__ lse, int H, int Hk, int nsplit) {
  const int rho = blockIdx.y, h = blockIdx.x;
  const int G = H / Hk;
  for (int idx = threadIdx.x; idx < G * kD; idx += blockDim.x) {
    const int g = idx / kD, c = idx % kD;
    const size_t base = ((size_t)rho * Hk + h) * nsplit;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, part_ml[((base + s) * G + g) * 2]);
    float Lsum = 0.f, acc = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float ms = part_ml[((base + s) * G + g) * 2];
      if (ms == -INFINITY) continue;
      const float f = fast_exp2(ms - M);
      Lsum += f * part_ml[((base + s) * G + g) * 2 + 1];
      acc += f * part_o[((base + s) * G + g) * kD + c];
    }
    const int hq = h * G + g;
    const __nv_bfloat16 ob = __float2bfloat16_rn(acc / Lsum);
    o[((size_t)rho * H + hq) * kD + c] = *reinterpret_cast<const uint16_t *>(&ob);
    if (lse != nullptr && c == 0) lse[(size_t)rho * H + hq] = (M + log2f(Lsum)) * 0.6931471805599453f;
  }
}

int num_splits(const bsa_decode_shape_t &s) {
  return (s.top_k + 1 + kPagesPerSplit - 1) / kPagesPerSplit;
}

}  // namespace

size_t decode_workspace_bytes(const bsa_decode_shape_t &s) {
  const size_t G = (size_t)(s.num_heads / s.num_kv_heads);
  const size_t pairs = (size_t)s.num_reqs * s.num_kv_heads;
  const size_t scores = pairs * s.max_pages_per_req * sizeof(float);
  const size_t ml = pairs * num_splits(s) * G * 2 * sizeof(float);
  const size_t ob = pairs * num_splits(s) * G * kD * sizeof(float);
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return up(scores) + up(ml) + up(ob);
}

cudaError_t launch_decode(const bsa_decode_shape_t &s, const void *q, const void *k_cache,
                          const void *v_cache, const float *page_summ,
                          const int32_t *block_table, const int32_t *context_lens, float scale,
                          void *o, float *lse, int32_t *sel, int32_t *sel_counts,
                          int32_t *dev_status, void *ws, cudaStream_t st) {
  (void)dev_status;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const int G = s.num_heads / s.num_kv_heads;
  const int nsplit = num_splits(s);
  const size_t pairs = (size_t)s.num_reqs * s.num_kv_heads;
  char *w = static_cast<char *>(ws);
  float *scores = reinterpret_cast<float *>(w);
  w += up(pairs * s.max_pages_per_req * sizeof(float));
  float *part_ml = reinterpret_cast<float *>(w);
  w += up(pairs * nsplit * G * 2 * sizeof(float));
  float *part_o = reinterpret_cast<float *>(w);

  const uint16_t *qb = static_cast<const uint16_t *>(q);
  dec_score_kernel<<<dim3((s.max_pages_per_req + 63) / 64, s.num_kv_heads, s.num_reqs),
                     kScoreThreads, 0, st>>>(qb, page_summ, block_table, context_lens, scores,
                                             s.num_heads, s.num_kv_heads, s.max_pages_per_req);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t sm = (size_t)s.max_pages_per_req * sizeof(uint32_t);
  if (sm > 40 * 1024) {
    e = cudaFuncSetAttribute(dec_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm);
    if (e != cudaSuccess) return e;
  }
  dec_select_kernel<<<dim3(s.num_kv_heads, s.num_reqs), kSelThreads, sm, st>>>(
      scores, context_lens, sel, sel_counts, s.num_kv_heads, s.max_pages_per_req, s.top_k);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const float scale_log2 = scale * 1.4426950408889634f;
  const dim3 agrid(nsplit, s.num_kv_heads, s.num_reqs);
#define BSA_DEC_ATTN(GG)                                                                      \
  dec_attn_kernel<GG><<<agrid, kPagesPerSplit * 32, 0, st>>>(                                 \
      qb, static_cast<const uint16_t *>(k_cache), static_cast<const uint16_t *>(v_cache),     \
      block_table, context_lens, sel, sel_counts, scale_log2, part_ml, part_o, s.num_heads,   \
      s.num_kv_heads, s.max_pages_per_req, s.top_k, nsplit)
  switch (G) {
    case 1: BSA_DEC_ATTN(1); break;
    case 2: BSA_DEC_ATTN(2); break;
    case 4: BSA_DEC_ATTN(4); break;
    case 8: BSA_DEC_ATTN(8); break;
    default: return cudaErrorInvalidValue;
  }
#undef BSA_DEC_ATTN
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dec_merge_kernel<<<dim3(s.num_kv_heads, s.num_reqs), 128, 0, st>>>(
      part_ml, part_o, static_cast<uint16_t *>(o), lse, s.num_heads, s.num_kv_heads, nsplit);
  return cudaGetLastError();
}

}  // namespace bsa
