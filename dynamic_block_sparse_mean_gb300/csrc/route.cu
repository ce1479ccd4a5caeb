// a2 + a3: the block router of "2.1 · 粗粒度选择" §2.1.
//   scores  g[i,h,r,j] = max over the group's query heads and the valid tokens
//           of block r of q . c_j, j < r (eq.(6), pool = max; unscaled)
//   select  forced diagonal (+ sink), then top-k or the clamped threshold of
//           eq.(7); ranking (score desc, index asc); rows deduplicated and
//           sorted ascending (eq.(1) address order).
// Scores are fp32 FFMA dot products (fp32-accurate: the selection is compared
// bit-exactly, up to a 1e-5 tie band, with a float64 oracle).
#include <algorithm>

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

BSA_DEV float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

struct SelectParams {
  float *S;
  const int32_t *cu, *qoff;
  int32_t *J, *counts;
  int Nq, Nk, Hk, b, mode, k_max, k_min;
  float tau_delta;
  int force_sink, window, num_global;
  const int32_t *global_blocks;
  // screen: S holds q . (c_hi + c_mid); null Qn means S is exact
  const float *Qn, *cn, *rn;
  const uint16_t *Q, *C3;
  size_t c3_rows;
  int T, G, d;
  // rows the bounds cannot settle: a queue, and per row the candidates to rescore
  int32_t *queue_len;  // zeroed by the split kernel
  int32_t *queue;      // [rows]
  int32_t *nlist;      // [rows]: candidates listed, or -1: every j < r
  int32_t *rlist;      // [rows][kCap]
};

constexpr uint8_t kTaken = 1, kExact = 2, kIn = 4, kOut = 8;
constexpr int kCap = 64;       // candidates listed per row; more: the whole row is rescored
constexpr int kChunk = 16;     // candidates per rescoring pass over the row's queries
constexpr int kRescoreThreads = 256;

// One histogram pass of a warp radix select over the candidates' order keys
// (candidates not taken and not already decided in / out): returns (bin, keys
// above the bin, keys in the bin) for the `remaining`-th key.
template <typename KeyF>
BSA_DEV int3 radix_pass(KeyF key, const uint8_t *flags, int r, uint32_t prefix, uint32_t mask,
                        int shift, int remaining, int32_t *hist, int lane) {
  for (int e = lane; e < 256; e += 32) hist[e] = 0;
  __syncwarp();
  for (int j = lane; j < r; j += 32)
    if (!(flags[j] & (kTaken | kIn | kOut))) {
      const uint32_t kk = key(j);
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
  bin = __shfl_sync(0xffffffffu, bin, max(src, 0));
  above = __shfl_sync(0xffffffffu, above, max(src, 0));
  inbin = __shfl_sync(0xffffffffu, inbin, max(src, 0));
  __syncwarp();  // every lane has read hist before the next pass clears it
  return make_int3(max(bin, 0), above, inbin);
}

// The order key of the k-th largest candidate key (1 <= k <= candidates).
template <typename KeyF>
BSA_DEV uint32_t kth_key(KeyF key, const uint8_t *flags, int r, int k, int32_t *hist, int lane) {
  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    const int3 res = radix_pass(key, flags, r, prefix, mask, shift, remaining, hist, lane);
    remaining -= res.y;
    prefix |= (uint32_t)res.x << shift;
    mask |= 0xFFu << shift;
  }
  return prefix;
}

BSA_DEV float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

BSA_DEV int warp_sum(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// A router row: (i, h, qb) of the flattened row id, the logical block r it
// selects for (qb, or in a chunked prefill qb + the blocks cached before the
// chunk), and its query tokens.
struct SelRow {
  int row, i, h, qb, r, s0, n, nvalid;
  bool live;
};

BSA_DEV SelRow sel_row(const SelectParams &p, int row) {
  SelRow x;
  x.row = row;
  x.qb = row % p.Nq;
  x.i = row / (p.Nq * p.Hk);
  x.h = (row / p.Nq) % p.Hk;
  x.s0 = p.cu[x.i];
  x.n = p.cu[x.i + 1] - x.s0;
  const int nb = (x.n + p.b - 1) / p.b;
  x.r = x.qb;
  bool ok = true;
  if (p.qoff != nullptr) {
    const int pre = p.qoff[x.i];
    ok = chunk_ok(pre, x.n, p.b, p.Nk);
    if (ok) x.r += pre / p.b;
  }
  x.live = ok && x.qb < nb;
  x.nvalid = min(p.b, x.n - x.qb * p.b);
  return x;
}

// Shared memory of a selecting warp: Nk scores, Nk bounds, a 256-bin histogram,
// Nk flag bytes.
struct SelSmem {
  float *sc, *eb;
  int32_t *hist;
  uint8_t *flags;
};

BSA_DEV SelSmem sel_smem(uint8_t *sm, int Nk) {
  SelSmem m;
  m.sc = reinterpret_cast<float *>(sm);
  m.eb = m.sc + Nk;
  m.hist = reinterpret_cast<int32_t *>(m.eb + Nk);
  m.flags = reinterpret_cast<uint8_t *>(m.hist + 256);
  return m;
}

// Loads the row's scores and, screened, their bounds e_j = Qn (|c - c_hi - c_mid| +
// 2^-15 |c|) (Cauchy-Schwarz for the dropped part; 2d fp32 accumulations of products
// of norm |q| |c| for the rest), and marks the forced blocks F_r (union routing:
// local window, global list, sink; the diagonal r is never a candidate) taken, so
// the dynamic choice never spends budget on them; a block named twice is kept
// once.  Returns the number of forced history blocks (j < r).
BSA_DEV int sel_load(const SelectParams &p, const SelRow &x, const SelSmem &m, bool screen,
                     int lane) {
  const float *Srow = p.S + (size_t)x.row * p.Nk;
  const size_t crow = ((size_t)x.i * p.Hk + x.h) * p.Nk;
  const float qn = screen ? p.Qn[x.row] : 0.f;
  const int wlo = max(0, x.r - max(1, p.window) + 1);
  for (int j = lane; j < x.r; j += 32) {
    m.sc[j] = Srow[j];
    const bool forced = j >= wlo || (p.force_sink && j == 0);
    m.eb[j] = screen ? 1.001f * qn * (p.rn[crow + j] + 3.1e-5f * p.cn[crow + j]) : 0.f;
    m.flags[j] = (forced ? kTaken : 0) | (screen ? 0 : kExact);
  }
  __syncwarp();
  if (lane < p.num_global) {
    const int gb = p.global_blocks[lane];
    if (gb >= 0 && gb < x.r) m.flags[gb] |= kTaken;
  }
  __syncwarp();
  int nhist = 0;
  for (int j = lane; j < x.r; j += 32) nhist += (m.flags[j] & kTaken) ? 1 : 0;
  return warp_sum(nhist);
}

// Dynamic picks for a count |A| of eq.(7): k_r = min(k_max, max(k_min, |F| + |A|),
// |F| + |candidates|), minus the forced blocks, clamped to the candidates.
BSA_DEV int k_for(const SelectParams &p, int a, int nforced, int ncand) {
  const int k_r = min(p.k_max, min(max(p.k_min, nforced + a), nforced + ncand));
  return max(0, min(k_r - nforced, ncand));
}

// Selection of one row from scores that are exact where it matters: every
// candidate is either exact (lo = hi = score) or settled by its bounds.  Threshold
// mode: tau = (max candidate score) - delta from the exact maximum when every
// candidate that may hold it is exact, else from the upper bound (then no candidate
// straddles tau, so the count is the same).  Top-k: candidates whose lower end is
// above the (k+1)-th upper end are in, those whose upper end is below the k-th lower
// end out, the rest (exact) compete under (score desc, index asc) by a radix select
// (8 bits per pass from the top; it stops once the bin of the k-th key holds exactly
// the keys still needed).  Writes J (ascending, -1 padded) and the count.
BSA_DEV void sel_finish(const SelectParams &p, const SelRow &x, const SelSmem &m, int nhist,
                        int lane) {
  const int r = x.r;
  float *sc = m.sc;
  const float *eb = m.eb;
  uint8_t *flags = m.flags;
  const int nforced = nhist + 1;  // + the diagonal
  const int ncand = r - nhist;
  auto lo = [&](int j) { return (flags[j] & kExact) ? sc[j] : __fsub_rd(sc[j], eb[j]); };
  auto hi = [&](int j) { return (flags[j] & kExact) ? sc[j] : __fadd_ru(sc[j], eb[j]); };
  bool all_exact = true;
  for (int j = lane; j < r; j += 32)
    if (!(flags[j] & (kTaken | kExact))) all_exact = false;
  all_exact = __all_sync(0xffffffffu, all_exact);

  int k_dyn;
  if (p.mode == BSA_ROUTE_TOPK) {
    k_dyn = max(0, min(p.k_max - nforced, ncand));
  } else {
    float ml = -INFINITY, mh = -INFINITY;
    for (int j = lane; j < r; j += 32)
      if (!(flags[j] & kTaken)) {
        ml = fmaxf(ml, lo(j));
        mh = fmaxf(mh, hi(j));
      }
    ml = warp_max(ml);
    mh = warp_max(mh);
    bool max_exact = true;
    float mx = -INFINITY;
    for (int j = lane; j < r; j += 32)
      if (!(flags[j] & kTaken) && hi(j) >= ml) {
        if (flags[j] & kExact) mx = fmaxf(mx, sc[j]);
        else max_exact = false;
      }
    max_exact = __all_sync(0xffffffffu, max_exact);
    mx = warp_max(mx);
    const float tau = max_exact ? mx - p.tau_delta : __fsub_ru(mh, p.tau_delta);
    int a = 0;
    for (int j = lane; j < r; j += 32)
      if (!(flags[j] & kTaken) && lo(j) >= tau) ++a;
    k_dyn = k_for(p, warp_sum(a), nforced, ncand);
  }

  if (!all_exact && k_dyn > 0 && k_dyn < ncand) {
    const uint32_t t_lo = kth_key([&](int j) { return order_key(lo(j)); }, flags, r, k_dyn, m.hist, lane);
    const uint32_t t_hi = kth_key([&](int j) { return order_key(hi(j)); }, flags, r, k_dyn + 1, m.hist, lane);
    for (int j = lane; j < r; j += 32)
      if (!(flags[j] & kTaken)) {
        if (order_key(lo(j)) > t_hi) flags[j] |= kIn;
        else if (order_key(hi(j)) < t_lo) flags[j] |= kOut;
      }
    __syncwarp();
  }
  // The pool still to choose from (candidates neither in nor out; exact, or every
  // candidate when the scores are exact) and the picks left for it.
  int n_in = 0, n_out = 0;
  for (int j = lane; j < r; j += 32) {
    n_in += (flags[j] & kIn) ? 1 : 0;
    n_out += (flags[j] & kOut) ? 1 : 0;
  }
  n_in = warp_sum(n_in);
  n_out = warp_sum(n_out);
  const int npool = ncand - n_in - n_out;
  const int kp = k_dyn - n_in;

  uint32_t prefix = 0, mask = 0;
  int remaining = kp;  // pool picks still to place at or below the current bin
  if (kp > 0 && kp < npool) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      const int3 res = radix_pass([&](int j) { return order_key(sc[j]); }, flags, r, prefix, mask,
                                  shift, remaining, m.hist, lane);
      remaining -= res.y;
      prefix |= (uint32_t)res.x << shift;
      mask |= 0xFFu << shift;
      // the k-th key's bin holds exactly the keys still needed: all are picked
      if (res.z == remaining) break;
    }
  }
  // One ordered pass: forced blocks, sure picks, pool candidates above the k-th
  // key's bin and the first `remaining` inside it (ties to the lower block index).
  int32_t *Jrow = p.J + (size_t)x.row * p.k_max;
  int w = 0, eq_seen = 0;
  for (int j0 = 0; j0 <= r; j0 += 32) {
    const int j = j0 + lane;
    bool keep = false, eq = false;
    if (j < r) {
      if (flags[j] & (kTaken | kIn)) {
        keep = true;
      } else if (flags[j] & kOut) {
        keep = false;
      } else if (kp >= npool) {
        keep = kp > 0;
      } else if (kp > 0) {
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
  for (int e = w + lane; e < p.k_max; e += 32) Jrow[e] = -1;
  if (lane == 0) p.counts[x.row] = w;
}

BSA_DEV void sel_empty(const SelectParams &p, int row, int lane) {
  int32_t *Jrow = p.J + (size_t)row * p.k_max;
  for (int e = lane; e < p.k_max; e += 32) Jrow[e] = -1;
  if (lane == 0) p.counts[row] = 0;
}

// Phase 1, one warp per router row.  Exact scores: the selection.  Screened
// scores: each candidate's exact score lies in [S - e, S + e] (rounded outward).
// Threshold mode bounds tau = (max) - delta by [max lo - delta, max hi - delta] and
// the count |A| by the candidates surely above / possibly above it, hence the picks
// k by [k_lo, k_hi].  For every such k, a candidate whose lower end exceeds the
// (k_lo+1)-th largest upper end is surely picked, one whose upper end is below the
// k_hi-th largest lower end surely not.  When every candidate is settled (and |A|
// is) the row is finished here; otherwise the unsettled candidates, plus in
// threshold mode the ones that may hold the maximum or straddle tau, are listed
// and the row is queued: after they are rescored exactly, every candidate of the
// row is exact or settled for the actual k (intervals only shrink, so the settled
// ones stay settled).
__global__ void __launch_bounds__(32) route_plan_kernel(const SelectParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int lane = threadIdx.x;
  grid_dep_wait();  // the scores come from the previous launch
  const SelRow x = sel_row(p, blockIdx.x);
  if (!x.live) {
    sel_empty(p, x.row, lane);
    grid_dep_launch();
    return;
  }
  const SelSmem m = sel_smem(smem, p.Nk);
  const bool screen = p.Qn != nullptr;
  const int nhist = sel_load(p, x, m, screen, lane);
  if (screen) {
    const int r = x.r, nforced = nhist + 1, ncand = r - nhist;
    const float *sc = m.sc, *eb = m.eb;
    const uint8_t *flags = m.flags;
    auto lo = [&](int j) { return __fsub_rd(sc[j], eb[j]); };
    auto hi = [&](int j) { return __fadd_ru(sc[j], eb[j]); };
    int k_lo, k_hi;
    bool tau_open = false;
    float ml = -INFINITY, tau_l = 0.f, tau_h = 0.f;
    if (p.mode == BSA_ROUTE_TOPK) {
      k_lo = k_hi = max(0, min(p.k_max - nforced, ncand));
    } else {
      float mh = -INFINITY;
      for (int j = lane; j < r; j += 32)
        if (!(flags[j] & kTaken)) {
          ml = fmaxf(ml, lo(j));
          mh = fmaxf(mh, hi(j));
        }
      ml = warp_max(ml);
      mh = warp_max(mh);
      tau_l = __fsub_rd(ml, p.tau_delta);
      tau_h = __fsub_ru(mh, p.tau_delta);
      int a_lo = 0, a_hi = 0;
      for (int j = lane; j < r; j += 32)
        if (!(flags[j] & kTaken)) {
          a_lo += lo(j) >= tau_h ? 1 : 0;
          a_hi += hi(j) >= tau_l ? 1 : 0;
        }
      a_lo = warp_sum(a_lo);
      a_hi = warp_sum(a_hi);
      k_lo = k_for(p, a_lo, nforced, ncand);
      k_hi = k_for(p, a_hi, nforced, ncand);
      // tau matters only when the candidates straddling it change the picks
      tau_open = k_lo != k_hi;
    }
    // Settled bounds for every k in [k_lo, k_hi]: the (k_lo+1)-th largest upper end
    // and the k_hi-th largest lower end (resolved to the last bit: a coarser bound
    // would leave many more candidates to rescore).
    uint32_t t_in = 0xFFFFFFFFu, t_out = 0u;  // in: order_key(lo) > t_in; out: order_key(hi) < t_out
    bool none_in = false;
    if (k_hi == 0) {
      t_out = 0xFFFFFFFFu;  // nothing can be picked: every candidate is out
      none_in = true;
    } else if (k_lo < ncand) {
      t_in = kth_key([&](int j) { return order_key(hi(j)); }, flags, r, k_lo + 1, m.hist, lane);
      if (k_hi < ncand)
        t_out = kth_key([&](int j) { return order_key(lo(j)); }, flags, r, k_hi, m.hist, lane);
    } else {
      t_in = 0u;  // k_lo >= ncand: every candidate is picked
    }
    // list what is not settled
    int32_t *lst = p.rlist + (size_t)x.row * kCap;
    int n = 0;
    for (int j0 = 0; j0 < r; j0 += 32) {
      const int j = j0 + lane;
      bool want = false;
      if (j < r && !(flags[j] & kTaken)) {
        const bool in = !none_in && order_key(lo(j)) > t_in;
        const bool out = k_hi == 0 || order_key(hi(j)) < t_out;
        want = !(in || out) && !(k_lo >= ncand);
        if (tau_open && (hi(j) >= ml || (lo(j) < tau_h && hi(j) >= tau_l))) want = true;
      }
      const unsigned mw = __ballot_sync(0xffffffffu, want);
      const int pos = n + __popc(mw & ((1u << lane) - 1u));
      if (want && pos < kCap) lst[pos] = j;
      n += __popc(mw);
    }
    if (n > 0) {
      if (lane == 0) {
        p.nlist[x.row] = n <= kCap ? n : -1;
        p.queue[atomicAdd(p.queue_len, 1)] = x.row;
      }
      grid_dep_launch();
      return;
    }
    // Every candidate settled (so k_lo = k_hi): the row is the forced blocks, the
    // sure picks and the diagonal, in one ordered pass.
    int32_t *Jrow = p.J + (size_t)x.row * p.k_max;
    int w = 0;
    for (int j0 = 0; j0 <= r; j0 += 32) {
      const int j = j0 + lane;
      bool keep = j == r;
      if (j < r) keep = (flags[j] & kTaken) || (!none_in && order_key(lo(j)) > t_in);
      const unsigned km = __ballot_sync(0xffffffffu, keep);
      if (keep && w + __popc(km & ((1u << lane) - 1u)) < p.k_max)
        Jrow[w + __popc(km & ((1u << lane) - 1u))] = j;
      w += __popc(km);
    }
    for (int e = w + lane; e < p.k_max; e += 32) Jrow[e] = -1;
    if (lane == 0) p.counts[x.row] = min(w, p.k_max);
    grid_dep_launch();
    return;
  }
  sel_finish(p, x, m, nhist, lane);
  grid_dep_launch();
}

// Phase 2: exact scores of the listed candidates of every queued row, the max
// over the row's valid query rows of q . c_j in fp32 FFMA with c_j = lo + mid + hi
// from the split planes.  A CTA takes a queued row; its 256 threads each take
// every 256th query row (all loads of a row issued before use) against up to
// kChunk staged candidates, then the per-candidate maxima are reduced across the
// CTA and written over the screened scores in S.
template <int D>
__global__ void __launch_bounds__(kRescoreThreads) route_rescore_kernel(const SelectParams p) {
  __shared__ __align__(16) float cbuf[kChunk * D];
  __shared__ float red[kRescoreThreads / 32][kChunk];
  __shared__ int ids[kChunk];
  grid_dep_wait();  // the queue comes from the previous launch
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int nq = *p.queue_len;
  const size_t plane = p.c3_rows * D;
  for (int qi = blockIdx.x; qi < nq; qi += gridDim.x) {
    const SelRow x = sel_row(p, p.queue[qi]);
    const int nl = p.nlist[x.row];
    const int total = nl < 0 ? x.r : nl;  // -1: every j < r
    const int32_t *lst = p.rlist + (size_t)x.row * kCap;
    const size_t crow = ((size_t)x.i * p.Hk + x.h) * p.Nk;
    const int nrows = p.G * x.nvalid;
    for (int c0 = 0; c0 < total; c0 += kChunk) {
      const int nc = min(kChunk, total - c0);
      if (threadIdx.x < nc) ids[threadIdx.x] = nl < 0 ? c0 + threadIdx.x : lst[c0 + threadIdx.x];
      __syncthreads();
      for (int e = threadIdx.x; e < nc * D; e += kRescoreThreads) {
        const size_t at = (crow + ids[e / D]) * D + e % D;
        cbuf[e] = bf16_to_f32(p.C3[2 * plane + at]) + bf16_to_f32(p.C3[plane + at]) +
                  bf16_to_f32(p.C3[at]);
      }
      __syncthreads();
      float best[kChunk];
#pragma unroll
      for (int c = 0; c < kChunk; ++c) best[c] = -INFINITY;
      for (int rho = threadIdx.x; rho < nrows; rho += kRescoreThreads) {
        const int hq = x.h * p.G + rho / x.nvalid, t = rho % x.nvalid;
        const uint4 *qrow = reinterpret_cast<const uint4 *>(
            p.Q + ((size_t)hq * p.T + x.s0 + x.qb * p.b + t) * D);
        uint4 u[D / 8];
#pragma unroll
        for (int k = 0; k < D / 8; ++k) u[k] = __ldg(qrow + k);
        float acc[kChunk];
#pragma unroll
        for (int c = 0; c < kChunk; ++c) acc[c] = 0.f;
#pragma unroll
        for (int k = 0; k < D / 8; ++k) {
          const uint32_t w[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
          float qv[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            qv[2 * e] = __uint_as_float(w[e] << 16);
            qv[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
          }
#pragma unroll
          for (int c = 0; c < kChunk; ++c)
            if (c < nc) {
              const float4 a = *reinterpret_cast<const float4 *>(cbuf + c * D + 8 * k);
              const float4 b4 = *reinterpret_cast<const float4 *>(cbuf + c * D + 8 * k + 4);
              float v = acc[c];
              v = fmaf(qv[0], a.x, v);
              v = fmaf(qv[1], a.y, v);
              v = fmaf(qv[2], a.z, v);
              v = fmaf(qv[3], a.w, v);
              v = fmaf(qv[4], b4.x, v);
              v = fmaf(qv[5], b4.y, v);
              v = fmaf(qv[6], b4.z, v);
              v = fmaf(qv[7], b4.w, v);
              acc[c] = v;
            }
        }
#pragma unroll
        for (int c = 0; c < kChunk; ++c) best[c] = fmaxf(best[c], acc[c]);
      }
#pragma unroll
      for (int c = 0; c < kChunk; ++c) {
        const float v = warp_max(best[c]);
        if (lane == 0) red[warp][c] = v;
      }
      __syncthreads();
      if (threadIdx.x < nc) {
        float v = red[0][threadIdx.x];
#pragma unroll
        for (int w8 = 1; w8 < kRescoreThreads / 32; ++w8) v = fmaxf(v, red[w8][threadIdx.x]);
        p.S[(size_t)x.row * p.Nk + ids[threadIdx.x]] = v;
      }
      __syncthreads();
    }
  }
  grid_dep_launch();
}

// Phase 3, one warp per queued row: the listed candidates are exact now, every
// other one is settled by its bounds, and the row is selected.
__global__ void __launch_bounds__(32) route_final_kernel(const SelectParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int lane = threadIdx.x;
  grid_dep_wait();  // the rescored scores come from the previous launch
  const int nq = *p.queue_len;
  const SelSmem m = sel_smem(smem, p.Nk);
  for (int qi = blockIdx.x; qi < nq; qi += gridDim.x) {
    const SelRow x = sel_row(p, p.queue[qi]);
    const int nhist = sel_load(p, x, m, true, lane);
    const int nl = p.nlist[x.row];
    const int32_t *lst = p.rlist + (size_t)x.row * kCap;
    if (nl < 0) {
      for (int j = lane; j < x.r; j += 32) m.flags[j] |= kExact;
    } else {
      for (int e = lane; e < nl; e += 32) m.flags[lst[e]] |= kExact;
    }
    __syncwarp();
    sel_finish(p, x, m, nhist, lane);
    __syncwarp();
  }
  grid_dep_launch();
}

}  // namespace

// Workspace: [bf16 split of C and the screen's norms, BF16 path only][score
// matrix, unless the caller passes its own `scores` buffer][BF16 screen: the queue
// of rows to rescore (length, rows), per row the listed count and kCap candidate
// ids].  With a cache (chunked prefill) the summaries come from its pages and
// score rows hold N_k entries.
static size_t up256r(size_t x) { return (x + 255) & ~(size_t)255; }

size_t route_workspace_bytes(const bsa_shape_t &s, const bsa_route_params_t &,
                             const bsa_kv_cache_t *cache) {
  const size_t split = s.dtype == BSA_BF16 ? route_tc_workspace_bytes(s, cache) : 0;
  const size_t Nk = cache != nullptr ? cache->max_context_blocks : s.max_blocks;
  const size_t rows = (size_t)s.num_seqs * s.num_kv_heads * s.max_blocks;
  const size_t queue = s.dtype == BSA_BF16
                           ? up256r(4) + up256r(rows * 4) + up256r(rows * 4) + up256r(rows * kCap * 4)
                           : 0;
  return split + up256r(rows * Nk * sizeof(float)) + queue;
}

size_t route_select_smem(int Nk) { return (size_t)Nk * 9 + 256 * 4 + 16; }

bool route_select_fits(int Nk, int) { return route_select_smem(Nk) <= 227 * 1024; }

cudaError_t launch_route(const bsa_shape_t &s, const bsa_route_params_t &p, const void *Q,
                         const float *C, const bsa_kv_cache_t *cache, int32_t *J,
                         int32_t *counts, float *scores, int32_t *dev_status, void *ws,
                         cudaStream_t st) {
  const size_t split = s.dtype == BSA_BF16 ? route_tc_workspace_bytes(s, cache) : 0;
  const int Nk = cache != nullptr ? cache->max_context_blocks : s.max_blocks;
  const int rows = s.num_seqs * s.num_kv_heads * s.max_blocks;
  char *w = static_cast<char *>(ws) + split;
  float *S = scores != nullptr ? scores : reinterpret_cast<float *>(w);
  w += up256r((size_t)rows * Nk * sizeof(float));
  const int G = s.num_heads / s.num_kv_heads;
  const dim3 grid(s.max_blocks, s.num_kv_heads, s.num_seqs);
  // The BF16 path screens when asked to, or automatically when a row pools at least
  // 512 query rows (the measured break-even: below it the per-row bound and
  // selection work costs more than the third of the score products it saves),
  // unless the caller asked for the score matrix, which is then computed exactly
  // (it is a debugging output compared entry by entry).
  const bool screen = s.dtype == BSA_BF16 && scores == nullptr &&
                      (p.screen > 0 || (p.screen == 0 && G * s.block >= 512));
  SelectParams sp;
  sp.S = S;
  sp.cu = s.cu_seqlens;
  sp.qoff = cache != nullptr ? cache->prefix_lens : nullptr;
  sp.J = J;
  sp.counts = counts;
  sp.Nq = s.max_blocks;
  sp.Nk = Nk;
  sp.Hk = s.num_kv_heads;
  sp.b = s.block;
  sp.mode = p.mode;
  sp.k_max = p.k_max;
  sp.k_min = p.k_min;
  sp.tau_delta = p.tau_delta;
  sp.force_sink = p.force_sink;
  sp.window = p.window;
  sp.num_global = p.num_global;
  sp.global_blocks = p.global_blocks;
  sp.Qn = sp.cn = sp.rn = nullptr;
  sp.Q = sp.C3 = nullptr;
  sp.c3_rows = 0;
  sp.T = s.total_tokens;
  sp.G = G;
  sp.d = s.head_dim;
  sp.queue_len = sp.queue = sp.nlist = sp.rlist = nullptr;
  if (s.dtype == BSA_BF16) {
    sp.queue_len = reinterpret_cast<int32_t *>(w);
    w += up256r(4);
    sp.queue = reinterpret_cast<int32_t *>(w);
    w += up256r((size_t)rows * 4);
    sp.nlist = reinterpret_cast<int32_t *>(w);
    w += up256r((size_t)rows * 4);
    sp.rlist = reinterpret_cast<int32_t *>(w);
  }
  cudaError_t e;
  if (s.dtype == BSA_BF16) {
    e = launch_route_scores_tc(s, Q, C, cache, S, screen, ws, sp.queue_len, dev_status, st);
    if (e != cudaSuccess) return e;
  } else {
    route_scores_kernel<float><<<grid, kThreads, 0, st>>>(
        static_cast<const float *>(Q), C, s.cu_seqlens, S, s.total_tokens, s.max_blocks,
        s.num_kv_heads, G, s.head_dim, s.block);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (screen) {
    const RouteScreen rs = route_tc_screen(s, cache, ws);
    sp.Qn = rs.Qn;
    sp.cn = rs.cn;
    sp.rn = rs.rn;
    sp.C3 = rs.C3;
    sp.c3_rows = rs.c3_rows;
    sp.Q = static_cast<const uint16_t *>(Q);
  }
  const size_t sm = route_select_smem(Nk);
  if (sm > 48 * 1024) {
    if ((e = cudaFuncSetAttribute(route_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)sm)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(route_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)sm)) != cudaSuccess)
      return e;
  }
  e = launch_dependent(route_plan_kernel, dim3(rows), dim3(32), sm, st, sp);
  if (e != cudaSuccess || !screen) return e;
  const int persistent = std::max(1, std::min(rows, 2 * num_sms()));
  e = s.head_dim == 128
          ? launch_dependent(route_rescore_kernel<128>, dim3(persistent), dim3(kRescoreThreads), 0,
                             st, sp)
          : launch_dependent(route_rescore_kernel<64>, dim3(persistent), dim3(kRescoreThreads), 0,
                             st, sp);
  if (e != cudaSuccess) return e;
  return launch_dependent(route_final_kernel, dim3(std::max(1, std::min(rows, 8 * num_sms()))),
                          dim3(32), sm, st, sp);
}

}  // namespace bsa
