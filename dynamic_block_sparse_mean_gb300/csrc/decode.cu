// a6: paged sparse decode ("2.1 · 粗粒度选择" §2.2: decode reads the block
// summaries, O(N_k d_r), then only the selected K/V; §3.1: the router emits
// logical page ids, the block table maps them to physical pages when the
// attention runs).  Four launches, all HBM-bound:
//   score   q . page summary for the complete pages 0 .. L-2 of each
//           (request, KV head), max over the group's query heads
//   select  exact top-k by (score desc, index asc) via a 4-pass radix select,
//           plus the last page L-1, written in ascending order
//   attn    tensor cores: each unit of two selected pages gives a partial
//           softmax (m, l, u) per query head (eqs.(3)-(5) within the unit)
//   merge   combines the unit partials of a (request, KV head) into o and lse
// Request lengths are checked on the device before any indexed access: a length
// of 0 is an idle slot of a padded batch (no pages kept, o = 0, lse = -inf, no
// error); a negative length or one past max_pages * 64 is BSA_ERR_CACHE with the
// same empty result.  A block-table entry outside [0, num_phys_pages) is
// BSA_ERR_CACHE too: its page scores -inf, and if it is still kept (fewer pages
// than top_k) the attention reads zeros in its place.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace bsa {
namespace {

constexpr int kD = 128;          // decode head_dim
constexpr int kMaxG = 8;         // query heads per KV head supported (1, 2, 4 or 8)
constexpr int kPage = 64;        // tokens per page
constexpr int kScoreThreads = 256;
constexpr int kSelThreads = 256;

// ---------------------------------------------------------------- score
// grid (ceil(max_pages / 64), R): 64 logical pages of one request per CTA, for
// every KV head.  The CTA stages the pages' block-table entries and the request's
// queries once (fp32 rows of kQStride floats in dynamic shared memory); each warp
// then takes (KV head, 8 pages) items.  Every load instruction reads one whole
// 512-byte summary row (lane = float4 column), so a warp's request touches four
// cache lines; the 8 G partial dot products per lane are then summed across the
// warp by a reduce-scatter (31 shuffles for G = 4 instead of 5 per dot product).
constexpr int kQStride = kD + 4;

// Reduce-scatter of N per-lane partial sums over the 32 lanes of a warp (halving
// butterfly): at offset o a lane keeps the half of its values selected by bit o
// of its lane index and adds its partner's copy of that half.  With N = 8 G
// values indexed j = 8-page row * G + head, lane l ends with the full sums of
// j = l >> (5 - log2 N) (N <= 32: the remaining offsets add plainly) or of
// j = 2 l, 2 l + 1 (N = 64): in every case row = l >> 2.
template <int N, int O>
BSA_DEV void rs_step(float (&v)[64], int lane) {
  if constexpr (O >= 1) {
    if constexpr (N > 1) {
      const bool up = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        const float send = up ? v[i] : v[i + N / 2];
        const float keep = up ? v[i + N / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      rs_step<N / 2, O / 2>(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      rs_step<1, O / 2>(v, lane);
    }
  }
}

// A request length the decode accepts: 1 .. max_pages * page (0 is an idle slot).
BSA_DEV bool len_ok(int len, int max_pages) { return len >= 1 && len <= max_pages * kPage; }

template <int G>
__global__ void __launch_bounds__(kScoreThreads) dec_score_kernel(
    const uint16_t *__restrict__ q, const float *__restrict__ ps, const int32_t *__restrict__ bt,
    const int32_t *__restrict__ lens, float *__restrict__ scores, int32_t *status, int Hk,
    int max_pages, int num_phys) {
  extern __shared__ __align__(16) float qs[];  // [H][kQStride]
  __shared__ int phys_s[64];
  const int rho = blockIdx.y;
  const int H = G * Hk;
  const int len = lens[rho];
  if (!len_ok(len, max_pages)) return;  // reported by the select kernel
  const int L = (len + kPage - 1) / kPage;
  const int p_begin = blockIdx.x * 64;
  if (p_begin >= L - 1) return;
  const int npg = min(L - 1, p_begin + 64) - p_begin;
  if (threadIdx.x < npg) {
    int ph = __ldg(bt + (size_t)rho * max_pages + p_begin + threadIdx.x);
    if (ph < 0 || ph >= num_phys) {  // a stale or foreign page id: never read through it
      set_status(status, BSA_ERR_CACHE);
      ph = -1;
    }
    phys_s[threadIdx.x] = ph;
  }
  for (int e = threadIdx.x; e < H * kD; e += blockDim.x)
    qs[(e / kD) * kQStride + e % kD] = bf16_to_f32(q[(size_t)rho * H * kD + e]);
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int ngrp = (npg + 7) / 8;
  for (int item = warp; item < Hk * ngrp; item += kScoreThreads / 32) {
    const int h = item / ngrp, p0 = (item - h * ngrp) * 8;
    {  // this warp's next item towards L2: lane = (page, 128-byte line of its summary row)
      const int nitem = item + kScoreThreads / 32;
      if (nitem < Hk * ngrp) {
        const int nh = nitem / ngrp, np0 = (nitem - nh * ngrp) * 8 + (lane >> 2);
        const int ph = np0 < npg ? phys_s[np0] : -1;
        if (ph >= 0)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(ps + ((size_t)ph * Hk + nh) * kD + (lane & 3) * 32));
      }
    }
    float4 c[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {  // a missing page of the last group repeats the first
      const int pg = p0 + k < npg ? p0 + k : p0;
      const int ph = phys_s[pg];
      c[k] = ph >= 0 ? __ldg(reinterpret_cast<const float4 *>(ps + ((size_t)ph * Hk + h) * kD) + lane)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float v[64];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float4 qq = *reinterpret_cast<const float4 *>(qs + (h * G + g) * kQStride + 4 * lane);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        v[k * G + g] = qq.x * c[k].x + qq.y * c[k].y + qq.z * c[k].z + qq.w * c[k].w;
    }
    rs_step<8 * G, 16>(v, lane);
    float best = G == 8 ? fmaxf(v[0], v[1]) : v[0];  // max over the group's heads
    best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 1));
    best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 2));
    const int row = lane >> 2;
    if ((lane & 3) == 0 && p0 + row < npg)
      scores[((size_t)rho * Hk + h) * max_pages + p_begin + p0 + row] =
          phys_s[p0 + row] >= 0 ? best : -INFINITY;
  }
  grid_dep_launch();
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
    int32_t *__restrict__ sel_counts, int32_t *status, int Hk, int max_pages, int top_k) {
  extern __shared__ uint32_t keys[];  // max_pages
  __shared__ int hist[256];
  __shared__ int scan_buf[32];
  __shared__ int s_bin, s_above;
  const int rho = blockIdx.y, h = blockIdx.x;
  int32_t *out = sel + ((size_t)rho * Hk + h) * (top_k + 1);
  grid_dep_wait();  // scores come from the previous launch
  const int len = lens[rho];
  if (!len_ok(len, max_pages)) {  // idle (0) or invalid: no pages kept
    if (len != 0 && h == 0 && threadIdx.x == 0) set_status(status, BSA_ERR_CACHE);
    for (int e = threadIdx.x; e <= top_k; e += blockDim.x) out[e] = -1;
    if (threadIdx.x == 0) sel_counts[(size_t)rho * Hk + h] = 0;
    grid_dep_launch();
    return;
  }
  const int L = (len + 63) / 64;
  const int N = L - 1;  // scored pages
  const float *sc = scores + ((size_t)rho * Hk + h) * max_pages;
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
      const int bin_count = hist[s_bin];
      remaining -= s_above;
      prefix |= (uint32_t)s_bin << shift;
      mask |= 0xFFu << shift;
      __syncthreads();
      // The bin holding the k-th key holds exactly the keys still needed: all of
      // them are selected, whatever their lower bits, so the select is complete.
      if (bin_count == remaining) break;
    }
  }
  // Compact in index order: keys above the k-th key's bin (compared on the
  // resolved top bits, `mask`), then the first `remaining` keys of that bin (ties
  // go to the lower page index).
  const int per = (N + blockDim.x - 1) / blockDim.x;
  const int lo = min(N, (int)threadIdx.x * per), hi = min(N, lo + per);
  int n_eq = 0;
  for (int e = lo; e < hi; ++e) n_eq += (k < N && (keys[e] & mask) == prefix) ? 1 : 0;
  const int2 eq = block_scan(n_eq, scan_buf);
  int taken = 0, eq_seen = eq.x;
  for (int e = lo; e < hi; ++e) {
    bool s;
    if (k >= N) {
      s = true;
    } else if ((keys[e] & mask) > prefix) {
      s = true;
    } else if ((keys[e] & mask) == prefix) {
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
    } else if ((keys[e] & mask) > prefix) {
      s = true;
    } else if ((keys[e] & mask) == prefix) {
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
  grid_dep_launch();
}

// ---------------------------------------------------------------- attention
// Persistent, one CTA per SM, on the tensor cores.  A unit is two selected pages
// of one (request, KV head) — 128 keys — and yields one partial (m, l, u) per
// query head of the group:
//   S^T = K Q^T   M = 128 keys,  N = 16 (the group's queries, padded), K = d
//   O^T = V^T P^T M = d = 128,   N = 16,                                K = 128 keys
// A unit holding one page only reads the second page at an out-of-range page
// coordinate, which the tensor copy fills with zeros, and masks its keys.
// Warp roles (320 threads):
//   warps 0-3  softmax: thread = one key row of S^T (TMEM lane)
//   warp 4     producer: resolves the page indices of 32 units at a time, then
//              stages K, V (two 64-column panels x two pages) and Q by TMA
//   warp 5     MMA issuer (one thread); owns the TMEM allocation
//   warps 6-9  epilogue: thread = one d row of O^T (warp 6 + q reads TMEM lane
//              quarter (q + 2) mod 4), writes the unit's partial (m, l, u)
// The softmax warps hand a unit to the epilogue warps once its P and row sums are
// written and go on to the next unit while the unit's PV runs and its partial is
// written out; a buffer (b = unit parity) is reused two units later only after the
// epilogue has released it.
// TMEM (64 columns): S_0, S_1, O_0, O_1 (16 columns each), double-buffered by unit.
constexpr int kDecThreads = 320;
constexpr int kDecEpi = 6;       // first of the four epilogue warps
constexpr int kDecProducer = 4;
constexpr int kDecMma = 5;
constexpr int kNS = 3;                       // K/V/Q stages
constexpr int kKVBytes = 2 * kPage * kD * 2;  // two pages of K (or V): 32 KB
constexpr int kQPanel = 16 * 128;             // 16 rows x 128 bytes
constexpr int kQRows = 8;                     // query rows copied (G <= 8)
constexpr int kStageBytes = 2 * kKVBytes + 2 * kQPanel;  // K | V | Q
constexpr int kPBytes = 2 * kQPanel;          // P^T: 16 rows x 128 keys (two panels)
constexpr int kTxBytes = 2 * kKVBytes + 2 * kQRows * 128;
// shared memory map (offsets from a 1024-byte aligned base)
constexpr int kOffStages = 0;
constexpr int kOffP = kOffStages + kNS * kStageBytes;
constexpr int kOffHdr = kOffP + 2 * kPBytes;        // per stage: unit, valid A, valid B
constexpr int kOffRed = kOffHdr + kNS * 16;          // [2][4][16] max, [2][4][16] sum
constexpr int kOffEpi = kOffRed + 2 * 2 * 4 * 16 * 4; // [2] unit handed to the epilogue
constexpr int kOffBar = kOffEpi + 16;
// barriers: FULL[kNS], EMPTY[kNS], SFULL[2], PFULL[2], OFULL[2], MX[2], EPI[2] (a unit
// handed to the epilogue), EPIFREE[2] (its buffer released by the epilogue), FINAL
constexpr int B_FULL = 0, B_EMPTY = kNS, B_SFULL = 2 * kNS, B_PFULL = B_SFULL + 2,
              B_OFULL = B_PFULL + 2, B_MX = B_OFULL + 2, B_EPI = B_MX + 2,
              B_EPIFREE = B_EPI + 2, B_FIN = B_EPIFREE + 2;
constexpr int kNumBars = B_FIN + 1;
constexpr int kOffCtl = kOffBar + kNumBars * 8;     // tmem base, abort flag
constexpr int kDecSmem = kOffCtl + 16 + 1024;
static_assert(kDecSmem <= 232448, "shared memory budget");
constexpr uint32_t kColS = 0, kColO = 32;
// kind::f16 descriptors: QK with both operands K-major; PV with A (= V^T) MN-major.
constexpr uint32_t kIdescQK = idesc_bf16(128, 16, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 16, false) | (1u << 15);

struct DecParams {
  const int32_t *bt, *lens, *sel, *sel_counts;
  float *part_ml, *part_o;
  int32_t *status;
  float scale_log2;
  int H, Hk, G, max_pages, top_k, nchunk, units, oob_page, num_phys;
};

// Tensor-map page coordinate (phys * H_kv + h) of logical page lp, or the
// zero-filled out-of-range coordinate for an id outside the cache.
BSA_DEV int dec_page_coord(const DecParams &p, int rho, int h, int lp) {
  const int ph = __ldg(p.bt + (size_t)rho * p.max_pages + lp);
  if (ph < 0 || ph >= p.num_phys) {
    set_status(p.status, BSA_ERR_CACHE);
    return p.oob_page;
  }
  return ph * p.Hk + h;
}

BSA_DEV void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

BSA_DEV void bar_warps_wait(uint32_t bar, uint32_t parity, volatile int32_t *abort_flag,
                            int32_t *status, bool &ok) {
  ok = ok && mbar_wait(bar, parity, abort_flag, status);
  ok = __all_sync(0xffffffffu, ok);
}

template <int G>
__global__ void __launch_bounds__(kDecThreads, 1)
    dec_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const DecParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *sm = smem_raw + (sbase - raw);
  auto bar = [&](int k) { return sbase + kOffBar + 8u * (uint32_t)k; };
  int32_t *hdr = reinterpret_cast<int32_t *>(sm + kOffHdr);
  float *red_m = reinterpret_cast<float *>(sm + kOffRed);
  float *red_l = red_m + 2 * 4 * 16;
  int32_t *epi_u = reinterpret_cast<int32_t *>(sm + kOffEpi);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffCtl);
  volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(sm + kOffCtl + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_SFULL + b), 1);
      mbar_init(bar(B_PFULL + b), 4);
      mbar_init(bar(B_OFULL + b), 1);
      mbar_init(bar(B_MX + b), 4);
      mbar_init(bar(B_EPI + b), 4);
      mbar_init(bar(B_EPIFREE + b), 4);
    }
    mbar_init(bar(B_FIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kDecMma) {
    tmem_alloc(smem_u32(tmem_slot), 64);
    tmem_relinquish();
  }
  if (warp == kDecProducer && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int per_pair = p.top_k + 1;
  grid_dep_wait();    // the selection comes from the previous launch
  grid_dep_launch();  // the merge may be scheduled now; it waits for this grid

  if (warp == kDecProducer) {
    // ------------------------------------------------------------ producer
    int j = 0;
    int last[kNS];
    for (int s = 0; s < kNS; ++s) last[s] = -1;
    bool ok = true;
    for (int b0 = blockIdx.x; ok && b0 < p.units; b0 += 32 * gridDim.x) {
      const int u = b0 + lane * gridDim.x;
      int zA = 0, zB = 0, qrow = 0, vA = 0, vB = 0;
      bool live = false;
      if (u < p.units) {
        const int pair = u / p.nchunk, c = u - pair * p.nchunk;
        const int cnt = __ldg(p.sel_counts + pair);
        const int rho = pair / p.Hk, h = pair - rho * p.Hk;
        const int n = __ldg(p.lens + rho);
        if (2 * c < cnt && len_ok(n, p.max_pages)) {
          live = true;
          const int32_t *sp = p.sel + (size_t)pair * per_pair + 2 * c;
          const int lpA = checked_index(__ldg(sp), 0, p.max_pages - 1, p.status);
          zA = dec_page_coord(p, rho, h, lpA);
          vA = min(kPage, n - lpA * kPage);
          if (2 * c + 1 < cnt) {
            const int lpB = checked_index(__ldg(sp + 1), 0, p.max_pages - 1, p.status);
            zB = dec_page_coord(p, rho, h, lpB);
            vB = min(kPage, n - lpB * kPage);
          } else {
            zB = p.oob_page;  // zero-filled by the copy, keys masked
          }
          qrow = rho * p.H + h * p.G;
        }
      }
      uint32_t todo = __ballot_sync(0xffffffffu, live);
      while (todo != 0u) {
        const int src = __ffs(todo) - 1;
        todo &= todo - 1u;
        const int uu = __shfl_sync(0xffffffffu, u, src);
        const int a = __shfl_sync(0xffffffffu, zA, src);
        const int b = __shfl_sync(0xffffffffu, zB, src);
        const int qr = __shfl_sync(0xffffffffu, qrow, src);
        const int va = __shfl_sync(0xffffffffu, vA, src);
        const int vb = __shfl_sync(0xffffffffu, vB, src);
        if (lane == 0) {
          const int st = j % kNS;
          const uint32_t ph = ((j / kNS) & 1) ^ 1;
          ok = mbar_wait(bar(B_EMPTY + st), ph, abort_flag, p.status);
          if (ok) {
            hdr[st * 4 + 0] = uu;
            hdr[st * 4 + 1] = va;
            hdr[st * 4 + 2] = vb;
            const uint32_t full = bar(B_FULL + st);
            mbar_arrive_expect_tx(full, kTxBytes);
            last[st] = ph ^ 1;
            const uint32_t stg = sbase + kOffStages + st * kStageBytes;
            for (int pn = 0; pn < 2; ++pn) {
              tma_load_3d(stg + pn * 16384, &tmK, full, pn * 64, 0, a);
              tma_load_3d(stg + pn * 16384 + 8192, &tmK, full, pn * 64, 0, b);
            }
            for (int pn = 0; pn < 2; ++pn)
              tma_load_3d(stg + 2 * kKVBytes + pn * kQPanel, &tmQ, full, pn * 64, qr, 0);
            for (int pn = 0; pn < 2; ++pn) {
              tma_load_3d(stg + kKVBytes + pn * 16384, &tmV, full, pn * 64, 0, a);
              tma_load_3d(stg + kKVBytes + pn * 16384 + 8192, &tmV, full, pn * 64, 0, b);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        ++j;
      }
    }
    if (lane == 0) {
      if (ok) {  // end of work: a stage whose header holds unit -1
        const int st = j % kNS;
        if (mbar_wait(bar(B_EMPTY + st), ((j / kNS) & 1) ^ 1, abort_flag, p.status)) {
          hdr[st * 4 + 0] = -1;
          mbar_arrive(bar(B_FULL + st));
        }
      } else {  // copies in flight land before the CTA leaves
        for (int s = 0; s < kNS; ++s)
          if (last[s] >= 0) mbar_wait_drain(bar(B_FULL + s), last[s]);
      }
    }
  } else if (warp == kDecMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t stg0 = sbase + kOffStages, pb0 = sbase + kOffP;
      auto qk = [&](int i) {
        const int st = i % kNS, b = i & 1;
        const uint32_t k0 = stg0 + st * kStageBytes, q0 = k0 + 2 * kKVBytes;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_bf16_ss(tmem + kColS + 16 * b,
                      sdesc_sw128(k0 + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024),
                      sdesc_sw128(q0 + (kk / 4) * kQPanel + (kk % 4) * 32, 16, 1024), kIdescQK,
                      kk > 0 ? 1u : 0u);
        mma_commit(bar(B_SFULL + b));
      };
      auto pv = [&](int i) {
        const int st = i % kNS, b = i & 1;
        const uint32_t v0 = stg0 + st * kStageBytes + kKVBytes, p0 = pb0 + b * kPBytes;
#pragma unroll
        for (int kk = 0; kk < 2 * kPage / 16; ++kk)
          mma_bf16_ss(tmem + kColO + 16 * b, sdesc_sw128(v0 + kk * 2048, 16384, 1024),
                      sdesc_sw128(p0 + (kk / 4) * kQPanel + (kk % 4) * 32, 16, 1024), kIdescPV,
                      kk > 0 ? 1u : 0u);
        mma_commit(bar(B_OFULL + b));
        mma_commit(bar(B_EMPTY + st));
      };
      bool ok = mbar_wait(bar(B_FULL + 0), 0, abort_flag, p.status);
      bool more = ok && hdr[0] >= 0;
      if (more) {
        tc_fence_after();
        qk(0);
      }
      for (int i = 0; more; ++i) {
        // QK of the next unit goes ahead of PV of this one
        const int i1 = i + 1, st1 = i1 % kNS;
        if (!(ok = mbar_wait(bar(B_FULL + st1), (i1 / kNS) & 1, abort_flag, p.status))) break;
        const bool next = hdr[st1 * 4] >= 0;
        if (next) {
          tc_fence_after();
          qk(i1);
        }
        if (!(ok = mbar_wait(bar(B_PFULL + (i & 1)), (i / 2) & 1, abort_flag, p.status))) break;
        tc_fence_after();
        pv(i);
        more = next;
      }
      // Every MMA issued so far completes before TMEM is released.
      mma_commit(bar(B_FIN));
      mbar_wait_drain(bar(B_FIN), 0);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax
    const int t = warp * 32 + lane;  // key row of S^T
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    // byte offset of P^T[g][t] inside one P buffer (128-byte swizzle, 8-row atoms)
    const uint32_t t_panel = (uint32_t)(t >> 6) * kQPanel, t_chunk = (uint32_t)((t & 63) >> 3),
                   t_in = (uint32_t)(t & 7) * 2;
    bool ok = true;
    for (int i = 0;; ++i) {
      const int st = i % kNS, b = i & 1;
      bar_warps_wait(bar(B_FULL + st), (i / kNS) & 1, abort_flag, p.status, ok);
      if (!ok) break;
      const int u = hdr[st * 4 + 0];
      // buffer b (row statistics, unit slot, O_b) was released by the epilogue for
      // unit i - 2
      if (i >= 2) bar_warps_wait(bar(B_EPIFREE + b), ((i - 2) / 2) & 1, abort_flag, p.status, ok);
      if (!ok) break;
      if (u < 0) {  // end of work, passed on to the epilogue
        if (t == 0) epi_u[b] = -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_EPI + b));
        break;
      }
      const int va = hdr[st * 4 + 1], vb = hdr[st * 4 + 2];
      const bool valid = t < kPage ? t < va : t - kPage < vb;
      bar_warps_wait(bar(B_SFULL + b), (i / 2) & 1, abort_flag, p.status, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t r[16];
      tmem_ld16(tmem + lane_base + kColS + 16 * b, r);
      float x[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        x[g] = valid ? __uint_as_float(r[g]) * p.scale_log2 : -INFINITY;
        float m = x[g];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) red_m[(b * 4 + warp) * 16 + g] = m;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_MX + b));
      bar_warps_wait(bar(B_MX + b), (i / 2) & 1, abort_flag, p.status, ok);
      if (!ok) break;
      float l[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float M = fmaxf(fmaxf(red_m[(b * 4 + 0) * 16 + g], red_m[(b * 4 + 1) * 16 + g]),
                              fmaxf(red_m[(b * 4 + 2) * 16 + g], red_m[(b * 4 + 3) * 16 + g]));
        // a unit's first page always holds a valid key, so M is finite
        const float pg = fast_exp2(x[g] - M);
        l[g] = pg;
        const __nv_bfloat16 pb = __float2bfloat16_rn(pg);
        const uint32_t off = t_panel + (uint32_t)g * 128u + ((t_chunk ^ (uint32_t)(g & 7)) << 4) + t_in;
        *reinterpret_cast<__nv_bfloat16 *>(sm + kOffP + b * kPBytes + off) = pb;
      }
      // Rows G-15 of P^T are never written: they only feed columns of O^T that are
      // never read (likewise rows G-15 of the staged queries).
      fence_proxy_async_smem();  // P^T is read by the tensor cores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL + b));
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float sum = l[g];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (lane == 0) red_l[(b * 4 + warp) * 16 + g] = sum;
      }
      if (t == 0) epi_u[b] = u;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_EPI + b));
    }
  } else if (warp >= kDecEpi) {
    // ------------------------------------------------------------ epilogue
    const int q = warp % 4;            // TMEM lane quarter
    const int t = q * 32 + lane;       // d row of O^T
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    bool ok = true;
    for (int i = 0;; ++i) {
      const int b = i & 1;
      bar_warps_wait(bar(B_EPI + b), (i / 2) & 1, abort_flag, p.status, ok);
      if (!ok) break;
      const int u = epi_u[b];
      if (u < 0) break;
      bar_warps_wait(bar(B_OFULL + b), (i / 2) & 1, abort_flag, p.status, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t r[16];
      tmem_ld16(tmem + lane_base + kColO + 16 * b, r);
      float *po = p.part_o + (size_t)u * G * kD;
#pragma unroll
      for (int g = 0; g < G; ++g) po[g * kD + t] = __uint_as_float(r[g]);
      if (t < G) {
        float lsum = 0.f, mt = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g)
          if (g == t) {
            lsum = red_l[(b * 4 + 0) * 16 + g] + red_l[(b * 4 + 1) * 16 + g] +
                   red_l[(b * 4 + 2) * 16 + g] + red_l[(b * 4 + 3) * 16 + g];
            mt = fmaxf(fmaxf(red_m[(b * 4 + 0) * 16 + g], red_m[(b * 4 + 1) * 16 + g]),
                       fmaxf(red_m[(b * 4 + 2) * 16 + g], red_m[(b * 4 + 3) * 16 + g]));
          }
        p.part_ml[((size_t)u * G + t) * 2] = mt;
        p.part_ml[((size_t)u * G + t) * 2 + 1] = lsum;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_EPIFREE + b));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kDecMma) {
    __syncwarp();
    tmem_dealloc(tmem, 64);
  }
}

// grid (H_kv, R), G * 128 threads (one output element each): combine the unit
// partials of a (request, KV head) with eqs.(3)-(5) in the log2 domain.  Warp g
// first turns the partials' (m, l) of query head g into weights 2^(m_k - M) and
// the total l; then every thread sums its column of u with loads kept in flight.
constexpr int kMaxChunks = (64 + 2) / 2;  // units per (request, KV head) at top_k = 64

__global__ void __launch_bounds__(kMaxG * kD) dec_merge_kernel(
    const float *__restrict__ part_ml, const float *__restrict__ part_o,
    const int32_t *__restrict__ sel_counts, uint16_t *__restrict__ o, float *__restrict__ lse,
    int H, int Hk, int nchunk) {
  __shared__ float wgt[kMaxG][kMaxChunks];
  __shared__ float tot_l[kMaxG], tot_m[kMaxG];
  const int rho = blockIdx.y, h = blockIdx.x;
  const int G = H / Hk;
  const int pair = rho * Hk + h;
  grid_dep_wait();  // the partials come from the previous launch
  const int nu = (sel_counts[pair] + 1) / 2;
  if (nu == 0) {  // no page kept (idle or invalid request): empty softmax
    const int gg = threadIdx.x / kD, cc = threadIdx.x % kD, hq = h * G + gg;
    o[((size_t)rho * H + hq) * kD + cc] = 0;
    if (lse != nullptr && cc == 0) lse[(size_t)rho * H + hq] = -INFINITY;
    return;
  }
  const size_t u0 = (size_t)pair * nchunk;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (warp < G) {
    const int g = warp;
    float mk[2], lk[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int k = lane + 32 * r;
      mk[r] = k < nu ? part_ml[((u0 + k) * G + g) * 2] : -INFINITY;
      lk[r] = k < nu ? part_ml[((u0 + k) * G + g) * 2 + 1] : 0.f;
    }
    float M = fmaxf(mk[0], mk[1]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int k = lane + 32 * r;
      const float f = k < nu ? fast_exp2(mk[r] - M) : 0.f;
      if (k < kMaxChunks) wgt[g][k] = f;
      L += f * lk[r];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (lane == 0) {
      tot_l[g] = L;
      tot_m[g] = M;
    }
  }
  __syncthreads();
  const int g = threadIdx.x / kD, c = threadIdx.x % kD;
  const float *col = part_o + (u0 * G + g) * kD + c;
  float acc = 0.f;
#pragma unroll 8
  for (int k = 0; k < nu; ++k) acc = fmaf(wgt[g][k], col[(size_t)k * G * kD], acc);
  const int hq = h * G + g;
  const __nv_bfloat16 ob = __float2bfloat16_rn(acc / tot_l[g]);
  o[((size_t)rho * H + hq) * kD + c] = *reinterpret_cast<const uint16_t *>(&ob);
  if (lse != nullptr && c == 0)
    lse[(size_t)rho * H + hq] = (tot_m[g] + log2f(tot_l[g])) * 0.6931471805599453f;
}

int num_chunks(const bsa_decode_shape_t &s) { return (s.top_k + 2) / 2; }

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

// Workspace: scores [R, H_kv, max_pages] | unit partials (m, l) | unit partials u.
size_t decode_workspace_bytes(const bsa_decode_shape_t &s) {
  const size_t G = (size_t)(s.num_heads / s.num_kv_heads);
  const size_t units = (size_t)s.num_reqs * s.num_kv_heads * num_chunks(s);
  const size_t pairs = (size_t)s.num_reqs * s.num_kv_heads;
  return up256(pairs * s.max_pages_per_req * sizeof(float)) + up256(units * G * 2 * sizeof(float)) +
         up256(units * G * kD * sizeof(float));
}

cudaError_t launch_decode(const bsa_decode_shape_t &s, const void *q, const void *k_cache,
                          const void *v_cache, const float *page_summ,
                          const int32_t *block_table, const int32_t *context_lens, float scale,
                          void *o, float *lse, int32_t *sel, int32_t *sel_counts,
                          int32_t *dev_status, void *ws, cudaStream_t st) {
  const int G = s.num_heads / s.num_kv_heads;
  const int nchunk = num_chunks(s);
  const size_t pairs = (size_t)s.num_reqs * s.num_kv_heads;
  const size_t units = pairs * nchunk;
  char *w = static_cast<char *>(ws);
  float *scores = reinterpret_cast<float *>(w);
  w += up256(pairs * s.max_pages_per_req * sizeof(float));
  float *part_ml = reinterpret_cast<float *>(w);
  w += up256(units * G * 2 * sizeof(float));
  float *part_o = reinterpret_cast<float *>(w);

  CUtensorMap mq, mk, mv;
  const uint64_t zpages = (uint64_t)s.num_phys_pages * s.num_kv_heads;
  if (!make_tmap_3d_bf16(&mq, q, kD, (uint64_t)s.num_reqs * s.num_heads, 1, 64, kQRows, 1) ||
      !make_tmap_3d_bf16(&mk, k_cache, kD, kPage, zpages, 64, kPage, 1) ||
      !make_tmap_3d_bf16(&mv, v_cache, kD, kPage, zpages, 64, kPage, 1))
    return cudaErrorInvalidValue;

  const uint16_t *qb = static_cast<const uint16_t *>(q);
  const int qs_bytes = s.num_heads * kQStride * (int)sizeof(float);
  const dim3 sgrid((s.max_pages_per_req + 63) / 64, s.num_reqs);
  cudaError_t e;
#define BSA_DEC_SCORE(GG)                                                                     \
  do {                                                                                        \
    e = cudaFuncSetAttribute(dec_score_kernel<GG>,                                            \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, qs_bytes);          \
    if (e != cudaSuccess) return e;                                                           \
    dec_score_kernel<GG><<<sgrid, kScoreThreads, qs_bytes, st>>>(                             \
        qb, page_summ, block_table, context_lens, scores, dev_status, s.num_kv_heads,           \
        s.max_pages_per_req, s.num_phys_pages);                                               \
  } while (0)
  switch (G) {
    case 1: BSA_DEC_SCORE(1); break;
    case 2: BSA_DEC_SCORE(2); break;
    case 4: BSA_DEC_SCORE(4); break;
    case 8: BSA_DEC_SCORE(8); break;
    default: return cudaErrorInvalidValue;
  }
#undef BSA_DEC_SCORE
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t sm = (size_t)s.max_pages_per_req * sizeof(uint32_t);
  if (sm > 40 * 1024) {
    e = cudaFuncSetAttribute(dec_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm);
    if (e != cudaSuccess) return e;
  }
  e = launch_dependent(dec_select_kernel, dim3(s.num_kv_heads, s.num_reqs), dim3(kSelThreads), sm,
                       st, scores, context_lens, sel, sel_counts, dev_status, s.num_kv_heads,
                       s.max_pages_per_req, s.top_k);
  if (e != cudaSuccess) return e;

  DecParams p;
  p.bt = block_table;
  p.lens = context_lens;
  p.sel = sel;
  p.sel_counts = sel_counts;
  p.part_ml = part_ml;
  p.part_o = part_o;
  p.status = dev_status;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.H = s.num_heads;
  p.Hk = s.num_kv_heads;
  p.G = G;
  p.max_pages = s.max_pages_per_req;
  p.top_k = s.top_k;
  p.nchunk = nchunk;
  p.units = (int)units;
  p.oob_page = (int)zpages;
  p.num_phys = s.num_phys_pages;
  auto *kern = G == 1 ? dec_tc_kernel<1> : G == 2 ? dec_tc_kernel<2> : G == 4 ? dec_tc_kernel<4>
                                                                              : dec_tc_kernel<8>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmem);
  if (e != cudaSuccess) return e;
  const int grid = (int)std::min<size_t>((size_t)num_sms(), units);
  e = launch_dependent(kern, dim3(grid), dim3(kDecThreads), kDecSmem, st, mq, mk, mv, p);
  if (e != cudaSuccess) return e;
  return launch_dependent(dec_merge_kernel, dim3(s.num_kv_heads, s.num_reqs), dim3(G * kD), 0, st,
                          part_ml, part_o, sel_counts, static_cast<uint16_t *>(o), lse,
                          s.num_heads, s.num_kv_heads, nchunk);
}

}  // namespace bsa
