// a2 on the tensor cores: router scores g[i,h,r,j] = max over the group's query
// rows of block r of q . c_j, j < r ("2.1 · 粗粒度选择" §2.1 eq.(6), pool = max).
//
// The selection is compared bit-exactly (up to a 1e-5 tie band) with a float64
// oracle, so the scores must be fp32-accurate where they decide.  Q is exact in
// bf16; each fp32 summary is split without error into three bf16 terms
// c = c_hi + c_mid + c_lo (the residuals of bf16 rounding are exact in fp32).
//   exact  (parts = 3) q . c accumulated on the tensor cores in fp32 as
//          q . c_lo + q . c_mid + q . c_hi (small terms first);
//   screen (parts = 2) q . (c_hi + c_mid), two thirds of the work.  The rest,
//          q . delta with delta = c - c_hi - c_mid, is bounded by |q| |delta|; the
//          epilogue records the largest query norm of each row so that the
//          selection can bound every screened score and rescore exactly only the
//          candidates whose interval meets the selection boundary.
//
// MMA orientation: M = 128 summaries (TMEM lanes), N = up to 256 query rows
// (TMEM columns), K = d.  The max over query rows is then a per-thread max over
// the TMEM columns of its own lane — no cross-thread reduction.
//
// Persistent kernel, one CTA per SM, 192 threads:
//   warps 0-3  epilogue: tcgen05.ld of a 128 x N accumulator, masked row max,
//              write / max-merge into S
//   warp 4     TMA producer: query chunks (G*b rows, <= 256 per chunk) and
//              16 KB panels of the split summaries, through rings of 2 and 4
//   warp 5     MMA issuer (lane 0), double-buffered accumulators in TMEM
//   warp 6     watcher: waits on the copies' mbarriers and meets the MMA warp on
//              named barriers (an mbarrier check would cost the issuing thread a few
//              hundred cycles while the MMAs stream their operands from shared memory)
// Work order: rows with the longest and the shortest history alternately.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace bsa {
namespace {

constexpr int kThreads = 224;
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kWatchWarp = 6;
// named barriers (watcher + MMA warp, taken by both once per query chunk / panel)
constexpr uint32_t kNbQ = 1, kNbA = 2, kNbThreads = 64;
constexpr int kQStages = 2;
constexpr int kAStages = 4;
constexpr int kAStage = 128 * 128;  // one 128-byte panel of one split part, 128 summaries

template <int D>
struct RCfg {
  static constexpr int kPanels = D / 64;
  static constexpr int kQStage = 256 * D * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffA = kOffQ + kQStages * kQStage;
  static constexpr int kOffBar = kOffA + kAStages * kAStage;
  static constexpr int B_QFULL = 0, B_QEMPTY = kQStages;
  static constexpr int B_AFULL = 2 * kQStages, B_AEMPTY = B_AFULL + kAStages;
  static constexpr int B_DFULL = B_AEMPTY + kAStages, B_DEMPTY = B_DFULL + 2;
  static constexpr int B_FINAL = B_DEMPTY + 2;
  static constexpr int kNumBars = B_FINAL + 1;
  static constexpr int kOffCtl = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes =
      kOffCtl + 16 + 1024 < 120 * 1024 ? 120 * 1024 : kOffCtl + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct RouteTcParams {
  const int32_t *cu;
  const int32_t *qoff;  // chunked prefill: tokens cached before each chunk (else null)
  float *S;
  float *Qn;            // screen: per row, the largest query norm (zeroed by the split)
  int32_t *status;
  int B, Nq, Hk, G, b;
  int Nk;         // summaries per (sequence, KV head) = row length of S (N_q without a cache)
  int nch;        // query chunks per row: ceil(G*b / 256)
  int parts;      // split parts per summary: 3 exact, 2 screen
};

// Router row: query block qb of sequence i and KV head h (its queries in the packed
// Q), logical block r = qb (+ the cached blocks before a chunk) scored against
// summaries 0 .. r-1.
struct RUnit {
  int i, h, r, qb, s0, nvalid;
  bool valid;
};

BSA_DEV RUnit runit(const RouteTcParams &p, int u) {
  RUnit x;
  const int BH = p.B * p.Hk;
  // Rank k of the longest-first order, taken alternately from its two ends (0, N-1, 1,
  // N-2, ...): along a CTA's stride long rows (tensor-bound) and short ones (bound by
  // their query copies) alternate, so the copies overlap the products.
  const int k = u / BH;
  const int kk = (k & 1) ? p.Nq - 1 - (k >> 1) : (k >> 1);
  x.qb = p.Nq - 1 - kk;
  const int ih = u % BH;
  x.i = ih / p.Hk;
  x.h = ih % p.Hk;
  x.s0 = __ldg(p.cu + x.i);
  const int n = __ldg(p.cu + x.i + 1) - x.s0;
  const int nb = (n + p.b - 1) / p.b;
  bool ok = true;
  x.r = x.qb;
  if (p.qoff != nullptr) {
    const int pre = __ldg(p.qoff + x.i);
    ok = chunk_ok(pre, n, p.b, p.Nk);
    if (ok) x.r += pre / p.b;
  }
  x.valid = ok && x.r >= 1 && x.qb < nb;
  x.nvalid = min(p.b, n - x.qb * p.b);
  return x;
}

BSA_DEV int chunk_cols(const RouteTcParams &p, int ch) { return min(256, p.G * p.b - 256 * ch); }

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    route_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmC,
                    const RouteTcParams p) {
  using C = RCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *sm = smem_raw + (sbase - raw);
  const uint32_t bars = sbase + C::kOffBar;
  auto bar = [&](int k) { return bars + 8u * (uint32_t)k; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::kOffCtl);
  volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(sm + C::kOffCtl + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(bar(C::B_QFULL + s), 1);
      // the MMA's commit, plus the four epilogue warps when they read query norms
      mbar_init(bar(C::B_QEMPTY + s), p.Qn != nullptr ? 5 : 1);
    }
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(bar(C::B_AFULL + s), 1);
      mbar_init(bar(C::B_AEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_DFULL + s), 1);
      mbar_init(bar(C::B_DEMPTY + s), 4);
    }
    mbar_init(bar(C::B_FINAL), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmC);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();    // Q, C and the split come from earlier launches
  const int total = p.B * p.Hk * p.Nq;
  const uint32_t smQ = sbase + C::kOffQ, smA = sbase + C::kOffA;
  const int heads_per_chunk = 256 / p.b;

  if (warp == kTmaWarp) {
    if (lane == 0) {
      int qi = 0, ai = 0;
      int lastQ[kQStages], lastA[kAStages];
      for (int s = 0; s < kQStages; ++s) lastQ[s] = -1;
      for (int s = 0; s < kAStages; ++s) lastA[s] = -1;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total; u += gridDim.x) {
        const RUnit x = runit(p, u);
        if (!x.valid) continue;
        const int nmt = (x.r + 127) / 128;
        const int crow = (x.i * p.Hk + x.h) * p.Nk;
        for (int ch = 0; ok && ch < p.nch; ++ch, ++qi) {
          const int qs = qi % kQStages;
          if (!(ok = mbar_wait(bar(C::B_QEMPTY + qs), ((qi / kQStages) & 1) ^ 1, abort_flag, p.status)))
            break;
          mbar_arrive_expect_tx(bar(C::B_QFULL + qs), C::kQStage);
          lastQ[qs] = (qi / kQStages) & 1;
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_3d(smQ + qs * C::kQStage + pn * 32768, &tmQ, bar(C::B_QFULL + qs), pn * 64,
                        x.s0 + x.qb * p.b, x.h * p.G + ch * heads_per_chunk);
          for (int mt = 0; ok && mt < nmt; ++mt)
            for (int part = p.parts - 1; ok && part >= 0; --part)
              for (int pn = 0; pn < C::kPanels; ++pn, ++ai) {
                const int as = ai % kAStages;
                if (!(ok = mbar_wait(bar(C::B_AEMPTY + as), ((ai / kAStages) & 1) ^ 1, abort_flag,
                                     p.status)))
                  break;
                mbar_arrive_expect_tx(bar(C::B_AFULL + as), kAStage);
                lastA[as] = (ai / kAStages) & 1;
                tma_load_3d(smA + as * kAStage, &tmC, bar(C::B_AFULL + as), pn * 64,
                            crow + 128 * mt, part);
              }
        }
      }
      if (!ok) {
        for (int s = 0; s < kQStages; ++s)
          if (lastQ[s] >= 0) mbar_wait_drain(bar(C::B_QFULL + s), lastQ[s]);
        for (int s = 0; s < kAStages; ++s)
          if (lastA[s] >= 0) mbar_wait_drain(bar(C::B_AFULL + s), lastA[s]);
      }
    }
  } else if (warp == kMmaWarp) {
    // Lane 0 issues; the whole warp takes the named barriers, once per chunk and panel
    // whether or not a wait gave up, so the watcher's and its own always pair up.
    int qi = 0, ai = 0, di = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const RUnit x = runit(p, u);
      if (!x.valid) continue;
      const int nmt = (x.r + 127) / 128;
      for (int ch = 0; ch < p.nch; ++ch, ++qi) {
        const int qs = qi % kQStages;
        const uint32_t idesc = idesc_bf16(128, chunk_cols(p, ch), false);
        nbar_sync(kNbQ, kNbThreads);  // the query chunk landed
        for (int mt = 0; mt < nmt; ++mt, ++di) {
          const int db = di % 2;
          if (lane == 0 && ok)
            ok = mbar_wait(bar(C::B_DEMPTY + db), ((di / 2) & 1) ^ 1, abort_flag, p.status);
          __syncwarp();
          bool first = true;
          for (int part = p.parts - 1; part >= 0; --part)
            for (int pn = 0; pn < C::kPanels; ++pn, ++ai) {
              const int as = ai % kAStages;
              nbar_sync(kNbA, kNbThreads);  // the summary panel landed
              if (lane == 0 && ok) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  const uint64_t a = sdesc_sw128(smA + as * kAStage + kk * 32, 16, 1024);
                  const uint64_t bdesc =
                      sdesc_sw128(smQ + qs * C::kQStage + pn * 32768 + kk * 32, 16, 1024);
                  mma_bf16_ss(tmem + db * 256, a, bdesc, idesc, first ? 0u : 1u);
                  first = false;
                }
                mma_commit(bar(C::B_AEMPTY + as));
              }
              __syncwarp();
            }
          if (lane == 0 && ok) mma_commit(bar(C::B_DFULL + db));
          __syncwarp();
        }
        if (lane == 0 && ok) mma_commit(bar(C::B_QEMPTY + qs));
        __syncwarp();
      }
    }
    if (lane == 0) {
      mma_commit(bar(C::B_FINAL));
      mbar_wait_drain(bar(C::B_FINAL), 0);
    }
    __syncwarp();
  } else if (warp == kWatchWarp) {
    // ------------------------------------------------------------ copy watcher
    int qi = 0, ai = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const RUnit x = runit(p, u);
      if (!x.valid) continue;
      const int nmt = (x.r + 127) / 128;
      for (int ch = 0; ch < p.nch; ++ch, ++qi) {
        const int qs = qi % kQStages;
        if (lane == 0 && ok)
          ok = mbar_wait(bar(C::B_QFULL + qs), (qi / kQStages) & 1, abort_flag, p.status);
        __syncwarp();
        ok = __shfl_sync(0xffffffffu, ok, 0);
        nbar_sync(kNbQ, kNbThreads);
        for (int mt = 0; mt < nmt; ++mt)
          for (int part = p.parts - 1; part >= 0; --part)
            for (int pn = 0; pn < C::kPanels; ++pn, ++ai) {
              const int as = ai % kAStages;
              if (lane == 0 && ok)
                ok = mbar_wait(bar(C::B_AFULL + as), (ai / kAStages) & 1, abort_flag, p.status);
              __syncwarp();
              ok = __shfl_sync(0xffffffffu, ok, 0);
              nbar_sync(kNbA, kNbThreads);
            }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-3)
    const int row = warp * 32 + lane;  // TMEM lane = summary within the M-tile
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    int di = 0, qi = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total; u += gridDim.x) {
      const RUnit x = runit(p, u);
      if (!x.valid) continue;
      const int nmt = (x.r + 127) / 128;
      const size_t srow = (size_t)(x.i * p.Hk + x.h) * p.Nq + x.qb;
      float *Srow = p.S + srow * p.Nk;
      const bool full = x.nvalid == p.b;
      for (int ch = 0; ok && ch < p.nch; ++ch, ++qi) {
        const int ncols = chunk_cols(p, ch);
        if (p.Qn != nullptr) {
          // Largest norm of the chunk's valid query rows, read from the staged chunk:
          // thread t takes rows t and t + 128; a row's 16-byte pieces are summed in
          // a rotated order (the sum ignores the swizzle; the rotation spreads the
          // quarter-warp's loads over all banks).
          const int qs = qi % kQStages;
          if (!(ok = mbar_wait(bar(C::B_QFULL + qs), (qi / kQStages) & 1, abort_flag, p.status)))
            break;
          float nmax = 0.f;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int rho = row + 128 * half;
            if (rho < ncols && (rho % p.b) < x.nvalid) {
              float ss = 0.f;
#pragma unroll
              for (int pn = 0; pn < C::kPanels; ++pn)
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  const uint8_t *src = sm + C::kOffQ + qs * C::kQStage + pn * 32768 + rho * 128 +
                                       (((k + rho) & 7) << 4);
                  const uint4 v = *reinterpret_cast<const uint4 *>(src);
                  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
                    ss = fmaf(lo, lo, fmaf(hi, hi, ss));
                  }
                }
              nmax = fmaxf(nmax, ss);
            }
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) nmax = fmaxf(nmax, __shfl_xor_sync(0xffffffffu, nmax, off));
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bar(C::B_QEMPTY + qs));
            // a bound, so rounded up: sqrt is correctly rounded; the sum of squares
            // of d terms is within d 2^-24 of exact
            const float nrm = sqrtf(nmax) * 1.0001f;
            atomicMax(reinterpret_cast<int *>(p.Qn + srow), __float_as_int(nrm));
          }
        }
        for (int mt = 0; mt < nmt; ++mt, ++di) {
          const int db = di % 2;
          if (!(ok = mbar_wait(bar(C::B_DFULL + db), (di / 2) & 1, abort_flag, p.status))) break;
          tc_fence_after();
          float m = -INFINITY;
          int c0 = 0;
          if (full)  // every column valid: 128 at a time with the reducing load
            for (; c0 + 128 <= ncols; c0 += 128)
              m = fmaxf(m, tmem_max128(tmem + lane_base + db * 256 + c0));
          for (; c0 < ncols; c0 += 32) {
            uint32_t rr[32];
            tmem_ld32(tmem + lane_base + db * 256 + c0, rr);
            if (full) {
#pragma unroll
              for (int c = 0; c < 32; ++c) m = fmaxf(m, __uint_as_float(rr[c]));
            } else {
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (((ch * 256 + c0 + c) % p.b) < x.nvalid) m = fmaxf(m, __uint_as_float(rr[c]));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::B_DEMPTY + db));
          const int j = mt * 128 + row;
          if (j < x.r) Srow[j] = ch == 0 ? m : fmaxf(Srow[j], m);
        }
      }
    }
  }

  grid_dep_launch();  // the next launch may be scheduled; it waits for this grid
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

// One summary row c (D fp32, one warp) -> three bf16 planes with c = hi + mid + lo
// exactly up to the last bf16 rounding (the residuals of bf16 rounding are exact in
// fp32), and the row's norms |c| and |c - hi - mid| for the screen's bound (each
// rounded up: a correctly rounded sqrt of a sum of D squares within D 2^-24).
template <int D>
BSA_DEV void split_row(const float (&c)[D / 32], uint16_t *__restrict__ C3, size_t n, size_t e0,
                       float *cn, float *rn, size_t row, int lane) {
  float sc = 0.f, sr = 0.f;
#pragma unroll
  for (int k = 0; k < D / 32; ++k) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(c[k]);
    const float r1 = c[k] - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    const size_t e = e0 + k;
    C3[e] = *reinterpret_cast<const uint16_t *>(&hi);
    C3[n + e] = *reinterpret_cast<const uint16_t *>(&mid);
    C3[2 * n + e] = *reinterpret_cast<const uint16_t *>(&lo);
    sc = fmaf(c[k], c[k], sc);
    sr = fmaf(r2, r2, sr);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    sc += __shfl_xor_sync(0xffffffffu, sc, off);
    sr += __shfl_xor_sync(0xffffffffu, sr, off);
  }
  if (lane == 0) {
    cn[row] = sqrtf(sc) * 1.0001f;
    rn[row] = sqrtf(sr) * 1.0001f;
  }
}

// C [rows, D] fp32 -> planes [3, rows, D] and norms; one warp per row.  Also zeroes
// the per-row query-norm maxima Qn [qrows] that the score kernel raises.
template <int D>
__global__ void split3_kernel(const float *__restrict__ C, uint16_t *__restrict__ C3,
                              float *__restrict__ cn, float *__restrict__ rn, float *__restrict__ Qn,
                              int32_t *qlen, size_t rows, size_t qrows) {
  grid_dep_wait();  // C comes from the previous launch
  if (qlen != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *qlen = 0;
  const int lane = threadIdx.x % 32;
  const size_t warps = (size_t)gridDim.x * blockDim.x / 32;
  const size_t w0 = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; Qn != nullptr && q < qrows;
       q += (size_t)gridDim.x * blockDim.x)
    Qn[q] = 0.f;
  for (size_t row = w0; row < rows; row += warps) {
    float c[D / 32];
#pragma unroll
    for (int k = 0; k < D / 32; ++k) c[k] = C[row * D + lane * (D / 32) + k];
    split_row<D>(c, C3, rows * D, row * D + lane * (D / 32), cn, rn, row, lane);
  }
  grid_dep_launch();
}

// Chunked prefill: the page summaries of every context block, gathered through
// the block table into rows (i, h, j < N_k) and split three ways as split3_kernel
// does; blocks past a sequence's context, and every block of a sequence whose
// prefix is unusable (flagged here), are zero.
template <int D>
__global__ void gather_split3_kernel(const float *__restrict__ ps, const int32_t *__restrict__ bt,
                                     const int32_t *__restrict__ prefix,
                                     const int32_t *__restrict__ cu, uint16_t *__restrict__ C3,
                                     float *__restrict__ cn, float *__restrict__ rn,
                                     float *__restrict__ Qn, int32_t *qlen, int32_t *status,
                                     int Hk, int Nk, int maxp, int P, int b, size_t rows,
                                     size_t qrows) {
  grid_dep_wait();  // the summaries may come from the previous launch
  if (qlen != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *qlen = 0;
  const int lane = threadIdx.x % 32;
  const size_t warps = (size_t)gridDim.x * blockDim.x / 32;
  const size_t w0 = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; Qn != nullptr && q < qrows;
       q += (size_t)gridDim.x * blockDim.x)
    Qn[q] = 0.f;
  for (size_t row = w0; row < rows; row += warps) {
    const int j = (int)(row % Nk);
    const int ih = (int)(row / Nk);
    const int h = ih % Hk, i = ih / Hk;
    const int pre = prefix[i], len = cu[i + 1] - cu[i];
    const float *src = nullptr;
    if (len == 0) {
      // an idle sequence: no rows
    } else if (chunk_ok(pre, len, b, Nk)) {
      if (j < pre / b + (len + b - 1) / b) {
        const int phys = bt[(size_t)i * maxp + j];
        if (phys >= 0 && phys < P)
          src = ps + ((size_t)phys * Hk + h) * D;
        else if (lane == 0)
          set_status(status, BSA_ERR_CACHE);
      }
    } else if (j == 0 && h == 0 && lane == 0) {
      set_status(status, BSA_ERR_CACHE);
    }
    float c[D / 32];
#pragma unroll
    for (int k = 0; k < D / 32; ++k) c[k] = src != nullptr ? src[lane * (D / 32) + k] : 0.f;
    split_row<D>(c, C3, rows * D, row * D + lane * (D / 32), cn, rn, row, lane);
  }
  grid_dep_launch();
}

// Workspace of the tensor-core scores: the split planes [3, rows_c, D] bf16, then
// |c| and |c - hi - mid| per summary row (fp32), then the per-row query-norm maxima
// [B * H_kv * N_q] (fp32).
size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

struct RouteTcWs {
  uint16_t *C3;
  float *cn, *rn, *Qn;
};

RouteTcWs route_tc_ws(const bsa_shape_t &s, const bsa_kv_cache_t *cache, void *ws) {
  const int Nk = cache != nullptr ? cache->max_context_blocks : s.max_blocks;
  const size_t rows = (size_t)s.num_seqs * s.num_kv_heads * Nk;
  char *w = static_cast<char *>(ws);
  RouteTcWs r;
  r.C3 = reinterpret_cast<uint16_t *>(w);
  w += up256(rows * s.head_dim * 3 * sizeof(uint16_t));
  r.cn = reinterpret_cast<float *>(w);
  w += up256(rows * sizeof(float));
  r.rn = reinterpret_cast<float *>(w);
  w += up256(rows * sizeof(float));
  r.Qn = reinterpret_cast<float *>(w);
  return r;
}

// C == nullptr: a chunk over the paged cache (summaries gathered from it).
template <int D>
cudaError_t launch_d(const bsa_shape_t &s, const void *Q, const float *C,
                     const bsa_kv_cache_t *cache, float *S, bool screen, void *ws,
                     int32_t *qlen, int32_t *dev_status, cudaStream_t st) {
  using Cf = RCfg<D>;
  const int Nk = cache != nullptr ? cache->max_context_blocks : s.max_blocks;
  const size_t rows = (size_t)s.num_seqs * s.num_kv_heads * Nk;
  const size_t qrows = (size_t)s.num_seqs * s.num_kv_heads * s.max_blocks;
  const RouteTcWs w = route_tc_ws(s, cache, ws);
  float *Qn = screen ? w.Qn : nullptr;
  const dim3 sgrid((unsigned)std::min<size_t>((rows * 32 + 255) / 256, 4096));
  cudaError_t e0 =
      cache != nullptr
          ? launch_dependent(gather_split3_kernel<D>, sgrid, dim3(256), 0, st, cache->page_summ,
                             cache->block_table, cache->prefix_lens, s.cu_seqlens, w.C3, w.cn,
                             w.rn, Qn, qlen, dev_status, s.num_kv_heads, Nk,
                             cache->max_pages_per_req, cache->num_phys_pages, s.block, rows, qrows)
          : launch_dependent(split3_kernel<D>, sgrid, dim3(256), 0, st, C, w.C3, w.cn, w.rn, Qn,
                             qlen, rows, qrows);
  if (e0 != cudaSuccess) return e0;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int G = s.num_heads / s.num_kv_heads;
  CUtensorMap mq, mc;
  if (!make_tmap_3d_bf16(&mq, Q, D, s.total_tokens, s.num_heads, 64, s.block, 256 / s.block) ||
      !make_tmap_3d_bf16(&mc, w.C3, D, rows, 3, 64, 128, 1))
    return cudaErrorInvalidValue;
  RouteTcParams p;
  p.cu = s.cu_seqlens;
  p.qoff = cache != nullptr ? cache->prefix_lens : nullptr;
  p.Nk = Nk;
  p.S = S;
  p.Qn = Qn;
  p.status = dev_status;
  p.B = s.num_seqs;
  p.Nq = s.max_blocks;
  p.Hk = s.num_kv_heads;
  p.G = G;
  p.b = s.block;
  p.nch = (G * s.block + 255) / 256;
  p.parts = screen ? 2 : 3;
  e = cudaFuncSetAttribute(route_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cf::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = (int)std::min<size_t>(num_sms(), std::max<size_t>(1, rows));
  return launch_dependent(route_tc_kernel<D>, dim3(grid), dim3(kThreads), Cf::kSmemBytes, st, mq,
                          mc, p);
}

}  // namespace

size_t route_tc_workspace_bytes(const bsa_shape_t &s, const bsa_kv_cache_t *cache) {
  const int Nk = cache != nullptr ? cache->max_context_blocks : s.max_blocks;
  const size_t rows = (size_t)s.num_seqs * s.num_kv_heads * Nk;
  const size_t qrows = (size_t)s.num_seqs * s.num_kv_heads * s.max_blocks;
  return up256(rows * s.head_dim * 3 * sizeof(uint16_t)) + 2 * up256(rows * sizeof(float)) +
         up256(qrows * sizeof(float));
}

RouteScreen route_tc_screen(const bsa_shape_t &s, const bsa_kv_cache_t *cache, void *ws) {
  const RouteTcWs w = route_tc_ws(s, cache, ws);
  RouteScreen r;
  r.C3 = w.C3;
  r.cn = w.cn;
  r.rn = w.rn;
  r.Qn = w.Qn;
  r.c3_rows = (size_t)s.num_seqs * s.num_kv_heads *
              (cache != nullptr ? cache->max_context_blocks : s.max_blocks);
  return r;
}

cudaError_t launch_route_scores_tc(const bsa_shape_t &s, const void *Q, const float *C,
                                   const bsa_kv_cache_t *cache, float *S, bool screen, void *ws,
                                   int32_t *qlen, int32_t *dev_status, cudaStream_t st) {
  if (s.head_dim == 64) return launch_d<64>(s, Q, C, cache, S, screen, ws, qlen, dev_status, st);
  return launch_d<128>(s, Q, C, cache, S, screen, ws, qlen, dev_status, st);
}

}  // namespace bsa
