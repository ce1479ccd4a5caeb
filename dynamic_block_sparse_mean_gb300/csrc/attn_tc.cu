// a5, BF16 tensor-core path: exact attention on the selected tiles only
// ("2.1 · 粗粒度选择" §1.2: eq.(1) address list, eq.(2) S = Q_r K_j^T / sqrt(d_h),
// masks before the softmax, online-softmax recurrences (3)-(5), output u / l).
//
// Persistent kernel, one CTA per SM.  A work unit is (router row, pair of
// M-tiles): the G*b query rows of a row (all query heads of the KV-head group
// share the row's blocks, GQA) are cut into 128-row M-tiles, two per CTA, so
// every K/V tile staged in shared memory feeds 256 query rows.
//
// Warp roles (320 threads):
//   warps 0-3  softmax / epilogue for M-tile 0 (thread = one query row = one TMEM lane)
//   warps 4-7  softmax / epilogue for M-tile 1
//   warp 8     TMA producer: Q tiles, then K_j and V_j of each selected block j
//   warp 9     MMA issuer (one thread): S_t = Q_t K_j^T into TMEM, O_t += P_t V_j
// TMEM (512 columns): O_0, O_1 (d columns each) and S_0, S_1 (b columns each).
// P is written by the softmax threads into shared memory in the 128-byte
// swizzled K-major layout the MMA reads.
//
// The running max used for the exponentials is refreshed only when the row max
// grows by more than 8 (log2 units); O and l are then rescaled in TMEM.  u / l is
// unchanged by the choice of reference, so this is eqs.(3)-(5) with a lagged m.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace bsa {
namespace {

constexpr int kThreads = 320;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;

template <int D, int BK>
struct Cfg {
  static constexpr int kPanels = D / 64;      // 128-byte panels along d
  static constexpr int kPPanels = BK / 64;    // 128-byte panels of P along the keys
  static constexpr int kQTile = 128 * D * 2;
  static constexpr int kKVTile = BK * D * 2;
  static constexpr int kPTile = 128 * BK * 2;
  static constexpr int NSK = (D == 128 && BK == 128) ? 2 : 3;
  static constexpr int NSV = (D == 128 && BK == 128) ? 1 : 3;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQTile;
  static constexpr int kOffV = kOffK + NSK * kKVTile;
  static constexpr int kOffP = kOffV + NSV * kKVTile;
  static constexpr int kOffBar = kOffP + 2 * kPTile;
  // barrier slots
  static constexpr int B_QFULL = 0, B_QEMPTY = 1;
  static constexpr int B_KFULL = 2, B_KEMPTY = B_KFULL + NSK;
  static constexpr int B_VFULL = B_KEMPTY + NSK, B_VEMPTY = B_VFULL + NSV;
  static constexpr int B_SFULL = B_VEMPTY + NSV, B_PFULL = B_SFULL + 2;
  static constexpr int B_ODONE = B_PFULL + 2, B_OFREE = B_ODONE + 2;
  static constexpr int B_FINAL = B_OFREE + 2;
  static constexpr int kNumBars = B_FINAL + 1;
  static constexpr int kOffCtl = kOffBar + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kSmemUsed = kOffCtl + 16;
  // 1 KB for base alignment; at least 120 KB so that exactly one CTA (which owns
  // all 512 TMEM columns) is resident per SM.
  static constexpr int kSmemBytes = kSmemUsed + 1024 < 120 * 1024 ? 120 * 1024 : kSmemUsed + 1024;
  // TMEM columns of O_t and S_t
  BSA_DEV static uint32_t colO(int t) { return (uint32_t)(t * D); }
  BSA_DEV static uint32_t colS(int t) { return 256u + (uint32_t)(t * BK); }
  static constexpr uint32_t kIdescQK = idesc_bf16(128, BK, false);
  static constexpr uint32_t kIdescPV = idesc_bf16(128, D, true);
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(256 + 2 * BK <= kTmemCols && 2 * D <= 256, "TMEM budget");
};

struct AttnParams {
  const int32_t *cu;
  const int32_t *row_ptr;
  const int32_t *col_idx;
  const int32_t *work;
  const int32_t *bucket_off;
  uint16_t *O;
  float *lse;
  int32_t *status;
  int T, H, Hk, G, Nq, mtiles, npairs;
  float scale_log2;
};

struct Unit {
  int row, r, h, i, s0, n, kv0, nkv, pair, nt;
};

BSA_DEV Unit decode_unit(const AttnParams &p, int u) {
  Unit x;
  const int slot = u / p.npairs;
  x.pair = u - slot * p.npairs;
  x.row = __ldg(p.work + slot);
  x.r = x.row % p.Nq;
  x.h = (x.row / p.Nq) % p.Hk;
  x.i = x.row / (p.Nq * p.Hk);
  x.s0 = __ldg(p.cu + x.i);
  x.n = __ldg(p.cu + x.i + 1) - x.s0;
  x.kv0 = __ldg(p.row_ptr + x.row);
  x.nkv = __ldg(p.row_ptr + x.row + 1) - x.kv0;
  x.nt = min(2, p.mtiles - 2 * x.pair);
  return x;
}

template <int D, int BK>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using C = Cfg<D, BK>;
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
    mbar_init(bar(C::B_QFULL), 1);
    mbar_init(bar(C::B_QEMPTY), 1);
    for (int s = 0; s < C::NSK; ++s) {
      mbar_init(bar(C::B_KFULL + s), 1);
      mbar_init(bar(C::B_KEMPTY + s), 1);
    }
    for (int s = 0; s < C::NSV; ++s) {
      mbar_init(bar(C::B_VFULL + s), 1);
      mbar_init(bar(C::B_VEMPTY + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::B_SFULL + t), 1);
      mbar_init(bar(C::B_PFULL + t), 4);
      mbar_init(bar(C::B_ODONE + t), 1);
      mbar_init(bar(C::B_OFREE + t), 4);
    }
    mbar_init(bar(C::B_FINAL), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int total_units = __ldg(p.bucket_off + BSA_NUM_BUCKETS) * p.npairs;
  const uint32_t smQ = sbase + C::kOffQ, smK = sbase + C::kOffK;
  const uint32_t smV = sbase + C::kOffV, smP = sbase + C::kOffP;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int kv_g = 0, ucount = 0;
      int issuedK[C::NSK], issuedV[C::NSV], issuedQ = -1;
      for (int s = 0; s < C::NSK; ++s) issuedK[s] = -1;
      for (int s = 0; s < C::NSV; ++s) issuedV[s] = -1;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x, ++ucount) {
        const Unit x = decode_unit(p, u);
        if (!(ok = mbar_wait(bar(C::B_QEMPTY), (ucount & 1) ^ 1, abort_flag, p.status))) break;
        mbar_arrive_expect_tx(bar(C::B_QFULL), x.nt * C::kQTile);
        issuedQ = ucount & 1;
        for (int t = 0; t < x.nt; ++t) {
          const int hq0 = x.h * p.G + ((2 * x.pair + t) * 128) / BK;
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_3d(smQ + t * C::kQTile + pn * 16384, &tmQ, bar(C::B_QFULL), pn * 64,
                        x.s0 + x.r * BK, hq0);
        }
        for (int j = 0; j < x.nkv; ++j, ++kv_g) {
          const int kb = __ldg(p.col_idx + x.kv0 + j);
          const int y = x.s0 + kb * BK;
          const int ks = kv_g % C::NSK, vs = kv_g % C::NSV;
          if (!(ok = mbar_wait(bar(C::B_KEMPTY + ks), ((kv_g / C::NSK) & 1) ^ 1, abort_flag,
                               p.status)))
            break;
          mbar_arrive_expect_tx(bar(C::B_KFULL + ks), C::kKVTile);
          issuedK[ks] = (kv_g / C::NSK) & 1;
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_3d(smK + ks * C::kKVTile + pn * (BK * 128), &tmK, bar(C::B_KFULL + ks),
                        pn * 64, y, x.h);
          if (!(ok = mbar_wait(bar(C::B_VEMPTY + vs), ((kv_g / C::NSV) & 1) ^ 1, abort_flag,
                               p.status)))
            break;
          mbar_arrive_expect_tx(bar(C::B_VFULL + vs), C::kKVTile);
          issuedV[vs] = (kv_g / C::NSV) & 1;
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_3d(smV + vs * C::kKVTile + pn * (BK * 128), &tmV, bar(C::B_VFULL + vs),
                        pn * 64, y, x.h);
        }
      }
      if (!ok) {  // let every copy already in flight land before the CTA leaves
        if (issuedQ >= 0) mbar_wait_drain(bar(C::B_QFULL), issuedQ);
        for (int s = 0; s < C::NSK; ++s)
          if (issuedK[s] >= 0) mbar_wait_drain(bar(C::B_KFULL + s), issuedK[s]);
        for (int s = 0; s < C::NSV; ++s)
          if (issuedV[s] >= 0) mbar_wait_drain(bar(C::B_VFULL + s), issuedV[s]);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int kv_g = 0, ucount = 0;
      int kvt[2] = {0, 0}, ut[2] = {0, 0};
      bool ok = true;
      auto issue_qk = [&](int t, int ks) {
        const uint32_t qa = smQ + t * C::kQTile, kbse = smK + ks * C::kKVTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk % 4) * 32u;
          const uint64_t a = sdesc_sw128(qa + (kk / 4) * 16384 + off, 16, 1024);
          const uint64_t b = sdesc_sw128(kbse + (kk / 4) * (BK * 128) + off, 16, 1024);
          mma_bf16_ss(tmem + C::colS(t), a, b, C::kIdescQK, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int vs, bool acc) {
        const uint32_t pa = smP + t * C::kPTile, vb = smV + vs * C::kKVTile;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t a = sdesc_sw128(pa + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(vb + kk * 2048, BK * 128, 1024);
          mma_bf16_ss(tmem + C::colO(t), a, b, C::kIdescPV, (acc || kk > 0) ? 1u : 0u);
        }
      };
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x, ++ucount) {
        const Unit x = decode_unit(p, u);
        if (!(ok = mbar_wait(bar(C::B_QFULL), ucount & 1, abort_flag, p.status))) break;
        tc_fence_after();
        {
          const int ks = kv_g % C::NSK;
          if (!(ok = mbar_wait(bar(C::B_KFULL + ks), (kv_g / C::NSK) & 1, abort_flag, p.status)))
            break;
          tc_fence_after();
          for (int t = 0; t < x.nt; ++t) {
            issue_qk(t, ks);
            mma_commit(bar(C::B_SFULL + t));
          }
          mma_commit(bar(C::B_KEMPTY + ks));
          if (x.nkv == 1) mma_commit(bar(C::B_QEMPTY));
        }
        for (int j = 0; ok && j < x.nkv; ++j) {
          const int g = kv_g + j;
          const int vs = g % C::NSV;
          if (!(ok = mbar_wait(bar(C::B_VFULL + vs), (g / C::NSV) & 1, abort_flag, p.status)))
            break;
          tc_fence_after();
          for (int t = 0; t < x.nt; ++t) {
            if (!(ok = mbar_wait(bar(C::B_PFULL + t), kvt[t] & 1, abort_flag, p.status))) break;
            tc_fence_after();
            if (j == 0) {
              if (!(ok = mbar_wait(bar(C::B_OFREE + t), (ut[t] & 1) ^ 1, abort_flag, p.status)))
                break;
              tc_fence_after();
            }
            issue_pv(t, vs, j > 0);
            mma_commit(bar(C::B_ODONE + t));
            ++kvt[t];
            if (j + 1 < x.nkv) {
              const int ks1 = (g + 1) % C::NSK;
              if (t == 0) {
                if (!(ok = mbar_wait(bar(C::B_KFULL + ks1), ((g + 1) / C::NSK) & 1, abort_flag,
                                     p.status)))
                  break;
                tc_fence_after();
              }
              issue_qk(t, ks1);
              mma_commit(bar(C::B_SFULL + t));
            }
          }
          if (!ok) break;
          mma_commit(bar(C::B_VEMPTY + vs));
          if (j + 1 < x.nkv) {
            mma_commit(bar(C::B_KEMPTY + (g + 1) % C::NSK));
            if (j + 2 == x.nkv) mma_commit(bar(C::B_QEMPTY));
          }
        }
        for (int t = 0; t < x.nt; ++t) ++ut[t];
        kv_g += x.nkv;
      }
      // Every MMA issued so far completes before TMEM is released.
      mma_commit(bar(C::B_FINAL));
      mbar_wait_drain(bar(C::B_FINAL), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int t = warp / 4;           // M-tile of this warpgroup
    const int wq = warp % 4;          // TMEM lane quarter
    const int rho = wq * 32 + lane;   // row of the M-tile
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::colS(t);
    const uint32_t tO = tmem + lane_base + C::colO(t);
    uint8_t *Prow = sm + C::kOffP + t * C::kPTile + rho * 128;
    int kvt = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
      const Unit x = decode_unit(p, u);
      if (t >= x.nt) continue;
      const int grow = (2 * x.pair + t) * 128 + rho;   // row within the group's G*b rows
      const bool row_valid = grow < p.G * BK;
      const int hq = x.h * p.G + grow / BK;
      const int tq = x.r * BK + grow % BK;             // sequence-relative query position
      const int tok_in_blk = grow % BK;
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < x.nkv; ++j) {
        const int kb = __ldg(p.col_idx + x.kv0 + j);
        if (!(ok = mbar_wait(bar(C::B_SFULL + t), kvt & 1, abort_flag, p.status))) break;
        tc_fence_after();
        float s[BK];
#pragma unroll
        for (int c0 = 0; c0 < BK; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(tS + c0, rr);
#pragma unroll
          for (int c = 0; c < 32; ++c) s[c0 + c] = __uint_as_float(rr[c]);
        }
        if (kb == x.r) {  // diagonal block: token-level causal triangle
#pragma unroll
          for (int c = 0; c < BK; ++c)
            if (c > tok_in_blk) s[c] = -INFINITY;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < BK; ++c) mx = fmaxf(mx, s[c]);
        const float m_new = fmaxf(m_used, mx * p.scale_log2);
        if (j > 0) {
          // PV of the previous block must be done before O is rescaled or P rewritten.
          if (!(ok = mbar_wait(bar(C::B_ODONE + t), (kvt - 1) & 1, abort_flag, p.status))) break;
          tc_fence_after();
          const bool resc = m_new > m_used + kRescaleThreshold;
          if (__any_sync(0xffffffffu, resc)) {
            const float alpha = resc ? fast_exp2(m_used - m_new) : 1.f;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t rr[32];
              tmem_ld32(tO + c0, rr);
#pragma unroll
              for (int c = 0; c < 32; ++c) rr[c] = __float_as_uint(__uint_as_float(rr[c]) * alpha);
              tmem_st32(tO + c0, rr);
            }
            l *= alpha;
            if (resc) m_used = m_new;
          }
        } else {
          m_used = m_new;
        }
        const float mref = (m_used == -INFINITY) ? 0.f : m_used;
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < BK; ++c) {
          s[c] = fast_exp2(fmaf(s[c], p.scale_log2, -mref));
          rs += s[c];
        }
        l += rs;
        // P row -> shared memory, 128-byte swizzled K-major (16-byte chunk c8 of row rho at c8 ^ (rho & 7)).
#pragma unroll
        for (int c8 = 0; c8 < BK / 8; ++c8) {
          const int pn = c8 / 8, ch = c8 % 8;
          uint4 v;
          v.x = pack_bf16x2(s[c8 * 8 + 0], s[c8 * 8 + 1]);
          v.y = pack_bf16x2(s[c8 * 8 + 2], s[c8 * 8 + 3]);
          v.z = pack_bf16x2(s[c8 * 8 + 4], s[c8 * 8 + 5]);
          v.w = pack_bf16x2(s[c8 * 8 + 6], s[c8 * 8 + 7]);
          *reinterpret_cast<uint4 *>(Prow + pn * 16384 + ((ch ^ (rho & 7)) * 16)) = v;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_PFULL + t));
        ++kvt;
      }
      if (!ok) break;
      // epilogue: O = u / l, lse = (m + log2 l) ln 2
      if (!(ok = mbar_wait(bar(C::B_ODONE + t), (kvt - 1) & 1, abort_flag, p.status))) break;
      tc_fence_after();
      const bool store = row_valid && tq < x.n;
      const float inv_l = 1.f / l;
      uint16_t *orow = p.O + ((size_t)hq * p.T + x.s0 + tq) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(tO + c0, rr);
        if (store) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + c0);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(rr[q4 * 8 + 0]) * inv_l, __uint_as_float(rr[q4 * 8 + 1]) * inv_l);
            v.y = pack_bf16x2(__uint_as_float(rr[q4 * 8 + 2]) * inv_l, __uint_as_float(rr[q4 * 8 + 3]) * inv_l);
            v.z = pack_bf16x2(__uint_as_float(rr[q4 * 8 + 4]) * inv_l, __uint_as_float(rr[q4 * 8 + 5]) * inv_l);
            v.w = pack_bf16x2(__uint_as_float(rr[q4 * 8 + 6]) * inv_l, __uint_as_float(rr[q4 * 8 + 7]) * inv_l);
            dst[q4] = v;
          }
        }
      }
      if (store && p.lse != nullptr)
        p.lse[(size_t)hq * p.T + x.s0 + tq] = (m_used + fast_log2(l)) * 0.6931471805599453f;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_OFREE + t));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

template <int D, int BK>
cudaError_t launch_tc(const bsa_shape_t &s, const void *Q, const void *K, const void *V,
                      const int32_t *row_ptr, const int32_t *col_idx, const int32_t *work,
                      const int32_t *bucket_off, float scale, void *O, float *lse,
                      int32_t *dev_status, cudaStream_t st) {
  using C = Cfg<D, BK>;
  CUtensorMap mq, mk, mv;
  if (!make_tmap_3d_bf16(&mq, Q, D, s.total_tokens, s.num_heads, 64, BK, 128 / BK) ||
      !make_tmap_3d_bf16(&mk, K, D, s.total_tokens, s.num_kv_heads, 64, BK, 1) ||
      !make_tmap_3d_bf16(&mv, V, D, s.total_tokens, s.num_kv_heads, 64, BK, 1))
    return cudaErrorInvalidValue;
  AttnParams p;
  p.cu = s.cu_seqlens;
  p.row_ptr = row_ptr;
  p.col_idx = col_idx;
  p.work = work;
  p.bucket_off = bucket_off;
  p.O = static_cast<uint16_t *>(O);
  p.lse = lse;
  p.status = dev_status;
  p.T = s.total_tokens;
  p.H = s.num_heads;
  p.Hk = s.num_kv_heads;
  p.G = s.num_heads / s.num_kv_heads;
  p.Nq = s.max_blocks;
  p.mtiles = (p.G * BK + 127) / 128;
  p.npairs = (p.mtiles + 1) / 2;
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D, BK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long max_units = (long long)s.num_seqs * s.num_kv_heads * s.max_blocks * p.npairs;
  const int grid = (int)std::min<long long>(num_sms(), std::max<long long>(1, max_units));
  attn_tc_kernel<D, BK><<<grid, kThreads, C::kSmemBytes, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_tc(const bsa_shape_t &s, const void *Q, const void *K,
                                const void *V, const int32_t *row_ptr, const int32_t *col_idx,
                                const int32_t *work, const int32_t *bucket_off, float scale,
                                void *O, float *lse, int32_t *dev_status, cudaStream_t st) {
  if (s.head_dim == 64 && s.block == 64)
    return launch_tc<64, 64>(s, Q, K, V, row_ptr, col_idx, work, bucket_off, scale, O, lse,
                             dev_status, st);
  if (s.head_dim == 64 && s.block == 128)
    return launch_tc<64, 128>(s, Q, K, V, row_ptr, col_idx, work, bucket_off, scale, O, lse,
                              dev_status, st);
  if (s.head_dim == 128 && s.block == 64)
    return launch_tc<128, 64>(s, Q, K, V, row_ptr, col_idx, work, bucket_off, scale, O, lse,
                              dev_status, st);
  return launch_tc<128, 128>(s, Q, K, V, row_ptr, col_idx, work, bucket_off, scale, O, lse,
                             dev_status, st);
}

}  // namespace bsa
