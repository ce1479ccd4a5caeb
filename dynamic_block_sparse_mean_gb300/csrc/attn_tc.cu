// a5, BF16 tensor-core path: exact attention on the selected tiles only
// ("2.1 · 粗粒度选择" §1.2: eq.(1) address list, eq.(2) S = Q_r K_j^T / sqrt(d_h),
// masks before the softmax, online-softmax recurrences (3)-(5), output u / l).
//
// Persistent kernel, one CTA per SM.  A work unit is (router row, pair of
// M-tiles): the G*b query rows of a row (all query heads of the KV-head group
// share the row's blocks, GQA) are cut into 128-row M-tiles, two per CTA, so
// every K/V tile staged in shared memory feeds 256 query rows.
//
// Keys are walked in steps of 128: one 128-key block, or two 64-key blocks
// placed side by side in one shared-memory stage (a trailing odd block is loaded
// twice and its copy masked).  Every MMA therefore has N = 128, the shape at
// which tcgen05 runs at its full rate (N = 64 runs at two thirds).
//
// Warp roles (512 threads):
//   warps 0-3   softmax for M-tile 0 (thread = one query row = one TMEM lane)
//   warps 4-7   softmax for M-tile 1
//   warp 8      TMA producer: Q tiles, then the K and V rows of each key step
//   warps 9-10  MMA issuers, one thread each: warp 9 + t issues M-tile t's products
//   warp 11     idle (completes the warpgroup of warps 8-10)
//   warps 12-15 output epilogue of both M-tiles (warp 12 + q reads TMEM lane quarter q)
// A unit's last softmax step hands each row's 1 / l to the epilogue warpgroup through
// shared memory and goes straight on to the next unit; the epilogue reads O out of
// tensor memory, releases it to the next unit's PV and writes the tile out while the
// softmax already works on the next unit.  The warpgroups split the register file
// (setmaxnreg): the softmax takes more than the 128 registers a thread has at launch,
// the TMA / MMA warps and the epilogue give theirs up.
// TMEM (512 columns): O_0, O_1 (d columns each), S_0, S_1 (128 columns each).  The
// softmax overwrites the first 64 columns of S_t with P (bf16 pairs) and the PV
// product reads P straight from tensor memory.
//
// Issue order of M-tile t's MMA thread for step s (one batch):
//     PV_t(s)   [after P_t(s)]      O_t += P_t(s) V(s)
//     QK_t(s+1) [after K(s+1)]      S_t  = Q_t K(s+1)^T
// tcgen05.mma operations of one thread execute in issue order, so QK_t(s+1)
// overwrites S_t only after PV_t(s) has read P_t(s).  Each M-tile has its own
// issuing thread, and the two alternate batch by batch (a ping-pong of two named
// barriers, which unlike an mbarrier do not wait behind the MMAs' shared-memory
// operand reads), so the tensor pipe sees PV_0 QK_0 | PV_1 QK_1 | PV_0 ... and the two
// tiles' softmaxes stay half a step apart.  A barrier check stalls its own
// thread's MMA issue for about a hundred cycles, even on a completed phase
// (measured on GB300: four checks per 32 MMAs of one thread slow the pipe from 64
// to 80 cycles per MMA; two threads with the same checks keep it at 64), so each
// issuer's checks now overlap the other tile's batch.  A K / V stage and the Q
// tiles are released by one commit of each issuer; an issuer without a tile in a
// unit walks its steps all the same.
//
// The running max used for the exponentials is refreshed only when the row max
// grows by more than 8 (log2 units); O and l are then rescaled in TMEM.  u / l is
// unchanged by the choice of reference, so this is eqs.(3)-(5) with a lagged m.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace bsa {
namespace {

constexpr int kThreads = 512;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;    // M-tile 0's issuer; M-tile 1's is kMmaWarp + 1; owns TMEM
constexpr int kEpiWarp = 12;   // first of the four epilogue warps
// Registers per thread after the split, for the softmax warpgroups, the warpgroup of
// the TMA and MMA warps, and the epilogue warpgroup.  The four warpgroups hold
// 4 x 128 x 128 registers at launch, and the split must stay within them (an
// increase waits until other warpgroups have released enough).
constexpr uint32_t kRegSoftmax = 176, kRegIssue = 56, kRegEpi = 104;
static_assert(2 * kRegSoftmax + kRegIssue + kRegEpi <= 4 * 128, "register split");
constexpr int kTmemCols = 512;
constexpr int kStep = 128;  // keys per step
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kNbTurn = 1;  // named barriers 1, 2: the issuers' turns
constexpr uint32_t kNbP = 3;     // named barriers 3, 4: P_t written (warpgroup t + issuer t)

template <int D, int BK>
struct Cfg {
  static constexpr int kPanels = D / 64;        // 128-byte panels along d
  static constexpr int kBPS = kStep / BK;       // key blocks per step (2 or 1)
  static constexpr int kQTile = 128 * D * 2;
  static constexpr int kStage = kStep * D * 2;  // K (or V) rows of one step
  static constexpr int kPanel = kStep * 128;    // one 128-byte panel of a stage
  static constexpr int NS = D == 128 ? 2 : 4;   // K/V stages
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQTile;
  static constexpr int kOffV = kOffK + NS * kStage;
  static constexpr int kStageO = 128 * 128;      // output staging: 128 rows x 64 columns
  static constexpr int kOffStageO = kOffV + NS * kStage;  // one half-tile per M-tile
  static constexpr int kOffBar = kOffStageO + 2 * kStageO;
  // barrier slots
  static constexpr int B_QFULL = 0, B_QEMPTY = 1;
  static constexpr int B_KFULL = 2, B_KEMPTY = B_KFULL + NS;
  static constexpr int B_VFULL = B_KEMPTY + NS, B_VEMPTY = B_VFULL + NS;
  static constexpr int B_SFULL = B_VEMPTY + NS;
  static constexpr int B_OFREE = B_SFULL + 2;
  static constexpr int B_OFINAL = B_OFREE + 2;    // all PV of a unit done (once per unit)
  static constexpr int B_OSTAGED = B_OFINAL + 2;  // a staged output half is complete (4 warps)
  static constexpr int B_OSFREE = B_OSTAGED + 2;  // the staging buffer was read by its store
  static constexpr int B_FINAL = B_OSFREE + 2;    // one per issuer
  static constexpr int B_STATS = B_FINAL + 2;     // a unit's 1 / l of tile t staged (4 warps)
  static constexpr int B_STATSFREE = B_STATS + 2; // ... and read by the epilogue (4 warps)
  static constexpr int kNumBars = B_STATSFREE + 2;
  static constexpr int kOffCtl = kOffBar + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kOffStat = kOffCtl + 16;           // 1 / l of each tile's 128 rows
  static constexpr int kSmemUsed = kOffStat + 2 * 128 * 4;
  // 1 KB for base alignment; at least 120 KB so that exactly one CTA (which owns
  // all 512 TMEM columns) is resident per SM.
  static constexpr int kSmemBytes = kSmemUsed + 1024 < 120 * 1024 ? 120 * 1024 : kSmemUsed + 1024;
  BSA_DEV static uint32_t colO(int t) { return (uint32_t)(t * D); }
  BSA_DEV static uint32_t colS(int t) { return 256u + (uint32_t)(t * kStep); }
  static constexpr uint32_t kIdescQK = idesc_bf16(128, kStep, false);
  static constexpr uint32_t kIdescPV = idesc_bf16(128, D, true);
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(2 * D <= 256, "TMEM budget");
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
  // Chunked prefill over a paged cache (CHUNK kernels only): tokens cached before
  // each sequence's chunk, the block table and its row length.
  const int32_t *qoff;
  const int32_t *bt;
  int maxp;
  int num_phys;   // physical pages of the cache (CHUNK kernels only)
  int T, H, Hk, G, Nq, mtiles, npairs;
  float scale_log2;
};

// A work unit: logical block r of the row (the diagonal) and, in a chunk, its
// query block qb in the packed Q / O (r = qb + the blocks cached before the
// chunk); without a cache both are r.
struct Unit {
  int row, r, qb, h, i, s0, n, kv0, nkv, pair, nt;
};

template <bool CHUNK>
BSA_DEV int qblock(const Unit &x) {
  if constexpr (CHUNK) return x.qb;
  return x.r;
}

template <bool CHUNK>
BSA_DEV Unit decode_unit(const AttnParams &p, int u) {
  Unit x;
  const int slot = u / p.npairs;
  x.pair = u - slot * p.npairs;
  x.row = __ldg(p.work + slot);
  x.r = x.row % p.Nq;
  x.h = (x.row / p.Nq) % p.Hk;
  x.i = x.row / (p.Nq * p.Hk);
  if constexpr (CHUNK) {
    x.qb = x.r;
    x.r += __ldg(p.qoff + x.i) / 64;
  }
  x.s0 = __ldg(p.cu + x.i);
  x.n = __ldg(p.cu + x.i + 1) - x.s0;
  x.kv0 = __ldg(p.row_ptr + x.row);
  x.nkv = __ldg(p.row_ptr + x.row + 1) - x.kv0;
  x.nt = min(2, p.mtiles - 2 * x.pair);
  return x;
}

// Tensor coordinates (token row, head) of the K / V tile of entry jb of a unit's
// row: the packed [H_kv, T, d] layout, or in a chunk the page the block table
// names in the cache viewed as rows of [P * H_kv * 64, d] (the page index is
// clamped to the table; a physical id outside the cache reads zeros).
template <bool CHUNK, int BK>
BSA_DEV int2 kv_coord(const AttnParams &p, const Unit &w, int jb) {
  const int j = checked_index(__ldg(p.col_idx + w.kv0 + jb), 0, w.r, p.status);
  if constexpr (CHUNK) {
    const int pg = min(max(j, 0), p.maxp - 1);
    const int phys =
        checked_index(__ldg(p.bt + (size_t)w.i * p.maxp + pg), 0, p.num_phys - 1, p.status);
    return make_int2((phys * p.Hk + w.h) * 64, 0);
  } else {
    return make_int2(w.s0 + j * BK, w.h);
  }
}

// Same with A (P, bf16 pairs) read from tensor memory.
BSA_DEV void mma_ts_lo(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t hi,
                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 bd;\n\t"
      "mov.b64 bd, {%2, %5};\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(hi)
      : "memory");
}

// Shared -> global tensor store of one box (bulk async group of this thread).
BSA_DEV void tma_store_3d(const CUtensorMap *map, uint32_t src, int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}
BSA_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk store of this thread has finished reading shared memory.
BSA_DEV void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until every committed bulk store of this thread has completed.
BSA_DEV void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }


// 16 TMEM columns of this thread's lane, not waited (tmem_wait_st before the
// values are consumed).
BSA_DEV void tmem_st16_nowait(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

BSA_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 64 consecutive TMEM columns of this thread's lane: two loads, one wait.
BSA_DEV void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]),
        "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
        "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
        "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]),
        "=r"(r[62]), "=r"(r[63])
      : "r"(taddr), "r"(taddr + 32u)
      : "memory");
}

BSA_DEV float max3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}

BSA_DEV uint64_t pack2(float lo, float hi) {
  return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
BSA_DEV float lo_of(uint64_t v) { return __uint_as_float((uint32_t)v); }
BSA_DEV float hi_of(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

BSA_DEV uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
BSA_DEV uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Max of 64 values (tree of three-input maxes).
BSA_DEV float max64(const float (&v)[64]) {
  float a[22];
#pragma unroll
  for (int k = 0; k < 21; ++k) a[k] = max3(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
  a[21] = v[63];
  float b[8];
#pragma unroll
  for (int k = 0; k < 7; ++k) b[k] = max3(a[3 * k], a[3 * k + 1], a[3 * k + 2]);
  b[7] = a[21];
  return max3(max3(b[0], b[1], b[2]), max3(b[3], b[4], b[5]), fmaxf(b[6], b[7]));
}

// Load 64 S columns, apply the step's mask (columns >= lim are -inf; lim = 64
// means none), into floats.
BSA_DEV void load_masked(uint32_t taddr, int lim, float (&v)[64]) {
  uint32_t rr[64];
  tmem_ld64(taddr, rr);
#pragma unroll
  for (int c = 0; c < 64; ++c) v[c] = c < lim ? __uint_as_float(rr[c]) : -INFINITY;
}


// P for one step: S columns 32 q .. 32 q + 31 -> P columns 16 q .. 16 q + 15 (bf16
// pairs), for q = 0..3.  The load of quarter q + 1 is in flight while quarter q is
// exponentiated, and the P stores are waited once at the end; a P quarter only
// overwrites S columns already read.  MASKED applies the step's column limits
// (lim[h] for the half h of 64 columns).  Returns the row sum of the new P.
template <bool MASKED>
BSA_DEV float exp_step(uint32_t tS, uint64_t scale2, uint64_t negm, const int (&lim)[2]) {
  uint32_t buf[2][32];
  uint64_t acc0 = 0, acc1 = 0;
  tmem_ld32_async(tS, buf[0]);
  tmem_wait_ld(buf[0]);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (q < 3) tmem_ld32_async(tS + 32 * (q + 1), buf[(q + 1) & 1]);
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      float a = __uint_as_float(buf[q & 1][2 * c]), b = __uint_as_float(buf[q & 1][2 * c + 1]);
      if (MASKED) {
        const int col = (q & 1) * 32 + 2 * c;  // column within the 64-column half q / 2
        a = col < lim[q >> 1] ? a : -INFINITY;
        b = col + 1 < lim[q >> 1] ? b : -INFINITY;
      }
      const uint64_t z = fma2(pack2(a, b), scale2, negm);
      const float e0 = fast_exp2(lo_of(z)), e1 = fast_exp2(hi_of(z));
      pk[c] = pack_bf16x2(e0, e1);
      if (c & 1)
        acc1 = add2(acc1, pack2(e0, e1));
      else
        acc0 = add2(acc0, pack2(e0, e1));
    }
    tmem_st16_nowait(tS + 16 * q, pk);
    if (q < 3) tmem_wait_ld(buf[(q + 1) & 1]);
  }
  tmem_wait_st();
  const uint64_t acc = add2(acc0, acc1);
  return lo_of(acc) + hi_of(acc);
}

// Warpgroup-wide change of this warp's register allocation (every warp of the
// warpgroup executes the same one).
template <uint32_t R>
BSA_DEV void reg_alloc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}
template <uint32_t R>
BSA_DEV void reg_dealloc() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}

template <int D, int BK, bool CHUNK>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   const AttnParams p) {
  using C = Cfg<D, BK>;
  constexpr int BPS = C::kBPS;
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
    mbar_init(bar(C::B_QEMPTY), 2);  // released by both issuers
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(bar(C::B_KFULL + s), 1);
      mbar_init(bar(C::B_KEMPTY + s), 2);
      mbar_init(bar(C::B_VFULL + s), 1);
      mbar_init(bar(C::B_VEMPTY + s), 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::B_SFULL + t), 1);
      mbar_init(bar(C::B_OFREE + t), 4);
      mbar_init(bar(C::B_OFINAL + t), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::B_OSTAGED + t), 4);
      mbar_init(bar(C::B_OSFREE + t), 1);
      mbar_init(bar(C::B_STATS + t), 4);
      mbar_init(bar(C::B_STATSFREE + t), 4);
    }
    mbar_init(bar(C::B_FINAL), 1);
    mbar_init(bar(C::B_FINAL + 1), 1);
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
  grid_dep_wait();    // Q, K, V and the worklist may come from earlier launches

  const int total_units = __ldg(p.bucket_off + BSA_NUM_BUCKETS) * p.npairs;
  const uint32_t smQ = sbase + C::kOffQ, smK = sbase + C::kOffK, smV = sbase + C::kOffV;

  // Each role changes its register allocation first (warps 8-11 together, each
  // softmax warpgroup, the epilogue warpgroup).
  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    reg_dealloc<kRegIssue>();
    if (lane == 0) {
      int stp = 0, ucount = 0;   // global step counter (stage ring), units
      int issuedK[C::NS], issuedV[C::NS], issuedQ = -1;
      for (int s = 0; s < C::NS; ++s) issuedK[s] = issuedV[s] = -1;
      bool ok = true;
      Unit nx;
      if (blockIdx.x < total_units) nx = decode_unit<CHUNK>(p, blockIdx.x);
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x, ++ucount) {
        const Unit x = nx;
        if (u + (int)gridDim.x < total_units) nx = decode_unit<CHUNK>(p, u + gridDim.x);  // prefetch
        if (!(ok = mbar_wait(bar(C::B_QEMPTY), (ucount & 1) ^ 1, abort_flag, p.status))) break;
        mbar_arrive_expect_tx(bar(C::B_QFULL), x.nt * C::kQTile);
        issuedQ = ucount & 1;
        for (int t = 0; t < x.nt; ++t) {
          const int hq0 = x.h * p.G + ((2 * x.pair + t) * 128) / BK;
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_3d(smQ + t * C::kQTile + pn * 16384, &tmQ, bar(C::B_QFULL), pn * 64,
                        x.s0 + qblock<CHUNK>(x) * BK, hq0);
        }
        const int nsteps = (x.nkv + BPS - 1) / BPS;
        // No copy is prefetched into L2: prefetching the K / V steps one or two steps
        // ahead made the launch slower (128k workload 7.10 ms without, 7.19 one step
        // ahead, 7.30 two; the 2-stage ring already keeps a step ahead), and so did
        // prefetching the next unit's Q tiles at the start of a unit (6.98 ms without).
        for (int s = 0; s < nsteps; ++s, ++stp) {
          int2 y[BPS];
#pragma unroll
          for (int e = 0; e < BPS; ++e)  // a missing block repeats the last one
            y[e] = kv_coord<CHUNK, BK>(p, x, min(s * BPS + e, x.nkv - 1));
          const int st = stp % C::NS;
          const uint32_t ph = ((stp / C::NS) & 1) ^ 1;
          if (!(ok = mbar_wait(bar(C::B_KEMPTY + st), ph, abort_flag, p.status))) break;
          mbar_arrive_expect_tx(bar(C::B_KFULL + st), C::kStage);
          issuedK[st] = ph ^ 1;
#pragma unroll
          for (int e = 0; e < BPS; ++e)
            for (int pn = 0; pn < C::kPanels; ++pn)
              tma_load_3d(smK + st * C::kStage + pn * C::kPanel + e * BK * 128, &tmK,
                          bar(C::B_KFULL + st), pn * 64, y[e].x, y[e].y);
          if (!(ok = mbar_wait(bar(C::B_VEMPTY + st), ph, abort_flag, p.status))) break;
          mbar_arrive_expect_tx(bar(C::B_VFULL + st), C::kStage);
          issuedV[st] = ph ^ 1;
#pragma unroll
          for (int e = 0; e < BPS; ++e)
            for (int pn = 0; pn < C::kPanels; ++pn)
              tma_load_3d(smV + st * C::kStage + pn * C::kPanel + e * BK * 128, &tmV,
                          bar(C::B_VFULL + st), pn * 64, y[e].x, y[e].y);
        }
      }
      if (!ok) {  // let every copy already in flight land before the CTA leaves
        if (issuedQ >= 0) mbar_wait_drain(bar(C::B_QFULL), issuedQ);
        for (int s = 0; s < C::NS; ++s) {
          if (issuedK[s] >= 0) mbar_wait_drain(bar(C::B_KFULL + s), issuedK[s]);
          if (issuedV[s] >= 0) mbar_wait_drain(bar(C::B_VFULL + s), issuedV[s]);
        }
      }
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ------------------------------------------------------------ MMA issuers
    reg_dealloc<kRegIssue>();
    const int t = warp - kMmaWarp;  // the M-tile this warp's lane 0 issues for
    {
      const bool lead = lane == 0;  // waits and issues; the whole warp takes the turns
      int stp = 0, ucount = 0;
      int ks = 0;   // steps of this tile (S / P phases)
      int ut = 0;   // units of this tile (O-free / O-final phases)
      bool ok = true;
      // Descriptors differ only in their low word; K-step offsets within a panel
      // are compile-time constants, so each MMA costs one add.
      const uint32_t qlo0 = desc_lo(smQ, 16), klo0 = desc_lo(smK, 16);
      const uint32_t vlo0 = desc_lo(smV, C::kPanel);
      const uint32_t dhi = kDescHi;
      auto issue_qk = [&](int st) {
        const uint32_t alo = qlo0 + (uint32_t)(t * C::kQTile) / 16u;
        const uint32_t blo = klo0 + (uint32_t)(st * C::kStage) / 16u;
        const uint32_t d = tmem + C::colS(t);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk % 4) * 2u;
          mma_ss_lo(d, alo + (kk / 4) * (16384u / 16u) + off,
                    blo + (kk / 4) * (uint32_t)(C::kPanel / 16) + off, dhi, C::kIdescQK,
                    kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int st, bool acc) {
        const uint32_t blo = vlo0 + (uint32_t)(st * C::kStage) / 16u;
        const uint32_t a = tmem + C::colS(t), d = tmem + C::colO(t);
#pragma unroll
        for (int kk = 0; kk < kStep / 16; ++kk)
          mma_ts_lo(d, a + kk * 8, blo + kk * (2048u / 16u), dhi, C::kIdescPV,
                    (acc || kk > 0) ? 1u : 0u);
      };
      // Batches alternate between the issuers: issuer 0's batch b follows issuer 1's
      // batch b - 1, issuer 1's batch b follows issuer 0's batch b.  The turn passes
      // through two named barriers (issuer 0 -> 1, issuer 1 -> 0) that both warps
      // take once per batch, blocking: a named barrier does not go through shared
      // memory, where an mbarrier check waits behind the MMAs' operand reads.  Both
      // issuers walk every batch of every unit, after a failed wait too (they then
      // skip the waits and the MMAs), so the two barriers always pair up.
      int nb = 0;
      auto my_turn = [&]() {
        __syncwarp();
        if (t == 1) nbar_sync(kNbTurn, 64);
        else if (nb > 0) nbar_sync(kNbTurn + 1, 64);
      };
      auto turn_done = [&]() {
        __syncwarp();
        nbar_sync(kNbTurn + t, 64);
        ++nb;
      };
      auto wait = [&](int b, uint32_t parity) {
        if (lead && ok) ok = mbar_wait(bar(b), parity, abort_flag, p.status);
      };
      Unit nx;
      if (blockIdx.x < total_units) nx = decode_unit<CHUNK>(p, blockIdx.x);
      for (int u = blockIdx.x; u < total_units; u += gridDim.x, ++ucount) {
        const Unit x = nx;
        if (u + (int)gridDim.x < total_units) nx = decode_unit<CHUNK>(p, u + gridDim.x);  // prefetch
        const int nsteps = (x.nkv + BPS - 1) / BPS;
        const bool active = t < x.nt;
        // Every barrier a batch needs is checked before the issuer takes its turn,
        // while the other tile's batch runs; the turn is then the only wait between
        // the two warps' batches.
        wait(C::B_QFULL, ucount & 1);
        {  // QK of step 0
          const int st = stp % C::NS;
          wait(C::B_KFULL + st, (stp / C::NS) & 1);
          my_turn();
          if (lead && ok) {
            tc_fence_after();
            if (active) {
              issue_qk(st);
              mma_commit(bar(C::B_SFULL + t));
            }
            mma_commit(bar(C::B_KEMPTY + st));
            if (nsteps == 1) mma_commit(bar(C::B_QEMPTY));
          }
          turn_done();
        }
        for (int s = 0; s < nsteps; ++s) {
          const int g = stp + s, st = g % C::NS;
          const int g1 = g + 1, st1 = g1 % C::NS;
          const bool more = s + 1 < nsteps;
          wait(C::B_VFULL + st, (g / C::NS) & 1);
          if (active) {
            __syncwarp();
            nbar_sync(kNbP + t, 160);  // P_t(s) is in tensor memory
            if (s == 0) wait(C::B_OFREE + t, (ut & 1) ^ 1);
          }
          if (more) wait(C::B_KFULL + st1, (g1 / C::NS) & 1);
          my_turn();
          if (lead && ok) {
            tc_fence_after();
            if (active) {
              issue_pv(st, s > 0);
              if (!more) mma_commit(bar(C::B_OFINAL + t));
            }
            mma_commit(bar(C::B_VEMPTY + st));
            if (more) {
              if (active) {
                issue_qk(st1);
                mma_commit(bar(C::B_SFULL + t));
              }
              mma_commit(bar(C::B_KEMPTY + st1));
              if (s + 2 == nsteps) mma_commit(bar(C::B_QEMPTY));
            }
          }
          turn_done();
        }
        if (active) {
          ks += nsteps;
          ++ut;
        }
        stp += nsteps;
      }
      // issuer 1's last batch hands the turn to issuer 0 once more
      if (t == 0 && nb > 0) {
        __syncwarp();
        nbar_sync(kNbTurn + 1, 64);
      }
      // Every MMA this thread issued completes before TMEM is released.
      if (lead) {
        mma_commit(bar(C::B_FINAL + t));
        mbar_wait_drain(bar(C::B_FINAL + t), 0);
      }
      __syncwarp();
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax
    reg_alloc<kRegSoftmax>();
    const int t = warp / 4;           // M-tile of this warpgroup
    const int wq = warp % 4;          // TMEM lane quarter
    const int rho = wq * 32 + lane;   // row of the M-tile
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tO = tmem + lane_base + C::colO(t);
    const uint32_t tS = tmem + lane_base + C::colS(t);
    int kstep = 0;                    // steps of this tile (S / P / O-done phases)
    int units = 0;                    // units of this tile (row statistics handed over)
    float *stat_inv_l = reinterpret_cast<float *>(sm + C::kOffStat) + t * 128;
    bool ok = true;
    const uint64_t scale2 = pack2(p.scale_log2, p.scale_log2);
    // Position of the diagonal block r in a unit's row (the token-level triangle),
    // found by the whole warp; -1 if the row does not hold it.
    auto diag_of = [&](const Unit &w) {
      int dj = -1;
      for (int j0 = 0; j0 < w.nkv; j0 += 32) {
        const int j = j0 + lane;
        const unsigned hit =
            __ballot_sync(0xffffffffu, j < w.nkv && __ldg(p.col_idx + w.kv0 + j) == w.r);
        if (hit != 0u && dj < 0) dj = j0 + __ffs(hit) - 1;
      }
      return dj;
    };
    Unit nx;
    int nx_diag = -1;
    if (blockIdx.x < total_units) {
      nx = decode_unit<CHUNK>(p, blockIdx.x);
      nx_diag = diag_of(nx);
    }
    // Every step of every unit of this tile takes the P barrier with issuer t, after a
    // failed wait too (the work is then skipped), so the two sides always pair up.
    for (int u = blockIdx.x; u < total_units; u += gridDim.x) {
      const Unit x = nx;
      const int diag_j = nx_diag;
      const bool has_next = u + (int)gridDim.x < total_units;
      if (has_next) nx = decode_unit<CHUNK>(p, u + gridDim.x);  // prefetch
      if (t >= x.nt) {
        if (has_next) nx_diag = diag_of(nx);
        continue;
      }
      const int nsteps = (x.nkv + BPS - 1) / BPS;
      const int grow = (2 * x.pair + t) * 128 + rho;   // row within the group's G*b rows
      const bool row_valid = grow < p.G * BK;
      const int hq = x.h * p.G + grow / BK;
      const int tok_in_blk = grow % BK;
      const int tq = qblock<CHUNK>(x) * BK + tok_in_blk;  // query position in the packed Q
      float m_used = -INFINITY, l = 0.f;
      for (int s = 0; s < nsteps; ++s, ++kstep) {
        // Column limits of the two 64-column halves of this step: keys past the
        // query (diagonal block) or past the row's last block are masked.
        int lim[2] = {64, 64};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int jb = (BPS == 2) ? s * 2 + hh : s;       // block holding this half
          const int key0 = (BPS == 2) ? 0 : hh * 64;        // first key of the half in its block
          if (jb >= x.nkv) lim[hh] = 0;
          else if (jb == diag_j) lim[hh] = max(0, min(64, tok_in_blk - key0 + 1));
        }
        if (ok) ok = mbar_wait(bar(C::B_SFULL + t), kstep & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          __syncwarp();
          nbar_sync(kNbP + t, 160);
          if (s == 0 && has_next) nx_diag = diag_of(nx);
          continue;
        }
        tc_fence_after();
        float mx;
        // tcgen05 loads are warp-collective: the path must be the same for every
        // lane (the diagonal's limits differ from lane to lane).
        if (__all_sync(0xffffffffu, lim[0] == 64 && lim[1] == 64)) {  // no mask: reducing loads
          mx = tmem_max128(tS);
        } else {
          float v[64];
          load_masked(tS, lim[0], v);
          mx = max64(v);
          load_masked(tS + 64, lim[1], v);
          mx = fmaxf(mx, max64(v));
        }
        const float m_new = fmaxf(m_used, mx * p.scale_log2);
        if (s > 0) {
          const bool resc = m_new > m_used + kRescaleThreshold;
          if (__any_sync(0xffffffffu, resc)) {
            // O already holds PV(s-1): the commit that signalled S(s) was issued
            // after PV(s-1) and tracks every earlier MMA of the issuing thread.
            const float alpha = resc ? fast_exp2(m_used - m_new) : 1.f;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t ro[32];
              tmem_ld32(tO + c0, ro);
#pragma unroll
              for (int c = 0; c < 32; ++c) ro[c] = __float_as_uint(__uint_as_float(ro[c]) * alpha);
              tmem_st32(tO + c0, ro);
            }
            l *= alpha;
            if (resc) m_used = m_new;
          }
        } else {
          m_used = m_new;
        }
        const float mref = (m_used == -INFINITY) ? 0.f : m_used;
        const uint64_t negm = pack2(-mref, -mref);
        if (__all_sync(0xffffffffu, lim[0] == 64 && lim[1] == 64))
          l += exp_step<false>(tS, scale2, negm, lim);
        else
          l += exp_step<true>(tS, scale2, negm, lim);
        tc_fence_before();
        __syncwarp();
        nbar_sync(kNbP + t, 160);
        // The next unit's diagonal position: its load overlaps the wait for S(1).
        if (s == 0 && has_next) nx_diag = diag_of(nx);
      }
      if (!ok) continue;
      // Hand the row's 1 / l to the epilogue warpgroup (its slot is free once the
      // epilogue has read the previous unit's) and write lse = (m + log2 l) ln 2.
      if (units > 0) ok = mbar_wait(bar(C::B_STATSFREE + t), (units - 1) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        continue;
      }
      stat_inv_l[rho] = 1.f / l;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_STATS + t));
      ++units;
      if (row_valid && tq < x.n && p.lse != nullptr)
        p.lse[(size_t)hq * p.T + x.s0 + tq] = (m_used + fast_log2(l)) * 0.6931471805599453f;
    }
  } else if (warp >= kEpiWarp) {
    // ------------------------------------------------------------ epilogue, both M-tiles
    reg_dealloc<kRegEpi>();
    const int wq = warp % 4;          // TMEM lane quarter
    const int rho = wq * 32 + lane;   // row of the M-tile
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const float *stat_inv_l = reinterpret_cast<const float *>(sm + C::kOffStat);
    const bool elected = wq == 0 && lane == 0;  // issues the tensor stores
    int ut[2] = {0, 0};               // units of each tile (O-final / statistics phases)
    int ostage[2] = {0, 0};           // output staging uses of each tile
    bool store_pending[2] = {false, false};  // elected: a tile's last staged store not yet waited
    bool ok = true;
    Unit nx;
    if (blockIdx.x < total_units) nx = decode_unit<CHUNK>(p, blockIdx.x);
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
      const Unit x = nx;
      if (u + (int)gridDim.x < total_units) nx = decode_unit<CHUNK>(p, u + gridDim.x);  // prefetch
      for (int t = 0; ok && t < x.nt; ++t) {
        // O = u / l once the unit's last PV of tile t is done and its 1 / l is staged
        ok = mbar_wait(bar(C::B_OFINAL + t), ut[t] & 1, abort_flag, p.status);
        if (ok) ok = mbar_wait(bar(C::B_STATS + t), ut[t] & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        ++ut[t];
        tc_fence_after();
        const int grow = (2 * x.pair + t) * 128 + rho;   // row within the group's G*b rows
        const int tq = qblock<CHUNK>(x) * BK + grow % BK;  // query position in the packed Q
        const bool store = grow < p.G * BK && tq < x.n;
        const int hq = x.h * p.G + grow / BK;
        const float inv_l = stat_inv_l[t * 128 + rho];
        const uint32_t tO = tmem + lane_base + C::colO(t);
        // Read the whole O row as bf16 pairs first, release O (to the next unit's PV)
        // and the statistics slot, and only then write the row out.
        uint32_t ob[D / 2];
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ro[32];
          tmem_ld32(tO + c0, ro);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            ob[c0 / 2 + e] = pack_bf16x2(__uint_as_float(ro[2 * e]) * inv_l,
                                         __uint_as_float(ro[2 * e + 1]) * inv_l);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(C::B_OFREE + t));
          mbar_arrive(bar(C::B_STATSFREE + t));
        }
        // A tile whose 128 rows are all valid query rows of a full block goes out
        // through shared memory and tensor stores (one 64-column half at a time, in
        // the 128-byte-swizzled layout of the store box); other tiles (sequence
        // tails, partial groups) store their valid rows directly.
        const bool via_tma =
            (2 * x.pair + t + 1) * 128 <= p.G * BK && (qblock<CHUNK>(x) + 1) * BK <= x.n;
        if (via_tma) {
          const uint32_t stg = sbase + C::kOffStageO + t * C::kStageO;
#pragma unroll
          for (int hh = 0; hh < C::kPanels; ++hh, ++ostage[t]) {
            // the last half of the tile's previous unit is waited for only now, when
            // the buffer is needed again
            if (elected && store_pending[t]) {
              bulk_wait_read();
              mbar_arrive(bar(C::B_OSFREE + t));
              store_pending[t] = false;
            }
            // the previous store out of this buffer has finished reading it
            if (!__all_sync(0xffffffffu, ok = mbar_wait(bar(C::B_OSFREE + t), (ostage[t] & 1) ^ 1,
                                                        abort_flag, p.status))) {
              ok = false;
              break;
            }
#pragma unroll
            for (int c = 0; c < 8; ++c)
              st_shared_v4(stg + rho * 128 + ((c ^ (rho & 7)) << 4), ob[hh * 32 + 4 * c],
                           ob[hh * 32 + 4 * c + 1], ob[hh * 32 + 4 * c + 2], ob[hh * 32 + 4 * c + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_OSTAGED + t));
            if (elected) {
              ok = mbar_wait(bar(C::B_OSTAGED + t), ostage[t] & 1, abort_flag, p.status);
              if (ok) {
                tma_store_3d(&tmO, stg, hh * 64, x.s0 + qblock<CHUNK>(x) * BK,
                             x.h * p.G + ((2 * x.pair + t) * 128) / BK);
                bulk_commit();
                if (hh + 1 < C::kPanels) {
                  bulk_wait_read();
                  mbar_arrive(bar(C::B_OSFREE + t));
                } else {
                  store_pending[t] = true;
                }
              }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);  // the elected thread's outcome, warp-wide
            if (!ok) break;
          }
        } else if (store) {
          uint4 *dst = reinterpret_cast<uint4 *>(p.O + ((size_t)hq * p.T + x.s0 + tq) * D);
#pragma unroll
          for (int q4 = 0; q4 < D / 8; ++q4)
            dst[q4] = make_uint4(ob[4 * q4], ob[4 * q4 + 1], ob[4 * q4 + 2], ob[4 * q4 + 3]);
        }
      }
    }
  } else {
    reg_dealloc<kRegIssue>();  // warp 11: no role
  }

  if (warp == kEpiWarp && lane == 0) bulk_wait_all();  // output stores done
  grid_dep_launch();  // the next launch may be scheduled; it waits for this grid
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// cache == nullptr: K / V packed [H_kv, T, d]; otherwise a chunk over the paged
// cache (block 64 = the page), K / V read from its pages.
template <int D, int BK, bool CHUNK>
cudaError_t launch_tc(const bsa_shape_t &s, const void *Q, const void *K, const void *V,
                      const bsa_kv_cache_t *cache, const int32_t *row_ptr,
                      const int32_t *col_idx, const int32_t *work, const int32_t *bucket_off,
                      float scale, void *O, float *lse, int32_t *dev_status, cudaStream_t st) {
  using C = Cfg<D, BK>;
  CUtensorMap mq, mk, mv;
  CUtensorMap mo;
  bool ok = make_tmap_3d_bf16(&mo, O, D, s.total_tokens, s.num_heads, 64, BK, 128 / BK) &&
            make_tmap_3d_bf16(&mq, Q, D, s.total_tokens, s.num_heads, 64, BK, 128 / BK);
  if constexpr (CHUNK) {
    const uint64_t rows = (uint64_t)cache->num_phys_pages * s.num_kv_heads * 64;
    ok = ok && make_tmap_3d_bf16(&mk, cache->k_cache, D, rows, 1, 64, 64, 1) &&
         make_tmap_3d_bf16(&mv, cache->v_cache, D, rows, 1, 64, 64, 1);
  } else {
    ok = ok && make_tmap_3d_bf16(&mk, K, D, s.total_tokens, s.num_kv_heads, 64, BK, 1) &&
         make_tmap_3d_bf16(&mv, V, D, s.total_tokens, s.num_kv_heads, 64, BK, 1);
  }
  if (!ok) return cudaErrorInvalidValue;
  AttnParams p;
  p.cu = s.cu_seqlens;
  p.row_ptr = row_ptr;
  p.col_idx = col_idx;
  p.work = work;
  p.bucket_off = bucket_off;
  p.O = static_cast<uint16_t *>(O);
  p.lse = lse;
  p.status = dev_status;
  p.qoff = CHUNK ? cache->prefix_lens : nullptr;
  p.bt = CHUNK ? cache->block_table : nullptr;
  p.maxp = CHUNK ? cache->max_pages_per_req : 0;
  p.num_phys = CHUNK ? cache->num_phys_pages : 0;
  p.T = s.total_tokens;
  p.H = s.num_heads;
  p.Hk = s.num_kv_heads;
  p.G = s.num_heads / s.num_kv_heads;
  p.Nq = s.max_blocks;
  p.mtiles = (p.G * BK + 127) / 128;
  p.npairs = (p.mtiles + 1) / 2;
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D, BK, CHUNK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // The softmax warpgroups' setmaxnreg increase waits, without a bound, until the
  // other warpgroups have released enough registers: refuse to launch a build whose
  // per-thread launch count cannot cover the split (checked once per instantiation).
  static const cudaError_t regs_ok = [] {
    cudaFuncAttributes fa;
    const cudaError_t r = cudaFuncGetAttributes(&fa, attn_tc_kernel<D, BK, CHUNK>);
    if (r != cudaSuccess) return r;
    return fa.numRegs * kThreads >= (int)(2 * kRegSoftmax + kRegIssue + kRegEpi) * 128
               ? cudaSuccess
               : cudaErrorInvalidConfiguration;
  }();
  if (regs_ok != cudaSuccess) return regs_ok;
  const long long max_units = (long long)s.num_seqs * s.num_kv_heads * s.max_blocks * p.npairs;
  const int grid = (int)std::min<long long>(num_sms(), std::max<long long>(1, max_units));
  return launch_dependent(attn_tc_kernel<D, BK, CHUNK>, dim3(grid), dim3(kThreads),
                          C::kSmemBytes, st, mq, mk, mv, mo, p);
}

}  // namespace

cudaError_t launch_attention_tc(const bsa_shape_t &s, const void *Q, const void *K,
                                const void *V, const int32_t *row_ptr, const int32_t *col_idx,
                                const int32_t *work, const int32_t *bucket_off, float scale,
                                void *O, float *lse, int32_t *dev_status, cudaStream_t st) {
  if (s.head_dim == 64 && s.block == 64)
    return launch_tc<64, 64, false>(s, Q, K, V, nullptr, row_ptr, col_idx, work, bucket_off,
                                    scale, O, lse, dev_status, st);
  if (s.head_dim == 64 && s.block == 128)
    return launch_tc<64, 128, false>(s, Q, K, V, nullptr, row_ptr, col_idx, work, bucket_off,
                                     scale, O, lse, dev_status, st);
  if (s.head_dim == 128 && s.block == 64)
    return launch_tc<128, 64, false>(s, Q, K, V, nullptr, row_ptr, col_idx, work, bucket_off,
                                     scale, O, lse, dev_status, st);
  return launch_tc<128, 128, false>(s, Q, K, V, nullptr, row_ptr, col_idx, work, bucket_off,
                                    scale, O, lse, dev_status, st);
}

cudaError_t launch_attention_chunk(const bsa_shape_t &s, const bsa_kv_cache_t &cache,
                                   const void *Q, const int32_t *row_ptr, const int32_t *col_idx,
                                   const int32_t *work, const int32_t *bucket_off, float scale,
                                   void *O, float *lse, int32_t *dev_status, cudaStream_t st) {
  if (s.head_dim == 64)
    return launch_tc<64, 64, true>(s, Q, nullptr, nullptr, &cache, row_ptr, col_idx, work,
                                   bucket_off, scale, O, lse, dev_status, st);
  return launch_tc<128, 64, true>(s, Q, nullptr, nullptr, &cache, row_ptr, col_idx, work,
                                  bucket_off, scale, O, lse, dev_status, st);
}

}  // namespace bsa
