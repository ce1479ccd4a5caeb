// Backward of the sparse attention on the tensor cores (BF16, head_dim 128): the
// same gradients as the SIMT path ("2.1 · 粗粒度选择" §2.2: training reuses the
// forward's index and softmax statistics; the forward of §1.2 eqs.(1)-(5)), as
// tcgen05 MMAs on 64-key tiles with fp32 accumulators in TMEM:
//   S = Q K^T,  dP = dO V^T                     (M = 128 query rows, N = 64 keys)
//   P = exp(S * scale - lse),  dS = P (dP - D),  D = rowsum(dO * O)
//   dQ  = scale * dS K       (query-major pass, M = 128 query rows, N = d)
//   dV^T = dO^T P,  dK^T = scale * Q^T dS   (key-major pass, M = d = 128, N = 64 keys)
// Two passes so that every output element has one writer and no atomics touch the
// gradients: the dQ pass walks the forward's worklist (row -> its key blocks); the
// dK / dV pass walks the transposed index (key block -> the rows that selected
// it, ascending), built here from a row bitmap per key block, its population
// counts and a scan.  Both passes recompute S and dP.  Masks are the forward's:
// the causal triangle inside the diagonal block and query rows past the sequence
// end or past the KV-head group.
//
// Operands sit in shared memory in the 128-byte-swizzled layout TMA writes: a
// tile of R rows x 64 bf16 columns is R rows of 128 bytes, 16-byte chunk c of row
// p at p * 128 + ((c ^ (p & 7)) << 4).  Q / dO / K / V tiles come by TMA; P and dS
// are written by the softmax warps in the same layout, which serves both as a
// K-major operand (dS of dQ = dS K) and as an MN-major one (P, dS of the
// key-major products, and K / Q / dO read transposed).
//
// Both passes run 320 threads: two softmax warpgroups that take alternate tiles
// (each warp reads the TMEM lanes of its quarter), a TMA warp and an MMA warp.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace bsa {
namespace {

constexpr int kD = 128;

constexpr float kLog2e = 1.4426950408889634f;

// kind::f16 instruction descriptors: S / dP (A, B K-major, N = 64 keys); dQ
// (A = dS K-major, B = K MN-major, N = d); dV^T / dK^T (A, B both MN-major).
constexpr uint32_t kIdescS = idesc_bf16(128, 64, false);
constexpr uint32_t kIdescS128 = idesc_bf16(128, 128, false);
constexpr uint32_t kIdescDQ = idesc_bf16(128, kD, true);
constexpr uint32_t kIdescKV = idesc_bf16(128, 64, true) | (1u << 15);

struct BwdTcParams {
  const int32_t *cu;
  const int32_t *row_ptr;
  const int32_t *col_idx;
  const int32_t *work;
  const int32_t *bucket_off;
  const int32_t *kt_ptr;     // key-major index: rows of key block kb at kt_rows[kt_ptr[kb] ..)
  const int32_t *kt_rows;
  const int32_t *kt_work;    // key blocks with rows, longest list first
  const int32_t *kt_bucket;  // kt_bucket[7] = number of such key blocks
  const float *lse;
  const float *Dv;
  uint16_t *dQ;
  uint16_t *dK;
  uint16_t *dV;
  int32_t *status;
  int T, Hk, G, Nq, mtiles;
  float scale, scale_log2;
};

// Row rho of an M-tile of 128 query rows of work row (r, h): rows are the group's
// G heads x b tokens in that order (the TMA box of Q loads 128 / b heads of b
// tokens), so tile t, row rho is head h*G + (t*128 + rho) / b, token (..) % b.
struct QRow {
  bool valid;    // a query of the sequence inside the group
  int tok;       // token within the query block
  size_t idx;    // (head, token) index into [H, T]
};

template <int BK>
BSA_DEV QRow qrow(const BwdTcParams &p, int t, int rho, int h, int r, int s0, int n) {
  QRow q;
  const int grow = t * 128 + rho;
  q.tok = grow % BK;
  q.valid = grow < p.G * BK && r * BK + q.tok < n;
  q.idx = (size_t)(h * p.G + grow / BK) * p.T + s0 + r * BK + q.tok;
  return q;
}

// 16 TMEM columns of this thread's lane, not waited (see tmem_ld32_async).
BSA_DEV void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Wait for this thread's TMEM loads into the two 16-register buffers.
BSA_DEV void tmem_wait_ld16x2(uint32_t (&r)[16], uint32_t (&q)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(q[0]), "+r"(q[1]),
                 "+r"(q[2]), "+r"(q[3]), "+r"(q[4]), "+r"(q[5]), "+r"(q[6]), "+r"(q[7]),
                 "+r"(q[8]), "+r"(q[9]), "+r"(q[10]), "+r"(q[11]), "+r"(q[12]), "+r"(q[13]),
                 "+r"(q[14]), "+r"(q[15])
               :
               : "memory");
}

// Packed pairs of fp32 (low word = first element) and the sm_100+ pair arithmetic.
BSA_DEV uint64_t f2_pack(float lo, float hi) {
  return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
BSA_DEV uint64_t f2_pack(uint32_t lo, uint32_t hi) { return (uint64_t)lo | ((uint64_t)hi << 32); }
BSA_DEV float f2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
BSA_DEV float f2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
BSA_DEV uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
BSA_DEV uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
BSA_DEV uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// P and dS of the 64 keys of one TMEM S / dP tile row into shared memory (P only
// when smP != 0), 16 columns at a time: the next 16 columns' loads are in flight
// while the current ones are computed, and only 64 registers hold loaded values
// (holding all 128 at once left the compiler no room to overlap the exp / multiply
// chains of different columns, which made this routine four times slower).
// Keys past the query on the diagonal (key0 + column > tok), and invalid rows,
// get P = dS = 0.
// WAIT: the dS buffer may still be read by the previous dQ product; wait for its
// release (bounded) before the first store, after the first 16 columns are computed.
template <bool WAIT = false>
BSA_DEV void tile_grad64(uint32_t tS, uint32_t tDP, uint32_t smP, uint32_t smDS, int rho,
                         bool valid, bool diag, int key0, int tok, float scale_log2, float lse2,
                         float Drow, uint32_t wbar = 0u, uint32_t wparity = 0u,
                         volatile int32_t *abort_flag = nullptr, int32_t *status = nullptr,
                         bool *ok = nullptr) {
  uint32_t sb[2][16], db[2][16];
  const int lim = !valid ? 0 : (diag ? min(64, max(0, tok - key0 + 1)) : 64);  // first masked column
  const uint64_t sc2 = f2_pack(scale_log2, scale_log2), nl2 = f2_pack(-lse2, -lse2);
  const uint64_t nd2 = f2_pack(-Drow, -Drow);
  tmem_ld16_async(tS, sb[0]);
  tmem_ld16_async(tDP, db[0]);
  tmem_wait_ld16x2(sb[0], db[0]);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (c < 3) {
      tmem_ld16_async(tS + 16 * (c + 1), sb[(c + 1) & 1]);
      tmem_ld16_async(tDP + 16 * (c + 1), db[(c + 1) & 1]);
    }
    const uint32_t(&sv)[16] = sb[c & 1];
    const uint32_t(&dv)[16] = db[c & 1];
    uint32_t pk[8], dk[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int col = 16 * c + 2 * e;
      const uint64_t z = f2_fma(f2_pack(sv[2 * e], sv[2 * e + 1]), sc2, nl2);
      const float p0 = col < lim ? fast_exp2(f2_lo(z)) : 0.f;
      const float p1 = col + 1 < lim ? fast_exp2(f2_hi(z)) : 0.f;
      const uint64_t ds = f2_mul(f2_pack(p0, p1), f2_add(f2_pack(dv[2 * e], dv[2 * e + 1]), nd2));
      pk[e] = pack_bf16x2(p0, p1);
      dk[e] = pack_bf16x2(f2_lo(ds), f2_hi(ds));
    }
    if (WAIT && c == 0) {
      *ok = __all_sync(0xffffffffu, mbar_wait(wbar, wparity, abort_flag, status));
      if (!*ok) {  // leave no TMEM load in flight
        tmem_wait_ld16x2(sb[1], db[1]);
        return;
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // 16-byte chunk 2c + h of the 128-byte row
      const uint32_t off = rho * 128 + (((2 * c + h) ^ (rho & 7)) << 4);
      if (smP != 0u) st_shared_v4(smP + off, pk[4 * h], pk[4 * h + 1], pk[4 * h + 2], pk[4 * h + 3]);
      st_shared_v4(smDS + off, dk[4 * h], dk[4 * h + 1], dk[4 * h + 2], dk[4 * h + 3]);
    }
    if (c < 3) tmem_wait_ld16x2(sb[(c + 1) & 1], db[(c + 1) & 1]);
  }
}

// S = X Y^T for one 128-row X tile (two 16 KB panels) and one 64-row Y tile
// (two 8 KB panels), K = d.
// Descriptors differ in their low word only, and the K-step offsets are constants.
BSA_DEV void mma_xyT(uint32_t d_tmem, uint32_t x, uint32_t y) {
  const uint32_t xl = desc_lo(x, 16), yl = desc_lo(y, 16);
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk)
    mma_ss_lo(d_tmem, xl + ((kk / 4) * 16384 + (kk % 4) * 32) / 16,
              yl + ((kk / 4) * 8192 + (kk % 4) * 32) / 16, kDescHi, kIdescS, kk > 0 ? 1u : 0u);
}

// D += A B with A (bf16 pairs, row = lane) read from tensor memory.
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

// 8 TMEM columns of this thread's lane, not waited.
BSA_DEV void tmem_st8_nowait(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                   taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
               "r"(r[7])
               : "memory");
}

// dS of the 64 keys of one TMEM S / dP tile row written back to tensor memory as
// bf16 pairs (32 columns at tDS, key 2 c and 2 c + 1 in column c: the layout of a
// tensor-memory A operand), 16 columns at a time as tile_grad64 does.  Once the
// last S / dP columns are loaded the warp takes named barrier `sread` (over
// `sread_threads` threads: the S / dP buffer may then be overwritten); the stores
// are waited before returning.
BSA_DEV void tile_grad64_tmem(uint32_t tS, uint32_t tDP, uint32_t tDS, bool valid, bool diag,
                              int key0, int tok, float scale_log2, float lse2, float Drow,
                              uint32_t sread, uint32_t sread_threads) {
  uint32_t sb[2][16], db[2][16];
  const int lim = !valid ? 0 : (diag ? min(64, max(0, tok - key0 + 1)) : 64);  // first masked column
  const uint64_t sc2 = f2_pack(scale_log2, scale_log2), nl2 = f2_pack(-lse2, -lse2);
  const uint64_t nd2 = f2_pack(-Drow, -Drow);
  tmem_ld16_async(tS, sb[0]);
  tmem_ld16_async(tDP, db[0]);
  tmem_wait_ld16x2(sb[0], db[0]);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (c < 3) {
      tmem_ld16_async(tS + 16 * (c + 1), sb[(c + 1) & 1]);
      tmem_ld16_async(tDP + 16 * (c + 1), db[(c + 1) & 1]);
    }
    const uint32_t(&sv)[16] = sb[c & 1];
    const uint32_t(&dv)[16] = db[c & 1];
    uint32_t dk[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int col = 16 * c + 2 * e;
      const uint64_t z = f2_fma(f2_pack(sv[2 * e], sv[2 * e + 1]), sc2, nl2);
      const float p0 = col < lim ? fast_exp2(f2_lo(z)) : 0.f;
      const float p1 = col + 1 < lim ? fast_exp2(f2_hi(z)) : 0.f;
      const uint64_t ds = f2_mul(f2_pack(p0, p1), f2_add(f2_pack(dv[2 * e], dv[2 * e + 1]), nd2));
      dk[e] = pack_bf16x2(f2_lo(ds), f2_hi(ds));
    }
    tmem_st8_nowait(tDS + 8 * c, dk);
    if (c < 3) tmem_wait_ld16x2(sb[(c + 1) & 1], db[(c + 1) & 1]);
    if (c == 2) {  // every S / dP column of this warp is in registers
      tc_fence_before();
      __syncwarp();
      nbar_sync(sread, sread_threads);
    }
  }
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// S = X Y^T for one 128-row X tile and one 128-row Y tile (two 16 KB panels each),
// K = d, N = 128.
BSA_DEV void mma_xyT128(uint32_t d_tmem, uint32_t x, uint32_t y) {
  const uint32_t xl = desc_lo(x, 16), yl = desc_lo(y, 16);
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk)
    mma_ss_lo(d_tmem, xl + ((kk / 4) * 16384 + (kk % 4) * 32) / 16,
              yl + ((kk / 4) * 16384 + (kk % 4) * 32) / 16, kDescHi, kIdescS128, kk > 0 ? 1u : 0u);
}

// ---------------------------------------------------------------- key-major index

// Mark, per key block, the rows that selected it: bit r of the key block's
// ceil(N_q / 32) words.
__global__ void kt_mark_kernel(const int32_t *__restrict__ row_ptr,
                               const int32_t *__restrict__ col_idx, int nrows, int Nq, int W,
                               uint32_t *__restrict__ bits, int32_t *__restrict__ status) {
  for (int row = blockIdx.x * blockDim.x + threadIdx.x; row < nrows;
       row += gridDim.x * blockDim.x) {
    const int r = row % Nq, base = row - r;
    for (int e = row_ptr[row]; e < row_ptr[row + 1]; ++e) {
      const int j = col_idx[e];
      if (j >= 0 && j <= r)
        atomicOr(bits + (size_t)(base + j) * W + r / 32, 1u << (r % 32));
      else if (BSA_BOUNDS_CHECK)
        set_status(status, BSA_ERR_INDEX_RANGE);  // skipped in every build
    }
  }
}

// Rows per key block: the population count of its bitmap (a row named twice in a
// malformed worklist still counts once, matching what the emit writes).
__global__ void kt_count_kernel(const uint32_t *__restrict__ bits, int nrows, int W,
                                int32_t *__restrict__ cnt) {
  for (int kb = blockIdx.x * blockDim.x + threadIdx.x; kb < nrows;
       kb += gridDim.x * blockDim.x) {
    int c = 0;
    for (int w = 0; w < W; ++w) c += __popc(bits[(size_t)kb * W + w]);
    cnt[kb] = c;
  }
}

// One warp per key block: its rows in ascending order at kt_rows[kt_ptr[kb] ..), so
// the dK / dV sums run in the same order on every call.
__global__ void kt_emit_kernel(const uint32_t *__restrict__ bits,
                               const int32_t *__restrict__ kt_ptr, int32_t *__restrict__ kt_rows,
                               int nrows, int W) {
  const int lane = threadIdx.x % 32;
  for (int kb = (blockIdx.x * blockDim.x + threadIdx.x) / 32; kb < nrows;
       kb += gridDim.x * blockDim.x / 32) {
    int pos = kt_ptr[kb];
    for (int w0 = 0; w0 < W; w0 += 32) {
      const int w = w0 + lane;
      uint32_t m = w < W ? bits[(size_t)kb * W + w] : 0u;
      const int c = __popc(m);
      int incl = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      int out = pos + incl - c;
      while (m != 0u) {
        const int b = __ffs(m) - 1;
        kt_rows[out++] = w * 32 + b;
        m &= m - 1u;
      }
      pos += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
}

// ---------------------------------------------------------------- dQ pass

// One CTA per (work row, M-tile), one per SM: Q and dO of the tile stay in shared
// memory; the row's keys stream in steps of 128 (one 128-key block, or two 64-key
// blocks side by side; an odd last block is loaded twice and its copy masked)
// through a three-stage K ring and a two-stage V ring, so every S / dP product has
// N = 128 (the N = 64 form runs at 58 % of the N = 128 rate per FLOP).  TMEM holds
// S and dP of one step (256 columns, single-buffered), the dQ accumulator (128) and
// two dS buffers (64 each): the softmax warps write dS back to tensor memory as
// bf16 pairs and dQ += dS K reads it as the A operand, so no shared-memory dS
// buffer has to be released before the next step's dS is written.  The MMA thread
// issues S / dP(s) as soon as the softmax warps have loaded S / dP(s - 1) (before
// they finish dS(s - 1)), then dQ += dS(s - 1) K(s - 1).  Warpgroup g (warps 4 g ..
// 4 g + 3, one query row per thread) takes the 64 keys 64 g .. 64 g + 63 of every
// step.  320 threads: warps 0-7 softmax, warp 8 TMA, warp 9 MMA.
namespace dq {
constexpr int kThreads = 352;
constexpr int NK = 3, NV = 2;  // K and V ring stages (32 KB each: 128 keys x d)
constexpr int kOffQ = 0, kOffDO = 32768, kOffK = 65536, kOffV = kOffK + NK * 32768;
constexpr int kOffBar = kOffV + NV * 32768;
constexpr int B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_KEMPTY = B_KFULL + NK;
constexpr int B_VFULL = B_KEMPTY + NK;
constexpr int B_VEMPTY = B_VFULL + NV, B_SFULL = B_VEMPTY + NV;
// DSFREE per dS buffer: dQ(s) has read it
constexpr int B_DSFREE = B_SFULL + 1, B_DQFULL = B_DSFREE + 2;
// named barriers, each taken once per step by all of its warps: K / V of the step
// landed (watcher + MMA warp), S / dP loaded by the softmax and dS written (8 softmax
// warps + MMA warp)
constexpr uint32_t kNbKV = 1, kNbSR = 2, kNbDS = 3, kKVThreads = 64, kSoftThreads = 288;
constexpr int kOffCtl = kOffBar + (B_DQFULL + 1) * 8;
constexpr int kSmemBytes = kOffCtl + 16 + 1024;
constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 384, kTmemCols = 512;
static_assert(kSmemBytes <= 232448, "shared memory budget");
}  // namespace dq

// Persistent: one CTA per SM walks the work items (router row, 128-row M-tile) of the
// worklist's longest-first order with a stride of the grid.  Ring stages, barrier phases
// and dS buffers follow step and item counters that run on across items, so the next
// item's Q / dO load starts once the current item's last S / dP products have read
// theirs, and its first steps overlap the current item's last dQ products and dQ store.
template <int BK>
__global__ void __launch_bounds__(dq::kThreads, 1) bwd_dq_tc_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
    const BwdTcParams p) {
  using namespace dq;
  constexpr int BPS = 128 / BK;  // key blocks per 128-key step
  const int total = __ldg(p.bucket_off + BSA_NUM_BUCKETS) * p.mtiles;  // work items
  if ((int)blockIdx.x >= total) return;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *sm = smem_raw + (sbase - raw);
  auto bar = [&](int k) { return sbase + kOffBar + 8u * (uint32_t)k; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffCtl);
  volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(sm + kOffCtl + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    for (int st = 0; st < NK; ++st) {
      mbar_init(bar(B_KFULL + st), 1);
      mbar_init(bar(B_KEMPTY + st), 1);
    }
    for (int st = 0; st < NV; ++st) {
      mbar_init(bar(B_VFULL + st), 1);
      mbar_init(bar(B_VEMPTY + st), 1);
    }
    mbar_init(bar(B_SFULL), 1);
    for (int b = 0; b < 2; ++b) mbar_init(bar(B_DSFREE + b), 1);
    mbar_init(bar(B_DQFULL), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t smQ = sbase + kOffQ, smDO = sbase + kOffDO, smK = sbase + kOffK,
                 smV = sbase + kOffV;

  struct Item {
    int t, r, h, s0, n, kv0, nkv, nsteps;
  };
  auto item_of = [&](int u) {
    Item w;
    w.t = u % p.mtiles;
    const int row = __ldg(p.work + u / p.mtiles);
    w.r = row % p.Nq;
    w.h = (row / p.Nq) % p.Hk;
    const int i = row / (p.Nq * p.Hk);
    w.s0 = __ldg(p.cu + i);
    w.n = __ldg(p.cu + i + 1) - w.s0;
    w.kv0 = __ldg(p.row_ptr + row);
    w.nkv = __ldg(p.row_ptr + row + 1) - w.kv0;
    w.nsteps = (w.nkv + BPS - 1) / BPS;
    return w;
  };
  // every role walks the same items; the next item is decoded one ahead
  const int stride = (int)gridDim.x;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool ok = true;
      int issued_k[NK], issued_v[NV], issued_q = -1;
      for (int st = 0; st < NK; ++st) issued_k[st] = -1;
      for (int st = 0; st < NV; ++st) issued_v[st] = -1;
      int gs = 0, it = 0;
      Item nx = item_of(blockIdx.x);
      for (int u = blockIdx.x; ok && u < total; u += stride, ++it) {
        const Item w = nx;
        if (u + stride < total) nx = item_of(u + stride);
        const int hq0 = w.h * p.G + (w.t * 128) / BK;
        // the previous item's last S / dP products have read its Q / dO
        if (it >= 1 && !(ok = mbar_wait(bar(B_QEMPTY), (it - 1) & 1, abort_flag, p.status)))
          break;
        mbar_arrive_expect_tx(bar(B_QFULL), 4 * 16384);
        issued_q = it & 1;
        for (int pn = 0; pn < 2; ++pn) {
          tma_load_3d(smQ + pn * 16384, &tmQ, bar(B_QFULL), pn * 64, w.s0 + w.r * BK, hq0);
          tma_load_3d(smDO + pn * 16384, &tmDO, bar(B_QFULL), pn * 64, w.s0 + w.r * BK, hq0);
        }
        // token row of 64-key half hf of step s (a missing second block repeats the first)
        auto key_row = [&](int s, int hf) {
          if (BPS == 1)
            return w.s0 + checked_index(__ldg(p.col_idx + w.kv0 + s), 0, w.r, p.status) * BK +
                   hf * 64;
          const int e = min(2 * s + hf, w.nkv - 1);
          return w.s0 + checked_index(__ldg(p.col_idx + w.kv0 + e), 0, w.r, p.status) * BK;
        };
        for (int s = 0; s < w.nsteps; ++s, ++gs) {
          const int sk = gs % NK, sv = gs % NV;
          const int y0 = key_row(s, 0), y1 = key_row(s, 1);
          if (gs >= NK &&
              !(ok = mbar_wait(bar(B_KEMPTY + sk), ((gs - NK) / NK) & 1, abort_flag, p.status)))
            break;
          mbar_arrive_expect_tx(bar(B_KFULL + sk), 4 * 8192);
          issued_k[sk] = (gs / NK) & 1;
          for (int pn = 0; pn < 2; ++pn) {  // panel pn: d columns 64 pn .. 64 pn + 63, 128 rows
            tma_load_3d(smK + sk * 32768 + pn * 16384, &tmK, bar(B_KFULL + sk), pn * 64, y0, w.h);
            tma_load_3d(smK + sk * 32768 + pn * 16384 + 8192, &tmK, bar(B_KFULL + sk), pn * 64,
                        y1, w.h);
          }
          if (gs >= NV &&
              !(ok = mbar_wait(bar(B_VEMPTY + sv), ((gs - NV) / NV) & 1, abort_flag, p.status)))
            break;
          mbar_arrive_expect_tx(bar(B_VFULL + sv), 4 * 8192);
          issued_v[sv] = (gs / NV) & 1;
          for (int pn = 0; pn < 2; ++pn) {
            tma_load_3d(smV + sv * 32768 + pn * 16384, &tmV, bar(B_VFULL + sv), pn * 64, y0, w.h);
            tma_load_3d(smV + sv * 32768 + pn * 16384 + 8192, &tmV, bar(B_VFULL + sv), pn * 64,
                        y1, w.h);
          }
        }
      }
      // every copy issued lands before the CTA leaves
      if (issued_q >= 0) mbar_wait_drain(bar(B_QFULL), issued_q);
      for (int st = 0; st < NK; ++st)
        if (issued_k[st] >= 0) mbar_wait_drain(bar(B_KFULL + st), issued_k[st]);
      for (int st = 0; st < NV; ++st)
        if (issued_v[st] >= 0) mbar_wait_drain(bar(B_VFULL + st), issued_v[st]);
      (void)ok;
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // Lane 0 issues; the whole warp takes the named barriers, once per step each, so
    // none of them can be left waiting.
    {
      // dQ += dS(g) K(g): 128 keys in steps of 16, dS from TMEM; `first` starts the
      // item's accumulator
      auto dq_product = [&](int g, bool first) {
        const int b = g & 1;
        const uint32_t bl = desc_lo(smK + (g % NK) * 32768, 16384);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_lo(tmem + kColDQ, tmem + kColDS + 64 * b + 8 * kk, bl + kk * 128, kDescHi,
                    kIdescDQ, (!first || kk > 0) ? 1u : 0u);
        mma_commit(bar(B_KEMPTY + g % NK));
        mma_commit(bar(B_DSFREE + b));
      };
      int gs = 0, it = 0;
      Item nx = item_of(blockIdx.x);
      for (int u = blockIdx.x; u < total; u += stride, ++it) {
        const Item w = nx;
        if (u + stride < total) nx = item_of(u + stride);
        for (int s = 0; s < w.nsteps; ++s) {
          const int g = gs + s;
          // S / dP(g - 1) loaded by the softmax: the single S / dP buffer is free (the
          // previous item's last step was waited for below; this one is taken first:
          // the softmax waits on it in the middle of its step)
          if (s >= 1) nbar_sync(kNbSR, kSoftThreads);
          nbar_sync(kNbKV, kKVThreads);  // K / V(g) landed (and the item's Q / dO at s = 0)
          if (lane == 0) {
            tc_fence_after();
            mma_xyT128(tmem + kColS, smQ, smK + (g % NK) * 32768);
            mma_xyT128(tmem + kColDP, smDO, smV + (g % NV) * 32768);
            mma_commit(bar(B_SFULL));
            mma_commit(bar(B_VEMPTY + g % NV));  // V(g) has no other reader
            if (s + 1 == w.nsteps) mma_commit(bar(B_QEMPTY));  // the item's Q / dO are read
          }
          __syncwarp();
          if (s >= 1) {
            // dS(g - 1) written; at s = 1 the softmax warps have also finished reading
            // the previous item's dQ, which this item's first product overwrites
            nbar_sync(kNbDS, kSoftThreads);
            if (lane == 0) {
              tc_fence_after();
              dq_product(g - 1, s == 1);
            }
            __syncwarp();
          }
        }
        nbar_sync(kNbSR, kSoftThreads);
        nbar_sync(kNbDS, kSoftThreads);
        if (lane == 0) {
          tc_fence_after();
          dq_product(gs + w.nsteps - 1, w.nsteps == 1);
          mma_commit(bar(B_DQFULL));
        }
        __syncwarp();
        gs += w.nsteps;
      }
      if (lane == 0 && it > 0) mbar_wait_drain(bar(B_DQFULL), (it - 1) & 1);  // before TMEM is freed
      __syncwarp();
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ copy watcher
    bool ok = true;
    int gs = 0, it = 0;
    Item nx = item_of(blockIdx.x);
    for (int u = blockIdx.x; u < total; u += stride, ++it) {
      const Item w = nx;
      if (u + stride < total) nx = item_of(u + stride);
      for (int s = 0; s < w.nsteps; ++s, ++gs) {
        if (ok && s == 0) ok = mbar_wait_poll(bar(B_QFULL), it & 1, abort_flag, p.status);
        if (ok) ok = mbar_wait_poll(bar(B_KFULL + gs % NK), (gs / NK) & 1, abort_flag, p.status);
        if (ok) ok = mbar_wait_poll(bar(B_VFULL + gs % NV), (gs / NV) & 1, abort_flag, p.status);
        ok = __all_sync(0xffffffffu, ok);
        nbar_sync(kNbKV, kKVThreads);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int g = warp / 4, wq = warp % 4;  // warpgroup g: keys 64 g .. 64 g + 63 of a step
    const int rho = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    bool ok = true;
    int gs = 0, it = 0;
    Item nx = item_of(blockIdx.x);
    for (int u = blockIdx.x; u < total; u += stride, ++it) {
      const Item w = nx;
      if (u + stride < total) nx = item_of(u + stride);
      const QRow q = qrow<BK>(p, w.t, rho, w.h, w.r, w.s0, w.n);
      const float lse2 = q.valid ? __ldg(p.lse + q.idx) * kLog2e : 0.f;
      const float Drow = q.valid ? __ldg(p.Dv + q.idx) : 0.f;
      for (int s = 0; s < w.nsteps; ++s) {
        const int gg = gs + s, b = gg & 1;
        // this warpgroup's 64 keys: half g of the step's 128-key block, or its 64-key
        // block (absent past the row's last block)
        const int e = BPS == 1 ? s : 2 * s + g;
        const bool present = e < w.nkv;
        const int j = present ? __ldg(p.col_idx + w.kv0 + e) : -1;
        const int key0 = BPS == 1 ? 64 * g : 0;
        if (ok) ok = mbar_wait(bar(B_SFULL), gg & 1, abort_flag, p.status);
        // dS buffer b was read by dQ(gg - 2) (issued one step ago)
        if (ok && gg >= 2)
          ok = mbar_wait(bar(B_DSFREE + b), ((gg - 2) >> 1) & 1, abort_flag, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          tc_fence_after();
          tile_grad64_tmem(tmem + lane_base + kColS + 64 * g, tmem + lane_base + kColDP + 64 * g,
                           tmem + lane_base + kColDS + 64 * b + 32 * g, q.valid && present,
                           j == w.r, key0, q.tok, p.scale_log2, lse2, Drow, kNbSR,
                           kSoftThreads);
        } else {
          nbar_sync(kNbSR, kSoftThreads);
        }
        tc_fence_before();
        nbar_sync(kNbDS, kSoftThreads);
      }
      gs += w.nsteps;
      // epilogue: warpgroup g writes columns 64 g .. 64 g + 63 of its rows' dQ
      if (ok) ok = mbar_wait(bar(B_DQFULL), it & 1, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        uint4 *dst = reinterpret_cast<uint4 *>(p.dQ + q.idx * kD + 64 * g);
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_base + kColDQ + 64 * g + c0, rr);
          uint32_t o[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            o[e] = pack_bf16x2(__uint_as_float(rr[2 * e]) * p.scale,
                               __uint_as_float(rr[2 * e + 1]) * p.scale);
          if (q.valid)
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[c0 / 8 + v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- dK / dV pass

// One CTA per (key block, 64-key tile), one per SM: K and V of the tile stay in
// shared memory; the query tiles of every row that selected the block stream
// through a two-stage ring (Q and dO).  S and dP of tile n land in one of two TMEM
// buffers while the softmax warps turn tile n-1 into P and dS (two shared-memory
// buffers each), which then feed dV^T += dO^T P and dK^T += Q^T dS.  320 threads:
// two softmax warpgroups on alternate tiles (warpgroup 0 writes dV, 1 dK at the
// end), warp 8 TMA, warp 9 MMA.
namespace kv {
constexpr int kThreads = 320;
constexpr int kOffK = 0, kOffV = 16384, kOffQ = 32768, kOffDO = kOffQ + 2 * 32768;
constexpr int kOffP = kOffDO + 2 * 32768, kOffDS = kOffP + 2 * 16384;
constexpr int kOffBar = kOffDS + 2 * 16384;
constexpr int B_KVFULL = 0, B_QFULL = 1, B_QEMPTY = 3, B_SFULL = 5, B_SFREE = 7;
constexpr int B_PDSFULL = 9, B_PDSFREE = 11, B_DONE = 13, B_DOFULL = 14, B_DOEMPTY = 16;
constexpr int kOffCtl = kOffBar + 18 * 8;
constexpr int kSmemBytes = kOffCtl + 16 + 1024;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 320, kTmemCols = 512;
static_assert(kSmemBytes <= 232448, "shared memory budget");
}  // namespace kv

template <int BK>
__global__ void __launch_bounds__(kv::kThreads, 1) bwd_dkdv_tc_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
    const BwdTcParams p) {
  using namespace kv;
  constexpr int KT = BK / 64;
  const int u = blockIdx.x;
  if (u >= __ldg(p.kt_bucket + BSA_NUM_BUCKETS) * KT) return;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *sm = smem_raw + (sbase - raw);
  auto bar = [&](int k) { return sbase + kOffBar + 8u * (uint32_t)k; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffCtl);
  volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(sm + kOffCtl + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(bar(B_KVFULL), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_QFULL + b), 1);
      mbar_init(bar(B_QEMPTY + b), 1);
      mbar_init(bar(B_DOFULL + b), 1);
      mbar_init(bar(B_DOEMPTY + b), 1);
      mbar_init(bar(B_SFULL + b), 1);
      mbar_init(bar(B_SFREE + b), 4);
      mbar_init(bar(B_PDSFULL + b), 4);
      mbar_init(bar(B_PDSFREE + b), 1);
    }
    mbar_init(bar(B_DONE), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int e = u % KT;
  const int kb = __ldg(p.kt_work + u / KT);  // (i * H_kv + h) * N_q + j
  const int j = kb % p.Nq, h = (kb / p.Nq) % p.Hk, i = kb / (p.Nq * p.Hk);
  const int s0 = __ldg(p.cu + i), n = __ldg(p.cu + i + 1) - s0;
  const int l0 = __ldg(p.kt_ptr + kb), ntiles = (__ldg(p.kt_ptr + kb + 1) - l0) * p.mtiles;
  const int key_row = s0 + j * BK + e * 64;  // first key of the tile in the packed K / V
  const uint32_t smK = sbase + kOffK, smV = sbase + kOffV, smQ = sbase + kOffQ,
                 smDO = sbase + kOffDO, smP = sbase + kOffP, smDS = sbase + kOffDS;
  auto row_of = [&](int nt) { return __ldg(p.kt_rows + l0 + nt / p.mtiles); };

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool ok = true;
      int issued_q[2] = {-1, -1}, issued_do[2] = {-1, -1};
      mbar_arrive_expect_tx(bar(B_KVFULL), 4 * 8192);
      for (int pn = 0; pn < 2; ++pn) {
        tma_load_3d(smK + pn * 8192, &tmK, bar(B_KVFULL), pn * 64, key_row, h);
        tma_load_3d(smV + pn * 8192, &tmV, bar(B_KVFULL), pn * 64, key_row, h);
      }
      auto tile_coord = [&](int nt, int &y, int &hq) {
        y = s0 + row_of(nt) * BK;
        hq = h * p.G + ((nt % p.mtiles) * 128) / BK;
      };
      // Q / dO of the tiles two and three ahead go to L2 now, so that the ring's
      // copies (issued only when a stage frees) find them there
      auto prefetch = [&](int nt) {
        if (nt >= ntiles) return;
        int y, hq;
        tile_coord(nt, y, hq);
        for (int pn = 0; pn < 2; ++pn) {
          tma_prefetch_l2_3d(&tmQ, pn * 64, y, hq);
          tma_prefetch_l2_3d(&tmDO, pn * 64, y, hq);
        }
      };
      prefetch(0);
      prefetch(1);
      for (int nt = 0; nt < ntiles; ++nt) {
        const int st = nt & 1;
        int y, hq;
        tile_coord(nt, y, hq);
        prefetch(nt + 2);
        if (nt >= 2 && !(ok = mbar_wait(bar(B_QEMPTY + st), ((nt - 2) >> 1) & 1, abort_flag,
                                        p.status)))
          break;
        mbar_arrive_expect_tx(bar(B_QFULL + st), 2 * 16384);
        issued_q[st] = (nt >> 1) & 1;
        for (int pn = 0; pn < 2; ++pn)
          tma_load_3d(smQ + st * 32768 + pn * 16384, &tmQ, bar(B_QFULL + st), pn * 64, y, hq);
        if (nt >= 2 && !(ok = mbar_wait(bar(B_DOEMPTY + st), ((nt - 2) >> 1) & 1, abort_flag,
                                        p.status)))
          break;
        mbar_arrive_expect_tx(bar(B_DOFULL + st), 2 * 16384);
        issued_do[st] = (nt >> 1) & 1;
        for (int pn = 0; pn < 2; ++pn)
          tma_load_3d(smDO + st * 32768 + pn * 16384, &tmDO, bar(B_DOFULL + st), pn * 64, y, hq);
      }
      // every copy issued lands before the CTA leaves (on the normal path the MMA
      // warp has consumed them all; after an abort this waits out the flights)
      mbar_wait_drain(bar(B_KVFULL), 0);
      for (int st = 0; st < 2; ++st) {
        if (issued_q[st] >= 0) mbar_wait_drain(bar(B_QFULL + st), issued_q[st]);
        if (issued_do[st] >= 0) mbar_wait_drain(bar(B_DOFULL + st), issued_do[st]);
      }
      (void)ok;
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(bar(B_KVFULL), 0, abort_flag, p.status);
      // dK^T += Q^T dS, then dV^T += dO^T P of tile nt: Q's stage is released
      // first, so its next copy starts while the dV products run
      auto kv_products = [&](int nt) {
        const int b = nt & 1;
        const uint32_t dol = desc_lo(smDO + b * 32768, 16384), pl = desc_lo(smP + b * 16384, 16384);
        const uint32_t ql = desc_lo(smQ + b * 32768, 16384), dsl = desc_lo(smDS + b * 16384, 16384);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // 128 query rows in steps of 16 (2048 bytes)
          mma_ss_lo(tmem + kColDK, ql + kk * 128, dsl + kk * 128, kDescHi, kIdescKV,
                    (nt > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(B_QEMPTY + b));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss_lo(tmem + kColDV, dol + kk * 128, pl + kk * 128, kDescHi, kIdescKV,
                    (nt > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(B_DOEMPTY + b));
        mma_commit(bar(B_PDSFREE + b));
      };
      for (int nt = 0; ok && nt < ntiles; ++nt) {
        const int b = nt & 1;
        if (!(ok = mbar_wait(bar(B_QFULL + b), (nt >> 1) & 1, abort_flag, p.status))) break;
        if (nt >= 2 &&
            !(ok = mbar_wait(bar(B_SFREE + b), ((nt - 2) >> 1) & 1, abort_flag, p.status)))
          break;
        tc_fence_after();
        mma_xyT(tmem + kColS + 64 * b, smQ + b * 32768, smK);
        if (!(ok = mbar_wait(bar(B_DOFULL + b), (nt >> 1) & 1, abort_flag, p.status))) break;
        tc_fence_after();
        mma_xyT(tmem + kColDP + 64 * b, smDO + b * 32768, smV);
        mma_commit(bar(B_SFULL + b));
        if (nt >= 1) {
          if (!(ok = mbar_wait(bar(B_PDSFULL + (b ^ 1)), ((nt - 1) >> 1) & 1, abort_flag,
                               p.status)))
            break;
          tc_fence_after();
          kv_products(nt - 1);
        }
      }
      if (ok && ntiles > 0 &&
          (ok = mbar_wait(bar(B_PDSFULL + ((ntiles - 1) & 1)), ((ntiles - 1) >> 1) & 1,
                          abort_flag, p.status))) {
        tc_fence_after();
        kv_products(ntiles - 1);
      }
      mma_commit(bar(B_DONE));
      mbar_wait_drain(bar(B_DONE), 0);  // MMAs done before TMEM is freed
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int g = warp / 4, wq = warp % 4;  // warpgroup g takes the tiles nt = g (mod 2)
    const int rho = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    bool ok = true;
    // the row of this warpgroup's next tile and its statistics are loaded one tile ahead
    auto stats = [&](int nt, QRow &q, float &lse2, float &Drow, int &r) {
      r = row_of(nt);
      q = qrow<BK>(p, nt % p.mtiles, rho, h, r, s0, n);
      lse2 = q.valid ? __ldg(p.lse + q.idx) * kLog2e : 0.f;
      Drow = q.valid ? __ldg(p.Dv + q.idx) : 0.f;
    };
    QRow qn;
    float lse_n = 0.f, D_n = 0.f;
    int r_n = 0;
    if (g < ntiles) stats(g, qn, lse_n, D_n, r_n);
    for (int nt = g; nt < ntiles; nt += 2) {
      const int b = nt & 1;
      const QRow q = qn;
      const float lse2 = lse_n, Drow = D_n;
      const bool diag = r_n == j;
      if (nt + 2 < ntiles) stats(nt + 2, qn, lse_n, D_n, r_n);
      if (!(ok = mbar_wait(bar(B_SFULL + b), (nt >> 1) & 1, abort_flag, p.status))) break;
      // P / dS of tile nt-2 have been consumed by its dK / dV products
      if (nt >= 2 &&
          !(ok = mbar_wait(bar(B_PDSFREE + b), ((nt - 2) >> 1) & 1, abort_flag, p.status)))
        break;
      tc_fence_after();
      tile_grad64(tmem + lane_base + kColS + 64 * b, tmem + lane_base + kColDP + 64 * b,
                  smP + b * 16384, smDS + b * 16384, rho, q.valid, diag, e * 64, q.tok,
                  p.scale_log2, lse2, Drow);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(B_SFREE + b));
        mbar_arrive(bar(B_PDSFULL + b));
      }
    }
    // epilogue: TMEM lane = head-dim column d, 64 columns = the tile's keys;
    // warpgroup 0 writes dV, warpgroup 1 dK
    if (ok && mbar_wait(bar(B_DONE), 0, abort_flag, p.status)) {
      tc_fence_after();
      const int d = rho;
      uint16_t *out = g == 0 ? p.dV : p.dK;
      const float mul = g == 0 ? 1.f : p.scale;
      const uint32_t col = g == 0 ? kColDV : kColDK;
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_base + col + c0, rr);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int key = j * BK + e * 64 + c0 + c;  // sequence-relative key position
          if (key < n) {
            const __nv_bfloat16 v = __float2bfloat16_rn(__uint_as_float(rr[c]) * mul);
            out[((size_t)h * p.T + s0 + key) * kD + d] = *reinterpret_cast<const uint16_t *>(&v);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- dK / dV pass, 128-key blocks

// b = 128: one CTA per key block with its 128 keys on the TMEM lanes (M = 128), so
// P and dS never leave tensor memory: S^T = K Q^T and dP^T = V dO^T (N = 64 query
// rows of one head and half a query block per tile), the softmax warps turn them
// into P^T and dS^T (bf16 pairs written over the S^T / dP^T columns they read:
// the A operand layout), and dV += P^T dO, dK += dS^T Q run as TS products with
// N = d.  Shared memory holds K, V and a four-stage ring of Q / dO tiles (no P / dS
// buffers).  The MMA warp hears from the softmax warps and of landed copies through
// named barriers: an mbarrier check costs it a few hundred cycles while the MMAs
// stream operands from shared memory, and the MMA queue runs dry meanwhile.  Per key lane, the query columns a tile may use are [lo, hi): the
// causal triangle on the diagonal block (key <= query), the sequence end, and keys
// past the sequence end use none.  The query-row statistics (lse, D) of a tile are
// staged per warp in shared memory and read as broadcasts.  352 threads: two
// softmax warpgroups on alternate tiles (warpgroup 0 writes dV, 1 dK at the end),
// warp 8 TMA, warp 9 MMA, warp 10 turns the copies' mbarriers into named barriers.
namespace kv128 {
constexpr int kThreads = 352;
constexpr int NQ = 4;  // Q / dO stages (Q 16 KB | dO 16 KB)
constexpr int kOffK = 0, kOffV = 32768, kOffQ = 65536;
constexpr int kStage = 32768;
constexpr int kOffStat = kOffQ + NQ * kStage;  // per softmax warp: lse2[64] | D[64]
constexpr int kOffBar = kOffStat + 8 * 512;
constexpr int B_KVFULL = 0, B_QFULL = 1, B_QEMPTY = B_QFULL + NQ, B_SFULL = B_QEMPTY + NQ;
constexpr int B_DONE = B_SFULL + 2;
// named barriers: softmax warpgroup g done with its tile (4 warps + the MMA warp), and
// Q / dO stage st landed (the watcher warp + the MMA warp)
constexpr uint32_t kNbPDS = 1, kNbQ = 3, kPdsThreads = 160, kQThreads = 64;
constexpr int kOffCtl = kOffBar + (B_DONE + 1) * 8;
constexpr int kSmemBytes = kOffCtl + 16 + 1024;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384, kTmemCols = 512;
static_assert(kSmemBytes <= 232448, "shared memory budget");
}  // namespace kv128

// P^T and dS^T of one 64-column S^T / dP^T tile row (this key lane, 64 query columns)
// written back over the columns read (chunk c -> columns 8 c .. 8 c + 7), 16 columns
// at a time with the next chunk's loads in flight.  Columns outside [lo, hi) get
// P = dS = 0; st = this warp's staged lse2 / D.
BSA_DEV void tile_grad64_t(uint32_t tS, uint32_t tDP, const float *st, int lo, int hi,
                           float scale_log2) {
  uint32_t sb[2][16], db[2][16];
  const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
  tmem_ld16_async(tS, sb[0]);
  tmem_ld16_async(tDP, db[0]);
  tmem_wait_ld16x2(sb[0], db[0]);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (c < 3) {
      tmem_ld16_async(tS + 16 * (c + 1), sb[(c + 1) & 1]);
      tmem_ld16_async(tDP + 16 * (c + 1), db[(c + 1) & 1]);
    }
    const uint32_t(&sv)[16] = sb[c & 1];
    const uint32_t(&dv)[16] = db[c & 1];
    uint32_t pk[8], dk[8];
#pragma unroll
    for (int e4 = 0; e4 < 4; ++e4) {  // four columns: two packed pairs
      const float4 l4 = *reinterpret_cast<const float4 *>(st + 16 * c + 4 * e4);
      const float4 d4 = *reinterpret_cast<const float4 *>(st + 64 + 16 * c + 4 * e4);
#pragma unroll
      for (int hp = 0; hp < 2; ++hp) {
        const int e = 2 * e4 + hp, col = 16 * c + 2 * e;
        const float la = hp ? l4.z : l4.x, lb = hp ? l4.w : l4.y;
        const float da = hp ? d4.z : d4.x, db_ = hp ? d4.w : d4.y;
        const uint64_t z = f2_fma(f2_pack(sv[2 * e], sv[2 * e + 1]), sc2, f2_pack(-la, -lb));
        const float p0 = col >= lo && col < hi ? fast_exp2(f2_lo(z)) : 0.f;
        const float p1 = col + 1 >= lo && col + 1 < hi ? fast_exp2(f2_hi(z)) : 0.f;
        const uint64_t ds =
            f2_mul(f2_pack(p0, p1), f2_add(f2_pack(dv[2 * e], dv[2 * e + 1]), f2_pack(-da, -db_)));
        pk[e] = pack_bf16x2(p0, p1);
        dk[e] = pack_bf16x2(f2_lo(ds), f2_hi(ds));
      }
    }
    tmem_st8_nowait(tS + 8 * c, pk);
    tmem_st8_nowait(tDP + 8 * c, dk);
    if (c < 3) tmem_wait_ld16x2(sb[(c + 1) & 1], db[(c + 1) & 1]);
  }
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kv128::kThreads, 1) bwd_dkdv128_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
    const BwdTcParams p) {
  using namespace kv128;
  constexpr int BK = 128;
  const int u = blockIdx.x;
  if (u >= __ldg(p.kt_bucket + BSA_NUM_BUCKETS)) return;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *sm = smem_raw + (sbase - raw);
  auto bar = [&](int k) { return sbase + kOffBar + 8u * (uint32_t)k; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffCtl);
  volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(sm + kOffCtl + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(bar(B_KVFULL), 1);
    for (int st = 0; st < NQ; ++st) {
      mbar_init(bar(B_QFULL + st), 1);
      mbar_init(bar(B_QEMPTY + st), 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(bar(B_SFULL + b), 1);
    mbar_init(bar(B_DONE), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Synchronisation: mbarrier waits are bounded and made warp-uniform; every named
  // barrier is reached once per tile by each of its warps whether or not a wait gave
  // up, so none of them can be left waiting.
  const int kb = __ldg(p.kt_work + u);  // (i * H_kv + h) * N_q + j
  const int j = kb % p.Nq, h = (kb / p.Nq) % p.Hk, i = kb / (p.Nq * p.Hk);
  const int s0 = __ldg(p.cu + i), n = __ldg(p.cu + i + 1) - s0;
  const int tpr = 2 * p.G;  // 64-row query tiles per selecting row: G heads x 2 halves
  const int l0 = __ldg(p.kt_ptr + kb), ntiles = (__ldg(p.kt_ptr + kb + 1) - l0) * tpr;
  const uint32_t smK = sbase + kOffK, smV = sbase + kOffV, smQ = sbase + kOffQ;
  auto row_of = [&](int nt) { return __ldg(p.kt_rows + l0 + nt / tpr); };

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool ok = true;
      int issued[NQ];
      for (int st = 0; st < NQ; ++st) issued[st] = -1;
      mbar_arrive_expect_tx(bar(B_KVFULL), 8 * 8192);
      for (int pn = 0; pn < 2; ++pn)
        for (int hf = 0; hf < 2; ++hf) {
          tma_load_3d(smK + pn * 16384 + hf * 8192, &tmK, bar(B_KVFULL), pn * 64,
                      s0 + j * BK + hf * 64, h);
          tma_load_3d(smV + pn * 16384 + hf * 8192, &tmV, bar(B_KVFULL), pn * 64,
                      s0 + j * BK + hf * 64, h);
        }
      for (int nt = 0; nt < ntiles; ++nt) {
        const int st = nt % NQ;
        if (nt >= NQ &&
            !(ok = mbar_wait(bar(B_QEMPTY + st), ((nt - NQ) / NQ) & 1, abort_flag, p.status)))
          break;
        const int r = row_of(nt), tt = nt % tpr;
        const int y = s0 + r * BK + 64 * (tt & 1), hq = h * p.G + (tt >> 1);
        mbar_arrive_expect_tx(bar(B_QFULL + st), 4 * 8192);
        issued[st] = (nt / NQ) & 1;
        for (int pn = 0; pn < 2; ++pn) {  // Q | dO, each two 8 KB panels of 64 rows
          tma_load_3d(smQ + st * kStage + pn * 8192, &tmQ, bar(B_QFULL + st), pn * 64, y, hq);
          tma_load_3d(smQ + st * kStage + 16384 + pn * 8192, &tmDO, bar(B_QFULL + st), pn * 64,
                      y, hq);
        }
      }
      mbar_wait_drain(bar(B_KVFULL), 0);
      for (int st = 0; st < NQ; ++st)
        if (issued[st] >= 0) mbar_wait_drain(bar(B_QFULL + st), issued[st]);
      (void)ok;
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    {
      bool ok = true;
      if (lane == 0) ok = mbar_wait(bar(B_KVFULL), 0, abort_flag, p.status);
      // dV += P^T dO, dK += dS^T Q of tile nt (64 query rows in steps of 16)
      auto kv_products = [&](int nt) {
        const int b = nt & 1, st = nt % NQ;
        const uint32_t ql = desc_lo(smQ + st * kStage, 8192);
        const uint32_t dol = desc_lo(smQ + st * kStage + 16384, 8192);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts_lo(tmem + kColDV, tmem + kColS + 64 * b + 8 * kk, dol + kk * 128, kDescHi,
                    kIdescDQ, (nt > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts_lo(tmem + kColDK, tmem + kColDP + 64 * b + 8 * kk, ql + kk * 128, kDescHi,
                    kIdescDQ, (nt > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(B_QEMPTY + st));
      };
      // S^T / dP^T of tile nt into buffer nt & 1 (its last reader, kv_products(nt - 2),
      // was issued before by this thread)
      auto s_products = [&](int nt) {
        const int b = nt & 1, st = nt % NQ;
        mma_xyT(tmem + kColS + 64 * b, smK, smQ + st * kStage);
        mma_xyT(tmem + kColDP + 64 * b, smV, smQ + st * kStage + 16384);
        mma_commit(bar(B_SFULL + b));
      };
      // lane 0 issues; the whole warp takes the named barriers.  Tile nt's products
      // and tile nt + 2's S^T / dP^T go out back to back after one pair of checks.
      for (int nt = 0; nt < 2 && nt < ntiles; ++nt) {
        nbar_sync(kNbQ + nt, kQThreads);
        if (lane == 0 && ok) {
          tc_fence_after();
          s_products(nt);
        }
        __syncwarp();
      }
      for (int nt = 0; nt < ntiles; ++nt) {
        const bool next = nt + 2 < ntiles;
        nbar_sync(kNbPDS + (nt & 1), kPdsThreads);
        if (next) nbar_sync(kNbQ + (nt + 2) % NQ, kQThreads);
        if (lane == 0 && ok) {
          tc_fence_after();
          kv_products(nt);
          if (next) s_products(nt + 2);
        }
        __syncwarp();
      }
      if (lane == 0) {
        mma_commit(bar(B_DONE));
        mbar_wait_drain(bar(B_DONE), 0);  // MMAs done before TMEM is freed
      }
      __syncwarp();
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ copy watcher
    bool ok = true;
    for (int nt = 0; nt < ntiles; ++nt) {
      if (ok) ok = mbar_wait(bar(B_QFULL + nt % NQ), (nt / NQ) & 1, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
      nbar_sync(kNbQ + nt % NQ, kQThreads);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int g = warp / 4, wq = warp % 4;  // warpgroup g takes the tiles nt = g (mod 2)
    const int kin = wq * 32 + lane;         // this lane's key within the block
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const bool key_ok = j * BK + kin < n;
    float *stat = reinterpret_cast<float *>(sm + kOffStat) + warp * 128;
    // lse / D of query columns lane and lane + 32 of tile nt (0 past the sequence
    // end), loaded one tile of this warpgroup ahead of their use
    auto stat_load = [&](int nt, float(&v)[4]) {
      if (nt >= ntiles) return;
      const int r = row_of(nt), tt = nt % tpr;
      const int qtok0 = 64 * (tt & 1);
      const size_t q0 = (size_t)(h * p.G + (tt >> 1)) * p.T + s0 + r * BK + qtok0;
      const int nq = min(64, n - (r * BK + qtok0));
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = lane + 32 * e;
        v[e] = c < nq ? __ldg(p.lse + q0 + c) : 0.f;
        v[2 + e] = c < nq ? __ldg(p.Dv + q0 + c) : 0.f;
      }
    };
    float nxt[4] = {0.f, 0.f, 0.f, 0.f};
    stat_load(g, nxt);
    bool ok = true;
    for (int nt = g; nt < ntiles; nt += 2) {
      const int b = nt & 1;
      const int r = row_of(nt), tt = nt % tpr;
      const int qtok0 = 64 * (tt & 1);                  // first query of the tile in block r
      const int nq = min(64, n - (r * BK + qtok0));     // valid query columns
      // stage this tile's lse2 / D for the broadcasts, then start the next tile's loads
      stat[lane] = nxt[0] * kLog2e;
      stat[lane + 32] = nxt[1] * kLog2e;
      stat[64 + lane] = nxt[2];
      stat[96 + lane] = nxt[3];
      __syncwarp();
      stat_load(nt + 2, nxt);
      const int lo = (j == r) ? max(0, kin - qtok0) : 0;  // causal: key <= query
      const int hi = key_ok ? nq : 0;
      if (ok) ok = mbar_wait(bar(B_SFULL + b), (nt >> 1) & 1, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        tile_grad64_t(tmem + lane_base + kColS + 64 * b, tmem + lane_base + kColDP + 64 * b, stat,
                      lo, hi, p.scale_log2);
      }
      tc_fence_before();
      nbar_sync(kNbPDS + g, kPdsThreads);
    }
    // epilogue: TMEM lane = key, 128 columns = d; warpgroup 0 writes dV, 1 dK
    if (ok) ok = mbar_wait(bar(B_DONE), 0, abort_flag, p.status);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      uint16_t *out = g == 0 ? p.dV : p.dK;
      const float mul = g == 0 ? 1.f : p.scale;
      const uint32_t col = g == 0 ? kColDV : kColDK;
      uint4 *dst = reinterpret_cast<uint4 *>(out + ((size_t)h * p.T + s0 + j * BK + kin) * kD);
#pragma unroll
      for (int c0 = 0; c0 < kD; c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_base + col + c0, rr);
        uint32_t o[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          o[e] = pack_bf16x2(__uint_as_float(rr[2 * e]) * mul, __uint_as_float(rr[2 * e + 1]) * mul);
        if (key_ok)
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[c0 / 8 + v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

template <int BK>
cudaError_t launch_bk(const bsa_shape_t &s, const void *Q, const void *K, const void *V,
                      const void *dO, BwdTcParams p, cudaStream_t st) {
  CUtensorMap mq, mdo, mk, mv;
  if (!make_tmap_3d_bf16(&mq, Q, kD, s.total_tokens, s.num_heads, 64, BK, 128 / BK) ||
      !make_tmap_3d_bf16(&mdo, dO, kD, s.total_tokens, s.num_heads, 64, BK, 128 / BK) ||
      !make_tmap_3d_bf16(&mk, K, kD, s.total_tokens, s.num_kv_heads, 64, 64, 1) ||
      !make_tmap_3d_bf16(&mv, V, kD, s.total_tokens, s.num_kv_heads, 64, 64, 1))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(bwd_dq_tc_kernel<BK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, dq::kSmemBytes);
  if (e != cudaSuccess) return e;
  if constexpr (BK == 64) {
    e = cudaFuncSetAttribute(bwd_dkdv_tc_kernel<BK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kv::kSmemBytes);
  } else {
    e = cudaFuncSetAttribute(bwd_dkdv128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kv128::kSmemBytes);
  }
  if (e != cudaSuccess) return e;
  const long long rows = (long long)s.num_seqs * s.num_kv_heads * s.max_blocks;
  const unsigned dq_grid = (unsigned)std::min<long long>(rows * p.mtiles, num_sms());
  bwd_dq_tc_kernel<BK><<<dq_grid, dq::kThreads, dq::kSmemBytes, st>>>(mq, mdo, mk, mv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if constexpr (BK == 64) {
    bwd_dkdv_tc_kernel<BK><<<(unsigned)rows, kv::kThreads, kv::kSmemBytes, st>>>(mq, mdo, mk, mv,
                                                                                 p);
  } else {
    // query tiles of 64 rows of one head: their own tensor maps
    CUtensorMap mq64, mdo64;
    if (!make_tmap_3d_bf16(&mq64, Q, kD, s.total_tokens, s.num_heads, 64, 64, 1) ||
        !make_tmap_3d_bf16(&mdo64, dO, kD, s.total_tokens, s.num_heads, 64, 64, 1))
      return cudaErrorInvalidValue;
    bwd_dkdv128_kernel<<<(unsigned)rows, kv128::kThreads, kv128::kSmemBytes, st>>>(mq64, mdo64, mk,
                                                                                 mv, p);
  }
  return cudaGetLastError();
}

}  // namespace

bool attention_bwd_tc_supported(const bsa_shape_t &s) {
  return s.dtype == BSA_BF16 && s.head_dim == kD && (s.block == 64 || s.block == 128);
}

// [count | kt_work | kt_ptr (+1) | kt_bucket | row bitmap (ceil(N_q / 32) words per key
// block) | kt_rows (one per (row, block) pair of any valid worklist: at most r + 1 per row)]
size_t attention_bwd_tc_index_bytes(const bsa_shape_t &s) {
  const size_t rows = (size_t)s.num_seqs * s.num_kv_heads * s.max_blocks;
  const size_t W = ((size_t)s.max_blocks + 31) / 32;
  const size_t pairs = (size_t)s.num_seqs * s.num_kv_heads * s.max_blocks * (s.max_blocks + 1) / 2;
  return 2 * up256(rows * 4) + up256((rows + 1) * 4) + up256((BSA_NUM_BUCKETS + 1) * 4) +
         up256(rows * W * 4) + up256(pairs * 4);
}

cudaError_t launch_attention_bwd_tc(const bsa_shape_t &s, const void *Q, const void *K,
                                    const void *V, const void *dO, const float *lse,
                                    const float *Dv, const int32_t *row_ptr,
                                    const int32_t *col_idx, const int32_t *work,
                                    const int32_t *bucket_off, float scale, void *dQ, void *dK,
                                    void *dV, void *ws, int32_t *dev_status, cudaStream_t st) {
  const int nrows = s.num_seqs * s.num_kv_heads * s.max_blocks;
  const int W = (s.max_blocks + 31) / 32;
  char *w = static_cast<char *>(ws);
  int32_t *cnt = reinterpret_cast<int32_t *>(w);
  w += up256((size_t)nrows * 4);
  int32_t *kt_work = reinterpret_cast<int32_t *>(w);
  w += up256((size_t)nrows * 4);
  int32_t *kt_ptr = reinterpret_cast<int32_t *>(w);
  w += up256(((size_t)nrows + 1) * 4);
  int32_t *kt_bucket = reinterpret_cast<int32_t *>(w);
  w += up256((BSA_NUM_BUCKETS + 1) * 4);
  uint32_t *bits = reinterpret_cast<uint32_t *>(w);
  w += up256((size_t)nrows * W * 4);
  int32_t *kt_rows = reinterpret_cast<int32_t *>(w);

  // zero the row bitmap and the key gradients: a key block that no row selected
  // keeps dK = dV = 0
  cudaError_t e = cudaMemsetAsync(bits, 0, (size_t)nrows * W * 4, st);
  if (e != cudaSuccess) return e;
  const size_t kv_bytes = (size_t)s.num_kv_heads * s.total_tokens * kD * 2;
  if ((e = cudaMemsetAsync(dK, 0, kv_bytes, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dV, 0, kv_bytes, st)) != cudaSuccess) return e;
  const int blocks = std::max(1, std::min(4 * num_sms(), (nrows + 255) / 256));
  kt_mark_kernel<<<blocks, 256, 0, st>>>(row_ptr, col_idx, nrows, s.max_blocks, W, bits,
                                         dev_status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  kt_count_kernel<<<blocks, 256, 0, st>>>(bits, nrows, W, cnt);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = launch_length_scan(cnt, kt_ptr, kt_work, kt_bucket, nrows, st)) != cudaSuccess)
    return e;
  const int eblocks = (int)std::max<size_t>(
      1, std::min<size_t>((size_t)8 * num_sms(), ((size_t)nrows * 32 + 255) / 256));
  kt_emit_kernel<<<eblocks, 256, 0, st>>>(bits, kt_ptr, kt_rows, nrows, W);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  BwdTcParams p;
  p.cu = s.cu_seqlens;
  p.row_ptr = row_ptr;
  p.col_idx = col_idx;
  p.work = work;
  p.bucket_off = bucket_off;
  p.kt_ptr = kt_ptr;
  p.kt_rows = kt_rows;
  p.kt_work = kt_work;
  p.kt_bucket = kt_bucket;
  p.lse = lse;
  p.Dv = Dv;
  p.dQ = static_cast<uint16_t *>(dQ);
  p.dK = static_cast<uint16_t *>(dK);
  p.dV = static_cast<uint16_t *>(dV);
  p.status = dev_status;
  p.T = s.total_tokens;
  p.Hk = s.num_kv_heads;
  p.G = s.num_heads / s.num_kv_heads;
  p.Nq = s.max_blocks;
  p.mtiles = (p.G * s.block + 127) / 128;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  if (s.block == 64) return launch_bk<64>(s, Q, K, V, dO, p, st);
  return launch_bk<128>(s, Q, K, V, dO, p, st);
}

}  // namespace bsa
