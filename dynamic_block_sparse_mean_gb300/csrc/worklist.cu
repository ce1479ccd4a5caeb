// a4: J -> CSR worklist ("2.1 · 粗粒度选择" §3.1 index representations: the fixed
// table J and the CSR row_ptr / col_idx form; PaperTrace 5-1 "从索引输出到工作表":
// rows grouped into length buckets and handed to one persistent launch).
//   1. rows kernel   validates each row and records its length (grid-wide)
//   2. scan kernel   row_ptr by prefix sum, and the work list: a stable counting
//                    sort of rows, long rows by exact length, short ones by
//                    capacity bucket, longest first (one CTA); the capacity
//                    buckets are contiguous ranges of it
//   3. fill kernel   copies the block ids into col_idx (grid-wide)
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace bsa {
namespace {

constexpr int kScanThreads = 1024;

// Logical block of row (i, h, qb): qb, or in a chunked prefill qb + the blocks
// cached before the chunk (qoff: cached tokens per sequence); -1 when the row is
// not one (past the sequence's end, or the sequence's prefix is unusable).
BSA_DEV int row_block(const int32_t *__restrict__ cu, const int32_t *__restrict__ qoff, int row,
                      int Nq, int Nk, int Hk, int b, int32_t *dev_status) {
  const int qb = row % Nq, i = row / (Nq * Hk);
  const int n = cu[i + 1] - cu[i];
  if (qb >= (n + b - 1) / b) return -1;
  if (qoff == nullptr) return qb;
  const int pre = qoff[i];
  if (!chunk_ok(pre, n, b, Nk)) {
    if (qb == 0 && (row / Nq) % Hk == 0) set_status(dev_status, BSA_ERR_CACHE);
    return -1;
  }
  return qb + pre / b;
}

// Row code: 0 = not a row (past the sequence end); c > 0 = copy c ids from J;
// -1 = the row holds only its diagonal block (empty row, or a malformed row).
__global__ void wl_rows_kernel(const int32_t *__restrict__ J, const int32_t *__restrict__ counts,
                               const int32_t *__restrict__ cu, const int32_t *__restrict__ qoff,
                               int32_t *__restrict__ code, int32_t *dev_status, int nrows, int Nq,
                               int Nk, int Hk, int b, int k_max) {
  grid_dep_wait();  // J and counts may come from the previous launch
  for (int row = blockIdx.x * blockDim.x + threadIdx.x; row < nrows;
       row += gridDim.x * blockDim.x) {
    const int r = row_block(cu, qoff, row, Nq, Nk, Hk, b, dev_status);
    if (r < 0) {
      code[row] = 0;
      continue;
    }
    const int c = counts[row];
    if (c < 0 || c > k_max) {
      set_status(dev_status, BSA_ERR_COUNT);
      code[row] = -1;
      continue;
    }
    if (c == 0) {
      code[row] = -1;
      continue;
    }
    const int32_t *Jr = J + (size_t)row * k_max;
    int prev = -1, err = 0;
    for (int e = 0; e < c; ++e) {
      const int v = Jr[e];
      if (v < 0 || v > r) {
        err = BSA_ERR_INDEX_RANGE;
        break;
      }
      if (v <= prev) {
        err = BSA_ERR_INDEX_ORDER;
        break;
      }
      prev = v;
    }
    if (err) set_status(dev_status, err);
    code[row] = err ? -1 : c;
  }
  grid_dep_launch();
}

// Exclusive scan over the block of N values per thread at once (warp shuffles,
// then a scan of the 32 warp totals): v becomes each thread's exclusive prefix,
// tot the block totals.
template <int N>
BSA_DEV void block_scan_n(int (&v)[N], int (&tot)[N], int (*wsum)[N]) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  int inc[N];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    inc[k] = v[k];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc[k], off);
      if (lane >= off) inc[k] += y;
    }
  }
  if (lane == 31)
#pragma unroll
    for (int k = 0; k < N; ++k) wsum[warp][k] = inc[k];
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < N; ++k) {
      int w = wsum[lane][k], x = w;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
      }
      wsum[lane][k] = x - w;  // exclusive prefix of this warp
      if (lane == 31) wsum[32][k] = x;
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < N; ++k) {
    v[k] = inc[k] - v[k] + wsum[warp][k];
    tot[k] = wsum[32][k];
  }
}

// One CTA: row_ptr by prefix sum of the row lengths, and the work list of the rows
// with at least one block: the rows longer than `exact_above` blocks first, longest
// first (lengths above 256 count as 256), then the others by capacity bucket, largest
// first; rows of equal key in row-id order (a stable counting sort).  A persistent
// launch that hands the list out round-robin ends close to the ideal when long rows
// of different lengths are in exact order (varlen workload: 2.6 % above the ideal by
// bucket, 1.0 % with exact order above 32 blocks); for short rows of nearly equal
// length the row-id order of the buckets, which keeps a KV head's rows together,
// measured faster.  The capacity buckets are contiguous ranges of the list: bucket s
// (capacity 256 >> s) starts after the rows longer than its capacity.  For the
// row_ptr scan thread t owns a contiguous chunk of rows; for the sort warp w does,
// walking it 32 rows at a time (equal keys inside a group of 32 ranked by lane).
__global__ void __launch_bounds__(kScanThreads) wl_scan_kernel(
    const int32_t *__restrict__ code, int32_t *__restrict__ row_ptr, int32_t *__restrict__ work,
    int32_t *__restrict__ bucket_off, int nrows, int exact_above) {
  grid_dep_wait();  // the row codes come from the previous launch
  constexpr int NB = BSA_NUM_BUCKETS;
  // sort keys: 256 - min(length, 256) above exact_above, 256 - exact_above + bucket
  // below (exact_above is 0 or a power of two from 4 to 128)
  constexpr int NK = 256;
  constexpr int NW = kScanThreads / 32;   // warps
  __shared__ int wsum[33][1];
  __shared__ int hist[NK][NW];  // per (key, warp): rows, then the first position
  const int t = threadIdx.x, warp = t / 32, lane = t % 32;
  // row_ptr: prefix sum of the lengths (an error row, code -1, holds one block)
  {
    const int chunk = (nrows + kScanThreads - 1) / kScanThreads;
    const int lo = min(nrows, t * chunk), hi = min(nrows, lo + chunk);
    int v[1] = {0}, tot[1];
    for (int row = lo; row < hi; ++row) {
      const int c = code[row];
      v[0] += c < 0 ? 1 : c;
    }
    block_scan_n<1>(v, tot, wsum);
    int off = v[0];
    for (int row = lo; row < hi; ++row) {
      const int c = code[row];
      row_ptr[row] = off;
      off += c < 0 ? 1 : c;
    }
    if (t == 0) row_ptr[nrows] = tot[0];
  }
  for (int k = t; k < NK * NW; k += kScanThreads) (&hist[0][0])[k] = 0;
  __syncthreads();
  const int wchunk = (nrows + NW - 1) / NW;
  const int wlo = min(nrows, warp * wchunk), whi = min(nrows, wlo + wchunk);
  auto key_of = [&](int row) {  // -1: an empty row, not listed
    if (row >= whi) return -1;
    const int c = code[row];
    const int len = c < 0 ? 1 : c;
    if (len <= 0) return -1;
    if (len > exact_above) return NK - min(len, NK);
    int cap = 4, sb = 6;  // capacity bucket: 256 -> 0, ..., 4 -> 6
    while (cap < len && sb > 0) {
      cap <<= 1;
      --sb;
    }
    return NK - exact_above + sb;
  };
  // rows per (key, warp)
  for (int r0 = wlo; r0 < whi; r0 += 32) {
    const int key = key_of(r0 + lane);
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && lane == __ffs(peers) - 1) hist[key][warp] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // first position of each (key, warp): exclusive scan in key-major order, 8 entries
  // per thread
  constexpr int PER = NK * NW / kScanThreads;
  static_assert(PER * kScanThreads == NK * NW, "scan split");
  int *flat = &hist[0][0];
  int loc[PER], v[1] = {0}, tot[1];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    loc[i] = flat[PER * t + i];
    v[0] += loc[i];
  }
  __syncthreads();
  block_scan_n<1>(v, tot, wsum);
  int acc = v[0];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    flat[PER * t + i] = acc;
    acc += loc[i];
  }
  __syncthreads();
  if (t == 0) {
    bucket_off[0] = 0;
#pragma unroll
    for (int q = 1; q < NB; ++q)  // rows longer than 256 >> q
      bucket_off[q] = hist[(256 >> q) >= exact_above ? NK - (256 >> q) : NK - exact_above + q][0];
    bucket_off[NB] = tot[0];
  }
  // placement: the (key, warp) start, plus the rows of the same key before this one
  for (int r0 = wlo; r0 < whi; r0 += 32) {
    const int row = r0 + lane, key = key_of(row);
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int base = key >= 0 ? hist[key][warp] : 0;
    if (key >= 0) work[base + __popc(peers & ((1u << lane) - 1u))] = row;
    __syncwarp();
    if (key >= 0 && lane == __ffs(peers) - 1) hist[key][warp] = base + __popc(peers);
    __syncwarp();
  }
  grid_dep_launch();
}

__global__ void wl_fill_kernel(const int32_t *__restrict__ J, const int32_t *__restrict__ code,
                               const int32_t *__restrict__ row_ptr, int32_t *__restrict__ col_idx,
                               const int32_t *__restrict__ cu, const int32_t *__restrict__ qoff,
                               int nrows, int Nq, int Nk, int Hk, int b, int k_max) {
  grid_dep_wait();  // codes and row_ptr come from the previous launches
  for (int row = blockIdx.x * blockDim.x + threadIdx.x; row < nrows;
       row += gridDim.x * blockDim.x) {
    const int c = code[row];
    if (c == 0) continue;
    int32_t *out = col_idx + row_ptr[row];
    if (c < 0) {  // the diagonal: the row's logical block
      out[0] = row_block(cu, qoff, row, Nq, Nk, Hk, b, nullptr);
      continue;
    }
    const int32_t *Jr = J + (size_t)row * k_max;
    for (int e = 0; e < c; ++e) out[e] = Jr[e];
  }
  grid_dep_launch();
}

// Density 1 (every causal block): row r of a sequence with nb blocks holds 0..r.
__global__ void wl_causal_rows_kernel(const int32_t *__restrict__ cu, int32_t *__restrict__ code,
                                      int nrows, int Nq, int Hk, int b) {
  for (int row = blockIdx.x * blockDim.x + threadIdx.x; row < nrows;
       row += gridDim.x * blockDim.x) {
    const int r = row % Nq, i = row / (Nq * Hk);
    const int nb = (cu[i + 1] - cu[i] + b - 1) / b;
    code[row] = r < nb ? r + 1 : 0;
  }
}

__global__ void wl_causal_fill_kernel(const int32_t *__restrict__ code,
                                      const int32_t *__restrict__ row_ptr,
                                      int32_t *__restrict__ col_idx, int nrows) {
  // one warp per row: the row's block ids 0 .. c - 1
  const int lane = threadIdx.x % 32;
  for (int row = (blockIdx.x * blockDim.x + threadIdx.x) / 32; row < nrows;
       row += gridDim.x * blockDim.x / 32) {
    const int c = code[row];
    int32_t *out = col_idx + row_ptr[row];
    for (int e = lane; e < c; e += 32) out[e] = e;
  }
}

// Scratch of bsa_build_worklist_noalloc: one row code per row, shared by every
// call on a device.  Host code must not pass this name to a kernel (on the host
// it is only a stand-in); it passes the address cudaGetSymbolAddress returns.
__device__ __align__(256) int32_t g_noalloc_rows[BSA_WORKLIST_NOALLOC_MAX_ROWS];

}  // namespace

// The driver's cuCtxGetCurrent, reached through the runtime (no libcuda link).
PFN_cuCtxGetCurrent_v4000 ctx_get_current_fn() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
  });
  return fn;
}

// Device address of g_noalloc_rows on the current device, looked up with that
// device current and cached per device together with the CUDA context it was
// looked up in.  A call from another context of the device (the caller reset
// the device, or made its own context current) looks the address up again.
cudaError_t worklist_noalloc_scratch(int32_t **out) {
  constexpr int kMaxDevices = 64;
  static int32_t *cache[kMaxDevices] = {nullptr};
  static CUcontext cache_ctx[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CUcontext ctx = nullptr;
  auto get_ctx = ctx_get_current_fn();
  if (get_ctx == nullptr || get_ctx(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
  std::lock_guard<std::mutex> lock(mu);
  if (ctx == nullptr || cache[dev] == nullptr || cache_ctx[dev] != ctx) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_rows);  // makes the device's context current
    if (e != cudaSuccess) return e;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorUnknown;
    cache[dev] = static_cast<int32_t *>(p);
    cache_ctx[dev] = ctx;
  }
  *out = cache[dev];
  return cudaSuccess;
}

size_t worklist_workspace_bytes(const bsa_shape_t &s, int32_t) {
  return (size_t)s.num_seqs * s.num_kv_heads * s.max_blocks * sizeof(int32_t);
}

cudaError_t launch_worklist(const bsa_shape_t &s, int32_t k_max, const int32_t *J,
                            const int32_t *counts, int32_t *row_ptr, int32_t *col_idx,
                            int32_t *work, int32_t *bucket_off, int32_t *dev_status, void *ws,
                            cudaStream_t st, const bsa_kv_cache_t *cache) {
  const int nrows = s.num_seqs * s.num_kv_heads * s.max_blocks;
  int32_t *code = static_cast<int32_t *>(ws);
  const int blocks = min(4 * num_sms(), (nrows + 255) / 256);
  const int32_t *qoff = cache != nullptr ? cache->prefix_lens : nullptr;
  const int Nk = cache != nullptr ? cache->max_context_blocks : s.max_blocks;
  cudaError_t e = launch_dependent(wl_rows_kernel, dim3(max(blocks, 1)), dim3(256), 0, st, J,
                                   counts, s.cu_seqlens, qoff, code, dev_status, nrows,
                                   s.max_blocks, Nk, s.num_kv_heads, s.block, k_max);
  if (e != cudaSuccess) return e;
  e = launch_dependent(wl_scan_kernel, dim3(1), dim3(kScanThreads), 0, st, code, row_ptr, work,
                       bucket_off, nrows, 32);
  if (e != cudaSuccess) return e;
  return launch_dependent(wl_fill_kernel, dim3(max(blocks, 1)), dim3(256), 0, st, J, code,
                          row_ptr, col_idx, s.cu_seqlens, qoff, nrows, s.max_blocks, Nk,
                          s.num_kv_heads, s.block, k_max);
}

cudaError_t launch_length_scan(const int32_t *len, int32_t *row_ptr, int32_t *work,
                               int32_t *bucket_off, int nrows, cudaStream_t st) {
  wl_scan_kernel<<<1, kScanThreads, 0, st>>>(len, row_ptr, work, bucket_off, nrows, 128);
  return cudaGetLastError();
}

size_t causal_worklist_capacity(const bsa_shape_t &s) {
  return (size_t)s.num_seqs * s.num_kv_heads * s.max_blocks * (s.max_blocks + 1) / 2;
}

cudaError_t launch_causal_worklist(const bsa_shape_t &s, int32_t *row_ptr, int32_t *col_idx,
                                   int32_t *work, int32_t *bucket_off, void *ws, cudaStream_t st) {
  const int nrows = s.num_seqs * s.num_kv_heads * s.max_blocks;
  int32_t *code = static_cast<int32_t *>(ws);
  const int blocks = max(1, min(4 * num_sms(), (nrows + 255) / 256));
  wl_causal_rows_kernel<<<blocks, 256, 0, st>>>(s.cu_seqlens, code, nrows, s.max_blocks,
                                                s.num_kv_heads, s.block);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  wl_scan_kernel<<<1, kScanThreads, 0, st>>>(code, row_ptr, work, bucket_off, nrows, 0);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int fblocks = max(1, min(8 * num_sms(), (nrows + 7) / 8));
  wl_causal_fill_kernel<<<fblocks, 256, 0, st>>>(code, row_ptr, col_idx, nrows);
  return cudaGetLastError();
}

// Coverage of eq.(10): C = exp(lse_sparse - lse_dense) elementwise over [H, T].
namespace {
__global__ void coverage_kernel(const float *__restrict__ ls, const float *__restrict__ ld,
                                float *__restrict__ C, size_t n) {
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x)
    C[e] = expf(ls[e] - ld[e]);
}
}  // namespace

cudaError_t launch_coverage(const bsa_shape_t &s, const float *lse_sparse, const float *lse_dense,
                            float *C, cudaStream_t st) {
  const size_t n = (size_t)s.num_heads * s.total_tokens;
  const int blocks = (int)std::min<size_t>((size_t)8 * num_sms(), (n + 255) / 256);
  coverage_kernel<<<std::max(blocks, 1), 256, 0, st>>>(lse_sparse, lse_dense, C, n);
  return cudaGetLastError();
}

}  // namespace bsa
