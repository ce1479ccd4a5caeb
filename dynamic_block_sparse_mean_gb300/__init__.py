"""GB300-native dynamic block-sparse attention with a mean-pooled block router.

A thin binding over libbsa.so (include/bsa.h): it marshals torch tensors'
device pointers and the current CUDA stream into the C ABI.  Every step of
the computation runs in the library's CUDA kernels; there is no CPU path.

Typical prefill use::

    import dynamic_block_sparse_mean_gb300 as bsa
    plan = bsa.PrefillPlan(cu_seqlens_host, num_heads=32, num_kv_heads=8, head_dim=128,
                           block=64, route=bsa.RouteParams(bsa.ROUTE_TOPK, k_max=32))
    out, lse = plan.run(q, k, v)        # q [H, T, d], k / v [H_kv, T, d] bf16 on cuda
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass, field

import numpy as np
import torch

from . import _lib
from ._lib import BsaError, NUM_BUCKETS, check

ROUTE_TOPK = 0
ROUTE_THRESHOLD = 1

__all__ = ["ROUTE_TOPK", "ROUTE_THRESHOLD", "RouteParams", "PrefillShape", "PrefillPlan",
           "DecodePlan", "BsaError", "block_summaries", "route", "build_worklist",
           "attention_fwd", "attention_bwd", "causal_worklist", "coverage", "page_summaries",
           "page_summaries_append", "decode_paged", "check_status", "library_path",
           "HostPrefill", "PagedKVCache", "Chunk", "ChunkPlan", "chunk_append", "route_chunk",
           "build_worklist_chunk", "attention_chunk", "selftest_wait_timeout", "token_recall",
           "recall_tiles_per_seq"]


def library_path() -> str:
    return _lib.LIB_PATH


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return _lib.BSA_BF16
    if dt == torch.float32:
        return _lib.BSA_FP32
    raise TypeError(f"unsupported dtype {dt}: bfloat16 or float32")


@dataclass
class RouteParams:
    """Router parameters (bsa_route_params_t).  Union routing: `window` keeps the
    most recent blocks of every row (diagonal included), `global_blocks` a short
    list of block ids kept by every row that can see them; the dynamic top-k or
    threshold choice covers the rest of the history."""
    mode: int = ROUTE_TOPK
    k_max: int = 32
    k_min: int = 0
    tau_delta: float = 0.0
    force_sink: bool = False
    window: int = 1
    global_blocks: tuple = ()
    screen: int = 0   # bf16 score screening: 0 automatic, 1 always, -1 never
    _gdev: object = field(default=None, repr=False, compare=False)

    def _globals_on(self, device):
        if not self.global_blocks:
            return None
        if self._gdev is None or self._gdev.device != torch.device(device):
            self._gdev = torch.as_tensor([int(g) for g in self.global_blocks], dtype=torch.int32,
                                         device=device)
        return self._gdev

    def c(self, device=None) -> _lib.RouteParams:
        g = self._globals_on(device) if device is not None else None
        return _lib.RouteParams(self.mode, self.k_max, self.k_min, self.tau_delta,
                                1 if self.force_sink else 0, self.window,
                                0 if g is None else g.numel(),
                                None if g is None else g.data_ptr(), int(self.screen))


@dataclass
class PrefillShape:
    """Shape of a packed batch; cu_seqlens is the device tensor [B + 1] int32."""
    num_seqs: int
    total_tokens: int
    max_seqlen: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block: int
    dtype: torch.dtype
    cu_seqlens: torch.Tensor

    @property
    def max_blocks(self) -> int:
        return (self.max_seqlen + self.block - 1) // self.block

    @property
    def num_rows(self) -> int:
        return self.num_seqs * self.num_kv_heads * self.max_blocks

    def c(self) -> _lib.Shape:
        return _lib.Shape(self.num_seqs, self.total_tokens, self.max_seqlen, self.num_heads,
                          self.num_kv_heads, self.head_dim, self.block, self.max_blocks,
                          _dtype_code(self.dtype), ctypes.c_void_p(self.cu_seqlens.data_ptr()))

    @staticmethod
    def make(cu_seqlens_host, num_heads, num_kv_heads, head_dim, block, dtype=torch.bfloat16,
             device="cuda") -> "PrefillShape":
        cu = np.asarray(cu_seqlens_host, dtype=np.int64)
        lens = np.diff(cu)
        return PrefillShape(len(lens), int(cu[-1]), int(lens.max()), num_heads, num_kv_heads,
                            head_dim, block, dtype,
                            torch.as_tensor(cu.astype(np.int32), device=device))


@dataclass
class Worklist:
    row_ptr: torch.Tensor
    col_idx: torch.Tensor
    work: torch.Tensor
    bucket_off: torch.Tensor


def check_status(dev_status: torch.Tensor) -> None:
    """Raise if a kernel recorded a device-side error (synchronises on the tensor)."""
    code = int(dev_status.item())
    if code != 0:
        raise BsaError("device", code)


def block_summaries(k: torch.Tensor, shape: PrefillShape, out: torch.Tensor | None = None):
    """[B, H_kv, N_q, d] fp32 mean key of every block (bsa_block_summaries)."""
    if out is None:
        out = torch.empty(shape.num_seqs, shape.num_kv_heads, shape.max_blocks, shape.head_dim,
                          dtype=torch.float32, device=k.device)
    s = shape.c()
    check("bsa_block_summaries", _lib.lib().bsa_block_summaries(ctypes.byref(s), _p(k), _p(out),
                                                                 _stream()))
    return out


def route_workspace_bytes(shape: PrefillShape, params: RouteParams) -> int:
    s, p = shape.c(), params.c()
    return int(_lib.lib().bsa_route_workspace_size(ctypes.byref(s), ctypes.byref(p)))


def route(q, C, shape: PrefillShape, params: RouteParams, J=None, counts=None, scores=None,
          ws=None, dev_status=None):
    """J [B, H_kv, N_q, k_max] and counts [B, H_kv, N_q] (bsa_route)."""
    dev = q.device
    if J is None:
        J = torch.empty(shape.num_seqs, shape.num_kv_heads, shape.max_blocks, params.k_max,
                        dtype=torch.int32, device=dev)
    if counts is None:
        counts = torch.empty(shape.num_seqs, shape.num_kv_heads, shape.max_blocks,
                             dtype=torch.int32, device=dev)
    if ws is None:
        ws = torch.empty(max(256, route_workspace_bytes(shape, params)), dtype=torch.uint8,
                         device=dev)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    s, p = shape.c(), params.c(dev)
    check("bsa_route", _lib.lib().bsa_route(ctypes.byref(s), ctypes.byref(p), _p(q), _p(C), _p(J),
                                            _p(counts), _p(scores), _p(dev_status), _p(ws),
                                            ws.numel(), _stream()))
    return J, counts


def build_worklist(J, counts, shape: PrefillShape, k_max: int, dev_status, wl: Worklist | None = None,
                   ws=None) -> Worklist:
    dev = J.device
    rows = shape.num_rows
    if wl is None:
        wl = Worklist(torch.empty(rows + 1, dtype=torch.int32, device=dev),
                      torch.empty(max(1, rows * k_max), dtype=torch.int32, device=dev),
                      torch.empty(max(1, rows), dtype=torch.int32, device=dev),
                      torch.empty(NUM_BUCKETS + 1, dtype=torch.int32, device=dev))
    s = shape.c()
    if ws is None:
        n = int(_lib.lib().bsa_worklist_workspace_size(ctypes.byref(s), k_max))
        ws = torch.empty(max(256, n), dtype=torch.uint8, device=dev)
    check("bsa_build_worklist", _lib.lib().bsa_build_worklist(
        ctypes.byref(s), k_max, _p(J), _p(counts), _p(wl.row_ptr), _p(wl.col_idx), _p(wl.work),
        _p(wl.bucket_off), _p(dev_status), _p(ws), ws.numel(), _stream()))
    return wl


def attention_fwd(q, k, v, wl: Worklist, shape: PrefillShape, dev_status, scale: float = 0.0,
                  out=None, lse=None, want_lse: bool = True):
    """O [H, T, d] (q's dtype) and lse [H, T] fp32 on the worklist's tiles."""
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(shape.num_heads, shape.total_tokens, dtype=torch.float32, device=q.device)
    s = shape.c()
    check("bsa_attention_fwd", _lib.lib().bsa_attention_fwd(
        ctypes.byref(s), _p(q), _p(k), _p(v), _p(wl.row_ptr), _p(wl.col_idx), _p(wl.work),
        _p(wl.bucket_off), float(scale), _p(out), _p(lse), _p(dev_status), _stream()))
    return out, lse


def attention_bwd(q, k, v, o, do, lse, wl: Worklist, shape: PrefillShape, scale: float = 0.0,
                  dq=None, dk=None, dv=None, ws=None, dev_status=None):
    """dQ, dK, dV of the sparse attention for the upstream gradient do, reusing the
    forward's worklist and lse (bsa_attention_bwd)."""
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    s = shape.c()
    if ws is None:
        n = int(_lib.lib().bsa_attention_bwd_workspace_size(ctypes.byref(s)))
        ws = torch.empty(max(256, n), dtype=torch.uint8, device=q.device)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=q.device)
    check("bsa_attention_bwd", _lib.lib().bsa_attention_bwd(
        ctypes.byref(s), _p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(wl.row_ptr),
        _p(wl.col_idx), _p(wl.work), _p(wl.bucket_off), float(scale), _p(dq), _p(dk), _p(dv),
        _p(dev_status), _p(ws), ws.numel(), _stream()))
    return dq, dk, dv


def causal_worklist(shape: PrefillShape, device, wl: Worklist | None = None, ws=None) -> Worklist:
    """Worklist of every causal block (bsa_build_causal_worklist): fed to
    attention_fwd it gives dense causal attention with the same kernel."""
    s = shape.c()
    rows = shape.num_rows
    if wl is None:
        cap = int(_lib.lib().bsa_causal_worklist_capacity(ctypes.byref(s)))
        wl = Worklist(torch.empty(rows + 1, dtype=torch.int32, device=device),
                      torch.empty(max(1, cap), dtype=torch.int32, device=device),
                      torch.empty(max(1, rows), dtype=torch.int32, device=device),
                      torch.empty(NUM_BUCKETS + 1, dtype=torch.int32, device=device))
    if ws is None:
        n = int(_lib.lib().bsa_worklist_workspace_size(ctypes.byref(s), 1))
        ws = torch.empty(max(256, n), dtype=torch.uint8, device=device)
    check("bsa_build_causal_worklist", _lib.lib().bsa_build_causal_worklist(
        ctypes.byref(s), _p(wl.row_ptr), _p(wl.col_idx), _p(wl.work), _p(wl.bucket_off), _p(ws),
        ws.numel(), _stream()))
    return wl


def selftest_wait_timeout(dev_status):
    """Run the bounded-wait self-test (bsa_selftest_wait_timeout): dev_status
    receives BSA_ERR_TIMEOUT (19) and the context stays usable."""
    check("bsa_selftest_wait_timeout",
          _lib.lib().bsa_selftest_wait_timeout(_p(dev_status), _stream()))


def coverage(lse_sparse, lse_dense, shape: PrefillShape, out=None):
    """Coverage C_i of eq.(10), [H, T] fp32 (bsa_coverage)."""
    if out is None:
        out = torch.empty_like(lse_sparse)
    s = shape.c()
    check("bsa_coverage", _lib.lib().bsa_coverage(ctypes.byref(s), _p(lse_sparse), _p(lse_dense),
                                                  _p(out), _stream()))
    return out


def recall_tiles_per_seq(shape: PrefillShape) -> int:
    """64-token query tiles per sequence of the recall tile numbering."""
    s = shape.c()
    return int(_lib.lib().bsa_recall_tiles_per_seq(ctypes.byref(s)))


def token_recall(q, k, J, counts, shape: PrefillShape, t_top: int, tiles=None, hits=None,
                 dev_status=None):
    """|G_i ∩ N(i)| per query for the dense top-t teacher (bsa_token_recall): hits
    [H, T] int32, written for the queries of `tiles` (a device int32 tensor of tile
    ids (i * H + hq) * recall_tiles_per_seq + c, or None for every tile)."""
    if hits is None:
        hits = torch.full((shape.num_heads, shape.total_tokens), -1, dtype=torch.int32,
                          device=q.device)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=q.device)
    s = shape.c()
    check("bsa_token_recall", _lib.lib().bsa_token_recall(
        ctypes.byref(s), int(t_top), _p(q), _p(k), _p(J), _p(counts), int(J.shape[-1]),
        _p(tiles), 0 if tiles is None else int(tiles.numel()), _p(hits), _p(dev_status),
        _stream()))
    return hits


class PrefillPlan:
    """All buffers of one prefill shape, allocated once; run() enqueues the four calls
    (summaries, route, worklist, attention) on the current stream."""

    def __init__(self, cu_seqlens_host, num_heads: int, num_kv_heads: int, head_dim: int,
                 block: int, route: RouteParams, dtype=torch.bfloat16, device="cuda",
                 keep_scores: bool = False):
        self.shape = PrefillShape.make(cu_seqlens_host, num_heads, num_kv_heads, head_dim, block,
                                       dtype, device)
        self.params = route
        sh, dev = self.shape, device
        self.C = torch.empty(sh.num_seqs, num_kv_heads, sh.max_blocks, head_dim,
                             dtype=torch.float32, device=dev)
        self.J = torch.empty(sh.num_seqs, num_kv_heads, sh.max_blocks, route.k_max,
                             dtype=torch.int32, device=dev)
        self.counts = torch.empty(sh.num_seqs, num_kv_heads, sh.max_blocks, dtype=torch.int32,
                                  device=dev)
        self.scores = (torch.empty(sh.num_seqs, num_kv_heads, sh.max_blocks, sh.max_blocks,
                                   dtype=torch.float32, device=dev) if keep_scores else None)
        self.route_ws = torch.empty(max(256, route_workspace_bytes(sh, route)), dtype=torch.uint8,
                                    device=dev)
        rows = sh.num_rows
        self.wl = Worklist(torch.empty(rows + 1, dtype=torch.int32, device=dev),
                           torch.empty(max(1, rows * route.k_max), dtype=torch.int32, device=dev),
                           torch.empty(max(1, rows), dtype=torch.int32, device=dev),
                           torch.empty(NUM_BUCKETS + 1, dtype=torch.int32, device=dev))
        s = sh.c()
        self.wl_ws = torch.empty(max(256, int(_lib.lib().bsa_worklist_workspace_size(
            ctypes.byref(s), route.k_max))), dtype=torch.uint8, device=dev)
        self.out = torch.empty(num_heads, sh.total_tokens, head_dim, dtype=dtype, device=dev)
        self.lse = torch.empty(num_heads, sh.total_tokens, dtype=torch.float32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    # kernels each stage launches on the BF16 path (bsa_block_summaries 1;
    # bsa_route 3: summary split, tensor-core scores, selection;
    # bsa_build_worklist 3; bsa_attention_fwd 1)
    LAUNCHES = {"summaries": 1, "route": 3, "worklist": 3, "attention": 1}

    def summaries(self, k):
        block_summaries(k, self.shape, out=self.C)

    def select(self, q):
        route(q, self.C, self.shape, self.params, J=self.J, counts=self.counts,
              scores=self.scores, ws=self.route_ws, dev_status=self.status)

    def worklist(self):
        build_worklist(self.J, self.counts, self.shape, self.params.k_max, self.status,
                       wl=self.wl, ws=self.wl_ws)

    def route(self, q, k):
        self.summaries(k)
        self.select(q)
        self.worklist()

    def attend(self, q, k, v, scale: float = 0.0):
        return attention_fwd(q, k, v, self.wl, self.shape, self.status, scale, out=self.out,
                             lse=self.lse)

    def run(self, q, k, v, scale: float = 0.0):
        self.route(q, k)
        return self.attend(q, k, v, scale)

    def coverage(self, q, k, v, scale: float = 0.0):
        """Coverage C_i of eq.(10) of the current route: the lse of the routed
        attention against the lse of the same kernel over every causal block.
        Returns (C [H, T], O_dense, lse_dense); run() must have been called."""
        if getattr(self, "_dense_wl", None) is None:
            self._dense_wl = causal_worklist(self.shape, q.device)
        Od, ld = attention_fwd(q, k, v, self._dense_wl, self.shape, self.status, scale)
        return coverage(self.lse, ld, self.shape), Od, ld


class HostPrefill:
    """Prefill of batches that live in host memory, with the copies overlapped.

    Two device slots (inputs and a PrefillPlan each) alternate between batches:
    while batch s computes, the upload of batch s + 1 runs on one copy stream and
    the download of batch s - 1's output on another.  Inside a batch the inputs
    are uploaded in the order the path needs them (K for the summaries, then Q
    for the router, then V for the attention), so the first kernels start before
    the whole batch has arrived.  submit() only enqueues; the output host buffer
    is complete once synchronize() (or the returned event) has passed.  Host
    buffers should be pinned for the copies to run asynchronously.
    """

    def __init__(self, cu_seqlens_host, num_heads: int, num_kv_heads: int, head_dim: int,
                 block: int, route: RouteParams, dtype=torch.bfloat16, device="cuda"):
        self.device = torch.device(device)
        self.plans = [PrefillPlan(cu_seqlens_host, num_heads, num_kv_heads, head_dim, block, route,
                                  dtype, device) for _ in range(2)]
        T = self.plans[0].shape.total_tokens
        self.q = [torch.empty(num_heads, T, head_dim, dtype=dtype, device=device) for _ in range(2)]
        self.k = [torch.empty(num_kv_heads, T, head_dim, dtype=dtype, device=device)
                  for _ in range(2)]
        self.v = [torch.empty(num_kv_heads, T, head_dim, dtype=dtype, device=device)
                  for _ in range(2)]
        self.h2d = torch.cuda.Stream(device=self.device)
        self.d2h = torch.cuda.Stream(device=self.device)
        self.compute = torch.cuda.current_stream(self.device)
        self._inputs_free = [None, None]   # compute of the slot's last batch done
        self._output_free = [None, None]   # download of the slot's last output done
        self._n = 0

    @property
    def status(self):
        return self.plans[0].status, self.plans[1].status

    def submit(self, q_host, k_host, v_host, out_host) -> torch.cuda.Event:
        """Enqueue one batch: upload q / k / v (host [H, T, d] / [H_kv, T, d]), run
        the path, download O into out_host.  Returns the event of the download."""
        s = self._n % 2
        self._n += 1
        plan = self.plans[s]
        ev = lambda: torch.cuda.Event()  # noqa: E731
        k_in, q_in, v_in = ev(), ev(), ev()
        with torch.cuda.stream(self.h2d):
            if self._inputs_free[s] is not None:
                self.h2d.wait_event(self._inputs_free[s])
            self.k[s].copy_(k_host, non_blocking=True)
            k_in.record(self.h2d)
            self.q[s].copy_(q_host, non_blocking=True)
            q_in.record(self.h2d)
            self.v[s].copy_(v_host, non_blocking=True)
            v_in.record(self.h2d)
        with torch.cuda.stream(self.compute):
            self.compute.wait_event(k_in)
            plan.summaries(self.k[s])
            self.compute.wait_event(q_in)
            plan.select(self.q[s])
            plan.worklist()
            self.compute.wait_event(v_in)
            if self._output_free[s] is not None:
                self.compute.wait_event(self._output_free[s])
            plan.attend(self.q[s], self.k[s], self.v[s])
            done = ev()
            done.record(self.compute)
            self._inputs_free[s] = done
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(done)
            out_host.copy_(plan.out, non_blocking=True)
            out_done = ev()
            out_done.record(self.d2h)
            self._output_free[s] = out_done
        return out_done

    def synchronize(self):
        for st in (self.h2d, self.compute, self.d2h):
            st.synchronize()


# ---------------------------------------------------------------- chunked prefill


@dataclass
class PagedKVCache:
    """Paged KV cache with its page summaries (bsa_kv_cache_t): k_cache, v_cache
    [P, H_kv, 64, d] bf16; page_summ [P, H_kv, d] fp32 page means and, optionally,
    page_sum the running sums that streaming decode appends continue from;
    block_table [B, max_pages] int32 physical page of each logical block."""
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    page_summ: torch.Tensor
    block_table: torch.Tensor
    page_sum: torch.Tensor | None = None

    PAGE = 64

    @staticmethod
    def allocate(num_phys_pages: int, num_kv_heads: int, head_dim: int, block_table,
                 device="cuda", with_sums: bool = True) -> "PagedKVCache":
        P, Hk, d = num_phys_pages, num_kv_heads, head_dim
        z = lambda *sh, dt: torch.zeros(*sh, dtype=dt, device=device)  # noqa: E731
        return PagedKVCache(z(P, Hk, 64, d, dt=torch.bfloat16), z(P, Hk, 64, d, dt=torch.bfloat16),
                            z(P, Hk, d, dt=torch.float32),
                            torch.as_tensor(block_table, dtype=torch.int32, device=device),
                            z(P, Hk, d, dt=torch.float32) if with_sums else None)

    def c(self, chunk: "Chunk") -> _lib.KVCache:
        return _lib.KVCache(self.k_cache.data_ptr(), self.v_cache.data_ptr(),
                            self.page_summ.data_ptr(),
                            None if self.page_sum is None else self.page_sum.data_ptr(),
                            self.block_table.data_ptr(), chunk.prefix_lens.data_ptr(),
                            self.block_table.shape[1], self.k_cache.shape[0],
                            chunk.max_context_blocks)


@dataclass
class Chunk:
    """One chunk of a chunked prefill: `shape` packs the tokens each sequence adds
    (block 64, bf16), `prefix_lens` [B] int32 the tokens already cached (multiples
    of 64), max_context_blocks >= every ceil((prefix + n) / 64)."""
    shape: PrefillShape
    prefix_lens: torch.Tensor
    max_context_blocks: int

    @staticmethod
    def make(prefix_lens_host, chunk_lens_host, num_heads: int, num_kv_heads: int,
             head_dim: int, device="cuda", max_context_blocks: int | None = None) -> "Chunk":
        pre = np.asarray(prefix_lens_host, dtype=np.int64)
        lens = np.asarray(chunk_lens_host, dtype=np.int64)
        cu = np.zeros(len(lens) + 1, dtype=np.int64)
        cu[1:] = np.cumsum(lens)
        shape = PrefillShape.make(cu, num_heads, num_kv_heads, head_dim, 64, torch.bfloat16,
                                  device)
        if max_context_blocks is None:
            max_context_blocks = int(((pre + lens + 63) // 64).max())
        return Chunk(shape, torch.as_tensor(pre.astype(np.int32), device=device),
                     max_context_blocks)


def chunk_append(k, v, chunk: Chunk, cache: PagedKVCache, dev_status):
    """Write the chunk's keys / values (k, v [H_kv, T, d]) into their pages and
    summarise those pages (bsa_chunk_append)."""
    s, c = chunk.shape.c(), cache.c(chunk)
    check("bsa_chunk_append", _lib.lib().bsa_chunk_append(
        ctypes.byref(s), ctypes.byref(c), _p(k), _p(v), _p(dev_status), _stream()))


def route_chunk_workspace_bytes(chunk: Chunk, cache: PagedKVCache, params: RouteParams) -> int:
    s, c, p = chunk.shape.c(), cache.c(chunk), params.c()
    return int(_lib.lib().bsa_route_chunk_workspace_size(ctypes.byref(s), ctypes.byref(c),
                                                         ctypes.byref(p)))


def route_chunk(q, chunk: Chunk, cache: PagedKVCache, params: RouteParams, dev_status, J=None,
                counts=None, scores=None, ws=None):
    """J [B, H_kv, N_q, k_max] logical block ids and counts of the chunk's query
    blocks, routed against the cached page summaries (bsa_route_chunk)."""
    sh, dev = chunk.shape, q.device
    if J is None:
        J = torch.empty(sh.num_seqs, sh.num_kv_heads, sh.max_blocks, params.k_max,
                        dtype=torch.int32, device=dev)
    if counts is None:
        counts = torch.empty(sh.num_seqs, sh.num_kv_heads, sh.max_blocks, dtype=torch.int32,
                             device=dev)
    if ws is None:
        ws = torch.empty(max(256, route_chunk_workspace_bytes(chunk, cache, params)),
                         dtype=torch.uint8, device=dev)
    s, c, p = sh.c(), cache.c(chunk), params.c(dev)
    check("bsa_route_chunk", _lib.lib().bsa_route_chunk(
        ctypes.byref(s), ctypes.byref(c), ctypes.byref(p), _p(q), _p(J), _p(counts), _p(scores),
        _p(dev_status), _p(ws), ws.numel(), _stream()))
    return J, counts


def build_worklist_chunk(J, counts, chunk: Chunk, cache: PagedKVCache, k_max: int, dev_status,
                         wl: Worklist | None = None, ws=None) -> Worklist:
    dev, rows = J.device, chunk.shape.num_rows
    if wl is None:
        wl = Worklist(torch.empty(rows + 1, dtype=torch.int32, device=dev),
                      torch.empty(max(1, rows * k_max), dtype=torch.int32, device=dev),
                      torch.empty(max(1, rows), dtype=torch.int32, device=dev),
                      torch.empty(NUM_BUCKETS + 1, dtype=torch.int32, device=dev))
    s, c = chunk.shape.c(), cache.c(chunk)
    if ws is None:
        n = int(_lib.lib().bsa_worklist_workspace_size(ctypes.byref(s), k_max))
        ws = torch.empty(max(256, n), dtype=torch.uint8, device=dev)
    check("bsa_build_worklist_chunk", _lib.lib().bsa_build_worklist_chunk(
        ctypes.byref(s), ctypes.byref(c), k_max, _p(J), _p(counts), _p(wl.row_ptr),
        _p(wl.col_idx), _p(wl.work), _p(wl.bucket_off), _p(dev_status), _p(ws), ws.numel(),
        _stream()))
    return wl


def attention_chunk(q, wl: Worklist, chunk: Chunk, cache: PagedKVCache, dev_status,
                    scale: float = 0.0, out=None, lse=None, want_lse: bool = True):
    """O [H, T, d] bf16 and lse [H, T] fp32 of the chunk's queries over the
    selected cache pages (bsa_attention_chunk)."""
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(chunk.shape.num_heads, chunk.shape.total_tokens, dtype=torch.float32,
                          device=q.device)
    s, c = chunk.shape.c(), cache.c(chunk)
    check("bsa_attention_chunk", _lib.lib().bsa_attention_chunk(
        ctypes.byref(s), ctypes.byref(c), _p(q), _p(wl.row_ptr), _p(wl.col_idx), _p(wl.work),
        _p(wl.bucket_off), float(scale), _p(out), _p(lse), _p(dev_status), _stream()))
    return out, lse


class ChunkPlan:
    """Buffers of one chunk shape, allocated once; run() enqueues the four calls of
    a chunked-prefill step (append, route, worklist, attention) on the current
    stream."""

    LAUNCHES = {"append": 1, "route": 3, "worklist": 3, "attention": 1}

    def __init__(self, chunk: Chunk, cache: PagedKVCache, route: RouteParams, device="cuda"):
        self.chunk, self.cache, self.params = chunk, cache, route
        sh, dev = chunk.shape, device
        self.J = torch.empty(sh.num_seqs, sh.num_kv_heads, sh.max_blocks, route.k_max,
                             dtype=torch.int32, device=dev)
        self.counts = torch.empty(sh.num_seqs, sh.num_kv_heads, sh.max_blocks, dtype=torch.int32,
                                  device=dev)
        self.route_ws = torch.empty(max(256, route_chunk_workspace_bytes(chunk, cache, route)),
                                    dtype=torch.uint8, device=dev)
        rows = sh.num_rows
        self.wl = Worklist(torch.empty(rows + 1, dtype=torch.int32, device=dev),
                           torch.empty(max(1, rows * route.k_max), dtype=torch.int32, device=dev),
                           torch.empty(max(1, rows), dtype=torch.int32, device=dev),
                           torch.empty(NUM_BUCKETS + 1, dtype=torch.int32, device=dev))
        s = sh.c()
        self.wl_ws = torch.empty(max(256, int(_lib.lib().bsa_worklist_workspace_size(
            ctypes.byref(s), route.k_max))), dtype=torch.uint8, device=dev)
        self.out = torch.empty(sh.num_heads, sh.total_tokens, sh.head_dim, dtype=torch.bfloat16,
                               device=dev)
        self.lse = torch.empty(sh.num_heads, sh.total_tokens, dtype=torch.float32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def run(self, q, k, v, scale: float = 0.0):
        ch, ca = self.chunk, self.cache
        chunk_append(k, v, ch, ca, self.status)
        route_chunk(q, ch, ca, self.params, self.status, J=self.J, counts=self.counts,
                    ws=self.route_ws)
        build_worklist_chunk(self.J, self.counts, ch, ca, self.params.k_max, self.status,
                             wl=self.wl, ws=self.wl_ws)
        return attention_chunk(q, self.wl, ch, ca, self.status, scale, out=self.out, lse=self.lse)


# ---------------------------------------------------------------- decode


def _dshape(q, k_cache, block_table, top_k: int) -> _lib.DecodeShape:
    R, H, d = q.shape
    P, Hk, page, _ = k_cache.shape
    return _lib.DecodeShape(R, H, Hk, d, page, block_table.shape[1], P, top_k)


def page_summaries(k_cache, block_table, context_lens, out=None):
    """[P, H_kv, d] fp32 mean key of every referenced page (bsa_page_summaries)."""
    P, Hk, page, d = k_cache.shape
    if out is None:
        out = torch.zeros(P, Hk, d, dtype=torch.float32, device=k_cache.device)
    s = _lib.DecodeShape(block_table.shape[0], Hk, Hk, d, page, block_table.shape[1], P, 1)
    check("bsa_page_summaries", _lib.lib().bsa_page_summaries(
        ctypes.byref(s), _p(k_cache), _p(block_table), _p(context_lens), _p(out), _stream()))
    return out


def page_summaries_append(k_cache, block_table, context_lens, page_sum, page_summ):
    """eq.(11) streaming update for the key each request just appended
    (bsa_page_summaries_append): page_sum is the running-sum state, page_summ the
    means; context_lens are the counts after the append (0 skips a request)."""
    P, Hk, page, d = k_cache.shape
    s = _lib.DecodeShape(block_table.shape[0], Hk, Hk, d, page, block_table.shape[1], P, 1)
    check("bsa_page_summaries_append", _lib.lib().bsa_page_summaries_append(
        ctypes.byref(s), _p(k_cache), _p(block_table), _p(context_lens), _p(page_sum),
        _p(page_summ), _stream()))
    return page_summ


class DecodePlan:
    """Buffers for one decode batch shape; run() enqueues bsa_decode_paged."""

    def __init__(self, num_reqs, num_heads, num_kv_heads, head_dim, page_size, max_pages,
                 num_phys_pages, top_k, device="cuda"):
        self.cshape = _lib.DecodeShape(num_reqs, num_heads, num_kv_heads, head_dim, page_size,
                                       max_pages, num_phys_pages, top_k)
        self.top_k = top_k
        n = int(_lib.lib().bsa_decode_workspace_size(ctypes.byref(self.cshape)))
        self.ws = torch.empty(max(256, n), dtype=torch.uint8, device=device)
        self.out = torch.empty(num_reqs, num_heads, head_dim, dtype=torch.bfloat16, device=device)
        self.lse = torch.empty(num_reqs, num_heads, dtype=torch.float32, device=device)
        self.sel = torch.empty(num_reqs, num_kv_heads, top_k + 1, dtype=torch.int32, device=device)
        self.sel_counts = torch.empty(num_reqs, num_kv_heads, dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def run(self, q, k_cache, v_cache, page_summ, block_table, context_lens, scale: float = 0.0):
        check("bsa_decode_paged", _lib.lib().bsa_decode_paged(
            ctypes.byref(self.cshape), _p(q), _p(k_cache), _p(v_cache), _p(page_summ),
            _p(block_table), _p(context_lens), float(scale), _p(self.out), _p(self.lse),
            _p(self.sel), _p(self.sel_counts), _p(self.status), _p(self.ws), self.ws.numel(),
            _stream()))
        return self.out, self.lse, self.sel, self.sel_counts


def decode_paged(q, k_cache, v_cache, page_summ, block_table, context_lens, top_k: int = 32,
                 scale: float = 0.0):
    R, H, d = q.shape
    P, Hk, page, _ = k_cache.shape
    plan = DecodePlan(R, H, Hk, d, page, block_table.shape[1], P, top_k, device=q.device)
    return plan.run(q, k_cache, v_cache, page_summ, block_table, context_lens, scale)
