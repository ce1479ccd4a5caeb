"""Seeded synthetic inputs shared by the GPU path's tests and benches and by the oracle.

This module only draws numbers and lays them out; it holds none of the
method's arithmetic (no summaries, scores, selection or softmax).  Every array
is drawn on the CPU with numpy's PCG64 so the GPU path and the oracle see the
same bits.  BF16 tensors are carried as uint16 bit patterns (round to nearest
even from float32).

Value recipes (the pages describe the structure only in words, so the exact
recipe is a reading):
  iid          Q, K, V i.i.d. N(0, 1).
  planted      per KV head, 2% of the key blocks (drawn from 1 .. N-2) are each
               paired with a later query block u; every key of block j gets +3 w,
               w the unit-normalised mean of that group's queries in block u.
  window_bias  on 20% of the KV heads (and their query heads), dims 0-1 of Q and
               K get A (cos(theta beta), sin(theta beta)), beta the token's
               sequence-relative block index, A = 2, theta = pi / 32, so q.k
               gains A^2 cos(theta (u - j)), largest for recent blocks.
  lowrank      K[h, t] += U_h z_{h, block(t)}, U_h in R^{d x 8} with N(0, 1/8)
               entries and one z ~ N(0, I_8) per (head, block): keys of a block
               share a direction, so blocks cluster.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

from .workloads import DecodeWorkload, PrefillWorkload

_CHUNK = 1 << 22


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(32, os.cpu_count() or 1))


def normal_f32(shape, seed: int, tag: int) -> np.ndarray:
    """N(0, 1) float32 of `shape`, drawn in fixed 4M-element chunks from spawned
    PCG64 streams, so the result does not depend on the thread count."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    nchunks = max(1, (n + _CHUNK - 1) // _CHUNK)
    children = np.random.SeedSequence([seed, tag]).spawn(nchunks)

    def work(c: int) -> None:
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(children[c]))
        out[lo:hi] = g.standard_normal(hi - lo, dtype=np.float32)

    if nchunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out.reshape(shape)


def normal_bf16(shape, seed: int, tag: int) -> np.ndarray:
    """N(0, 1) rounded to bf16 (uint16 bits); chunked and threaded like normal_f32."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    nchunks = max(1, (n + _CHUNK - 1) // _CHUNK)
    children = np.random.SeedSequence([seed, tag]).spawn(nchunks)

    def work(c: int) -> None:
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(children[c]))
        out[lo:hi] = f32_to_bf16_bits(g.standard_normal(hi - lo, dtype=np.float32))

    if nchunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out.reshape(shape)


@dataclass
class PrefillInputs:
    q: np.ndarray                 # [H, T, d]   uint16 (bf16 bits) or float32
    k: np.ndarray                 # [H_kv, T, d]
    v: np.ndarray                 # [H_kv, T, d]
    cu_seqlens: np.ndarray        # [B + 1] int32
    block: int
    dtype: str                    # "bf16" or "fp32"
    planted: list = field(default_factory=list)   # (h_kv, key block j, query block u)

    @property
    def lengths(self) -> np.ndarray:
        return np.diff(self.cu_seqlens)

    def as_f64(self, name: str) -> np.ndarray:
        a = getattr(self, name)
        if self.dtype == "bf16":
            return bf16_bits_to_f32(a).astype(np.float64)
        return a.astype(np.float64)


def draw_lengths(num_seqs: int, lo: int, hi: int, seed: int) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7])))
    return g.integers(lo, hi + 1, size=num_seqs).astype(np.int64)


def gen_prefill(lengths, num_heads: int, num_kv_heads: int, head_dim: int, block: int,
                seed: int, structure: str = "iid", dtype: str = "bf16") -> PrefillInputs:
    """Packed head-major prefill inputs for sequences of the given lengths."""
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    H, Hk, d, b = num_heads, num_kv_heads, head_dim, block
    G = H // Hk
    planted = []

    if dtype == "fp32":
        q = normal_f32((H, T, d), seed, 1)
        k = normal_f32((Hk, T, d), seed, 2)
        v = normal_f32((Hk, T, d), seed, 3)
    else:
        q = normal_bf16((H, T, d), seed, 1)
        v = normal_bf16((Hk, T, d), seed, 3)
        k = None

    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 11])))

    if structure in ("planted", "lowrank"):
        kf = normal_f32((Hk, T, d), seed, 2) if k is None else k
        qf = bf16_bits_to_f32(q) if dtype == "bf16" else q
        for i in range(len(lengths)):
            s0, n = int(cu[i]), int(lengths[i])
            nb = (n + b - 1) // b
            for h in range(Hk):
                if structure == "planted":
                    npl = int(math.floor(0.02 * nb))
                    if nb < 3 or npl == 0:
                        continue
                    js = g.choice(np.arange(1, nb - 1), size=min(npl, nb - 2), replace=False)
                    for j in sorted(int(x) for x in js):
                        u = int(g.integers(j + 1, nb))
                        qb = qf[h * G:(h + 1) * G, s0 + u * b: s0 + min(n, (u + 1) * b), :]
                        w = qb.reshape(-1, d).mean(axis=0)
                        w = w / max(float(np.linalg.norm(w)), 1e-30)
                        kf[h, s0 + j * b: s0 + min(n, (j + 1) * b), :] += np.float32(3.0) * w
                        planted.append((h, j, u))
                else:
                    U = g.standard_normal((d, 8)).astype(np.float32) * np.float32(1.0 / math.sqrt(8.0))
                    Z = g.standard_normal((nb, 8)).astype(np.float32)
                    comp = Z @ U.T                                   # [nb, d]
                    rep = np.repeat(comp, b, axis=0)[:n]             # token t gets its block's row
                    kf[h, s0:s0 + n, :] += rep
        k = kf if dtype == "fp32" else f32_to_bf16_bits(kf)
    elif k is None:
        k = normal_bf16((Hk, T, d), seed, 2)

    if structure == "window_bias":
        nbias = max(1, int(round(0.2 * Hk)))
        heads = sorted(int(x) for x in g.choice(Hk, size=nbias, replace=False))
        A, theta = 2.0, math.pi / 32.0
        for i in range(len(lengths)):
            s0, n = int(cu[i]), int(lengths[i])
            beta = np.arange(n) // b
            code = np.stack([A * np.cos(theta * beta), A * np.sin(theta * beta)], axis=1).astype(np.float32)
            for h in heads:
                for arr, hs in ((k, [h]), (q, list(range(h * G, (h + 1) * G)))):
                    for hh in hs:
                        if dtype == "bf16":
                            cur = bf16_bits_to_f32(arr[hh, s0:s0 + n, 0:2])
                            arr[hh, s0:s0 + n, 0:2] = f32_to_bf16_bits(cur + code)
                        else:
                            arr[hh, s0:s0 + n, 0:2] += code
    elif structure not in ("iid", "planted", "lowrank"):
        raise ValueError(f"unknown structure {structure!r}")

    return PrefillInputs(q=q, k=k, v=v, cu_seqlens=cu.astype(np.int32), block=b,
                         dtype=dtype, planted=planted)


def make_prefill(w: PrefillWorkload, dtype: str = "bf16") -> PrefillInputs:
    if w.seqlen is not None:
        lengths = [w.seqlen] * w.num_seqs
    else:
        lengths = draw_lengths(w.num_seqs, w.seqlen_range[0], w.seqlen_range[1], w.seed)
    return gen_prefill(lengths, w.num_heads, w.num_kv_heads, w.head_dim, w.block,
                       w.seed, w.structure, dtype)


@dataclass
class DecodeInputs:
    q: np.ndarray            # [R, H, d] uint16 bf16 bits
    k_cache: np.ndarray      # [P, H_kv, page, d] uint16
    v_cache: np.ndarray      # [P, H_kv, page, d] uint16
    block_table: np.ndarray  # [R, max_pages] int32, -1 past each request's pages
    context_lens: np.ndarray  # [R] int32
    page_size: int


def gen_decode(context_lens, num_heads: int, num_kv_heads: int, head_dim: int,
               page_size: int, seed: int, max_pages: int | None = None) -> DecodeInputs:
    """A paged BF16 KV cache whose physical pages are a random permutation of
    the requests' logical pages, plus one query token per request."""
    lens = np.asarray(context_lens, dtype=np.int64)
    R = len(lens)
    npages = (lens + page_size - 1) // page_size
    P = int(npages.sum())
    if max_pages is None:
        max_pages = int(npages.max())
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 13])))
    perm = g.permutation(P).astype(np.int32)
    bt = np.full((R, max_pages), -1, dtype=np.int32)
    off = 0
    for r in range(R):
        bt[r, :npages[r]] = perm[off:off + npages[r]]
        off += int(npages[r])
    q = normal_bf16((R, num_heads, head_dim), seed, 1)
    kc = normal_bf16((P, num_kv_heads, page_size, head_dim), seed, 2)
    vc = normal_bf16((P, num_kv_heads, page_size, head_dim), seed, 3)
    return DecodeInputs(q=q, k_cache=kc, v_cache=vc, block_table=bt,
                        context_lens=lens.astype(np.int32), page_size=page_size)


def make_decode(w: DecodeWorkload, num_reqs: int | None = None) -> DecodeInputs:
    R = w.num_reqs if num_reqs is None else num_reqs
    lens = draw_lengths(w.num_reqs, w.len_range[0], w.len_range[1], w.seed)[:R]
    max_pages = (w.len_range[1] + w.page_size - 1) // w.page_size
    return gen_decode(lens, w.num_heads, w.num_kv_heads, w.head_dim, w.page_size,
                      w.seed, max_pages=max_pages)
