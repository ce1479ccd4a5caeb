"""Algorithmic work counters used to turn measured times into throughput.

Conventions ("2.1 · 粗粒度选择" §2.2, last paragraph of the worked budget: say
whether effective token pairs, physical tile FLOPs or profiler counts are used):

  attention FLOPs  PHYSICAL TILE FLOPs: every selected block of a row is one
                   full b x b tile for each of the G query heads of the row, and
                   costs 2 b^2 d for QK^T plus 2 b^2 d for PV (eq.(9) counts the
                   same physical pairs).  Diagonal and tail tiles count full.
  effective pairs  (query, key) pairs the causal / tail mask leaves, reported
                   beside the physical count.
  router FLOPs     2 d per (query row, scored history block), max-pooling free.
  decode bytes     summaries of the scored pages + the valid K and V tokens of
                   the selected pages + q, o, block-table entries.
"""
from __future__ import annotations

import numpy as np


def attention_tile_flops(counts: np.ndarray, G: int, b: int, d: int) -> float:
    """counts [B, H_kv, N_q] (rows past a sequence's end hold 0)."""
    tiles = int(np.asarray(counts, dtype=np.int64).sum())
    return float(tiles) * G * 4.0 * b * b * d


def attention_bytes(H: int, Hk: int, T: int, d: int, elem: int = 2) -> float:
    """Compulsory HBM bytes of one attention pass: Q, K, V read once, O written
    once, lse written once (the floor; re-reads of K/V tiles hit L2)."""
    return float(elem) * d * T * (2 * H + 2 * Hk) + 4.0 * H * T


def effective_pairs(J: np.ndarray, counts: np.ndarray, cu_seqlens, b: int, G: int) -> float:
    """Causally visible (query, key) pairs inside the selected tiles, all query heads."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    total = 0
    for i in range(len(cu) - 1):
        n = int(cu[i + 1] - cu[i])
        nb = (n + b - 1) // b
        for r in range(nb):
            nq = min(n, (r + 1) * b) - r * b
            c = counts[i, :, r]
            ids = J[i, :, r]
            for h in range(counts.shape[1]):
                for j in ids[h, :c[h]]:
                    if j < r:
                        total += nq * b
                    else:  # diagonal: token t sees keys r*b .. t
                        total += nq * (nq + 1) // 2
    return float(total) * G


def router_flops(cu_seqlens, b: int, H: int, d: int) -> float:
    """2 d per (valid query row of every head, history block j < r)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    total = 0
    for i in range(len(cu) - 1):
        n = int(cu[i + 1] - cu[i])
        nb = (n + b - 1) // b
        r = np.arange(nb)
        rows = np.minimum(n, (r + 1) * b) - r * b
        total += int((rows * r).sum())
    return 2.0 * d * H * total


def summaries_bytes(Hk: int, T: int, d: int, n_blocks_total: int, elem: int = 2) -> float:
    return float(elem) * Hk * T * d + 4.0 * Hk * n_blocks_total * d


def decode_bytes(context_lens, sel, sel_counts, num_heads: int, Hk: int, d: int,
                 page: int) -> dict:
    """Algorithmic bytes of one paged decode step."""
    lens = np.asarray(context_lens, dtype=np.int64)
    L = (lens + page - 1) // page
    summ = float(((L - 1) * Hk * d * 4).sum())
    kv = 0
    for rho in range(len(lens)):
        for h in range(Hk):
            for p in sel[rho, h, :sel_counts[rho, h]]:
                kv += min(page, int(lens[rho]) - int(p) * page)
    kv_bytes = float(kv) * d * 2 * 2
    qo = float(len(lens)) * num_heads * d * 2 * 2 + float(len(lens)) * num_heads * 4
    bt = float((L * 4).sum())
    return {"summaries": summ, "kv": kv_bytes, "q_o_lse": qo, "block_table": bt,
            "total": summ + kv_bytes + qo + bt}


def router_bytes(H: int, Hk: int, T: int, d: int, num_seqs: int, max_blocks: int,
                 k_max: int, elem: int = 2) -> float:
    """Compulsory HBM bytes of the router call (scores + selection): Q read once,
    the fp32 summaries read once, J and the counts written once."""
    rows = float(num_seqs) * Hk * max_blocks
    return (float(elem) * H * T * d + 4.0 * rows * d + 4.0 * rows * k_max + 4.0 * rows)
