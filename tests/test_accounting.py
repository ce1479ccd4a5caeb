"""The bench's work counters (dynamic_block_sparse_mean_gb300/accounting.py) against
the worked budget of "2.1 · 粗粒度选择" §2.2 (eq.(9), golden file) and against brute
force over the oracle's explicit masks, so that the TFLOP/s and GB/s the bench
reports rest on checked numerators."""
import json
import os

import numpy as np

import oracle
from dynamic_block_sparse_mean_gb300 import accounting

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_tile_flops_follow_eq9_physical_pairs():
    gold = json.load(open(os.path.join(GOLDEN, "budget_example.json")))
    n, b, N, k = gold["n"], gold["b"], gold["num_blocks"], gold["blocks_per_row"]
    counts = np.full((1, 1, N), k)
    d, G = 128, 1
    # each physical (query, key) pair costs 2 d for QK^T and 2 d for PV
    assert accounting.attention_tile_flops(counts, G, b, d) == gold["eq9_physical_pairs"] * 4 * d
    assert accounting.attention_tile_flops(counts, 4, b, d) == 4 * gold["eq9_physical_pairs"] * 4 * d
    assert n == N * b


def test_effective_pairs_equal_mask_population():
    rng = np.random.default_rng(5)
    b, G, Hk = 16, 2, 2
    cu = np.array([0, 50, 50, 101])                 # ragged, an empty sequence in the middle
    info = oracle.seq_info(cu, b)
    Nq = max(nb for _, _, nb in info)
    k = 3
    J = np.full((3, Hk, Nq, k), -1, dtype=np.int64)
    counts = np.zeros((3, Hk, Nq), dtype=np.int64)
    brute = 0
    for i, (_, n, nb) in enumerate(info):
        for h in range(Hk):
            for r in range(nb):
                ids = sorted(set(rng.choice(r + 1, size=min(k - 1, r + 1), replace=False).tolist())
                             | {r})[:k]
                J[i, h, r, :len(ids)] = ids
                counts[i, h, r] = len(ids)
                mult = oracle.block_multiplicity(ids, nb, r)
                q_lo, q_hi = r * b, min(n, (r + 1) * b)
                brute += int(oracle.key_mask(q_lo, q_hi, mult, b).sum())
    assert accounting.effective_pairs(J, counts, cu, b, G) == brute * G


def test_router_flops_count_every_scored_history_block():
    cu = np.array([0, 130, 194])
    b, H, d = 64, 4, 32
    brute = 0
    for _, n, nb in oracle.seq_info(cu, b):
        for r in range(nb):
            rows = min(n, (r + 1) * b) - r * b
            brute += rows * r                        # every valid query row scores blocks 0..r-1
    assert accounting.router_flops(cu, b, H, d) == 2 * d * H * brute


def test_decode_bytes_by_hand():
    lens = np.array([130, 64])                       # 3 pages (2 scored), 1 page (none scored)
    sel = np.array([[[0, 2, -1]], [[0, -1, -1]]])    # H_kv = 1
    cnt = np.array([[2], [1]])
    H, Hk, d, page = 4, 1, 8, 64
    got = accounting.decode_bytes(lens, sel, cnt, H, Hk, d, page)
    assert got["summaries"] == (2 + 0) * Hk * d * 4
    assert got["kv"] == (64 + 2 + 64) * d * 2 * 2  # page 0 full, page 2 holds 2 keys, page 0 full
    assert got["q_o_lse"] == 2 * H * d * 2 * 2 + 2 * H * 4
    assert got["block_table"] == (3 + 1) * 4
    assert got["total"] == sum(got[k] for k in ("summaries", "kv", "q_o_lse", "block_table"))


def test_attention_bytes_floor():
    H, Hk, T, d = 32, 8, 32768, 128
    # Q and O over H heads, K and V over H_kv heads, bf16; lse fp32
    assert accounting.attention_bytes(H, Hk, T, d) == 2 * d * T * (2 * H + 2 * Hk) + 4 * H * T
    assert accounting.attention_bytes(H, Hk, T, d) == 675282944.0   # the bench's figure
