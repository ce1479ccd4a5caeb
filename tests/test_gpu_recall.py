"""GPU parity of the token-recall measurement (bsa_token_recall) against the float64
oracle: |G_i ∩ N(i)| for the dense top-t teacher G_i and the routed candidate keys
N(i) ("2.1 · 粗粒度选择" §1.1, the recall@k paragraph).

The counts are integers and must equal the oracle's, except where fp32 rounding
can reorder keys at the t-th score: the kernel's score of a key differs from the
exact one by at most d * 2^-24 * sum_i |q_i k_i| (a sum of d exact bf16 products
in fp32), so the count may differ from the oracle's only by the number of keys
whose score interval overlaps that of the t-th key and whose membership in N(i)
differs from it.
"""
import numpy as np
import pytest
import torch

import dynamic_block_sparse_mean_gb300 as bsa
import oracle
from dynamic_block_sparse_mean_gb300 import synth
from parity_utils import oracle_view, shape_of, upload

pytestmark = pytest.mark.gpu


def _allowed_diff(Qv, Kv, cu, b, G, J, cnt, t_top, hq, tok):
    """Number of keys that fp32 rounding may swap across the teacher boundary."""
    i = int(np.searchsorted(cu, tok, side="right") - 1)
    s0 = int(cu[i])
    t = tok - s0
    if t + 1 <= t_top:
        return 0
    q = Qv[hq, tok]
    Ks = Kv[hq // G, s0:s0 + t + 1]
    g = Ks @ q
    err = Ks.shape[1] * 2.0 ** -24 * (np.abs(Ks) @ np.abs(q))
    order = oracle.rank_order(g, np.arange(t + 1))
    kth = order[t_top - 1]
    lo, hi = g[kth] - err[kth], g[kth] + err[kth]
    near = (g + err >= lo) & (g - err <= hi)
    r = t // b
    sel = set(int(x) for x in J[i, hq // G, r, :cnt[i, hq // G, r]]) or {r}
    inside = np.array([s // b in sel for s in range(t + 1)])
    return int(near[inside].sum()) if not inside[near].all() else 0


def _compare(x, H, Hk, J, cnt, t_top, hits, queries):
    Qv, Kv = oracle_view(x, "q"), oracle_view(x, "k")
    want = oracle.token_recall(Qv, Kv, x.cu_seqlens, x.block, H // Hk, J, cnt, t_top, queries)
    cu = np.asarray(x.cu_seqlens, dtype=np.int64)
    Qf, Kf = np.asarray(Qv[:, :, :]), np.asarray(Kv[:, :, :])
    exact = 0
    for (hq, tok), (h_o, g_o) in want.items():
        h_g = int(hits[hq, tok])
        if h_g == h_o:
            exact += 1
            continue
        slack = _allowed_diff(Qf, Kf, cu, x.block, H // Hk, J, cnt, t_top, hq, tok)
        assert abs(h_g - h_o) <= slack, (hq, tok, h_g, h_o, slack)
    return exact / max(1, len(want))


@pytest.mark.parametrize("lengths,H,Hk,d,b,t_top", [
    ([700, 129, 64, 1300], 4, 2, 128, 64, 32),
    ([1000, 300], 8, 2, 128, 128, 64),
    ([640, 33], 4, 4, 64, 64, 16),
])
def test_token_recall_matches_oracle_all_queries(lengths, H, Hk, d, b, t_top):
    x = synth.gen_prefill(lengths, H, Hk, d, b, 23, "iid", "bf16")
    q, k, v = upload(x)
    sh = shape_of(x, H, Hk)
    Jo, co, _, _ = oracle.route(oracle_view(x, "q"), oracle_view(x, "k"), x.cu_seqlens, b,
                                H // Hk, oracle.TOPK, 4, force_sink=True)
    J = torch.as_tensor(Jo.astype(np.int32), device="cuda")
    cnt = torch.as_tensor(co.astype(np.int32), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    hits = bsa.token_recall(q, k, J, cnt, sh, t_top, dev_status=st).cpu().numpy()
    torch.cuda.synchronize()
    bsa.check_status(st)
    T = int(x.cu_seqlens[-1])
    queries = [(hq, tok) for hq in range(H) for tok in range(T)]
    assert _compare(x, H, Hk, Jo, co, t_top, hits, queries) > 0.99


def test_token_recall_listed_tiles_only_and_limits():
    lengths, H, Hk, d, b = [3000, 1700], 8, 2, 128, 64
    x = synth.gen_prefill(lengths, H, Hk, d, b, 29, "iid", "bf16")
    q, k, v = upload(x)
    sh = shape_of(x, H, Hk)
    Qv, Kv = oracle_view(x, "q"), oracle_view(x, "k")
    Jo, co, _, _ = oracle.route(Qv, Kv, x.cu_seqlens, b, H // Hk, oracle.TOPK, 6)
    J = torch.as_tensor(Jo.astype(np.int32), device="cuda")
    cnt = torch.as_tensor(co.astype(np.int32), device="cuda")
    per = bsa.recall_tiles_per_seq(sh)
    assert per == (3000 + 63) // 64
    rng = np.random.default_rng(4)
    tiles = sorted(set(int(t) for t in rng.integers(0, 2 * H * per, size=24)))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    hits = bsa.token_recall(q, k, J, cnt, sh, 64, dev_status=st,
                            tiles=torch.as_tensor(tiles, dtype=torch.int32, device="cuda"))
    hits = hits.cpu().numpy()
    bsa.check_status(st)
    cu = np.asarray(x.cu_seqlens)
    queries = []
    for tile in tiles:
        c, ih = tile % per, tile // per
        hq, i = ih % H, ih // H
        queries += [(hq, int(cu[i]) + t) for t in range(64 * c, min(64 * c + 64, lengths[i]))]
    _compare(x, H, Hk, Jo, co, 64, hits, queries)
    listed = np.zeros_like(hits, dtype=bool)
    for hq, tok in queries:
        listed[hq, tok] = True
    assert (hits[~listed] == -1).all()            # untouched outside the listed tiles
    # density 1: every teacher key is a candidate
    Ja, ca = oracle.causal_all_blocks(x.cu_seqlens, b, Hk)
    hd = bsa.token_recall(q, k, torch.as_tensor(Ja.astype(np.int32), device="cuda"),
                          torch.as_tensor(ca.astype(np.int32), device="cuda"), sh, 64).cpu().numpy()
    pos = np.concatenate([np.arange(n) for n in lengths])
    assert (hd == np.minimum(64, pos + 1)[None, :]).all()
    # a teacher larger than every visible set: hits = the visible keys of the selected blocks
    hb = bsa.token_recall(q, k, J, cnt, sh, 1 << 30).cpu().numpy()
    want = oracle.token_recall(Qv, Kv, x.cu_seqlens, b, H // Hk, Jo, co, 1 << 30,
                               [(hq, tok) for hq in (0, 5) for tok in range(0, 4700, 7)])
    for (hq, tok), (h_o, _) in want.items():
        assert hb[hq, tok] == h_o
    # a tile id outside the batch is reported
    st.zero_()
    bsa.token_recall(q, k, J, cnt, sh, 64, dev_status=st,
                     tiles=torch.as_tensor([2 * H * per], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert int(st.item()) == 16
