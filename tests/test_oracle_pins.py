"""Pins for the float64 oracle: each test checks it against something other than
itself — a library routine, a closed form, brute force, an exhaustive search,
an invariant of the mathematics, or a number printed on the pages."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from dynamic_block_sparse_mean_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _inputs(lengths, H, Hk, d, b, seed, structure="iid"):
    x = synth.gen_prefill(lengths, H, Hk, d, b, seed, structure)
    return x, x.as_f64("q"), x.as_f64("k"), x.as_f64("v")


# ---------------------------------------------------------------- attention


def _sdpa_dense(Q, K, V, cu, G):
    """Dense causal attention per sequence through torch's library routine (float64)."""
    H, T, d = Q.shape
    out = np.zeros_like(Q)
    lse = np.zeros((H, T))
    for i in range(len(cu) - 1):
        s0, s1 = int(cu[i]), int(cu[i + 1])
        q = torch.from_numpy(Q[:, s0:s1])
        k = torch.from_numpy(K[:, s0:s1]).repeat_interleave(G, dim=0)
        v = torch.from_numpy(V[:, s0:s1]).repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True)[0]
        out[:, s0:s1] = o.numpy()
        s = (q @ k.transpose(-1, -2)) / math.sqrt(d)
        mask = torch.ones(s1 - s0, s1 - s0, dtype=torch.bool).tril()
        lse[:, s0:s1] = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=-1).numpy()
    return out, lse


def test_all_causal_blocks_equal_dense_causal_attention():
    x, Q, K, V = _inputs([200, 77, 128], H=4, Hk=2, d=32, b=32, seed=5)
    J, cnt = oracle.causal_all_blocks(x.cu_seqlens, 32, 2)
    O, lse = oracle.attention(Q, K, V, x.cu_seqlens, 32, 2, J, cnt)
    Od, lsed = _sdpa_dense(Q, K, V, x.cu_seqlens, 2)
    assert np.abs(O - Od).max() < 1e-12
    assert np.abs(lse - lsed).max() < 1e-12


def test_tile_order_does_not_change_result():
    x, Q, K, V = _inputs([300], H=2, Hk=1, d=16, b=32, seed=6)
    J, cnt, _, _ = oracle.route(Q, K, x.cu_seqlens, 32, 2, oracle.TOPK, k_max=4, force_sink=True)
    rng = np.random.default_rng(0)
    Js = J.copy()
    for idx in np.ndindex(J.shape[:3]):
        c = cnt[idx]
        Js[idx][:c] = rng.permutation(J[idx][:c])
    O1, l1 = oracle.attention(Q, K, V, x.cu_seqlens, 32, 2, J, cnt)
    O2, l2 = oracle.attention(Q, K, V, x.cu_seqlens, 32, 2, Js, cnt)
    assert np.array_equal(O1, O2) and np.array_equal(l1, l2)


def test_online_softmax_recurrences_match_direct_softmax_in_any_order():
    rng = np.random.default_rng(1)
    S = rng.normal(size=(7, 96)) * 3
    Vv = rng.normal(size=(96, 5))
    e = np.exp(S - S.max(1, keepdims=True))
    direct = (e / e.sum(1, keepdims=True)) @ Vv
    direct_lse = np.log(np.exp(S).sum(1))
    for trial in range(5):
        cols = rng.permutation(96)
        cuts = np.sort(rng.choice(np.arange(1, 96), size=4, replace=False))
        parts = np.split(cols, cuts)
        O, lse = oracle.online_softmax_merge([S[:, p] for p in parts], [Vv[p] for p in parts])
        assert np.abs(O - direct).max() < 1e-13
        assert np.abs(lse - direct_lse).max() < 1e-12


def test_duplicate_block_changes_result_so_dedup_is_required():
    x, Q, K, V = _inputs([256], H=1, Hk=1, d=16, b=32, seed=7)
    J, cnt, _, _ = oracle.route(Q, K, x.cu_seqlens, 32, 1, oracle.TOPK, k_max=3)
    r = 6
    ids = list(J[0, 0, r, :cnt[0, 0, r]])
    Jd = np.full((1, 1, J.shape[2], 8), -1)
    Jd[0, 0, r, :len(ids) + 1] = sorted(ids + [ids[0]])
    cd = np.zeros_like(cnt)
    cd[0, 0, r] = len(ids) + 1
    rows = [(0, 0, r)]
    Os, _ = oracle.attention(Q, K, V, x.cu_seqlens, 32, 1, Jd, cd, rows=rows)
    Om, _ = oracle.attention(Q, K, V, x.cu_seqlens, 32, 1, Jd, cd, rows=rows, multiset=True)
    Oref, _ = oracle.attention(Q, K, V, x.cu_seqlens, 32, 1, J, cnt, rows=rows)
    sl = slice(r * 32, (r + 1) * 32)
    assert np.array_equal(Os[0, sl], Oref[0, sl])           # set semantics ignore the repeat
    assert np.abs(Om[0, sl] - Os[0, sl]).max() > 2e-2        # counting it twice moves O


def test_empty_row_falls_back_to_diagonal():
    x, Q, K, V = _inputs([192], H=2, Hk=2, d=8, b=64, seed=8)
    J = np.full((1, 2, 3, 2), -1)
    cnt = np.zeros((1, 2, 3), dtype=np.int64)
    O0, l0 = oracle.attention(Q, K, V, x.cu_seqlens, 64, 1, J, cnt)
    for r in range(3):
        J[0, :, r, 0] = r
    cnt[:] = 1
    O1, l1 = oracle.attention(Q, K, V, x.cu_seqlens, 64, 1, J, cnt)
    assert np.array_equal(O0, O1) and np.array_equal(l0, l1)


def test_causal_mask_worked_example_position_130():
    gold = json.load(open(os.path.join(GOLDEN, "budget_example.json")))["causal_example"]
    b, pos = gold["b"], gold["pos"]
    blk, first, last = oracle.causal_visibility(pos, b)
    assert (blk, first, last) == (gold["block"], gold["sees_first"], gold["sees_last"])
    mult = oracle.block_multiplicity([0, 1, 2], 3, 2)
    m = oracle.key_mask(2 * b, 3 * b, mult, b)
    visible = np.nonzero(m[pos - 2 * b])[0]
    assert visible[0] == gold["sees_first"] and visible[-1] == gold["sees_last"]
    assert len(visible) == gold["sees_last"] + 1
    assert np.nonzero(m[pos - 2 * b, 2 * b:])[0][0] + 2 * b == gold["diag_first"]


def test_gqa_query_head_permutation_permutes_outputs():
    x, Q, K, V = _inputs([256], H=8, Hk=2, d=16, b=32, seed=9)
    J, cnt, _, _ = oracle.route(Q, K, x.cu_seqlens, 32, 4, oracle.TOPK, k_max=4)
    perm = np.array([2, 0, 3, 1, 5, 7, 4, 6])        # within each group of 4
    J2, cnt2, _, _ = oracle.route(Q[perm], K, x.cu_seqlens, 32, 4, oracle.TOPK, k_max=4)
    assert np.array_equal(J, J2) and np.array_equal(cnt, cnt2)   # candidates are per KV head
    O, l = oracle.attention(Q, K, V, x.cu_seqlens, 32, 4, J, cnt)
    O2, l2 = oracle.attention(Q[perm], K, V, x.cu_seqlens, 32, 4, J, cnt)
    assert np.abs(O2 - O[perm]).max() < 1e-14 and np.abs(l2 - l[perm]).max() < 1e-14


def test_group_score_is_max_of_single_head_routing():
    """With H = H_kv each head routes alone; the group score is the max of those."""
    x, Q, K, V = _inputs([320, 100], H=6, Hk=2, d=16, b=32, seed=10)
    C = oracle.block_summaries(K, x.cu_seqlens, 32)
    g = oracle.route_scores(Q, C, x.cu_seqlens, 32, 3)
    for h in range(2):
        singles = [oracle.route_scores(Q[hq:hq + 1], C[:, h:h + 1], x.cu_seqlens, 32, 1)[:, 0]
                   for hq in range(3 * h, 3 * h + 3)]
        assert np.array_equal(g[:, h], np.maximum.reduce(singles))


# ---------------------------------------------------------------- brute force


def test_tiny_vectorised_oracle_equals_brute_force():
    b, G = 16, 2
    x, Q, K, V = _inputs([100, 37, 64], H=2, Hk=1, d=8, b=b, seed=11)
    C = oracle.block_summaries(K, x.cu_seqlens, b)
    Cb = oracle.brute_summaries(K.tolist(), x.cu_seqlens, b)
    assert np.abs(C - np.array(Cb)).max() < 1e-13
    g = oracle.route_scores(Q, C, x.cu_seqlens, b, G)
    gb = oracle.brute_scores(Q.tolist(), Cb, x.cu_seqlens, b, G)
    for (i, h, r, j), v in gb.items():
        assert abs(g[i, h, r, j] - v) < 1e-12
    J, cnt, _, _ = oracle.route(Q, K, x.cu_seqlens, b, G, oracle.TOPK, k_max=3, force_sink=True)
    O, lse = oracle.attention(Q, K, V, x.cu_seqlens, b, G, J, cnt)
    Ob, Lb = oracle.brute_attention(Q.tolist(), K.tolist(), V.tolist(), x.cu_seqlens, b, G,
                                    J.tolist(), cnt.tolist())
    for (hq, t), o in Ob.items():
        assert np.abs(O[hq, t] - np.array(o)).max() < 1e-12
        assert abs(lse[hq, t] - Lb[(hq, t)]) < 1e-12
    assert len(Ob) == Q.shape[0] * Q.shape[1]


def test_topk_selection_equals_exhaustive_enumeration():
    rng = np.random.default_rng(12)
    for trial in range(40):
        r = int(rng.integers(1, 9))
        g = np.round(rng.normal(size=r), 1)       # rounding creates exact ties
        for sink in (False, True):
            for k_max in (1, 2, 3, 5):
                sel = oracle.select_row(g, r, oracle.TOPK, k_max, force_sink=sink)
                F = {r} | ({0} if sink else set())
                cand = {j: g[j] for j in range(r) if j not in F}
                k_dyn = max(0, k_max - len(F))
                want = oracle.brute_topk_by_enumeration(cand, k_dyn) if cand and k_dyn else []
                assert sel == sorted(F | set(want))


def test_threshold_rule_hand_worked_row():
    # eq.(7) worked by hand: scores of history blocks 0..5 of row r = 6.
    g = np.array([1.0, 3.0, 2.5, 0.9, 2.0, 2.9])
    # delta 1.0 -> tau 2.0 -> A = {1, 2, 4, 5}; k_r = min(8, max(2, 1 + 4), 7) = 5.
    assert oracle.select_row(g, 6, oracle.THRESHOLD, 8, 2, 1.0) == [1, 2, 4, 5, 6]
    # k_max 3 clamps to the diagonal plus the two best: 1 (3.0) and 5 (2.9).
    assert oracle.select_row(g, 6, oracle.THRESHOLD, 3, 2, 1.0) == [1, 5, 6]
    # k_min 6 lifts the row to six blocks: the five best history blocks plus r.
    assert oracle.select_row(g, 6, oracle.THRESHOLD, 8, 6, 1.0) == [0, 1, 2, 4, 5, 6]
    # the row never exceeds the r + 1 causal blocks.
    assert oracle.select_row(g[:2], 2, oracle.THRESHOLD, 64, 4, 2.0) == [0, 1, 2]
    # row 0 holds only its diagonal.
    assert oracle.select_row(np.array([]), 0, oracle.THRESHOLD, 64, 4, 2.0) == [0]
    # top-k with the sink forced: F = {0, 6}, two dynamic picks 1 and 5.
    assert oracle.select_row(g, 6, oracle.TOPK, 4, force_sink=True) == [0, 1, 5, 6]
    # equal scores go to the lower block index.
    assert oracle.select_row(np.array([1.0, 2.0, 2.0, 2.0]), 4, oracle.TOPK, 3) == [1, 2, 4]


def test_union_routing_hand_worked_row():
    # N_u = L_u ∪ G ∪ I_u for row r = 6 with scores of history blocks 0..5:
    # window 3 -> L = {4, 5, 6}; global list [1] -> F = {1, 4, 5, 6}.
    g = np.array([1.0, 3.0, 2.5, 0.9, 2.0, 2.9])
    # k_max 6 leaves two dynamic picks among {0, 2, 3}: 2 (2.5) and 0 (1.0).  Blocks 1
    # (3.0) and 5 (2.9) score highest but are already kept, so they spend no budget.
    assert oracle.select_row(g, 6, oracle.TOPK, 6, window=3, global_blocks=[1]) == [0, 1, 2, 4, 5, 6]
    assert oracle.select_row(g, 6, oracle.TOPK, 5, window=3, global_blocks=[1]) == [1, 2, 4, 5, 6]
    # a global block inside the window is kept once and frees no extra slot
    assert oracle.select_row(g, 6, oracle.TOPK, 5, window=3, global_blocks=[5]) == \
        oracle.select_row(g, 6, oracle.TOPK, 5, window=3) == [1, 2, 4, 5, 6]
    # blocks after r are invisible (causal) whatever the global list says
    assert oracle.select_row(g[:3], 3, oracle.TOPK, 3, window=1, global_blocks=[2, 7]) == [1, 2, 3]
    # threshold mode, eq.(7) over the non-forced candidates {0, 2, 3}: delta 1.0 ->
    # tau 1.5 -> A = {2}; k_r = min(8, max(2, |F| + 1), |F| + 3) = 5 -> F plus block 2.
    assert oracle.select_row(g, 6, oracle.THRESHOLD, 8, 2, 1.0, window=3, global_blocks=[1]) == \
        [1, 2, 4, 5, 6]


def test_union_selection_properties_and_enumeration():
    rng = np.random.default_rng(21)
    for trial in range(60):
        r = int(rng.integers(0, 10))
        g = np.round(rng.normal(size=r), 1)
        w = int(rng.integers(0, 5))
        glob = sorted(set(int(x) for x in rng.integers(0, 12, size=int(rng.integers(0, 4)))))
        sink = bool(rng.integers(0, 2))
        for k_max in (1, 3, 6, 12):
            sel = oracle.select_row(g, r, oracle.TOPK, k_max, force_sink=sink, window=w,
                                    global_blocks=glob)
            assert sel == sorted(set(sel)) and all(0 <= j <= r for j in sel)
            window = set(range(max(0, r - max(1, w) + 1), r + 1))
            kept = window | {j for j in glob if j <= r} | ({0} if sink else set())
            assert kept <= set(sel)                              # every forced block is kept
            dyn = [j for j in sel if j not in kept]
            assert len(sel) == max(len(kept), min(k_max, r + 1))  # the budget counts forced blocks
            # the dynamic part is the exhaustive best subset of the remaining history
            cand = {j: g[j] for j in range(r) if j not in kept}
            k_dyn = max(0, k_max - len(kept))
            want = oracle.brute_topk_by_enumeration(cand, k_dyn) if cand and k_dyn else []
            assert sorted(dyn) == sorted(want)
        # a window reaching block 0 selects the whole causal row
        assert oracle.select_row(g, r, oracle.TOPK, r + 1, window=r + 1) == list(range(r + 1))


def test_coverage_matches_library_logsumexp_and_limits():
    # eq.(10) C_i = exp(lse over the selected keys - lse over all causal keys), both
    # log-sum-exps from torch; all causal blocks give C = 1; a superset of blocks
    # never covers less.
    x, Q, K, V = _inputs([300, 200], 4, 2, 32, 64, seed=31)
    G, b = 2, 64
    Jo, co, _, _ = oracle.route(Q, K, x.cu_seqlens, b, G, oracle.TOPK, 2)
    C = oracle.coverage(Q, K, x.cu_seqlens, b, G, Jo, co)
    info = oracle.seq_info(x.cu_seqlens, b)
    for (i, h, r) in oracle.all_rows(x.cu_seqlens, b, 2):
        s0, n, nb = info[i]
        sel = [int(v) for v in Jo[i, h, r, :co[i, h, r]]]
        for hq in range(h * G, (h + 1) * G):
            for t in range(r * b, min(n, (r + 1) * b), 17):
                s = torch.from_numpy(K[h, s0:s0 + t + 1] @ Q[hq, s0 + t]) / math.sqrt(32)
                keep = torch.from_numpy(np.isin(np.arange(t + 1) // b, sel))
                want = math.exp(float(torch.logsumexp(s[keep], 0) - torch.logsumexp(s, 0)))
                assert abs(C[hq, s0 + t] - want) < 1e-12
    Ja, ca = oracle.causal_all_blocks(x.cu_seqlens, b, 2)
    assert np.nanmax(np.abs(oracle.coverage(Q, K, x.cu_seqlens, b, G, Ja, ca) - 1.0)) < 1e-12
    Jb, cb, _, _ = oracle.route(Q, K, x.cu_seqlens, b, G, oracle.TOPK, 3)
    Cb = oracle.coverage(Q, K, x.cu_seqlens, b, G, Jb, cb)
    ok = ~np.isnan(C)
    assert (Cb[ok] >= C[ok] - 1e-12).all()


def _recall_hand_case():
    """n = 8, b = 2 (4 blocks), d = 1, H = 4 query heads over H_kv = 2 (G = 2), all
    queries 1.0, so a query's dense scores are the keys themselves."""
    K = np.zeros((2, 8, 1))
    K[0, :, 0] = [0.5, 3.0, 2.0, -1.0, 4.0, 0.1, 2.5, 1.0]
    K[1, :, 0] = [1.0, 1.0, 1.0, 1.0, 0.0, 0.0, 0.0, 0.0]      # ties at the top
    Q = np.ones((4, 8, 1))
    J = np.full((1, 2, 4, 4), -1)
    cnt = np.zeros((1, 2, 4), dtype=np.int64)
    for h in range(2):
        for r in range(4):
            J[0, h, r, 0], cnt[0, h, r] = r, 1                  # diagonal only
    J[0, 0, 3, :2], cnt[0, 0, 3] = [1, 3], 2
    J[0, 1, 3, :2], cnt[0, 1, 3] = [0, 3], 2
    cnt[0, 0, 2] = 0                                            # empty row -> {2}
    return Q, K, J, cnt


def test_token_recall_hand_worked_cases():
    # Top-3 teacher (P2 §1.1 recall paragraph), worked by hand:
    #  KV head 0, token 7: scores 0..7 = K0 -> top-3 {4, 1, 6}; N = blocks {1, 3} =
    #   keys {2, 3, 6, 7} -> 1 hit.  token 6: visible 0..6 (itself included) -> top-3
    #   {4, 1, 6}, 1 hit.  token 5: empty row -> block {2} = keys {4, 5}; top-3
    #   {4, 1, 2} -> 1 hit.  token 1: only 2 visible keys, |G| = 2, both in block 0.
    #  KV head 1 (all visible scores tie at 1.0 up to key 3): token 7 -> top-3 by
    #   lower index {0, 1, 2}; N = blocks {0, 3} = {0, 1, 6, 7} -> 2 hits.  token 3:
    #   N = block {1} = {2, 3}; top-3 {0, 1, 2} -> 1 hit.
    Q, K, J, cnt = _recall_hand_case()
    want = {7: (1, 3), 6: (1, 3), 5: (1, 3), 1: (2, 2)}
    want1 = {7: (2, 3), 3: (1, 3)}
    for hq in range(4):     # query heads 0, 1 share KV head 0; 2, 3 share KV head 1
        table = want if hq < 2 else want1
        got = oracle.token_recall(Q, K, [0, 8], 2, 2, J, cnt, 3, [(hq, t) for t in table])
        assert {t: got[(hq, t)] for t in table} == table


def test_token_recall_limits_and_monotonicity():
    x, Q, K, V = _inputs([300, 200], 4, 2, 32, 64, seed=33)
    G, b, t_top = 2, 64, 16
    rng = np.random.default_rng(5)
    queries = [(int(rng.integers(4)), int(rng.integers(500))) for _ in range(60)]
    # every causal block selected: the teacher is always inside the candidate set
    Ja, ca = oracle.causal_all_blocks(x.cu_seqlens, b, 2)
    for (hq, tok), (hits, gs) in oracle.token_recall(Q, K, x.cu_seqlens, b, G, Ja, ca, t_top,
                                                     queries).items():
        assert hits == gs == min(t_top, tok - (0 if tok < 300 else 300) + 1)
    # a teacher larger than the visible keys is the whole visible set: hits = the
    # query's allowed keys under the explicit mask of the row
    Jo, co, _, _ = oracle.route(Q, K, x.cu_seqlens, b, G, oracle.TOPK, 2)
    big = oracle.token_recall(Q, K, x.cu_seqlens, b, G, Jo, co, 10 ** 6, queries)
    info = oracle.seq_info(x.cu_seqlens, b)
    for (hq, tok), (hits, gs) in big.items():
        i = 0 if tok < 300 else 1
        s0, n, nb = info[i]
        t = tok - s0
        r = t // b
        mult = oracle.block_multiplicity(Jo[i, hq // G, r, :co[i, hq // G, r]], nb, r)
        assert gs == t + 1 and hits == int(oracle.key_mask(t, t + 1, mult, b).sum())
    # more blocks never lose a teacher key
    small = oracle.token_recall(Q, K, x.cu_seqlens, b, G, Jo, co, t_top, queries)
    Jb, cb, _, _ = oracle.route(Q, K, x.cu_seqlens, b, G, oracle.TOPK, 4)
    large = oracle.token_recall(Q, K, x.cu_seqlens, b, G, Jb, cb, t_top, queries)
    assert all(large[q][0] >= small[q][0] for q in small)


def test_backward_matches_central_differences():
    # d/dx sum(O * dO) by central differences of the forward oracle, for random
    # entries of Q, K and V (independent of autograd).
    x, Q, K, V = _inputs([150, 70], 4, 2, 8, 32, seed=61)
    G, b = 2, 32
    Jo, co, _, _ = oracle.route(Q, K, x.cu_seqlens, b, G, oracle.TOPK, 2)
    rng = np.random.default_rng(62)
    dO = rng.normal(size=Q.shape)
    dQ, dK, dV = oracle.attention_backward(Q, K, V, x.cu_seqlens, b, G, Jo, co, dO)

    def loss(Q_, K_, V_):
        O, _ = oracle.attention(Q_, K_, V_, x.cu_seqlens, b, G, Jo, co)
        return float((O * dO).sum())

    eps = 1e-6
    for name, A, grad in (("q", Q, dQ), ("k", K, dK), ("v", V, dV)):
        for _ in range(6):
            idx = tuple(int(rng.integers(n)) for n in A.shape)
            Ap, Am = A.copy(), A.copy()
            Ap[idx] += eps
            Am[idx] -= eps
            args_p = {"q": (Ap, K, V), "k": (Q, Ap, V), "v": (Q, K, Ap)}[name]
            args_m = {"q": (Am, K, V), "k": (Q, Am, V), "v": (Q, K, Am)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_backward_row_and_key_block_equal_the_full_backward():
    # The sampled backward (one router row's dQ; one key block's dK / dV summed over
    # the rows that selected it) against the whole-sequence backward, itself pinned to
    # central differences and to the dense gradients above.  Rows include an empty
    # one (R-7: it holds its diagonal) and ragged tails.
    x, Q, K, V = _inputs([170, 75], 4, 2, 8, 32, seed=65)
    G, b = 2, 32
    Jo, co, _, _ = oracle.route(Q, K, x.cu_seqlens, b, G, oracle.TOPK, 3, force_sink=True)
    co = co.copy()
    co[0, 1, 3] = 0  # an empty row
    dO = np.random.default_rng(66).normal(size=Q.shape)
    dQ, dK, dV = oracle.attention_backward(Q, K, V, x.cu_seqlens, b, G, Jo, co, dO)
    for i, (s0, n, nb) in enumerate(oracle.seq_info(x.cu_seqlens, b)):
        for h in range(2):
            for r in range(nb):
                dq, _, _ = oracle.attention_backward_row(Q, K, V, x.cu_seqlens, b, G, Jo, co, dO,
                                                         (i, h, r))
                q_lo, q_hi = r * b, min(n, (r + 1) * b)
                assert np.abs(dq - dQ[h * G:(h + 1) * G, s0 + q_lo:s0 + q_hi]).max() < 1e-12
            for j in range(nb):
                dk, dv = oracle.attention_backward_key_block(Q, K, V, x.cu_seqlens, b, G, Jo, co,
                                                             dO, i, h, j)
                lo, hi = j * b, min(n, (j + 1) * b)
                assert np.abs(dk - dK[h, s0 + lo:s0 + hi]).max() < 1e-12
                assert np.abs(dv - dV[h, s0 + lo:s0 + hi]).max() < 1e-12


def test_backward_at_density_one_equals_sdpa_gradients():
    x, Q, K, V = _inputs([200, 90], 4, 2, 16, 32, seed=63)
    G, b = 2, 32
    Ja, ca = oracle.causal_all_blocks(x.cu_seqlens, b, 2)
    dO = np.random.default_rng(64).normal(size=Q.shape)
    dQ, dK, dV = oracle.attention_backward(Q, K, V, x.cu_seqlens, b, G, Ja, ca, dO)
    for i in range(len(x.cu_seqlens) - 1):
        s0, s1 = int(x.cu_seqlens[i]), int(x.cu_seqlens[i + 1])
        q = torch.tensor(Q[:, s0:s1], requires_grad=True)
        k = torch.tensor(K[:, s0:s1], requires_grad=True)
        v = torch.tensor(V[:, s0:s1], requires_grad=True)
        o = torch.nn.functional.scaled_dot_product_attention(
            q[None], k.repeat_interleave(G, dim=0)[None], v.repeat_interleave(G, dim=0)[None],
            is_causal=True)[0]
        gq, gk, gv = torch.autograd.grad((o * torch.from_numpy(dO[:, s0:s1])).sum(), (q, k, v))
        assert np.abs(gq.numpy() - dQ[:, s0:s1]).max() < 1e-11
        assert np.abs(gk.numpy() - dK[:, s0:s1]).max() < 1e-11
        assert np.abs(gv.numpy() - dV[:, s0:s1]).max() < 1e-11


# ---------------------------------------------------------------- summaries


def test_summaries_closed_form_with_partial_tail():
    # k_t = a + t c: a block's mean is a + c * (mean position of its valid keys).
    n, b, d = 150, 64, 4
    a, c = np.array([1.0, -2.0, 0.5, 3.0]), np.array([0.25, 0.5, -1.0, 2.0])
    K = (a[None, :] + np.arange(n)[:, None] * c[None, :])[None]
    C = oracle.block_summaries(K, np.array([0, n]), b)
    for j, (lo, hi) in enumerate([(0, 64), (64, 128), (128, 150)]):
        assert np.abs(C[0, 0, j] - (a + c * (lo + hi - 1) / 2.0)).max() < 1e-12


def test_streaming_summary_equals_batch_mean():
    rng = np.random.default_rng(13)
    keys = rng.normal(size=(64, 16))
    st = oracle.streaming_summary(keys)
    for r in (1, 7, 33, 64):
        assert np.abs(st[r - 1] - keys[:r].mean(0)).max() < 1e-14


def test_summary_never_sees_another_sequence():
    x, Q, K, V = _inputs([70, 50], H=1, Hk=1, d=4, b=64, seed=14)
    C = oracle.block_summaries(K, x.cu_seqlens, 64)
    assert np.abs(C[0, 0, 1] - K[0, 64:70].mean(0)).max() < 1e-14
    assert np.abs(C[1, 0, 0] - K[0, 70:120].mean(0)).max() < 1e-14


# ---------------------------------------------------------------- error bound


def test_missed_mass_error_bound():
    x, Q, K, V = _inputs([512], H=2, Hk=1, d=16, b=32, seed=15)
    J, cnt, _, _ = oracle.route(Q, K, x.cu_seqlens, 32, 2, oracle.TOPK, k_max=3)
    O, _ = oracle.attention(Q, K, V, x.cu_seqlens, 32, 2, J, cnt)
    Jd, cd = oracle.causal_all_blocks(x.cu_seqlens, 32, 1)
    Od, _ = oracle.attention(Q, K, V, x.cu_seqlens, 32, 2, Jd, cd)
    Vmax = np.abs(V).max()
    scale = 1.0 / 4.0
    checked = 0
    for t in range(0, 512, 7):
        r = t // 32
        ids = J[0, 0, r, :cnt[0, 0, r]]
        for hq in range(2):
            delta = oracle.missed_mass(Q[hq, t], K[0], t, ids, 32, scale)
            err = np.abs(Od[hq, t] - O[hq, t]).max()
            assert err <= 2 * Vmax * delta + 1e-12
            checked += 1
    assert checked > 100


# ---------------------------------------------------------------- budget numbers


def test_budget_counters_reproduce_worked_example():
    gold = json.load(open(os.path.join(GOLDEN, "budget_example.json")))
    n, b, N = gold["n"], gold["b"], gold["num_blocks"]
    assert (n + b - 1) // b == N
    dense = oracle.dense_causal_pairs(n)
    assert float(f"{dense:.{gold['eq8_significant_digits']}g}") == gold["eq8_dense_pairs_approx"]
    assert oracle.physical_pairs([gold["blocks_per_row"]] * N, b, b) == gold["eq9_physical_pairs"]
    kd, useful = gold["dynamic_blocks"], gold["useful_tokens_per_dynamic_block"]
    assert N * b * kd * useful == gold["logical_dynamic_pairs"]
    assert oracle.physical_pairs([kd] * N, b, b) == gold["physical_dynamic_pairs"]
    assert gold["physical_dynamic_pairs"] // gold["logical_dynamic_pairs"] == gold["waste_factor"]
    # two of the eight blocks overlap between branches: dedup leaves six unique tiles.
    row = [120, 121, 0, 121, 5, 17, 0, 60]
    assert oracle.unique_tiles(row) == gold["unique_blocks_after_dedup"]
    assert oracle.physical_pairs([oracle.unique_tiles(row)] * N, b, b) == gold["dedup_physical_pairs"]
    assert gold["million_tokens"] // 64 == gold["blocks_at_million_b64"]
    assert gold["blocks_at_million_b64"] < 2 ** 15            # still fits a signed 16-bit id
    assert abs(gold["hier_recall_each"] ** 2 - gold["hier_recall_joint"]) < 1e-15


# ---------------------------------------------------------------- decode


def test_decode_with_every_page_selected_is_dense_attention():
    d, page = 16, 8
    x = synth.gen_decode([37, 64, 9], num_heads=4, num_kv_heads=2, head_dim=d, page_size=page, seed=16)
    q = synth.bf16_bits_to_f32(x.q).astype(np.float64)
    kc = synth.bf16_bits_to_f32(x.k_cache).astype(np.float64)
    vc = synth.bf16_bits_to_f32(x.v_cache).astype(np.float64)
    o, lse, sel, cnt = oracle.decode(q, kc, vc, x.block_table, x.context_lens, page, top_k=100)
    for rho, n in enumerate(x.context_lens):
        L = (n + page - 1) // page
        phys = x.block_table[rho, :L]
        for hq in range(4):
            h = hq // 2
            Kl = kc[phys, h].reshape(-1, d)[:n]
            Vl = vc[phys, h].reshape(-1, d)[:n]
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[rho, hq])[None, None], torch.from_numpy(Kl)[None], torch.from_numpy(Vl)[None])[0, 0]
            assert np.abs(o[rho, hq] - ref.numpy()).max() < 1e-12
            s = Kl @ q[rho, hq] / math.sqrt(d)
            assert abs(lse[rho, hq] - float(torch.logsumexp(torch.from_numpy(s), 0))) < 1e-12
        assert cnt[rho, 0] == L


def test_decode_is_invariant_to_physical_page_placement():
    d, page = 8, 4
    x = synth.gen_decode([30, 21], num_heads=2, num_kv_heads=1, head_dim=d, page_size=page, seed=17)
    args = [synth.bf16_bits_to_f32(a).astype(np.float64) for a in (x.q, x.k_cache, x.v_cache)]
    o1, l1, s1, c1 = oracle.decode(*args, x.block_table, x.context_lens, page, top_k=3)
    P = x.k_cache.shape[0]
    perm = np.random.default_rng(3).permutation(P)
    inv = np.argsort(perm)
    kc2, vc2 = args[1][perm], args[2][perm]          # physical page p moves to slot inv[p]
    bt2 = np.where(x.block_table >= 0, inv[np.maximum(x.block_table, 0)], -1)
    o2, l2, s2, c2 = oracle.decode(args[0], kc2, vc2, bt2, x.context_lens, page, top_k=3)
    assert np.array_equal(s1, s2) and np.array_equal(c1, c2)
    assert np.abs(o1 - o2).max() < 1e-14


def test_multiset_mode_equals_attention_over_concatenated_keys():
    """The literal Concat of the unified object: a block listed twice contributes its
    keys twice; checked against SDPA over the explicitly concatenated key list."""
    x, Q, K, V = _inputs([256], H=1, Hk=1, d=16, b=32, seed=18)
    r, ids = 5, [0, 2, 2, 5]
    J = np.full((1, 1, 8, 4), -1)
    J[0, 0, r] = ids
    cnt = np.zeros((1, 1, 8), dtype=np.int64)
    cnt[0, 0, r] = 4
    O, lse = oracle.attention(Q, K, V, x.cu_seqlens, 32, 1, J, cnt, rows=[(0, 0, r)], multiset=True)
    for t in range(r * 32, (r + 1) * 32):
        keys = [s for j in ids for s in range(j * 32, (j + 1) * 32) if s <= t]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(Q[0, t])[None, None], torch.from_numpy(K[0, keys])[None],
            torch.from_numpy(V[0, keys])[None])[0, 0]
        assert np.abs(O[0, t] - ref.numpy()).max() < 1e-12


def test_decode_scores_mean_summaries_and_always_keeps_last_page():
    # d = 2, pages of 2 tokens, context 7: complete pages 0..2, last page 3 holds one key.
    q = np.array([[[1.0, 0.0]]])
    keys = np.array([[1.0, 0], [-0.8, 0],      # page 0: max 1.0 but mean 0.1
                     [0.5, 0], [0.5, 0],       # page 1: mean 0.5 (best by mean)
                     [0.3, 0], [0.3, 0],       # page 2: mean 0.3
                     [100.0, 0], [0.0, 0]])    # page 3: last page, never scored
    kc = keys.reshape(4, 1, 2, 2)
    vc = np.arange(16, dtype=np.float64).reshape(4, 1, 2, 2)
    bt = np.array([[0, 1, 2, 3]], dtype=np.int32)
    o, lse, sel, cnt = oracle.decode(q, kc, vc, bt, np.array([7]), 2, top_k=1)
    assert list(sel[0, 0, :cnt[0, 0]]) == [1, 3]
    o2, _, sel2, cnt2 = oracle.decode(q, kc, vc, bt, np.array([7]), 2, top_k=2)
    assert list(sel2[0, 0, :cnt2[0, 0]]) == [1, 2, 3]
    # keys 2, 3 and 6 (t < 7) enter the softmax; the padding key 7 does not.
    s = np.array([0.5, 0.5, 100.0]) / math.sqrt(2)
    w = np.exp(s - s.max()) / np.exp(s - s.max()).sum()
    ref = w @ vc.reshape(8, 2)[[2, 3, 6]]
    assert np.abs(o[0, 0] - ref).max() < 1e-12


def _paged_from_prompt(K, V, cu, b, seed, garbage=np.nan):
    """Pages of b tokens holding every sequence's whole prompt, placed by a random
    permutation; slots past a sequence's end hold `garbage`."""
    Hk, _, d = K.shape
    lens = np.diff(cu)
    pages = (lens + b - 1) // b
    perm = np.random.default_rng(seed).permutation(int(pages.sum()))
    kc = np.full((len(perm), Hk, b, d), garbage)
    vc = np.full((len(perm), Hk, b, d), garbage)
    bt = np.full((len(lens), int(pages.max())), -1, dtype=np.int64)
    off = 0
    for i, (n, L) in enumerate(zip(lens, pages)):
        bt[i, :L] = perm[off:off + L]
        off += L
        for p in range(L):
            lo, hi = int(cu[i]) + p * b, int(cu[i]) + min(int(n), (p + 1) * b)
            kc[bt[i, p], :, :hi - lo] = K[:, lo:hi]
            vc[bt[i, p], :, :hi - lo] = V[:, lo:hi]
    return kc, vc, bt


def test_chunked_prefill_equals_single_pass():
    """R-16 with [P2] §3.1: a prompt processed chunk by chunk through a paged cache
    (pages in random physical order, the whole prompt already written, unwritten
    page slots NaN) gives for every chunk the single-pass router rows and outputs:
    later keys and unwritten slots never enter, and chunk block q is logical block
    prefix / b + q.  The second sequence finishes early (an empty chunk)."""
    b, H, Hk, d = 64, 4, 2, 32
    G = H // Hk
    x = synth.gen_prefill([700, 300], H, Hk, d, b, 31, "iid", "fp32")
    Q, K, V = (getattr(x, n).astype(np.float64) for n in "qkv")
    cu = x.cu_seqlens
    Jo, co, _, _ = oracle.route(Q, K, cu, b, G, oracle.TOPK, 4, force_sink=True)
    Oo, lo = oracle.attention(Q, K, V, cu, b, G, Jo, co)
    kc, vc, bt = _paged_from_prompt(K, V, cu, b, 5)
    bounds = [[0, 256, 640, 700], [0, 64, 300, 300]]
    for step in range(3):
        pre = [bd[step] for bd in bounds]
        lens = [bd[step + 1] - bd[step] for bd in bounds]
        ccu = np.concatenate([[0], np.cumsum(lens)])
        qc = np.concatenate([Q[:, cu[i] + pre[i]: cu[i] + pre[i] + lens[i]] for i in range(2)],
                            axis=1)
        Jc, cc, Oc, lc = oracle.chunked_prefill(qc, kc, vc, bt, pre, ccu, b, G, oracle.TOPK, 4,
                                                force_sink=True)
        for i in range(2):
            nq = (lens[i] + b - 1) // b
            r0 = pre[i] // b
            assert np.array_equal(cc[i, :, :nq], co[i, :, r0:r0 + nq])
            assert np.array_equal(Jc[i, :, :nq], Jo[i, :, r0:r0 + nq])
            assert (cc[i, :, nq:] == 0).all()
            sl = slice(cu[i] + pre[i], cu[i] + pre[i] + lens[i])
            got = slice(ccu[i], ccu[i + 1])
            assert np.allclose(Oc[:, got], Oo[:, sl], rtol=0, atol=1e-12)
            assert np.allclose(lc[:, got], lo[:, sl], rtol=0, atol=1e-12)


def test_chunked_prefill_union_threshold_equals_single_pass():
    """The same chunk-by-chunk identity under threshold routing with a local window
    and a global list (union routing): the chunk's rows use their logical block for
    the window, the global ids and the threshold's candidate set."""
    b, H, Hk, d = 32, 2, 1, 16
    G = H // Hk
    x = synth.gen_prefill([600], H, Hk, d, b, 41, "iid", "fp32")
    Q, K, V = (getattr(x, n).astype(np.float64) for n in "qkv")
    cu = x.cu_seqlens
    kw = dict(k_min=2, tau_delta=1.5, force_sink=False, window=3, global_blocks=(1, 7))
    Jo, co, _, _ = oracle.route(Q, K, cu, b, G, oracle.THRESHOLD, 8, **kw)
    Oo, lo = oracle.attention(Q, K, V, cu, b, G, Jo, co)
    kc, vc, bt = _paged_from_prompt(K, V, cu, b, 9)
    for pre, n in ((0, 224), (224, 320), (544, 56)):
        qc = Q[:, pre:pre + n]
        Jc, cc, Oc, lc = oracle.chunked_prefill(qc, kc, vc, bt, [pre], [0, n], b, G,
                                                oracle.THRESHOLD, 8, **kw)
        nq, r0 = (n + b - 1) // b, pre // b
        assert np.array_equal(cc[0, :, :nq], co[0, :, r0:r0 + nq])
        assert np.array_equal(Jc[0, :, :nq], Jo[0, :, r0:r0 + nq])
        assert np.allclose(Oc[:, :n], Oo[:, pre:pre + n], rtol=0, atol=1e-12)
        assert np.allclose(lc[:, :n], lo[:, pre:pre + n], rtol=0, atol=1e-12)


def test_decode_group_score_is_the_max_over_query_heads():
    # Two query heads share one KV head (G = 2); d = 2, pages of 2 tokens, context 6.
    # Page means c_0 = (0.9, 0), c_1 = (0.5, 0.5); page 2 is the last page.
    # q_0 = (1, 0), q_1 = (-1, 2): scores q_h . c_p are
    #   page 0: 0.9 and -0.9   (max 0.9, sum 0.0)
    #   page 1: 0.5 and  0.5   (max 0.5, sum 1.0)
    # so pooling by max keeps page 0, pooling by sum or mean would keep page 1.
    q = np.array([[[1.0, 0.0], [-1.0, 2.0]]])                 # [R=1, H=2, d=2]
    keys = np.array([[0.9, 0.0], [0.9, 0.0],
                     [0.5, 0.5], [0.5, 0.5],
                     [0.0, 0.0], [0.0, 0.0]])
    kc = keys.reshape(3, 1, 2, 2)
    vc = np.arange(12, dtype=np.float64).reshape(3, 1, 2, 2)
    bt = np.array([[0, 1, 2]], dtype=np.int32)
    _, _, sel, cnt, sc = oracle.decode(q, kc, vc, bt, np.array([6]), 2, top_k=1,
                                       return_scores=True)
    per_head = np.array([[0.9, 0.5], [-0.9, 0.5]])            # by hand, as above
    assert np.allclose(sc[(0, 0)], per_head.max(axis=0))
    assert list(sel[0, 0, :cnt[0, 0]]) == [0, 2]               # page 0 and the last page
    assert per_head.sum(axis=0).argmax() == 1                  # a sum would have kept page 1
