"""Plain, slow, float64 CPU oracle for coarse-grained dynamic block-sparse attention.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
anything in this package.  The library (``dynamic_block_sparse_mean_gb300``)
never calls it and shares no code with it; the only module both sides use is
the seeded input generator ``dynamic_block_sparse_mean_gb300.synth``, which
holds none of the method's arithmetic.

Sources (cited by page title and section / equation):
  [P2]  "2.1 · 粗粒度选择: 从内容分组到动态稀疏块" (PaperTrace, sparse-attention 2-1)
  [P3]  PaperTrace sparse-attention 5-1, the page on turning indexer output into
        kernel worklists (headings "从索引输出到工作表", "稀疏 softmax 仍要保持数值一致",
        "如何验证内核真的兑现算法收益")
  [P1]  charlestar.github.io feed, the DeepSeek Sparse Attention indexer entry
        (tiled local top-k followed by a merge, stable ties)

What is computed follows the unified object of [P2] §3.2: summaries
c_v = f(K_v), scores s_uv = g(Q_u, c_v), a selected set I_u over v <= u, and
O_u = Attn(Q_u, Concat K_v, Concat V_v) over the selected blocks taken as a SET
(a block enters the softmax once, [P2] §1.2 after eq.(5) and §3.2).  The
attention is the plain definition: the whole causal score row is materialised,
an explicit mask is built from J, and softmax and AV follow.  Routing is a
selection rule, so it is written out step by step.

Readings where the pages leave a step open (each repeated at its function):
  R-1  summary divisor is the number of valid keys in the block (eq.(11));
       keys past the sequence end never enter a summary ([P2] §4.1).
  R-2  router scores are unscaled q.c_j (eq.(6) has no 1/sqrt(d_h)).
  R-3  query pooling is the max over every valid query row of the block and
       over all query heads of the KV-head group (GQA shares candidates).
  R-4  only complete history blocks j < r are scored; the diagonal r is always
       kept as the triangle branch, block 0 too when the sink is forced; forced
       blocks are not dynamic candidates; k_max counts forced blocks.
  R-5  threshold: tau_r = (max candidate score) - delta; |A| counts candidates
       with score >= tau_r; k_r = min(k_max, max(k_min, |F| + |A|), |F| + |cand|)
       with F the forced set; keep F plus the best k_r - |F| candidates.
  R-6  ranking is (score descending, block index ascending).
  R-7  an empty row falls back to the diagonal block {r}.
  R-8  token-level causal mask s <= t inside the diagonal tile; blocks are
       sequence-relative and never cross a sequence boundary.
  R-9  softmax scale 1/sqrt(d_h) (eq.(2)); lse is the natural-log
       logsumexp over the allowed keys.
  R-11 decode: pages are the routing blocks; the last logical page is always
       kept and never scored; complete pages 0 .. L-2 are scored.
  R-16 chunked prefill: a chunk starts on the page grid (the cached prefix is a
       whole number of pages = routing blocks), so its query blocks are logical
       blocks prefix / b + q and the result is the single-pass prefill's.

Pins (tests/test_oracle_*.py): dense causal attention through
torch.nn.functional.scaled_dot_product_attention when every causal block is
selected; tile-order invariance; a duplicate block changes the multiset result;
empty row equals {r}; GQA permutation; brute force on tiny inputs; the error
bound of [P2] §4; the online-softmax recurrences against the direct softmax;
eq.(11) streaming means; the worked budget numbers of [P2] §2.2 (golden file);
token recall against the dense top-t teacher worked by hand (ties, GQA, an
empty row), equal to 1 at density 1 and to the explicit mask's key count when
the teacher covers every visible key; the backward against central differences,
against autograd of the dense causal attention at density 1, and its one-row /
one-key-block restriction against the whole-sequence backward.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import torch

TOPK = 0
THRESHOLD = 1


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def _f64(x):
    """A slice of an input as float64 (inputs may be any array-like that
    returns real values when indexed; conversion happens per slice)."""
    return np.asarray(x, dtype=np.float64)


def seq_info(cu_seqlens, b: int):
    """(start, length, number of blocks) per sequence; blocks are ceil(n / b)
    ([P2] section 1 opening: N_q = ceil(n / b))."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    out = []
    for i in range(len(cu) - 1):
        s0, n = int(cu[i]), int(cu[i + 1] - cu[i])
        out.append((s0, n, (n + b - 1) // b))
    return out


def max_blocks(cu_seqlens, b: int) -> int:
    return max((nb for _, _, nb in seq_info(cu_seqlens, b)), default=0)


def rank_order(scores, idx):
    """Indices sorted by (score descending, index ascending) — the stable tie rule (R-6)."""
    scores = np.asarray(scores, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    return idx[np.lexsort((idx, -scores))]


# ----------------------------------------------------------------------------
# a1: block summaries
# ----------------------------------------------------------------------------

def block_summaries(K, cu_seqlens, b: int):
    """Mean-pooled key summary c_j of every block of every sequence and KV head.

    [P2] §2.1 eq.(6): c_j = (1/b_k) sum_s k_{j,s}; with the divisor taken as the
    number of keys the block actually holds (eq.(11), r_j), so a partial tail
    block averages its valid keys only and padding never enters ([P2] §4.1).
    Returns C [B, H_kv, N_q, d]; blocks past a sequence's end are zero.
    """
    Hk, _, d = K.shape
    info = seq_info(cu_seqlens, b)
    Nq = max((nb for _, _, nb in info), default=0)
    C = np.zeros((len(info), Hk, Nq, d))
    for i, (s0, n, nb) in enumerate(info):
        for j in range(nb):
            lo, hi = s0 + j * b, s0 + min(n, (j + 1) * b)
            C[i, :, j, :] = _f64(K[:, lo:hi, :]).sum(axis=1) / (hi - lo)
    return C


def streaming_summary(keys):
    """eq.(11) of [P2] §3.1 (block summaries as cache state): s <- s + k_t and
    c = s / r after every appended key; returns the summary after each step."""
    s = np.zeros(keys.shape[-1])
    out = []
    for r, k in enumerate(np.asarray(keys, dtype=np.float64), start=1):
        s = s + k
        out.append(s / r)
    return np.array(out)


# ----------------------------------------------------------------------------
# a2: router scores
# ----------------------------------------------------------------------------

def route_scores(Q, C, cu_seqlens, b: int, G: int, rows=None):
    """g[i, h, r, j] = max over query heads of group h and valid tokens t of block r
    of Q[hq, t] . c_{i,h,j}, for history blocks j < r; -inf elsewhere.

    [P2] §2.1 eq.(6) with pool = max (R-3, "max over the block's queries") and the
    GQA group pooled by max ([P2] §4, group options max / mean / union);
    unscaled (R-2); only complete history j < r is scored ([P2] §2.1, causal
    block rule; §4.1, a summary never holds keys the query cannot see).
    `rows`, if given, is an iterable of (i, h, r) to compute.
    """
    info = seq_info(cu_seqlens, b)
    B, Hk, Nq, d = C.shape
    g = np.full((B, Hk, Nq, Nq), -np.inf)
    if rows is None:
        rows = [(i, h, r) for i, (_, _, nb) in enumerate(info) for h in range(Hk) for r in range(nb)]
    for (i, h, r) in rows:
        if r == 0 or r >= info[i][2]:
            continue
        g[i, h, r, :r] = route_scores_row(Q, C, cu_seqlens, b, G, (i, h, r))
    return g


def route_scores_row(Q, C, cu_seqlens, b: int, G: int, row):
    """The scores g[i, h, r, 0 .. r-1] of one router row (see route_scores)."""
    i, h, r = row
    d = C.shape[3]
    s0, n, _ = seq_info(cu_seqlens, b)[i]
    qr = _f64(Q[h * G:(h + 1) * G, s0 + r * b: s0 + min(n, (r + 1) * b), :]).reshape(-1, d)
    return (qr @ C[i, h, :r, :].T).max(axis=0)


# ----------------------------------------------------------------------------
# a3: selection
# ----------------------------------------------------------------------------

def forced_blocks(r: int, force_sink: bool, window: int = 1, global_blocks=()):
    """Blocks every row r keeps, outside the dynamic budget.

    The diagonal r is always kept (triangle branch, [P2] §2.1 causal rule); block 0
    when the sink is forced (R-4).  Union routing ([P2] §3.2, N_u = L_u ∪ G ∪ I_u,
    with the representations of [P2] §3.1): the local window L_r = the `window`
    most recent blocks r - window + 1 .. r (an implicit rule; window <= 1 is the
    diagonal alone) and the global list G (blocks at or before r; later blocks are
    invisible under the causal rule).  The union is a set: a block named by two
    branches is kept once (R-15)."""
    f = set(range(max(0, r - max(1, window) + 1), r + 1))
    if force_sink:
        f.add(0)
    f |= {int(g) for g in global_blocks if 0 <= int(g) <= r}
    return f


def select_row(g_row, r: int, mode: int, k_max: int, k_min: int = 0,
               tau_delta: float = 0.0, force_sink: bool = False, window: int = 1,
               global_blocks=()):
    """Selected key blocks of query block r, deduplicated and sorted by address.

    Top-k: [P2] §2.1 "top-k, threshold and capacity" — every row gets the same
    budget k_max (forced blocks included, R-4).
    Threshold: eq.(7) k_r = min(k_max, max(k_min, |{j : g_rj >= tau_r}|)) with
    tau_r relative to the row maximum (R-5).
    Dedup and ascending order: [P2] §1.2 (eq.(1) address list, sorted for
    locality) and §3.2 (union then dedup).  The dynamic candidates exclude every
    forced block, window included ([P2] §3.1: dynamic top-k leaves out the blocks
    the local window covers).
    """
    F = forced_blocks(r, force_sink, window, global_blocks)
    cand = np.array([j for j in range(r) if j not in F], dtype=np.int64)
    if mode == TOPK:
        k_dyn = max(0, k_max - len(F))
    elif mode == THRESHOLD:
        if len(cand) == 0:
            k_dyn = 0
        else:
            sc = np.asarray(g_row, dtype=np.float64)[cand]
            tau = sc.max() - tau_delta
            a = int((sc >= tau).sum())
            k_r = min(k_max, max(k_min, len(F) + a), len(F) + len(cand))
            k_dyn = max(0, k_r - len(F))
    else:
        raise ValueError(mode)
    chosen = []
    if k_dyn > 0 and len(cand) > 0:
        chosen = [int(x) for x in rank_order(np.asarray(g_row, dtype=np.float64)[cand], cand)[:k_dyn]]
    return sorted(F | set(chosen))


def route(Q, K, cu_seqlens, b: int, G: int, mode: int, k_max: int, k_min: int = 0,
          tau_delta: float = 0.0, force_sink: bool = False, rows=None, window: int = 1,
          global_blocks=()):
    """Summaries, scores and selection: returns J [B, H_kv, N_q, k_max] (-1 padded),
    counts [B, H_kv, N_q], scores g and summaries C.  Rows not requested keep
    count 0 and -1 entries."""
    C = block_summaries(K, cu_seqlens, b)
    g = route_scores(Q, C, cu_seqlens, b, G, rows)
    B, Hk, Nq, _ = C.shape
    J = np.full((B, Hk, Nq, k_max), -1, dtype=np.int64)
    counts = np.zeros((B, Hk, Nq), dtype=np.int64)
    info = seq_info(cu_seqlens, b)
    if rows is None:
        rows = [(i, h, r) for i, (_, _, nb) in enumerate(info) for h in range(Hk) for r in range(nb)]
    for (i, h, r) in rows:
        if r >= info[i][2]:
            continue
        sel = select_row(g[i, h, r], r, mode, k_max, k_min, tau_delta, force_sink, window,
                         global_blocks)
        J[i, h, r, :len(sel)] = sel
        counts[i, h, r] = len(sel)
    return J, counts, g, C


# ----------------------------------------------------------------------------
# a5: attention on the selected tiles (plain definition with an explicit mask)
# ----------------------------------------------------------------------------

def block_multiplicity(ids, nb: int, r: int, multiset: bool = False):
    """How many times each key block enters the softmax.  Set semantics (default):
    once, whatever J repeats ([P2] §1.2 after eq.(5); §3.2 'dedup before the
    kernel').  Multiset: once per occurrence, the literal Concat of §3.2, used
    only to show that a duplicate changes the result.  An empty row falls back
    to the diagonal block (R-7; [P3] sparse-softmax section)."""
    mult = np.zeros(nb, dtype=np.float64)
    ids = [int(x) for x in ids]
    if not ids:
        ids = [r]
    for j in ids:
        if multiset:
            mult[j] += 1.0
        else:
            mult[j] = 1.0
    return mult


def key_mask(q_lo: int, q_hi: int, mult, b: int):
    """Explicit boolean mask [q_hi - q_lo, q_hi]: query t (sequence-relative,
    q_lo <= t < q_hi) may see key s iff block(s) is selected and s <= t
    ([P2] §1.2 'causal mask before softmax'; §2.1 causal block rule; the first
    index representation of [P2] §3.1 is this dense mask)."""
    kidx = np.arange(q_hi)
    t = np.arange(q_lo, q_hi)
    sel = np.asarray(mult)[kidx // b] > 0
    return sel[None, :] & (kidx[None, :] <= t[:, None])


def attention_rows(Q, K, V, cu_seqlens, b: int, G: int, J, counts, rows, scale=None,
                   multiset: bool = False, O=None, lse=None):
    """O and lse for the requested (i, h_kv, r) rows.

    For every query head of the group and every valid query token t of block r,
    the whole causal score row S = q k^T / sqrt(d_h) ([P2] §1.2 eq.(2)) is
    materialised over keys 0 .. t_max of the sequence (keys after the block's
    last query are masked by causality for every query of the block), the mask
    {s : block(s) in J_r, s <= t} is applied before the softmax ([P2] §1.2,
    masks before softmax; §4.1 token-level triangle in the diagonal block), and
    O = softmax(S) V, lse = logsumexp(S) (R-9).
    """
    H, T, d = Q.shape
    if O is None:
        O = np.full((H, T, d), np.nan)
    if lse is None:
        lse = np.full((H, T), np.nan)
    info = seq_info(cu_seqlens, b)
    for (i, h, r) in rows:
        s0, n, nb = info[i]
        if r >= nb:
            continue
        Ob, lb = attention_row(Q, K, V, cu_seqlens, b, G, J, counts, (i, h, r), scale, multiset)
        q_lo, q_hi = r * b, min(n, (r + 1) * b)
        O[h * G:(h + 1) * G, s0 + q_lo:s0 + q_hi] = Ob
        lse[h * G:(h + 1) * G, s0 + q_lo:s0 + q_hi] = lb
    return O, lse


def attention_row(Q, K, V, cu_seqlens, b: int, G: int, J, counts, row, scale=None,
                  multiset: bool = False):
    """One router row (i, h_kv, r): returns O [G, n_r, d] and lse [G, n_r] for the
    group's query heads and the n_r valid query tokens of block r (same
    definition as attention_rows)."""
    i, h, r = row
    d = Q.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    s0, n, nb = seq_info(cu_seqlens, b)[i]
    cnt = int(counts[i, h, r])
    mult = block_multiplicity(J[i, h, r, :cnt], nb, r, multiset)
    q_lo, q_hi = r * b, min(n, (r + 1) * b)
    wkey = mult[np.arange(q_hi) // b]
    allowed = key_mask(q_lo, q_hi, mult, b)
    Kp, Vp = _f64(K[h, s0:s0 + q_hi]), _f64(V[h, s0:s0 + q_hi])
    Ob = np.empty((G, q_hi - q_lo, d))
    lb = np.empty((G, q_hi - q_lo))
    for g, hq in enumerate(range(h * G, (h + 1) * G)):
        S = (_f64(Q[hq, s0 + q_lo:s0 + q_hi]) @ Kp.T) * scale
        S = np.where(allowed, S, -np.inf)
        m = S.max(axis=1, keepdims=True)
        E = wkey[None, :] * np.exp(S - m)
        l = E.sum(axis=1, keepdims=True)
        Ob[g] = (E @ Vp) / l
        lb[g] = (m + np.log(l))[:, 0]
    return Ob, lb


def all_rows(cu_seqlens, b: int, Hk: int):
    return [(i, h, r) for i, (_, _, nb) in enumerate(seq_info(cu_seqlens, b))
            for h in range(Hk) for r in range(nb)]


def attention(Q, K, V, cu_seqlens, b: int, G: int, J, counts, scale=None, rows=None,
              multiset: bool = False):
    Hk = K.shape[0]
    if rows is None:
        rows = all_rows(cu_seqlens, b, Hk)
    return attention_rows(Q, K, V, cu_seqlens, b, G, J, counts, rows, scale, multiset)


def attention_backward(Q, K, V, cu_seqlens, b: int, G: int, J, counts, dO, scale=None):
    """Gradients dQ, dK, dV of the sparse attention for the upstream gradient dO
    (float64), the backward of the same plain definition as `attention`: per
    sequence and KV head the allowed-key mask {s : block(s) in J_r, s <= t} is
    built explicitly, the masked softmax attention of every query head of the group
    is formed, and torch autograd (a library primitive) differentiates
    sum(O * dO).  dK and dV sum over the group's query heads (GQA).  Training needs
    this backward ([P2] §2.2 training paragraph; [P3] verification: gradients of
    the fixed-candidate kernel against the dense-then-mask reference)."""
    H, T, d = Q.shape
    Hk = K.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dQ = np.zeros((H, T, d))
    dK = np.zeros((Hk, T, d))
    dV = np.zeros((Hk, T, d))
    for i, (s0, n, nb) in enumerate(seq_info(cu_seqlens, b)):
        if n == 0:
            continue
        for h in range(Hk):
            allowed = np.zeros((n, n), dtype=bool)
            for r in range(nb):
                cnt = int(counts[i, h, r])
                sel = [int(x) for x in J[i, h, r, :cnt]] or [r]
                keys = np.zeros(n, dtype=bool)
                for j in set(sel):
                    keys[j * b:min(n, (j + 1) * b)] = True
                for t in range(r * b, min(n, (r + 1) * b)):
                    allowed[t] = keys & (np.arange(n) <= t)
            mask = torch.from_numpy(allowed)
            k = torch.tensor(np.asarray(K[h, s0:s0 + n], dtype=np.float64), requires_grad=True)
            v = torch.tensor(np.asarray(V[h, s0:s0 + n], dtype=np.float64), requires_grad=True)
            for hq in range(h * G, (h + 1) * G):
                q = torch.tensor(np.asarray(Q[hq, s0:s0 + n], dtype=np.float64), requires_grad=True)
                sc = (q @ k.T) * scale
                sc = sc.masked_fill(~mask, float("-inf"))
                o = torch.softmax(sc, dim=-1) @ v
                g = torch.from_numpy(np.asarray(dO[hq, s0:s0 + n], dtype=np.float64))
                gq, gk, gv = torch.autograd.grad((o * g).sum(), (q, k, v))
                dQ[hq, s0:s0 + n] = gq.numpy()
                dK[h, s0:s0 + n] += gk.numpy()
                dV[h, s0:s0 + n] += gv.numpy()
    return dQ, dK, dV


def attention_backward_row(Q, K, V, cu_seqlens, b: int, G: int, J, counts, dO, row,
                           scale=None):
    """The backward of one router row (i, h_kv, r) alone, for sampled checks at sizes
    where `attention_backward` cannot materialise a sequence: the same definition
    (mask {s : block(s) in J_r, s <= t} before the softmax, O = softmax(S) V, torch
    autograd of sum(O * dO)) over the row's query tokens of every query head of the
    group.  The row's queries meet no other row, so its dQ [G, n_r, d] is exact; its
    keys 0 .. t_max receive this row's share of dK and dV [t_max + 1, d] (summed over
    the group's heads), which the rows selecting a key block add up to that block's
    dK and dV (`attention_backward_key_block`)."""
    i, h, r = row
    d = Q.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    s0, n, nb = seq_info(cu_seqlens, b)[i]
    cnt = int(counts[i, h, r])
    mult = block_multiplicity(J[i, h, r, :cnt], nb, r)
    q_lo, q_hi = r * b, min(n, (r + 1) * b)
    mask = torch.from_numpy(key_mask(q_lo, q_hi, mult, b))
    k = torch.tensor(_f64(K[h, s0:s0 + q_hi]), requires_grad=True)
    v = torch.tensor(_f64(V[h, s0:s0 + q_hi]), requires_grad=True)
    dq = np.empty((G, q_hi - q_lo, d))
    dk = np.zeros((q_hi, d))
    dv = np.zeros((q_hi, d))
    for g, hq in enumerate(range(h * G, (h + 1) * G)):
        q = torch.tensor(_f64(Q[hq, s0 + q_lo:s0 + q_hi]), requires_grad=True)
        sc = ((q @ k.T) * scale).masked_fill(~mask, float("-inf"))
        o = torch.softmax(sc, dim=-1) @ v
        gout = torch.from_numpy(_f64(dO[hq, s0 + q_lo:s0 + q_hi]))
        gq, gk, gv = torch.autograd.grad((o * gout).sum(), (q, k, v))
        dq[g] = gq.numpy()
        dk += gk.numpy()
        dv += gv.numpy()
    return dq, dk, dv


def attention_backward_key_block(Q, K, V, cu_seqlens, b: int, G: int, J, counts, dO, i: int,
                                 h: int, j: int, scale=None):
    """dK and dV [n_j, d] of key block j of sequence i and KV head h: the sum, over
    every row r >= j whose selected SET holds j (an empty row holds {r}, R-7), of
    that row's share from `attention_backward_row`."""
    s0, n, nb = seq_info(cu_seqlens, b)[i]
    lo, hi = j * b, min(n, (j + 1) * b)
    dk = np.zeros((hi - lo, Q.shape[2]))
    dv = np.zeros((hi - lo, Q.shape[2]))
    for r in range(j, nb):
        cnt = int(counts[i, h, r])
        sel = {int(x) for x in J[i, h, r, :cnt]} or {r}
        if j not in sel:
            continue
        _, gk, gv = attention_backward_row(Q, K, V, cu_seqlens, b, G, J, counts, dO, (i, h, r),
                                           scale)
        dk += gk[lo:hi]
        dv += gv[lo:hi]
    return dk, dv


def causal_all_blocks(cu_seqlens, b: int, Hk: int):
    """J selecting every causal block 0..r of every row (density 1.0)."""
    info = seq_info(cu_seqlens, b)
    Nq = max((nb for _, _, nb in info), default=0)
    J = np.full((len(info), Hk, Nq, Nq), -1, dtype=np.int64)
    counts = np.zeros((len(info), Hk, Nq), dtype=np.int64)
    for i, (_, _, nb) in enumerate(info):
        for r in range(nb):
            J[i, :, r, :r + 1] = np.arange(r + 1)
            counts[i, :, r] = r + 1
    return J, counts


# ----------------------------------------------------------------------------
# online softmax recurrences (eqs. (3)-(5))
# ----------------------------------------------------------------------------

def online_softmax_merge(S_tiles, V_tiles):
    """Merge score tiles one at a time with [P2] §1.2 eqs.(3)-(5): running row
    max m, exp-sum l and unnormalised output u; returns (u / l, m + ln l)."""
    m = None
    for S, Vt in zip(S_tiles, V_tiles):
        S = np.asarray(S, dtype=np.float64)
        m_hat = S.max(axis=-1)
        p = np.exp(S - m_hat[:, None])
        l_hat = p.sum(axis=-1)
        u_hat = p @ np.asarray(Vt, dtype=np.float64)
        if m is None:
            m, l, u = m_hat, l_hat, u_hat
            continue
        m_new = np.maximum(m, m_hat)                                  # (3)
        a, c = np.exp(m - m_new), np.exp(m_hat - m_new)
        l = a * l + c * l_hat                                         # (4)
        u = a[:, None] * u + c[:, None] * u_hat                       # (5)
        m = m_new
    return u / l[:, None], m + np.log(l)


# ----------------------------------------------------------------------------
# quality and budget diagnostics
# ----------------------------------------------------------------------------

def dense_probabilities(q, Kseq, t: int, scale: float):
    """Dense causal softmax of one query at position t over keys 0..t."""
    s = (np.asarray(Kseq[:t + 1], dtype=np.float64) @ np.asarray(q, dtype=np.float64)) * scale
    e = np.exp(s - s.max())
    return e / e.sum()


def missed_mass(q, Kseq, t: int, allowed_blocks, b: int, scale: float):
    """delta = dense probability mass on keys outside the selected set ([P2] §4);
    1 - delta is the coverage C_i of eq.(10)."""
    a = dense_probabilities(q, Kseq, t, scale)
    inside = np.isin(np.arange(t + 1) // b, np.asarray(list(allowed_blocks)))
    return float(a[~inside].sum())


def coverage(Q, K, cu_seqlens, b: int, G: int, J, counts, rows=None, scale=None):
    """Coverage C_i of eq.(10) ([P2] §3.1, second validation layer): for every query
    token i of the requested rows and every query head of the group, the dense
    causal softmax probability mass that falls on the keys the row selected,
    C_i = sum over j in N(i) of alpha_ij^dense.  [H, T], NaN outside the rows.
    An empty row keeps only its diagonal (R-7)."""
    H, T, d = Q.shape
    Hk = K.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if rows is None:
        rows = all_rows(cu_seqlens, b, Hk)
    C = np.full((H, T), np.nan)
    info = seq_info(cu_seqlens, b)
    for (i, h, r) in rows:
        s0, n, nb = info[i]
        if r >= nb:
            continue
        cnt = int(counts[i, h, r])
        sel = [int(x) for x in J[i, h, r, :cnt]] or [r]
        Kseq = K[h, s0:s0 + n]
        for hq in range(h * G, (h + 1) * G):
            for t in range(r * b, min(n, (r + 1) * b)):
                a = dense_probabilities(Q[hq, s0 + t], Kseq, t, scale)
                inside = np.isin(np.arange(t + 1) // b, np.asarray(sel))
                C[hq, s0 + t] = float(a[inside].sum())
    return C


def dense_scores(q, Kseq, t: int):
    """Unscaled dense scores q . k_s of one query at sequence position t over its
    visible keys s = 0 .. t (the softmax scale does not change their order)."""
    return np.asarray(Kseq[:t + 1], dtype=np.float64) @ np.asarray(q, dtype=np.float64)


def token_recall(Q, K, cu_seqlens, b: int, G: int, J, counts, t_top: int, queries):
    """Token recall@t against the dense teacher ([P2] §1.1, the paragraph on
    recall@k: G_i = the dense attention's top-t keys of query i, N(i) = its
    candidate keys, token recall = |G_i ∩ N(i)| / |G_i|; the physical tile
    budget is reported beside it).

    queries: (query head hq, packed token index) pairs.  For query i at sequence
    position t, G_i holds the min(t_top, t + 1) visible keys (s <= t, same
    sequence) of largest dense score, ranked by (score desc, index asc) (R-6);
    N(i) holds the visible keys whose block is in the J row (i, hq // G, t // b),
    an empty row keeping its diagonal (R-7).  Returns {(hq, token): (|G_i ∩ N(i)|,
    |G_i|)}."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    out = {}
    for hq, tok in queries:
        i = int(np.searchsorted(cu, tok, side="right") - 1)
        s0 = int(cu[i])
        t = int(tok) - s0
        h, r = hq // G, t // b
        cnt = int(counts[i, h, r])
        sel = set(int(x) for x in J[i, h, r, :cnt]) or {r}
        g = dense_scores(Q[hq, tok], K[h, s0:s0 + t + 1], t)
        top = rank_order(g, np.arange(t + 1))[:t_top]
        hits = sum(1 for s in top if int(s) // b in sel)
        out[(int(hq), int(tok))] = (hits, len(top))
    return out


def dense_causal_pairs(n: int) -> int:
    """eq.(8) of [P2] §2.2: n (n + 1) / 2 token pairs for one head."""
    return n * (n + 1) // 2


def physical_pairs(row_counts, bq: int, bk: int) -> int:
    """Physical tile pairs: every selected block of a row is a full bq x bk tile
    (eq.(9) of [P2] §2.2 counts 128 x 8 x 64 x 64)."""
    return int(np.asarray(row_counts, dtype=np.int64).sum()) * bq * bk


def unique_tiles(row) -> int:
    """Unique physical tiles of a row ([P2] §2.2: the after-dedup tile count)."""
    return len(set(int(x) for x in row))


def causal_visibility(pos: int, b: int):
    """Block of query position pos and the first / last key it may see
    ([P2] §2.1 causal rule: position 130 at b = 64 is in block 2 and sees 0..130)."""
    return pos // b, 0, pos


# ----------------------------------------------------------------------------
# decode
# ----------------------------------------------------------------------------

def decode(q, k_cache, v_cache, block_table, context_lens, page: int, top_k: int,
           scale=None, reqs=None, return_scores: bool = False):
    """Paged single-token decode with the same router.

    For request rho and KV head h: L = ceil(len / page) logical pages; the
    complete pages 0 .. L-2 are summarised by their mean key (eq.(6)) and scored
    with max over the group's query heads (R-3); the best top_k by (score desc,
    index asc) plus the last page L-1 (R-11) are kept in ascending order; the
    logical ids are mapped to physical pages through the block table ([P2]
    §3.1 paged KV: the router emits monotone logical ids, the block table maps
    them at attention time); softmax over the selected pages' valid tokens.
    Decode cost is reading the summaries plus the selected K/V ([P2] §2.2).
    Returns o [R, H, d], lse [R, H], sel [R, H_kv, top_k + 1] (-1 padded), counts,
    and with return_scores a dict {(rho, h): page scores} as a fifth value.
    """
    q = np.asarray(q, dtype=np.float64)
    R, H, d = q.shape
    Hk = k_cache.shape[1]
    G = H // Hk
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.full((R, H, d), np.nan)
    lse = np.full((R, H), np.nan)
    sel = np.full((R, Hk, top_k + 1), -1, dtype=np.int64)
    cnt = np.zeros((R, Hk), dtype=np.int64)
    scores = {}
    if reqs is None:
        reqs = range(R)
    for rho in reqs:
        n = int(context_lens[rho])
        L = (n + page - 1) // page
        phys = np.asarray(block_table[rho, :L], dtype=np.int64)
        for h in range(Hk):
            Kl = _f64(k_cache[phys, h]).reshape(L * page, d)[:n]
            Vl = _f64(v_cache[phys, h]).reshape(L * page, d)[:n]
            qg = q[rho, h * G:(h + 1) * G]
            if L > 1:
                c = Kl[:(L - 1) * page].reshape(L - 1, page, d).mean(axis=1)
                gsc = (qg @ c.T).max(axis=0)
                chosen = [int(x) for x in rank_order(gsc, np.arange(L - 1))[:top_k]]
            else:
                gsc = np.zeros(0)
                chosen = []
            scores[(rho, h)] = gsc
            ids = sorted(set(chosen) | {L - 1})
            sel[rho, h, :len(ids)] = ids
            cnt[rho, h] = len(ids)
            keys = np.concatenate([np.arange(p * page, min(n, (p + 1) * page)) for p in ids])
            S = (qg @ Kl[keys].T) * scale
            m = S.max(axis=1, keepdims=True)
            E = np.exp(S - m)
            l = E.sum(axis=1, keepdims=True)
            o[rho, h * G:(h + 1) * G] = (E @ Vl[keys]) / l
            lse[rho, h * G:(h + 1) * G] = (m + np.log(l))[:, 0]
    if return_scores:
        return o, lse, sel, cnt, scores
    return o, lse, sel, cnt


# ----------------------------------------------------------------------------
# chunked prefill over a paged cache
# ----------------------------------------------------------------------------

def chunked_prefill(q_chunk, k_cache, v_cache, block_table, prefix_lens, chunk_cu, b: int,
                    G: int, mode: int, k_max: int, k_min: int = 0, tau_delta: float = 0.0,
                    force_sink: bool = False, window: int = 1, global_blocks=(), scale=None):
    """One chunk of a chunked prefill whose keys and values already sit in the
    paged cache ([P2] §3.1: block summaries are cache state kept beside the KV
    cache; the router's logical block ids are mapped to physical pages by the
    block table; [P2] §2.2: a query block's routing needs only the summaries of
    its history).

    Sequence i has prefix_lens[i] tokens cached before the chunk and adds the
    chunk_cu[i+1] - chunk_cu[i] tokens of q_chunk; its context of prefix + n keys
    and values is read out of the pages block_table[i][0..] (page size b, R-16:
    the prefix is a multiple of b, so chunk query block q is the logical block
    r = prefix / b + q).  Everything else is the single-pass definition applied
    to that context: block-mean summaries, scores, selection (`route`) and the
    masked attention (`attention`), for the chunk's query blocks only.
    Returns J [B, H_kv, N_q, k_max] (logical ids, -1 padded), counts [B, H_kv, N_q],
    O [H, T_chunk, d] and lse [H, T_chunk]; N_q = ceil(max chunk length / b).
    """
    q_chunk = np.asarray(q_chunk, dtype=np.float64)
    H, Tc, d = q_chunk.shape
    Hk = k_cache.shape[1]
    cu = np.asarray(chunk_cu, dtype=np.int64)
    B = len(cu) - 1
    lens = np.diff(cu)
    Nq = int(((lens + b - 1) // b).max()) if B else 0
    J = np.full((B, Hk, Nq, k_max), -1, dtype=np.int64)
    counts = np.zeros((B, Hk, Nq), dtype=np.int64)
    O = np.full((H, Tc, d), np.nan)
    lse = np.full((H, Tc), np.nan)
    for i in range(B):
        pre, n, s0 = int(prefix_lens[i]), int(lens[i]), int(cu[i])
        if n == 0:
            continue  # an idle sequence: its prefix may end anywhere
        assert pre % b == 0, "R-16: a chunk starts on the page grid"
        ctx = pre + n
        L = (ctx + b - 1) // b
        phys = np.asarray(block_table[i, :L], dtype=np.int64)
        Kc = np.stack([_f64(k_cache[phys, h]).reshape(L * b, d)[:ctx] for h in range(Hk)])
        Vc = np.stack([_f64(v_cache[phys, h]).reshape(L * b, d)[:ctx] for h in range(Hk)])
        Qc = np.zeros((H, ctx, d))
        Qc[:, pre:] = q_chunk[:, s0:s0 + n]
        one = np.array([0, ctx])
        rows = [(0, h, r) for h in range(Hk) for r in range(pre // b, L)]
        Jc, cc, _, _ = route(Qc, Kc, one, b, G, mode, k_max, k_min, tau_delta, force_sink,
                             rows=rows, window=window, global_blocks=global_blocks)
        Oc, lc = attention(Qc, Kc, Vc, one, b, G, Jc, cc, scale=scale, rows=rows)
        nq = L - pre // b
        J[i, :, :nq] = Jc[0, :, pre // b:L]
        counts[i, :, :nq] = cc[0, :, pre // b:L]
        O[:, s0:s0 + n] = Oc[:, pre:]
        lse[:, s0:s0 + n] = lc[:, pre:]
    return J, counts, O, lse


# ----------------------------------------------------------------------------
# brute force (scalar loops, tiny inputs only)
# ----------------------------------------------------------------------------

def brute_summaries(K, cu_seqlens, b: int):
    """Scalar-loop block means (n <= 256 only)."""
    Hk, _, d = len(K), len(K[0]), len(K[0][0])
    info = seq_info(cu_seqlens, b)
    Nq = max(nb for _, _, nb in info)
    C = [[[[0.0] * d for _ in range(Nq)] for _ in range(Hk)] for _ in info]
    for i, (s0, n, nb) in enumerate(info):
        for h in range(Hk):
            for j in range(nb):
                cntv = 0
                acc = [0.0] * d
                for t in range(j * b, min(n, (j + 1) * b)):
                    cntv += 1
                    for e in range(d):
                        acc[e] += float(K[h][s0 + t][e])
                C[i][h][j] = [a / cntv for a in acc]
    return C


def brute_scores(Q, C, cu_seqlens, b: int, G: int):
    """Scalar-loop router scores g[i][h][r][j] (None where not scored)."""
    info = seq_info(cu_seqlens, b)
    Hk = len(C[0])
    d = len(Q[0][0])
    out = {}
    for i, (s0, n, nb) in enumerate(info):
        for h in range(Hk):
            for r in range(nb):
                for j in range(r):
                    best = -math.inf
                    for hq in range(h * G, (h + 1) * G):
                        for t in range(r * b, min(n, (r + 1) * b)):
                            s = 0.0
                            for e in range(d):
                                s += float(Q[hq][s0 + t][e]) * C[i][h][j][e]
                            best = max(best, s)
                    out[(i, h, r, j)] = best
    return out


def brute_topk_by_enumeration(scores: dict, k: int):
    """The unique k-subset whose every member outranks every non-member under
    (score desc, index asc), found by trying all subsets (R-6)."""
    keys = sorted(scores)
    k = min(k, len(keys))
    hits = []
    for sub in itertools.combinations(keys, k):
        inside, outside = set(sub), [j for j in keys if j not in sub]
        ok = all((scores[a] > scores[o]) or (scores[a] == scores[o] and a < o)
                 for a in inside for o in outside)
        if ok:
            hits.append(sorted(sub))
    assert len(hits) == 1
    return hits[0]


def brute_attention(Q, K, V, cu_seqlens, b: int, G: int, J, counts, scale=None):
    """Scalar-loop masked softmax attention (n <= 256 only)."""
    H, d = len(Q), len(Q[0][0])
    Hk = len(K)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    info = seq_info(cu_seqlens, b)
    O, L = {}, {}
    for i, (s0, n, nb) in enumerate(info):
        for h in range(Hk):
            for r in range(nb):
                cnt = int(counts[i][h][r])
                ids = set(int(x) for x in J[i][h][r][:cnt]) or {r}
                for hq in range(h * G, (h + 1) * G):
                    for t in range(r * b, min(n, (r + 1) * b)):
                        sc = []
                        for s in range(0, t + 1):
                            if s // b in ids:
                                dot = 0.0
                                for e in range(d):
                                    dot += float(Q[hq][s0 + t][e]) * float(K[h][s0 + s][e])
                                sc.append((s, dot * scale))
                        m = max(v for _, v in sc)
                        den = sum(math.exp(v - m) for _, v in sc)
                        o = [0.0] * d
                        for s, v in sc:
                            w = math.exp(v - m) / den
                            for e in range(d):
                                o[e] += w * float(V[h][s0 + s][e])
                        O[(hq, s0 + t)] = o
                        L[(hq, s0 + t)] = m + math.log(den)
    return O, L
