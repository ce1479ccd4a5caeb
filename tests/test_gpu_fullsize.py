"""Full-size parity: each large workload runs through PrefillPlan / DecodePlan
exactly as bench.py launches it; sampled rows (every sequence's first, last
and tail rows for every KV head, plus random rows) are recomputed one by one by
the float64 oracle.  Router rows are compared tie-aware; attention rows are
recomputed by the oracle on the index the GPU used for that row (which the
router check has just shown to be the oracle's, up to ties)."""
import numpy as np
import pytest
import torch

import dynamic_block_sparse_mean_gb300 as bsa
import oracle
from dynamic_block_sparse_mean_gb300 import synth, workloads
from parity_utils import (BF16_LSE_ABS, BF16_MAX_ABS, BF16_MEAN_ABS, TIE_BAND, BF16View,
                          check_route_rows, dev_tensor, sample_rows)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

PREFILL = [(workloads.PROMPT_32K, 48), (workloads.VARLEN_256K, 24), (workloads.LONG_128K, 12)]


class RowScores:
    """Sparse score rows: g[i, h, r, :r] for the sampled rows only."""

    def __init__(self):
        self.rows = {}

    def __getitem__(self, idx):
        i, h, r, sl = idx
        return self.rows[(i, h, r)][sl]


@pytest.mark.parametrize("w,n_random", PREFILL, ids=[w.name for w, _ in PREFILL])
def test_prefill_workload_sampled_rows(w, n_random):
    x = synth.make_prefill(w)
    q, k, v = (dev_tensor(a, "bf16") for a in (x.q, x.k, x.v))
    plan = bsa.PrefillPlan(x.cu_seqlens, w.num_heads, w.num_kv_heads, w.head_dim, w.block,
                           bsa.RouteParams(w.mode, w.k_max, w.k_min, w.tau_delta, w.force_sink))
    out, lse = plan.run(q, k, v)
    torch.cuda.synchronize()
    bsa.check_status(plan.status)
    J, cnt = plan.J.cpu().numpy(), plan.counts.cpu().numpy()
    Q, K, V = BF16View(x.q), BF16View(x.k), BF16View(x.v)
    G = w.group
    C = oracle.block_summaries(K, x.cu_seqlens, w.block)
    rows = sample_rows(x.cu_seqlens, w.block, w.num_kv_heads, n_random, seed=w.seed)
    # router: every sampled row, scores against all of its history blocks
    g = RowScores()
    Jo = np.full(J.shape, -1, dtype=np.int64)
    co = np.zeros(cnt.shape, dtype=np.int64)
    for (i, h, r) in rows:
        g.rows[(i, h, r)] = (oracle.route_scores_row(Q, C, x.cu_seqlens, w.block, G, (i, h, r))
                             if r > 0 else np.zeros(0))
        sel = oracle.select_row(g.rows[(i, h, r)], r, w.mode, w.k_max, w.k_min, w.tau_delta,
                                w.force_sink)
        Jo[i, h, r, :len(sel)] = sel
        co[i, h, r] = len(sel)
    check_route_rows(J, cnt, Jo, co, g, rows, w.mode, w.force_sink, w.tau_delta)
    # attention on the GPU's index for the sampled rows
    errs, means, lerr = [], [], []
    out_np = None
    info = oracle.seq_info(x.cu_seqlens, w.block)
    for (i, h, r) in rows[: max(8, len(rows) // 2)]:
        Ob, lb = oracle.attention_row(Q, K, V, x.cu_seqlens, w.block, G, J, cnt, (i, h, r))
        s0, n, _ = info[i]
        t0, t1 = s0 + r * w.block, s0 + min(n, (r + 1) * w.block)
        Og = out[h * G:(h + 1) * G, t0:t1].float().cpu().numpy()
        lg = lse[h * G:(h + 1) * G, t0:t1].cpu().numpy()
        d = np.abs(Og - Ob)
        errs.append(d.max())
        means.append(d.mean())
        lerr.append(np.abs(lg - lb).max())
    assert max(errs) <= BF16_MAX_ABS, max(errs)
    assert float(np.mean(means)) <= BF16_MEAN_ABS, np.mean(means)
    assert max(lerr) <= BF16_LSE_ABS, max(lerr)


def test_decode_workload_sampled_requests():
    w = workloads.DECODE_64
    x = synth.make_decode(w)
    q = dev_tensor(x.q, "bf16")
    kc, vc = dev_tensor(x.k_cache, "bf16"), dev_tensor(x.v_cache, "bf16")
    bt = torch.as_tensor(x.block_table, device="cuda")
    cl = torch.as_tensor(x.context_lens, device="cuda")
    ps = bsa.page_summaries(kc, bt, cl)
    plan = bsa.DecodePlan(w.num_reqs, w.num_heads, w.num_kv_heads, w.head_dim, w.page_size,
                          x.block_table.shape[1], x.k_cache.shape[0], w.top_k)
    o, lse, sel, sc = plan.run(q, kc, vc, ps, bt, cl)
    torch.cuda.synchronize()
    bsa.check_status(plan.status)
    reqs = [0, int(np.argmax(x.context_lens)), int(np.argmin(x.context_lens)), 37]
    q64 = synth.bf16_bits_to_f32(x.q).astype(np.float64)
    oo, lo, so, co, scores = oracle.decode(q64, BF16View(x.k_cache), BF16View(x.v_cache),
                                           x.block_table, x.context_lens, w.page_size, w.top_k,
                                           reqs=reqs, return_scores=True)
    sel, sc = sel.cpu().numpy(), sc.cpu().numpy()
    for rho in reqs:
        for h in range(w.num_kv_heads):
            assert sc[rho, h] == co[rho, h] == w.top_k + 1
            dg, do = set(sel[rho, h, :-1]), set(so[rho, h, :-1])
            assert sel[rho, h, -1] == so[rho, h, -1]
            if dg != do:
                gs = scores[(rho, h)]
                s_k = min(gs[j] for j in do)
                assert all(abs(gs[j] - s_k) <= TIE_BAND for j in dg ^ do)
    og = o.float().cpu().numpy()[reqs]
    d = np.abs(og - oo[reqs])
    assert d.max() <= BF16_MAX_ABS and d.mean() <= BF16_MEAN_ABS
    assert np.abs(lse.cpu().numpy()[reqs] - lo[reqs]).max() <= BF16_LSE_ABS


BACKWARD = [(workloads.PROMPT_32K, 6, 3, 24), (workloads.LONG_128K, 3, 2, 10)]
BWD_REL = 2e-2  # bf16 gradients: max |diff| / max |ref|, as in test_gpu_backward.py


@pytest.mark.parametrize("w,n_rows,n_blocks,max_sel", BACKWARD, ids=[w.name for w, *_ in BACKWARD])
def test_backward_workload_sampled(w, n_rows, n_blocks, max_sel):
    """The backward at full size, launched as bench.py launches it (the forward's
    worklist and lse), on sampled outputs the oracle computes one by one: dQ of
    whole router rows, and dK / dV of key blocks selected by at most max_sel rows
    (the oracle sums those rows' shares), on the index the GPU used."""
    x = synth.make_prefill(w)
    q, k, v = (dev_tensor(a, "bf16") for a in (x.q, x.k, x.v))
    plan = bsa.PrefillPlan(x.cu_seqlens, w.num_heads, w.num_kv_heads, w.head_dim, w.block,
                           bsa.RouteParams(w.mode, w.k_max, w.k_min, w.tau_delta, w.force_sink))
    out, lse = plan.run(q, k, v)
    rng = np.random.default_rng(w.seed + 7)
    dO_bits = synth.f32_to_bf16_bits(rng.normal(size=x.q.shape).astype(np.float32))
    do = dev_tensor(dO_bits, "bf16")
    dq, dk, dv = bsa.attention_bwd(q, k, v, out, do, lse, plan.wl, plan.shape)
    torch.cuda.synchronize()
    bsa.check_status(plan.status)
    J, cnt = plan.J.cpu().numpy(), plan.counts.cpu().numpy()
    Q, K, V, dO = BF16View(x.q), BF16View(x.k), BF16View(x.v), BF16View(dO_bits)
    G, b = w.group, w.block
    info = oracle.seq_info(x.cu_seqlens, b)

    def rel(got, ref):
        return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))

    rows = sample_rows(x.cu_seqlens, b, w.num_kv_heads, 0, seed=w.seed)
    picked = [rows[int(e)] for e in rng.choice(len(rows), size=min(n_rows, len(rows)),
                                              replace=False)]
    for (i, h, r) in picked:
        ref, _, _ = oracle.attention_backward_row(Q, K, V, x.cu_seqlens, b, G, J, cnt, dO,
                                                  (i, h, r))
        s0, n, _ = info[i]
        t0, t1 = s0 + r * b, s0 + min(n, (r + 1) * b)
        got = dq[h * G:(h + 1) * G, t0:t1].float().cpu().numpy()
        assert rel(got, ref) <= BWD_REL, ("dQ", (i, h, r), rel(got, ref))
    # key blocks with a few selecting rows, spread over sequences, heads and positions
    nsel = {}
    for i, (s0, n, nb) in enumerate(info):
        for h in range(w.num_kv_heads):
            for r in range(nb):
                for j in {int(e) for e in J[i, h, r, :cnt[i, h, r]]} or {r}:
                    nsel[(i, h, j)] = nsel.get((i, h, j), 0) + 1
    cands = sorted(key for key, c in nsel.items() if 2 <= c <= max_sel)
    assert cands
    for e in rng.choice(len(cands), size=min(n_blocks, len(cands)), replace=False):
        i, h, j = cands[int(e)]
        ref_k, ref_v = oracle.attention_backward_key_block(Q, K, V, x.cu_seqlens, b, G, J, cnt,
                                                           dO, i, h, j)
        s0, n, _ = info[i]
        t0, t1 = s0 + j * b, s0 + min(n, (j + 1) * b)
        got_k = dk[h, t0:t1].float().cpu().numpy()
        got_v = dv[h, t0:t1].float().cpu().numpy()
        assert rel(got_k, ref_k) <= BWD_REL, ("dK", (i, h, j), rel(got_k, ref_k))
        assert rel(got_v, ref_v) <= BWD_REL, ("dV", (i, h, j), rel(got_v, ref_v))
