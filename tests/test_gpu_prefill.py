"""GPU parity of the prefill path (summaries, router, worklist, attention) against
the float64 oracle on identical seeded inputs, through the C ABI."""
import numpy as np
import pytest
import torch

import dynamic_block_sparse_mean_gb300 as bsa
import oracle
from dynamic_block_sparse_mean_gb300 import synth
from parity_utils import (BF16_LSE_ABS, BF16_MAX_ABS, BF16_MEAN_ABS, FP32_REL, TIE_BAND,
                          attention_errors, check_buckets, check_route_rows, expected_csr,
                          oracle_view, shape_of, upload, worklist_from_oracle)

pytestmark = pytest.mark.gpu

# (name, lengths, H, H_kv, d, b, mode, k_max, k_min, tau_delta, sink)
CASES = [
    ("tiny_n1024_d64_b64", [1024], 2, 2, 64, 64, oracle.TOPK, 4, 0, 0.0, True),
    ("ragged_gqa4_d128_b64", [700, 129, 64, 1500], 8, 2, 128, 64, oracle.TOPK, 6, 0, 0.0, False),
    ("gqa8_d128_b128_sink", [1000, 300], 16, 2, 128, 128, oracle.TOPK, 5, 0, 0.0, True),
    ("gqa2_d128_b64_threshold", [777, 1300], 4, 2, 128, 64, oracle.THRESHOLD, 8, 2, 2.0, False),
    ("gqa3_d64_b64", [640, 33], 6, 2, 64, 64, oracle.TOPK, 3, 0, 0.0, False),
    ("gqa1_d64_b128", [900], 2, 2, 64, 128, oracle.TOPK, 4, 0, 0.0, True),
]


def _run_case(case, dtype="bf16", seed=7):
    name, lengths, H, Hk, d, b, mode, k_max, k_min, tau, sink = case
    x = synth.gen_prefill(lengths, H, Hk, d, b, seed, "iid", dtype)
    q, k, v = upload(x)
    sh = shape_of(x, H, Hk)
    params = bsa.RouteParams(mode, k_max, k_min, tau, sink)
    return x, q, k, v, sh, params


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_summaries_match_oracle(case):
    x, q, k, v, sh, params = _run_case(case)
    C = bsa.block_summaries(k, sh).cpu().numpy()
    Co = oracle.block_summaries(oracle_view(x, "k"), x.cu_seqlens, x.block)
    assert C.shape == Co.shape
    assert np.abs(C - Co).max() < 1e-5


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_router_matches_oracle_tie_aware(case):
    x, q, k, v, sh, params = _run_case(case)
    H, Hk = case[2], case[3]
    C = bsa.block_summaries(k, sh)
    scores = torch.full((sh.num_seqs, Hk, sh.max_blocks, sh.max_blocks), float("nan"), device="cuda")
    J, cnt = bsa.route(q, C, sh, params, scores=scores)
    Jo, co, go, _ = oracle.route(oracle_view(x, "q"), oracle_view(x, "k"), x.cu_seqlens, x.block,
                                 H // Hk, params.mode, params.k_max, params.k_min, params.tau_delta,
                                 params.force_sink)
    rows = oracle.all_rows(x.cu_seqlens, x.block, Hk)
    check_route_rows(J.cpu().numpy(), cnt.cpu().numpy(), Jo, co, go, rows, params.mode,
                     params.force_sink, params.tau_delta)
    # the score matrix itself: fp32-accurate against float64
    sg = scores.cpu().numpy()
    valid = np.isfinite(go)
    assert np.abs(sg[valid] - go[valid]).max() < 2e-6 * max(1.0, np.abs(go[valid]).max())
    # rows past a sequence's end are empty and -1 filled
    info = oracle.seq_info(x.cu_seqlens, x.block)
    cn = cnt.cpu().numpy()
    for i, (_, _, nb) in enumerate(info):
        assert (cn[i, :, nb:] == 0).all()


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_router_screen_matches_oracle_tie_aware(case):
    # Without a score matrix the BF16 router screens with q . (c_hi + c_mid) and
    # rescores only the candidates its error bound cannot place.
    x, q, k, v, sh, params = _run_case(case, seed=8)
    params.screen = 1
    H, Hk = case[2], case[3]
    C = bsa.block_summaries(k, sh)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    J, cnt = bsa.route(q, C, sh, params, dev_status=st)
    torch.cuda.synchronize()
    bsa.check_status(st)
    Jo, co, go, _ = oracle.route(oracle_view(x, "q"), oracle_view(x, "k"), x.cu_seqlens, x.block,
                                 H // Hk, params.mode, params.k_max, params.k_min, params.tau_delta,
                                 params.force_sink)
    rows = oracle.all_rows(x.cu_seqlens, x.block, Hk)
    check_route_rows(J.cpu().numpy(), cnt.cpu().numpy(), Jo, co, go, rows, params.mode,
                     params.force_sink, params.tau_delta)


@pytest.mark.parametrize("mode", [oracle.TOPK, oracle.THRESHOLD])
def test_router_screen_with_every_candidate_tied(mode):
    # Keys repeat with period b, so every complete block holds the same keys: all
    # summaries and all candidate scores tie exactly, no bound can place any
    # candidate, and every one is rescored (several rounds per row); ties go to the
    # lower block index on both sides, so J must equal the oracle's exactly.
    lengths, H, Hk, d, b = [1500, 700], 4, 2, 128, 64
    x = synth.gen_prefill(lengths, H, Hk, d, b, 11, "iid", "bf16")
    cu = x.cu_seqlens
    for i, n in enumerate(lengths):
        s0 = int(cu[i])
        for t in range(b, n):
            x.k[:, s0 + t] = x.k[:, s0 + t % b]
    q, k, v = upload(x)
    sh = shape_of(x, H, Hk)
    params = (bsa.RouteParams(oracle.TOPK, 6, 0, 0.0, True, screen=1) if mode == oracle.TOPK else
              bsa.RouteParams(oracle.THRESHOLD, 8, 2, 2.0, False, screen=1))
    C = bsa.block_summaries(k, sh)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    J, cnt = bsa.route(q, C, sh, params, dev_status=st)
    torch.cuda.synchronize()
    bsa.check_status(st)
    Jo, co, go, _ = oracle.route(oracle_view(x, "q"), oracle_view(x, "k"), cu, b, H // Hk,
                                 params.mode, params.k_max, params.k_min, params.tau_delta,
                                 params.force_sink)
    assert np.array_equal(cnt.cpu().numpy(), co)
    Jg = J.cpu().numpy()
    for (i, h, r) in oracle.all_rows(cu, b, Hk):
        assert list(Jg[i, h, r, :co[i, h, r]]) == list(Jo[i, h, r, :co[i, h, r]]), (i, h, r)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_worklist_csr_and_buckets(case):
    x, q, k, v, sh, params = _run_case(case)
    H, Hk = case[2], case[3]
    Jo, co, _, _ = oracle.route(oracle_view(x, "q"), oracle_view(x, "k"), x.cu_seqlens, x.block,
                                H // Hk, params.mode, params.k_max, params.k_min, params.tau_delta,
                                params.force_sink)
    co = co.copy()
    co[0, 0, min(2, co.shape[2] - 1)] = 0       # one empty row: falls back to {r}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wl = worklist_from_oracle(Jo, co, sh, params.k_max, status)
    bsa.check_status(status)
    rp, ci = expected_csr(Jo, co, x.cu_seqlens, x.block)
    assert np.array_equal(wl.row_ptr.cpu().numpy(), rp)
    assert np.array_equal(wl.col_idx.cpu().numpy()[:len(ci)], ci)
    check_buckets(wl, rp)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_attention_bf16_on_oracle_index(case):
    x, q, k, v, sh, params = _run_case(case)
    H, Hk = case[2], case[3]
    G = H // Hk
    Jo, co, _, _ = oracle.route(oracle_view(x, "q"), oracle_view(x, "k"), x.cu_seqlens, x.block,
                                G, params.mode, params.k_max, params.k_min, params.tau_delta,
                                params.force_sink)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wl = worklist_from_oracle(Jo, co, sh, params.k_max, status)
    O, lse = bsa.attention_fwd(q, k, v, wl, sh, status)
    torch.cuda.synchronize()
    bsa.check_status(status)
    Oo, lo = oracle.attention(oracle_view(x, "q"), oracle_view(x, "k"), oracle_view(x, "v"),
                              x.cu_seqlens, x.block, G, Jo, co)
    Og = O.float().cpu().numpy()
    lg = lse.cpu().numpy()
    mask = np.ones(lo.shape, dtype=bool)
    mx, mean, lmx, _, _ = attention_errors(Og, lg, Oo, lo, mask)
    assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS, (mx, mean)
    assert lmx <= BF16_LSE_ABS, lmx


@pytest.mark.parametrize("case", [CASES[0], CASES[1], CASES[2]], ids=[c[0] for c in CASES[:3]])
def test_attention_fp32_path(case):
    x, q, k, v, sh, params = _run_case(case, dtype="fp32")
    H, Hk = case[2], case[3]
    G = H // Hk
    Qo, Ko, Vo = (getattr(x, n).astype(np.float64) for n in "qkv")
    Jo, co, _, _ = oracle.route(Qo, Ko, x.cu_seqlens, x.block, G, params.mode, params.k_max,
                                params.k_min, params.tau_delta, params.force_sink)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wl = worklist_from_oracle(Jo, co, sh, params.k_max, status)
    O, lse = bsa.attention_fwd(q, k, v, wl, sh, status)
    torch.cuda.synchronize()
    bsa.check_status(status)
    Oo, lo = oracle.attention(Qo, Ko, Vo, x.cu_seqlens, x.block, G, Jo, co)
    Og, lg = O.cpu().numpy(), lse.cpu().numpy()
    assert np.abs(Og - Oo).max() / np.abs(Oo).max() <= FP32_REL
    assert np.abs(lg - lo).max() / np.abs(lo).max() <= FP32_REL
    # the FP32 router too: the same tie-aware rule
    C = bsa.block_summaries(k, sh)
    J, cnt = bsa.route(q, C, sh, params)
    _, _, go, _ = oracle.route(Qo, Ko, x.cu_seqlens, x.block, G, params.mode, params.k_max,
                               params.k_min, params.tau_delta, params.force_sink)
    check_route_rows(J.cpu().numpy(), cnt.cpu().numpy(), Jo, co, go,
                     oracle.all_rows(x.cu_seqlens, x.block, Hk), params.mode, params.force_sink,
                     params.tau_delta)


def test_all_causal_blocks_equal_dense_attention():
    """Density 1.0: every causal block selected is dense causal attention."""
    x = synth.gen_prefill([1024, 333], 8, 2, 128, 64, 21)
    q, k, v = upload(x)
    sh = shape_of(x, 8, 2)
    Jo, co = oracle.causal_all_blocks(x.cu_seqlens, 64, 2)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wl = worklist_from_oracle(Jo, co, sh, Jo.shape[-1], status)
    O, lse = bsa.attention_fwd(q, k, v, wl, sh, status)
    Oo, lo = oracle.attention(oracle_view(x, "q"), oracle_view(x, "k"), oracle_view(x, "v"),
                              x.cu_seqlens, 64, 4, Jo, co)
    mx, mean, lmx, _, _ = attention_errors(O.float().cpu().numpy(), lse.cpu().numpy(), Oo, lo,
                                           np.ones(lo.shape, dtype=bool))
    bsa.check_status(status)
    assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS and lmx <= BF16_LSE_ABS


def test_shuffled_tile_order_stays_within_tolerance():
    """Tiles merged in any order give the same result up to rounding."""
    x = synth.gen_prefill([1500], 8, 2, 128, 64, 22)
    q, k, v = upload(x)
    sh = shape_of(x, 8, 2)
    Jo, co, _, _ = oracle.route(oracle_view(x, "q"), oracle_view(x, "k"), x.cu_seqlens, 64, 4,
                                oracle.TOPK, 8)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wl = worklist_from_oracle(Jo, co, sh, 8, status)
    rp = wl.row_ptr.cpu().numpy()
    ci = wl.col_idx.cpu().numpy().copy()
    rng = np.random.default_rng(0)
    for rr in range(len(rp) - 1):
        ci[rp[rr]:rp[rr + 1]] = rng.permutation(ci[rp[rr]:rp[rr + 1]])
    wl.col_idx.copy_(torch.as_tensor(ci, device="cuda"))
    O, lse = bsa.attention_fwd(q, k, v, wl, sh, status)
    Oo, lo = oracle.attention(oracle_view(x, "q"), oracle_view(x, "k"), oracle_view(x, "v"),
                              x.cu_seqlens, 64, 4, Jo, co)
    mx, mean, lmx, _, _ = attention_errors(O.float().cpu().numpy(), lse.cpu().numpy(), Oo, lo,
                                           np.ones(lo.shape, dtype=bool))
    bsa.check_status(status)
    assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS and lmx <= BF16_LSE_ABS


@pytest.mark.parametrize("kind,code", [("duplicate", 17), ("descending", 17), ("future", 16),
                                       ("negative", 16), ("count", 18)])
def test_worklist_rejects_malformed_rows(kind, code):
    x = synth.gen_prefill([640], 2, 1, 64, 64, 23)
    sh = shape_of(x, 2, 1)
    J = np.full((1, 1, 10, 4), -1, dtype=np.int32)
    cnt = np.zeros((1, 1, 10), dtype=np.int32)
    for r in range(10):
        J[0, 0, r, 0] = r
        cnt[0, 0, r] = 1
    r = 5
    bad = {"duplicate": [1, 1, 5], "descending": [3, 1, 5], "future": [1, 6],
           "negative": [-2, 5], "count": [1, 2, 5]}[kind]
    J[0, 0, r, :len(bad)] = bad
    cnt[0, 0, r] = len(bad) if kind != "count" else 9
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsa.build_worklist(torch.as_tensor(J, device="cuda"), torch.as_tensor(cnt, device="cuda"), sh,
                       4, status)
    assert int(status.item()) == code


def test_duplicate_through_multiset_would_change_result():
    """The worklist refuses duplicates, and counting one twice (the oracle's
    multiset mode) would move the output past the tolerance."""
    x = synth.gen_prefill([512], 2, 1, 64, 64, 24)
    Jd = np.full((1, 1, 8, 4), -1)
    Jd[0, 0, 5, :3] = [2, 2, 5]
    cd = np.zeros((1, 1, 8), dtype=np.int64)
    cd[0, 0, 5] = 3
    Os, _ = oracle.attention(oracle_view(x, "q"), oracle_view(x, "k"), oracle_view(x, "v"),
                             x.cu_seqlens, 64, 2, Jd, cd, rows=[(0, 0, 5)])
    Om, _ = oracle.attention(oracle_view(x, "q"), oracle_view(x, "k"), oracle_view(x, "v"),
                             x.cu_seqlens, 64, 2, Jd, cd, rows=[(0, 0, 5)], multiset=True)
    assert np.nanmax(np.abs(Os - Om)) > BF16_MAX_ABS
    sh = shape_of(x, 2, 1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsa.build_worklist(torch.as_tensor(Jd.astype(np.int32), device="cuda"),
                       torch.as_tensor(cd.astype(np.int32), device="cuda"), sh, 4, status)
    assert int(status.item()) == 17


def test_plan_end_to_end_small():
    """PrefillPlan (the public API) on the tiny workload against the oracle."""
    w = __import__("dynamic_block_sparse_mean_gb300.workloads", fromlist=["TINY"]).TINY
    x = synth.make_prefill(w)
    q, k, v = upload(x)
    plan = bsa.PrefillPlan(x.cu_seqlens, w.num_heads, w.num_kv_heads, w.head_dim, w.block,
                           bsa.RouteParams(w.mode, w.k_max, w.k_min, w.tau_delta, w.force_sink))
    O, lse = plan.run(q, k, v)
    torch.cuda.synchronize()
    bsa.check_status(plan.status)
    Jo, co, go, _ = oracle.route(oracle_view(x, "q"), oracle_view(x, "k"), x.cu_seqlens, w.block,
                                 w.group, w.mode, w.k_max, w.k_min, w.tau_delta, w.force_sink)
    check_route_rows(plan.J.cpu().numpy(), plan.counts.cpu().numpy(), Jo, co, go,
                     oracle.all_rows(x.cu_seqlens, w.block, w.num_kv_heads), w.mode, w.force_sink)
    Oo, lo = oracle.attention(oracle_view(x, "q"), oracle_view(x, "k"), oracle_view(x, "v"),
                              x.cu_seqlens, w.block, w.group, plan.J.cpu().numpy(),
                              plan.counts.cpu().numpy())
    mx, mean, lmx, _, _ = attention_errors(O.float().cpu().numpy(), lse.cpu().numpy(), Oo, lo,
                                           np.ones(lo.shape, dtype=bool))
    assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS and lmx <= BF16_LSE_ABS


# Union routing N_u = L_u ∪ G ∪ I_u: (name, lengths, H, H_kv, d, b, mode, k_max, k_min,
# tau_delta, sink, window, global list).  The last case repeats a global block and
# names blocks inside the window and past the sequence end.
UNION_CASES = [
    ("union_w3_g2_sink_topk", [1500, 700], 8, 2, 128, 64, oracle.TOPK, 10, 0, 0.0, True, 3, (2, 5)),
    ("union_w4_g1_threshold", [1300, 900], 4, 2, 128, 64, oracle.THRESHOLD, 12, 2, 2.0, False, 4,
     (1,)),
    ("union_w2_dup_b128", [2000], 16, 2, 128, 128, oracle.TOPK, 6, 0, 0.0, False, 2, (0, 3, 3, 40)),
]


def _union_case(case, seed=11):
    name, lengths, H, Hk, d, b, mode, k_max, k_min, tau, sink, window, glob = case
    x = synth.gen_prefill(lengths, H, Hk, d, b, seed, "iid", "bf16")
    q, k, v = upload(x)
    sh = shape_of(x, H, Hk)
    params = bsa.RouteParams(mode, k_max, k_min, tau, sink, window=window, global_blocks=glob)
    return x, q, k, v, sh, params


@pytest.mark.parametrize("case", UNION_CASES, ids=[c[0] for c in UNION_CASES])
def test_union_router_matches_oracle(case):
    x, q, k, v, sh, params = _union_case(case)
    H, Hk = case[2], case[3]
    C = bsa.block_summaries(k, sh)
    J, cnt = bsa.route(q, C, sh, params)
    Jo, co, go, _ = oracle.route(oracle_view(x, "q"), oracle_view(x, "k"), x.cu_seqlens, x.block,
                                 H // Hk, params.mode, params.k_max, params.k_min, params.tau_delta,
                                 params.force_sink, window=params.window,
                                 global_blocks=params.global_blocks)
    rows = oracle.all_rows(x.cu_seqlens, x.block, Hk)
    check_route_rows(J.cpu().numpy(), cnt.cpu().numpy(), Jo, co, go, rows, params.mode,
                     params.force_sink, params.tau_delta, window=params.window,
                     global_blocks=params.global_blocks)


@pytest.mark.parametrize("case", UNION_CASES, ids=[c[0] for c in UNION_CASES])
def test_union_routing_end_to_end(case):
    x, q, k, v, sh, params = _union_case(case)
    H, Hk = case[2], case[3]
    G = H // Hk
    plan = bsa.PrefillPlan(x.cu_seqlens, H, Hk, case[4], case[5], params, device="cuda")
    O, lse = plan.run(q, k, v)
    torch.cuda.synchronize()
    bsa.check_status(plan.status)
    # the oracle's attention over the index the GPU chose (checked above against the
    # oracle's own selection) gives the exact expected output for that index
    Jg = plan.J.cpu().numpy().astype(np.int64)
    cg = plan.counts.cpu().numpy().astype(np.int64)
    Oo, lo = oracle.attention(oracle_view(x, "q"), oracle_view(x, "k"), oracle_view(x, "v"),
                              x.cu_seqlens, x.block, G, Jg, cg)
    mx, mean, lmx, _, _ = attention_errors(O.float().cpu().numpy(), lse.cpu().numpy(), Oo, lo,
                                           np.ones(lo.shape, dtype=bool))
    assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS and lmx <= BF16_LSE_ABS, (mx, mean, lmx)


# Density-1 worklist and the coverage C_i of eq.(10).
DENSE_CASES = [
    ("dense_ragged_gqa4", [700, 129, 1500], 8, 2, 128, 64, None),
    # N_q = 258 > BSA_MAX_K: rows longer than any routed row; sampled rows only
    ("dense_258_blocks", [257 * 64 + 10], 2, 1, 64, 64, [(0, 0, 0), (0, 0, 128), (0, 0, 256), (0, 0, 257)]),
]


@pytest.mark.parametrize("case", DENSE_CASES, ids=[c[0] for c in DENSE_CASES])
def test_causal_worklist_gives_dense_attention(case):
    name, lengths, H, Hk, d, b, rows = case
    x = synth.gen_prefill(lengths, H, Hk, d, b, 13, "iid", "bf16")
    q, k, v = upload(x)
    sh = shape_of(x, H, Hk)
    wl = bsa.causal_worklist(sh, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    O, lse = bsa.attention_fwd(q, k, v, wl, sh, status)
    torch.cuda.synchronize()
    bsa.check_status(status)
    # CSR: row r of a sequence holds 0 .. r, rows past a sequence's end are empty
    info = oracle.seq_info(x.cu_seqlens, b)
    rp = wl.row_ptr.cpu().numpy()
    lens = np.diff(rp)
    Nq = sh.max_blocks
    for i, (_, _, nb) in enumerate(info):
        for h in range(Hk):
            base = (i * Hk + h) * Nq
            assert list(lens[base:base + Nq]) == [r + 1 for r in range(nb)] + [0] * (Nq - nb)
    ci = wl.col_idx.cpu().numpy()
    for row in (0, Nq - 1, len(lens) - 1):
        if lens[row]:
            assert list(ci[rp[row]:rp[row + 1]]) == list(range(lens[row]))
    bo = wl.bucket_off.cpu().numpy()
    assert bo[-1] == int((lens > 0).sum())
    # dense causal attention through the same kernel
    Ja, ca = oracle.causal_all_blocks(x.cu_seqlens, b, Hk)
    Oo, lo = oracle.attention(oracle_view(x, "q"), oracle_view(x, "k"), oracle_view(x, "v"),
                              x.cu_seqlens, b, H // Hk, Ja, ca, rows=rows)
    mask = ~np.isnan(lo)
    mx, mean, lmx, _, _ = attention_errors(O.float().cpu().numpy(), lse.cpu().numpy(), Oo, lo, mask)
    assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS and lmx <= BF16_LSE_ABS, (mx, mean, lmx)


def test_coverage_matches_oracle():
    lengths, H, Hk, d, b = [900, 400], 8, 2, 128, 64
    x = synth.gen_prefill(lengths, H, Hk, d, b, 17, "iid", "bf16")
    q, k, v = upload(x)
    params = bsa.RouteParams(oracle.TOPK, 4, 0, 0.0, True)
    plan = bsa.PrefillPlan(x.cu_seqlens, H, Hk, d, b, params, device="cuda")
    plan.run(q, k, v)
    C, _, _ = plan.coverage(q, k, v)
    torch.cuda.synchronize()
    bsa.check_status(plan.status)
    Jg = plan.J.cpu().numpy().astype(np.int64)
    cg = plan.counts.cpu().numpy().astype(np.int64)
    Co = oracle.coverage(oracle_view(x, "q"), oracle_view(x, "k"), x.cu_seqlens, b, H // Hk, Jg, cg)
    Cg = C.cpu().numpy()
    assert not np.isnan(Co).any()
    # C = exp(lse_sparse - lse_dense): each lse within BF16_LSE_ABS of float64
    assert np.abs(Cg - Co).max() <= 2 * BF16_LSE_ABS + 1e-4, np.abs(Cg - Co).max()
    assert Cg.min() > 0 and Cg.max() <= 1 + 2 * BF16_LSE_ABS
