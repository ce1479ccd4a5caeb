"""GPU parity on the edge cases of the method, through the C ABI, against the
float64 oracle: empty sequences inside, before and after a packed batch, one-key
sequences, a block plus one key, the largest row capacity (k_max = 256) with more
history blocks than a row holds, and the largest decode head count and page budget.

[P2] section 1 (packed batch of ragged lengths, N_q = ceil(n / b)), §2.1 (a row
keeps at most k_max blocks, eq.(7)), §4.1 (partial tail blocks).
"""
import numpy as np
import pytest
import torch

import dynamic_block_sparse_mean_gb300 as bsa
import oracle
from dynamic_block_sparse_mean_gb300 import synth
from parity_utils import (BF16_LSE_ABS, BF16_MAX_ABS, BF16_MEAN_ABS, FP32_REL, attention_errors,
                          check_buckets, check_decode, check_route_rows, dev_tensor, expected_csr,
                          oracle_view, rows_token_mask, sample_rows, shape_of, upload,
                          worklist_from_oracle)

pytestmark = pytest.mark.gpu

# (name, lengths, H, H_kv, d, b, mode, k_max, k_min, tau_delta, sink, rows of the
# attention check: None = every row, else the number of random rows added to every
# sequence's first, last and tail rows)
EDGE_CASES = [
    ("empty_and_one_key_b64", [1, 0, 65, 64, 0, 2049, 63], 4, 2, 128, 64, oracle.TOPK, 4, 0, 0.0,
     True, None),
    ("leading_trailing_empty_b128_d64", [0, 300, 1, 0], 4, 1, 64, 128, oracle.THRESHOLD, 3, 1,
     1.0, False, None),
    # 300 blocks: rows past 255 choose 256 of up to 299 candidates
    ("kmax256_topk_b64_d64", [19200, 100], 2, 1, 64, 64, oracle.TOPK, 256, 0, 0.0, False, 12),
    # every candidate passes the threshold, so the k_max clamp of eq.(7) decides
    ("kmax256_threshold_b128", [33280], 2, 2, 128, 128, oracle.THRESHOLD, 256, 8, 1.0e4, True, 8),
]
IDS = [c[0] for c in EDGE_CASES]


def _setup(case, dtype="bf16", seed=5):
    name, lengths, H, Hk, d, b, mode, k_max, k_min, tau, sink, _ = case
    x = synth.gen_prefill(lengths, H, Hk, d, b, seed, "iid", dtype)
    q, k, v = upload(x)
    sh = shape_of(x, H, Hk)
    params = bsa.RouteParams(mode, k_max, k_min, tau, sink)
    return x, q, k, v, sh, params


def _oracle_route(x, params, G, dtype="bf16"):
    if dtype == "bf16":
        Qo, Ko = oracle_view(x, "q"), oracle_view(x, "k")
    else:
        Qo, Ko = x.q.astype(np.float64), x.k.astype(np.float64)
    return oracle.route(Qo, Ko, x.cu_seqlens, x.block, G, params.mode, params.k_max,
                        params.k_min, params.tau_delta, params.force_sink)


@pytest.mark.parametrize("case", EDGE_CASES, ids=IDS)
def test_edge_summaries_router_worklist(case):
    x, q, k, v, sh, params = _setup(case)
    H, Hk = case[2], case[3]
    C = bsa.block_summaries(k, sh)
    J, cnt = bsa.route(q, C, sh, params)
    torch.cuda.synchronize()
    Jo, co, go, Co = _oracle_route(x, params, H // Hk)
    Cg = C.cpu().numpy()
    assert Cg.shape == Co.shape
    assert np.abs(Cg - Co).max() < 1e-5          # zero rows of empty sequences included
    rows = oracle.all_rows(x.cu_seqlens, x.block, Hk)
    Jg, cg = J.cpu().numpy(), cnt.cpu().numpy()
    check_route_rows(Jg, cg, Jo, co, go, rows, params.mode, params.force_sink, params.tau_delta)
    for i, (_, n, nb) in enumerate(oracle.seq_info(x.cu_seqlens, x.block)):
        assert (cg[i, :, nb:] == 0).all() and (Jg[i, :, nb:] == -1).all(), (i, n)
    if params.k_max == 256:
        assert cg.max() == 256                    # the capacity was reached
    # the worklist of the GPU's own index
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wl = bsa.build_worklist(J, cnt, sh, params.k_max, status)
    torch.cuda.synchronize()
    bsa.check_status(status)
    rp, ci = expected_csr(Jg, cg, x.cu_seqlens, x.block)
    assert np.array_equal(wl.row_ptr.cpu().numpy(), rp)
    assert np.array_equal(wl.col_idx.cpu().numpy()[:len(ci)], ci)
    check_buckets(wl, rp)


@pytest.mark.parametrize("case", EDGE_CASES, ids=IDS)
def test_edge_attention_bf16(case):
    x, q, k, v, sh, params = _setup(case)
    H, Hk = case[2], case[3]
    G = H // Hk
    Jo, co, _, _ = _oracle_route(x, params, G)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wl = worklist_from_oracle(Jo, co, sh, params.k_max, status)
    O, lse = bsa.attention_fwd(q, k, v, wl, sh, status)
    torch.cuda.synchronize()
    bsa.check_status(status)
    n_random = case[11]
    rows = sample_rows(x.cu_seqlens, x.block, Hk, n_random or 0, 3, all_rows=n_random is None)
    Oo, lo = oracle.attention(oracle_view(x, "q"), oracle_view(x, "k"), oracle_view(x, "v"),
                              x.cu_seqlens, x.block, G, Jo, co, rows=rows)
    mask = rows_token_mask(x.cu_seqlens, x.block, G, rows, H, x.q.shape[1])
    mx, mean, lmx, _, _ = attention_errors(O.float().cpu().numpy(), lse.cpu().numpy(), Oo, lo, mask)
    assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS and lmx <= BF16_LSE_ABS, (mx, mean, lmx)


@pytest.mark.parametrize("case", EDGE_CASES[:2], ids=IDS[:2])
def test_edge_attention_fp32_and_router(case):
    x, q, k, v, sh, params = _setup(case, dtype="fp32")
    H, Hk = case[2], case[3]
    G = H // Hk
    Jo, co, go, _ = _oracle_route(x, params, G, "fp32")
    C = bsa.block_summaries(k, sh)
    J, cnt = bsa.route(q, C, sh, params)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wl = worklist_from_oracle(Jo, co, sh, params.k_max, status)
    O, lse = bsa.attention_fwd(q, k, v, wl, sh, status)
    torch.cuda.synchronize()
    bsa.check_status(status)
    check_route_rows(J.cpu().numpy(), cnt.cpu().numpy(), Jo, co, go,
                     oracle.all_rows(x.cu_seqlens, x.block, Hk), params.mode, params.force_sink,
                     params.tau_delta)
    Qo, Ko, Vo = (getattr(x, n).astype(np.float64) for n in "qkv")
    Oo, lo = oracle.attention(Qo, Ko, Vo, x.cu_seqlens, x.block, G, Jo, co)
    assert np.abs(O.cpu().numpy() - Oo).max() / np.abs(Oo).max() <= FP32_REL
    assert np.abs(lse.cpu().numpy() - lo).max() / np.abs(lo).max() <= FP32_REL


@pytest.mark.parametrize("case,dtype,tol", [(EDGE_CASES[0], "bf16", 2e-2),
                                            (EDGE_CASES[1], "fp32", 1e-3)], ids=IDS[:2])
def test_edge_backward(case, dtype, tol):
    x, q, k, v, sh, params = _setup(case, dtype=dtype)
    H, Hk = case[2], case[3]
    G = H // Hk
    Jo, co, _, _ = _oracle_route(x, params, G, dtype)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wl = worklist_from_oracle(Jo, co, sh, params.k_max, status)
    O, lse = bsa.attention_fwd(q, k, v, wl, sh, status)
    dO_f = np.random.default_rng(9).normal(size=x.q.shape).astype(np.float32)
    if dtype == "bf16":
        bits = synth.f32_to_bf16_bits(dO_f)
        do, dO64 = dev_tensor(bits, "bf16"), synth.bf16_bits_to_f32(bits).astype(np.float64)
        Qo, Ko, Vo = (oracle_view(x, n) for n in "qkv")
    else:
        do, dO64 = dev_tensor(dO_f, "fp32"), dO_f.astype(np.float64)
        Qo, Ko, Vo = (getattr(x, n).astype(np.float64) for n in "qkv")
    dq, dk, dv = bsa.attention_bwd(q, k, v, O, do, lse, wl, sh)
    torch.cuda.synchronize()
    bsa.check_status(status)
    gq, gk, gv = oracle.attention_backward(Qo, Ko, Vo, x.cu_seqlens, x.block, G, Jo, co, dO64)
    for got, ref, what in ((dq, gq, "dQ"), (dk, gk, "dK"), (dv, gv, "dV")):
        err = np.abs(got.float().cpu().numpy().astype(np.float64) - ref).max() / np.abs(ref).max()
        assert err <= tol, (what, err)


def test_edge_plan_with_empty_sequences():
    """The public PrefillPlan over a batch with empty and one-key sequences."""
    case = EDGE_CASES[0]
    x, q, k, v, sh, params = _setup(case)
    H, Hk = case[2], case[3]
    plan = bsa.PrefillPlan(x.cu_seqlens, H, Hk, case[4], case[5], params)
    O, lse = plan.run(q, k, v)
    torch.cuda.synchronize()
    bsa.check_status(plan.status)
    Jg, cg = plan.J.cpu().numpy(), plan.counts.cpu().numpy()
    Jo, co, go, _ = _oracle_route(x, params, H // Hk)
    check_route_rows(Jg, cg, Jo, co, go, oracle.all_rows(x.cu_seqlens, x.block, Hk), params.mode,
                     params.force_sink)
    Oo, lo = oracle.attention(oracle_view(x, "q"), oracle_view(x, "k"), oracle_view(x, "v"),
                              x.cu_seqlens, x.block, H // Hk, Jg, cg)
    mx, mean, lmx, _, _ = attention_errors(O.float().cpu().numpy(), lse.cpu().numpy(), Oo, lo,
                                           np.ones(lo.shape, dtype=bool))
    assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS and lmx <= BF16_LSE_ABS


def _decode(x, top_k, G):
    q, kc, vc = (dev_tensor(a, "bf16") for a in (x.q, x.k_cache, x.v_cache))
    bt = torch.as_tensor(x.block_table, device="cuda")
    cl = torch.as_tensor(x.context_lens, device="cuda")
    ps = bsa.page_summaries(kc, bt, cl)
    o, lse, sel, cnt = bsa.decode_paged(q, kc, vc, ps, bt, cl, top_k=top_k)
    torch.cuda.synchronize()
    check_decode(x, top_k, o.float().cpu().numpy(), lse.cpu().numpy(), sel.cpu().numpy(),
                 cnt.cpu().numpy(), range(len(x.context_lens)), G)


def test_decode_largest_heads_and_page_budget():
    """H = 256 query heads over 32 KV heads (G = 8), top_k = 64: one key, one
    page exactly, one key past a page, history exactly top_k pages, and more
    history than top_k."""
    lens = [1, 64, 65, 64 * 65, 5000, 4097]
    x = synth.gen_decode(lens, 256, 32, 128, 64, seed=61, max_pages=80)
    _decode(x, 64, 8)


def test_decode_one_page_budget_mha():
    """G = 1 (64 KV heads, one query head each) with top_k = 1."""
    x = synth.gen_decode([1, 129, 3000, 640], 64, 64, 128, 64, seed=62)
    _decode(x, 1, 1)
