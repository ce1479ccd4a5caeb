"""GPU parity of the paged decode path against the float64 oracle."""
import numpy as np
import pytest
import torch

import dynamic_block_sparse_mean_gb300 as bsa
import oracle
from dynamic_block_sparse_mean_gb300 import synth
from parity_utils import BF16View, check_decode, dev_tensor

pytestmark = pytest.mark.gpu


def _upload(x):
    return (dev_tensor(x.q, "bf16"), dev_tensor(x.k_cache, "bf16"), dev_tensor(x.v_cache, "bf16"),
            torch.as_tensor(x.block_table, device="cuda"),
            torch.as_tensor(x.context_lens, device="cuda"))


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_decode_small(G):
    Hk = 2
    rng = np.random.default_rng(G)
    lens = rng.integers(1, 4000, size=7)
    lens[0], lens[1] = 64, 65          # one page exactly; a second page with one key
    x = synth.gen_decode(lens, G * Hk, Hk, 128, 64, seed=30 + G, max_pages=70)
    q, kc, vc, bt, cl = _upload(x)
    ps = bsa.page_summaries(kc, bt, cl)
    top_k = 8
    o, lse, sel, cnt = bsa.decode_paged(q, kc, vc, ps, bt, cl, top_k=top_k)
    torch.cuda.synchronize()
    check_decode(x, top_k, o.float().cpu().numpy(), lse.cpu().numpy(), sel.cpu().numpy(),
                 cnt.cpu().numpy(), range(len(lens)), G)


def test_page_summaries_match_page_means():
    x = synth.gen_decode([130, 64, 1000], 4, 2, 128, 64, seed=40)
    q, kc, vc, bt, cl = _upload(x)
    ps = bsa.page_summaries(kc, bt, cl).cpu().numpy()
    kv = BF16View(x.k_cache)
    for rho, n in enumerate(x.context_lens):
        L = (n + 63) // 64
        for p in range(L):
            phys = x.block_table[rho, p]
            valid = min(64, n - 64 * p)
            ref = kv[phys][:, :valid].mean(axis=1)            # [H_kv, d]
            assert np.abs(ps[phys] - ref).max() < 1e-5


def test_decode_every_page_selected_matches_dense():
    """top_k >= pages: every page is read, so decode is dense attention."""
    x = synth.gen_decode([500, 1200], 8, 2, 128, 64, seed=41)
    q, kc, vc, bt, cl = _upload(x)
    ps = bsa.page_summaries(kc, bt, cl)
    o, lse, sel, cnt = bsa.decode_paged(q, kc, vc, ps, bt, cl, top_k=64)
    torch.cuda.synchronize()
    check_decode(x, 64, o.float().cpu().numpy(), lse.cpu().numpy(), sel.cpu().numpy(),
                 cnt.cpu().numpy(), range(2), 4)


def test_streaming_page_summaries_follow_eq11():
    # Keys appended one per step from empty pages (eq.(11): s <- s + k, c = s / r);
    # the lengths cross page boundaries (page 64) in both directions.
    final = np.array([63, 64, 65, 130, 1, 200])
    x = synth.gen_decode(final, 4, 2, 128, 64, seed=51, max_pages=4)
    q, kc, vc, bt, cl = _upload(x)
    P, Hk, page, d = kc.shape
    psum = torch.zeros(P, Hk, d, dtype=torch.float32, device="cuda")
    summ = torch.zeros(P, Hk, d, dtype=torch.float32, device="cuda")
    for t in range(int(final.max())):
        lens_t = np.where(t < final, t + 1, 0).astype(np.int32)   # 0: no append this step
        bsa.page_summaries_append(kc, bt, torch.as_tensor(lens_t, device="cuda"), psum, summ)
    torch.cuda.synchronize()
    batch = bsa.page_summaries(kc, bt, cl)
    sg, bg = summ.cpu().numpy(), batch.cpu().numpy()
    kf = synth.bf16_bits_to_f32(x.k_cache).astype(np.float64)
    for rho, n in enumerate(final):
        for p in range((n + 63) // 64):
            phys = int(x.block_table[rho, p])
            keys = kf[phys, :, :min(64, n - p * 64)]        # the page's valid keys, in order
            for h in range(Hk):
                want = oracle.streaming_summary(keys[h])[-1]
                assert np.abs(sg[phys, h] - want).max() < 1e-5
                assert np.abs(sg[phys, h] - bg[phys, h]).max() < 1e-5


BSA_ERR_CACHE = 20


def _run_plan(x, top_k, cl=None, bt=None):
    q, kc, vc, bt0, cl0 = _upload(x)
    bt = bt0 if bt is None else torch.as_tensor(bt, device="cuda")
    cl = cl0 if cl is None else torch.as_tensor(np.asarray(cl, dtype=np.int32), device="cuda")
    ps = bsa.page_summaries(kc, bt, cl)
    R, H, d = q.shape
    P, Hk, page, _ = kc.shape
    plan = bsa.DecodePlan(R, H, Hk, d, page, bt.shape[1], P, top_k)
    plan.sel.fill_(777)                      # sentinel: every row must be rewritten
    plan.sel_counts.fill_(777)
    plan.run(q, kc, vc, ps, bt, cl)
    torch.cuda.synchronize()
    return (plan.out.float().cpu().numpy(), plan.lse.cpu().numpy(), plan.sel.cpu().numpy(),
            plan.sel_counts.cpu().numpy(), int(plan.status.item()))


def _assert_empty(o, lse, sel, cnt, rho):
    assert (cnt[rho] == 0).all() and (sel[rho] == -1).all()
    assert (o[rho] == 0).all() and np.isneginf(lse[rho]).all()


def test_decode_idle_and_invalid_lengths():
    """Length 0 is an idle slot (empty result, no error); a length past the block
    table is BSA_ERR_CACHE with the same empty result; neighbours are exact."""
    max_pages = 30
    lens = [700, 0, 1500, 200]
    x = synth.gen_decode(lens, 8, 2, 128, 64, seed=61, max_pages=max_pages)
    o, lse, sel, cnt, st = _run_plan(x, 8)
    assert st == 0
    _assert_empty(o, lse, sel, cnt, 1)
    check_decode(x, 8, o, lse, sel, cnt, [0, 2, 3], 4)

    bad = [700, 0, 1500, max_pages * 64 + 1]     # request 3 overruns its block-table row
    o, lse, sel, cnt, st = _run_plan(x, 8, cl=bad)
    assert st == BSA_ERR_CACHE
    _assert_empty(o, lse, sel, cnt, 1)
    _assert_empty(o, lse, sel, cnt, 3)
    check_decode(x, 8, o, lse, sel, cnt, [0, 2], 4)

    neg = [700, -5, 1500, 200]
    o, lse, sel, cnt, st = _run_plan(x, 8, cl=neg)
    assert st == BSA_ERR_CACHE
    _assert_empty(o, lse, sel, cnt, 1)
    check_decode(x, 8, o, lse, sel, cnt, [0, 2, 3], 4)


def test_decode_page_id_outside_cache():
    """A block-table entry outside [0, P) is reported and never read through: as a
    scored page it scores -inf (not kept); as a kept page it reads zeros."""
    x = synth.gen_decode([900, 2000, 300], 8, 2, 128, 64, seed=62)
    P = x.k_cache.shape[0]
    bt = x.block_table.copy()
    bt[1, 3] = P + 5            # request 1: a scored page among 31 (top 8 kept)
    bt[2, 1] = -7               # request 2: 5 pages, all kept (4 scored <= top_k)
    o, lse, sel, cnt, st = _run_plan(x, 8, bt=bt)
    assert st == BSA_ERR_CACHE
    check_decode(x, 8, o, lse, sel, cnt, [0], 4)
    for h in range(2):
        assert 3 not in sel[1, h, :cnt[1, h]].tolist()
        assert sel[2, h, :cnt[2, h]].tolist() == [0, 1, 2, 3, 4]
    assert np.isfinite(o[1:]).all() and np.isfinite(lse[1:]).all()
