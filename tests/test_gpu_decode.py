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
