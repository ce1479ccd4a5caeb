"""GPU parity of the chunked prefill over a paged KV cache ("2.1 · 粗粒度选择" §3.1:
summaries are cache state beside the KV cache, logical block ids mapped through a
block table; §2.2: routing a query block needs only its history's summaries),
through the C ABI, against the float64 oracle and against the single-pass prefill.

A prompt batch is cut into steps; in every step each sequence adds a chunk that
starts on the page grid (or adds nothing: an idle sequence, whose prefix may end
anywhere).  The chunk's keys and values are appended to the cache, its query
blocks routed against the cached summaries, and the selected pages attended.
"""
import numpy as np
import pytest
import torch

import dynamic_block_sparse_mean_gb300 as bsa
import oracle
from dynamic_block_sparse_mean_gb300 import synth
from parity_utils import (BF16_LSE_ABS, BF16_MAX_ABS, BF16_MEAN_ABS, BF16View, attention_errors,
                          check_route_rows, oracle_view, upload)

pytestmark = pytest.mark.gpu

PAGE = 64

# (name, chunk boundaries per sequence (token offsets, one list per sequence, equal
# numbers of steps), H, H_kv, d, route parameters)
CASES = [
    ("gqa4_d128_topk_sink", [[0, 512, 1024, 1500], [0, 128, 128, 700], [0, 64, 64, 64],
                             [0, 100, 100, 100]], 8, 2, 128,
     dict(mode=oracle.TOPK, k_max=6, force_sink=True)),
    ("gqa2_d64_threshold_union", [[0, 256, 1280, 2000], [0, 0, 640, 901]], 4, 2, 64,
     dict(mode=oracle.THRESHOLD, k_max=10, k_min=2, tau_delta=2.0, window=2,
          global_blocks=(1, 4))),
    # the same chunking with the router's score screen forced on (bounded screened
    # scores, exact rescoring of the candidates at the boundary)
    ("gqa4_d128_topk_sink_screened", [[0, 512, 1024, 1500], [0, 128, 128, 700], [0, 64, 64, 64],
                                      [0, 100, 100, 100]], 8, 2, 128,
     dict(mode=oracle.TOPK, k_max=6, force_sink=True, screen=1)),
]
IDS = [c[0] for c in CASES]


def _setup(case, seed=17):
    name, bounds, H, Hk, d, rp = case
    lengths = [bd[-1] for bd in bounds]
    x = synth.gen_prefill(lengths, H, Hk, d, PAGE, seed, "iid", "bf16")
    pages = [(n + PAGE - 1) // PAGE for n in lengths]
    perm = np.random.default_rng(seed).permutation(sum(pages) + 3)   # 3 pages nobody uses
    bt = np.full((len(lengths), max(pages) + 2), -1, dtype=np.int32)
    off = 0
    for i, L in enumerate(pages):
        bt[i, :L] = perm[off:off + L]
        off += L
    cache = bsa.PagedKVCache.allocate(len(perm), Hk, d, bt)
    params = bsa.RouteParams(**rp)
    return x, bounds, cache, params


def _step_inputs(x, bounds, step, q, k, v):
    """Chunk `step` of every sequence, packed: (prefix, lens, chunk tensors)."""
    cu = x.cu_seqlens
    pre = [bd[step] for bd in bounds]
    lens = [bd[step + 1] - bd[step] for bd in bounds]
    idx = np.concatenate([np.arange(cu[i] + pre[i], cu[i] + pre[i] + lens[i])
                          for i in range(len(bounds))]).astype(np.int64)
    ti = torch.as_tensor(idx, device="cuda")
    return pre, lens, q[:, ti].contiguous(), k[:, ti].contiguous(), v[:, ti].contiguous()


def _run_chunks(case):
    """Every step through ChunkPlan; returns the inputs and, per step, the chunk's
    (prefix, lens, J, counts, O, lse) on the host."""
    x, bounds, cache, params = _setup(case)
    H, Hk, d = case[2], case[3], case[4]
    q, k, v = upload(x)
    nsteps = len(bounds[0]) - 1
    max_ctx = (max(bd[-1] for bd in bounds) + PAGE - 1) // PAGE
    out = []
    for step in range(nsteps):
        pre, lens, qc, kc, vc = _step_inputs(x, bounds, step, q, k, v)
        if sum(lens) == 0:
            continue
        chunk = bsa.Chunk.make(pre, lens, H, Hk, d, max_context_blocks=max_ctx)
        plan = bsa.ChunkPlan(chunk, cache, params)
        O, lse = plan.run(qc, kc, vc)
        torch.cuda.synchronize()
        bsa.check_status(plan.status)
        out.append((pre, lens, plan.J.cpu().numpy(), plan.counts.cpu().numpy(),
                    O.float().cpu().numpy(), lse.cpu().numpy()))
    return x, cache, params, out


def _to_full_rows(x, steps, Hk, k_max):
    """The chunks' J / counts placed at their logical rows of a single-pass J."""
    info = oracle.seq_info(x.cu_seqlens, PAGE)
    Nq = max(nb for _, _, nb in info)
    J = np.full((len(info), Hk, Nq, k_max), -1, dtype=np.int64)
    cnt = np.zeros((len(info), Hk, Nq), dtype=np.int64)
    rows = []
    for pre, lens, Jc, cc, _, _ in steps:
        for i in range(len(lens)):
            nq = (lens[i] + PAGE - 1) // PAGE
            r0 = pre[i] // PAGE
            J[i, :, r0:r0 + nq] = Jc[i, :, :nq]
            cnt[i, :, r0:r0 + nq] = cc[i, :, :nq]
            rows += [(i, h, r) for h in range(Hk) for r in range(r0, r0 + nq)]
    return J, cnt, sorted(rows)


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_chunk_append_fills_pages_and_summaries(case):
    x, cache, params, _ = _run_chunks(case)
    Hk = case[3]
    K = BF16View(x.k)
    kc = cache.k_cache.cpu().view(torch.int16).numpy().view(np.uint16)
    vcache = cache.v_cache.cpu().view(torch.int16).numpy().view(np.uint16)
    ps = cache.page_summ.cpu().numpy()
    psum = cache.page_sum.cpu().numpy()
    bt = cache.block_table.cpu().numpy()
    Co = oracle.block_summaries(K, x.cu_seqlens, PAGE)
    for i, (s0, n, nb) in enumerate(oracle.seq_info(x.cu_seqlens, PAGE)):
        for p in range(nb):
            phys, lo, hi = bt[i, p], s0 + p * PAGE, s0 + min(n, (p + 1) * PAGE)
            # keys and values copied bit for bit; the last page's free slots zeroed
            assert np.array_equal(kc[phys, :, :hi - lo], x.k[:, lo:hi])
            assert np.array_equal(vcache[phys, :, :hi - lo], x.v[:, lo:hi])
            assert (kc[phys, :, hi - lo:] == 0).all() and (vcache[phys, :, hi - lo:] == 0).all()
            # eq.(11): mean of the page's keys, and the running sum beside it
            assert np.abs(ps[phys] - Co[i, :, p]).max() < 1e-5
            assert np.abs(psum[phys] - Co[i, :, p] * (hi - lo)).max() < 1e-5 * (hi - lo)
    unused = sorted(set(range(cache.k_cache.shape[0])) - set(bt[bt >= 0].tolist()))
    assert unused and (ps[unused] == 0).all()        # pages nobody owns are untouched


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_chunked_router_matches_oracle(case):
    x, cache, params, steps = _run_chunks(case)
    H, Hk = case[2], case[3]
    Jg, cg, rows = _to_full_rows(x, steps, Hk, params.k_max)
    Jo, co, go, _ = oracle.route(oracle_view(x, "q"), oracle_view(x, "k"), x.cu_seqlens, PAGE,
                                 H // Hk, params.mode, params.k_max, params.k_min,
                                 params.tau_delta, params.force_sink, window=params.window,
                                 global_blocks=params.global_blocks)
    assert rows == oracle.all_rows(x.cu_seqlens, PAGE, Hk)     # every row routed exactly once
    check_route_rows(Jg, cg, Jo, co, go, rows, params.mode, params.force_sink, params.tau_delta,
                     window=params.window, global_blocks=params.global_blocks)


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_chunked_attention_matches_oracle(case):
    """Each chunk's O / lse against the oracle's attention of the whole prompt on
    the index the GPU chose (so ties cannot move the comparison); the oracle's
    chunked prefill equals that single-pass result by its own pin."""
    x, cache, params, steps = _run_chunks(case)
    H, Hk = case[2], case[3]
    G = H // Hk
    Jg, cg, rows = _to_full_rows(x, steps, Hk, params.k_max)
    Oo, lo = oracle.attention(oracle_view(x, "q"), oracle_view(x, "k"), oracle_view(x, "v"),
                              x.cu_seqlens, PAGE, G, Jg, cg, rows=rows)
    cu = x.cu_seqlens
    for pre, lens, _, _, O, lse in steps:
        ccu = np.concatenate([[0], np.cumsum(lens)])
        for i in range(len(lens)):
            if lens[i] == 0:
                continue
            full = slice(cu[i] + pre[i], cu[i] + pre[i] + lens[i])
            got = slice(ccu[i], ccu[i + 1])
            d = np.abs(O[:, got] - Oo[:, full])
            assert d.max() <= BF16_MAX_ABS and d.mean() <= BF16_MEAN_ABS, (i, d.max(), d.mean())
            assert np.abs(lse[:, got] - lo[:, full]).max() <= BF16_LSE_ABS


def test_chunk_attention_on_oracle_chunk_index():
    """bsa_build_worklist_chunk + bsa_attention_chunk fed the oracle's own chunked
    J (oracle.chunked_prefill over the GPU-written cache) give its O and lse."""
    case = CASES[0]
    x, cache, params, _ = _run_chunks(case)
    H, Hk, d = case[2], case[3], case[4]
    bounds = case[1]
    q, k, v = upload(x)
    kc, vc = BF16View(cache.k_cache.cpu().view(torch.int16).numpy().view(np.uint16)), \
        BF16View(cache.v_cache.cpu().view(torch.int16).numpy().view(np.uint16))
    bt = cache.block_table.cpu().numpy()
    pre, lens, qc, _, _ = _step_inputs(x, bounds, 2, q, k, v)       # the last step
    ccu = np.concatenate([[0], np.cumsum(lens)])
    qh = synth.bf16_bits_to_f32(qc.cpu().view(torch.int16).numpy().view(np.uint16))
    Jo, co, Oo, lo = oracle.chunked_prefill(qh.astype(np.float64), kc, vc, bt, pre, ccu, PAGE,
                                            H // Hk, params.mode, params.k_max,
                                            force_sink=params.force_sink)
    chunk = bsa.Chunk.make(pre, lens, H, Hk, d,
                           max_context_blocks=(max(bd[-1] for bd in bounds) + 63) // 64)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    J = torch.as_tensor(Jo.astype(np.int32), device="cuda").contiguous()
    cnt = torch.as_tensor(co.astype(np.int32), device="cuda").contiguous()
    wl = bsa.build_worklist_chunk(J, cnt, chunk, cache, params.k_max, status)
    O, lse = bsa.attention_chunk(qc, wl, chunk, cache, status)
    torch.cuda.synchronize()
    bsa.check_status(status)
    mask = np.zeros(lo.shape, dtype=bool)
    mask[:, :ccu[-1]] = True
    mx, mean, lmx, _, _ = attention_errors(O.float().cpu().numpy(), lse.cpu().numpy(), Oo, lo, mask)
    assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS and lmx <= BF16_LSE_ABS, (mx, mean, lmx)


@pytest.mark.parametrize("case", [CASES[0], CASES[2]], ids=[CASES[0][0], CASES[2][0]])
def test_chunked_equals_single_pass_bit_for_bit(case):
    """The summaries of appended pages, the router's scores and the attention
    tiles are the single-pass ones in the same order, so the chunked J and O equal
    the single-pass PrefillPlan's exactly."""
    x, cache, params, steps = _run_chunks(case)
    H, Hk, d = case[2], case[3], case[4]
    q, k, v = upload(x)
    plan = bsa.PrefillPlan(x.cu_seqlens, H, Hk, d, PAGE, params)
    O1, lse1 = plan.run(q, k, v)
    torch.cuda.synchronize()
    bsa.check_status(plan.status)
    Jg, cg, rows = _to_full_rows(x, steps, Hk, params.k_max)
    J1, c1 = plan.J.cpu().numpy(), plan.counts.cpu().numpy()
    for (i, h, r) in rows:
        assert cg[i, h, r] == c1[i, h, r]
        assert np.array_equal(Jg[i, h, r, :cg[i, h, r]], J1[i, h, r, :c1[i, h, r]])
    O1, lse1 = O1.float().cpu().numpy(), lse1.cpu().numpy()
    cu = x.cu_seqlens
    for pre, lens, _, _, O, lse in steps:
        ccu = np.concatenate([[0], np.cumsum(lens)])
        for i in range(len(lens)):
            full = slice(cu[i] + pre[i], cu[i] + pre[i] + lens[i])
            assert np.array_equal(O[:, ccu[i]:ccu[i + 1]], O1[:, full])
            assert np.array_equal(lse[:, ccu[i]:ccu[i + 1]], lse1[:, full])


def test_chunk_rejects_prefix_off_the_page_grid():
    """A chunk whose prefix is not whole pages (or whose context passes N_k) is
    reported in dev_status (BSA_ERR_CACHE) and contributes no rows; the other
    sequences of the batch are routed as usual."""
    H, Hk, d = 4, 2, 128
    x = synth.gen_prefill([300, 200], H, Hk, d, PAGE, 3, "iid", "bf16")
    q, k, v = upload(x)
    bt = np.arange(16, dtype=np.int32).reshape(2, 8)
    cache = bsa.PagedKVCache.allocate(16, Hk, d, bt)
    params = bsa.RouteParams(oracle.TOPK, 4)
    for pre, lens in (([0, 100], [300, 100]),        # second prefix off the grid
                      ([0, 448], [300, 100])):       # second context past N_k = 8
        chunk = bsa.Chunk.make(pre, lens, H, Hk, d, max_context_blocks=8)
        plan = bsa.ChunkPlan(chunk, cache, params)
        qc, kc, vc = (t[:, :400].contiguous() for t in (q, k, v))
        plan.run(qc, kc, vc)
        torch.cuda.synchronize()
        assert int(plan.status.item()) == 20
        cnt = plan.counts.cpu().numpy()
        assert (cnt[1] == 0).all() and (cnt[0, :, :5] > 0).all()
        assert int(plan.wl.bucket_off[-1].item()) == 5 * Hk     # only the first sequence's rows
