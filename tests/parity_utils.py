"""Helpers for GPU-vs-oracle parity tests: moving seeded inputs to the device,
running the library through its Python binding, and the tie-aware index compare.

The tolerances are those the spec contract states: router indices and
counts bit-exact up to a 1e-5 tie band on the fp32 scores; BF16 attention
max-abs <= 2e-2 and mean-abs <= 2e-3 against the float64 oracle; FP32 attention
relative error (max |diff| / max |ref|) <= 1e-3 for O and lse.
"""
from __future__ import annotations

import numpy as np
import torch

import dynamic_block_sparse_mean_gb300 as bsa
import oracle
from dynamic_block_sparse_mean_gb300 import synth

TIE_BAND = 1e-5
BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
BF16_LSE_ABS = 1e-3
FP32_REL = 1e-3


def dev_tensor(a: np.ndarray, dtype: str):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def upload(x: synth.PrefillInputs):
    return dev_tensor(x.q, x.dtype), dev_tensor(x.k, x.dtype), dev_tensor(x.v, x.dtype)


def shape_of(x: synth.PrefillInputs, H, Hk):
    dt = torch.bfloat16 if x.dtype == "bf16" else torch.float32
    return bsa.PrefillShape.make(x.cu_seqlens, H, Hk, x.q.shape[2], x.block, dt)


def sample_rows(cu, b, Hk, n_random, seed, all_rows=False):
    """Every sequence's first, last and partial-tail rows for every KV head, plus
    n_random random rows (all rows when all_rows)."""
    info = oracle.seq_info(cu, b)
    if all_rows:
        return oracle.all_rows(cu, b, Hk)
    rows = set()
    for i, (_, n, nb) in enumerate(info):
        for h in range(Hk):
            rows.update({(i, h, 0), (i, h, nb - 1), (i, h, max(0, nb - 2))})
    rng = np.random.default_rng(seed)
    for _ in range(n_random):
        i = int(rng.integers(len(info)))
        rows.add((i, int(rng.integers(Hk)), int(rng.integers(info[i][2]))))
    return sorted(rows)


def check_route_rows(J_gpu, cnt_gpu, J_ora, cnt_ora, g_ora, rows, mode, force_sink,
                     tau_delta=0.0, band=TIE_BAND, window=1, global_blocks=()):
    """Tie-aware comparison of selected sets.

    Forced blocks must be present; each GPU row must be ascending, unique and -1
    padded.  Blocks that the two sides select differently must all lie within
    `band` of the oracle's k-th selected dynamic score (or of tau_r in threshold
    mode); counts must agree exactly in top-k mode and may differ in threshold
    mode only by the number of candidates within `band` of tau_r.  Finally the
    GPU's dynamic set must dominate its complement under the oracle's scores, up
    to the band.  Returns the number of rows whose sets differed (inside the band)."""
    differing = 0
    for (i, h, r) in rows:
        cg, co = int(cnt_gpu[i, h, r]), int(cnt_ora[i, h, r])
        row = [int(x) for x in J_gpu[i, h, r]]
        assert all(x == -1 for x in row[cg:]), (i, h, r, row)
        sg = row[:cg]
        assert sg == sorted(set(sg)), (i, h, r, sg)
        so = [int(x) for x in J_ora[i, h, r, :co]]
        F = oracle.forced_blocks(r, force_sink, window, global_blocks)
        assert F <= set(sg), (i, h, r, sg)
        g = np.asarray(g_ora[i, h, r, :r], dtype=np.float64)
        cand = [j for j in range(r) if j not in F]
        dg, do = set(sg) - F, set(so) - F
        if mode == oracle.TOPK:
            assert cg == co, (i, h, r, cg, co)
        else:
            if cand:
                tau = g[cand].max() - tau_delta
                nb_tau = sum(1 for j in cand if abs(g[j] - tau) <= band)
            else:
                nb_tau = 0
            assert abs(cg - co) <= nb_tau, (i, h, r, cg, co, nb_tau)
        if dg != do:
            differing += 1
            if cg == co and do:
                s_k = min(g[j] for j in do)
                for j in dg ^ do:
                    assert abs(g[j] - s_k) <= band, (i, h, r, j, g[j], s_k)
        rest = [j for j in cand if j not in dg]
        if dg and rest:
            assert min(g[j] for j in dg) >= max(g[j] for j in rest) - band, (i, h, r)
    return differing


def worklist_from_oracle(Jo, co, sh, k_max, status):
    """Build the GPU worklist from the oracle's J and counts (int64 -> int32,
    -1 padded to k_max)."""
    J = torch.as_tensor(Jo.astype(np.int32), device="cuda").contiguous()
    cnt = torch.as_tensor(co.astype(np.int32), device="cuda").contiguous()
    if J.shape[-1] < k_max:
        J = torch.nn.functional.pad(J, (0, k_max - J.shape[-1]), value=-1)
    return bsa.build_worklist(J, cnt, sh, k_max, status)


def expected_csr(Jo, co, cu, b):
    """The CSR row_ptr / col_idx the worklist must hold for the oracle's index:
    rows past a sequence's end are empty, an empty row inside falls back to {r}."""
    B, Hk, Nq = co.shape
    info = oracle.seq_info(cu, b)
    rp, ci = [0], []
    for i in range(B):
        for h in range(Hk):
            for r in range(Nq):
                if r < info[i][2]:
                    ids = [int(v) for v in Jo[i, h, r, :co[i, h, r]]] or [r]
                    ci += ids
                rp.append(len(ci))
    return np.array(rp), np.array(ci)


def capacity(n):
    """A row's capacity bucket: max(4, next power of two of its length)."""
    return max(4, 1 << int(np.ceil(np.log2(max(1, n)))))


def check_buckets(wl, rp):
    """`work` lists every non-empty row once: rows longer than 32 blocks first,
    longest first (lengths above 256 count as 256), then the others by capacity,
    largest first, row-id order among equal keys; each row lies in the bucket of its
    capacity."""
    bo = wl.bucket_off.cpu().numpy()
    work = wl.work.cpu().numpy()[:bo[-1]]
    lens = np.diff(rp)
    rows = np.nonzero(lens)[0].tolist()

    def key(w):
        n = int(lens[w])
        return (0, -min(n, 256), w) if n > 32 else (1, -capacity(n), w)

    assert work.tolist() == sorted(rows, key=key)
    for s in range(7):
        seg = work[bo[s]:bo[s + 1]]
        assert all(capacity(lens[w]) == 256 >> s for w in seg)


def rows_token_mask(cu, b, G, rows, H, T):
    """Boolean [H, T] of the query tokens covered by the given rows."""
    m = np.zeros((H, T), dtype=bool)
    info = oracle.seq_info(cu, b)
    for (i, h, r) in rows:
        s0, n, _ = info[i]
        m[h * G:(h + 1) * G, s0 + r * b: s0 + min(n, (r + 1) * b)] = True
    return m


def attention_errors(O_gpu, lse_gpu, O_ora, lse_ora, mask):
    d = np.abs(O_gpu[mask] - O_ora[mask])
    dl = np.abs(lse_gpu[mask] - lse_ora[mask])
    return float(d.max()), float(d.mean()), float(dl.max()), float(np.abs(O_ora[mask]).max()), \
        float(np.abs(lse_ora[mask]).max())


def check_decode(x, top_k, o, lse, sel, cnt, reqs, G):
    """Decode parity for the requests `reqs`: the kept page set (tie-aware, last
    page always kept), then O and lse within the BF16 tolerances."""
    q64 = synth.bf16_bits_to_f32(x.q).astype(np.float64)
    oo, lo, so, co, sc = oracle.decode(q64, BF16View(x.k_cache), BF16View(x.v_cache),
                                       x.block_table, x.context_lens, x.page_size, top_k,
                                       reqs=reqs, return_scores=True)
    Hk = x.k_cache.shape[1]
    for rho in reqs:
        for h in range(Hk):
            n = int(x.context_lens[rho])
            L = (n + 63) // 64
            cg = int(cnt[rho, h])
            assert cg == int(co[rho, h]) == min(top_k, L - 1) + 1
            sg = [int(v) for v in sel[rho, h, :cg]]
            assert sg == sorted(set(sg)) and sg[-1] == L - 1
            assert all(int(v) == -1 for v in sel[rho, h, cg:])
            dg, do = set(sg[:-1]), set(int(v) for v in so[rho, h, :cg - 1])
            g = sc[(rho, h)]
            if dg != do:
                s_k = min(g[j] for j in do)
                for j in dg ^ do:
                    assert abs(g[j] - s_k) <= TIE_BAND
    rows = np.array(list(reqs))
    d = np.abs(o[rows].astype(np.float64) - oo[rows])
    assert d.max() <= BF16_MAX_ABS and d.mean() <= BF16_MEAN_ABS, (d.max(), d.mean())
    assert np.abs(lse[rows] - lo[rows]).max() <= BF16_LSE_ABS


class BF16View:
    """Index a bf16-bit uint16 array and get float64 values back (converts only
    the requested slice), so the oracle can walk full-size inputs."""

    def __init__(self, bits: np.ndarray):
        self.bits = bits
        self.shape = bits.shape

    def __getitem__(self, idx):
        return synth.bf16_bits_to_f32(np.ascontiguousarray(self.bits[idx])).astype(np.float64)


def oracle_view(x: synth.PrefillInputs, name: str):
    a = getattr(x, name)
    return BF16View(a) if x.dtype == "bf16" else a.astype(np.float64)
