"""Child process of test_gpu_bounds.py: runs the ABI calls at small ragged shapes
with whichever library BSA_BOUNDS_CHECK selects and saves every output to an
.npz; with --corrupt (bounds-checked library only) it also runs the index-reading
calls on tables holding out-of-range entries and saves the status each records.

    python tests/bounds_child.py OUT.npz [--corrupt]
"""
from __future__ import annotations

import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import dynamic_block_sparse_mean_gb300 as bsa  # noqa: E402
import oracle  # noqa: E402
from dynamic_block_sparse_mean_gb300 import _lib, synth  # noqa: E402
from parity_utils import dev_tensor, shape_of, upload  # noqa: E402

LENGTHS = [700, 129, 64, 1, 300]


def host(t):
    t = t.detach()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.cpu().numpy()


def prefill(dtype, d, b, H, Hk, out, tag, corrupt):
    x = synth.gen_prefill(LENGTHS, H, Hk, d, b, 5, "iid", dtype)
    q, k, v = upload(x)
    sh = shape_of(x, H, Hk)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    C = bsa.block_summaries(k, sh)
    J, cnt = bsa.route(q, C, sh, bsa.RouteParams(oracle.TOPK, 4, 0, 0.0, True), dev_status=st)
    wl = bsa.build_worklist(J, cnt, sh, 4, st)
    O, lse = bsa.attention_fwd(q, k, v, wl, sh, st)
    do = dev_tensor(synth.gen_prefill(LENGTHS, H, Hk, d, b, 6, "iid", dtype).q, dtype)
    dq, dk, dv = bsa.attention_bwd(q, k, v, O, do, lse, wl, sh, dev_status=st)
    torch.cuda.synchronize()
    out[f"{tag}_status"] = np.array([int(st.item())])
    for name, t in (("J", J), ("cnt", cnt), ("O", O), ("lse", lse), ("dq", dq), ("dk", dk),
                    ("dv", dv)):
        out[f"{tag}_{name}"] = host(t)
    if not corrupt:
        return
    # Entries below 0, past the row's diagonal and far past the table: each must be
    # reported (BSA_ERR_INDEX_RANGE) and clamped by the bounds-checked kernels.
    col = wl.col_idx.clone()
    n = col.numel()
    bad = torch.tensor([-5, 10 ** 6, 7], dtype=torch.int32, device="cuda")
    pos = torch.tensor([0, n // 2, n - 1], dtype=torch.long, device="cuda")
    col[pos] = bad
    # the last entry of the last row is that row's diagonal; 7 blocks past it
    # is past r whatever r is (rows are causal)
    last_row_r = int(wl.col_idx[n - 1].item())
    col[n - 1] = last_row_r + 7
    bad_wl = bsa.Worklist(wl.row_ptr, col, wl.work, wl.bucket_off)
    for what in ("fwd", "bwd"):
        st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
        if what == "fwd":
            bsa.attention_fwd(q, k, v, bad_wl, sh, st2)
        else:
            bsa.attention_bwd(q, k, v, O, do, lse, bad_wl, sh, dev_status=st2)
        torch.cuda.synchronize()
        out[f"{tag}_corrupt_{what}_status"] = np.array([int(st2.item())])


def decode(out):
    x = synth.gen_decode([900, 0, 3000, 64, 65], 16, 2, 128, 64, seed=7, max_pages=60)
    q = dev_tensor(x.q, "bf16")
    kc, vc = dev_tensor(x.k_cache, "bf16"), dev_tensor(x.v_cache, "bf16")
    bt = torch.as_tensor(x.block_table, device="cuda")
    cl = torch.as_tensor(x.context_lens, device="cuda")
    P, Hk, page, d = kc.shape
    ps = bsa.page_summaries(kc, bt, cl)
    plan = bsa.DecodePlan(q.shape[0], q.shape[1], Hk, d, page, bt.shape[1], P, 8)
    plan.run(q, kc, vc, ps, bt, cl)
    torch.cuda.synchronize()
    out["dec_status"] = np.array([int(plan.status.item())])
    out["dec_out"], out["dec_lse"] = host(plan.out), host(plan.lse)
    out["dec_sel"], out["dec_cnt"] = host(plan.sel), host(plan.sel_counts)


def chunk(out, corrupt):
    H, Hk, d = 8, 2, 128
    lengths = [300, 700, 0]
    x = synth.gen_prefill([1000, 700, 200], H, Hk, d, 64, 9, "iid", "bf16")
    q, k, v = upload(x)
    pages = [16, 11, 4]
    bt = np.full((3, 16), -1, dtype=np.int32)
    perm = np.random.default_rng(1).permutation(sum(pages)).astype(np.int32)
    off = 0
    for i, n in enumerate(pages):
        bt[i, :n] = perm[off:off + n]
        off += n
    P = sum(pages)
    z = lambda *s: torch.zeros(s, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    zf = lambda *s: torch.zeros(s, dtype=torch.float32, device="cuda")  # noqa: E731
    bt_dev = torch.as_tensor(bt, device="cuda")
    cache = bsa.PagedKVCache(z(P, Hk, 64, d), z(P, Hk, 64, d), zf(P, Hk, d), bt_dev,
                             zf(P, Hk, d))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cu = x.cu_seqlens
    idx = np.concatenate([np.arange(cu[i], cu[i] + n) for i, n in enumerate(lengths)])
    ti = torch.as_tensor(idx, device="cuda")
    qc, kc, vc = (t[:, ti].contiguous() for t in (q, k, v))
    ch = bsa.Chunk.make([0, 0, 128], lengths, H, Hk, d, max_context_blocks=16)
    bsa.chunk_append(kc, vc, ch, cache, st)
    params = bsa.RouteParams(oracle.TOPK, 6, 0, 0.0, True)
    J, cnt = bsa.route_chunk(qc, ch, cache, params, st)
    wl = bsa.build_worklist_chunk(J, cnt, ch, cache, 6, st)
    O, lse = bsa.attention_chunk(qc, wl, ch, cache, st)
    torch.cuda.synchronize()
    out["chunk_status"] = np.array([int(st.item())])
    out["chunk_O"], out["chunk_lse"] = host(O), host(lse)
    if not corrupt:
        return
    # a block-table entry past the cache's pages, read by the chunk attention only
    bt_bad = bt.copy()
    bt_bad[1, 0] = P + 1000
    cache.block_table.copy_(torch.as_tensor(bt_bad, device="cuda"))
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsa.attention_chunk(qc, wl, ch, cache, st2)
    torch.cuda.synchronize()
    out["chunk_corrupt_status"] = np.array([int(st2.item())])


def main():
    path = sys.argv[1]
    corrupt = "--corrupt" in sys.argv
    checked = int(_lib.lib().bsa_bounds_checked())
    if corrupt and checked != 1:
        raise SystemExit("--corrupt runs only on the bounds-checked library")
    torch.cuda.set_device(0)
    out = {"bounds_checked": np.array([checked])}
    prefill("bf16", 128, 64, 8, 2, out, "bf16_b64", corrupt)
    prefill("bf16", 128, 128, 8, 2, out, "bf16_b128", corrupt)
    prefill("fp32", 64, 64, 4, 2, out, "fp32_d64", corrupt)
    decode(out)
    chunk(out, corrupt)
    np.savez(path, **out)


if __name__ == "__main__":
    main()
