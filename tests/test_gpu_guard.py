"""Guard bands around every output and workspace buffer of every ABI call.

Each buffer a call writes (outputs, workspaces, status words) is allocated at the
size include/bsa.h states, with 4 KB of a poison byte pattern on both sides; the
call runs at small ragged shapes on the tensor-core and the SIMT paths, and the
poison must be intact afterwards.  A kernel that writes past either end of a
buffer (an index off by one, a row of -1, a tail tile stored in full) shows up
here without any memory checker.
"""
import ctypes

import numpy as np
import pytest
import torch

import dynamic_block_sparse_mean_gb300 as bsa
import oracle
from dynamic_block_sparse_mean_gb300 import _lib, synth
from parity_utils import dev_tensor, shape_of, upload

pytestmark = pytest.mark.gpu

GUARD = 4096
POISON = 0xA5


class Guards:
    """Allocates guarded device buffers and checks all of them at the end."""

    def __init__(self):
        self.bufs = []

    def __call__(self, shape, dtype, fill=None):
        shape = tuple(int(s) for s in np.atleast_1d(shape))
        elem = torch.empty(0, dtype=dtype).element_size()
        nbytes = max(1, int(np.prod(shape))) * elem
        raw = torch.full((GUARD + nbytes + GUARD,), POISON, dtype=torch.uint8, device="cuda")
        view = raw[GUARD:GUARD + nbytes].view(dtype)[:int(np.prod(shape))].view(shape)
        if fill is not None:
            view.fill_(fill)
        self.bufs.append((raw, nbytes, shape, dtype))
        return view

    def ws(self, nbytes):
        return self((max(1, int(nbytes)),), torch.uint8)

    def check(self):
        torch.cuda.synchronize()
        for k, (raw, nbytes, shape, dtype) in enumerate(self.bufs):
            head, tail = raw[:GUARD], raw[GUARD + nbytes:]
            assert bool((head == POISON).all()), f"buffer {k} {shape} {dtype}: written before its start"
            assert bool((tail == POISON).all()), f"buffer {k} {shape} {dtype}: written past its end"


def _status(g):
    return g((1,), torch.int32, 0)


@pytest.mark.parametrize("dtype,d,b,H,Hk", [("bf16", 128, 64, 8, 2), ("bf16", 128, 128, 16, 2),
                                            ("bf16", 64, 64, 4, 4), ("fp32", 64, 64, 4, 2)])
def test_prefill_calls_stay_inside_their_buffers(dtype, d, b, H, Hk):
    g = Guards()
    lengths = [700, 129, 64, 1, 300]
    x = synth.gen_prefill(lengths, H, Hk, d, b, 5, "iid", dtype)
    q, k, v = upload(x)
    sh = shape_of(x, H, Hk)
    B, Nq, T = sh.num_seqs, sh.max_blocks, sh.total_tokens
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    st = _status(g)
    C = g((B, Hk, Nq, d), torch.float32)
    bsa.block_summaries(k, sh, out=C)
    params = bsa.RouteParams(oracle.TOPK, 5, 0, 0.0, True)
    J, cnt = g((B, Hk, Nq, 5), torch.int32), g((B, Hk, Nq), torch.int32)
    ws = g.ws(bsa.route_workspace_bytes(sh, params))
    bsa.route(q, C, sh, params, J=J, counts=cnt, ws=ws, dev_status=st)
    scores = g((B, Hk, Nq, Nq), torch.float32)
    J2, cnt2 = g((B, Hk, Nq, 5), torch.int32), g((B, Hk, Nq), torch.int32)
    bsa.route(q, C, sh, params, J=J2, counts=cnt2, scores=scores, ws=g.ws(
        bsa.route_workspace_bytes(sh, params)), dev_status=st)
    thr = bsa.RouteParams(oracle.THRESHOLD, 8, 2, 2.0, False, window=2, global_blocks=(3,))
    J3, cnt3 = g((B, Hk, Nq, 8), torch.int32), g((B, Hk, Nq), torch.int32)
    bsa.route(q, C, sh, thr, J=J3, counts=cnt3, ws=g.ws(bsa.route_workspace_bytes(sh, thr)),
              dev_status=st)
    rows = sh.num_rows
    s = sh.c()

    def wl_bufs(cap):
        return bsa.Worklist(g((rows + 1,), torch.int32), g((cap,), torch.int32),
                            g((rows,), torch.int32), g((bsa.NUM_BUCKETS + 1,), torch.int32))

    wl = wl_bufs(rows * 5)
    bsa.build_worklist(J, cnt, sh, 5, st, wl=wl,
                       ws=g.ws(_lib.lib().bsa_worklist_workspace_size(ctypes.byref(s), 5)))
    wl_na = wl_bufs(rows * 5)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    assert _lib.lib().bsa_build_worklist_noalloc(
        ctypes.byref(s), 5, p(J), p(cnt), p(wl_na.row_ptr), p(wl_na.col_idx), p(wl_na.work),
        p(wl_na.bucket_off), p(st), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    O, lse = g((H, T, d), tdt), g((H, T), torch.float32)
    bsa.attention_fwd(q, k, v, wl, sh, st, out=O, lse=lse)
    cap = int(_lib.lib().bsa_causal_worklist_capacity(ctypes.byref(s)))
    dwl = wl_bufs(cap)
    bsa.causal_worklist(sh, "cuda", wl=dwl,
                        ws=g.ws(_lib.lib().bsa_worklist_workspace_size(ctypes.byref(s), 1)))
    Od, ld = g((H, T, d), tdt), g((H, T), torch.float32)
    bsa.attention_fwd(q, k, v, dwl, sh, st, out=Od, lse=ld)
    cov = g((H, T), torch.float32)
    bsa.coverage(lse, ld, sh, out=cov)
    hits = g((H, T), torch.int32, -1)
    bsa.token_recall(q, k, J, cnt, sh, 16, hits=hits, dev_status=st)
    do = dev_tensor(synth.gen_prefill(lengths, H, Hk, d, b, 6, "iid", dtype).q, dtype)
    dq, dk, dv = g((H, T, d), tdt), g((Hk, T, d), tdt), g((Hk, T, d), tdt)
    bsa.attention_bwd(q, k, v, O, do, lse, wl, sh, dq=dq, dk=dk, dv=dv,
                      ws=g.ws(_lib.lib().bsa_attention_bwd_workspace_size(ctypes.byref(s))),
                      dev_status=st)
    bsa.selftest_wait_timeout(st)
    g.check()
    assert int(st.item()) == 19          # only the self-test's timeout was recorded


def test_decode_calls_stay_inside_their_buffers():
    g = Guards()
    lens = [900, 0, 3000, 64, 65]
    x = synth.gen_decode(lens, 16, 2, 128, 64, seed=7, max_pages=60)
    q = dev_tensor(x.q, "bf16")
    kc, vc = dev_tensor(x.k_cache, "bf16"), dev_tensor(x.v_cache, "bf16")
    bt = torch.as_tensor(x.block_table, device="cuda")
    cl = torch.as_tensor(x.context_lens, device="cuda")
    P, Hk, page, d = kc.shape
    R, H = q.shape[0], q.shape[1]
    ps = g((P, Hk, d), torch.float32, 0.0)
    bsa.page_summaries(kc, bt, cl, out=ps)
    psum, psumm = g((P, Hk, d), torch.float32, 0.0), g((P, Hk, d), torch.float32, 0.0)
    bsa.page_summaries_append(kc, bt, cl, psum, psumm)
    for top_k in (8, 64):
        plan = bsa.DecodePlan(R, H, Hk, d, page, bt.shape[1], P, top_k)
        plan.ws = g.ws(plan.ws.numel())
        plan.out, plan.lse = g((R, H, d), torch.bfloat16), g((R, H), torch.float32)
        plan.sel, plan.sel_counts = g((R, Hk, top_k + 1), torch.int32), g((R, Hk), torch.int32)
        plan.status = _status(g)
        plan.run(q, kc, vc, ps, bt, cl)
        torch.cuda.synchronize()
        assert int(plan.status.item()) == 0
    g.check()


def test_chunk_calls_stay_inside_their_buffers():
    g = Guards()
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
    cache = bsa.PagedKVCache(g((P, Hk, 64, d), torch.bfloat16, 0.0), g((P, Hk, 64, d), torch.bfloat16, 0.0),
                             g((P, Hk, d), torch.float32, 0.0), torch.as_tensor(bt, device="cuda"),
                             g((P, Hk, d), torch.float32, 0.0))
    params = bsa.RouteParams(oracle.TOPK, 6, 0, 0.0, True)
    st = _status(g)
    cu = x.cu_seqlens
    idx = np.concatenate([np.arange(cu[i], cu[i] + n) for i, n in enumerate(lengths)])
    ti = torch.as_tensor(idx, device="cuda")
    qc, kc, vc = (t[:, ti].contiguous() for t in (q, k, v))
    chunk = bsa.Chunk.make([0, 0, 128], lengths, H, Hk, d, max_context_blocks=16)
    sh = chunk.shape
    B, Nq, T = sh.num_seqs, sh.max_blocks, sh.total_tokens
    bsa.chunk_append(kc, vc, chunk, cache, st)
    J, cnt = g((B, Hk, Nq, 6), torch.int32), g((B, Hk, Nq), torch.int32)
    bsa.route_chunk(qc, chunk, cache, params, st, J=J, counts=cnt,
                    ws=g.ws(bsa.route_chunk_workspace_bytes(chunk, cache, params)))
    rows = sh.num_rows
    s = sh.c()
    wl = bsa.Worklist(g((rows + 1,), torch.int32), g((rows * 6,), torch.int32),
                      g((rows,), torch.int32), g((bsa.NUM_BUCKETS + 1,), torch.int32))
    bsa.build_worklist_chunk(J, cnt, chunk, cache, 6, st, wl=wl,
                             ws=g.ws(_lib.lib().bsa_worklist_workspace_size(ctypes.byref(s), 6)))
    O, lse = g((H, T, d), torch.bfloat16), g((H, T), torch.float32)
    bsa.attention_chunk(qc, wl, chunk, cache, st, out=O, lse=lse)
    g.check()
    assert int(st.item()) == 0
