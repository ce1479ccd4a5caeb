"""bsa_build_worklist_noalloc must build the same worklist as bsa_build_worklist.

It exists for callers that cannot give the library scratch memory — a serving
runtime that plans all of its GPU buffers ahead and owns only the inputs and
outputs, or code running where a cudaMalloc would synchronise the device — so
it keeps its scratch in a fixed device array inside libbsa.so.  This test calls
both entry points through the C ABI on the same inputs, twice in a row with
different shapes (the second call runs over whatever the first left in the
shared array), and requires identical integer outputs.  It lives in the file
pytest collects last so that a stop-at-first-failure run has already run every
other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import dynamic_block_sparse_mean_gb300 as bsa
from dynamic_block_sparse_mean_gb300 import _lib

pytestmark = pytest.mark.gpu


def _random_index(lengths, Hk, b, k_max, seed):
    """A valid J / counts pair: each row holds its diagonal plus random history
    blocks, ascending; a few rows are left empty (they fall back to the diagonal)."""
    rng = np.random.default_rng(seed)
    nb = [(n + b - 1) // b for n in lengths]
    Nq = max(nb)
    J = np.full((len(lengths), Hk, Nq, k_max), -1, dtype=np.int32)
    cnt = np.zeros((len(lengths), Hk, Nq), dtype=np.int32)
    for i, n_blocks in enumerate(nb):
        for h in range(Hk):
            for r in range(n_blocks):
                if rng.random() < 0.05:
                    continue
                extra = rng.choice(r, size=min(r, int(rng.integers(0, k_max))), replace=False) if r else []
                ids = sorted(set(int(e) for e in extra) | {r})[-k_max:]
                J[i, h, r, :len(ids)] = ids
                cnt[i, h, r] = len(ids)
    return J, cnt


def _buffers(rows, k_max):
    return (torch.full((rows + 1,), -7, dtype=torch.int32, device="cuda"),
            torch.full((rows * k_max,), -7, dtype=torch.int32, device="cuda"),
            torch.full((rows,), -7, dtype=torch.int32, device="cuda"),
            torch.full((8,), -7, dtype=torch.int32, device="cuda"),
            torch.zeros(1, dtype=torch.int32, device="cuda"))


def _both(lengths, Hk, b, k_max, seed):
    J, cnt = _random_index(lengths, Hk, b, k_max, seed)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    sh = bsa.PrefillShape.make(cu, Hk, Hk, 64, b)
    s = sh.c()
    dJ, dc = torch.as_tensor(J, device="cuda"), torch.as_tensor(cnt, device="cuda")
    lib = _lib.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731

    ref = _buffers(sh.num_rows, k_max)
    ws = torch.empty(max(256, lib.bsa_worklist_workspace_size(ctypes.byref(s), k_max)),
                     dtype=torch.uint8, device="cuda")
    assert lib.bsa_build_worklist(ctypes.byref(s), k_max, p(dJ), p(dc), *(p(t) for t in ref),
                                  p(ws), ws.numel(), stream) == 0
    got = _buffers(sh.num_rows, k_max)
    assert lib.bsa_build_worklist_noalloc(ctypes.byref(s), k_max, p(dJ), p(dc),
                                          *(p(t) for t in got), stream) == 0
    torch.cuda.synchronize()
    return ref, got, sh


def _assert_same(ref, got):
    rp, ci, wk, bo, st = (t.cpu().numpy() for t in ref)
    rp2, ci2, wk2, bo2, st2 = (t.cpu().numpy() for t in got)
    assert st[0] == 0 and st2[0] == 0
    assert np.array_equal(rp, rp2) and np.array_equal(bo, bo2)
    assert np.array_equal(ci[:rp[-1]], ci2[:rp2[-1]])
    assert np.array_equal(wk[:bo[-1]], wk2[:bo2[-1]])


def test_noalloc_worklist_matches_regular_on_two_calls_in_a_row():
    ref, got, sh = _both([3000, 700, 64, 1], Hk=4, b=64, k_max=12, seed=1)
    _assert_same(ref, got)
    ref, got, sh = _both([9000, 2000], Hk=2, b=128, k_max=20, seed=2)
    _assert_same(ref, got)


def test_noalloc_worklist_rejects_shapes_beyond_its_array():
    n = (_lib_max_rows() + 1) * 64
    sh = bsa.PrefillShape.make([0, n], 1, 1, 64, 64)
    s = sh.c()
    dummy = ctypes.c_void_p(256)
    assert _lib.lib().bsa_build_worklist_noalloc(ctypes.byref(s), 4, *([dummy] * 7), None) == 2


def _lib_max_rows():
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "include", "bsa.h")).read()
    return eval(re.search(r"#define BSA_WORKLIST_NOALLOC_MAX_ROWS \((.*?)\)", hdr).group(1))


def _sparse_index_at_cap(S, Hk, Nq, seed):
    """J / counts for S sequences x Hk KV heads x Nq blocks: each row holds up to
    three history blocks below its diagonal at random gaps, plus the diagonal;
    5 % of rows are left empty (they fall back to the diagonal)."""
    rng = np.random.default_rng(seed)
    r = np.broadcast_to(np.arange(Nq), (S, Hk, Nq))
    gaps = np.cumsum(1 + rng.integers(0, 40, size=(S, Hk, Nq, 3)), axis=-1)   # d1 < d2 < d3
    hist = r[..., None] - gaps[..., ::-1]                                      # ascending
    ids = np.concatenate([np.where(hist >= 0, hist, -1), r[..., None]], axis=-1)
    key = np.where(ids >= 0, ids, np.iinfo(np.int32).max)                     # -1s to the end
    ids = np.take_along_axis(ids, np.argsort(key, axis=-1, kind="stable"), axis=-1)
    cnt = (ids >= 0).sum(-1)
    empty = rng.random((S, Hk, Nq)) < 0.05
    ids[empty] = -1
    cnt[empty] = 0
    return ids.astype(np.int32), cnt.astype(np.int32)


def test_noalloc_worklist_at_its_row_limit():
    """A shape with exactly BSA_WORKLIST_NOALLOC_MAX_ROWS rows is accepted and gives
    the workspace version's worklist."""
    S, Hk, b, k_max = 4, 8, 64, 4
    Nq = _lib_max_rows() // (S * Hk)
    assert S * Hk * Nq == _lib_max_rows()
    J, cnt = _sparse_index_at_cap(S, Hk, Nq, seed=3)
    cu = np.arange(S + 1, dtype=np.int64) * Nq * b
    sh = bsa.PrefillShape.make(cu, Hk, Hk, 64, b)
    assert sh.num_rows == _lib_max_rows()
    s = sh.c()
    dJ, dc = torch.as_tensor(J, device="cuda"), torch.as_tensor(cnt, device="cuda")
    lib = _lib.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    ref = _buffers(sh.num_rows, k_max)
    ws = torch.empty(max(256, lib.bsa_worklist_workspace_size(ctypes.byref(s), k_max)),
                     dtype=torch.uint8, device="cuda")
    assert lib.bsa_build_worklist(ctypes.byref(s), k_max, p(dJ), p(dc), *(p(t) for t in ref),
                                  p(ws), ws.numel(), stream) == 0
    got = _buffers(sh.num_rows, k_max)
    assert lib.bsa_build_worklist_noalloc(ctypes.byref(s), k_max, p(dJ), p(dc),
                                          *(p(t) for t in got), stream) == 0
    torch.cuda.synchronize()
    _assert_same(ref, got)
    rp = ref[0].cpu().numpy()
    assert rp[-1] == int(np.maximum(cnt, 1).sum())     # empty rows became {r}
