"""The C-ABI library loads, exports every entry point include/bsa.h declares, and
rejects bad arguments on the host before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

from dynamic_block_sparse_mean_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "bsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bsa_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from dynamic_block_sparse_mean_gb300 import build
        build.build()
    return _lib.lib()


def test_header_declares_the_hot_path_calls():
    names = _declared()
    for n in ("bsa_block_summaries", "bsa_route", "bsa_build_worklist", "bsa_attention_fwd",
              "bsa_decode_paged", "bsa_page_summaries", "bsa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_declared()) <= set(_lib.PROTOTYPES), "binding prototypes cover the header"


def test_version_and_status_strings(lib):
    hdr = open(os.path.join(ROOT, "include", "bsa.h")).read()
    assert lib.bsa_version() == int(re.search(r"#define BSA_VERSION (\d+)", hdr).group(1))
    for code in _lib.STATUS_NAMES:
        assert lib.bsa_status_string(code)


def _route_split_bytes(rows, d, qrows):
    """The BF16 router's workspace besides the score matrix: the three-way bf16 split
    of the summaries, their two norms, one query-norm bound per router row, and the
    rescoring queue (its length, the queued rows, per row a count and 64 candidate
    ids), each rounded up to 256 bytes."""
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    return (up(rows * d * 3 * 2) + 2 * up(rows * 4) + up(qrows * 4) +
            up(4) + 2 * up(qrows * 4) + up(qrows * 64 * 4))


def _shape(**kw):
    base = dict(num_seqs=1, total_tokens=1024, max_seqlen=1024, num_heads=2, num_kv_heads=2,
                head_dim=64, block=64, max_blocks=16, dtype=0, cu_seqlens=0x1000)
    base.update(kw)
    return _lib.Shape(**base)


def test_host_side_argument_errors(lib):
    null = None
    s = _shape()
    bad = _shape(cu_seqlens=None)
    assert lib.bsa_block_summaries(ctypes.byref(bad), ctypes.c_void_p(16), ctypes.c_void_p(16), null) == 1
    assert lib.bsa_block_summaries(ctypes.byref(s), null, ctypes.c_void_p(16), null) == 1
    assert lib.bsa_block_summaries(ctypes.byref(_shape(max_blocks=15)), ctypes.c_void_p(16),
                                   ctypes.c_void_p(16), null) == 1
    assert lib.bsa_block_summaries(ctypes.byref(_shape(head_dim=96)), ctypes.c_void_p(16),
                                   ctypes.c_void_p(16), null) == 2
    assert lib.bsa_block_summaries(ctypes.byref(_shape(num_heads=3)), ctypes.c_void_p(16),
                                   ctypes.c_void_p(16), null) == 1
    empty = _shape(total_tokens=0, max_seqlen=0, max_blocks=0)       # a batch without tokens
    assert lib.bsa_block_summaries(ctypes.byref(empty), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                   null) == 1
    p = _lib.RouteParams(0, 300, 0, 0.0, 0)
    args = [ctypes.c_void_p(16)] * 4
    assert lib.bsa_route(ctypes.byref(s), ctypes.byref(p), *args, null, null, null, 0, null) == 2
    p = _lib.RouteParams(0, 4, 0, 0.0, 0)
    assert lib.bsa_route(ctypes.byref(s), ctypes.byref(p), *args, null, null, null, 0, null) == 3
    p = _lib.RouteParams(5, 4, 0, 0.0, 0)
    assert lib.bsa_route(ctypes.byref(s), ctypes.byref(p), *args, null, null, null, 0, null) == 1
    # union routing: the forced set must fit the row capacity, the list its bound
    gl = ctypes.c_void_p(16)
    for bad_p in (_lib.RouteParams(0, 4, 0, 0.0, 0, 5, 0, None),       # window > k_max
                  _lib.RouteParams(0, 4, 0, 0.0, 1, 2, 2, gl),         # 2 + 2 + sink > 4
                  _lib.RouteParams(0, 64, 0, 0.0, 0, 1, 33, gl),       # list too long
                  _lib.RouteParams(0, 64, 0, 0.0, 0, 1, 1, None)):     # list missing
        assert lib.bsa_route(ctypes.byref(s), ctypes.byref(bad_p), *args, null, null, null, 0,
                             null) == 1
    ok_p = _lib.RouteParams(0, 4, 0, 0.0, 1, 2, 1, gl)                # 2 + 1 + sink = 4
    assert lib.bsa_route(ctypes.byref(s), ctypes.byref(ok_p), *args, null, null, null, 0, null) == 3
    assert lib.bsa_route_workspace_size(ctypes.byref(s), ctypes.byref(p)) == \
        _route_split_bytes(32, 64, 32) + 1 * 2 * 16 * 16 * 4
    wl = [ctypes.c_void_p(16)] * 7
    assert lib.bsa_build_worklist(ctypes.byref(s), 4, *wl, null, 0, null) == 3
    assert lib.bsa_build_worklist(ctypes.byref(s), 0, *wl, null, 0, null) == 2
    a = [ctypes.c_void_p(16)] * 7
    assert lib.bsa_attention_fwd(ctypes.byref(s), *a, ctypes.c_float(0.0), ctypes.c_void_p(16),
                                 null, null, null) == 1          # dev_status missing
    assert lib.bsa_attention_fwd(ctypes.byref(s), *a, ctypes.c_float(float("nan")),
                                 ctypes.c_void_p(16), null, ctypes.c_void_p(16), null) == 1
    ds = _lib.DecodeShape(4, 32, 8, 128, 64, 100, 400, 32)
    dargs = [ctypes.c_void_p(16)] * 6
    assert lib.bsa_decode_paged(ctypes.byref(ds), *dargs, ctypes.c_float(0.0), ctypes.c_void_p(16),
                                null, ctypes.c_void_p(16), ctypes.c_void_p(16), null, null, 0,
                                null) == 3
    ds_bad = _lib.DecodeShape(4, 32, 8, 64, 64, 100, 400, 32)
    assert lib.bsa_decode_paged(ctypes.byref(ds_bad), *dargs, ctypes.c_float(0.0),
                                ctypes.c_void_p(16), null, ctypes.c_void_p(16), ctypes.c_void_p(16),
                                null, null, 0, null) == 2
    assert lib.bsa_decode_workspace_size(ctypes.byref(ds)) > 0
    # token recall: t_top >= 1, a tile count only with a tile list, k_max in range
    p16 = ctypes.c_void_p(16)
    rec = lambda t, km, tiles, nt: lib.bsa_token_recall(  # noqa: E731
        ctypes.byref(s), t, p16, p16, p16, p16, km, tiles, nt, p16, p16, null)
    assert rec(0, 4, null, 0) == 1
    assert rec(64, 4, null, 3) == 1
    assert rec(64, 300, null, 0) == 2
    assert lib.bsa_recall_tiles_per_seq(ctypes.byref(s)) == 16


def test_chunk_calls_reject_bad_cache_descriptors(lib):
    null, p16 = None, ctypes.c_void_p(16)
    s = _shape()                                            # block 64, d 64, bf16, N_q 16

    def cache(**kw):
        base = dict(k_cache=16, v_cache=16, page_summ=16, page_sum=None, block_table=16,
                    prefix_lens=16, max_pages_per_req=32, num_phys_pages=100,
                    max_context_blocks=16)
        base.update(kw)
        return _lib.KVCache(**base)

    def append(sh, c):
        return lib.bsa_chunk_append(ctypes.byref(sh), ctypes.byref(c), p16, p16, p16, null)

    assert append(s, cache(prefix_lens=None)) == 1
    assert append(s, cache(max_context_blocks=15)) == 1       # below the chunk's N_q
    assert append(s, cache(max_context_blocks=33)) == 1       # past the block table
    assert append(_shape(dtype=1), cache()) == 2              # the cache is bf16
    assert append(_shape(block=128, max_blocks=8), cache()) == 2   # page = block = 64
    assert append(s, cache(num_phys_pages=1 << 26)) == 2      # page rows past int32
    assert append(s, cache(k_cache=24)) == 1                  # 16-byte alignment
    assert lib.bsa_chunk_append(ctypes.byref(s), ctypes.byref(cache()), p16, p16, null,
                                null) == 1                    # dev_status missing
    p = _lib.RouteParams(0, 4, 0, 0.0, 0, 1, 0, None)
    c = cache()
    need = lib.bsa_route_chunk_workspace_size(ctypes.byref(s), ctypes.byref(c), ctypes.byref(p))
    assert need == _route_split_bytes(32, 64, 32) + 1 * 2 * 16 * 16 * 4
    args = [p16] * 4
    assert lib.bsa_route_chunk(ctypes.byref(s), ctypes.byref(c), ctypes.byref(p), *args, p16,
                               null, 0, null) == 3
    bad_p = _lib.RouteParams(0, 300, 0, 0.0, 0, 1, 0, None)
    assert lib.bsa_route_chunk(ctypes.byref(s), ctypes.byref(c), ctypes.byref(bad_p), *args, p16,
                               p16, 1 << 20, null) == 2
    wl = [p16] * 7
    assert lib.bsa_build_worklist_chunk(ctypes.byref(s), ctypes.byref(c), 4, *wl, null, 0,
                                        null) == 3
    a = [p16] * 5
    assert lib.bsa_attention_chunk(ctypes.byref(s), ctypes.byref(c), *a, ctypes.c_float(0.0), p16,
                                   null, null, null) == 1     # dev_status missing


def test_backward_host_checks_and_workspace(lib):
    null, p16 = None, ctypes.c_void_p(16)
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    # bf16, head_dim 128: D [H, T] plus the key-major index (counts, list, offsets,
    # buckets, a row bitmap of ceil(N_q / 32) words per key block, and the rows)
    s = _shape(head_dim=128)                 # B 1, T 1024, H 2, H_kv 2, b 64, N_q 16
    rows, W, pairs = 1 * 2 * 16, 1, 1 * 2 * 16 * 17 // 2
    want = up(2 * 1024 * 4) + 2 * up(rows * 4) + up((rows + 1) * 4) + up(8 * 4) + up(rows * W * 4) \
        + up(pairs * 4)
    assert lib.bsa_attention_bwd_workspace_size(ctypes.byref(s)) == want
    # fp32 or head_dim 64: D plus fp32 dK / dV accumulators
    s64 = _shape()
    kv = 2 * 1024 * 64 * 4
    assert lib.bsa_attention_bwd_workspace_size(ctypes.byref(s64)) == up(2 * 1024 * 4) + 2 * up(kv)
    args = [p16] * 10
    assert lib.bsa_attention_bwd(ctypes.byref(s), *args, ctypes.c_float(0.0), p16, p16, p16,
                                 null, p16, 1 << 30, null) == 1     # dev_status missing
    assert lib.bsa_attention_bwd(ctypes.byref(s), *args, ctypes.c_float(0.0), p16, p16, p16,
                                 p16, p16, 16, null) == 3           # workspace too small
    assert lib.bsa_attention_bwd(ctypes.byref(s), *args, ctypes.c_float(0.0), p16, p16, p16,
                                 p16, ctypes.c_void_p(16), 1 << 30, null) == 1   # ws not 256-aligned
    assert lib.bsa_attention_bwd(ctypes.byref(_shape(head_dim=96)), *args, ctypes.c_float(0.0),
                                 p16, p16, p16, p16, ctypes.c_void_p(256), 1 << 30, null) == 2


def test_selftest_entry_rejects_missing_status(lib):
    assert lib.bsa_selftest_wait_timeout(None, None) == 1
