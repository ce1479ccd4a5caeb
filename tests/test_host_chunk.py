"""Host-side bookkeeping of the chunked prefill (no GPU): the chunk's packed shape,
its logical-block offsets and the cache descriptor handed to the C ABI."""
import numpy as np
import torch

import dynamic_block_sparse_mean_gb300 as bsa


def test_chunk_shape_and_context_blocks():
    ch = bsa.Chunk.make([0, 128, 640], [300, 0, 65], 8, 2, 128, device="cpu")
    sh = ch.shape
    assert sh.cu_seqlens.tolist() == [0, 300, 300, 365]
    assert (sh.num_seqs, sh.total_tokens, sh.max_seqlen, sh.block) == (3, 365, 300, 64)
    assert sh.max_blocks == 5                                  # ceil(300 / 64)
    # contexts 300, 128 (idle) and 705 tokens: ceil(705 / 64) = 12 blocks
    assert ch.max_context_blocks == 12
    assert ch.prefix_lens.dtype == torch.int32 and ch.prefix_lens.tolist() == [0, 128, 640]


def test_cache_descriptor_fields():
    bt = np.arange(24, dtype=np.int32).reshape(2, 12)
    cache = bsa.PagedKVCache.allocate(30, 2, 64, bt, device="cpu")
    assert cache.k_cache.shape == (30, 2, 64, 64) and cache.k_cache.dtype == torch.bfloat16
    assert cache.page_summ.shape == (30, 2, 64) and cache.page_sum is not None
    ch = bsa.Chunk.make([64, 0], [10, 700], 4, 2, 64, device="cpu")
    c = cache.c(ch)
    assert (c.max_pages_per_req, c.num_phys_pages, c.max_context_blocks) == (12, 30, 11)
    assert c.block_table == cache.block_table.data_ptr()
    assert c.prefix_lens == ch.prefix_lens.data_ptr()
    assert c.page_sum == cache.page_sum.data_ptr()
    no_sums = bsa.PagedKVCache.allocate(30, 2, 64, bt, device="cpu", with_sums=False)
    assert no_sums.c(ch).page_sum is None
