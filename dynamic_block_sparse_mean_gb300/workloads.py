"""The five synthetic workloads the library is measured and parity-checked on.

Each workload is named by what it is and its sizes.  The shapes follow the
problem statement of "2.1 · 粗粒度选择" (PaperTrace, sparse-attention 2-1),
section 1 opening paragraph: Q, K, V of shape B x H x n x d_h, block size b,
N_q = ceil(n / b) query blocks, and an index J of at most k_b key blocks per
query block.  Layout in this library is head-major and packed: Q [H, T, d],
K and V [H_kv, T, d], sequence i owns tokens cu_seqlens[i] .. cu_seqlens[i+1].

Route parameters (what "k_max" means, forced blocks) are fixed here so that
the GPU path and the oracle read them from one place; no arithmetic of the
method lives in this module.
"""
from __future__ import annotations

from dataclasses import dataclass, field

ROUTE_TOPK = 0
ROUTE_THRESHOLD = 1


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    num_seqs: int
    seqlen: int | None          # fixed length; None for a variable-length batch
    seqlen_range: tuple[int, int] | None
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block: int
    mode: int                   # ROUTE_TOPK or ROUTE_THRESHOLD
    k_max: int                  # row capacity of J, forced blocks included
    k_min: int = 0
    tau_delta: float = 0.0
    force_sink: bool = False
    structure: str = "iid"      # generator recipe, see synth.py
    seed: int = 0

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    num_reqs: int
    len_range: tuple[int, int]
    num_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    top_k: int
    seed: int = 0


# Tiny case: n=1024, H=H_kv=2, d=64, b=64, top-4 with the diagonal and block 0
# forced, so two dynamic blocks per row once r >= 2.
TINY = PrefillWorkload(
    name="tiny_n1024_h2_d64_b64_top4", num_seqs=1, seqlen=1024, seqlen_range=None,
    num_heads=2, num_kv_heads=2, head_dim=64, block=64,
    mode=ROUTE_TOPK, k_max=4, force_sink=True, structure="iid", seed=1001)

# Long prompt with planted structure: n=32768, GQA 32/8, d=128, b=64, row
# capacity 32 (31 dynamic + the forced diagonal).
PROMPT_32K = PrefillWorkload(
    name="prompt_n32768_h32kv8_d128_b64_top32_planted", num_seqs=1, seqlen=32768,
    seqlen_range=None, num_heads=32, num_kv_heads=8, head_dim=128, block=64,
    mode=ROUTE_TOPK, k_max=32, force_sink=False, structure="planted", seed=1002)

# Variable-length packed batch, threshold routing (row max minus 2.0), clamps 4..64.
VARLEN_256K = PrefillWorkload(
    name="varlen_b8_n4k-64k_h32kv8_d128_b64_thresh2.0_k4-64", num_seqs=8, seqlen=None,
    seqlen_range=(4096, 65536), num_heads=32, num_kv_heads=8, head_dim=128, block=64,
    mode=ROUTE_THRESHOLD, k_max=64, k_min=4, tau_delta=2.0, force_sink=False,
    structure="window_bias", seed=1003)

# Very long sparse prefill: n=131072, GQA 64/8, b=128, top-16 dynamic plus the
# forced sink block 0 and the diagonal (row capacity 18).
LONG_128K = PrefillWorkload(
    name="long_n131072_h64kv8_d128_b128_top16+sink+diag", num_seqs=1, seqlen=131072,
    seqlen_range=None, num_heads=64, num_kv_heads=8, head_dim=128, block=128,
    mode=ROUTE_TOPK, k_max=18, force_sink=True, structure="lowrank", seed=1004)

# Paged sparse decode: 64 requests, one query token each, top-32 pages plus the last.
DECODE_64 = DecodeWorkload(
    name="decode_64req_len8k-128k_h32kv8_d128_page64_top32+last", num_reqs=64,
    len_range=(8192, 131072), num_heads=32, num_kv_heads=8, head_dim=128,
    page_size=64, top_k=32, seed=1005)

PREFILL_WORKLOADS = {w.name: w for w in (TINY, PROMPT_32K, VARLEN_256K, LONG_128K)}
