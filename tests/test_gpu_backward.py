"""GPU parity of the sparse-attention backward (dQ, dK, dV) against the float64
oracle (autograd of the masked definition), through the C ABI, on the index the
forward used."""
import numpy as np
import pytest
import torch

import dynamic_block_sparse_mean_gb300 as bsa
import oracle
from dynamic_block_sparse_mean_gb300 import synth
from parity_utils import dev_tensor, oracle_view, shape_of, upload

pytestmark = pytest.mark.gpu

# (name, lengths, H, H_kv, d, b, k_max, sink, dtype, max relative error)
CASES = [
    ("bwd_fp32_d64_b64_sink", [300, 129], 4, 2, 64, 64, 3, True, "fp32", 1e-3),
    ("bwd_bf16_gqa4_d128_b64", [700, 200], 8, 2, 128, 64, 4, False, "bf16", 2e-2),
    ("bwd_bf16_d128_b128", [600], 4, 1, 128, 128, 3, False, "bf16", 2e-2),
    ("bwd_fp32_d128_b64_tail", [400, 90], 4, 2, 128, 64, 3, True, "fp32", 1e-3),
    # tensor-core path: one query head per KV head (half of each M-tile masked), and
    # eight (four M-tiles per row)
    ("bwd_bf16_g1_d128_b64_sink", [500, 70], 2, 2, 128, 64, 4, True, "bf16", 2e-2),
    ("bwd_bf16_gqa8_d128_b64", [600, 1], 16, 2, 128, 64, 3, False, "bf16", 2e-2),
    # more work items than SMs (440 and 752 (row, M-tile) items): each persistent dQ
    # CTA walks several items, carrying ring stages, barrier phases and the dS buffer
    # across them; the 128-key case also runs 94 key-major dK / dV CTAs
    ("bwd_bf16_gqa4_d128_b64_multi", [4000, 3000], 8, 2, 128, 64, 6, True, "bf16", 2e-2),
    ("bwd_bf16_gqa8_d128_b128_multi", [6000], 16, 2, 128, 128, 4, True, "bf16", 2e-2),
    # 128-key blocks with one and two query heads per KV head (2 and 4 query tiles of
    # 64 rows per selecting row in the key-major pass), ragged tails
    ("bwd_bf16_g1_d128_b128", [700, 129], 2, 2, 128, 128, 3, True, "bf16", 2e-2),
    ("bwd_bf16_g2_d128_b128", [900, 60], 4, 2, 128, 128, 3, False, "bf16", 2e-2),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_oracle(case):
    name, lengths, H, Hk, d, b, k_max, sink, dtype, tol = case
    G = H // Hk
    x = synth.gen_prefill(lengths, H, Hk, d, b, 21, "iid", dtype)
    q, k, v = upload(x)
    sh = shape_of(x, H, Hk)
    Qo, Ko, Vo = oracle_view(x, "q"), oracle_view(x, "k"), oracle_view(x, "v")
    Jo, co, _, _ = oracle.route(Qo, Ko, x.cu_seqlens, b, G, oracle.TOPK, k_max, force_sink=sink)
    J = torch.as_tensor(Jo.astype(np.int32), device="cuda").contiguous()
    cnt = torch.as_tensor(co.astype(np.int32), device="cuda").contiguous()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wl = bsa.build_worklist(J, cnt, sh, k_max, status)
    O, lse = bsa.attention_fwd(q, k, v, wl, sh, status)
    rng = np.random.default_rng(22)
    dO_f = rng.normal(size=x.q.shape).astype(np.float32)
    if dtype == "bf16":
        dO_bits = synth.f32_to_bf16_bits(dO_f)
        do = dev_tensor(dO_bits, "bf16")
        dO64 = synth.bf16_bits_to_f32(dO_bits).astype(np.float64)
    else:
        do = dev_tensor(dO_f, "fp32")
        dO64 = dO_f.astype(np.float64)
    dq, dk, dv = bsa.attention_bwd(q, k, v, O, do, lse, wl, sh)
    torch.cuda.synchronize()
    bsa.check_status(status)
    # The oracle differentiates its own exact forward; the GPU uses its forward's O
    # (for D = dO . O) and lse, so the comparison covers both passes.
    gq, gk, gv = oracle.attention_backward(Qo, Ko, Vo, x.cu_seqlens, b, G, Jo, co, dO64)
    for got, ref, what in ((dq, gq, "dQ"), (dk, gk, "dK"), (dv, gv, "dV")):
        g = got.float().cpu().numpy().astype(np.float64)
        err = np.abs(g - ref).max() / np.abs(ref).max()
        assert err <= tol, (what, err)


def test_tensor_core_backward_is_deterministic():
    """The key-major pass sums a key block's rows in ascending order: two calls on
    the same inputs give the same bits."""
    x = synth.gen_prefill([900, 300], 8, 2, 128, 64, 23, "iid", "bf16")
    q, k, v = upload(x)
    sh = shape_of(x, 8, 2)
    Jo, co, _, _ = oracle.route(oracle_view(x, "q"), oracle_view(x, "k"), x.cu_seqlens, 64, 4,
                                oracle.TOPK, 5, force_sink=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wl = bsa.build_worklist(torch.as_tensor(Jo.astype(np.int32), device="cuda"),
                            torch.as_tensor(co.astype(np.int32), device="cuda"), sh, 5, status)
    O, lse = bsa.attention_fwd(q, k, v, wl, sh, status)
    do = dev_tensor(synth.f32_to_bf16_bits(np.random.default_rng(4).normal(size=x.q.shape)
                                           .astype(np.float32)), "bf16")
    a = [t.clone() for t in bsa.attention_bwd(q, k, v, O, do, lse, wl, sh, dev_status=status)]
    b = bsa.attention_bwd(q, k, v, O, do, lse, wl, sh, dev_status=status)
    torch.cuda.synchronize()
    bsa.check_status(status)
    for t0, t1 in zip(a, b):
        assert torch.equal(t0, t1)
