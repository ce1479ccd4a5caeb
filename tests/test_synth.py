"""The seeded input generator follows its stated recipes (no GPU): bf16 rounding is
round-to-nearest-even, draws do not depend on the thread count, and the planted,
window-bias and low-rank structures are what the workload table says."""
import math

import numpy as np
import torch

from dynamic_block_sparse_mean_gb300 import synth


def test_bf16_rounding_is_nearest_even_like_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32) * 100,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0], np.float32)])
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(synth.bf16_bits_to_f32(ours), torch.from_numpy(x).to(torch.bfloat16)
                          .float().numpy())


def test_draws_do_not_depend_on_thread_count(monkeypatch):
    shape = (3, (1 << 22) + 5)                       # more than one 4M-element chunk
    many = synth.normal_f32(shape, 7, 1)
    monkeypatch.setattr(synth, "_threads", lambda: 1)
    one = synth.normal_f32(shape, 7, 1)
    assert np.array_equal(many, one)
    assert abs(float(many.mean())) < 1e-2 and abs(float(many.std()) - 1.0) < 1e-2


def test_planted_blocks_follow_the_recipe():
    b, H, Hk, d = 64, 4, 2, 32
    x = synth.gen_prefill([64 * 300], H, Hk, d, b, 3, "planted", "fp32")
    base = synth.normal_f32((Hk, 64 * 300, d), 3, 2)
    nb = 300
    per_head = {h: [p for p in x.planted if p[0] == h] for h in range(Hk)}
    for h in range(Hk):
        assert len(per_head[h]) == math.floor(0.02 * nb)          # 2 % of the key blocks
    for (h, j, u) in x.planted:
        assert 1 <= j < nb - 1 and j < u < nb                      # paired with a later query block
        qb = x.q[h * 2:(h + 1) * 2, u * b:(u + 1) * b].reshape(-1, d).mean(axis=0)
        w = qb / np.linalg.norm(qb)
        delta = x.k[h, j * b:(j + 1) * b] - base[h, j * b:(j + 1) * b]
        assert np.allclose(delta, 3.0 * w[None, :], atol=1e-5)     # every key gets +3 w
    planted = {(h, j) for (h, j, _) in x.planted}
    for h in range(Hk):
        for j in range(nb):
            if (h, j) not in planted:
                assert np.array_equal(x.k[h, j * b:(j + 1) * b], base[h, j * b:(j + 1) * b])


def test_window_bias_adds_the_rotary_block_code():
    b, H, Hk, d = 64, 8, 8, 16
    n = 64 * 10
    x = synth.gen_prefill([n], H, Hk, d, b, 5, "window_bias", "fp32")
    kb = synth.normal_f32((Hk, n, d), 5, 2)
    changed = [h for h in range(Hk) if not np.array_equal(x.k[h], kb[h])]
    assert len(changed) == round(0.2 * Hk)                         # 20 % of the KV heads
    beta = np.arange(n) // b
    code = np.stack([2.0 * np.cos(math.pi / 32 * beta), 2.0 * np.sin(math.pi / 32 * beta)], 1)
    for h in changed:
        assert np.allclose(x.k[h, :, 0:2] - kb[h, :, 0:2], code, atol=1e-5)
        assert np.array_equal(x.k[h, :, 2:], kb[h, :, 2:])         # only dims 0 and 1


def test_lowrank_component_is_rank_eight_per_head():
    b, H, Hk, d = 16, 2, 2, 32
    n = 16 * 40
    x = synth.gen_prefill([n], H, Hk, d, b, 6, "lowrank", "fp32")
    kb = synth.normal_f32((Hk, n, d), 6, 2)
    for h in range(Hk):
        comp = x.k[h] - kb[h]
        blocks = comp.reshape(40, b, d)
        assert np.allclose(blocks, blocks[:, :1, :], atol=1e-5)   # one vector per block
        assert np.linalg.matrix_rank(blocks[:, 0, :].astype(np.float64), tol=1e-3) == 8
