"""The seeded input recipe (head_latent_attention_26_b300.synth), on CPU:
determinism, independence of named tensors, the stated distributions and a
valid block table."""

import math

import torch

from head_latent_attention_26_b300 import synth


def test_same_seed_same_values_and_names_independent():
    a = synth.normal((4, 64), 5, "x")
    b = synth.normal((4, 64), 5, "x")
    assert torch.equal(a, b)
    assert not torch.equal(a, synth.normal((4, 64), 5, "y"))
    assert not torch.equal(a, synth.normal((4, 64), 6, "x"))


def test_weight_shapes_and_fan_in_scale():
    d = synth.TINY
    W = synth.weights(d, 3, dtype=torch.float32)
    H, Hr = d.n_h * d.d_h, d.n_h * d.d_hr
    assert W["W_dkv"].shape == (d.d_c, d.d_model) and W["W_kr"].shape == (d.d_hr, d.d_model)
    assert W["W_dq"].shape == (d.d_cq, d.d_model) and W["W_uq"].shape == (H, d.d_cq)
    assert W["W_qr"].shape == (Hr, d.d_cq) and W["W_uk"].shape == (H, d.d_c)
    assert W["W_uv"].shape == (H, d.d_c) and W["W_o"].shape == (d.d_model, H)
    # std 1/sqrt(fan_in) on a large draw
    big = synth.normal((512, 4096), 9, "big", std=1 / math.sqrt(4096), dtype=torch.float32)
    assert abs(big.std().item() * math.sqrt(4096) - 1) < 0.01
    assert abs(big.mean().item()) * math.sqrt(4096) < 0.01


def test_bf16_values_are_rounded_once_from_fp32():
    x32 = synth.normal((1000,), 11, "r", dtype=torch.float32)
    x16 = synth.normal((1000,), 11, "r", dtype=torch.bfloat16)
    assert torch.equal(x32.to(torch.bfloat16), x16)


def test_block_table_is_a_permutation_of_the_pool():
    lens = [1, 64, 65, 300, 4096]
    table, n_pool = synth.block_table(lens, 64, 7, spare_blocks=3)
    nb = [(t + 63) // 64 for t in lens]
    assert n_pool == sum(nb) + 3 and table.shape == (len(lens), max(nb))
    used = []
    for b, n in enumerate(nb):
        assert torch.all(table[b, :n] >= 0) and torch.all(table[b, n:] == -1)
        used += table[b, :n].tolist()
    assert len(set(used)) == len(used) == sum(nb) and max(used) < n_pool
    again, _ = synth.block_table(lens, 64, 7, spare_blocks=3)
    assert torch.equal(table, again)


def test_lengths_counts_and_prefix():
    L = synth.ragged_lengths(1000, 512, 16384, 4)
    assert L.min() >= 512 and L.max() <= 16384
    q = synth.query_counts(1000, 4)
    assert set(q.tolist()) == {1, 2} and abs(q.float().mean().item() - 1.5) < 0.05
    assert synth.cu_from_counts([1, 2, 1]).tolist() == [0, 1, 3, 4]
    rows = synth.pick_rows(131072, 0.01, 4)
    assert len(rows) == 1311 and len(set(rows.tolist())) == 1311 and torch.all(rows[1:] > rows[:-1])


def test_dims():
    assert synth.V2.width == 576 and abs(synth.V2.scale - 1 / math.sqrt(192)) < 1e-15
    assert synth.TINY.width == 20
