"""Host logic of the output-weight L2 prefetch (no GPU): the ranges handed
to mla_set_decode_l2_prefetch are contiguous, 16-byte multiples, within the
byte budget, and W^O is cut at whole 128-row tiles."""

import pytest
import torch

from head_latent_attention_26_b300 import mla, synth

V2 = synth.V2


@pytest.fixture(scope="module")
def weights():
    w_uv = torch.empty(V2.n_h * V2.d_h, V2.d_c, dtype=torch.bfloat16)
    w_o = torch.empty(V2.d_model, V2.n_h * V2.d_h, dtype=torch.bfloat16)
    return w_uv, w_o


@pytest.mark.parametrize("budget", [0, 1000, 16 << 20, (16 << 20) + 100, 96 << 20, 1 << 40])
def test_output_weight_prefetch_ranges(weights, budget):
    w_uv, w_o = weights
    ranges = mla.output_weight_prefetch(w_uv, w_o, budget)
    nbytes = [t.numel() * t.element_size() for t in ranges]
    assert len(ranges) <= 2
    assert sum(nbytes) <= budget
    for t, n in zip(ranges, nbytes):
        assert t.is_contiguous() and n % 16 == 0 and n > 0 or budget < 16
    if budget == 0:
        assert ranges == ()
    if len(ranges) == 2:
        # all of W^UV first, then the leading whole tiles of W^O
        assert ranges[0].data_ptr() == w_uv.data_ptr() and nbytes[0] == w_uv.numel() * 2
        assert ranges[1].data_ptr() == w_o.data_ptr() and ranges[1].shape[0] % 128 == 0
        # the budget leaves less than one more tile of W^O unused
        assert budget - sum(nbytes) < 128 * w_o.shape[1] * 2 or ranges[1].shape[0] == w_o.shape[0]


def test_prefetch_binding_is_declared():
    assert "mla_set_decode_l2_prefetch" in mla.header_symbols()


def test_default_prefetch_only_for_one_launch_output_steps():
    # steps whose output projection is the one-launch kernel (up to 64 tokens)
    assert mla.default_prefetch_bytes(1) == mla.default_prefetch_bytes(64) == mla.OUT_WEIGHT_PREFETCH_BYTES
    assert mla.default_prefetch_bytes(65) == mla.default_prefetch_bytes(194) == 0
