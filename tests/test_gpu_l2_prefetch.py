"""The decode's L2 prefetch of a later kernel's weights (mla_set_decode_l2_prefetch)
is a hint to the memory system: with ranges set, mla_decode and mla_decode_q8
write bit for bit what they write without them, whatever the plan (whole
tokens per worker, split tokens), and bad ranges are refused on the host.
"""

import pytest
import torch

from head_latent_attention_26_b300 import build, synth
from _util import batch_meta, latent_inputs, scatter_rows
from test_gpu_q8 import q8_pool

pytestmark = pytest.mark.gpu

V2 = synth.V2


@pytest.fixture(scope="module")
def mla_mod():
    build.build()
    from head_latent_attention_26_b300 import mla
    return mla


@pytest.fixture(scope="module")
def v2(mla_mod):
    m = mla_mod.MLA(V2, 8192, torch.bfloat16)
    assert m.tensor_path
    return m


def test_prefetch_ranges_are_checked(v2, mla_mod):
    buf = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    for bad in (buf[1:1 + 4096], buf[:1000]):  # misaligned start, size not a multiple of 16
        with pytest.raises(mla_mod.MLAError) as e:
            v2.set_decode_l2_prefetch(bad)
        assert e.value.code == 1
    with pytest.raises(mla_mod.MLAError) as e:  # at most two ranges
        v2.set_decode_l2_prefetch(buf[:4096], buf[4096:8192], buf[8192:12288])
    assert e.value.code == 1
    v2.set_decode_l2_prefetch(buf[:4096], buf[4096:])
    v2.set_decode_l2_prefetch()


# (sequence lengths, query tokens per sequence, workers): one whole token per
# worker; tokens split over workers; more prefetch pieces than one range
CASES = [([4096] * 8, [1] * 8, 0), ([127, 63, 300, 1000], [1, 2, 1, 2], 3), ([200], [1], 0)]


def _weights(seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    w_uv = torch.randn(V2.n_h * V2.d_h, V2.d_c, generator=g, device="cuda").to(torch.bfloat16)
    w_o = torch.randn(V2.d_model, V2.n_h * V2.d_h, generator=g, device="cuda").to(torch.bfloat16)
    return w_uv, w_o


@pytest.mark.parametrize("seq_lens,q_counts,workers", CASES)
def test_decode_with_prefetch_is_unchanged(v2, seq_lens, q_counts, workers):
    seed = 1301 + sum(seq_lens)
    table, n_blocks, cu_q, lens, _ = batch_meta(seq_lens, q_counts, V2.block, seed)
    n_tok = int(sum(q_counts))
    q_lat, rows = latent_inputs(V2, n_tok, int(sum(seq_lens)), seed)
    per_seq = list(torch.split(rows, [int(t) for t in seq_lens]))
    pool = scatter_rows(per_seq, table, n_blocks, V2.block, V2.width)
    pool8 = q8_pool(per_seq, table, n_blocks)
    w_uv, w_o = _weights(seed)
    outs = {}
    for dec, p in (("bf16", pool), ("q8", pool8)):
        fn = v2.decode if dec == "bf16" else v2.decode_q8
        v2.set_decode_l2_prefetch()
        o0, l0 = fn(q_lat, p, table, lens, cu_q, num_workers=workers)
        v2.set_decode_l2_prefetch(w_uv, w_o[:2560])
        o1, l1 = fn(q_lat, p, table, lens, cu_q, num_workers=workers)
        v2.set_decode_l2_prefetch()
        v2.check()
        outs[dec] = (o0, l0, o1, l1)
    for dec, (o0, l0, o1, l1) in outs.items():
        assert not torch.isnan(o0.float()).any(), dec
        assert torch.equal(o0, o1) and torch.equal(l0, l1), dec
