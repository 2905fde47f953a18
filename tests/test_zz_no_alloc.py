"""mla_decode_noalloc: decode for callers that cannot allocate device memory.

Such a caller -- a plugin whose host engine owns the whole device-memory
budget, or a hot loop that must not risk cudaMalloc's synchronisation and
latency -- passes only inputs and outputs; the split-KV scratch comes from a
fixed array inside the library.  This file is collected last so that a failure
here cannot hide the results of the other tests.
"""

import pytest
import torch

from head_latent_attention_26_b300 import build, synth
from _util import LSE_TOL, OUT_TOL, batch_meta, latent_inputs, lse_err, row_rel_err, scatter_rows, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def case():
    build.build()
    from head_latent_attention_26_b300 import mla
    d = synth.V2
    m = mla.MLA(d, 20000, torch.bfloat16)
    assert m.tensor_path
    seq_lens, q_counts = [300, 2000, 64, 5000, 1], [1, 2, 1, 1, 1]
    table, n_blocks, cu_q, lens, _ = batch_meta(seq_lens, q_counts, d.block, 2024, spare_blocks=2)
    q_lat, rows = latent_inputs(d, sum(q_counts), sum(seq_lens), 2024)
    pool = scatter_rows(list(torch.split(rows, seq_lens)), table, n_blocks, d.block, d.width)
    return m, q_lat, pool, table, lens, cu_q


def test_noalloc_matches_workspace_decode_twice_in_a_row(case):
    m, q_lat, pool, table, lens, cu_q = case
    o_ref, l_ref = m.decode(q_lat, pool, table, lens, cu_q)
    m.check()
    o_ref, l_ref = to_np(o_ref), to_np(l_ref)
    for workers in (0, 7):  # two calls in a row share (and reuse) the fixed scratch
        o, l = m.decode_noalloc(q_lat, pool, table, lens, cu_q, num_workers=workers)
        m.check()
        assert row_rel_err(to_np(o), o_ref) < OUT_TOL, workers
        assert lse_err(to_np(l), l_ref) < LSE_TOL, workers


def test_noalloc_rejects_requests_beyond_its_scratch(case):
    from head_latent_attention_26_b300 import mla
    m, q_lat, pool, table, lens, cu_q = case
    with pytest.raises(mla.MLAError) as e:
        m.decode_noalloc(q_lat, pool, table, lens, cu_q, num_workers=33)  # at most 32 workers
    assert e.value.code == 3
