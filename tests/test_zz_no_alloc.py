"""mla_decode_noalloc: decode for callers that cannot allocate device memory.

Such a caller -- a plugin whose host engine owns the whole device-memory
budget, or a hot loop that must not risk cudaMalloc's synchronisation and
latency -- passes only inputs and outputs; the split-KV scratch comes from a
fixed array inside the library.  This file is collected last so that a failure
here cannot hide the results of the other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from head_latent_attention_26_b300 import build, synth
from _util import LSE_TOL, OUT_TOL, batch_meta, latent_inputs, lse_err, record, row_rel_err, scatter_rows, to_np

pytestmark = pytest.mark.gpu

SEQ_LENS, Q_COUNTS = [300, 2000, 64, 5000, 1], [1, 2, 1, 1, 1]


@pytest.fixture(scope="module")
def case():
    build.build()
    from head_latent_attention_26_b300 import mla
    d = synth.V2
    m = mla.MLA(d, 20000, torch.bfloat16)
    assert m.tensor_path
    table, n_blocks, cu_q, lens, _ = batch_meta(SEQ_LENS, Q_COUNTS, d.block, 2024, spare_blocks=2)
    q_lat, rows = latent_inputs(d, sum(Q_COUNTS), sum(SEQ_LENS), 2024)
    per_seq = list(torch.split(rows, SEQ_LENS))
    pool = scatter_rows(per_seq, table, n_blocks, d.block, d.width)
    return m, q_lat, pool, table, lens, cu_q, per_seq


def _oracle_check(d, q_lat, per_seq, o, l, what):
    cu = np.concatenate([[0], np.cumsum(Q_COUNTS)])
    for b, L in enumerate(SEQ_LENS):
        rows_b = to_np(per_seq[b])
        for k in range(Q_COUNTS[b]):
            n = int(cu[b]) + k
            t = L - Q_COUNTS[b] + k
            o_ref, l_ref = O.attend_latent(to_np(q_lat[n]), rows_b[:t + 1], d.d_c, d.d_h)
            e_o, e_l = row_rel_err(to_np(o[n]), o_ref), lse_err(to_np(l[n]), l_ref)
            record("decode without workspace vs oracle", e_o, e_l)
            assert e_o < OUT_TOL and e_l < LSE_TOL, (what, n, e_o, e_l)


def test_noalloc_matches_workspace_decode_and_oracle_twice_in_a_row(case):
    m, q_lat, pool, table, lens, cu_q, per_seq = case
    d = synth.V2
    o_ref, l_ref = m.decode(q_lat, pool, table, lens, cu_q)
    m.check()
    _oracle_check(d, q_lat, per_seq, o_ref, l_ref, "mla_decode")
    o_ref, l_ref = to_np(o_ref), to_np(l_ref)
    # two calls in a row share (and reuse) the fixed scratch; 32 workers is the
    # largest request it holds
    for workers in (0, 7, 32):
        o, l = m.decode_noalloc(q_lat, pool, table, lens, cu_q, num_workers=workers)
        m.check()
        assert row_rel_err(to_np(o), o_ref) < OUT_TOL, workers
        assert lse_err(to_np(l), l_ref) < LSE_TOL, workers
        _oracle_check(d, q_lat, per_seq, o, l, f"mla_decode_noalloc workers={workers}")


def test_noalloc_rejects_requests_beyond_its_scratch(case):
    from head_latent_attention_26_b300 import mla
    m, q_lat, pool, table, lens, cu_q, _ = case
    with pytest.raises(mla.MLAError) as e:
        m.decode_noalloc(q_lat, pool, table, lens, cu_q, num_workers=33)  # at most 32 workers
    assert e.value.code == 3
    # 8193 query tokens: rejected on the host before anything launches (the
    # pointers are valid, the token count alone is beyond the fixed scratch)
    lib, P = m.lib, ctypes.c_void_p
    o = torch.empty(1, 128, 512, dtype=torch.bfloat16, device="cuda")
    l = torch.empty(1, 128, dtype=torch.float32, device="cuda")
    s = P(torch.cuda.current_stream().cuda_stream)
    args = (m.h, q_lat.data_ptr(), pool.data_ptr(), pool.shape[0], table.data_ptr(), table.shape[1],
            lens.data_ptr(), cu_q.data_ptr(), lens.shape[0])
    assert lib.mla_decode_noalloc(*args, 8193, 0, o.data_ptr(), l.data_ptr(), s) == 3
    assert lib.mla_decode_noalloc(*args, 8193, 32, o.data_ptr(), l.data_ptr(), s) == 3
    m.check()  # nothing was launched, nothing recorded
