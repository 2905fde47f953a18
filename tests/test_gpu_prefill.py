"""GPU parity of the prefill path (the prompt's keys and values expanded per
head, then causal attention over every prompt position; [perforder]
"極限最適化の代償：MLA特有の学習負荷と独自Tritonカーネルという障壁", [kasblo]
"「キャッシュを減らせた」と「その割合だけ速い」は別の評価") through the C-ABI,
against the oracle's prefill_expanded on the same h and weights.

The cache rows come from mla_cache_append (identity block table, so the pool
is the rows in position order) and q^C, q^R from mla_q_proj.  Like the decode
tests, which hand both sides the same bf16 latent queries, the parity tests
hand the oracle's prefill_from_parts the same bf16 rows and query parts the
GPU prefill reads, so what is compared is the prefill's own arithmetic (the
expansion, the scores, the softmax and the weighted sum), at the gates of the
decode path.  (Run from h itself, the oracle's prefill_expanded also
differs from the GPU by the bf16 rounding of the query parts and the cache
rows, which a single key's lse, equal to one score, shows in full; that is
the earlier steps' rounding, not the prefill's.)
"""

import numpy as np
import pytest
import torch

import oracle as O
from head_latent_attention_26_b300 import build, synth
from _util import LSE_TOL, OUT_TOL, lse_err, record, row_rel_err, to_np

pytestmark = pytest.mark.gpu

V2 = synth.V2


@pytest.fixture(scope="module")
def v2():
    build.build()
    from head_latent_attention_26_b300 import mla
    m = mla.MLA(V2, 4096, torch.bfloat16)
    assert m.tensor_path
    return m


def _prefill_parts(v2, P, seed, h=None, W=None):
    """The GPU prefill and the bf16 inputs it read (rows, q^C, q^R)."""
    d = V2
    W = synth.weights(d, seed, device="cuda") if W is None else W
    h = synth.hidden(P, d, seed, device="cuda") if h is None else h
    n_blocks = (P + d.block - 1) // d.block
    table = torch.arange(n_blocks, dtype=torch.int32, device="cuda").view(1, -1)
    pool = torch.zeros(n_blocks, d.block, d.width, dtype=torch.bfloat16, device="cuda")
    zeros = torch.zeros(P, dtype=torch.int32, device="cuda")
    pos = torch.arange(P, dtype=torch.int32, device="cuda")
    v2.cache_append(h, torch.cat([W["W_dkv"], W["W_kr"]], dim=0).contiguous(), zeros, pos, table, pool)
    q_c, q_r = v2.q_proj(h, W["W_dq"], W["W_uq"], W["W_qr"])
    rows = pool.view(-1, d.width)[:P]
    o, lse = v2.prefill(rows, q_c, q_r, W["W_uk"], W["W_uv"])
    v2.check()
    return dict(h=h, W=W, rows=rows, q_c=q_c, q_r=q_r, o=o, lse=lse)


def _oracle_parts(r):
    rows = to_np(r["rows"])
    return O.prefill_from_parts(rows[:, :V2.d_c], rows[:, V2.d_c:], to_np(r["q_c"]), to_np(r["q_r"]),
                                to_np(r["W"]["W_uk"]), to_np(r["W"]["W_uv"]), base=V2.rope_base)


@pytest.mark.parametrize("P", [1, 64, 128, 130, 300])
def test_prefill_matches_oracle(v2, P):
    """Every position and head: one key, one partial tile, exactly one tile,
    a ragged second tile, three tiles with a ragged tail."""
    r = _prefill_parts(v2, P, 1300 + P)
    o_ref, lse_ref = _oracle_parts(r)
    e_o, e_l = row_rel_err(to_np(r["o"]), o_ref), lse_err(to_np(r["lse"]), lse_ref)
    record("prefill P<=300 (every position)", e_o, e_l)
    assert e_o < OUT_TOL and e_l < LSE_TOL, (e_o, e_l)


def test_prefill_is_causal(v2):
    """Changing the last prompt token leaves every earlier position's output
    bit for bit unchanged (each row sees only keys at or before it)."""
    P = 260
    d = V2
    W = synth.weights(d, 1311, device="cuda")
    h = synth.hidden(P, d, 1311, device="cuda")
    r1 = _prefill_parts(v2, P, 1311, h=h, W=W)
    o1, l1 = r1["o"].clone(), r1["lse"].clone()
    h2 = h.clone()
    h2[P - 1] = synth.hidden(1, d, 1312, device="cuda")[0]
    r2 = _prefill_parts(v2, P, 1311, h=h2, W=W)
    o2, l2 = r2["o"], r2["lse"]
    assert torch.equal(o1[:P - 1], o2[:P - 1]) and torch.equal(l1[:P - 1], l2[:P - 1])
    assert not torch.equal(o1[P - 1], o2[P - 1])


def test_prefill_p2048_sampled_rows(v2):
    """P=2048 (16 query tiles, 16 key tiles on the last): the oracle on the
    first 2048 positions, compared at sampled positions of every tile."""
    P = 2048
    r = _prefill_parts(v2, P, 1313)
    rows = sorted(set([0, 1, 127, 128, 129, 1023, 1024, 2046, 2047] + list(range(5, P, 97))))
    o_ref, lse_ref = _oracle_parts(r)
    e_o = row_rel_err(to_np(r["o"])[rows], o_ref[rows])
    e_l = lse_err(to_np(r["lse"])[rows], lse_ref[rows])
    record("prefill P=2048 sampled positions", e_o, e_l)
    assert e_o < OUT_TOL and e_l < LSE_TOL, (e_o, e_l)


def test_prefill_rejects_other_dims(v2):
    from head_latent_attention_26_b300 import mla
    tiny = mla.MLA(synth.TINY, 64, torch.float32)
    rows = torch.zeros(4, 20, dtype=torch.float32, device="cuda")
    q = torch.zeros(4, 4, 8, dtype=torch.float32, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        tiny.prefill(rows, q, q, q, q)
    assert e.value.code == 2
