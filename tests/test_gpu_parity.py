"""GPU parity: every step of the path, through the C-ABI, against the fp64 oracle.

Inputs are seeded and synthetic (head_latent_attention_26_b300.synth); the
oracle sees exactly the values the kernels see (bf16 widened to float64).
Tolerances (tests/_util.py): per-row max relative error 1e-2 on outputs,
|d lse| / max(1, |lse|) <= 2e-3, bit-exact for cache indexing.
"""

import math

import numpy as np
import pytest
import torch

import oracle as O
from head_latent_attention_26_b300 import build, synth
from _util import LSE_TOL, OUT_TOL, batch_meta, latent_inputs, lse_err, record, row_rel_err, scatter_rows, to_np

pytestmark = pytest.mark.gpu

V2 = synth.V2
TINY = synth.TINY
MAX_POS = 131072 + 64


@pytest.fixture(scope="module")
def mla_mod():
    build.build()
    from head_latent_attention_26_b300 import mla
    return mla


@pytest.fixture(scope="module")
def v2(mla_mod):
    m = mla_mod.MLA(V2, MAX_POS, torch.bfloat16)
    assert m.tensor_path
    return m


@pytest.fixture(scope="module")
def tiny(mla_mod):
    m = mla_mod.MLA(TINY, 64, torch.float32)
    assert not m.tensor_path
    return m


def _w_dkr(W):
    return torch.cat([W["W_dkv"], W["W_kr"]], dim=0).contiguous()


def _np_weights(W):
    return {k: to_np(v) for k, v in W.items()}


# ---------------------------------------------------------------------------
# Tiny layer (fp32 storage, generic kernels)
# ---------------------------------------------------------------------------

def test_tiny_layer_end_to_end(tiny):
    d, T = TINY, 64
    W = synth.weights(d, 1001, dtype=torch.float32, device="cuda")
    h = synth.hidden(T, d, 1001, dtype=torch.float32, device="cuda")
    table, n_blocks, cu_q, seq_lens, pos = batch_meta([T], [1], d.block, 1001)
    pool = torch.zeros(n_blocks, d.block, d.width, dtype=torch.float32, device="cuda")
    zeros = torch.zeros(T, dtype=torch.int32, device="cuda")
    allpos = torch.arange(T, dtype=torch.int32, device="cuda")
    tiny.cache_append(h, _w_dkr(W), zeros, allpos, table, pool)
    out = {}
    u = tiny.decode_step(h[T - 1:T].contiguous(), W, _w_dkr(W), zeros[:1], pos, table, pool, seq_lens, cu_q,
                         out=out)
    tiny.check()
    Wn = _np_weights(W)
    ref = O.decode_sequence(to_np(h), to_np(h)[T - 1], T - 1, Wn, n_h=d.n_h, base=d.rope_base)
    rows = to_np(pool.view(-1, d.width))[[O.cache_slot(table.cpu(), 0, j, d.block) for j in range(T)]]
    # fp32 storage and arithmetic: far inside the bf16 gates
    assert row_rel_err(rows, ref["rows"]) < 1e-4
    assert row_rel_err(to_np(out["q_lat"])[0], ref["q_lat"]) < 1e-4
    assert row_rel_err(to_np(out["o_lat"])[0], ref["o_lat"]) < 1e-4
    assert lse_err(to_np(out["lse"])[0], ref["lse"]) < 1e-5
    assert row_rel_err(to_np(u)[0], ref["u"]) < 1e-4


def test_tiny_every_position_sees_only_its_prefix(tiny):
    """64 sequences share one physical block; sequence t has t+1 rows, so its
    query sits at position t.  Checks the causal limit at every position."""
    d = TINY
    rows = synth.normal((64, d.width), 1002, "rows", dtype=torch.float32, device="cuda")
    q_lat = synth.normal((64, d.n_h, d.width), 1002, "q", dtype=torch.float32, device="cuda")
    pool = rows.view(1, 64, d.width).contiguous()
    table = torch.zeros(64, 1, dtype=torch.int32, device="cuda")
    seq_lens = torch.arange(1, 65, dtype=torch.int32, device="cuda")
    cu_q = torch.arange(0, 65, dtype=torch.int32, device="cuda")
    o_lat, lse = tiny.decode(q_lat, pool, table, seq_lens, cu_q)
    tiny.check()
    rn, qn = to_np(rows), to_np(q_lat)
    for t in range(64):
        o_ref, l_ref = O.attend_latent(qn[t], rn[:t + 1], d.d_c, d.d_h)
        assert row_rel_err(to_np(o_lat[t]), o_ref) < 1e-4, t
        assert lse_err(to_np(lse[t]), l_ref) < 1e-5, t


# ---------------------------------------------------------------------------
# DeepSeek-V2 sizes, bf16
# ---------------------------------------------------------------------------

def test_v2_cache_append_values_and_indexing(v2):
    d = V2
    seq_lens = [130, 64, 7]
    new = [50, 64, 7]  # append the last `new` rows of each sequence
    table, n_blocks, _, _, _ = batch_meta(seq_lens, [1, 1, 1], d.block, 1003, spare_blocks=3)
    W = synth.weights(d, 1003, device="cuda")
    x = synth.hidden(sum(new), d, 1003, device="cuda")
    seq_idx = torch.tensor(sum([[b] * n for b, n in enumerate(new)], []), dtype=torch.int32, device="cuda")
    pos = torch.tensor(sum([list(range(L - n, L)) for L, n in zip(seq_lens, new)], []), dtype=torch.int32,
                       device="cuda")
    sentinel = torch.tensor(0x3F3F, dtype=torch.int16)
    pool = torch.full((n_blocks, d.block, d.width), int(sentinel), dtype=torch.int16, device="cuda").view(torch.bfloat16)
    v2.cache_append(x, _w_dkr(W), seq_idx, pos, table, pool)
    v2.check()
    # values: oracle rows for the same tokens
    c, k_r = O.kv_latent(to_np(x), to_np(W["W_dkv"]), to_np(W["W_kr"]), to_np(pos), d.rope_base)
    ref_rows = np.concatenate([c, k_r], axis=1)
    tab = table.cpu()
    slots = [O.cache_slot(tab, int(b), int(p), d.block) for b, p in zip(seq_idx.tolist(), pos.tolist())]
    flat = pool.view(-1, d.width)
    assert row_rel_err(to_np(flat[slots]), ref_rows) < OUT_TOL
    # indexing: every other row keeps the sentinel bit pattern
    mask = torch.ones(flat.shape[0], dtype=torch.bool)
    mask[slots] = False
    untouched = flat.view(torch.int16)[mask.cuda()]
    assert bool((untouched == sentinel.cuda()).all())
    # the same tokens through an identity table land in the same bytes
    ident = torch.arange(table.numel(), dtype=torch.int32, device="cuda").view_as(table)
    pool2 = torch.zeros_like(pool)
    v2.cache_append(x, _w_dkr(W), seq_idx, pos, ident, pool2)
    v2.check()
    slots2 = [O.cache_slot(ident.cpu(), int(b), int(p), d.block) for b, p in zip(seq_idx.tolist(), pos.tolist())]
    a = flat.view(torch.int16)[slots]
    b2 = pool2.view(-1, d.width).view(torch.int16)[slots2]
    assert torch.equal(a, b2)


def test_v2_absorb_q(v2):
    d = V2
    W = synth.weights(d, 1004, device="cuda")
    n = 6
    q_c = synth.normal((n, d.n_h, d.d_h), 1004, "q_c", device="cuda")
    q_r = synth.normal((n, d.n_h, d.d_hr), 1004, "q_r", device="cuda")
    pos = torch.tensor([0, 1, 63, 4095, 70001, 131071], dtype=torch.int32, device="cuda")
    q_lat = v2.absorb_q(q_c, q_r, pos, W["W_uk"])
    v2.check()
    for i in range(n):
        ref = O.absorb_query(to_np(q_c[i]), O.rope(to_np(q_r[i]), int(pos[i]), d.rope_base), to_np(W["W_uk"]))
        assert row_rel_err(to_np(q_lat[i]), ref) < OUT_TOL, i


def _decode_case(v2, seq_lens, q_counts, seed, workers, spare=2, scale_rows=None):
    d = V2
    table, n_blocks, cu_q, lens, _ = batch_meta(seq_lens, q_counts, d.block, seed, spare_blocks=spare)
    n_tok = int(sum(q_counts))
    q_lat, rows = latent_inputs(d, n_tok, int(sum(seq_lens)), seed)
    if scale_rows is not None:
        rows[scale_rows.cuda()] *= 8  # exact in bf16
    per_seq = list(torch.split(rows, [int(t) for t in seq_lens]))
    pool = scatter_rows(per_seq, table, n_blocks, d.block, d.width, fill=float("nan"))
    o_lat, lse = v2.decode(q_lat, pool, table, lens, cu_q, num_workers=workers)
    v2.check()
    return q_lat, per_seq, table, cu_q, o_lat, lse


def _check_tokens(d, q_lat, per_seq, seq_lens, q_counts, o_lat, lse, tokens=None, heads=None, case=None):
    qn = None
    cu = np.concatenate([[0], np.cumsum(q_counts)])
    for b, L in enumerate(seq_lens):
        rows_b = None
        for k in range(int(q_counts[b])):
            n = int(cu[b]) + k
            if tokens is not None and n not in tokens:
                continue
            if rows_b is None:
                rows_b = to_np(per_seq[b])
            t = int(L) - int(q_counts[b]) + k
            q = to_np(q_lat[n]) if qn is None else qn[n]
            hs = list(range(d.n_h)) if heads is None else heads
            o_ref, l_ref = O.attend_latent(q, rows_b[:t + 1], d.d_c, d.d_h, heads=hs)
            e_o = row_rel_err(to_np(o_lat[n])[hs], o_ref)
            e_l = lse_err(to_np(lse[n])[hs], l_ref)
            if case:
                record(case, e_o, e_l)
            assert e_o < OUT_TOL and e_l < LSE_TOL, (b, n, t, e_o, e_l)


@pytest.mark.parametrize("seq_lens,q_counts,workers", [
    ([1], [1], 0),
    ([64], [1], 0),
    ([65], [1], 0),
    ([200], [1], 0),
    ([200], [1], 1),
    ([127, 63, 300, 1000], [1, 2, 1, 2], 0),
    ([127, 63, 300, 1000], [1, 2, 1, 2], 1),
    ([127, 63, 300, 1000], [1, 2, 1, 2], 3),
    ([127, 63, 300, 1000], [1, 2, 1, 2], 7),
    ([127, 63, 300, 1000], [1, 2, 1, 2], 40),
])
def test_v2_decode_tensor_path(v2, seq_lens, q_counts, workers):
    q_lat, per_seq, _, _, o_lat, lse = _decode_case(v2, seq_lens, q_counts, 1005 + sum(seq_lens), workers)
    _check_tokens(V2, q_lat, per_seq, seq_lens, q_counts, o_lat, lse, case="decode small cases")


def test_v2_decode_split_matches_unsplit(v2):
    seq_lens, q_counts = [2500, 1300], [1, 2]
    results = {}
    for w in (1, 2, 5, 74, 150):
        q_lat, per_seq, _, _, o_lat, lse = _decode_case(v2, seq_lens, q_counts, 1006, w)
        results[w] = (to_np(o_lat), to_np(lse))
    _check_tokens(V2, q_lat, per_seq, seq_lens, q_counts, o_lat, lse, case="decode split 1..150 workers")
    base_o, base_l = results[1]
    for w, (o, l) in results.items():
        assert row_rel_err(o, base_o) < OUT_TOL and lse_err(l, base_l) < LSE_TOL, w


def test_v2_layer_end_to_end(v2):
    """Whole step from hidden states: append 200 rows, query the last one,
    u against the expanded (K and V per head) fp64 oracle for all heads."""
    d, T = V2, 200
    W = synth.weights(d, 1007, device="cuda")
    h = synth.hidden(T, d, 1007, device="cuda")
    table, n_blocks, cu_q, seq_lens, pos = batch_meta([T], [1], d.block, 1007)
    pool = torch.zeros(n_blocks, d.block, d.width, dtype=torch.bfloat16, device="cuda")
    zeros = torch.zeros(T, dtype=torch.int32, device="cuda")
    allpos = torch.arange(T, dtype=torch.int32, device="cuda")
    v2.cache_append(h[:T - 1].contiguous(), _w_dkr(W), zeros[:T - 1], allpos[:T - 1], table, pool)
    out = {}
    u = v2.decode_step(h[T - 1:].contiguous(), W, _w_dkr(W), zeros[:1], pos, table, pool, seq_lens, cu_q,
                       out=out)
    v2.check()
    ref = O.decode_sequence(to_np(h), to_np(h)[T - 1], T - 1, _np_weights(W), n_h=d.n_h, base=d.rope_base)
    errs = {k: row_rel_err(to_np(out[k])[0], ref[k]) for k in ("q_lat", "o_lat")}
    errs["u"] = row_rel_err(to_np(u)[0], ref["u"])
    e_l = lse_err(to_np(out["lse"])[0], ref["lse"])
    for k, e in errs.items():
        record(f"T=200 layer from h: {k}", e, e_l if k == "o_lat" else None)
    assert all(e < OUT_TOL for e in errs.values()) and e_l < LSE_TOL, (errs, e_l)


@pytest.mark.parametrize("n_new", [1, 64, 300])
def test_q_proj_append_matches_the_two_calls(v2, n_new):
    """mla_q_proj_append (W^DQ and the cache-row product in one launch) against
    mla_q_proj + mla_cache_append on the same tokens: the same pool rows
    written (every other row keeps its sentinel, bit for bit), the rows and
    the query parts equal up to the order of the fp32 sums, and both against
    the oracle's cache rows and query parts."""
    d = V2
    seed = 1400 + n_new
    W = synth.weights(d, seed, device="cuda")
    x = synth.hidden(n_new, d, seed, device="cuda")
    lens = [n_new + 37]
    table, n_blocks, _, _, _ = batch_meta(lens, [n_new], d.block, seed, spare_blocks=2)
    seq_idx = torch.zeros(n_new, dtype=torch.int32, device="cuda")
    pos = torch.arange(37, 37 + n_new, dtype=torch.int32, device="cuda")
    sentinel = torch.full((n_blocks, d.block, d.width), 0x3F3F, dtype=torch.int16, device="cuda")
    pool_a = sentinel.clone().view(torch.bfloat16)
    pool_b = sentinel.clone().view(torch.bfloat16)
    q_c_a, q_r_a = v2.q_proj_append(x, W["W_dq"], W["W_uq"], W["W_qr"], _w_dkr(W), seq_idx, pos, table, pool_a)
    q_c_b, q_r_b = v2.q_proj(x, W["W_dq"], W["W_uq"], W["W_qr"])
    v2.cache_append(x, _w_dkr(W), seq_idx, pos, table, pool_b)
    v2.check()
    written_a = pool_a.view(torch.int16) != 0x3F3F
    written_b = pool_b.view(torch.int16) != 0x3F3F
    assert torch.equal(written_a.any(-1), written_b.any(-1))
    tab = table.cpu()
    slots = [O.cache_slot(tab, 0, int(p_), d.block) for p_ in pos.tolist()]
    rows_a = pool_a.view(-1, d.width)[slots]
    rows_b = pool_b.view(-1, d.width)[slots]
    assert int(written_a.view(-1, d.width).any(-1).sum()) == n_new
    assert row_rel_err(to_np(rows_a), to_np(rows_b)) < 2 ** -7
    assert row_rel_err(to_np(q_c_a), to_np(q_c_b)) < 2 ** -6 and row_rel_err(to_np(q_r_a), to_np(q_r_b)) < 2 ** -6
    Wn = _np_weights(W)
    c_ref, kr_ref = O.kv_latent(to_np(x), Wn["W_dkv"], Wn["W_kr"], pos.cpu().numpy(), d.rope_base)
    _, qc_ref, qr_ref = O.query_parts(to_np(x), Wn["W_dq"], Wn["W_uq"], Wn["W_qr"], d.n_h)
    e_rows = row_rel_err(to_np(rows_a), np.concatenate([c_ref, kr_ref], axis=1))
    e_qc, e_qr = row_rel_err(to_np(q_c_a), qc_ref), row_rel_err(to_np(q_r_a), qr_ref)
    record("q_proj_append: cache rows / q_c / q_r", max(e_rows, e_qc, e_qr))
    assert e_rows < OUT_TOL and e_qc < OUT_TOL and e_qr < OUT_TOL, (e_rows, e_qc, e_qr)


@pytest.mark.parametrize("n_new", [1, 64, 100])
def test_q_latent_append(v2, n_new):
    """mla_q_latent_append (up to 64 tokens: W^DQ with the cache rows, then per
    head W^UQ_i and W^UK_i^T chained on chip, and W^QR with RoPE; beyond 64:
    the separate kernels) against the oracle's latent query and cache rows,
    every other pool row untouched, and against the separate route."""
    d = V2
    seed = 1500 + n_new
    W = synth.weights(d, seed, device="cuda")
    x = synth.hidden(n_new, d, seed, device="cuda")
    lens = [n_new + 21]
    table, n_blocks, _, _, _ = batch_meta(lens, [n_new], d.block, seed, spare_blocks=2)
    seq_idx = torch.zeros(n_new, dtype=torch.int32, device="cuda")
    pos = torch.arange(21, 21 + n_new, dtype=torch.int32, device="cuda")
    sentinel = torch.full((n_blocks, d.block, d.width), 0x3F3F, dtype=torch.int16, device="cuda")
    pool_a = sentinel.clone().view(torch.bfloat16)
    pool_b = sentinel.clone().view(torch.bfloat16)
    q_lat = v2.q_latent_append(x, W["W_dq"], W["W_uq"], W["W_qr"], W["W_uk"], _w_dkr(W), seq_idx, pos, table, pool_a)
    q_c, q_r = v2.q_proj_append(x, W["W_dq"], W["W_uq"], W["W_qr"], _w_dkr(W), seq_idx, pos, table, pool_b)
    q_lat_b = v2.absorb_q(q_c, q_r, pos, W["W_uk"])
    v2.check()
    written = (pool_a.view(torch.int16) != 0x3F3F).view(-1, d.width).any(-1)
    tab = table.cpu()
    slots = [O.cache_slot(tab, 0, int(p_), d.block) for p_ in pos.tolist()]
    assert int(written.sum()) == n_new and bool(written[slots].all())
    Wn = _np_weights(W)
    xn = to_np(x)
    c_ref, kr_ref = O.kv_latent(xn, Wn["W_dkv"], Wn["W_kr"], pos.cpu().numpy(), d.rope_base)
    e_rows = row_rel_err(to_np(pool_a.view(-1, d.width)[slots]), np.concatenate([c_ref, kr_ref], axis=1))
    _, qc_ref, qr_raw = O.query_parts(xn, Wn["W_dq"], Wn["W_uq"], Wn["W_qr"], d.n_h)
    lat_ref = np.stack([O.absorb_query(qc_ref[n], O.rope(qr_raw[n], int(pos[n]), d.rope_base), Wn["W_uk"])
                        for n in range(n_new)])
    e_lat = row_rel_err(to_np(q_lat), lat_ref)
    record("q_latent_append: q_lat", e_lat)
    record("q_latent_append: cache rows", e_rows)
    assert e_lat < OUT_TOL and e_rows < OUT_TOL, (e_lat, e_rows)
    # the separate route rounds q^C and q^R to bf16 at the same points up to
    # the order of the sums (and rotates the stored q^R): a few bf16 steps
    assert row_rel_err(to_np(q_lat), to_np(q_lat_b)) < 2 ** -5


# ---------------------------------------------------------------------------
# Full-size workloads, sampled outputs, in the launch configuration of the bench
# ---------------------------------------------------------------------------

def test_v2_config_b1_t4096_end_to_end(v2):
    """B=1, T=4096: the cache is built by mla_cache_append from h ~ N(0,1);
    the last token's output u is checked against the expanded oracle."""
    d, T = V2, 4096
    W = synth.weights(d, 1008, device="cuda")
    h = synth.hidden(T, d, 1008, device="cuda")
    table, n_blocks, cu_q, seq_lens, pos = batch_meta([T], [1], d.block, 1008)
    pool = torch.zeros(n_blocks, d.block, d.width, dtype=torch.bfloat16, device="cuda")
    zeros = torch.zeros(T, dtype=torch.int32, device="cuda")
    allpos = torch.arange(T, dtype=torch.int32, device="cuda")
    v2.cache_append(h[:T - 1].contiguous(), _w_dkr(W), zeros[:T - 1], allpos[:T - 1], table, pool)
    out = {}
    u = v2.decode_step(h[T - 1:].contiguous(), W, _w_dkr(W), zeros[:1], pos, table, pool, seq_lens, cu_q,
                       out=out)
    v2.check()
    ref = O.decode_sequence(to_np(h), to_np(h)[T - 1], T - 1, _np_weights(W), n_h=d.n_h, base=d.rope_base)
    e_o, e_l = row_rel_err(to_np(out["o_lat"])[0], ref["o_lat"]), lse_err(to_np(out["lse"])[0], ref["lse"])
    e_u = row_rel_err(to_np(u)[0], ref["u"])
    record("B=1 T=4096 layer from h: o_lat / lse", e_o, e_l)
    record("B=1 T=4096 layer from h: u", e_u)
    assert e_o < OUT_TOL and e_l < LSE_TOL and e_u < OUT_TOL


def test_v2_config_b64_t4096_all_tokens(v2):
    """B=64, T=4096, permuted pool, the bench's launch configuration: every
    token, every head."""
    B, T = 64, 4096
    seq_lens, q_counts = [T] * B, [1] * B
    q_lat, per_seq, _, _, o_lat, lse = _decode_case(v2, seq_lens, q_counts, 1009, 0)
    _check_tokens(V2, q_lat, per_seq, seq_lens, q_counts, o_lat, lse, case="B=64 T=4096 decode (64 tokens)")


def test_v2_config_b1_t131072_hot_rows(v2):
    """B=1, T=131072 (128K context), 1% of rows scaled by 8: split-KV over all workers."""
    T = 131072
    hot = synth.pick_rows(T, 0.01, 1010)
    q_lat, per_seq, _, _, o_lat, lse = _decode_case(v2, [T], [1], 1010, 0, scale_rows=hot)
    _check_tokens(V2, q_lat, per_seq, [T], [1], o_lat, lse, case="B=1 T=131072 hot rows decode")


def test_v2_config_ragged_b128(v2):
    """B=128, lengths U[512,16384], 1 or 2 queries each; the newest rows are
    appended by mla_cache_append in the same run into a pool whose every other
    row holds a sentinel bit pattern.  Counts the cache bytes the pool holds
    after the append against (d_c + d_hr) * sum(T) * 2, checks that the append
    wrote exactly the new tokens' rows, and checks 48 sampled tokens plus every
    token of the first eight sequences against the oracle."""
    d, B = V2, 128
    seed = 1011
    lens = synth.ragged_lengths(B, 512, 16384, seed).tolist()
    qc = synth.query_counts(B, seed).tolist()
    table, n_blocks, cu_q, seq_lens, pos = batch_meta(lens, qc, d.block, seed, spare_blocks=3)
    n_tok = sum(qc)
    q_lat, rows = latent_inputs(d, n_tok, sum(lens), seed)
    per_seq = list(torch.split(rows, lens))
    # prior rows (all but each sequence's newest q_len) placed by the test;
    # everything else keeps the sentinel
    sentinel = 0x3F3F
    prior = [r[:L - q] for r, L, q in zip(per_seq, lens, qc)]
    pool = scatter_rows(prior, table, n_blocks, d.block, d.width)
    flat = pool.view(-1, d.width)
    written = torch.zeros(flat.shape[0], dtype=torch.bool, device="cuda")
    for b, r in enumerate(prior):
        j = torch.arange(r.shape[0], device="cuda")
        written[table[b][j // d.block].long() * d.block + (j % d.block)] = True
    flat.view(torch.int16)[~written] = sentinel
    before = flat.view(torch.int16).clone()
    W = synth.weights(d, seed, device="cuda")
    x = synth.hidden(n_tok, d, seed, device="cuda")
    seq_idx = torch.tensor(sum([[b] * q for b, q in enumerate(qc)], []), dtype=torch.int32, device="cuda")
    v2.cache_append(x, _w_dkr(W), seq_idx, pos, table, pool)
    o_lat, lse = v2.decode(q_lat, pool, table, seq_lens, cu_q)
    v2.check()
    after = flat.view(torch.int16)
    holds = (after != sentinel).any(dim=1)
    # the cache the pool holds: every sequence's T_b rows of d_c + d_hr bf16 values
    assert int(holds.sum()) * d.width * 2 == O.latent_cache_bytes(1, sum(lens), 1, d.d_c, d.d_hr, 2)
    # the append changed exactly the new tokens' rows, at the oracle's slots
    changed = torch.nonzero((after != before).any(dim=1)).flatten().cpu().tolist()
    tab = table.cpu()
    slots = [O.cache_slot(tab, int(b), int(p), d.block) for b, p in zip(seq_idx.tolist(), pos.tolist())]
    assert sorted(changed) == sorted(slots)
    c, k_r = O.kv_latent(to_np(x), to_np(W["W_dkv"]), to_np(W["W_kr"]), to_np(pos), d.rope_base)
    new_rows = np.concatenate([c, k_r], axis=1)
    e_rows = row_rel_err(to_np(flat[slots]), new_rows)
    record("ragged B=128 appended rows", e_rows)
    assert e_rows < OUT_TOL
    cu = np.concatenate([[0], np.cumsum(qc)])
    rng = np.random.default_rng(seed)
    picks = set(rng.choice(n_tok, 48, replace=False).tolist()) | set(range(int(cu[8])))
    for n in sorted(picks):
        b = int(np.searchsorted(cu, n, side="right") - 1)
        L = lens[b]
        t = L - (int(cu[b + 1]) - n)
        rows_b = to_np(per_seq[b])
        rows_b[L - qc[b]:] = new_rows[int(cu[b]):int(cu[b + 1])]
        o_ref, l_ref = O.attend_latent(to_np(q_lat[n]), rows_b[:t + 1], d.d_c, d.d_h)
        e_o, e_l = row_rel_err(to_np(o_lat[n]), o_ref), lse_err(to_np(lse[n]), l_ref)
        record("ragged B=128 decode (%d tokens)" % len(picks), e_o, e_l)
        assert e_o < OUT_TOL and e_l < LSE_TOL, (n, e_o, e_l)


# ---------------------------------------------------------------------------
# Errors: host validation, device bounds, bounded waits
# ---------------------------------------------------------------------------

def test_host_validation(v2, mla_mod):
    d = V2
    q_lat, _ = latent_inputs(d, 1, 64, 1012)
    pool = torch.zeros(1, d.block, d.width, dtype=torch.bfloat16, device="cuda")
    table = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
    lens = torch.tensor([10], dtype=torch.int32, device="cuda")
    cu_q = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    with pytest.raises(mla_mod.MLAError) as e:  # misaligned q_lat
        bad = torch.empty(q_lat.numel() + 8, dtype=torch.bfloat16, device="cuda")[1:1 + q_lat.numel()].view_as(q_lat)
        v2.decode(bad, pool, table, lens, cu_q)
    assert e.value.code == 1
    with pytest.raises(mla_mod.MLAError) as e:  # workspace too small
        v2.decode(q_lat, pool, table, lens, cu_q, ws=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.code == 3


def test_device_bounds_error_is_reported_not_faulted(v2):
    d = V2
    q_lat, rows = latent_inputs(d, 1, 128, 1013)
    pool = rows.view(2, d.block, d.width).contiguous()
    table = torch.tensor([[0, 7]], dtype=torch.int32, device="cuda")  # block 7 is outside the 2-block pool
    lens = torch.tensor([128], dtype=torch.int32, device="cuda")
    cu_q = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    v2.decode(q_lat, pool, table, lens, cu_q)
    assert v2.device_status() == 6
    assert v2.device_status() == 0  # reading clears it
    # and the library is still usable
    table_ok = torch.tensor([[0, 1]], dtype=torch.int32, device="cuda")
    v2.decode(q_lat, pool, table_ok, lens, cu_q)
    v2.check()


def test_bounded_wait_times_out_cleanly(v2):
    v2.set_wait_limit(1000)
    try:
        assert v2.selftest_wait_timeout() == 5
    finally:
        v2.set_wait_limit(0)
    v2.check()


# ---------------------------------------------------------------------------
# Projection kernels at every token-tile width (64 / 128 / 256 and several
# 256-token tiles), against the oracle's own projections
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n_tok", [1, 5, 64, 100, 300])
def test_v2_projections_token_tiles(v2, n_tok):
    d = V2
    seed = 1020 + n_tok
    W = synth.weights(d, seed, device="cuda")
    x = synth.hidden(n_tok, d, seed, device="cuda")
    q_c, q_r = v2.q_proj(x, W["W_dq"], W["W_uq"], W["W_qr"])
    o_lat = synth.normal((n_tok, d.n_h, d.d_c), seed, "o_lat", device="cuda")
    u = v2.out(o_lat, W["W_uv"], W["W_o"])
    v2.check()
    Wn = _np_weights(W)
    _, qc_ref, qr_ref = O.query_parts(to_np(x), Wn["W_dq"], Wn["W_uq"], Wn["W_qr"], d.n_h)
    rng = np.random.default_rng(seed)
    for n in sorted(set(rng.choice(n_tok, min(n_tok, 6), replace=False).tolist()) | {n_tok - 1}):
        assert row_rel_err(to_np(q_c[n]), qc_ref[n]) < OUT_TOL, n
        assert row_rel_err(to_np(q_r[n]), qr_ref[n]) < OUT_TOL, n
        u_ref = O.output_projection(O.up_project(to_np(o_lat[n]), Wn["W_uv"]), Wn["W_o"])
        assert row_rel_err(to_np(u[n]), u_ref) < OUT_TOL, n


def test_v2_cache_append_many_tokens(v2):
    """300 new rows of 3 sequences in one call (two 256-token tiles)."""
    d = V2
    seq_lens = [180, 64, 56]
    table, n_blocks, _, _, _ = batch_meta(seq_lens, [1, 1, 1], d.block, 1030, spare_blocks=1)
    W = synth.weights(d, 1030, device="cuda")
    x = synth.hidden(sum(seq_lens), d, 1030, device="cuda")
    seq_idx = torch.tensor(sum([[b] * n for b, n in enumerate(seq_lens)], []), dtype=torch.int32, device="cuda")
    pos = torch.tensor(sum([list(range(n)) for n in seq_lens], []), dtype=torch.int32, device="cuda")
    pool = torch.zeros(n_blocks, d.block, d.width, dtype=torch.bfloat16, device="cuda")
    v2.cache_append(x, _w_dkr(W), seq_idx, pos, table, pool)
    v2.check()
    c, k_r = O.kv_latent(to_np(x), to_np(W["W_dkv"]), to_np(W["W_kr"]), to_np(pos), d.rope_base)
    tab = table.cpu()
    slots = [O.cache_slot(tab, int(b), int(p), d.block) for b, p in zip(seq_idx.tolist(), pos.tolist())]
    assert row_rel_err(to_np(pool.view(-1, d.width)[slots]), np.concatenate([c, k_r], axis=1)) < OUT_TOL


@pytest.mark.parametrize("n_tok", [1, 70, 260])
def test_v2_absorb_q_token_tiles(v2, n_tok):
    d = V2
    seed = 1040 + n_tok
    W = synth.weights(d, seed, device="cuda")
    q_c = synth.normal((n_tok, d.n_h, d.d_h), seed, "q_c", device="cuda")
    q_r = synth.normal((n_tok, d.n_h, d.d_hr), seed, "q_r", device="cuda")
    pos = torch.randint(0, MAX_POS, (n_tok,), generator=torch.Generator().manual_seed(seed),
                        dtype=torch.int32).cuda()
    q_lat = v2.absorb_q(q_c, q_r, pos, W["W_uk"])
    v2.check()
    for n in sorted({0, n_tok // 2, n_tok - 1}):
        ref = O.absorb_query(to_np(q_c[n]), O.rope(to_np(q_r[n]), int(pos[n]), d.rope_base), to_np(W["W_uk"]))
        assert row_rel_err(to_np(q_lat[n]), ref) < OUT_TOL, n


# ---------------------------------------------------------------------------
# Folded query weight W~^UQ_i = W^UK_i^T W^UQ_i and the latent query from c^Q
# ---------------------------------------------------------------------------

def test_tiny_folded_query(tiny):
    d, n = TINY, 5
    W = synth.weights(d, 1050, dtype=torch.float32, device="cuda")
    x = synth.hidden(n, d, 1050, dtype=torch.float32, device="cuda")
    pos = torch.tensor([0, 1, 17, 40, 63], dtype=torch.int32, device="cuda")
    W_abs = tiny.absorb_weights(W["W_uq"], W["W_uk"])
    q_lat = tiny.q_proj_absorbed(x, W["W_dq"], W_abs, W["W_qr"], pos)
    tiny.check()
    Wn = _np_weights(W)
    W_abs_ref = O.absorbed_query_weight(Wn["W_uq"], Wn["W_uk"], d.n_h)
    assert row_rel_err(to_np(W_abs), W_abs_ref) < 1e-5
    c_q, q_c, q_r_raw = O.query_parts(to_np(x), Wn["W_dq"], Wn["W_uq"], Wn["W_qr"], d.n_h)
    for i in range(n):
        q_r = O.rope(q_r_raw[i], int(pos[i]), d.rope_base)
        ref = O.latent_query_precomputed(c_q[i], W_abs_ref, q_r, d.n_h)
        # the same latent query by the runtime route
        assert np.max(np.abs(ref - O.absorb_query(q_c[i], q_r, Wn["W_uk"]))) <= 1e-12 * np.max(np.abs(ref))
        assert row_rel_err(to_np(q_lat[i]), ref) < 1e-4, i


def test_v2_folded_weight(v2):
    d = V2
    W = synth.weights(d, 1051, device="cuda")
    W_abs = v2.absorb_weights(W["W_uq"], W["W_uk"])
    v2.check()
    assert W_abs.shape == (d.n_h * d.d_c, d.d_cq)
    W_uq, W_uk = to_np(W["W_uq"]), to_np(W["W_uk"])
    for i in (0, 1, 77, 127):
        rows = slice(i * d.d_h, (i + 1) * d.d_h)
        ref = O.absorbed_query_weight(W_uq[rows], W_uk[rows], 1)
        got = to_np(W_abs[i * d.d_c:(i + 1) * d.d_c])
        # fp32 sums of 128 products rounded once to bf16
        assert row_rel_err(got, ref) < 1e-2, i
        assert np.max(np.abs(got - ref)) <= 2 ** -8 * np.max(np.abs(ref)), i


@pytest.mark.parametrize("n_tok", [1, 64, 100, 300])
def test_v2_q_proj_absorbed_token_tiles(v2, n_tok):
    d = V2
    seed = 1060 + n_tok
    W = synth.weights(d, seed, device="cuda")
    x = synth.hidden(n_tok, d, seed, device="cuda")
    pos = torch.randint(0, MAX_POS, (n_tok,), generator=torch.Generator().manual_seed(seed),
                        dtype=torch.int32).cuda()
    W_abs = v2.absorb_weights(W["W_uq"], W["W_uk"])
    q_lat = v2.q_proj_absorbed(x, W["W_dq"], W_abs, W["W_qr"], pos)
    # the runtime route on the same inputs, for the same tokens
    q_c, q_r = v2.q_proj(x, W["W_dq"], W["W_uq"], W["W_qr"])
    q_lat_rt = v2.absorb_q(q_c, q_r, pos, W["W_uk"])
    v2.check()
    Wn = _np_weights(W)
    picks = sorted({0, n_tok // 3, n_tok // 2, n_tok - 1})
    c_q, q_c_ref, q_r_raw = O.query_parts(to_np(x[picks]), Wn["W_dq"], Wn["W_uq"], Wn["W_qr"], d.n_h)
    for j, n in enumerate(picks):
        ref = O.absorb_query(q_c_ref[j], O.rope(q_r_raw[j], int(pos[n]), d.rope_base), Wn["W_uk"])
        assert row_rel_err(to_np(q_lat[n]), ref) < OUT_TOL, n
        assert row_rel_err(to_np(q_lat_rt[n]), ref) < OUT_TOL, n
