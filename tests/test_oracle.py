"""Pins of the fp64 oracle against what the pages and plain mathematics fix.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong scale) fails at least one:

* the pages' worked example (tests/golden/worked_example.json);
* the pages' cache-size numbers (tests/golden/cache_sizes.json);
* RoPE closed forms (2-D rotation, the second frequency, invariants);
* softmax special cases (one key, equal scores, huge gaps, ln-weights);
* a two-head attention case whose outputs are computed by hand;
* the absorbed-versus-expanded identity;
* brute-force scalar loops on tiny inputs.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# The pages' worked example: score 7 in both orders
# --------------------------------------------------------------------------

def test_worked_example_both_orders():
    g = _golden("worked_example.json")
    U = np.array(g["U"], dtype=float)
    c = np.array([g["c"]], dtype=float)
    q = np.array(g["q"], dtype=float)
    no_rope = np.zeros((1, 0))
    # expand first: k = U c, then q . k
    k_c, v = O.expand_kv(c, U, U, 0, d_h=3)
    assert k_c[0].tolist() == g["k"]
    s_expanded = O.scores_expanded(q, no_rope[0], k_c, no_rope)
    assert s_expanded.tolist() == [g["score"]]
    # absorb first: U^T q, then . c
    q_lat = O.absorb_query(q[None], no_rope, U)
    assert q_lat[0].tolist() == g["Ut_q"]
    s_latent = O.scores_latent(q_lat[0], c)
    assert s_latent.tolist() == [g["score"]]


def test_worked_example_precomputed_weight():
    # The same example with the query itself produced by an up-projection:
    # W^UQ = [[1,0],[0,1],[1,0]] maps c^Q = (1,2) to q = (1,2,1), so the folded
    # weight W^UK^T W^UQ must send c^Q straight to U^T q = (2,3), and the
    # score against c is 7 again.  The folded weight's entries are fixed by
    # hand: folding in the other order, W^UQ^T W^UK, gives [[2,1],[0,1]].
    g = _golden("worked_example.json")
    U = np.array(g["U"], dtype=float)
    W_uq = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 0.0]])
    c_q = np.array([1.0, 2.0])
    assert (W_uq @ c_q).tolist() == g["q"]
    W_abs = O.absorbed_query_weight(W_uq, U, n_h=1)
    assert W_abs.tolist() == [[2.0, 0.0], [1.0, 1.0]]
    q_lat = O.latent_query_precomputed(c_q, W_abs, np.zeros((1, 0)), n_h=1)
    assert q_lat[0].tolist() == g["Ut_q"]
    assert O.scores_latent(q_lat[0], np.array([g["c"]], float)).tolist() == [g["score"]]
    assert (W_uq.T @ U).tolist() == [[2.0, 1.0], [0.0, 1.0]]


def test_worked_example_rejects_transposed_weight():
    # Using U^T where U belongs would change the answer (and the shapes).
    g = _golden("worked_example.json")
    U = np.array(g["U"], dtype=float)
    with pytest.raises(ValueError):
        O.expand_kv(np.array([g["c"]], float), U.T, U.T, 0, d_h=2)[0] @ np.array(g["q"], float)


# --------------------------------------------------------------------------
# Cache sizes and element counts
# --------------------------------------------------------------------------

def test_cache_size_closed_form():
    g = _golden("cache_sizes.json")
    for case in g["cases"]:
        n = O.latent_cache_bytes(case["B"], case["T"], case["L"], case["d_c"], case["d_r"], case["s"])
        if "bytes" in case:
            assert n == case["bytes"]
        assert n == case["MiB"] * 1024 * 1024
    assert O.mha_cache_elements(128, 128) == g["mha_elements_per_token"]["value"]
    assert O.mla_cache_elements(512, 64) == g["mla_elements_per_token"]["value"]
    assert round(O.mha_cache_elements(128, 128) / O.mla_cache_elements(512, 64)) == 57


def test_cache_slot_formula():
    table = [[5, 2, 7], [0, 3, -1]]
    assert O.cache_slot(table, 0, 0, 64) == 5 * 64
    assert O.cache_slot(table, 0, 63, 64) == 5 * 64 + 63
    assert O.cache_slot(table, 0, 64, 64) == 2 * 64
    assert O.cache_slot(table, 0, 130, 64) == 7 * 64 + 2
    assert O.cache_slot(table, 1, 127, 64) == 3 * 64 + 63


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------

def test_rope_position_zero_is_identity():
    x = np.random.default_rng(0).standard_normal((5, 8))
    assert np.array_equal(O.rope(x, 0), x)


def test_rope_two_d_rotation_closed_form():
    # d = 2: theta_0 = base^0 = 1, so position p turns (1, 0) into (cos p, sin p)
    for p in [1, 2, 7, 100]:
        y = O.rope(np.array([1.0, 0.0]), p)
        assert np.allclose(y, [math.cos(p), math.sin(p)], rtol=0, atol=1e-15)
        y = O.rope(np.array([0.0, 1.0]), p)
        assert np.allclose(y, [-math.sin(p), math.cos(p)], rtol=0, atol=1e-15)


def test_rope_second_frequency():
    # d = 4, base 10000: pair 1 turns by p * 10000^(-2/4) = p / 100
    for p in [3, 50, 4095]:
        y = O.rope(np.array([0.0, 0.0, 1.0, 0.0]), p)
        assert np.allclose(y, [0, 0, math.cos(p / 100), math.sin(p / 100)], rtol=0, atol=1e-13)
        y = O.rope(np.array([1.0, 0.0, 0.0, 0.0]), p)
        assert np.allclose(y, [math.cos(p), math.sin(p), 0, 0], rtol=0, atol=1e-13)


def test_rope_preserves_pair_norms_and_depends_on_offset_only():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for m, n in [(5, 2), (4100, 4097), (131071, 131068)]:
        qm, kn = O.rope(q, m), O.rope(k, n)
        assert np.allclose(np.hypot(qm[0::2], qm[1::2]), np.hypot(q[0::2], q[1::2]), atol=1e-12)
        # q(m).k(n) depends only on m - n ([kasblo] "分離したRoPE": relative position)
        assert abs(qm @ kn - O.rope(q, m - n) @ k) < 1e-9


# --------------------------------------------------------------------------
# Softmax and lse
# --------------------------------------------------------------------------

def test_softmax_single_key():
    a, lse = O.softmax_lse(np.array([3.25]))
    assert a.tolist() == [1.0] and lse == 3.25


def test_softmax_equal_scores_is_mean():
    a, lse = O.softmax_lse(np.full(5, -2.0))
    assert np.allclose(a, 0.2, atol=1e-16)
    assert abs(lse - (-2.0 + math.log(5))) < 1e-15


def test_softmax_log_weights():
    a, lse = O.softmax_lse(np.log([1.0, 2.0, 3.0]))
    assert np.allclose(a, [1 / 6, 2 / 6, 3 / 6], atol=1e-15)
    assert abs(lse - math.log(6)) < 1e-15


def test_softmax_huge_gap_is_one_hot():
    a, lse = O.softmax_lse(np.array([0.0, 1000.0, -1000.0]))
    assert a.tolist() == [0.0, 1.0, 0.0] and lse == 1000.0


# --------------------------------------------------------------------------
# A two-head case computed by hand
# --------------------------------------------------------------------------

def _hand_case():
    """n_h=2, d_h=2, d_hr=2, d_c=3, T=3; scale = 1/sqrt(2+2) = 1/2.

    Head 0 keys read c[0], values read c[2]; head 1 keys read c[1], values
    read 2*c[2].  c[:,0] = 2 ln(1,2,3) and c[:,1] = 2 ln(4,1,1), so the weights
    are (1,2,3)/6 for head 0 and (4,1,1)/6 for head 1; both lse = ln 6.
    """
    c = np.array([[2 * math.log(1), 2 * math.log(4), 10.0],
                  [2 * math.log(2), 2 * math.log(1), 20.0],
                  [2 * math.log(3), 2 * math.log(1), 30.0]])
    W_uk = np.zeros((4, 3)); W_uk[0, 0] = 1; W_uk[3, 1] = 1
    W_uv = np.zeros((4, 3)); W_uv[0, 2] = 1; W_uv[3, 2] = 2
    q_c = np.array([[1.0, 0.0], [0.0, 1.0]])
    q_r = np.zeros((2, 2))
    k_r = np.array([[7.0, -1.0], [0.5, 2.0], [3.0, 3.0]])  # multiplied by q_r = 0
    o_expect = np.array([[140 / 6, 0.0], [0.0, 30.0]])
    return c, k_r, W_uk, W_uv, q_c, q_r, o_expect


def test_hand_case_expanded():
    c, k_r, W_uk, W_uv, q_c, q_r, o_expect = _hand_case()
    o, lse = O.attend_expanded(q_c, q_r, c, k_r, W_uk, W_uv)
    assert np.allclose(o, o_expect, atol=1e-12)
    assert np.allclose(lse, [math.log(6), math.log(6)], atol=1e-14)
    # u = W^O [o_1; o_2]: pick o_1[0] and o_2[1] from the head-major concatenation
    W_o = np.zeros((2, 4)); W_o[0, 0] = 1; W_o[1, 3] = 1
    assert np.allclose(O.output_projection(o, W_o), [140 / 6, 30.0], atol=1e-12)


def test_hand_case_absorbed():
    c, k_r, W_uk, W_uv, q_c, q_r, o_expect = _hand_case()
    q_lat = O.absorb_query(q_c, q_r, W_uk)
    assert np.allclose(q_lat, [[1, 0, 0, 0, 0], [0, 1, 0, 0, 0]])
    rows = np.concatenate([c, k_r], axis=1)
    o_lat, lse = O.attend_latent(q_lat, rows, d_c=3, d_h=2)
    assert np.allclose(O.up_project(o_lat, W_uv), o_expect, atol=1e-12)
    assert np.allclose(lse, [math.log(6)] * 2, atol=1e-14)


def test_hand_case_positional_part():
    # scores driven only by the RoPE part: q^C = 0, q^R_0 = (1, 0), k^R_j[0] = 2 ln w_j
    c, _, W_uk, W_uv, _, _, _ = _hand_case()
    q_c = np.zeros((2, 2))
    q_r = np.array([[1.0, 0.0], [0.0, 0.0]])
    k_r = np.array([[2 * math.log(1), 5.0], [2 * math.log(2), -5.0], [2 * math.log(3), 1.0]])
    o, lse = O.attend_expanded(q_c, q_r, c, k_r, W_uk, W_uv)
    assert np.allclose(o[0], [140 / 6, 0.0], atol=1e-12)
    # head 1 sees all-zero scores: plain mean of its values 2*c[:,2]
    assert np.allclose(o[1], [0.0, 40.0], atol=1e-12)
    assert np.allclose(lse, [math.log(6), math.log(3)], atol=1e-14)


# --------------------------------------------------------------------------
# Causality through the block table
# --------------------------------------------------------------------------

def test_decode_batch_causal_two_queries():
    rng = np.random.default_rng(3)
    d_c, d_hr, d_h, n_h, block = 3, 2, 2, 2, 4
    rows = rng.standard_normal((8, d_c + d_hr))
    table = [[1, 0]]  # logical block 0 -> physical 1, logical 1 -> physical 0
    q_lat = rng.standard_normal((2, n_h, d_c + d_hr))
    seq_lens, cu_q = [2], [0, 2]
    res = O.decode_batch(q_lat, rows, table, seq_lens, cu_q, block, d_c, d_h)
    # token 0 at position 0 sees exactly one row (physical row 4): o~ = c_0
    o0, lse0 = res[0]
    assert np.allclose(o0, np.broadcast_to(rows[4, :d_c], (n_h, d_c)), atol=1e-15)
    s0 = rows[4] @ q_lat[0].T / math.sqrt(d_h + d_hr)
    assert np.allclose(lse0, s0, atol=1e-15)
    # changing the second row does not touch token 0 but does touch token 1
    rows2 = rows.copy(); rows2[5] += 1.0
    res2 = O.decode_batch(q_lat, rows2, table, seq_lens, cu_q, block, d_c, d_h)
    assert np.array_equal(res2[0][0], o0)
    assert not np.allclose(res2[1][0], res[1][0])


# --------------------------------------------------------------------------
# Absorbed == expanded, and split merging
# --------------------------------------------------------------------------

def _random_layer(seed, n_h=4, d_h=8, d_hr=4, d_c=16, d_cq=24, d=32):
    rng = np.random.default_rng(seed)
    W = {
        "W_dkv": rng.standard_normal((d_c, d)) / math.sqrt(d),
        "W_kr": rng.standard_normal((d_hr, d)) / math.sqrt(d),
        "W_dq": rng.standard_normal((d_cq, d)) / math.sqrt(d),
        "W_uq": rng.standard_normal((n_h * d_h, d_cq)) / math.sqrt(d_cq),
        "W_qr": rng.standard_normal((n_h * d_hr, d_cq)) / math.sqrt(d_cq),
        "W_uk": rng.standard_normal((n_h * d_h, d_c)) / math.sqrt(d_c),
        "W_uv": rng.standard_normal((n_h * d_h, d_c)) / math.sqrt(d_c),
        "W_o": rng.standard_normal((d, n_h * d_h)) / math.sqrt(n_h * d_h),
    }
    return W, rng


def test_absorbed_equals_expanded():
    W, rng = _random_layer(5)
    T = 64
    h = rng.standard_normal((T, 32))
    r = O.decode_sequence(h, h[T - 1], T - 1, W, n_h=4)
    o_abs = O.up_project(r["o_lat"], W["W_uv"])
    assert np.max(np.abs(o_abs - r["o"])) <= 1e-12 * np.max(np.abs(r["o"]))
    assert np.max(np.abs(r["lse_lat"] - r["lse"])) <= 1e-12 * max(1.0, np.max(np.abs(r["lse"])))


def test_precomputed_query_equals_runtime_absorption():
    # Two routes to the latent query: q^C = W^UQ c^Q then W^UK_i^T q^C_i per
    # head, or the folded weight applied to c^Q.  Four heads with distinct
    # weights, so a wrong head slice or a swapped operand shows.
    W, rng = _random_layer(11)
    h = rng.standard_normal((3, 32))
    c_q, q_c, q_r_raw = O.query_parts(h, W["W_dq"], W["W_uq"], W["W_qr"], n_h=4)
    W_abs = O.absorbed_query_weight(W["W_uq"], W["W_uk"], n_h=4)
    assert W_abs.shape == (4 * 16, 24)
    for n in range(3):
        q_r = O.rope(q_r_raw[n], n + 5)
        ref = O.absorb_query(q_c[n], q_r, W["W_uk"])
        got = O.latent_query_precomputed(c_q[n], W_abs, q_r, n_h=4)
        assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_absorbed_query_weight_brute_force():
    # every entry as an explicit scalar sum over the head's d_h rows
    rng = np.random.default_rng(12)
    n_h, d_h, d_c, d_cq = 3, 2, 4, 5
    W_uq = rng.standard_normal((n_h * d_h, d_cq))
    W_uk = rng.standard_normal((n_h * d_h, d_c))
    got = O.absorbed_query_weight(W_uq, W_uk, n_h)
    for i in range(n_h):
        for c in range(d_c):
            for k in range(d_cq):
                s = 0.0
                for e in range(d_h):
                    s += W_uk[i * d_h + e][c] * W_uq[i * d_h + e][k]
                assert abs(got[i * d_c + c][k] - s) <= 1e-13


# --------------------------------------------------------------------------
# Quantised latent cache: block codes
# --------------------------------------------------------------------------

def test_q8_exact_block():
    # codes k with scale 2^-4: the largest |x| is 127 * 2^-4, so d = 2^-4
    # exactly and every value comes back unchanged
    k = np.array([-127, -100, -64, -33, -17, -8, -5, -3, -2, -1, 0, 0, 1, 2, 3, 4,
                  5, 6, 7, 9, 12, 15, 20, 31, 32, 47, 63, 64, 90, 111, 126, 127])
    x = k * 2.0 ** -4
    q, d = O.quantize_q8_blocks(x[None])
    assert q.dtype == np.int8 and d.dtype == np.float16
    assert q[0].tolist() == k.tolist() and d.tolist() == [[2.0 ** -4]]
    assert O.dequantize_q8_blocks(q, d)[0].tolist() == x.tolist()


def test_q8_zero_block_and_ties():
    x = np.zeros((1, 64))
    # second block: largest 127/16, then exact half-way values 2.5, 0.5 and -1.5
    # (in units of the scale 1/16): ties go away from zero (3, 1, -2), which
    # round-half-to-even would send to 2, 0 and -2
    x[0, 32] = 127 / 16
    x[0, 33], x[0, 34], x[0, 35] = 2.5 / 16, 0.5 / 16, -1.5 / 16
    q, d = O.quantize_q8_blocks(x)
    assert d.tolist() == [[0.0, 1 / 16]]
    assert q[0, :32].tolist() == [0] * 32
    assert q[0, 32:36].tolist() == [127, 3, 1, -2]
    assert O.dequantize_q8_blocks(q, d)[0, :32].tolist() == [0.0] * 32


def test_q8_error_bound_extremes_and_idempotence():
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((50, 512)) * rng.uniform(0.01, 30, (50, 1))).astype(np.float32)
    q, d = O.quantize_q8_blocks(x)
    dq = O.dequantize_q8_blocks(q, d)
    d64 = d.astype(np.float64).repeat(32, axis=1)
    # every value within half a step of its code
    assert np.all(np.abs(x - dq) <= d64 / 2 * (1 + 1e-6))
    # the largest magnitude of every block takes code +-127
    blocks = np.abs(x.reshape(50, 16, 32))
    top = np.take_along_axis(q.reshape(50, 16, 32), blocks.argmax(axis=2)[..., None], axis=2)
    assert np.all(np.abs(top.astype(int)) == 127)
    # quantising the dequantised values gives back the same codes and scales
    q2, d2 = O.quantize_q8_blocks(dq.astype(np.float32))
    assert np.array_equal(q2, q) and np.array_equal(d2, d)


def test_q8_cache_rows_keep_rope_and_exact_cache_attends_alike():
    rng = np.random.default_rng(22)
    d_c, d_hr, T = 64, 8, 20
    # latent values on the exact grid of each block's scale (each block holds a 127)
    codes = rng.integers(-127, 128, (T, d_c))
    codes[:, ::32] = 127
    rows = np.concatenate([codes * 2.0 ** -5, rng.standard_normal((T, d_hr))], axis=1)
    q, d, k_r = O.quantize_cache_rows(rows, d_c)
    assert np.array_equal(k_r, rows[:, d_c:])
    back = O.dequantize_cache_rows(q, d, k_r)
    assert np.array_equal(back, rows)
    q_lat = rng.standard_normal((4, d_c + d_hr))
    o1, l1 = O.attend_latent(q_lat, rows, d_c=d_c, d_h=16)
    o2, l2 = O.attend_latent(q_lat, back, d_c=d_c, d_h=16)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# --------------------------------------------------------------------------
# Prefill: every prompt position at once (expanded form)
# --------------------------------------------------------------------------

def test_prefill_first_token_sees_only_itself():
    W, rng = _random_layer(31)
    h = rng.standard_normal((6, 32))
    o, lse, _ = O.prefill_expanded(h, W, n_h=4)
    c, k_r = O.kv_latent(h[:1], W["W_dkv"], W["W_kr"], [0])
    _, q_c, q_r_raw = O.query_parts(h[:1], W["W_dq"], W["W_uq"], W["W_qr"], 4)
    for i in range(4):
        k_c, v = O.expand_kv(c, W["W_uk"], W["W_uv"], i, 8)
        # one visible key: the output is its value, the lse its score
        assert np.allclose(o[0, i], v[0], atol=1e-13)
        s = (q_c[0, i] @ k_c[0] + q_r_raw[0, i] @ k_r[0]) / math.sqrt(12)  # position 0: no rotation
        assert abs(lse[0, i] - s) < 1e-12


def test_prefill_is_causal():
    W, rng = _random_layer(32)
    h = rng.standard_normal((7, 32))
    o, lse, u = O.prefill_expanded(h, W, n_h=4)
    h2 = h.copy()
    h2[4] += 3.0  # a later token changes
    o2, lse2, u2 = O.prefill_expanded(h2, W, n_h=4)
    assert np.array_equal(o2[:4], o[:4]) and np.array_equal(lse2[:4], lse[:4]) and np.array_equal(u2[:4], u[:4])
    assert not np.allclose(o2[4:], o[4:])


def test_prefill_matches_per_token_decode_and_brute_force():
    W, rng = _random_layer(33)
    P = 9
    h = rng.standard_normal((P, 32))
    o, lse, u = O.prefill_expanded(h, W, n_h=4)
    for t in range(P):
        r = O.decode_sequence(h[:t + 1], h[t], t, W, n_h=4, with_latent=False)
        assert np.max(np.abs(o[t] - r["o"])) <= 1e-12 * np.max(np.abs(r["o"]))
        assert np.max(np.abs(lse[t] - r["lse"])) <= 1e-12 * max(1.0, np.max(np.abs(r["lse"])))
        assert np.max(np.abs(u[t] - r["u"])) <= 1e-12 * np.max(np.abs(r["u"]))
    # scalar loops on a tiny layer
    n_h, d_h, d_hr, d_c, d_cq, d = 2, 2, 2, 3, 3, 4
    Wt, rng = _random_layer(34, n_h, d_h, d_hr, d_c, d_cq, d)
    ht = rng.standard_normal((4, d))
    ot, _, ut = O.prefill_expanded(ht, Wt, n_h=n_h)
    for t in range(4):
        o_b, u_b = _brute_decode(ht.tolist(), t, {k: v.tolist() for k, v in Wt.items()}, n_h, d_h, d_hr)
        assert np.allclose(ot[t].reshape(-1), o_b, atol=1e-12) and np.allclose(ut[t], u_b, atol=1e-12)


def test_merge_partials_equals_whole():
    rng = np.random.default_rng(7)
    q_lat = rng.standard_normal((4, 20))
    rows = rng.standard_normal((50, 20)) * 3
    whole_o, whole_l = O.attend_latent(q_lat, rows, d_c=16, d_h=8)
    parts = [(0, 7), (7, 31), (31, 50)]
    po, pl = zip(*[O.attend_latent(q_lat, rows[a:b], d_c=16, d_h=8) for a, b in parts])
    o, l = O.merge_partials(np.stack(po), np.stack(pl))
    assert np.allclose(o, whole_o, atol=1e-13) and np.allclose(l, whole_l, atol=1e-13)


# --------------------------------------------------------------------------
# Brute force with scalar loops on tiny inputs
# --------------------------------------------------------------------------

def _brute_decode(h, t, W, n_h, d_h, d_hr, base=10000.0):
    """Every step as explicit scalar sums, straight from the equations."""
    d = len(h[0])
    d_c = len(W["W_dkv"])
    d_cq = len(W["W_dq"])

    def matvec(M, x):
        return [sum(M[r][k] * x[k] for k in range(len(x))) for r in range(len(M))]

    def rot(x, p):
        out = list(x)
        for k in range(len(x) // 2):
            ang = p * base ** (-2.0 * k / len(x))
            out[2 * k] = x[2 * k] * math.cos(ang) - x[2 * k + 1] * math.sin(ang)
            out[2 * k + 1] = x[2 * k] * math.sin(ang) + x[2 * k + 1] * math.cos(ang)
        return out

    cs = [matvec(W["W_dkv"], h[j]) for j in range(t + 1)]
    krs = [rot(matvec(W["W_kr"], h[j]), j) for j in range(t + 1)]
    cq = matvec(W["W_dq"], h[t])
    qc_all = matvec(W["W_uq"], cq)
    qr_all = matvec(W["W_qr"], cq)
    o_all = []
    for i in range(n_h):
        qc = qc_all[i * d_h:(i + 1) * d_h]
        qr = rot(qr_all[i * d_hr:(i + 1) * d_hr], t)
        s = []
        vs = []
        for j in range(t + 1):
            kc = [sum(W["W_uk"][i * d_h + r][k] * cs[j][k] for k in range(d_c)) for r in range(d_h)]
            v = [sum(W["W_uv"][i * d_h + r][k] * cs[j][k] for k in range(d_c)) for r in range(d_h)]
            dot = sum(qc[r] * kc[r] for r in range(d_h)) + sum(qr[r] * krs[j][r] for r in range(d_hr))
            s.append(dot / math.sqrt(d_h + d_hr))
            vs.append(v)
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = sum(e)
        o_all.extend(sum(e[j] / z * vs[j][r] for j in range(t + 1)) for r in range(d_h))
    u = matvec(W["W_o"], o_all)
    return o_all, u


def test_brute_force_tiny():
    n_h, d_h, d_hr, d_c, d_cq, d = 2, 2, 2, 3, 3, 4
    W, rng = _random_layer(11, n_h, d_h, d_hr, d_c, d_cq, d)
    T = 5
    h = rng.standard_normal((T, d))
    for t in range(T):
        r = O.decode_sequence(h[:t + 1], h[t], t, W, n_h=n_h)
        o_b, u_b = _brute_decode(h.tolist(), t, {k: v.tolist() for k, v in W.items()}, n_h, d_h, d_hr)
        assert np.allclose(r["o"].reshape(-1), o_b, atol=1e-12)
        assert np.allclose(r["u"], u_b, atol=1e-12)
