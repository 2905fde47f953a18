"""Planted mistakes in the oracle must fail its pins.

Each case swaps one oracle function for a plausibly wrong version (a sign, a
scale, a head index, a position offset, a rounding rule, a dropped max
shift, a wrong merge weight) and runs every pin of tests/test_oracle.py; at
least one pin has to fail.  The mistakes are planted in the oracle, on the
CPU; nothing here touches the CUDA library."""

import numpy as np
import pytest

import oracle
import oracle.mla as M
import test_oracle as T

PINS = [getattr(T, n) for n in sorted(dir(T)) if n.startswith("test_") and callable(getattr(T, n))]


def _failing_pins():
    bad = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except Exception:  # noqa: BLE001 (any failure of the pin counts)
            bad.append(pin.__name__)
    return bad


def _rope_wrong_sign(orig):
    return lambda x, pos, base=10000.0: orig(x, -np.asarray(pos, dtype=np.float64), base)


def _kv_latent_position_off_by_one(orig):
    return lambda h, W_dkv, W_kr, pos, base=10000.0: orig(h, W_dkv, W_kr, np.asarray(pos) + 1, base)


def _attend_latent_wrong_scale(orig):
    # 1/sqrt(d_c + d_hr), the width of the absorbed dot product, instead of 1/sqrt(d_h + d_hr)
    return lambda q_lat, rows, d_c, d_h, heads=None: orig(q_lat, rows, d_c, d_c, heads)


def _absorb_query_head_zero(orig):
    def bad(q_c, q_r, W_uk):
        q_c = M.f64(q_c)
        n_h, d_h = q_c.shape
        return orig(q_c, q_r, np.tile(M.f64(W_uk)[:d_h], (n_h, 1)))
    return bad


def _up_project_head_zero(orig):
    def bad(o_lat, W_uv):
        o_lat = M.f64(o_lat)
        d_h = M.f64(W_uv).shape[0] // o_lat.shape[0]
        return orig(o_lat, np.tile(M.f64(W_uv)[:d_h], (o_lat.shape[0], 1)))
    return bad


def _softmax_without_max_shift(orig):
    def bad(s):
        e = np.exp(M.f64(s))
        z = e.sum(axis=-1, keepdims=True)
        return e / z, np.log(z[..., 0])
    return bad


def _merge_equal_weights(orig):
    def bad(o_parts, lse_parts):
        _, L = orig(o_parts, lse_parts)
        return np.mean(M.f64(o_parts), axis=0), L
    return bad


def _q8_round_half_even(orig):
    def bad(x, block=M.Q8_BLOCK):
        q, d = orig(x, block)
        x32 = np.asarray(x, dtype=np.float32)
        blocks = x32.reshape(x32.shape[:-1] + (x32.shape[-1] // block, block))
        d32 = d.astype(np.float32)[..., None]
        v = np.where(d32 > 0, blocks / np.where(d32 > 0, d32, np.float32(1)), np.float32(0))
        return np.clip(np.rint(v), -127, 127).astype(np.int8).reshape(x32.shape), d
    return bad


def _folded_weight_head_shift(orig):
    # head i folded with head i-1's W^UQ rows
    def bad(W_uq, W_uk, n_h):
        W_uq = M.f64(W_uq)
        return orig(np.roll(W_uq, W_uq.shape[0] // n_h, axis=0), W_uk, n_h)
    return bad


def _prefill_parts_mask_includes_next_key(orig):
    # the same planted mask error, in the attention from the prompt's parts
    def bad(c, k_r, q_c, q_r_raw, W_uk, W_uv, base=10000.0):
        c, k_r, q_c = M.f64(c), M.f64(k_r), M.f64(q_c)
        P, n_h = q_c.shape[0], q_c.shape[1]
        q_r = M.rope(M.f64(q_r_raw), np.arange(P)[:, None], base)
        d_h, d_hr = q_c.shape[2], q_r.shape[2]
        later = np.triu(np.ones((P, P), dtype=bool), 2)
        o, lse = np.empty((P, n_h, d_h)), np.empty((P, n_h))
        for i in range(n_h):
            k_c, v = M.expand_kv(c, W_uk, W_uv, i, d_h)
            s = (q_c[:, i] @ k_c.T + q_r[:, i] @ k_r.T) / np.sqrt(d_h + d_hr)
            s[later] = -np.inf
            a, lse[:, i] = M.softmax_lse(s)
            o[:, i] = a @ v
        return o, lse
    return bad


def _prefill_mask_includes_next_key(orig):
    # the causal mask lets row t see row t+1
    def bad(h, W, n_h, base=10000.0):
        h = M.f64(h)
        P = h.shape[0]
        pos = np.arange(P)
        c, k_r = M.kv_latent(h, W["W_dkv"], W["W_kr"], pos, base)
        _, q_c, q_r_raw = M.query_parts(h, W["W_dq"], W["W_uq"], W["W_qr"], n_h)
        q_r = M.rope(q_r_raw, pos[:, None], base)
        d_h, d_hr = q_c.shape[2], q_r.shape[2]
        later = np.triu(np.ones((P, P), dtype=bool), 2)
        o, lse = np.empty((P, n_h, d_h)), np.empty((P, n_h))
        for i in range(n_h):
            k_c, v = M.expand_kv(c, W["W_uk"], W["W_uv"], i, d_h)
            s = (q_c[:, i] @ k_c.T + q_r[:, i] @ k_r.T) / np.sqrt(d_h + d_hr)
            s[later] = -np.inf
            a, lse[:, i] = M.softmax_lse(s)
            o[:, i] = a @ v
        return o, lse, np.stack([M.output_projection(o[t], W["W_o"]) for t in range(P)])
    return bad


MUTATIONS = [
    ("rope", _rope_wrong_sign),
    ("kv_latent", _kv_latent_position_off_by_one),
    ("attend_latent", _attend_latent_wrong_scale),
    ("absorb_query", _absorb_query_head_zero),
    ("up_project", _up_project_head_zero),
    ("softmax_lse", _softmax_without_max_shift),
    ("merge_partials", _merge_equal_weights),
    ("quantize_q8_blocks", _q8_round_half_even),
    ("absorbed_query_weight", _folded_weight_head_shift),
    ("prefill_expanded", _prefill_mask_includes_next_key),
    ("prefill_from_parts", _prefill_parts_mask_includes_next_key),
]


def test_pins_pass_on_the_oracle_as_it_stands():
    assert _failing_pins() == []


@pytest.mark.parametrize("name,make", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, make):
    bad = make(getattr(M, name))
    monkeypatch.setattr(M, name, bad)
    monkeypatch.setattr(oracle, name, bad)
    assert _failing_pins(), f"no pin catches the planted mistake in {name}"
