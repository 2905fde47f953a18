"""Plain, slow, fp64 CPU oracle for MLA decode (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may use this module.  It shares no code with the CUDA
library: numpy in float64, one library matmul per step, no blocking, fusion or
reordering beyond what the equations state.

Sources (cited by page and section heading):

* [0h-n0]  "論文解説: DeepSeek-V2 — MoEモデルのKVキャッシュを93.3%削減する
  Multi-head Latent Attention" (0h-n0.github.io/posts/paper-2401-06066)
* [kasblo] MLA explainer at kasblo.com/?p=4663
* [qiita]  MLA notes at qiita.com/joule/items/57d9b3f4fc27959eaa0d

The method reaches the plain multi-head attention result exactly (the
absorption is an identity of matrix products, [0h-n0] "行列吸収トリック",
[qiita] "Absorption Trick"), so the primary oracle is the un-absorbed
definition: K and V are expanded per head and per cached token.  The absorbed
intermediates (latent query, latent output) are also written out, each from
its own defining equation, for per-kernel parity.

Readings taken where the pages are silent:

* RoPE: interleaved pairs (x[2k], x[2k+1]) rotated by angle pos * theta_k,
  theta_k = base ** (-2k / d_r); positions are 0-based.  The pages only say
  that pairs of numbers are rotated by position ([kasblo] "分離したRoPE").
* Score scale 1/sqrt(d_h + d_h^R) ([qiita] "Attention 計算").
* Causal, inclusive: a query at position t sees rows j <= t ([qiita]
  "Attention 計算", the sum over j = 1..t).
* No normalisation layers and no biases ([kasblo] "MLAはKとVを共通の潜在表現
  から作る" omits normalisation; [0h-n0] sketch uses bias=False).
* Head i of W^UK, W^UV, W^UQ owns rows [i*d_h, (i+1)*d_h); W^QR is head-major
  [n_h, d_h^R]; W^O consumes the head-major concatenation.

Parity status: every function below is pinned by a test under
``tests/test_oracle.py`` (worked example, closed forms, special cases with
hand-computed answers, invariants, brute force on tiny inputs).
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "f64",
    "rope",
    "kv_latent",
    "query_parts",
    "expand_kv",
    "scores_expanded",
    "softmax_lse",
    "attend_expanded",
    "output_projection",
    "absorb_query",
    "absorbed_query_weight",
    "latent_query_precomputed",
    "Q8_BLOCK",
    "quantize_q8_blocks",
    "dequantize_q8_blocks",
    "quantize_cache_rows",
    "dequantize_cache_rows",
    "scores_latent",
    "attend_latent",
    "up_project",
    "merge_partials",
    "cache_slot",
    "latent_cache_bytes",
    "mha_cache_elements",
    "mla_cache_elements",
    "decode_sequence",
    "decode_batch",
    "prefill_expanded",
    "prefill_from_parts",
]


def f64(x) -> np.ndarray:
    """Widen any array-like (numpy, or a CPU torch tensor) to float64 exactly."""
    if hasattr(x, "detach"):  # torch tensor: bf16 -> fp32 -> fp64 is exact
        x = x.detach().to("cpu").float().numpy()
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------
# Positional part: decoupled RoPE
# --------------------------------------------------------------------------

def rope(x, pos, base: float = 10000.0) -> np.ndarray:
    """Rotate consecutive pairs of the last axis of ``x`` by position.

    [kasblo] "位置情報は別の経路で持つ：分離したRoPE": pairs of numbers are
    rotated according to the position so that the dot product reflects the
    relative position.  [qiita] "RoPE の扱い": q^R = RoPE(W^QR c^Q),
    k^R = RoPE(W^KR h).  Reading: pair k = (x[2k], x[2k+1]) turns by the angle
    pos * base**(-2k/d_r), computed in float64.
    """
    x = f64(x)
    d = x.shape[-1]
    if d % 2:
        raise ValueError("RoPE needs an even width")
    k = np.arange(d // 2, dtype=np.float64)
    theta = base ** (-2.0 * k / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty(np.broadcast_shapes(x.shape, ang.shape[:-1] + (d,)), dtype=np.float64)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


# --------------------------------------------------------------------------
# What the cache holds: c^KV and k^R
# --------------------------------------------------------------------------

def kv_latent(h, W_dkv, W_kr, pos, base: float = 10000.0):
    """Per-token cache contents (c^KV_t, k^R_t).

    [0h-n0] "MLA: 低ランクKV結合圧縮": c^KV_t = W^DKV h_t with
    W^DKV in R^{d_c x d}.  [qiita] "RoPE の扱い": k^R_t = RoPE(W^KR h_t),
    shared by every head.  [0h-n0] "Decoupled RoPE": the cache stores c^KV
    (d_c) and k^R (d_h^R), 576 elements per token per layer at V2 sizes.

    h: [T, d]; W_dkv: [d_c, d]; W_kr: [d_hr, d]; pos: [T].
    Returns c [T, d_c] and k_r [T, d_hr] (k_r already rotated).
    """
    h = f64(h)
    c = h @ f64(W_dkv).T
    k_r = rope(h @ f64(W_kr).T, pos, base)
    return c, k_r


# --------------------------------------------------------------------------
# Query side
# --------------------------------------------------------------------------

def query_parts(h, W_dq, W_uq, W_qr, n_h: int):
    """Query compression and the raw (un-rotated) positional query.

    [qiita] "Query の圧縮": c^Q_t = W^DQ h_t, q^C_t = W^UQ c^Q_t.
    [qiita] "RoPE の扱い": q^R_{t,i} = RoPE(W^QR c^Q_t); this function returns
    W^QR c^Q_t before the rotation.

    h: [N, d]; W_dq: [d_cq, d]; W_uq: [n_h*d_h, d_cq]; W_qr: [n_h*d_hr, d_cq].
    Returns c_q [N, d_cq], q_c [N, n_h, d_h], q_r_raw [N, n_h, d_hr].
    """
    h = f64(h)
    c_q = h @ f64(W_dq).T
    q_c = (c_q @ f64(W_uq).T).reshape(h.shape[0], n_h, -1)
    q_r_raw = (c_q @ f64(W_qr).T).reshape(h.shape[0], n_h, -1)
    return c_q, q_c, q_r_raw


# --------------------------------------------------------------------------
# Expanded (un-absorbed) attention: the definition
# --------------------------------------------------------------------------

def _head_rows(W, i: int, d_h: int) -> np.ndarray:
    return W[i * d_h:(i + 1) * d_h]


def expand_kv(c, W_uk, W_uv, i: int, d_h: int):
    """Per-head key and value content of every cached token.

    [0h-n0] "MLA: 低ランクKV結合圧縮" / [qiita] "復元": k^C_t = W^UK c^KV_t,
    v^C_t = W^UV c^KV_t with W^UK, W^UV in R^{n_h d_h x d_c}; head i takes
    rows [i*d_h, (i+1)*d_h).  Returns k_c [T, d_h], v [T, d_h].
    """
    c = f64(c)
    k_c = c @ _head_rows(f64(W_uk), i, d_h).T
    v = c @ _head_rows(f64(W_uv), i, d_h).T
    return k_c, v


def scores_expanded(q_c_i, q_r_i, k_c, k_r) -> np.ndarray:
    """Unscaled scores q_{t,i}^T k_{j,i} with the concatenated vectors.

    [qiita] "最終的な Key と Query の結合": q_{t,i} = [q^C_{t,i}; q^R_{t,i}],
    k_{j,i} = [k^C_{j,i}; k^R_j].  Returns [T].
    """
    q = np.concatenate([f64(q_c_i), f64(q_r_i)])
    k = np.concatenate([f64(k_c), f64(k_r).reshape(len(k_c), -1)], axis=1)
    return k @ q


def softmax_lse(s):
    """Softmax over the last axis and its log-sum-exp (natural log).

    The max-shift only guards the exponent range: a = exp(s - m) / sum,
    lse = m + ln(sum exp(s - m)).
    """
    s = f64(s)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    z = np.sum(e, axis=-1, keepdims=True)
    return e / z, (m + np.log(z))[..., 0]


def attend_expanded(q_c, q_r, c, k_r, W_uk, W_uv, heads=None):
    """o_{t,i} for one query token over the cached rows it may see.

    [qiita] "Attention 計算":
        o_{t,i} = sum_j softmax_j( q_{t,i}^T k_{j,i} / sqrt(d_h + d_h^R) ) v^C_{j,i}
    Keys and values are expanded per head (the un-absorbed form).

    q_c: [n_h, d_h]; q_r: [n_h, d_hr] (rotated); c: [T, d_c] and k_r: [T, d_hr]
    are the rows j = 0..T-1 this query sees.  ``heads`` restricts the work to
    a subset of heads (rows of the result follow that order).
    Returns o [len(heads), d_h] and lse [len(heads)].
    """
    q_c, q_r = f64(q_c), f64(q_r)
    n_h, d_h = q_c.shape
    d_hr = q_r.shape[1]
    heads = range(n_h) if heads is None else heads
    inv = 1.0 / math.sqrt(d_h + d_hr)
    o, lse = [], []
    for i in heads:
        k_c, v = expand_kv(c, W_uk, W_uv, i, d_h)
        s = scores_expanded(q_c[i], q_r[i], k_c, k_r) * inv
        a, l = softmax_lse(s)
        o.append(a @ v)
        lse.append(l)
    return np.array(o), np.array(lse)


def output_projection(o, W_o) -> np.ndarray:
    """u_t = W^O [o_{t,1}; ...; o_{t,n_h}]  ([qiita] "Attention 計算").

    o: [n_h, d_h] (head-major concatenation); W_o: [d, n_h*d_h].
    """
    return f64(W_o) @ f64(o).reshape(-1)


# --------------------------------------------------------------------------
# Absorbed intermediates (each from its own defining equation)
# --------------------------------------------------------------------------

def absorb_query(q_c, q_r, W_uk) -> np.ndarray:
    """Latent query [W^UK_i^T q^C_i ; q^R_i] for every head.

    [0h-n0] "行列吸収トリック": (q^C)^T (W^UK_i c) = (W^UK_i^T q^C)^T c, so the
    content query moves into the d_c-dimensional latent space.
    q_c: [n_h, d_h]; q_r: [n_h, d_hr] (rotated); W_uk: [n_h*d_h, d_c].
    Returns [n_h, d_c + d_hr].
    """
    q_c, q_r, W_uk = f64(q_c), f64(q_r), f64(W_uk)
    n_h, d_h = q_c.shape
    qt = np.stack([_head_rows(W_uk, i, d_h).T @ q_c[i] for i in range(n_h)])
    return np.concatenate([qt, q_r], axis=1)


def absorbed_query_weight(W_uq, W_uk, n_h: int) -> np.ndarray:
    """The query weight with W^UK folded in: W~^UQ_i = W^UK_i^T W^UQ_i.

    [0h-n0] "行列吸収トリック": the product W^UK_i^T W^UQ_i can be formed once,
    ahead of inference, after which the latent content query is a single
    product of c^Q.  W_uq: [n_h*d_h, d_cq]; W_uk: [n_h*d_h, d_c].
    Returns [n_h*d_c, d_cq]; rows [i*d_c, (i+1)*d_c) belong to head i.
    """
    W_uq, W_uk = f64(W_uq), f64(W_uk)
    d_h = W_uq.shape[0] // n_h
    return np.concatenate([_head_rows(W_uk, i, d_h).T @ _head_rows(W_uq, i, d_h) for i in range(n_h)])


def latent_query_precomputed(c_q, W_uq_abs, q_r, n_h: int) -> np.ndarray:
    """Latent query [W~^UQ_i c^Q ; q^R_i] for every head, straight from c^Q.

    [0h-n0] "行列吸収トリック" with the folded weight of absorbed_query_weight.
    c_q: [d_cq]; W_uq_abs: [n_h*d_c, d_cq]; q_r: [n_h, d_hr] (rotated).
    Returns [n_h, d_c + d_hr].
    """
    qt = (f64(W_uq_abs) @ f64(c_q)).reshape(n_h, -1)
    return np.concatenate([qt, f64(q_r)], axis=1)


def scores_latent(q_lat_i, rows) -> np.ndarray:
    """Unscaled score q~_i . c_j + q^R_i . k^R_j against stored rows [c_j; k^R_j].

    [kasblo] "分離したRoPE": the score is the sum of the content match and the
    positional match.  rows: [T, d_c + d_hr]; returns [T].
    """
    return f64(rows) @ f64(q_lat_i)


def attend_latent(q_lat, rows, d_c: int, d_h: int, heads=None):
    """Latent output o~_i = sum_j a_ij c_j and lse_i, straight from the cache.

    [kasblo] "V側は、小さな表現の加重和を先に求める": sum_j a_j W^UV c_j equals
    W^UV sum_j a_j c_j, weights differing per head.  The scale stays
    1/sqrt(d_h + d_h^R) ([qiita] "Attention 計算").

    q_lat: [n_h, d_c + d_hr]; rows: [T, d_c + d_hr] (rows this query sees).
    Returns o_lat [len(heads), d_c] and lse [len(heads)].
    """
    q_lat, rows = f64(q_lat), f64(rows)
    n_h, width = q_lat.shape
    d_hr = width - d_c
    heads = range(n_h) if heads is None else heads
    inv = 1.0 / math.sqrt(d_h + d_hr)
    o, lse = [], []
    for i in heads:
        a, l = softmax_lse(scores_latent(q_lat[i], rows) * inv)
        o.append(a @ rows[:, :d_c])
        lse.append(l)
    return np.array(o), np.array(lse)


# --------------------------------------------------------------------------
# Quantised latent cache (int8 codes in blocks with one fp16 scale)
# --------------------------------------------------------------------------

Q8_BLOCK = 32


def quantize_q8_blocks(x, block: int = Q8_BLOCK):
    """int8 block codes of cached latent values.

    [0h-n0] "量子化との組み合わせ": the compressed c^KV can be stored further
    with KV-cache quantisation of the Q8_0 kind (llama.cpp's q8_0 cache type).
    The page names the format only; the reading taken is that format's
    definition: each run of `block` consecutive values shares one scale
    d = max|x| / 127 kept in fp16, and each value becomes the int8 code
    round(x / d), nearest with ties away from zero; an all-zero block has
    d = 0 and codes 0.  The scale and the codes are decided in fp32 (x and the
    fp16 scale widened to fp32, one correctly rounded fp32 division), the
    precision a GPU kernel would use, so both sides reach the same integers.

    x: [..., n] with n a multiple of `block`, values exact in fp32 and below
    127 * 65504 in magnitude.  Returns codes int8 [..., n] and scales float16
    [..., n / block].
    """
    x32 = np.asarray(x, dtype=np.float32)
    shp = x32.shape
    blocks = x32.reshape(shp[:-1] + (shp[-1] // block, block))
    amax = np.max(np.abs(blocks), axis=-1)
    d16 = (amax / np.float32(127.0)).astype(np.float16)
    d32 = d16.astype(np.float32)[..., None]
    safe = np.where(d32 > 0, d32, np.float32(1.0))
    v = np.where(d32 > 0, blocks / safe, np.float32(0.0)).astype(np.float32)
    q = np.sign(v) * np.floor(np.abs(v) + np.float32(0.5))
    return np.clip(q, -127, 127).astype(np.int8).reshape(shp), d16


def dequantize_q8_blocks(q, d, block: int = Q8_BLOCK) -> np.ndarray:
    """The values a quantised block stands for: code x scale (exact in float64)."""
    q64 = np.asarray(q, dtype=np.float64)
    shp = q64.shape
    d64 = np.asarray(d, dtype=np.float64)[..., None]
    return (q64.reshape(shp[:-1] + (shp[-1] // block, block)) * d64).reshape(shp)


def quantize_cache_rows(rows, d_c: int, block: int = Q8_BLOCK):
    """A cache of rows [c^KV ; k^R] with c^KV quantised and k^R kept as is.

    The positional key is shared by all heads and carries the rotation, so
    only the d_c latent values are quantised.  rows: [T, d_c + d_hr].
    Returns (codes int8 [T, d_c], scales float16 [T, d_c / block], k_r [T, d_hr]).
    """
    rows = np.asarray(rows)
    q, d = quantize_q8_blocks(rows[:, :d_c], block)
    return q, d, rows[:, d_c:]


def dequantize_cache_rows(q, d, k_r, block: int = Q8_BLOCK) -> np.ndarray:
    """Rows [dequantised c^KV ; k^R] in float64, the input attend_latent takes."""
    return np.concatenate([dequantize_q8_blocks(q, d, block), f64(k_r)], axis=1)


def up_project(o_lat, W_uv) -> np.ndarray:
    """o_{t,i} = W^UV_i o~_{t,i}: the value up-projection after the weighted sum.

    [kasblo] "V側は、小さな表現の加重和を先に求める"; [0h-n0] "行列吸収トリック"
    (W^UV folded towards the output).  o_lat: [n_h, d_c]; W_uv: [n_h*d_h, d_c].
    """
    o_lat, W_uv = f64(o_lat), f64(W_uv)
    n_h = o_lat.shape[0]
    d_h = W_uv.shape[0] // n_h
    return np.stack([_head_rows(W_uv, i, d_h) @ o_lat[i] for i in range(n_h)])


def merge_partials(o_parts, lse_parts):
    """Combine attention over disjoint key ranges into attention over their union.

    Not on the pages: the standard identity for splitting a softmax sum.
    With L = ln sum_s exp(lse_s): o = sum_s exp(lse_s - L) o_s.
    o_parts: [S, ..., d]; lse_parts: [S, ...].
    """
    o_parts, lse_parts = f64(o_parts), f64(lse_parts)
    m = np.max(lse_parts, axis=0)
    w = np.exp(lse_parts - m)
    z = np.sum(w, axis=0)
    L = m + np.log(z)
    o = np.sum((w / z)[..., None] * o_parts, axis=0)
    return o, L


# --------------------------------------------------------------------------
# Cache bookkeeping
# --------------------------------------------------------------------------

def cache_slot(block_table, b: int, pos: int, block: int) -> int:
    """Physical row of token ``pos`` of sequence ``b`` in a block-tabled pool.

    Not on the pages (the paged layout is a serving choice): logical block
    pos // block of sequence b lives in physical block block_table[b][pos // block],
    at row pos % block inside it.
    """
    return int(block_table[b][pos // block]) * block + pos % block


def latent_cache_bytes(B: int, T: int, L: int, d_c: int, d_r: int, s: int) -> int:
    """B * T * L * (d_c + d_r) * s bytes ([kasblo] "容量を計算する")."""
    return B * T * L * (d_c + d_r) * s


def mha_cache_elements(n_h: int, d_h: int) -> int:
    """2 n_h d_h elements per token per layer for plain MHA ([0h-n0] "背景と動機")."""
    return 2 * n_h * d_h


def mla_cache_elements(d_c: int, d_hr: int) -> int:
    """d_c + d_h^R elements per token per layer for MLA ([0h-n0] "Decoupled RoPE")."""
    return d_c + d_hr


# --------------------------------------------------------------------------
# Whole decode step
# --------------------------------------------------------------------------

def decode_sequence(h_rows, h_query, t: int, W: dict, n_h: int, base: float = 10000.0,
                    heads=None, with_latent: bool = True) -> dict:
    """One query token at position t of one sequence, end to end, in float64.

    h_rows: [t+1, d] hidden states of rows 0..t (the query's own row last);
    h_query: [d] the query token's hidden state (equal to h_rows[t] for a
    normal decode step).  W holds W_dkv, W_kr, W_dq, W_uq, W_qr, W_uk, W_uv, W_o.

    Expanded path ([qiita] "Attention 計算"): rows -> (c, k^R); query ->
    (q^C, q^R); K/V expanded per head; softmax over j <= t; u = W^O [o].
    The absorbed intermediates (q_lat, o_lat) are added when with_latent.
    """
    c, k_r = kv_latent(h_rows, W["W_dkv"], W["W_kr"], np.arange(t + 1), base)
    _, q_c, q_r_raw = query_parts(f64(h_query)[None], W["W_dq"], W["W_uq"], W["W_qr"], n_h)
    q_c, q_r = q_c[0], rope(q_r_raw[0], t, base)
    o, lse = attend_expanded(q_c, q_r, c, k_r, W["W_uk"], W["W_uv"], heads=heads)
    res = {"c": c, "k_r": k_r, "q_c": q_c, "q_r_raw": q_r_raw[0], "q_r": q_r, "o": o, "lse": lse}
    if heads is None:
        res["u"] = output_projection(o, W["W_o"])
    if with_latent:
        q_lat = absorb_query(q_c, q_r, W["W_uk"])
        rows = np.concatenate([c, k_r], axis=1)
        o_lat, lse_lat = attend_latent(q_lat, rows, c.shape[1], q_c.shape[1], heads=heads)
        res.update(q_lat=q_lat, rows=rows, o_lat=o_lat, lse_lat=lse_lat)
    return res


def prefill_expanded(h, W: dict, n_h: int, base: float = 10000.0, with_u: bool = True):
    """Causal attention for every token of a prompt at once, in the expanded form.

    [perforder] "極限最適化の代償：MLA特有の学習負荷と独自Tritonカーネルという障壁":
    in the prefill phase many tokens are processed together and the
    up-projection of the latent vector to full keys and values becomes a large
    matrix product; [kasblo] "「キャッシュを減らせた」と「その割合だけ速い」は別の評価"
    names the reference implementation's "naive" branch that keeps the
    expanded K/V.  The cache rows and query parts of the prompt come from h
    (positions 0..P-1); the attention itself is prefill_from_parts.

    h: [P, d].  Returns o [P, n_h, d_h], lse [P, n_h] and u [P, d] (None when
    with_u is False: the output projection is then skipped, the rest is the
    same arithmetic).
    """
    h = f64(h)
    P = h.shape[0]
    pos = np.arange(P)
    c, k_r = kv_latent(h, W["W_dkv"], W["W_kr"], pos, base)
    _, q_c, q_r_raw = query_parts(h, W["W_dq"], W["W_uq"], W["W_qr"], n_h)
    o, lse = prefill_from_parts(c, k_r, q_c, q_r_raw, W["W_uk"], W["W_uv"], base)
    u = np.stack([output_projection(o[t], W["W_o"]) for t in range(P)]) if with_u else None
    return o, lse, u


def prefill_from_parts(c, k_r, q_c, q_r_raw, W_uk, W_uv, base: float = 10000.0):
    """The prompt's causal attention from its cache rows and query parts.

    c [P, d_c] and k_r [P, d_hR] (already rotated) are the prompt's cache rows
    in position order, q_c [P, n_h, d_h] and q_r_raw [P, n_h, d_hR] (before
    rotation) its query parts.  Row t of the prompt attends rows 0..t
    ([qiita] "Attention 計算").  All P queries of a head at once: K/V expanded
    per head, S = (Q^C K^C^T + Q^R K^R^T) / sqrt(d_h + d_h^R) over the P x P
    positions, entries with j > t set to -inf, a row-wise softmax with its
    log-sum-exp, O = A V.  Returns o [P, n_h, d_h] and lse [P, n_h].
    """
    c, k_r, q_c = f64(c), f64(k_r), f64(q_c)
    P, n_h = q_c.shape[0], q_c.shape[1]
    pos = np.arange(P)
    q_r = rope(f64(q_r_raw), pos[:, None], base)
    d_h, d_hr = q_c.shape[2], q_r.shape[2]
    inv = 1.0 / math.sqrt(d_h + d_hr)
    later = np.triu(np.ones((P, P), dtype=bool), 1)  # key j after query t
    o = np.empty((P, n_h, d_h))
    lse = np.empty((P, n_h))
    for i in range(n_h):
        k_c, v = expand_kv(c, W_uk, W_uv, i, d_h)
        s = (q_c[:, i] @ k_c.T + q_r[:, i] @ k_r.T) * inv
        s[later] = -np.inf
        a, lse[:, i] = softmax_lse(s)
        o[:, i] = a @ v
    return o, lse


def decode_batch(q_lat, pool_rows, block_table, seq_lens, cu_q, block: int, d_c: int, d_h: int,
                 tokens=None, heads=None):
    """Latent attention for a ragged batch read through a block table.

    Query tokens of sequence b are rows cu_q[b]..cu_q[b+1]-1 of q_lat and sit
    at positions seq_lens[b]-q_len_b .. seq_lens[b]-1; each sees the rows at
    positions j <= its own ([qiita] "Attention 計算", sum over j <= t).
    pool_rows: [n_blocks*block, d_c + d_hr].  Returns {token: (o_lat, lse)}.
    """
    q_lat = f64(q_lat)
    pool_rows = f64(pool_rows) if not isinstance(pool_rows, np.ndarray) else pool_rows
    out = {}
    B = len(seq_lens)
    for b in range(B):
        q0, q1 = int(cu_q[b]), int(cu_q[b + 1])
        L = int(seq_lens[b])
        for n in range(q0, q1):
            if tokens is not None and n not in tokens:
                continue
            t = L - (q1 - n)
            idx = [cache_slot(block_table, b, j, block) for j in range(t + 1)]
            out[n] = attend_latent(q_lat[n], pool_rows[idx], d_c, d_h, heads=heads)
    return out
