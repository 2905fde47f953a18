"""GPU parity of the quantised latent cache ([0h-n0] "量子化との組み合わせ"):
mla_cache_append_q8 and mla_decode_q8 through the C-ABI against the oracle.

The codes and scales of a row are a function of the bf16 row the plain
append stores, so they are compared bit for bit with the oracle's
quantisation of that row; attention over a quantised pool is compared with
the oracle's attention over the dequantised rows, at the tolerances of the
bf16 cache.
"""

import numpy as np
import pytest
import torch

import oracle as O
from head_latent_attention_26_b300 import build, synth
from _util import (LSE_TOL, OUT_TOL, batch_meta, latent_inputs, lse_err, record, row_rel_err, to_np)

pytestmark = pytest.mark.gpu

V2 = synth.V2
ROW_BYTES = 672


@pytest.fixture(scope="module")
def v2():
    build.build()
    from head_latent_attention_26_b300 import mla
    m = mla.MLA(V2, 131072 + 64, torch.bfloat16)
    assert m.tensor_path
    return m


def _w_dkr(W):
    return torch.cat([W["W_dkv"], W["W_kr"]], dim=0).contiguous()


def q8_bytes(rows_bf16: torch.Tensor) -> np.ndarray:
    """[T, 672] bytes of quantised rows, by the oracle's quantisation of the
    given bf16 rows [T, 576] (codes, fp16 scales, the bf16 k^R bits)."""
    r = rows_bf16.detach().cpu()
    codes, scales, _ = O.quantize_cache_rows(r.float().numpy(), V2.d_c)
    out = np.empty((r.shape[0], ROW_BYTES), dtype=np.uint8)
    out[:, :512] = codes.view(np.uint8)
    out[:, 512:544] = scales.astype("<f2").view(np.uint8)
    out[:, 544:] = r[:, V2.d_c:].contiguous().view(torch.int16).numpy().view(np.uint8)
    return out


def q8_pool(rows_per_seq, table, n_blocks, fill=0):
    """A quantised pool holding each sequence's rows at its block-table slots."""
    pool = np.full((n_blocks * V2.block, ROW_BYTES), fill, dtype=np.uint8)
    tab = table.cpu()
    for b, rows in enumerate(rows_per_seq):
        T = rows.shape[0]
        if T == 0:
            continue
        slots = np.array([O.cache_slot(tab, b, j, V2.block) for j in range(T)])
        pool[slots] = q8_bytes(rows)
    return torch.from_numpy(pool).view(n_blocks, V2.block, ROW_BYTES).cuda()


def dequantised(rows_bf16: torch.Tensor) -> np.ndarray:
    codes, scales, k_r = O.quantize_cache_rows(rows_bf16.detach().cpu().float().numpy(), V2.d_c)
    return O.dequantize_cache_rows(codes, scales, k_r)


def test_q8_append_codes_and_scales_bit_exact(v2):
    """The quantised rows of new tokens match the oracle's quantisation of the
    plain append's bf16 rows byte for byte; every other pool row keeps its
    sentinel."""
    d = V2
    seq_lens = [130, 64, 7]
    new = [50, 64, 7]
    table, n_blocks, _, _, _ = batch_meta(seq_lens, [1, 1, 1], d.block, 1101, spare_blocks=3)
    W = synth.weights(d, 1101, device="cuda")
    x = synth.hidden(sum(new), d, 1101, device="cuda")
    seq_idx = torch.tensor(sum([[b] * n for b, n in enumerate(new)], []), dtype=torch.int32, device="cuda")
    pos = torch.tensor(sum([list(range(L - n, L)) for L, n in zip(seq_lens, new)], []), dtype=torch.int32,
                       device="cuda")
    pool_bf = torch.zeros(n_blocks, d.block, d.width, dtype=torch.bfloat16, device="cuda")
    v2.cache_append(x, _w_dkr(W), seq_idx, pos, table, pool_bf)
    pool_q = torch.full((n_blocks, d.block, ROW_BYTES), 0xA5, dtype=torch.uint8, device="cuda")
    v2.cache_append_q8(x, _w_dkr(W), seq_idx, pos, table, pool_q)
    v2.check()
    tab = table.cpu()
    slots = [O.cache_slot(tab, int(b), int(p), d.block) for b, p in zip(seq_idx.tolist(), pos.tolist())]
    rows_bf = pool_bf.view(-1, d.width)[slots]
    got = pool_q.view(-1, ROW_BYTES)[slots].cpu().numpy()
    want = q8_bytes(rows_bf)
    assert np.array_equal(got[:, :512], want[:, :512]), "codes"
    assert np.array_equal(got[:, 512:544], want[:, 512:544]), "scales"
    assert np.array_equal(got[:, 544:], want[:, 544:]), "k^R"
    mask = torch.ones(n_blocks * d.block, dtype=torch.bool)
    mask[slots] = False
    assert bool((pool_q.view(-1, ROW_BYTES)[mask.cuda()] == 0xA5).all())
    # the quantised values are within half a step of the bf16 row they encode
    deq = dequantised(rows_bf)
    ref = to_np(rows_bf)
    step = np.repeat(O.quantize_cache_rows(ref, d.d_c)[1].astype(np.float64), 32, axis=1)
    assert np.all(np.abs(deq[:, :512] - ref[:, :512]) <= step / 2 + 1e-12)


def _q8_case(v2, seq_lens, q_counts, seed, workers, scale_rows=None):
    d = V2
    table, n_blocks, cu_q, lens, _ = batch_meta(seq_lens, q_counts, d.block, seed, spare_blocks=2)
    n_tok = int(sum(q_counts))
    q_lat, rows = latent_inputs(d, n_tok, int(sum(seq_lens)), seed)
    if scale_rows is not None:
        rows[scale_rows.cuda()] *= 8
    per_seq = list(torch.split(rows, [int(t) for t in seq_lens]))
    pool = q8_pool(per_seq, table, n_blocks, fill=0xFF)
    o_lat, lse = v2.decode_q8(q_lat, pool, table, lens, cu_q, num_workers=workers)
    v2.check()
    return q_lat, per_seq, o_lat, lse


def _check(q_lat, per_seq, seq_lens, q_counts, o_lat, lse, case, tokens=None):
    d = V2
    cu = np.concatenate([[0], np.cumsum(q_counts)])
    for b, L in enumerate(seq_lens):
        deq = None
        for k in range(int(q_counts[b])):
            n = int(cu[b]) + k
            if tokens is not None and n not in tokens:
                continue
            if deq is None:
                deq = dequantised(per_seq[b])
            t = int(L) - int(q_counts[b]) + k
            o_ref, l_ref = O.attend_latent(to_np(q_lat[n]), deq[:t + 1], d.d_c, d.d_h)
            e_o, e_l = row_rel_err(to_np(o_lat[n]), o_ref), lse_err(to_np(lse[n]), l_ref)
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
    ([127, 63, 300, 1000], [1, 2, 1, 2], 7),
])
def test_q8_decode_small(v2, seq_lens, q_counts, workers):
    q_lat, per_seq, o_lat, lse = _q8_case(v2, seq_lens, q_counts, 1110 + sum(seq_lens), workers)
    _check(q_lat, per_seq, seq_lens, q_counts, o_lat, lse, "quantised cache decode small cases")


def test_q8_decode_b64_t4096_all_tokens(v2):
    B, T = 64, 4096
    q_lat, per_seq, o_lat, lse = _q8_case(v2, [T] * B, [1] * B, 1120, 0)
    _check(q_lat, per_seq, [T] * B, [1] * B, o_lat, lse, "quantised cache B=64 T=4096 decode (64 tokens)")


def test_q8_decode_b1_t131072_hot_rows(v2):
    T = 131072
    hot = synth.pick_rows(T, 0.01, 1121)
    q_lat, per_seq, o_lat, lse = _q8_case(v2, [T], [1], 1121, 0, scale_rows=hot)
    _check(q_lat, per_seq, [T], [1], o_lat, lse, "quantised cache B=1 T=131072 hot rows")


def test_q8_decode_from_appended_rows(v2):
    """The cache built by mla_cache_append_q8 (prior rows and the step's own
    rows), read by mla_decode_q8: checked against the oracle on the
    dequantised rows of the plain append."""
    d, T = V2, 300
    W = synth.weights(d, 1122, device="cuda")
    h = synth.hidden(T, d, 1122, device="cuda")
    table, n_blocks, cu_q, seq_lens, _ = batch_meta([T], [1], d.block, 1122)
    zeros = torch.zeros(T, dtype=torch.int32, device="cuda")
    allpos = torch.arange(T, dtype=torch.int32, device="cuda")
    pool_q = torch.zeros(n_blocks, d.block, ROW_BYTES, dtype=torch.uint8, device="cuda")
    pool_bf = torch.zeros(n_blocks, d.block, d.width, dtype=torch.bfloat16, device="cuda")
    v2.cache_append_q8(h, _w_dkr(W), zeros, allpos, table, pool_q)
    v2.cache_append(h, _w_dkr(W), zeros, allpos, table, pool_bf)
    q_lat, _ = latent_inputs(d, 1, 1, 1122)
    o_lat, lse = v2.decode_q8(q_lat, pool_q, table, seq_lens, cu_q)
    v2.check()
    tab = table.cpu()
    rows_bf = pool_bf.view(-1, d.width)[[O.cache_slot(tab, 0, j, d.block) for j in range(T)]]
    o_ref, l_ref = O.attend_latent(to_np(q_lat[0]), dequantised(rows_bf), d.d_c, d.d_h)
    e_o, e_l = row_rel_err(to_np(o_lat[0]), o_ref), lse_err(to_np(lse[0]), l_ref)
    record("quantised cache from mla_cache_append_q8", e_o, e_l)
    assert e_o < OUT_TOL and e_l < LSE_TOL


def test_q8_unsupported_dims(v2):
    from head_latent_attention_26_b300 import mla
    tiny = mla.MLA(synth.TINY, 64, torch.float32)
    q = torch.zeros(1, 4, 20, dtype=torch.float32, device="cuda")
    pool = torch.zeros(1, 64, ROW_BYTES, dtype=torch.uint8, device="cuda")
    table = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
    lens = torch.tensor([1], dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        tiny.decode_q8(q, pool, table, lens, cu, ws=torch.empty(256, dtype=torch.uint8, device="cuda"))
    assert e.value.code == 2
