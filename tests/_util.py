"""Shared helpers for the parity tests: tolerances, input recipes, pool filling."""

from __future__ import annotations

import numpy as np
import torch

from head_latent_attention_26_b300 import synth

# Tolerances: max relative error 1e-2 on outputs (per output row:
# max|gpu - ref| / max|ref|), 2e-3 on log-sum-exp (|d| / max(1, |lse|)),
# against the fp64 oracle for bf16 inputs with fp32 accumulation.
OUT_TOL = 1e-2
LSE_TOL = 2e-3


# worst error seen per test case, printed at the end of the session so that
# each configuration's margin against the gates is on record
MARGINS: dict = {}


def record(case: str, out_err: float = None, lse_err_: float = None):
    """Keep the largest output / lse error seen for `case`."""
    o, l = MARGINS.get(case, (0.0, 0.0))
    MARGINS[case] = (max(o, out_err or 0.0), max(l, lse_err_ or 0.0))


def row_rel_err(gpu, ref) -> float:
    """Largest per-row max|gpu-ref| / max|ref| over the leading axes."""
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    g = g.reshape(-1, g.shape[-1])
    r = r.reshape(-1, r.shape[-1])
    num = np.max(np.abs(g - r), axis=1)
    den = np.maximum(np.max(np.abs(r), axis=1), 1e-30)
    return float(np.max(num / den))


def lse_err(gpu, ref) -> float:
    g = np.asarray(gpu, dtype=np.float64).reshape(-1)
    r = np.asarray(ref, dtype=np.float64).reshape(-1)
    return float(np.max(np.abs(g - r) / np.maximum(1.0, np.abs(r))))


def to_np(t) -> np.ndarray:
    return t.detach().to("cpu").double().numpy()


def latent_inputs(d: synth.Dims, n_tok: int, rows_total: int, seed: int, device="cuda",
                  dtype=torch.bfloat16):
    """Latent queries and cached rows drawn with the statistics the real path
    produces for h ~ N(0,1), W ~ N(0, 1/fan_in): q~ ~ N(0, 1/4) (d_h terms of
    variance 1/d_c... summed: d_h/d_c), q^R ~ N(0,1), c ~ N(0,1), k^R ~ N(0,1),
    so scaled scores are about N(0, 1)."""
    qstd = float(np.sqrt(d.d_h / d.d_c))
    q_lat = torch.cat([synth.normal((n_tok, d.n_h, d.d_c), seed, "q_tilde", std=qstd, dtype=dtype, device=device),
                       synth.normal((n_tok, d.n_h, d.d_hr), seed, "q_rope", dtype=dtype, device=device)], dim=2)
    rows = synth.normal((rows_total, d.width), seed, "rows", dtype=dtype, device=device)
    return q_lat.contiguous(), rows


def scatter_rows(rows_per_seq, table, n_blocks, block, width, dtype=torch.bfloat16, device="cuda",
                 fill=0.0):
    """Place each sequence's rows in the pool through the block table."""
    pool = torch.full((n_blocks, block, width), fill, dtype=dtype, device=device)
    flat = pool.view(-1, width)
    for b, rows in enumerate(rows_per_seq):
        T = rows.shape[0]
        if T == 0:
            continue
        j = torch.arange(T, device=device)
        blk = table[b].to(device)[j // block].long()
        flat[blk * block + (j % block)] = rows.to(device=device, dtype=dtype)
    return pool


def batch_meta(seq_lens, q_counts, block, seed, spare_blocks=0, device="cuda"):
    """Block table, cu_q, seq_lens and per-token positions for a ragged batch."""
    table, n_blocks = synth.block_table(seq_lens, block, seed, spare_blocks)
    cu_q = synth.cu_from_counts(q_counts)
    pos = []
    for L, q in zip(seq_lens, q_counts):
        pos += [int(L) - int(q) + k for k in range(int(q))]
    return (table.to(device), n_blocks, cu_q.to(device),
            torch.tensor([int(x) for x in seq_lens], dtype=torch.int32, device=device),
            torch.tensor(pos, dtype=torch.int32, device=device))
