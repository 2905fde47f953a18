"""Seeded synthetic inputs for the MLA decode path.

This module holds no arithmetic of the method: it only draws random tensors,
block tables and lengths.  The same arrays feed both the CUDA library and the
fp64 oracle, so every comparison sees identical inputs.

Recipe (the workloads' shapes and distributions):
  * hidden states h ~ N(0, 1);
  * every weight W ~ N(0, 1/fan_in) with fan_in its input width;
  * values are drawn in float32 and rounded once to the storage dtype;
  * a cache pool of sum_b ceil(T_b / block) blocks is handed out to the
    sequences through a seeded random permutation of the physical blocks;
  * ragged lengths are uniform integers in [lo, hi]; query counts are 1 or 2
    with equal probability.

Each tensor has its own torch.Generator seeded from (seed, name), so adding a
tensor never changes the values of another.
"""

from __future__ import annotations

import math
import zlib
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Dims:
    """Layer sizes in the pages' notation (see include/mla.h)."""

    n_h: int
    d_h: int
    d_hr: int
    d_c: int
    d_cq: int
    d_model: int
    block: int = 64
    rope_base: float = 10000.0

    @property
    def width(self) -> int:
        """Elements of one cached row: d_c + d_hr."""
        return self.d_c + self.d_hr

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d_h + self.d_hr)


#: DeepSeek-V2 layer sizes: d=5120, n_h=128, d_h=128, d_h^R=64, d_c=512, d_c'=1536.
V2 = Dims(n_h=128, d_h=128, d_hr=64, d_c=512, d_cq=1536, d_model=5120, block=64)
#: Tiny single layer used for exhaustive parity: n_h=4, d_h=8, d_h^R=4, d_c=16, d_c'=24, d=32.
TINY = Dims(n_h=4, d_h=8, d_hr=4, d_c=16, d_cq=24, d_model=32, block=64)


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 0x9E3779B1 + zlib.crc32(name.encode())) & 0x7FFFFFFFFFFFFFFF)
    return g


def normal(shape, seed: int, name: str, std: float = 1.0, dtype=torch.bfloat16,
           device="cpu") -> torch.Tensor:
    """N(0, std^2) in float32, rounded once to ``dtype``."""
    g = _gen(seed, name, device)
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def weights(d: Dims, seed: int, dtype=torch.bfloat16, device="cpu") -> dict:
    """All projection matrices of one layer, [out, in] row-major, N(0, 1/fan_in)."""
    H, Hr = d.n_h * d.d_h, d.n_h * d.d_hr
    shapes = {
        "W_dkv": (d.d_c, d.d_model),
        "W_kr": (d.d_hr, d.d_model),
        "W_dq": (d.d_cq, d.d_model),
        "W_uq": (H, d.d_cq),
        "W_qr": (Hr, d.d_cq),
        "W_uk": (H, d.d_c),
        "W_uv": (H, d.d_c),
        "W_o": (d.d_model, H),
    }
    return {k: normal(s, seed, k, std=1.0 / math.sqrt(s[1]), dtype=dtype, device=device)
            for k, s in shapes.items()}


def hidden(n: int, d: Dims, seed: int, name: str = "h", dtype=torch.bfloat16,
           device="cpu") -> torch.Tensor:
    """n hidden states h ~ N(0, 1), [n, d_model]."""
    return normal((n, d.d_model), seed, name, dtype=dtype, device=device)


def block_table(seq_lens, block: int, seed: int, spare_blocks: int = 0):
    """Scatter every sequence's logical blocks over a randomly permuted pool.

    Returns (table [B, max_blocks] int32 with -1 past each sequence's end,
    n_pool_blocks).  ``spare_blocks`` extra physical blocks stay unowned.
    """
    lens = [int(t) for t in seq_lens]
    nb = [(t + block - 1) // block for t in lens]
    total = sum(nb) + spare_blocks
    perm = torch.randperm(total, generator=_gen(seed, "block_perm", "cpu"))
    max_blocks = max(nb) if nb else 1
    table = torch.full((len(lens), max_blocks), -1, dtype=torch.int32)
    k = 0
    for b, n in enumerate(nb):
        table[b, :n] = perm[k:k + n].to(torch.int32)
        k += n
    return table, total


def ragged_lengths(B: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """B integers uniform in [lo, hi]."""
    return torch.randint(lo, hi + 1, (B,), generator=_gen(seed, "lens", "cpu"), dtype=torch.int64)


def query_counts(B: int, seed: int) -> torch.Tensor:
    """B query counts, 1 or 2 with equal probability."""
    return torch.randint(1, 3, (B,), generator=_gen(seed, "q_lens", "cpu"), dtype=torch.int64)


def pick_rows(n_rows: int, frac: float, seed: int, name: str = "hot_rows") -> torch.Tensor:
    """A seeded subset of round(frac * n_rows) distinct row indices, sorted."""
    k = max(1, int(round(frac * n_rows)))
    perm = torch.randperm(n_rows, generator=_gen(seed, name, "cpu"))
    return torch.sort(perm[:k]).values


def cu_from_counts(counts) -> torch.Tensor:
    """Exclusive prefix sum with a trailing total: [0, c0, c0+c1, ...] (int32)."""
    c = torch.as_tensor(counts, dtype=torch.int64)
    return torch.cat([torch.zeros(1, dtype=torch.int64), torch.cumsum(c, 0)]).to(torch.int32)
