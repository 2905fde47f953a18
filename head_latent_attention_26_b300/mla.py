"""ctypes binding of libmla.so (include/mla.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (PyTorch provides device memory and
streams); their data pointers and the current stream are passed through.
There is no CPU fallback: without the built library, or without a CUDA
device, these calls raise.
"""

from __future__ import annotations

import ctypes
import os
import re

import torch

from .build import LIB, ROOT
from .synth import Dims

HEADER = os.path.join(ROOT, "include", "mla.h")

#: Bytes of the output projection's weights a decode step has the attention
#: fetch into L2 (a 126 MB L2 keeps about this much of a normal-priority
#: prefetch alive beside the evict-first cache stream).
OUT_WEIGHT_PREFETCH_BYTES = 96 << 20
#: Steps of more tokens than this run the output projection as two launches
#: and their decode re-reads more of its own data through L2 (queries, split
#: partials); there the prefetch cost the decode more than it saved (a ragged
#: batch of 194 tokens: decode +12 µs, output projection -1.9 µs).
OUT_WEIGHT_PREFETCH_MAX_TOKENS = 64


def default_prefetch_bytes(n_tok: int) -> int:
    """The L2 prefetch budget decode_step uses for a step of n_tok tokens."""
    return OUT_WEIGHT_PREFETCH_BYTES if n_tok <= OUT_WEIGHT_PREFETCH_MAX_TOKENS else 0


def output_weight_prefetch(W_uv: torch.Tensor, W_o: torch.Tensor, budget_bytes: int) -> tuple:
    """Ranges for MLA.set_decode_l2_prefetch ahead of the output projection:
    W^UV whole (its first phase reads it) and then the leading whole 128-row
    tiles of W^O, at most budget_bytes in all; () for a budget of 0."""
    uv = W_uv.numel() * W_uv.element_size()
    if budget_bytes <= 0:
        return ()
    if budget_bytes <= uv:
        return (W_uv.reshape(-1)[:budget_bytes // 16 * 16 // W_uv.element_size()],)
    rows = min(W_o.shape[0], (budget_bytes - uv) // (W_o.shape[1] * W_o.element_size()) // 128 * 128)
    return (W_uv, W_o[:rows]) if rows > 0 else (W_uv,)

MLA_OK = 0
STATUS = {
    0: "MLA_OK",
    1: "MLA_ERR_INVALID_ARG",
    2: "MLA_ERR_UNSUPPORTED",
    3: "MLA_ERR_WORKSPACE",
    4: "MLA_ERR_CUDA",
    5: "MLA_ERR_DEVICE_TIMEOUT",
    6: "MLA_ERR_DEVICE_BOUNDS",
}
BF16, F32 = 0, 1


class MLAError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)}")
        self.code = code


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_h", "d_h", "d_hr", "d_c", "d_cq", "d_model", "block")] + [
        ("rope_base", ctypes.c_float), ("scale", ctypes.c_float), ("dtype", ctypes.c_int)]


_lib = None
P, I, SZ, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_longlong

_SIGS = {
    "mla_create": (I, [ctypes.POINTER(_Dims), I, ctypes.POINTER(P)]),
    "mla_destroy": (None, [P]),
    "mla_status_string": (ctypes.c_char_p, [I]),
    "mla_num_sms": (I, [P]),
    "mla_uses_tensor_path": (I, [P]),
    "mla_set_wait_limit": (I, [P, LL]),
    "mla_set_decode_l2_prefetch": (I, [P, ctypes.POINTER(P), ctypes.POINTER(SZ), I]),
    "mla_q_proj_workspace_bytes": (SZ, [P, I]),
    "mla_q_proj": (I, [P, P, P, P, P, I, P, P, P, SZ, P]),
    "mla_cache_append": (I, [P, P, P, P, P, I, P, I, I, P, I, P]),
    "mla_q_proj_append": (I, [P, P, P, P, P, P, P, P, I, P, I, I, P, I, P, P, P, SZ, P]),
    "mla_q_latent_append_workspace_bytes": (SZ, [P, I]),
    "mla_q_latent_append": (I, [P, P, P, P, P, P, P, P, P, I, P, I, I, P, I, P, P, SZ, P]),
    "mla_cache_append_q8_workspace_bytes": (SZ, [P, I]),
    "mla_cache_append_q8": (I, [P, P, P, P, P, I, P, I, I, P, I, P, SZ, P]),
    "mla_absorb_q": (I, [P, P, P, P, I, P, P, P]),
    "mla_absorb_weights": (I, [P, P, P, P, P]),
    "mla_q_proj_absorbed": (I, [P, P, P, P, P, P, I, P, P, SZ, P]),
    "mla_decode_workspace_bytes": (SZ, [P, I, I]),
    "mla_decode": (I, [P, P, P, I, P, I, P, P, I, I, I, P, SZ, P, P, P]),
    "mla_decode_noalloc": (I, [P, P, P, I, P, I, P, P, I, I, I, P, P, P]),
    "mla_decode_q8": (I, [P, P, P, I, P, I, P, P, I, I, I, P, SZ, P, P, P]),
    "mla_prefill_workspace_bytes": (SZ, [P, I]),
    "mla_prefill": (I, [P, P, P, P, I, P, P, P, SZ, P, P, P]),
    "mla_out_workspace_bytes": (SZ, [P, I]),
    "mla_out": (I, [P, P, P, P, I, P, P, SZ, P]),
    "mla_check_device_status": (I, [P, P]),
    "mla_selftest_wait_timeout": (I, [P, P]),
    "mla_device_error_site": (I, [P, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(I)]),
}


def header_symbols() -> list:
    """Every function name declared in include/mla.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(mla_\w+)\s*\(", text, re.M)))


def load(path: str = LIB):
    """Load libmla.so and declare its signatures (no GPU needed)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with head_latent_attention_26_b300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _check(code: int, what: str):
    if code != MLA_OK:
        raise MLAError(code, what)


class MLA:
    """One attention layer's kernels on the current CUDA device.

    dims: layer sizes; max_pos: positions the RoPE table covers; dtype:
    torch.bfloat16 (storage and MMA type) or torch.float32.
    """

    def __init__(self, dims: Dims, max_pos: int, dtype=torch.bfloat16):
        if not torch.cuda.is_available():
            raise RuntimeError("MLA needs a CUDA device: there is no CPU fallback")
        self.lib = load()
        self.dims = dims
        self.dtype = dtype
        self.max_pos = max_pos
        d = _Dims(dims.n_h, dims.d_h, dims.d_hr, dims.d_c, dims.d_cq, dims.d_model, dims.block,
                  dims.rope_base, dims.scale, BF16 if dtype == torch.bfloat16 else F32)
        h = P()
        _check(self.lib.mla_create(ctypes.byref(d), max_pos, ctypes.byref(h)), "mla_create")
        self.h = h
        self._ws = {}

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            self.lib.mla_destroy(h)
            self.h = None

    # ---- plumbing ---------------------------------------------------------
    @property
    def tensor_path(self) -> bool:
        return bool(self.lib.mla_uses_tensor_path(self.h))

    @property
    def num_sms(self) -> int:
        return self.lib.mla_num_sms(self.h)

    def workspace(self, key: str, nbytes: int) -> torch.Tensor:
        """A cached device buffer of at least nbytes (allocated by torch)."""
        buf = self._ws.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
            self._ws[key] = buf
        return buf

    def set_wait_limit(self, polls: int):
        _check(self.lib.mla_set_wait_limit(self.h, polls), "mla_set_wait_limit")

    def set_decode_l2_prefetch(self, *ranges):
        """Device ranges (contiguous tensors or tensor views; at most two)
        that later decode calls fetch into L2 while they stream the cache,
        for the kernel that follows them (the output projection's weights);
        no argument clears.  The tensors are kept alive while they are set."""
        ptrs, sizes = (P * max(2, len(ranges)))(), (SZ * max(2, len(ranges)))()
        for i, t in enumerate(ranges):
            if not t.is_contiguous():
                raise ValueError("an L2 prefetch range must be contiguous")
            ptrs[i], sizes[i] = t.data_ptr(), t.numel() * t.element_size()
        _check(self.lib.mla_set_decode_l2_prefetch(self.h, ptrs, sizes, len(ranges)), "mla_set_decode_l2_prefetch")
        self._l2_prefetch = tuple(ranges)

    def check(self):
        """Synchronise and raise if any kernel recorded a device-side error."""
        _check(self.lib.mla_check_device_status(self.h, P(_stream())), "device status")

    def device_status(self) -> int:
        return self.lib.mla_check_device_status(self.h, P(_stream()))

    def error_site(self):
        """(site word, CTA, tile) of the first bounded wait that ran out, as
        read back by the last check (site word 0 = none)."""
        a, b, c = I(), I(), I()
        _check(self.lib.mla_device_error_site(self.h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
               "mla_device_error_site")
        return a.value, b.value, c.value

    def selftest_wait_timeout(self) -> int:
        _check(self.lib.mla_selftest_wait_timeout(self.h, P(_stream())), "selftest launch")
        return self.device_status()

    # ---- the path ---------------------------------------------------------
    def q_proj(self, x, W_dq, W_uq, W_qr, q_c=None, q_r=None):
        d, n = self.dims, x.shape[0]
        q_c = torch.empty(n, d.n_h, d.d_h, dtype=self.dtype, device=x.device) if q_c is None else q_c
        q_r = torch.empty(n, d.n_h, d.d_hr, dtype=self.dtype, device=x.device) if q_r is None else q_r
        nb = self.lib.mla_q_proj_workspace_bytes(self.h, n)
        ws = self.workspace("q_proj", nb)
        _check(self.lib.mla_q_proj(self.h, _ptr(x), _ptr(W_dq), _ptr(W_uq), _ptr(W_qr), n, _ptr(q_c), _ptr(q_r),
                                   _ptr(ws), ws.numel(), P(_stream())), "mla_q_proj")
        return q_c, q_r

    def cache_append(self, x, W_dkr, seq_idx, pos, block_table, pool):
        _check(self.lib.mla_cache_append(self.h, _ptr(x), _ptr(W_dkr), _ptr(seq_idx), _ptr(pos), x.shape[0],
                                         _ptr(block_table), block_table.shape[1], block_table.shape[0],
                                         _ptr(pool), pool.shape[0], P(_stream())), "mla_cache_append")
        return pool

    def q_proj_append(self, x, W_dq, W_uq, W_qr, W_dkr, seq_idx, pos, block_table, pool, q_c=None, q_r=None):
        """mla_q_proj_append: q_proj and cache_append of the same new tokens,
        the two products that read x in one launch.  Returns (q_c, q_r)."""
        d, n = self.dims, x.shape[0]
        q_c = torch.empty(n, d.n_h, d.d_h, dtype=self.dtype, device=x.device) if q_c is None else q_c
        q_r = torch.empty(n, d.n_h, d.d_hr, dtype=self.dtype, device=x.device) if q_r is None else q_r
        ws = self.workspace("q_proj", self.lib.mla_q_proj_workspace_bytes(self.h, n))
        _check(self.lib.mla_q_proj_append(self.h, _ptr(x), _ptr(W_dq), _ptr(W_uq), _ptr(W_qr), _ptr(W_dkr),
                                          _ptr(seq_idx), _ptr(pos), n, _ptr(block_table), block_table.shape[1],
                                          block_table.shape[0], _ptr(pool), pool.shape[0], _ptr(q_c), _ptr(q_r),
                                          _ptr(ws), ws.numel(), P(_stream())), "mla_q_proj_append")
        return q_c, q_r

    def q_latent_append(self, x, W_dq, W_uq, W_qr, W_uk, W_dkr, seq_idx, pos, block_table, pool, q_lat=None):
        """mla_q_latent_append: the latent query [n_tok, n_h, d_c + d_hr] of
        the new tokens and their cache rows (q_proj + cache_append + absorb_q
        in two launches for up to 64 tokens)."""
        d, n = self.dims, x.shape[0]
        q_lat = torch.empty(n, d.n_h, d.width, dtype=self.dtype, device=x.device) if q_lat is None else q_lat
        ws = self.workspace("q_latent", self.lib.mla_q_latent_append_workspace_bytes(self.h, n))
        _check(self.lib.mla_q_latent_append(self.h, _ptr(x), _ptr(W_dq), _ptr(W_uq), _ptr(W_qr), _ptr(W_uk),
                                            _ptr(W_dkr), _ptr(seq_idx), _ptr(pos), n, _ptr(block_table),
                                            block_table.shape[1], block_table.shape[0], _ptr(pool), pool.shape[0],
                                            _ptr(q_lat), _ptr(ws), ws.numel(), P(_stream())), "mla_q_latent_append")
        return q_lat

    def cache_append_q8(self, x, W_dkr, seq_idx, pos, block_table, pool_q8):
        """mla_cache_append_q8: the new tokens' rows, quantised, into a
        [n_blocks, block, 672] uint8 pool."""
        n = x.shape[0]
        ws = self.workspace("append_q8", self.lib.mla_cache_append_q8_workspace_bytes(self.h, n))
        _check(self.lib.mla_cache_append_q8(self.h, _ptr(x), _ptr(W_dkr), _ptr(seq_idx), _ptr(pos), n,
                                            _ptr(block_table), block_table.shape[1], block_table.shape[0],
                                            _ptr(pool_q8), pool_q8.shape[0], _ptr(ws), ws.numel(), P(_stream())),
               "mla_cache_append_q8")
        return pool_q8

    def absorb_q(self, q_c, q_r, pos, W_uk, q_lat=None):
        d, n = self.dims, q_c.shape[0]
        q_lat = torch.empty(n, d.n_h, d.width, dtype=self.dtype, device=q_c.device) if q_lat is None else q_lat
        _check(self.lib.mla_absorb_q(self.h, _ptr(q_c), _ptr(q_r), _ptr(pos), n, _ptr(W_uk), _ptr(q_lat),
                                     P(_stream())), "mla_absorb_q")
        return q_lat

    def absorb_weights(self, W_uq, W_uk, W_uq_abs=None):
        """The folded query weight W^UK_i^T W^UQ_i of every head, [n_h*d_c, d_cq]."""
        d = self.dims
        if W_uq_abs is None:
            W_uq_abs = torch.empty(d.n_h * d.d_c, d.d_cq, dtype=self.dtype, device=W_uq.device)
        _check(self.lib.mla_absorb_weights(self.h, _ptr(W_uq), _ptr(W_uk), _ptr(W_uq_abs), P(_stream())),
               "mla_absorb_weights")
        return W_uq_abs

    def q_proj_absorbed(self, x, W_dq, W_uq_abs, W_qr, pos, q_lat=None):
        """The latent query straight from x with the folded weight (replaces
        q_proj + absorb_q)."""
        d, n = self.dims, x.shape[0]
        q_lat = torch.empty(n, d.n_h, d.width, dtype=self.dtype, device=x.device) if q_lat is None else q_lat
        nb = self.lib.mla_q_proj_workspace_bytes(self.h, n)
        ws = self.workspace("q_proj", nb)
        _check(self.lib.mla_q_proj_absorbed(self.h, _ptr(x), _ptr(W_dq), _ptr(W_uq_abs), _ptr(W_qr), _ptr(pos), n,
                                            _ptr(q_lat), _ptr(ws), ws.numel(), P(_stream())), "mla_q_proj_absorbed")
        return q_lat

    def decode_workspace_bytes(self, n_tok: int, num_workers: int = 0) -> int:
        return self.lib.mla_decode_workspace_bytes(self.h, n_tok, num_workers)

    def decode(self, q_lat, pool, block_table, seq_lens, cu_q, num_workers: int = 0, o_lat=None, lse=None,
               ws=None):
        d, n = self.dims, q_lat.shape[0]
        o_lat = torch.empty(n, d.n_h, d.d_c, dtype=self.dtype, device=q_lat.device) if o_lat is None else o_lat
        lse = torch.empty(n, d.n_h, dtype=torch.float32, device=q_lat.device) if lse is None else lse
        if ws is None:
            ws = self.workspace("decode", self.decode_workspace_bytes(n, num_workers))
        _check(self.lib.mla_decode(self.h, _ptr(q_lat), _ptr(pool), pool.shape[0], _ptr(block_table),
                                   block_table.shape[1], _ptr(seq_lens), _ptr(cu_q), seq_lens.shape[0], n,
                                   num_workers, _ptr(ws), ws.numel(), _ptr(o_lat), _ptr(lse), P(_stream())),
               "mla_decode")
        return o_lat, lse

    def decode_q8(self, q_lat, pool_q8, block_table, seq_lens, cu_q, num_workers: int = 0, o_lat=None, lse=None,
                  ws=None):
        """mla_decode_q8: the attention over a quantised cache pool
        ([n_blocks, block, 672] uint8)."""
        d, n = self.dims, q_lat.shape[0]
        o_lat = torch.empty(n, d.n_h, d.d_c, dtype=self.dtype, device=q_lat.device) if o_lat is None else o_lat
        lse = torch.empty(n, d.n_h, dtype=torch.float32, device=q_lat.device) if lse is None else lse
        if ws is None:
            ws = self.workspace("decode", self.decode_workspace_bytes(n, num_workers))
        _check(self.lib.mla_decode_q8(self.h, _ptr(q_lat), _ptr(pool_q8), pool_q8.shape[0], _ptr(block_table),
                                      block_table.shape[1], _ptr(seq_lens), _ptr(cu_q), seq_lens.shape[0], n,
                                      num_workers, _ptr(ws), ws.numel(), _ptr(o_lat), _ptr(lse), P(_stream())),
               "mla_decode_q8")
        return o_lat, lse

    def decode_noalloc(self, q_lat, pool, block_table, seq_lens, cu_q, num_workers: int = 0, o_lat=None,
                       lse=None):
        """mla_decode_noalloc: the same attention, scratch in the library's
        fixed device array instead of a workspace argument."""
        d, n = self.dims, q_lat.shape[0]
        o_lat = torch.empty(n, d.n_h, d.d_c, dtype=self.dtype, device=q_lat.device) if o_lat is None else o_lat
        lse = torch.empty(n, d.n_h, dtype=torch.float32, device=q_lat.device) if lse is None else lse
        _check(self.lib.mla_decode_noalloc(self.h, _ptr(q_lat), _ptr(pool), pool.shape[0], _ptr(block_table),
                                           block_table.shape[1], _ptr(seq_lens), _ptr(cu_q), seq_lens.shape[0], n,
                                           num_workers, _ptr(o_lat), _ptr(lse), P(_stream())), "mla_decode_noalloc")
        return o_lat, lse

    def prefill(self, rows, q_c, q_r, W_uk, W_uv, o=None, lse=None):
        """mla_prefill: causal attention of a P-token prompt over its expanded
        keys and values.  rows [P, d_c + d_hr] (the prompt's cache rows in
        position order), q_c [P, n_h, d_h], q_r [P, n_h, d_hr] (before RoPE).
        Returns o [P, n_h, d_h] and lse [P, n_h]."""
        d, n = self.dims, rows.shape[0]
        o = torch.empty(n, d.n_h, d.d_h, dtype=self.dtype, device=rows.device) if o is None else o
        lse = torch.empty(n, d.n_h, dtype=torch.float32, device=rows.device) if lse is None else lse
        ws = self.workspace("prefill", self.lib.mla_prefill_workspace_bytes(self.h, n))
        _check(self.lib.mla_prefill(self.h, _ptr(rows), _ptr(q_c), _ptr(q_r), n, _ptr(W_uk), _ptr(W_uv), _ptr(ws),
                                    ws.numel(), _ptr(o), _ptr(lse), P(_stream())), "mla_prefill")
        return o, lse

    def out(self, o_lat, W_uv, W_o, u=None):
        d, n = self.dims, o_lat.shape[0]
        u = torch.empty(n, d.d_model, dtype=self.dtype, device=o_lat.device) if u is None else u
        ws = self.workspace("out", self.lib.mla_out_workspace_bytes(self.h, n))
        _check(self.lib.mla_out(self.h, _ptr(o_lat), _ptr(W_uv), _ptr(W_o), n, _ptr(u), _ptr(ws), ws.numel(),
                                P(_stream())), "mla_out")
        return u

    def decode_step(self, x, W: dict, W_dkr, seq_idx, pos, block_table, pool, seq_lens, cu_q,
                    num_workers: int = 0, out: dict | None = None,
                    l2_prefetch_bytes: int | None = None):
        """One whole decode step for new tokens x: the latent query and the
        new cache rows (one call), attention over the latent cache and the
        output projection.  While the attention streams the cache it fetches
        up to l2_prefetch_bytes of W^UV and W^O into L2 for the output
        projection (tensor path; None = default_prefetch_bytes(n_tok), 0 =
        none).  Returns u [n_tok, d_model]."""
        out = {} if out is None else out
        if l2_prefetch_bytes is None:
            l2_prefetch_bytes = default_prefetch_bytes(x.shape[0])
        q_lat = self.q_latent_append(x, W["W_dq"], W["W_uq"], W["W_qr"], W["W_uk"], W_dkr, seq_idx, pos,
                                     block_table, pool, out.get("q_lat"))
        ranges = output_weight_prefetch(W["W_uv"], W["W_o"], l2_prefetch_bytes) if self.tensor_path else ()
        if ranges:
            self.set_decode_l2_prefetch(*ranges)
        try:
            o_lat, lse = self.decode(q_lat, pool, block_table, seq_lens, cu_q, num_workers, out.get("o_lat"),
                                     out.get("lse"))
        finally:
            if ranges:
                self.set_decode_l2_prefetch()
        u = self.out(o_lat, W["W_uv"], W["W_o"], out.get("u"))
        out.update(q_lat=q_lat, o_lat=o_lat, lse=lse, u=u)
        return u
