"""Benchmark of one MLA decode step on B300.

Workloads (DeepSeek-V2 attention layer: d=5120, n_h=128, d_h=128, d_h^R=64,
d_c=512, d_c'=1536; 64-row cache blocks scattered over a seeded random
permutation of the pool):

  b64_t4096    (default) B=64 sequences x T=4096 cached rows, 1 new token each
  b1_t4096     B=1, T=4096
  b1_t131072   B=1, T=131072 (128K context), 1% of the cached rows scaled by 8
  ragged_b128  B=128, T_b ~ U[512, 16384], 1 or 2 new tokens per sequence
  b64_t4096_q8 b64_t4096 over the quantised latent cache (int8 codes of c^KV
               with an fp16 scale per 32 values, bf16 k^R: 672 B per row)
  prefill_p4096  a P=4096-token prompt: query projection, cache rows, and
               causal attention over the expanded keys and values

One step = the whole path for the step's new tokens: the latent query with
the cache append (mla_q_latent_append: query projection, cache rows, W^UK
absorption), latent attention (+ split combine), W^UV / W^O output.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

The timed steps are replayed as CUDA graphs of the library's C-ABI calls (the
calls are captured once; a replay launches the same kernels with no host work
in between), so the device time of the step is measured, not the host's
launch rate.  Event nodes around each step's decode call give the decode time
of every timed step.  Prints one JSON line.  Under torchrun every rank runs
an independent replica on its own GPU (the path has no exchange step); the
time is the max over ranks.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from head_latent_attention_26_b300 import synth  # noqa: E402

METRIC = "MLA decode tokens/s and latent-cache GB/s (% of HBM/tensor roofline), 1×B300"

# DRAM bytes (read + write) of one decode_tc_kernel launch on the B=64, T=4096
# workload with the given L2 prefetch, from an ncu capture of the kernel
# sources with these hashes; the figure is reported only while the sources
# still hash to them.
PROFILED_DECODE = {"sources": {"decode_tc.cu": "4594af35cf9b4dfa", "ptx.cuh": "c59e8751e182f4db"},
                   "workload": (64, 4096), "l2_prefetch_bytes": 100663296, "traffic_bytes": 415685632}


def _profiled_traffic(B: int, T: int, pf_bytes: int):
    import hashlib
    if (B, T, pf_bytes) != (*PROFILED_DECODE["workload"], PROFILED_DECODE["l2_prefetch_bytes"]):
        return None
    csrc = os.path.join(ROOT, "head_latent_attention_26_b300", "csrc")
    for name, digest in PROFILED_DECODE["sources"].items():
        with open(os.path.join(csrc, name), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != digest:
                return None
    return PROFILED_DECODE["traffic_bytes"]


SEED = 1003
B_DEFAULT, T_DEFAULT = 64, 4096
# A timed region at least this long runs the GPU at its sustained (power
# capped) tensor rate; shorter ones are compared with the burst rate.
SUSTAINED_REGION_S = 1.0

WORKLOADS = {
    "b64_t4096": dict(kind="uniform", B=64, T=4096, hot=0.0),
    "b1_t4096": dict(kind="uniform", B=1, T=4096, hot=0.0),
    "b1_t131072": dict(kind="uniform", B=1, T=131072, hot=0.01),
    "ragged_b128": dict(kind="ragged", B=128, lo=512, hi=16384, hot=0.0),
    # the headline step over the quantised latent cache (672-byte rows)
    "b64_t4096_q8": dict(kind="uniform", B=64, T=4096, hot=0.0, q8=True),
    # a 4096-token prompt through the expanded-K/V prefill
    "prefill_p4096": dict(kind="prefill", P=4096),
}
Q8_ROW_BYTES = 672


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    except (OSError, KeyError, ValueError):
        return 6400.0, 1800.0, 1400.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    return ws, rank


def _init_dist(ws: int, backend: str = "nccl"):
    """Joins the process group of a torchrun launch (nothing at N=1)."""
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend)


def _barrier(ws: int, cuda: bool = True):
    """All ranks meet, then this rank's device work drains."""
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    if cuda:
        torch.cuda.synchronize()


def _max_over_ranks(vals, ws: int, device="cuda"):
    """Element-wise maximum of the per-rank timings (every rank gets it)."""
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    if ws > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def _job_rate(units_per_rank: int, ws: int, ms: float) -> float:
    """Whole-job throughput: the units all ranks processed in one step over
    the slowest rank's step time."""
    return units_per_rank * ws / (ms * 1e-3)


def roofline_choice(t_hbm_s: float, t_tc_burst_s: float, t_tc_sus_s: float, region_s: float):
    """Which roof binds the decode kernel and the tensor peak it is held to.

    The tensor peak is the burst one unless the timed region lasts seconds (a
    kernel inside a long loop runs at the sustained, power-capped rate).  The
    binding roof is the slower of HBM and tensor: the larger lower bound on
    the kernel's time.  Returns (bound, t_roof_s, tensor_peak_kind)."""
    sustained = region_s >= SUSTAINED_REGION_S
    t_tc = t_tc_sus_s if sustained else t_tc_burst_s
    kind = "sustained" if sustained else "burst"
    if t_tc > t_hbm_s:
        return "tensor", t_tc, kind
    return "hbm", t_hbm_s, kind


_SAMPLER = r"""
import ctypes, sys, time
lib = ctypes.CDLL("libnvidia-ml.so.1")
assert lib.nvmlInit_v2() == 0
h = ctypes.c_void_p()
bus = sys.argv[1]
if not bus or lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
    assert lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(int(sys.argv[2])), ctypes.byref(h)) == 0
c, r = ctypes.c_uint(), ctypes.c_ulonglong()
get_r = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or lib.nvmlDeviceGetCurrentClocksThrottleReasons
if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(c)) == 0:
    print("max", c.value, flush=True)
while True:
    if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(c)) == 0 and get_r(h, ctypes.byref(r)) == 0:
        print(time.time(), c.value, r.value, flush=True)
    time.sleep(0.002)
"""


class ClockSampler:
    """SM clock and throttle-reason samples every 2 ms, read through NVML (the
    library nvidia-smi uses) by a separate process so the sampling does not
    compete with this process for the GIL.  Only samples taken while a timed
    region ran count (mark() brackets each region)."""

    REASONS = {"hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
               "sw_power_cap": 0x4}

    def __init__(self, torch_device: int):
        self.dev = torch_device
        self.proc = None
        self.lines = []
        self.thread = None
        self.windows = []

    def _bus_id(self) -> str:
        props = torch.cuda.get_device_properties(self.dev)
        bus = getattr(props, "pci_bus_id", None)
        if bus is None:
            return ""
        return f"{getattr(props, 'pci_domain_id', 0):08x}:{bus:02x}:{getattr(props, 'pci_device_id', 0):02x}.0"

    def start(self):
        try:
            self.proc = subprocess.Popen([sys.executable, "-c", _SAMPLER, self._bus_id(), str(self.dev)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=lambda: self.lines.extend(ln.strip() for ln in self.proc.stdout),
                                       daemon=True)
        self.thread.start()
        time.sleep(0.3)  # the sampler is up before the timed region starts

    def mark(self, t0: float, t1: float):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["sampler unavailable"], "samples": 0}
        time.sleep(0.01)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        smax, sm, reasons = None, [], set()
        for ln in self.lines:
            f = ln.split()
            if len(f) == 2 and f[0] == "max":
                smax = float(f[1])
            elif len(f) == 3:
                t = float(f[0])
                if self.windows and not any(a - 0.002 <= t <= b + 0.002 for a, b in self.windows):
                    continue
                sm.append(float(f[1]))
                for name, bit in self.REASONS.items():
                    if int(f[2]) & bit:
                        reasons.add(name)
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        return {"sm_mhz": med, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm),
                "source": "nvml, samples inside the timed regions"}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def workload_shape(name: str, batch=None, seq_len=None):
    """(lens, q_counts, hot_frac, description) of a named workload; --batch /
    --seq-len override the sizes of the uniform ones."""
    wl = WORKLOADS[name]
    if wl["kind"] == "uniform":
        B = batch if batch is not None else wl["B"]
        T = seq_len if seq_len is not None else wl["T"]
        desc = (f"MLA decode step, DeepSeek-V2 layer, B={B} sequences x T={T} cached rows, "
                "64-row blocks in a permuted pool, 1 new token per sequence")
        if wl["hot"]:
            desc += f", {wl['hot']:.0%} of cached rows scaled by 8"
        return [T] * B, [1] * B, wl["hot"], desc
    B = wl["B"]
    lens = synth.ragged_lengths(B, wl["lo"], wl["hi"], SEED).tolist()
    qc = synth.query_counts(B, SEED).tolist()
    desc = (f"MLA decode step, DeepSeek-V2 layer, ragged batch B={B}, T_b ~ U[{wl['lo']}, {wl['hi']}] "
            f"(sum {sum(lens)} rows), 1 or 2 new tokens per sequence ({sum(qc)} tokens), "
            "new rows appended by mla_cache_append inside the step")
    return lens, qc, wl["hot"], desc


def make_workload(lens, qc, hot: float, device="cuda"):
    """Weights, a pool holding each sequence's prior rows (T_b - q_b of them),
    and the step's inputs (q_b new tokens per sequence at the last positions)."""
    d = synth.V2
    W = synth.weights(d, SEED, device=device)
    W_dkr = torch.cat([W["W_dkv"], W["W_kr"]], dim=0).contiguous()
    B = len(lens)
    table, n_blocks = synth.block_table(lens, d.block, SEED)
    table = table.to(device)
    pool = torch.empty(n_blocks, d.block, d.width, dtype=torch.bfloat16, device=device)
    flat = pool.view(-1, d.width)
    # prior rows: c ~ N(0,1), k^R ~ N(0,1), the distribution W^DKV h and
    # RoPE(W^KR h) have for h ~ N(0,1), W ~ N(0, 1/fan_in)
    for b in range(B):
        n_prior = int(lens[b]) - int(qc[b])
        for j0 in range(0, n_prior, 65536):
            j1 = min(n_prior, j0 + 65536)
            rows = synth.normal((j1 - j0, d.width), SEED + b, f"prior_rows_{j0}", device=device)
            j = torch.arange(j0, j1, device=device)
            slots = table[b][j // d.block].long() * d.block + (j % d.block)
            flat[slots] = rows
    if hot:
        # a seeded share of each sequence's prior rows scaled by 8 (exact in bf16)
        for b in range(B):
            n_prior = int(lens[b]) - int(qc[b])
            j = synth.pick_rows(n_prior, hot, SEED + b).to(device)
            slots = table[b][j // d.block].long() * d.block + (j % d.block)
            flat[slots] *= 8
    n_tok = int(sum(qc))
    x = synth.hidden(n_tok, d, SEED, name="h_new", device=device)
    seq_idx, pos = [], []
    for b in range(B):
        for k in range(int(qc[b])):
            seq_idx.append(b)
            pos.append(int(lens[b]) - int(qc[b]) + k)
    inp = {
        "x": x,
        "seq_idx": torch.tensor(seq_idx, dtype=torch.int32, device=device),
        "pos": torch.tensor(pos, dtype=torch.int32, device=device),
        "seq_lens": torch.tensor([int(t) for t in lens], dtype=torch.int32, device=device),
        "cu_q": synth.cu_from_counts(qc).to(device),
    }
    return d, W, W_dkr, table, pool, inp


def quantise_pool_q8(pool):
    """Input set-up for the quantised-cache workload, in plain torch: each
    bf16 row [c (512) ; k^R (64)] as 672 bytes -- per run of 32 values of c an
    fp16 scale d = max|x| / 127 and int8 codes round(x / d) (nearest, ties
    away from zero), then the bf16 k^R bytes."""
    d = synth.V2
    flat = pool.view(-1, d.width)
    out = torch.empty(flat.shape[0], Q8_ROW_BYTES, dtype=torch.uint8, device=pool.device)
    for i in range(0, flat.shape[0], 65536):
        j = min(flat.shape[0], i + 65536)
        c = flat[i:j, :d.d_c].float().view(j - i, d.d_c // 32, 32)
        sc = (c.abs().amax(-1) / 127.0).half()
        sf = sc.float().unsqueeze(-1)
        q = torch.where(sf > 0, c / torch.where(sf > 0, sf, torch.ones_like(sf)), torch.zeros_like(c))
        code = (torch.sign(q) * torch.floor(q.abs() + 0.5)).clamp(-127, 127).to(torch.int8)
        out[i:j, :d.d_c] = code.view(j - i, d.d_c).view(torch.uint8)
        out[i:j, d.d_c:d.d_c + 32] = sc.contiguous().view(torch.uint8).view(j - i, 32)
        out[i:j, d.d_c + 32:] = flat[i:j, d.d_c:].contiguous().view(torch.uint8)
    return out.view(pool.shape[0], pool.shape[1], Q8_ROW_BYTES)


def algorithmic(B: int, T: int, d=synth.V2):
    """Bytes and flops the decode kernel must move / do for B sequences of T
    rows with one query token each (one launch)."""
    cache = B * T * d.width * 2
    q = B * d.n_h * d.width * 2
    out = B * d.n_h * d.d_c * 2 + B * d.n_h * 4
    flops = B * d.n_h * T * (2 * d.width + 2 * d.d_c)
    return cache, cache + q + out, flops


def algorithmic_tokens(visible, d=synth.V2, row_bytes=None):
    """The same for query tokens that see `visible[n]` cached rows each: per
    token its rows of cache (row_bytes each; default the bf16 row), its latent
    query read, its o_lat / lse written."""
    rows = int(sum(visible))
    n = len(visible)
    cache = rows * (row_bytes if row_bytes else d.width * 2)
    total = cache + n * d.n_h * d.width * 2 + n * d.n_h * d.d_c * 2 + n * d.n_h * 4
    flops = d.n_h * rows * (2 * d.width + 2 * d.d_c)
    return cache, total, flops


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def _capture(step, n_steps: int, events: bool):
    """A CUDA graph of n_steps calls of step(); with events, a pair of timing
    event nodes around each step's decode call (returned in order)."""
    g = torch.cuda.CUDAGraph()
    pairs = []
    with torch.cuda.graph(g):
        for _ in range(n_steps):
            step(pairs if events else None)
    return g, pairs


def _capture_chunks(step, K: int, events: bool, chunk: int = 256):
    graphs, pairs = [], []
    done = 0
    while done < K:
        n = min(chunk, K - done)
        g, p = _capture(step, n, events)
        graphs.append(g)
        pairs.extend(p)
        done += n
    return graphs, pairs


def _measure(m, step, e2e_step, args, ws: int, local: int) -> dict:
    """Times args.steps steps: captured as CUDA graphs with event nodes
    (step(pairs) appends its events), again without event nodes, and end to
    end (e2e_step: host copies in and out around a step, one graph replay per
    step from the host loop); SM clocks are sampled inside the timed regions."""
    # eager calls first: the library sets kernel attributes, encodes tensor
    # maps and sizes its launches once; the captured calls then do no host work
    step()
    torch.cuda.synchronize()
    m.check()
    warm, _ = _capture(step, max(3, args.warmup), events=False)
    graphs, pairs = _capture_chunks(step, args.steps, events=True)
    for _ in range(2):
        warm.replay()
    torch.cuda.synchronize()
    m.check()

    clocks = ClockSampler(local)
    clocks.start()
    _barrier(ws)
    w0 = time.time()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for g in graphs:
        g.replay()
    t1.record()
    _barrier(ws)
    clocks.mark(w0, time.time())
    m.check()
    ms = t0.elapsed_time(t1) / args.steps
    region_s = ms * args.steps * 1e-3

    # the same steps without event nodes (nothing between the kernels but the
    # stream order): the step time the timing nodes do not perturb
    graphs_plain, _ = _capture_chunks(step, args.steps, events=False)
    _barrier(ws)
    w0 = time.time()
    t0.record()
    for g in graphs_plain:
        g.replay()
    t1.record()
    _barrier(ws)
    clocks.mark(w0, time.time())
    ms_plain = t0.elapsed_time(t1) / args.steps
    del graphs_plain

    g_e2e, _ = _capture(e2e_step, 1, events=False)
    for _ in range(3):
        g_e2e.replay()
    _barrier(ws)
    w0 = time.time()
    t0.record()
    for _ in range(args.steps):
        g_e2e.replay()
    t1.record()
    _barrier(ws)
    clocks.mark(w0, time.time())
    e2e_ms = t0.elapsed_time(t1) / args.steps
    clk = clocks.stop()
    m.check()
    del graphs, warm, g_e2e
    return dict(ms=ms, ms_plain=ms_plain, pairs=pairs, e2e_ms=e2e_ms, clk=clk, region_s=region_s)




def l2_prefetch_setup(m, W, mb: float):
    """Has the decode fetch W^UV and the leading rows of W^O (whole 128-row
    tiles, up to `mb` MB in all) into L2; returns a description and the
    bytes."""
    from head_latent_attention_26_b300 import mla
    ranges = mla.output_weight_prefetch(W["W_uv"], W["W_o"], int(mb * 2**20))
    m.set_decode_l2_prefetch(*ranges)
    return _prefetch_desc(W, ranges), sum(t.numel() * t.element_size() for t in ranges)


def _prefetch_desc(W, ranges):
    if not ranges:
        return "none"
    desc = f"W^UV ({ranges[0].numel() * 2 / 1e6:.1f} MB)"
    if len(ranges) == 2:
        desc += f" and W^O rows 0..{ranges[1].shape[0] - 1} ({ranges[1].numel() * 2 / 1e6:.1f} MB)"
    return desc + " fetched into L2 during the decode for the output projection of the same step"


def run_ours(args):
    ws, rank = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    _init_dist(ws, "nccl")
    from head_latent_attention_26_b300 import build
    build.build()
    from head_latent_attention_26_b300 import mla
    lens, qc, hot, desc = workload_shape(args.workload, args.batch, args.seq_len)
    d, W, W_dkr, table, pool, inp = make_workload(lens, qc, hot)
    B, N = len(lens), int(sum(qc))
    q8 = WORKLOADS[args.workload].get("q8", False)
    if q8:
        pool = quantise_pool_q8(pool)
        desc += "; quantised latent cache (int8 codes of c^KV, fp16 scale per 32 values, bf16 k^R: 672 B per row)"
    m = mla.MLA(d, max(lens) + 64, torch.bfloat16)
    assert m.tensor_path
    bufs = {
        "q_c": torch.empty(N, d.n_h, d.d_h, dtype=torch.bfloat16, device="cuda"),
        "q_r": torch.empty(N, d.n_h, d.d_hr, dtype=torch.bfloat16, device="cuda"),
        "q_lat": torch.empty(N, d.n_h, d.width, dtype=torch.bfloat16, device="cuda"),
        "o_lat": torch.empty(N, d.n_h, d.d_c, dtype=torch.bfloat16, device="cuda"),
        "lse": torch.empty(N, d.n_h, dtype=torch.float32, device="cuda"),
        "u": torch.empty(N, d.d_model, dtype=torch.bfloat16, device="cuda"),
    }
    ws_dec = m.workspace("decode", m.decode_workspace_bytes(N, args.num_workers))
    # the decode streams the cache at about half the HBM rate; the rest
    # fetches the output projection's weights into L2 for the kernel that
    # follows it (by default where that pays: steps of up to 64 tokens)
    pf_mb = args.l2_prefetch_mb if args.l2_prefetch_mb is not None else mla.default_prefetch_bytes(N) / 2**20
    pf_desc, pf_bytes = l2_prefetch_setup(m, W, pf_mb)
    x_dev = torch.empty_like(inp["x"])
    x_dev.copy_(inp["x"])

    def step(pairs=None, x=None):
        x = x_dev if x is None else x
        if pairs is not None:
            ea = torch.cuda.Event(enable_timing=True, external=True)
            ea.record()
        if q8:
            m.q_proj(x, W["W_dq"], W["W_uq"], W["W_qr"], bufs["q_c"], bufs["q_r"])
            m.cache_append_q8(x, W_dkr, inp["seq_idx"], inp["pos"], table, pool)
        else:
            m.q_latent_append(x, W["W_dq"], W["W_uq"], W["W_qr"], W["W_uk"], W_dkr, inp["seq_idx"], inp["pos"],
                              table, pool, bufs["q_lat"])
        if pairs is not None:
            eb = torch.cuda.Event(enable_timing=True, external=True)
            eb.record()
        if q8:
            m.absorb_q(bufs["q_c"], bufs["q_r"], inp["pos"], W["W_uk"], bufs["q_lat"])
        if pairs is not None:
            e0 = torch.cuda.Event(enable_timing=True, external=True)
            e0.record()
        dec = m.decode_q8 if q8 else m.decode
        dec(bufs["q_lat"], pool, table, inp["seq_lens"], inp["cu_q"], args.num_workers, bufs["o_lat"], bufs["lse"],
            ws_dec)
        if pairs is not None:
            e1 = torch.cuda.Event(enable_timing=True, external=True)
            e1.record()
        m.out(bufs["o_lat"], W["W_uv"], W["W_o"], bufs["u"])
        if pairs is not None:
            e2 = torch.cuda.Event(enable_timing=True, external=True)
            e2.record()
            pairs.append((ea, eb, e0, e1, e2))

    # end to end through the public API with host buffers: every step copies
    # its inputs from pinned host memory, runs, and copies u back -- all inside
    # the timed region (one graph replay per step, launched from the host loop)
    h_x = inp["x"].cpu().pin_memory()
    h_pos = inp["pos"].cpu().pin_memory()
    h_lens = inp["seq_lens"].cpu().pin_memory()
    h_u = torch.empty(N, d.d_model, dtype=torch.bfloat16).pin_memory()

    def e2e_step(_=None):
        x_dev.copy_(h_x, non_blocking=True)
        inp["pos"].copy_(h_pos, non_blocking=True)
        inp["seq_lens"].copy_(h_lens, non_blocking=True)
        step()
        h_u.copy_(bufs["u"], non_blocking=True)

    res_t = _measure(m, step, e2e_step, args, ws, local)
    ms, ms_plain, pairs, e2e_ms, clk, region_s = (res_t[k] for k in ("ms", "ms_plain", "pairs", "e2e_ms", "clk",
                                                                       "region_s"))
    # per timed step: the query + append part (the latent query with the
    # cache append; the quantised cache: q_proj and its append), and the decode call (plan +
    # decode + combine), each between event nodes on the step's stream
    app_ms = sum(ea.elapsed_time(eb) for ea, eb, _, _, _ in pairs) / len(pairs)
    dec_ms = sum(e0.elapsed_time(e1) for _, _, e0, e1, _ in pairs) / len(pairs)
    out_ms = sum(e1.elapsed_time(e2) for _, _, _, e1, e2 in pairs) / len(pairs)
    # kernels per step: the latent query with the cache append 2 (W^DQ with
    # the cache rows; W^UQ -> W^UK^T per head with W^QR) -- the quantised
    # cache: q_proj 2, append 2 (the rows, then their codes), absorb 1 --,
    # decode 3 (plan, attention, combine), out 1 (W^UV then W^O)
    n_launch = 9 if q8 else 6

    ms, ms_plain, dec_ms, app_ms, out_ms, e2e_ms = _max_over_ranks([ms, ms_plain, dec_ms, app_ms, out_ms, e2e_ms], ws)
    if rank != 0:
        return None

    hbm, tf_burst, tf_sus, src = _peaks()
    visible = []
    for b in range(B):
        for k in range(int(qc[b])):
            visible.append(int(lens[b]) - int(qc[b]) + k + 1)
    cache_b, dec_bytes, flops = algorithmic_tokens(visible, d, Q8_ROW_BYTES if q8 else None)
    t = dec_ms * 1e-3
    gbs = dec_bytes / t / 1e9
    tflops = flops / t / 1e12
    t_hbm = dec_bytes / (hbm * 1e9)
    bound, t_roof, tc_kind = roofline_choice(t_hbm, flops / (tf_burst * 1e12), flops / (tf_sus * 1e12), region_s)
    tf_peak = tf_sus if tc_kind == "sustained" else tf_burst
    if bound == "tensor":
        roof = {"bound": "tensor", "achieved": round(tflops, 1), "peak": tf_peak, "unit": "TFLOP/s",
                "frac": round(tflops / tf_peak, 4)}
    else:
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4)}
    traffic = args.traffic if args.traffic is not None else (
        None if q8 else _profiled_traffic(B, lens[0] if len(set(lens)) == 1 else -1, pf_bytes))
    roof.update(kernel="decode_tc_kernel<quantised> (+plan, combine)" if q8 else "decode_tc_kernel (+plan, combine)",
                peak_source=f"{src} (MEASURED_PEAKS.json), "
                f"tensor peak {tc_kind} (timed region {region_s * 1e3:.1f} ms)",
                traffic=traffic,
                # the decode launch also reads these bytes for the next kernel (in `traffic`, not in `achieved`)
                l2_prefetch_bytes=pf_bytes,
                other={"hbm": {"achieved_gbs": round(gbs, 1), "peak": hbm, "frac": round(gbs / hbm, 4)},
                       "tensor": {"achieved_tflops": round(tflops, 1), "peak_sustained": tf_sus,
                                  "peak_burst": tf_burst, "frac_sustained": round(tflops / tf_sus, 4),
                                  "frac_burst": round(tflops / tf_burst, 4)}},
                algorithmic_bytes=dec_bytes, algorithmic_flops=flops, decode_us=round(dec_ms * 1e3, 2))
    n = ws
    # the headline: the K steps replayed with nothing between the kernels but
    # the stream order (the event nodes that time each call in the other
    # replay break the kernels' programmatic overlap)
    value = _job_rate(N, n, ms_plain)
    res = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_plain, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": desc, "batch": B, "tokens_per_step": N,
                   "seq_len": lens[0] if len(set(lens)) == 1 else f"U[{min(lens)}, {max(lens)}]",
                   "cached_rows": int(sum(lens)), "num_workers": args.num_workers,
                   "parallelism": f"replicas x{n}" if n > 1 else "single GPU",
                   "l2": f"no flush: every step streams {(298_024_960 + cache_b) / 1e6:.0f} MB of weights and "
                         "cache, more than the 126 MB L2",
                   "l2_prefetch": pf_desc,
                   "timing": "K steps captured as CUDA graphs of the C-ABI calls and replayed, timed by events "
                             "around the replays; the per-call times come from a second capture of the same "
                             "steps with event nodes around each call"},
        "ms_per_step_with_event_nodes": round(ms, 4),
        "latent_cache_gbs": round(cache_b / t / 1e9, 1),
        "decode_tokens_per_s": round(_job_rate(N, n, dec_ms), 1),
        "query_append_us": round(app_ms * 1e3, 2),
        "out_us": round(out_ms * 1e3, 2),
        "roofline": roof,
        "e2e": {"value": round(_job_rate(N, n, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h_x.numel() * 2 + h_pos.numel() * 4 + h_lens.numel() * 4,
                "d2h_bytes_per_step": h_u.numel() * 2},
        "gpu_launches": n_launch * args.steps,
        "clocks": clk,
    }
    if WORKLOADS[args.workload]["kind"] == "ragged":
        # the pool's valid rows: every sequence's T_b rows, (d_c + d_hr) bf16 values each
        res["cache_bytes"] = {"valid": int(sum(lens)) * d.width * 2,
                              "formula": "(d_c + d_hr) * sum(T) * 2",
                              "pool_bytes": pool.numel() * 2}
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(lens, qc, args.workload, budget_s=args.cpu_budget)
    return res


def prefill_work(P: int, d=synth.V2):
    """Algorithmic flops and bytes of one prefill call for a P-token prompt
    (positions 0..P-1): the K^C and V expansion (two products of P x d_c by
    d_c x n_h d_h) and the causal attention (per head sum_t (t+1) keys, each
    a 192-wide score and a 128-wide weighted sum); bytes = the rows, query
    parts and the two weights read, K^C and V written and read once, o and
    lse written."""
    hd = d.n_h * d.d_h
    f_exp = 2 * 2 * P * hd * d.d_c
    f_att = d.n_h * (P * (P + 1) // 2) * (2 * (d.d_h + d.d_hr) + 2 * d.d_h)
    byt = (P * d.width * 2 + P * hd * 2 + P * d.n_h * d.d_hr * 2 + 2 * hd * d.d_c * 2
           + 2 * (2 * P * hd * 2) + P * hd * 2 + P * d.n_h * 4)
    return f_exp + f_att, byt, f_exp, f_att


def run_prefill(args):
    """A P-token prompt: mla_q_proj, mla_cache_append (rows in position
    order), mla_prefill (K^C / V expansion + causal attention); events around
    the prefill call."""
    ws, rank = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    _init_dist(ws, "nccl")
    from head_latent_attention_26_b300 import build
    build.build()
    from head_latent_attention_26_b300 import mla
    P = args.seq_len if args.seq_len is not None else WORKLOADS[args.workload]["P"]
    d = synth.V2
    W = synth.weights(d, SEED, device="cuda")
    W_dkr = torch.cat([W["W_dkv"], W["W_kr"]], dim=0).contiguous()
    x_dev = synth.hidden(P, d, SEED, name="h_prompt", device="cuda")
    m = mla.MLA(d, P + 64, torch.bfloat16)
    assert m.tensor_path
    n_blocks = (P + d.block - 1) // d.block
    table = torch.arange(n_blocks, dtype=torch.int32, device="cuda").view(1, -1)
    pool = torch.empty(n_blocks, d.block, d.width, dtype=torch.bfloat16, device="cuda")
    rows = pool.view(-1, d.width)[:P]
    seq_idx = torch.zeros(P, dtype=torch.int32, device="cuda")
    pos = torch.arange(P, dtype=torch.int32, device="cuda")
    q_c = torch.empty(P, d.n_h, d.d_h, dtype=torch.bfloat16, device="cuda")
    q_r = torch.empty(P, d.n_h, d.d_hr, dtype=torch.bfloat16, device="cuda")
    o = torch.empty(P, d.n_h, d.d_h, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(P, d.n_h, dtype=torch.float32, device="cuda")

    def step(pairs=None):
        m.q_proj(x_dev, W["W_dq"], W["W_uq"], W["W_qr"], q_c, q_r)
        m.cache_append(x_dev, W_dkr, seq_idx, pos, table, pool)
        if pairs is not None:
            e0 = torch.cuda.Event(enable_timing=True, external=True)
            e0.record()
        m.prefill(rows, q_c, q_r, W["W_uk"], W["W_uv"], o, lse)
        if pairs is not None:
            e1 = torch.cuda.Event(enable_timing=True, external=True)
            e1.record()
            pairs.append((e0, e1))

    h_x = x_dev.cpu().pin_memory()
    h_o = torch.empty(P, d.n_h, d.d_h, dtype=torch.bfloat16).pin_memory()

    def e2e_step(_=None):
        x_dev.copy_(h_x, non_blocking=True)
        step()
        h_o.copy_(o, non_blocking=True)

    res_t = _measure(m, step, e2e_step, args, ws, local)
    pre_ms = sum(e0.elapsed_time(e1) for e0, e1 in res_t["pairs"]) / len(res_t["pairs"])
    ms, ms_plain, pre_ms, e2e_ms = _max_over_ranks([res_t["ms"], res_t["ms_plain"], pre_ms, res_t["e2e_ms"]], ws)
    if rank != 0:
        return None
    hbm, tf_burst, tf_sus, src = _peaks()
    flops, byt, f_exp, f_att = prefill_work(P, d)
    t = pre_ms * 1e-3
    bound, t_roof, tc_kind = roofline_choice(byt / (hbm * 1e9), flops / (tf_burst * 1e12), flops / (tf_sus * 1e12),
                                             res_t["region_s"])
    tf_peak = tf_sus if tc_kind == "sustained" else tf_burst
    if bound == "tensor":
        roof = {"bound": "tensor", "achieved": round(flops / t / 1e12, 1), "peak": tf_peak, "unit": "TFLOP/s",
                "frac": round(flops / t / 1e12 / tf_peak, 4)}
    else:
        roof = {"bound": "hbm", "achieved": round(byt / t / 1e9, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(byt / t / 1e9 / hbm, 4)}
    roof.update(kernel="mla_prefill (expansion GEMM + prefill_attn_kernel)", traffic=None,
                peak_source=f"{src} (MEASURED_PEAKS.json), tensor peak {tc_kind} (fp16 operands, the bf16 rate)",
                algorithmic_flops=flops, algorithmic_bytes=byt, expansion_flops=f_exp, attention_flops=f_att,
                prefill_us=round(pre_ms * 1e3, 2))
    n = ws
    res = {
        "metric": METRIC,
        "value": round(_job_rate(P, n, ms_plain), 1),
        "unit": "tokens/s",
        "n_gpus": n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_plain, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"MLA prefill, DeepSeek-V2 layer, one prompt of P={P} tokens (positions 0..P-1): "
                               "query projection, cache rows, K^C / V expansion and causal attention",
                   "batch": 1, "tokens_per_step": P, "seq_len": P,
                   "parallelism": f"replicas x{n}" if n > 1 else "single GPU",
                   "l2": "no flush: the step writes and reads the expanded K^C and V "
                         f"({2 * P * d.n_h * d.d_h * 2 / 1e6:.0f} MB), more than the 126 MB L2",
                   "timing": "K steps captured as CUDA graphs of the C-ABI calls and replayed, timed by events "
                             "around the replays; the prefill call's time comes from a second capture of the "
                             "same steps with event nodes around it"},
        "ms_per_step_with_event_nodes": round(ms, 4),
        "prefill_tokens_per_s": round(_job_rate(P, n, pre_ms), 1),
        "roofline": roof,
        "e2e": {"value": round(_job_rate(P, n, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h_x.numel() * 2, "d2h_bytes_per_step": h_o.numel() * 2},
        # q_proj 2, append 1, prefill 2 (expansion, attention)
        "gpu_launches": 5 * args.steps,
        "clocks": res_t["clk"],
    }
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline_prefill(P, args.cpu_budget)
    return res


# ---------------------------------------------------------------------------
# oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

def _oracle_inputs(B: int):
    """Weights and new-token states for the oracle legs, drawn on the host
    (same recipe and seeds; the host generator's values differ from the
    device generator's, which does not matter for timing)."""
    import oracle as O
    d = synth.V2
    W = synth.weights(d, SEED, device="cpu")
    return {k: O.f64(v) for k, v in W.items()}, synth.hidden(B, d, SEED, name="h_new", device="cpu")


def _prior_rows(B: int, T: int, b: int):
    """T - 1 prior rows of sequence b (the recipe of make_workload)."""
    d = synth.V2
    parts = [synth.normal((min(T - 1, j0 + 65536) - j0, d.width), SEED + b, f"prior_rows_{j0}", device="cpu")
             for j0 in range(0, max(T - 1, 1), 65536)]
    return torch.cat(parts)[:T - 1]


def _oracle_token(Wn, x, rows_bf16, T: int, b: int):
    """The oracle, as it stands, for one new token at position T - 1 after
    T - 1 cached rows: its cache row, query, expanded K/V over the T rows,
    softmax, W^O.  Returns u."""
    import numpy as np
    import oracle as O
    d = synth.V2
    rows = O.f64(rows_bf16)
    xb = O.f64(x[b % x.shape[0]:b % x.shape[0] + 1])
    c_new, kr_new = O.kv_latent(xb, Wn["W_dkv"], Wn["W_kr"], [T - 1], d.rope_base)
    c = np.concatenate([rows[:T - 1, :d.d_c], c_new])
    k_r = np.concatenate([rows[:T - 1, d.d_c:], kr_new])
    _, q_c, q_r_raw = O.query_parts(xb, Wn["W_dq"], Wn["W_uq"], Wn["W_qr"], d.n_h)
    o, _ = O.attend_expanded(q_c[0], O.rope(q_r_raw[0], T - 1, d.rope_base), c, k_r, Wn["W_uk"], Wn["W_uv"])
    return O.output_projection(o, Wn["W_o"])


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:  # noqa: BLE001
        return os.cpu_count() or 1


def _token_list(lens, qc):
    """(sequence, visible rows) of every query token, in token order."""
    out = []
    for b, (L, q) in enumerate(zip(lens, qc)):
        for k in range(int(q)):
            out.append((b, int(L) - int(q) + k + 1))
    return out


def cpu_baseline(lens, qc, workload: str, budget_s: float = 15.0):
    """Time the fp64 oracle on whole tokens of the workload until budget_s of
    oracle arithmetic has run (input generation is outside the timer)."""
    t_start = time.perf_counter()
    toks = _token_list(lens, qc)
    Wn, x = _oracle_inputs(len(toks))
    done, elapsed = 0, 0.0
    while done < len(toks) and (done == 0 or elapsed < budget_s):
        b, T = toks[done]
        rows = _prior_rows(len(lens), T, b)
        t0 = time.perf_counter()
        _oracle_token(Wn, x, rows, T, done)
        elapsed += time.perf_counter() - t0
        done += 1
    return {"value": round(done / elapsed, 4), "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{done} of {len(toks)} tokens of the {workload} workload (expanded K/V, fp64 numpy), "
                      f"{elapsed:.1f} s of oracle time; input generation untimed",
            "wall_s": round(time.perf_counter() - t_start, 1)}


def _oracle_prefill(Wn, h_bf16):
    """The oracle's prefill of a prompt (cache rows and query parts from h,
    expanded K/V, causal attention); the output projection is left out, as
    in the GPU prefill call."""
    import oracle as O
    d = synth.V2
    return O.prefill_expanded(O.f64(h_bf16), Wn, n_h=d.n_h, base=d.rope_base, with_u=False)


def _prefill_sample(P: int, budget_s: float):
    """The oracle's prefill of the largest power-of-two prompt prefix (64
    tokens up to P) that fits budget_s: prefixes double while four times the
    last one's time (an upper bound on the doubled prefix's, whose work grows
    at most with the square) stays within the budget.  Returns the weights,
    the prompt, the prefix length and its time."""
    Wn, _ = _oracle_inputs(1)
    h = synth.hidden(P, synth.V2, SEED, name="h_prompt", device="cpu")
    n = min(64, P)
    t0 = time.perf_counter()
    _oracle_prefill(Wn, h[:n])
    el = time.perf_counter() - t0
    while 2 * n <= P and 4 * el <= budget_s:
        n *= 2
        t0 = time.perf_counter()
        _oracle_prefill(Wn, h[:n])
        el = time.perf_counter() - t0
    return Wn, h, n, el


def cpu_baseline_prefill(P: int, budget_s: float = 15.0):
    t_start = time.perf_counter()
    _, _, n, el = _prefill_sample(P, budget_s)
    return {"value": round(n / el, 4), "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
            "sample": f"the first {n} of the {P} prompt tokens through the oracle's prefill (expanded K/V, fp64 "
                      f"numpy; attention cost grows with the prefix's square, so this rate is above the full "
                      f"prompt's), {el:.1f} s of oracle time",
            "wall_s": round(time.perf_counter() - t_start, 1)}


def run_reference_prefill(args):
    P = args.seq_len if args.seq_len is not None else WORKLOADS[args.workload]["P"]
    Wn, h, n, _ = _prefill_sample(P, max(1.0, args.cpu_budget / max(1, args.steps)))
    total = 0.0
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        _oracle_prefill(Wn, h[:n])
        if s >= args.warmup:
            total += time.perf_counter() - t0
    v = n * args.steps / total
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "tokens/s", "n_gpus": _dist()[0],
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"MLA prefill, one prompt of P={P} tokens", "batch": 1, "tokens_per_step": P,
                   "seq_len": P},
        "cpu_baseline": {"value": round(v, 4), "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
                         "sample": f"each step = the oracle's prefill of the first {n} of the {P} prompt tokens"},
        "e2e": {"value": round(v, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference(args):
    ws, rank = _dist()
    if rank != 0:
        return None
    if WORKLOADS[args.workload]["kind"] == "prefill":
        return run_reference_prefill(args)
    lens, qc, _, desc = workload_shape(args.workload, args.batch, args.seq_len)
    toks = _token_list(lens, qc)
    B = len(toks)
    Wn, x = _oracle_inputs(B)
    total_s = 0.0
    for s in range(args.warmup + args.steps):
        b, T = toks[s % B]
        rows = _prior_rows(len(lens), T, b)
        t0 = time.perf_counter()
        _oracle_token(Wn, x, rows, T, s % B)
        if s >= args.warmup:
            total_s += time.perf_counter() - t0
    v = args.steps / total_s
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(v, 4),
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_s / args.steps * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": desc, "batch": len(lens), "tokens_per_step": B,
                   "seq_len": lens[0] if len(set(lens)) == 1 else f"U[{min(lens)}, {max(lens)}]"},
        "cpu_baseline": {"value": round(v, 4), "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
                         "sample": f"each step = 1 of the {B} tokens of the workload through the fp64 oracle "
                                   "(expanded K/V); input generation untimed"},
        "e2e": {"value": round(v, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="b64_t4096")
    ap.add_argument("--batch", type=int, default=None, help="override B of a uniform workload")
    ap.add_argument("--seq-len", type=int, default=None, help="override T of a uniform workload")
    ap.add_argument("--num-workers", type=int, default=0)
    ap.add_argument("--l2-prefetch-mb", type=float, default=None,
                    help="W^UV and leading W^O rows the decode fetches into L2 for the output projection "
                         "(0 = none; default: 96 MiB for steps of up to 64 tokens, else none)")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per decode launch from an ncu capture of this kernel version")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        res = run_reference(args)
    elif WORKLOADS[args.workload]["kind"] == "prefill":
        res = run_prefill(args)
    else:
        res = run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
