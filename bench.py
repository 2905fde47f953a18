"""Benchmark of one MLA decode step on B300.

Workload (default): DeepSeek-V2 attention layer (d=5120, n_h=128, d_h=128,
d_h^R=64, d_c=512, d_c'=1536), batched decode B=64 sequences of T=4096 cached
rows each, one new token per sequence, 64-row cache blocks scattered over a
seeded random permutation of the pool.  One step = the whole path for the 64
new tokens: query projection, cache append, W^UK absorption, latent attention
(+ split combine), W^UV / W^O output.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  Under torchrun every rank runs an independent replica
on its own GPU (the path has no exchange step); the time is the max over ranks.
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

# DRAM bytes (read + write) of one decode_tc_kernel launch on this workload,
# from the ncu capture summarised in profiles/decode_tc_kernel_b64_t4096.md;
# valid only while the kernel sources hash to the captured ones.
PROFILED_DECODE = {"sources": {"decode_tc.cu": "661b9209bf3c159d", "ptx.cuh": "1fd1dc657a7fe061"},
                   "workload": (64, 4096), "traffic_bytes": 314375168}


def _profiled_traffic(B: int, T: int):
    import hashlib
    if (B, T) != PROFILED_DECODE["workload"]:
        return None
    csrc = os.path.join(ROOT, "head_latent_attention_26_b300", "csrc")
    for name, digest in PROFILED_DECODE["sources"].items():
        with open(os.path.join(csrc, name), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != digest:
                return None
    return PROFILED_DECODE["traffic_bytes"]
B_DEFAULT, T_DEFAULT = 64, 4096
SEED = 1003


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
        print(c.value, r.value, flush=True)
    time.sleep(0.005)
"""


class ClockSampler:
    """SM clock and throttle-reason samples every 5 ms while the timed region
    runs, read through NVML (the library nvidia-smi uses) by a separate
    process so the sampling does not compete with this process for the GIL."""

    REASONS = {"hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
               "sw_power_cap": 0x4}

    def __init__(self, torch_device: int):
        self.dev = torch_device
        self.proc = None
        self.lines = []
        self.thread = None

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

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["sampler unavailable"], "samples": 0}
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
            elif len(f) == 2:
                sm.append(float(f[0]))
                for name, bit in self.REASONS.items():
                    if int(f[1]) & bit:
                        reasons.add(name)
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        return {"sm_mhz": med, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm), "source": "nvml"}


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------

def make_workload(B: int, T: int, device="cuda"):
    """Weights, a pool holding T-1 prior rows per sequence, and the step's inputs."""
    d = synth.V2
    W = synth.weights(d, SEED, device=device)
    W_dkr = torch.cat([W["W_dkv"], W["W_kr"]], dim=0).contiguous()
    lens = [T] * B
    table, n_blocks = synth.block_table(lens, d.block, SEED)
    table = table.to(device)
    pool = torch.empty(n_blocks, d.block, d.width, dtype=torch.bfloat16, device=device)
    flat = pool.view(-1, d.width)
    # prior rows: c ~ N(0,1), k^R ~ N(0,1), the distribution W^DKV h and RoPE(W^KR h)
    # have for h ~ N(0,1), W ~ N(0, 1/fan_in)
    for b0 in range(0, B, 8):
        nb = min(8, B - b0)
        rows = synth.normal((nb * T, d.width), SEED + b0, "prior_rows", device=device)
        j = torch.arange(T, device=device)
        for k in range(nb):
            slots = table[b0 + k][j // d.block].long() * d.block + (j % d.block)
            flat[slots] = rows[k * T:(k + 1) * T]
        del rows
    x = synth.hidden(B, d, SEED, name="h_new", device=device)
    inp = {
        "x": x,
        "seq_idx": torch.arange(B, dtype=torch.int32, device=device),
        "pos": torch.full((B,), T - 1, dtype=torch.int32, device=device),
        "seq_lens": torch.full((B,), T, dtype=torch.int32, device=device),
        "cu_q": torch.arange(B + 1, dtype=torch.int32, device=device),
    }
    return d, W, W_dkr, table, pool, inp


def algorithmic(B: int, T: int, d=synth.V2):
    """Bytes and flops the decode kernel must move / do (one launch)."""
    cache = B * T * d.width * 2
    q = B * d.n_h * d.width * 2
    out = B * d.n_h * d.d_c * 2 + B * d.n_h * 4
    flops = B * d.n_h * T * (2 * d.width + 2 * d.d_c)
    return cache, cache + q + out, flops


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    ws, rank = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    _init_dist(ws, "nccl")
    from head_latent_attention_26_b300 import build
    build.build()
    from head_latent_attention_26_b300 import mla
    B, T = args.batch, args.seq_len
    d, W, W_dkr, table, pool, inp = make_workload(B, T)
    m = mla.MLA(d, T + 64, torch.bfloat16)
    assert m.tensor_path
    bufs = {
        "q_c": torch.empty(B, d.n_h, d.d_h, dtype=torch.bfloat16, device="cuda"),
        "q_r": torch.empty(B, d.n_h, d.d_hr, dtype=torch.bfloat16, device="cuda"),
        "q_lat": torch.empty(B, d.n_h, d.width, dtype=torch.bfloat16, device="cuda"),
        "o_lat": torch.empty(B, d.n_h, d.d_c, dtype=torch.bfloat16, device="cuda"),
        "lse": torch.empty(B, d.n_h, dtype=torch.float32, device="cuda"),
        "u": torch.empty(B, d.d_model, dtype=torch.bfloat16, device="cuda"),
    }
    ws_dec = m.workspace("decode", m.decode_workspace_bytes(B, args.num_workers))
    dec_ev = []

    def step(x, time_decode=False):
        m.q_proj(x, W["W_dq"], W["W_uq"], W["W_qr"], bufs["q_c"], bufs["q_r"])
        m.cache_append(x, W_dkr, inp["seq_idx"], inp["pos"], table, pool)
        m.absorb_q(bufs["q_c"], bufs["q_r"], inp["pos"], W["W_uk"], bufs["q_lat"])
        if time_decode:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
        m.decode(bufs["q_lat"], pool, table, inp["seq_lens"], inp["cu_q"], args.num_workers, bufs["o_lat"],
                 bufs["lse"], ws_dec)
        if time_decode:
            e1.record()
            dec_ev.append((e0, e1))
        m.out(bufs["o_lat"], W["W_uv"], W["W_o"], bufs["u"])

    for _ in range(args.warmup):
        step(inp["x"])
    m.check()

    def barrier():
        _barrier(ws)

    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        step(inp["x"], time_decode=True)
    t1.record()
    barrier()
    clk = clocks.stop()
    m.check()
    ms = t0.elapsed_time(t1) / args.steps
    dec_ms = sum(a.elapsed_time(b) for a, b in dec_ev) / len(dec_ev)
    launches_per_step = 2 + 1 + 1 + 3 + 2  # q_proj (W^DQ; W^UQ and W^QR fused), append, absorb, plan+decode+combine, out

    # end to end through the public API with host buffers: H2D of the step's
    # inputs, the step, D2H of u -- all inside the timed region
    h_x = inp["x"].cpu().pin_memory()
    h_pos = inp["pos"].cpu().pin_memory()
    h_lens = inp["seq_lens"].cpu().pin_memory()
    h_u = torch.empty(B, d.d_model, dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(inp["x"])
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        x_dev.copy_(h_x, non_blocking=True)
        inp["pos"].copy_(h_pos, non_blocking=True)
        inp["seq_lens"].copy_(h_lens, non_blocking=True)
        step(x_dev)
        h_u.copy_(bufs["u"], non_blocking=True)
    e1.record()
    barrier()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    m.check()

    # the two routes to the latent query for the same tokens: runtime
    # absorption (q_proj + absorb_q, the step above) and the folded weight
    # W^UK_i^T W^UQ_i formed once ahead of time (q_proj_absorbed)
    W_abs = m.absorb_weights(W["W_uq"], W["W_uk"])
    q_lat_f = torch.empty_like(bufs["q_lat"])
    n_q = max(3, min(args.steps, 300))

    def time_route(fn):
        for _ in range(3):
            fn()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n_q):
            fn()
        b.record()
        barrier()
        return a.elapsed_time(b) / n_q

    def runtime_route():
        m.q_proj(inp["x"], W["W_dq"], W["W_uq"], W["W_qr"], bufs["q_c"], bufs["q_r"])
        m.absorb_q(bufs["q_c"], bufs["q_r"], inp["pos"], W["W_uk"], bufs["q_lat"])

    rt_ms = time_route(runtime_route)
    fold_ms = time_route(lambda: m.q_proj_absorbed(inp["x"], W["W_dq"], W_abs, W["W_qr"], inp["pos"], q_lat_f))
    m.check()
    del W_abs
    ms, dec_ms, e2e_ms, rt_ms, fold_ms = _max_over_ranks([ms, dec_ms, e2e_ms, rt_ms, fold_ms], ws)
    if rank != 0:
        return None

    hbm, tf_burst, tf_sus, src = _peaks()
    cache_b, dec_bytes, flops = algorithmic(B, T, d)
    t = dec_ms * 1e-3
    gbs = dec_bytes / t / 1e9
    tflops = flops / t / 1e12
    # binding roofline of the decode kernel: the slower of HBM and tensor at the
    # measured peaks (sustained tensor peak: the kernel runs inside a long loop)
    t_hbm, t_tc = dec_bytes / (hbm * 1e9), flops / (tf_sus * 1e12)
    if t_tc >= t_hbm:
        roof = {"bound": "tensor", "achieved": round(tflops, 1), "peak": tf_sus, "unit": "TFLOP/s",
                "frac": round(tflops / tf_sus, 4)}
    else:
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4)}
    roof.update(kernel="decode_tc_kernel (+plan, combine)", peak_source=f"{src} (MEASURED_PEAKS.json)",
                traffic=args.traffic if args.traffic is not None else _profiled_traffic(B, T), other={"hbm": {"achieved_gbs": round(gbs, 1), "peak": hbm,
                                                     "frac": round(gbs / hbm, 4)},
                                             "tensor": {"achieved_tflops": round(tflops, 1),
                                                        "peak_sustained": tf_sus, "peak_burst": tf_burst,
                                                        "frac_sustained": round(tflops / tf_sus, 4),
                                                        "frac_burst": round(tflops / tf_burst, 4)}},
                algorithmic_bytes=dec_bytes, algorithmic_flops=flops, decode_us=round(dec_ms * 1e3, 2))
    n = ws
    value = _job_rate(B, n, ms)
    res = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"MLA decode step, DeepSeek-V2 layer, B={B} sequences x T={T} cached rows, "
                               "64-row blocks in a permuted pool, 1 new token per sequence",
                   "batch": B, "seq_len": T, "num_workers": args.num_workers,
                   "parallelism": f"replicas x{n}" if n > 1 else "single GPU",
                   "l2": "no flush: the step reads > L2 (302 MB cache + 300 MB weights)"},
        "latent_cache_gbs": round(cache_b / t / 1e9, 1),
        "decode_tokens_per_s": round(_job_rate(B, n, dec_ms), 1),
        "roofline": roof,
        "e2e": {"value": round(_job_rate(B, n, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h_x.numel() * 2 + h_pos.numel() * 4 + h_lens.numel() * 4,
                "d2h_bytes_per_step": h_u.numel() * 2},
        "query_routes": {"runtime_absorb_us": round(rt_ms * 1e3, 2), "folded_weight_us": round(fold_ms * 1e3, 2),
                         "weight_bytes": {"runtime": 2 * d.d_cq * (d.d_model + d.n_h * (d.d_h + d.d_hr))
                                          + 2 * d.n_h * d.d_h * d.d_c,
                                          "folded": 2 * d.d_cq * (d.d_model + d.n_h * (d.d_c + d.d_hr))},
                         "note": "W^DQ, W^UQ + W^QR, W^UK absorb (runtime) vs W^DQ, folded W^UK_i^T W^UQ_i + W^QR "
                                 f"(one launch), {n_q} back-to-back calls each, outside the timed step"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(B, T, budget_s=args.cpu_budget)
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
    d = synth.V2
    b0 = (b // 8) * 8
    g = synth.normal((min(8, B - b0) * T, d.width), SEED + b0, "prior_rows", device="cpu")
    return g[(b - b0) * T:(b - b0 + 1) * T]


def _oracle_token(Wn, x, rows_bf16, T: int, b: int):
    """The oracle, as it stands, for token b of the workload: its cache row,
    query, expanded K/V over the sequence's T rows, softmax, W^O.  Returns u."""
    import numpy as np
    import oracle as O
    d = synth.V2
    rows = O.f64(rows_bf16)
    c_new, kr_new = O.kv_latent(O.f64(x[b:b + 1]), Wn["W_dkv"], Wn["W_kr"], [T - 1], d.rope_base)
    c = np.concatenate([rows[:T - 1, :d.d_c], c_new])
    k_r = np.concatenate([rows[:T - 1, d.d_c:], kr_new])
    _, q_c, q_r_raw = O.query_parts(O.f64(x[b:b + 1]), Wn["W_dq"], Wn["W_uq"], Wn["W_qr"], d.n_h)
    o, _ = O.attend_expanded(q_c[0], O.rope(q_r_raw[0], T - 1, d.rope_base), c, k_r, Wn["W_uk"], Wn["W_uv"])
    return O.output_projection(o, Wn["W_o"])


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:  # noqa: BLE001
        return os.cpu_count() or 1


def cpu_baseline(B: int, T: int, budget_s: float = 15.0):
    """Time the fp64 oracle on whole tokens of the workload until budget_s of
    oracle arithmetic has run (input generation is outside the timer)."""
    t_start = time.perf_counter()
    Wn, x = _oracle_inputs(B)
    done, elapsed = 0, 0.0
    while done < B and (done == 0 or elapsed < budget_s):
        rows = _prior_rows(B, T, done)
        t0 = time.perf_counter()
        _oracle_token(Wn, x, rows, T, done)
        elapsed += time.perf_counter() - t0
        done += 1
    return {"value": round(done / elapsed, 4), "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{done} of {B} tokens of the B={B}, T={T} workload (expanded K/V, fp64 numpy), "
                      f"{elapsed:.1f} s of oracle time; input generation untimed",
            "wall_s": round(time.perf_counter() - t_start, 1)}


def run_reference(args):
    ws, rank = _dist()
    if rank != 0:
        return None
    B, T = args.batch, args.seq_len
    Wn, x = _oracle_inputs(B)
    total_s = 0.0
    for s in range(args.warmup + args.steps):
        rows = _prior_rows(B, T, s % B)
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
        "config": {"workload": f"MLA decode step, DeepSeek-V2 layer, B={B} sequences x T={T} cached rows, "
                               "64-row blocks in a permuted pool, 1 new token per sequence",
                   "batch": B, "seq_len": T},
        "cpu_baseline": {"value": round(v, 4), "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
                         "sample": f"each step = 1 of the B={B} tokens through the fp64 oracle "
                                   "(expanded K/V); input generation untimed"},
        "e2e": {"value": round(v, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--batch", type=int, default=B_DEFAULT)
    ap.add_argument("--seq-len", type=int, default=T_DEFAULT)
    ap.add_argument("--num-workers", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per decode launch from an ncu capture of this kernel version")
    args = ap.parse_args()
    if args.impl == "reference":
        res = run_reference(args)
    else:
        res = run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
