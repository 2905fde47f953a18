"""Host-side arithmetic of bench.py, on CPU: the roofline's algorithmic work
and the profiled-traffic guard."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_algorithmic_work_b64_t4096():
    # [kasblo] "容量を計算する": d_c + d_h^R = 576 bf16 values per cached token;
    # 64 sequences x 4096 rows
    cache, total, flops = bench.algorithmic(64, 4096)
    assert cache == 64 * 4096 * 576 * 2 == 301_989_888
    # plus the latent queries read once and o_lat (bf16) + lse (fp32) written
    assert total == cache + 64 * 128 * 576 * 2 + 64 * 128 * 512 * 2 + 64 * 128 * 4
    # per (token, head, key): a 576-wide score dot and a 512-wide value update
    assert flops == 64 * 128 * 4096 * (2 * 576 + 2 * 512) == 73_014_444_032


def test_algorithmic_work_scales_linearly():
    c1, t1, f1 = bench.algorithmic(1, 4096)
    c2, t2, f2 = bench.algorithmic(2, 8192)
    assert c2 == 4 * c1 and f2 == 4 * f1
    assert bench.algorithmic(1, 131072)[0] == 131072 * 1152


def test_profiled_traffic_guard():
    # the capture's traffic is reported only for its workload, L2 prefetch and sources
    pf = bench.PROFILED_DECODE["l2_prefetch_bytes"]
    assert bench._profiled_traffic(64, 2048, pf) is None
    assert bench._profiled_traffic(64, 4096, pf + 16) is None
    t = bench._profiled_traffic(64, 4096, pf)
    assert t is None or t == bench.PROFILED_DECODE["traffic_bytes"]
    # within a few percent of the algorithmic bytes plus the prefetched ones:
    # the cache is read once
    _, total, _ = bench.algorithmic(64, 4096)
    assert abs(bench.PROFILED_DECODE["traffic_bytes"] / (total + pf) - 1) < 0.03


@pytest.mark.parametrize("units,ws,ms,expect", [(64, 1, 0.2, 320000.0), (64, 4, 0.25, 1024000.0)])
def test_job_rate(units, ws, ms, expect):
    assert bench._job_rate(units, ws, ms) == pytest.approx(expect)
