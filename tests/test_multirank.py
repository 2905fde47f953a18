"""Host side of the bench's multi-rank path on CPU: two gloo ranks launched by
torch.distributed.run on 127.0.0.1 (no GPU, no oracle arithmetic)."""

from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(n: int, out_dir: str):
    env = dict(os.environ, MULTIRANK_OUT=out_dir, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "tests", "_multirank_worker.py")]
    r = subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=240)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    res = []
    for k in range(n):
        with open(os.path.join(out_dir, f"rank{k}.json")) as f:
            res.append(json.load(f))
    return res


@pytest.fixture(scope="module")
def two_ranks(tmp_path_factory):
    return _launch(2, str(tmp_path_factory.mktemp("multirank")))


def test_max_over_ranks(two_ranks):
    # rank r reported [1 + r, 4 - r, 2.5]: every rank must hold the element-wise max
    for r in two_ranks:
        assert r["world_size"] == 2
        assert r["max"] == [2.0, 4.0, 2.5]


def test_whole_job_rate(two_ranks):
    # 64 tokens per rank, 2 ranks, slowest rank 2 ms per step
    for r in two_ranks:
        assert r["rate"] == pytest.approx(64 * 2 / 2.0e-3)


def test_reference_arm_rank0_only(two_ranks):
    r0, r1 = sorted(two_ranks, key=lambda r: r["rank"])
    # rank 1 exits without work and prints nothing
    assert r1["calls"] == [] and r1["stdout"] == ""
    # rank 0 draws the inputs once and runs warm-up + timed tokens through the oracle legs
    assert r0["calls"] == ["inputs"] + ["rows", "token"] * 6
    lines = [ln for ln in r0["stdout"].splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 3
    assert line["warmup"] == 3 and line["higher_is_better"] is True
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    # 3 timed tokens of at least 2 ms each
    assert 0 < line["value"] <= 1 / 2e-3


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    bench._init_dist(1)  # no group at N=1
    assert bench._max_over_ranks([3.0, 1.0], 1, device="cpu") == [3.0, 1.0]
    assert bench._job_rate(64, 1, 0.25) == pytest.approx(256000.0)
