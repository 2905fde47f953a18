"""One rank of the multi-rank bench check (run by tests/test_multirank.py
under torch.distributed.run with the gloo backend, no GPU).

Exercises the host side of bench.py's N>1 path: joining the group, the
barrier, the max-over-ranks reduction of step times, the whole-job rate, and
the reference arm's rank-0-only rule.  The oracle legs are replaced by
counting stubs so no rank does oracle arithmetic; the test checks which rank
called them.  Writes its findings to $MULTIRANK_OUT/rank<r>.json."""

from __future__ import annotations

import contextlib
import io
import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def main():
    ws, rank = bench._dist()
    bench._init_dist(ws, "gloo")
    bench._barrier(ws, cuda=False)
    # per-rank "step times": rank r is slower on the first entry, faster on the second
    mx = bench._max_over_ranks([1.0 + rank, 4.0 - rank, 2.5], ws, device="cpu")
    rate = bench._job_rate(64, ws, mx[0])

    calls = []
    bench._oracle_inputs = lambda B: (calls.append("inputs"), ({}, None))[1]
    bench._prior_rows = lambda B, T, b: calls.append("rows")

    def token(Wn, x, rows, T, b):
        calls.append("token")
        time.sleep(0.002)

    bench._oracle_token = token
    out = io.StringIO()
    argv = sys.argv
    sys.argv = ["bench.py", "--impl", "reference", "--gpus", str(ws), "--steps", "3", "--warmup", "3",
                "--batch", "4", "--seq-len", "64"]
    with contextlib.redirect_stdout(out):
        bench.main()
    sys.argv = argv
    bench._barrier(ws, cuda=False)

    with open(os.path.join(os.environ["MULTIRANK_OUT"], f"rank{rank}.json"), "w") as f:
        json.dump({"rank": rank, "world_size": ws, "max": mx, "rate": rate, "calls": calls,
                   "stdout": out.getvalue()}, f)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
