"""Host logic of the multi-GPU bench path on CPU: two `gloo` ranks.

Each rank runs its own independent batch (weak scaling, no data-path
collective): the batches have the same shapes and differ in content; the
step time reported is the slowest rank's and the value aggregates every
rank's bytes. The reference arm prints on rank 0 only."""

from __future__ import annotations

import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out_dir: str):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    res = {}
    # slowest rank's time, identical on every rank
    res["max_ms"] = bench.max_over_ranks(10.0 + 5.0 * rank)
    res["value"] = bench.whole_job_gbs(world, 2e9, res["max_ms"])
    # each rank's batch: same shapes, different draws
    wl = bench.rank_workload(1, rank, 1, "cpu")
    req = wl.requests[0]
    res["shape"] = list(req.xk[0].shape)
    res["sum"] = float(req.xk[0].float().sum() + req.xv[3].float().sum() + wl.q.float().sum())
    gathered = [None] * world
    dist.all_gather_object(gathered, res["sum"])
    res["all_sums"] = gathered
    # the reference arm under torchrun: rank 0 alone prints one JSON line
    args = bench.parse_args_list(["--impl", "reference", "--workload", "cfg1", "--steps", "1", "--warmup", "0"])
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args, world, rank, 1, 1, "tiny")
    res["ref_lines"] = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(world)]
    assert r[0]["max_ms"] == r[1]["max_ms"] == 15.0
    assert r[0]["value"] == pytest.approx(2 * 2e9 / 15e-3 / 1e9)
    assert r[0]["shape"] == r[1]["shape"] == [256, 8, 128]
    assert r[0]["all_sums"] == r[1]["all_sums"]
    assert r[0]["all_sums"][0] != r[0]["all_sums"][1]  # independent batches
    assert len(r[0]["ref_lines"]) == 1 and r[1]["ref_lines"] == []
    line = json.loads(r[0]["ref_lines"][0])
    assert line["impl"] == "reference" and line["n_gpus"] == world and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench

    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_gbs(1, 1e9, 1.0) == pytest.approx(1000.0)
    a = bench.rank_workload(1, 0, 1, "cpu")
    b = bench.rank_workload(1, 0, 1, "cpu")
    assert torch.equal(a.requests[0].xk[0], b.requests[0].xk[0])  # reproducible per rank
