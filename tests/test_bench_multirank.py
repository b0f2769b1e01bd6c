"""bench.py's data-parallel path on CPU: two gloo ranks (no GPU).

Covers the job-wide aggregation (max of the step times over ranks, sum of
the decoded tokens), the line only rank 0 builds, the per-rank input shards,
and the reference arm printing exactly one line under torchrun."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import bench
from sink_sda_decode_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


# per-rank measurements of a fake run: rank 1 is the slower one for the step
# and the kernel, rank 0 for the end-to-end pass
_TIMES = {0: [2.0, 1.5, 4.0], 1: [3.0, 1.75, 3.5]}
_UNITS = {0: 64, 1: 48}


class _Args:
    steps, warmup, config = 5, 3, "h16"


def _rank_main(rank, ws, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      WORLD_SIZE=str(ws), RANK=str(rank), LOCAL_RANK=str(rank))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        w_ws, w_rank, _ = bench.dist_env()
        assert (w_ws, w_rank) == (ws, rank)
        times, units = bench.reduce_over_ranks(_TIMES[rank], _UNITS[rank], ws, torch.device("cpu"))
        res = {"times": times, "units": units}
        if rank == 0:
            w = inputs.config(0)
            r = {"h2d": 10, "d2h": 20, "clocks": {"sm_mhz": None}, "launches_per_step": 6}
            res["line"] = bench.report_line(_Args, w, ws, *times, units, r)
        with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
            json.dump(res, f)
    finally:
        torch.distributed.destroy_process_group()


def test_two_rank_aggregation_is_max_time_and_summed_tokens(tmp_path):
    ws = 2
    mp.start_processes(_rank_main, args=(ws, _free_port(), str(tmp_path)), nprocs=ws,
                       start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(ws)]
    for r in res:  # every rank sees the same job-wide numbers
        assert r["times"] == [3.0, 1.75, 4.0]
        assert r["units"] == 112.0
    assert "line" not in res[1]
    line = res[0]["line"]
    assert line["n_gpus"] == 2 and line["scaling"] == "weak"
    assert line["config"]["parallelism"] == "dp2 (independent token batches)"
    assert line["ms_per_step"] == 3.0
    assert line["value"] == pytest.approx(112 / 3.0e-3)
    assert line["e2e"]["value"] == pytest.approx(112 / 4.0e-3)
    assert line["roofline"]["kernel_ms"] == 1.75
    assert line["gpu_launches"] == 6 * _Args.steps
    json.dumps(line)


def test_single_process_reduction_is_identity():
    times, units = bench.reduce_over_ranks([1.0, 2.0, 3.0], 7, 1, torch.device("cpu"))
    assert times == [1.0, 2.0, 3.0] and units == 7.0


def test_rank_shards_are_independent_batches_of_one_recipe():
    a0, a1, d = inputs.config(0, shard=0), inputs.config(0, shard=1), inputs.config(0)
    assert np.array_equal(a0.kv_indices, d.kv_indices)
    assert torch.equal(a0.q, d.q)
    assert (a1.N, a1.H, a1.D, a1.total_pages) == (a0.N, a0.H, a0.D, a0.total_pages)
    assert sorted(np.diff(a1.kv_indptr)) == sorted(np.diff(a0.kv_indptr))  # lengths {0,1,17,64}
    assert not torch.equal(a1.q, a0.q)
    assert not np.array_equal(a1.kv_indices, a0.kv_indices)
    with pytest.raises(ValueError):
        inputs.config(0, shard=-1)


def test_reference_arm_prints_one_line_under_torchrun():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--config", "tiny", "--steps", "2", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
