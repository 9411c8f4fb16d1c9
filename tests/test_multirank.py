"""Host-side logic of the N > 1 bench path, on CPU with the gloo backend.

The path shards by whole requests: every rank runs its own independent batch
of the same workload, nothing crosses ranks on the data path, and the only
collectives are the barrier around the timed region and the max over ranks of
the elapsed times.  These tests run two real processes: one group through
torch.multiprocessing (the helpers bench.py uses), one through torchrun (the
launch the bench contract names), here with the oracle arm, which needs no GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from attention_packed_varlen_gb300 import workloads as wl  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = wl.prefill_workload_inputs(wl.PREFILL_ONLY_REQUEST, seed=bench.rank_prefill_seed(rank))
        # each rank times something different; the job time is the slowest
        my_time = 1.0 + 0.5 * rank
        slowest = bench.max_over_ranks_of(my_time, world, torch.device("cpu"))
        dist.barrier()
        rec = {"rank": rank, "slowest": slowest, "q_sum": float(inp.q.float().sum()),
               "n_seqs": len(inp.lengths), "lengths": [int(x) for x in inp.lengths], "beam_seeds": [bench.rank_beam_seed(b, rank) for b in bench.BEAM_WLS]}
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump(rec, f)
    finally:
        dist.destroy_process_group()


def test_two_ranks_shard_independent_batches_and_take_the_slowest(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    recs = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    assert all(r["slowest"] == 1.5 for r in recs)          # max over ranks, seen by every rank
    assert recs[0]["n_seqs"] == recs[1]["n_seqs"] == wl.PREFILL_ONLY_REQUEST.n_seqs
    assert recs[0]["lengths"] != recs[1]["lengths"]
    assert recs[0]["q_sum"] != recs[1]["q_sum"]             # independent batches, same workload
    assert set(recs[0]["beam_seeds"]).isdisjoint(recs[1]["beam_seeds"])


def test_job_throughput_counts_all_ranks_over_the_slowest():
    assert bench.job_throughput(10.0, 4, 2.0) == 20.0
    assert bench.max_over_ranks_of(3.0, 1, torch.device("cpu")) == 3.0


def test_torchrun_reference_arm_prints_one_line_from_rank_zero():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--ref-budget", "0.05"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_gpu_arm_refuses_to_run_without_cuda():
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "needs a CUDA GPU" in r.stderr
