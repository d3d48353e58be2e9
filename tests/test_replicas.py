"""The N > 1 path of the benchmark: independent replicas, one per rank, no
collective on the data path. The host logic that joins the ranks (barrier,
max of the ranks' step times, whole-job rate) runs here on two `gloo` ranks
on the CPU, through the same functions the benchmark calls under NCCL; the
reference arm runs under torchrun with two ranks and prints one line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, step_ms, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    w, r, local = bench.replica_env()
    assert (w, r, local) == (world, rank, rank)
    dist.init_process_group("gloo", rank=r, world_size=w)
    bench.rank_barrier(w)
    ms_all = bench.max_over_ranks(step_ms[rank], w, "cpu")
    rate = bench.job_rate(4, w, ms_all)
    bench.rank_barrier(w)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms_all": ms_all, "rate": rate}, f)


def test_two_gloo_ranks_agree_on_the_slowest_step(tmp_path):
    world = 2
    step_ms = [0.7164, 0.9031]  # rank 1 is the slow replica
    mp.spawn(_rank_main, args=(world, _free_port(), step_ms, str(tmp_path)),
             nprocs=world, join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for g in got:
        assert g["ms_all"] == max(step_ms)
        # 4 sequences per rank, 2 ranks, one token each per slowest step
        assert g["rate"] == pytest.approx(8 / (max(step_ms) * 1e-3), rel=1e-12)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5, 1, "cpu") == 0.5
    assert bench.job_rate(1, 1, 0.5) == pytest.approx(2000.0)
    bench.rank_barrier(1)  # no-op without a process group


def test_reference_arm_under_two_ranks_prints_one_line():
    """torchrun with two ranks: rank 0 times the oracle and prints one JSON
    line; rank 1 exits 0 without work."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
           "--workload", "tiny", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s"
    assert line["value"] > 0 and line["steps"] == 2 and line["warmup"] == 1
    assert line["config"]["workload"] == "tiny"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["value"] == line["value"]
