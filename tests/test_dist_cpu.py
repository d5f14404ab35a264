"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

Rows are independent, so N GPUs run N replicas of the per-GPU batch with no
collective on the data path; the only cross-rank steps are the barriers around
the timed region and one all-reduce that turns per-rank figures into whole-job
ones. These tests run those steps as two gloo ranks on the host, and run the
reference arm (the CPU oracle) under torchrun with two ranks: rank 0 alone
times and prints, the other rank exits 0 without work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def bench_module():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    return bench


def _rank_main(rank, world, port, per_rank, out_dir):
    bench = bench_module()
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                            rank=rank, world_size=world)
    try:
        us, e2e = per_rank[rank]
        dist.barrier()
        job_us, job_e2e = bench.job_figures(dist, torch, torch.device("cpu"), us, e2e, world)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"us": job_us, "e2e": job_e2e}, f)
    finally:
        dist.destroy_process_group()


def _run_ranks(per_rank, tmp_path):
    world = len(per_rank)
    mp.start_processes(_rank_main, args=(world, _free_port(), per_rank, str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    return [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]


def test_job_figures_two_ranks(tmp_path):
    # rank 1 is the slower one in the device-timed loop, rank 0 end to end:
    # the job's step time is rank 1's, its e2e rate twice rank 0's.
    got = _run_ranks([(10.25, 4.0e6), (31.5, 5.0e6)], tmp_path)
    for g in got:
        assert g["us"] == 31.5
        assert g["e2e"] == 2 * 4.0e6


def test_job_figures_equal_ranks(tmp_path):
    got = _run_ranks([(20.0, 3.0e6), (20.0, 3.0e6)], tmp_path)
    assert got[0] == got[1] == {"us": 20.0, "e2e": 6.0e6}


def test_job_figures_one_rank():
    assert bench_module().job_figures(None, torch, torch.device("cpu"), 12.5, 7.0e6, 1) \
        == (12.5, 7.0e6)


@pytest.mark.slow
def test_reference_arm_two_ranks():
    env = dict(os.environ, MASTER_ADDR="127.0.0.1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "3", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2 and line["steps"] == 3 and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "rows/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "rows/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
