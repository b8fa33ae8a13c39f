"""Host logic of bench.py on CPU: the max-over-ranks timing with 2 gloo ranks,
and the reference arm on a tiny workload (rank 0 prints, other ranks exit)."""
import json
import os
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", init_method="env://")
    got = bench.max_over_ranks(10.0 + rank * 5.0, world)
    bench.barrier(world)
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(repr(got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks(tmp_path):
    port = 29500 + (os.getpid() % 1000)
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    vals = [float(open(tmp_path / f"r{r}.txt").read()) for r in range(2)]
    assert vals == [15.0, 15.0]


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5


def _run_bench(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          env=env, timeout=600)


def test_reference_arm_prints_one_line():
    r = _run_bench({}, "--impl", "reference", "--workload", "tiny_1008", "--steps", "1", "--warmup", "3",
                   "--ref-rows", "4")
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"] == "tiny_1008"


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_bench({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--impl", "reference", "--workload",
                   "tiny_1008", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_below_three_is_rejected():
    r = _run_bench({}, "--impl", "reference", "--warmup", "1")
    assert r.returncode != 0
