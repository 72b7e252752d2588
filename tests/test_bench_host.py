"""Host side of bench.py, on the CPU: the reference arm's JSON line, its launch
under torch.distributed.run with two ranks (gloo), and the barrier / max-over-ranks
timing reduction that the GPU arm uses with N > 1 replicas."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BENCH = os.path.join(ROOT, "bench.py")
REQUIRED = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
            "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def json_lines(out: str) -> list[dict]:
    return [json.loads(line) for line in out.splitlines() if line.startswith("{")]


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, BENCH, "--impl", "reference", "--steps", "1", "--warmup", "0",
                        "--workload", "gpt2"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = json_lines(r.stdout)
    assert len(lines) == 1
    line = lines[0]
    assert REQUIRED <= set(line), REQUIRED - set(line)
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_under_torchrun_two_ranks():
    """N=2 under torch.distributed.run: rank 0 alone runs and prints, rank 1 exits 0."""
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(free_port()), BENCH,
                        "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "gpt2"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2 and lines[0]["impl"] == "reference"


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    spec = importlib.util.spec_from_file_location("bench_under_test", BENCH)
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.5 + rank, w)   # the job's time is the slowest rank's
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(slowest))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_timing_reduction_is_the_max_over_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    vals = [float((tmp_path / f"rank{r}.txt").read_text()) for r in range(world)]
    assert vals == [2.5, 2.5]


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the message shown when no GPU is present")
def test_gpu_arm_without_a_gpu_fails_loudly():
    r = subprocess.run([sys.executable, BENCH, "--steps", "1", "--warmup", "3", "--workload", "tiny",
                        "--no-cpu-baseline", "--no-e2e", "--no-prune"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode != 0
    assert not json_lines(r.stdout)


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", BENCH)
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    return bench


def test_clock_samples_are_taken_from_the_timed_region_only():
    import datetime
    bench = _load_bench()
    line = "0, {sm}, 2070, 1200.5, 0x{act}, Not Active, Not Active, {swt}, {cap}, 2026/12/02 21:48:{sec}"
    text = "\n".join([
        line.format(sm=2070, act="0", swt="Not Active", cap="Not Active", sec="09.900"),   # before: idle
        line.format(sm=1700, act="4", swt="Not Active", cap="Active", sec="10.100"),
        line.format(sm=1760, act="4", swt="Not Active", cap="Active", sec="10.300"),
        line.format(sm=1800, act="4", swt="Not Active", cap="Active", sec="10.500"),
        line.format(sm=1500, act="20", swt="Active", cap="Not Active", sec="11.200"),      # after the region
        "garbage line",
    ])
    lo = datetime.datetime(2026, 12, 2, 21, 48, 10)
    hi = datetime.datetime(2026, 12, 2, 21, 48, 10, 600000)
    c = bench.parse_clock_samples(text, (lo, hi))
    assert c["samples"] == 3 and c["samples_in_timed_region"] is True
    assert c["sm_mhz"] == 1760 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]                 # the thermal flag after the region is ignored
    # no sample inside the window (or no parsable timestamps): every sample is kept and flagged so
    far = (datetime.datetime(2027, 1, 1), datetime.datetime(2027, 1, 2))
    c = bench.parse_clock_samples(text, far)
    assert c["samples"] == 5 and c["samples_in_timed_region"] is False
    assert c["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]
    old = "\n".join(l.rsplit(",", 1)[0] for l in text.splitlines()[:3])   # lines without the timestamp field
    c = bench.parse_clock_samples(old, (lo, hi))
    assert c["samples"] == 3 and c["samples_in_timed_region"] is False
    assert bench.parse_clock_samples("", None) is None
