"""The benchmark's multi-process path on CPU (gloo, world size 2).

Rows are independent, so N GPUs run N replicas with no data-path collective;
the only cross-rank steps are the barrier around the timed region and the
max-over-ranks of its duration.  Both are exercised here without a GPU, and
the reference arm is checked to print exactly one line (rank 0) under torchrun.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    q.put((rank, bench.max_over_ranks(10.0 * (rank + 1))))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get() for _ in range(2))
    assert got == {0: 20.0, 1: 20.0}


def test_reference_arm_under_torchrun_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", "bench.py", "--impl", "reference",
           "--gpus", "2", "--config", "tiny", "--steps", "1", "--warmup", "0", "--cpu-rows", "2"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "rows/s"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    # the same config record as the GPU arm: the policy's split count (4 rows -> 32), L2 handling
    # and parallelism included
    assert d["config"]["splits"] == 32 and d["config"]["parallelism"] == "replicas"
    assert d["config"]["l2"].startswith("flushed")


def test_reference_arm_index_config_under_torchrun():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", "bench.py", "--impl", "reference",
           "--gpus", "2", "--config", "index", "--steps", "1", "--warmup", "0", "--requests", "4",
           "--ctx", "1000", "3000", "--cpu-rows", "1"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["requests"] == 4


def test_clock_sampler_reasons_and_summary():
    """NVML reason bits map to the names the timing rules use; the summary takes the median SM
    clock, the highest maximum and the union of reasons; no sampler source gives 'unsampled'."""
    import torch
    sys.path.insert(0, ROOT)
    import bench
    assert bench.nvml_reasons(0) == []
    assert bench.nvml_reasons(0x1 | 0x4) == ["sw_power_cap"]                      # idle bit ignored
    assert bench.nvml_reasons(0x8 | 0x20 | 0x40) == ["hw_slowdown", "hw_thermal_slowdown",
                                                     "sw_thermal_slowdown"]
    c = bench.ClockSampler(torch.device("cpu"))
    c.samples = [(2070.0, 2070.0, []), (1980.0, 2070.0, ["sw_power_cap"]), (2070.0, 2070.0, [])]
    assert c.summary()["sm_mhz"] == 2070.0 and c.summary()["reasons"] == ["sw_power_cap"]
    assert c.summary()["samples"] == 3 and c.summary()["sm_max_mhz"] == 2070.0
    c = bench.ClockSampler(torch.device("cpu"))
    c.samples = []
    assert c.summary()["reasons"] == ["unsampled"]
