"""The N > 1 path of bench.py on CPU: the product has no exchange step, so N
GPUs run N independent replicas; the process group carries only barriers and
the max-over-ranks timing.  These tests run that host logic as world-size-2
gloo groups (no GPU), and the reference arm under torchrun, where rank 0
alone works and prints."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, world, port, out_path):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    backend = bench.init_replicas(rank, "gloo")
    assert backend == "gloo"
    # each replica "timed" its own steps; the slowest one sets the job's time
    local_ms = 10.0 + 5.0 * rank
    total = bench.max_over_ranks(local_ms, "cpu")
    dist.barrier()
    with open(f"{out_path}.{rank}", "w") as f:
        json.dump({"rank": rank, "max_ms": total}, f)
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo(tmp_path):
    port = free_port()
    out = str(tmp_path / "r")
    mp.spawn(_replica, args=(2, port, out), nprocs=2, join=True)
    got = [json.load(open(f"{out}.{r}")) for r in range(2)]
    assert all(g["max_ms"] == 15.0 for g in got)


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--workload", "f32_64x64x64", "--steps", "1", "--warmup", "0"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0


def test_kernel_launch_count_per_call():
    """gpu_launches counts the zero fill that precedes a split fp32 product;
    plans come from the host planner (no GPU)."""
    sys.path.insert(0, ROOT)
    import bench
    from tests.conftest import build_library
    build_library()
    import tiled_dense_gemm_02_gb300 as tg
    a, b, c = 0x1000_0000, 0x2000_0000, 0x4000_0000

    def count(M, N, K, dtype, epilogue=False):
        st, p = tg.plan(M, N, K, a, K, b, N, c, N, dtype, None, sm_count=152)
        assert st == tg.OK
        return bench.kernel_launches_per_call(tg, p, epilogue)

    assert count(4096, 4096, 4096, tg.F32) == 2                   # 112 tiles of the last round split
    assert count(4096, 4096, 4096, tg.F32, epilogue=True) == 1    # an epilogue keeps whole tiles
    assert count(2048, 2048, 2048, tg.F32) == 1                   # one round, halves would not fit
    assert count(4096, 4096, 4096, tg.BF16_F32OUT) == 1
    assert count(1000, 1500, 4096, tg.BF16) == 1


def test_cpu_baseline_samples_are_bounded():
    """Both CPU baselines (the oracle and its cache-blocked variant) time a
    bounded sample of rows and report the cores they used."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as wl
    w = wl.BY_NAME["bf16_1000x1500x4096_ragged"]
    A, B = wl.make_inputs(w)
    for fn, kind in ((bench.cpu_oracle_sample, "oracle"), (bench.cpu_blocked_sample, "cache-blocked")):
        r = fn(w, A, B, 0.3)
        assert r["value"] > 0 and r["unit"] == "TFLOP/s" and r["cores"] >= 1
        assert kind in r["kind"] and "rows 0.." in r["sample"]
