"""bench.py with N > 1 ranks (one process per GPU under torchrun), on CPU:
the ranks' step times reduce to the slowest over gloo, the job's rate counts
every rank's tokens, and the reference arm prints one line, from rank 0.
(The decode step itself needs a GPU; its ranks share nothing, so the
multi-rank logic is what these cover.)"""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, times, out_dir: str):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench = _bench()
    ms = bench._slowest(times[rank], world, "cpu")
    rate = bench._job_rate(world, 4, ms)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "rate": rate}, f)


def test_two_ranks_take_the_slowest_time_and_count_all_tokens(tmp_path):
    times = [5.0, 7.5]
    mp.start_processes(_rank, args=(2, _free_port(), times, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for g in got:
        assert g["ms"] == 7.5
        assert g["rate"] == pytest.approx(2 * 4 / 7.5e-3)


def test_one_rank_is_its_own_time():
    bench = _bench()
    assert bench._slowest(3.25, 1, "cpu") == 3.25
    assert bench._job_rate(1, 1, 8.0) == pytest.approx(125.0)


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "small-layer-d512-kv128", "--steps", "1", "--warmup", "0",
           "--gpus", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
