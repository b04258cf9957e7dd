"""The N > 1 path of bench.py on CPU: replicas over `gloo`, world size 2.

Each rank runs its own copy of the step and nothing crosses ranks but the
barrier and the max over ranks of the timed region; the whole-job rate is
world x rows per step x steps / the slowest rank's time. The reference arm
prints only on rank 0; the other ranks exit 0 without work.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, out_q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        rate, job_ms = bench.job_throughput(local_ms[rank], rows_per_step=100, steps=5,
                                            world=world)
        out_q.put((rank, rate, job_ms))
    finally:
        dist.destroy_process_group()


def test_job_rate_is_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    local_ms = [10.0, 25.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, local_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, rate, job_ms in got:
        assert job_ms == pytest.approx(25.0)                       # the slowest rank
        assert rate == pytest.approx(2 * 100 * 5 / 0.025)          # both ranks' rows


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    rate, job_ms = bench.job_throughput(40.0, rows_per_step=8, steps=10, world=1)
    assert job_ms == 40.0 and rate == pytest.approx(8 * 10 / 0.040)


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_line_keeps_the_contract():
    # rank 0 of the reference arm (the fp64 oracle on the host cores) prints
    # one JSON line with the GPU arm's metric, unit and config and its own
    # cpu_baseline / e2e descriptions
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                        "tiny_mixed", "--steps", "2", "--warmup", "1"], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["config"]["workload"] == "tiny_mixed" and d["config"]["q_rows"] == 129
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["ms_per_step"] == pytest.approx(129 / d["value"] * 1e3)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["unit"] == d["unit"] and "oracle work" in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
