"""Multi-rank host logic of bench.py on CPU: two gloo ranks (world size 2).

The verify path does not shard (every rank runs an independent replica), so
the only cross-rank steps are the barriers around the timed region and the
max over ranks of the measured time.  These run here on the gloo backend; the
GPU launches use the same code with nccl.
"""
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


def _rank_body(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    ranks = bench.Ranks("gloo")
    try:
        ranks.barrier()
        # each rank "measured" a different time; all must agree on the slowest
        t = ranks.max(1.5 + rank * 2.0)
        v = bench.whole_job_tflops(ranks.world, 1e12, t)
        ranks.barrier()
        q.put((rank, ranks.world, t, v))
    finally:
        ranks.close()


def test_two_rank_barrier_and_max():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_body, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    assert codes == [0, 0], codes
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, w, t, v in got:
        assert w == world
        assert t == pytest.approx(3.5)          # max over ranks
        assert v == pytest.approx(2 * 1e12 / 3.5e-3 / 1e12)   # all ranks' work / slowest time


def test_whole_job_value_is_weak_scaling():
    import bench
    one = bench.whole_job_tflops(1, 1e12, 2.0)
    four = bench.whole_job_tflops(4, 1e12, 2.0)
    assert four == pytest.approx(4 * one)


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_single_rank_has_no_process_group():
    import bench
    env = {k: os.environ.pop(k) for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK") if k in os.environ}
    try:
        r = bench.Ranks("gloo")
        assert r.world == 1 and r.dist is None
        r.barrier()
        assert r.max(7.25) == 7.25
        r.close()
    finally:
        os.environ.update(env)


def test_bench_json_contract_keys():
    """The reference arm's line carries the contract's keys (runs the oracle on a tiny sample)."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "c2", "--steps", "1", "--warmup", "3"], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "gpu_launches"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["value"] > 0
