"""Host-side logic of bench.py that runs without a GPU: the multi-rank
timing reduction (world size 2 over gloo on CPU), the aggregate value, the
argument rules and the reference arm's rank handling."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # each rank reports a different step time; everyone must see the max
    t = bench.reduce_max(1.5 + rank, world)
    bench.barrier(world)
    v = bench.aggregate_value(64 * 100, world, t)
    q.put((rank, t, v))
    dist.destroy_process_group()


def test_two_rank_max_time_and_whole_job_value():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in out:
        assert t == 2.5
        assert v == pytest.approx(64 * 100 * 2 / 2.5)


def test_single_rank_identity():
    assert bench.reduce_max(3.25, 1) == 3.25
    assert bench.aggregate_value(640, 1, 2.0) == 320


def test_warmup_rule():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_clock_timestamp_parse_and_peaks():
    ts = bench.ClockSampler._ts("2026/12/02 07:21:31.123")
    assert ts is not None
    p = bench.load_peaks()
    assert p["hbm_gbs"] > 1000 and p["bf16_tflops"] > 100


@pytest.mark.slow
def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
