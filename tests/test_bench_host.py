"""Host-side logic of bench.py on the CPU: the max-over-ranks aggregation
under a world_size-2 gloo group, the algorithmic byte counts, and the
reference (oracle) arm end to end."""
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
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r took (r + 1) seconds for 10 units: whole-job value = 20 / 2
    value, t = bench.aggregate(float(rank + 1), 10.0, world)
    bench.barrier()
    q.put((rank, value, t))
    dist.destroy_process_group()


def test_aggregate_takes_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, value, t in got:
        assert t == 2.0 and value == 10.0


def test_aggregate_single_process_is_identity():
    assert bench.aggregate(0.5, 3.0, 1) == (6.0, 0.5)


def test_algorithmic_bytes():
    # codes 17408*5120/4 + f16 scales + x + y
    assert bench.q2_bytes(17408, 5120, 64) == 22282240 + 2785280 + 20480 + 69632
    assert bench.q2_bytes(17408, 5120, 128) == 22282240 + 1392640 + 20480 + 69632
    assert bench.q8_bytes(4096, 4096) == 16826368
    assert bench.q8_bytes(151936, 4096) == 623561728
    assert bench.qmm_flops(17408, 5120, 512) == 91268055040


def test_reference_arm_runs_on_cpu():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "4",
                        "--warmup", "3", "--ref-seconds", "2"], capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, RANK="0", WORLD_SIZE="1"))
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, RANK="1", WORLD_SIZE="2"))
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2", "--impl", "reference"])
