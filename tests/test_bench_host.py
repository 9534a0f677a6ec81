"""Host-side checks of bench.py: whole-job aggregation over ranks (gloo, world size 2),
the reference arm's JSON line, and the CPU oracle sample.  No GPU needed."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.dist_init(world, "gloo")
    units, seconds = bench.aggregate(10.0 * (rank + 1), 1.5 + rank, dist, "cpu")
    out.put((rank, units, seconds))
    dist.destroy_process_group()


def test_aggregate_sums_units_and_takes_max_time_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    for _, units, seconds in res:
        assert units == 30.0 and seconds == 2.5


def test_reference_arm_prints_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s"
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["higher_is_better"] is True


def test_cpu_oracle_sample_is_bounded():
    sys.path.insert(0, ROOT)
    import bench
    from sdpa_workloads import training
    v, desc = bench.cpu_oracle_sample(training(1024), seconds=0.2, rows_per_slice=128)
    assert v > 0 and "oracle" in desc


def test_visible_pair_flops_for_lengths_and_bottom_right():
    """The sweep's exact count of visible (row, key) pairs: full lengths with a top-left
    diagonal give s(s+1)/2 per head; a bottom-right diagonal with s_q = s_kv is the same;
    s_q < s_kv bottom-right adds the whole prefix to every row; no mask gives l_q*l_kv."""
    import bench
    from sdpa_workloads import Workload
    per = 4.0 * 3 * 64
    w = Workload("t", 2, 3, 3, 100, 100, 64, "bf16", causal=True, lens_q=(100, 40), lens_kv=(100, 40))
    assert bench.fwd_flops(w) == per * (100 * 101 // 2 + 40 * 41 // 2)
    w = Workload("t", 1, 3, 3, 100, 100, 64, "bf16", causal=True, bottom_right=True)
    assert bench.fwd_flops(w) == per * (100 * 101 // 2)
    w = Workload("t", 1, 3, 3, 30, 100, 64, "bf16", causal=True, bottom_right=True)
    assert bench.fwd_flops(w) == per * sum(70 + i + 1 for i in range(30))
    w = Workload("t", 2, 3, 3, 50, 80, 64, "bf16", lens_q=(50, 7), lens_kv=(80, 0))
    assert bench.fwd_flops(w) == per * (50 * 80)
    # a row whose diagonal falls before the first key sees nothing (bottom-right, l_q > l_kv)
    w = Workload("t", 1, 3, 3, 10, 4, 64, "bf16", causal=True, bottom_right=True)
    assert bench.fwd_flops(w) == per * sum(min(max(i - 6 + 1, 0), 4) for i in range(10))
