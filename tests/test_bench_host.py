"""Host-side logic of bench.py (no GPU): crossover interpolation, aggregation over ranks, clock
parsing, peaks fallback, and the max-over-ranks reduction on a 2-rank gloo group."""
import json
import math
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_crossover_interpolates_in_n():
    ns = [2048, 4096, 8192]
    # fused/pre = 0.8 at 4096 and 1.25 at 8192 -> log-ratio crosses 0 halfway in N
    n, how = bench.crossover(ns, [1.0, 0.8, 1.25], [1.0 / 0.9, 1.0, 1.0])
    assert abs(n - 6144.0) < 1e-6 and "fused faster below" in how
    n, how = bench.crossover(ns, [1, 1, 1], [2, 2, 2])
    assert n is None and "fused faster at every N" in how
    n, how = bench.crossover(ns, [2, 2, 2], [1, 1, 1])
    assert n is None and "pre-rotate faster" in how


def test_aggregate_counts_all_ranks_over_slowest():
    assert bench.aggregate(0.1374, 100, 4, 2.0) == pytest.approx(0.1374 * 100 * 4 / 2.0)


def test_parse_clocks_window_and_reasons():
    lines = [
        "2026/12/02 10:00:00.000, 0, 1900 MHz, 2070 MHz, 900 W, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:01.000, 0, 1800 MHz, 2070 MHz, 1300 W, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:00:09.000, 0, 500 MHz, 2070 MHz, 100 W, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    import datetime
    t0 = datetime.datetime(2026, 12, 2, 10, 0, 0).timestamp()
    c = bench.parse_clocks("\n".join(lines), t0, t0 + 1.0)
    assert c["sm_mhz"] == 1850 and c["sm_max_mhz"] == 2070 and c["reasons"] == ["sw_power_cap"]
    assert bench.parse_clocks("", t0, t0 + 1) is None


def test_peaks_fallback(tmp_path):
    p = bench.load_peaks(str(tmp_path / "missing.json"))
    assert p["source"] == "fallback" and p["bf16_tflops"] == 1900.0
    f = tmp_path / "peaks.json"
    f.write_text(json.dumps({"hbm_gbs": 1.0, "bf16_tflops": 2.0}))
    p = bench.load_peaks(str(f))
    assert p["source"] == "measured" and p["bf16_tflops_sustained"] == 2.0


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(1.0 + rank, world)
    bench.barrier(world)
    q.put((rank, t, bench.aggregate(1.0, 10, world, t)))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert all(p.exitcode == 0 for p in procs)
    assert [r[1] for r in res] == [2.0, 2.0]          # both ranks see the slowest time
    assert res[0][2] == pytest.approx(10.0)            # 1 unit x 10 steps x 2 ranks / 2 s
