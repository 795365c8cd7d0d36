"""Host-side logic of bench.py, on CPU: whole-job aggregation, clock parsing, the
multi-rank gather under a world-size-2 gloo group, and the reference (CPU oracle) arm."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_aggregate_sums_units_and_takes_slowest_rank():
    v, t = bench.aggregate([1.0, 2.0, 1.5], [10.0, 10.0, 10.0])
    assert t == 2.0 and v == 15.0


def test_clock_summary():
    rows = [
        ["2026/01/01 00:00:00.000", "0", "1800", "2070", "900", "0x0", "Not Active", "Not Active", "Not Active",
         "Active"],
        ["2026/01/01 00:00:00.100", "0", "1900", "2070", "950", "0x0", "Not Active", "Not Active", "Not Active",
         "Not Active"],
        ["2026/01/01 00:00:00.200", "0", "2000", "2070", "980", "0x0", "Not Active", "Active", "Not Active",
         "Not Active"],
    ]
    c = bench.ClockSampler.summarise(rows)
    assert c["sm_mhz"] == 1900 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist = bench.dist_init(world, "gloo")
    # rank r pretends to have taken 1 + r seconds for 100 units
    got = bench.allgather_floats(dist, world, [1.0 + rank, 100.0], "cpu")
    v, t = bench.aggregate([g[0] for g in got], [g[1] for g in got])
    q.put((rank, v, t))
    dist.destroy_process_group()


def test_two_rank_gloo_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, v, t in res:
        assert t == 2.0 and v == 100.0  # 200 units over the slowest rank's 2 s


def test_reference_arm_prints_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                          "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_traffic_record_requires_unchanged_kernel(tmp_path, monkeypatch):
    assert bench.recorded_traffic("no_such_kernel.cu") is None


def test_kernel_source_sha_covers_included_headers(tmp_path, monkeypatch):
    """A change to a header the kernel includes makes its traffic record stale."""
    csrc = tmp_path / "ternary_weight_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "include").mkdir()
    (csrc / "k.cu").write_text('#include "h.cuh"\nint k;\n')
    (csrc / "h.cuh").write_text("int h;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    a = bench.kernel_source_sha("k.cu")
    (csrc / "h.cuh").write_text("int h2;\n")
    b = bench.kernel_source_sha("k.cu")
    assert a and b and a != b
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.txt").write_text("k.cu %s 123 test\n" % b)
    assert bench.recorded_traffic("k.cu") == 123.0
    (csrc / "k.cu").write_text('#include "h.cuh"\nint k2;\n')
    assert bench.recorded_traffic("k.cu") is None
