"""Host-side logic of bench.py on CPU: multi-rank timing aggregation (gloo),
clock parsing, the traffic record rule and the reference (oracle) arm."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    got = bench.max_over_ranks(1.5 + rank, world)
    bench.barrier(world)
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(repr(got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    vals = [float(open(tmp_path / f"r{r}.txt").read()) for r in range(2)]
    assert vals == [2.5, 2.5]


def test_single_rank_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_clock_summary_parsing():
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(0)
    c.out = ("0, 1980, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
             "0, 2070, 2070, 950.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
             "0, 2010, 2070, 940.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n")
    s = c.summary()
    assert s["sm_mhz"] == 2010 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3


def test_traffic_record_requires_unchanged_source(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    prof = tmp_path / "profiles"
    prof.mkdir()
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    import hashlib
    digest = hashlib.sha256(b"kernel v1").hexdigest()
    (prof / "traffic.json").write_text(json.dumps({"k": {"source_sha256": digest, "dram_bytes_per_launch": 123}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("k.cu", "k") == 123
    src.write_text("kernel v2")
    assert bench.kernel_traffic("k.cu", "k") is None


@pytest.mark.slow
def test_reference_arm_prints_one_line():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "4",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
