"""Host logic of bench.py without a GPU: the multi-rank reduction over a
world-size-2 gloo group, per-rank latent seeds, and the reference arm's JSON
line (the float64 oracle timed on the host cores)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    m = bench.reduce_max(10.0 + rank, dist)
    bench.barrier(dist)
    q.put((rank, m, bench.rank_seed(1000, rank)))
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    import multiprocessing as mp
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    assert [r[1] for r in res] == [11.0, 11.0]
    assert res[0][2] != res[1][2]


def test_reduce_max_without_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5) == 3.5
    assert bench.out_pixels((4, 16, 64, 64)) == 4 * 512 * 512


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "Mpix/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_conv_traffic_is_read_only_for_the_kernel_it_was_captured_on(tmp_path):
    """The roofline's DRAM traffic comes from a machine-readable ncu summary
    that records the sha256 of the conv kernel's source at capture: it is
    used only while the source is that file."""
    sys.path.insert(0, ROOT)
    import bench
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps({"igemm_sha256": bench.igemm_source_sha(),
                                "dram_over_algorithmic": 0.95, "captures": []}))
    assert bench.conv_traffic_ratio(str(path))[0] == 0.95
    path.write_text(json.dumps({"igemm_sha256": "0" * 64, "dram_over_algorithmic": 0.95,
                                "captures": []}))
    assert bench.conv_traffic_ratio(str(path)) == (None, None)
    assert bench.conv_traffic_ratio(str(tmp_path / "none.json")) == (None, None)
