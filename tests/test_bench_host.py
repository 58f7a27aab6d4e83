"""Multi-rank host logic of bench.py on the CPU: two gloo ranks (world size 2) set up the
process group, draw distinct seeds, meet at the barriers and agree on the max over ranks."""
import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent.parent

WORKER = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import bench
rank, ws = bench.dist_setup()
bench.barrier(ws)
step_ms = 1.0 + rank * 0.75          # rank 1 is the slow one
m = bench.max_over_ranks(step_ms, ws)
seed = bench.seed_for_rank(3, rank)
bench.barrier(ws)
import torch.distributed as dist
backend = dist.get_backend()
dist.destroy_process_group()
print(json.dumps({"rank": rank, "ws": ws, "max": m, "seed": seed, "backend": backend}))
"""


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_agree_on_max_and_draw_distinct_seeds():
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER, str(ROOT)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    res = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        res.append(json.loads(out.strip().splitlines()[-1]))
    res.sort(key=lambda r: r["rank"])
    assert [r["ws"] for r in res] == [2, 2]
    assert all(r["backend"] == "gloo" for r in res)
    assert [r["max"] for r in res] == [1.75, 1.75]
    assert res[0]["seed"] != res[1]["seed"]


def test_single_rank_needs_no_process_group():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    code = ("import sys; sys.path.insert(0, sys.argv[1]); import bench; r, ws = bench.dist_setup(); "
            "bench.barrier(ws); print(r, ws, bench.max_over_ranks(2.5, ws), bench.seed_for_rank(4, r))")
    out = subprocess.run([sys.executable, "-c", code, str(ROOT)], env=env, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == ["0", "1", "2.5", "4"]


def test_profiled_traffic_is_dropped_when_the_kernel_source_changes(tmp_path, monkeypatch):
    import importlib
    sys.path.insert(0, str(ROOT))
    bench = importlib.import_module("bench")
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    import hashlib
    h = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "p.md").write_text(f"source_sha256_16: {h}\ntraffic_bytes_per_launch: 1234\n")
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    assert bench.profiled_traffic("p.md", ["k.cu"]) == 1234
    src.write_text("kernel v2")
    assert bench.profiled_traffic("p.md", ["k.cu"]) is None
    assert bench.profiled_traffic("missing.md", ["k.cu"]) is None


def test_reference_arm_runs_the_fixed_oracle_sample():
    """bench.py --impl reference on the CPU: one JSON line whose sample is the fixed, seeded row set
    that the GPU arm's cpu_baseline uses too (16 rows per host thread, at most the step's rows)."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    out = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference", "--workload", "decode_8k",
                          "--steps", "2", "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tok/s" and line["value"] > 0
    assert line["cpu_baseline"]["cores"] == 2 and "fixed 1 query rows" in line["cpu_baseline"]["sample"]
    sys.path.insert(0, str(ROOT))
    import bench
    from compressed_sparse_attention_03_gb300 import inputs

    wl = inputs.WORKLOADS["prefill_4k"]
    a, b = bench.oracle_rows(wl, 16), bench.oracle_rows(wl, 16)
    assert len(a) == 256 and np.array_equal(a, b) and np.all(np.diff(a) > 0)
