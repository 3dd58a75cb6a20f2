"""CPU checks of bench.py's host logic: the reference arm's JSON line, the
replica (N > 1) launch under torchrun with two gloo ranks, the max over
ranks used for the whole-job time, and the source hash that keeps a committed
traffic figure to the code it was measured on."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
        "cpu_baseline", "e2e", "impl"}


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def test_reference_arm_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--ref-rows", "32"], cwd=ROOT, capture_output=True,
                         text=True, timeout=600, check=True).stdout
    lines = _json_lines(out)
    assert len(lines) == 1
    d = lines[0]
    assert KEYS <= set(d)
    assert d["impl"] == "reference" and d["unit"] == "Gpixel/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["host"]["nproc"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["config"]["sample_rows"] == 32
    assert d["config"]["workload"] == "c4_sheet_24000x33600_rgba"


def test_reference_arm_two_gloo_ranks_print_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--ref-rows", "16"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900, env=env,
                         check=True).stdout
    lines = _json_lines(out)
    assert len(lines) == 1                      # rank 0 only
    assert lines[0]["n_gpus"] == 2 and lines[0]["impl"] == "reference"


def _max_worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=2)
    q.put((rank, bench.max_over_ranks(1.5 + rank, 2)))
    bench.barrier(2)
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_max_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 2.5, 1: 2.5}


def test_traffic_figure_only_for_the_sources_it_was_measured_on(tmp_path, monkeypatch):
    """bench.py reports a committed ncu traffic figure only while the kernel
    sources hash to the value recorded beside it; comments do not count."""
    sys.path.insert(0, ROOT)
    import bench
    src = tmp_path / "connected_component_labelling_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "k.cuh").write_text("__global__ void k() { int a = 1; }  // first\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.source_sha()
    entry = {"source_sha": sha, "kernels": {"w": {"tile_local": 4.9}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(entry))
    assert bench.traffic_per_px("tile_local", "w") == 4.9
    assert bench.traffic_per_px("number", "w") is None
    (src / "k.cuh").write_text("__global__ void k() { int a = 1; }  /* changed comment */\n")
    assert bench.source_sha() == sha and bench.traffic_per_px("tile_local", "w") == 4.9
    (src / "k.cuh").write_text("__global__ void k() { int a = 2; }\n")
    assert bench.source_sha() != sha and bench.traffic_per_px("tile_local", "w") is None
