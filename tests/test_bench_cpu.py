"""Host-side parts of bench.py, on CPU: the reference (oracle) arm, and the
N > 1 plumbing (process group, barrier, max over ranks) with the gloo
backend at world size 2.  The GPU arm itself needs a GPU and is exercised by
the benchmark runs."""

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


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def test_reference_arm_single_process():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny64",
                        "--sample", "32", "--steps", "2", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["value"] == line["value"]


def test_reference_arm_world2_prints_once():
    port = _free_port()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes", "1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                        str(port), "bench.py", "--impl", "reference", "--config", "tiny64",
                        "--sample", "32", "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2


def _worker(rank, world, port, out):
    # CPU ranks even on a machine with GPUs: the gloo path is what is tested
    os.environ["CUDA_VISIBLE_DEVICES"] = ""
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    out.put((rank, bench.max_over_ranks(float(rank + 1), w, "cpu")))
    dist.destroy_process_group()


def test_dist_helpers_gloo_world2():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    port = _free_port()
    q = ctx.Queue()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in ps)
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 2.0, 1: 2.0}


def _bench_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_clock_summary():
    B = _bench_module()
    lines = ["0, 2070, 2070, 812.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
             "0, 2055, 2070, 1390.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
             "garbage line\n",
             "0, [N/A], 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active\n",
             "0, 1800, 2070, 1400.0, 0x0000000000000008, Active, Not Active, Not Active, Not Active\n"]
    c = B.summarize_clocks(lines)
    assert c["samples"] == 3 and c["sm_mhz"] == 2055 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert B.summarize_clocks([]) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_traffic_from_profile_checks_the_kernel_source(tmp_path):
    import hashlib
    B = _bench_module()
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k() {}\n")
    h = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    prof = tmp_path / "p.md"
    prof.write_text("# summary\ntraffic_bytes_per_launch: 1234\nkernel_source_sha256_16: %s\n" % h)
    assert B.traffic_per_launch(str(src), str(prof)) == 1234.0
    src.write_text("__global__ void k() { /* changed */ }\n")
    assert B.traffic_per_launch(str(src), str(prof)) is None          # stale capture
    assert B.traffic_per_launch(str(tmp_path / "missing.cu"), str(prof)) is None
    # a missing summary reads as unmeasured, not as an error
    assert B.traffic_per_launch("kronecker_factored_gptq_gb300/csrc/prop_tc.cu",
                                str(tmp_path / "none.md")) is None
