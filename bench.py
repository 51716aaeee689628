"""Benchmark of the BaKron solver hot path on GB300.

One step = the whole path on one batch of synthetic input already resident in
HBM: the per-row grid (bakron_rowscale), factor preparation (bakron_prepare:
damping, RevCholesky, inversion of A and B) and the solve (bakron_quantize).
The headline workload is the 8192 x 8192 matrix of the pages' Table 3
(summary page "FastKron: Efficient Quantization with Kronecker-Factored
Hessians"), with synthetic W, A and B (see kronecker_factored_gptq_gb300
.workloads.c8192).  The metric counts mn(m+n) flops per solve.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank solves its own replica (no collective on
the data path; a barrier and a max over ranks bracket the timing).  Rank 0
prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle on the
host cores instead (a bounded sample of the same workload per step).
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "BaKron solve sec & TFLOP/s at 8192x8192 fp32 (% of GB300 TF32/FP32 peak)"
UNIT = "TFLOP/s"
# Dense peaks.  MEASURED_PEAKS.json holds the measured bf16 GEMM rate; the TF32
# tensor peak is that times the nominal tf32/bf16 ratio (1.1 / 2.25).  The
# FP32 FMA peak is 152 SMs x 128 lanes x 2 flops x the maximum SM clock.
NOMINAL_TF32_OVER_BF16 = 1.1 / 2.25
FP32_LANES = 152 * 128


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    d = {}
    if os.path.exists(p):
        d = json.load(open(p))
        src = "measured"
    else:
        d = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
             "sm_max_mhz": 2070.0}
        src = "fallback"
    tf32 = d["bf16_tflops"] * NOMINAL_TF32_OVER_BF16
    tf32_s = d.get("bf16_tflops_sustained", d["bf16_tflops"]) * NOMINAL_TF32_OVER_BF16
    fp32 = FP32_LANES * 2 * d.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
    return {"src": src, "tf32_tflops": tf32, "tf32_tflops_sustained": tf32_s,
            "fp32_tflops": fp32, "hbm_gbs": d["hbm_gbs"]}


def traffic_per_launch(kernel_file, profile_file):
    """DRAM bytes per launch of the dominant kernel, from the committed ncu
    summary; None when the kernel's source changed since the capture."""
    import hashlib
    try:
        src = open(os.path.join(ROOT, kernel_file), "rb").read()
        text = open(os.path.join(ROOT, profile_file)).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line:
            k, _, v = line.partition(":")
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != hashlib.sha256(src).hexdigest()[:16]:
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="bakron_clocks_", suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return summarize_clocks(lines)


def summarize_clocks(lines):
    """Median SM clock under load, the maximum clock, and every throttle
    reason seen Active, from nvidia-smi CSV lines in ClockSampler.FIELDS
    order (noheader, nounits); malformed lines are skipped."""
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
        except ValueError:
            continue
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i].lower() == "active"})
    sm = [r[0] for r in rows]
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows),
            "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ dist

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def flops_model(m, n):
    return float(m) * n * (m + n)


# ------------------------------------------------------------------ oracle

def oracle_sample(w, a):
    """The fp64 oracle (prepare + BaKron solve) on the leading a x a
    sub-problem of workload w, with the leading principal blocks of A and B.
    Returns (seconds, flops under the mn(m+n) model)."""
    import oracle as O
    a = min(a, w.m, w.n)
    t0 = time.perf_counter()
    _, UA = O.prepare(w.A[:a, :a], w.damp_A)
    _, UB = O.prepare(w.B[:a, :a], w.damp_B)
    Wa = w.W[:a, :a]
    s = O.row_scale(Wa, w.qmax)
    O.bakron(Wa, UA, UB, s, w.qmin, w.qmax)
    return time.perf_counter() - t0, flops_model(a, a)


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] or [os.cpu_count()])
    except Exception:
        return os.cpu_count()


def run_reference(args, world, rank):
    if rank != 0:
        return
    from kronecker_factored_gptq_gb300 import workloads as WL
    w = WL.load(args.config, seed=args.seed)
    a = args.sample
    for _ in range(args.warmup):
        oracle_sample(w, a)
    ts = []
    fl = 0.0
    for _ in range(args.steps):
        t, f = oracle_sample(w, a)
        ts.append(t)
        fl += f
    total = sum(ts)
    value = fl / total / 1e12
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "%s, leading %dx%d sub-problem per step" % (w.name, a, a),
                   "m": a, "n": a},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "fp64 oracle prepare + BaKron solve of the leading %dx%d "
                                   "sub-problem of %s, %d steps" % (a, a, w.name, args.steps)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ours

def run_ours(args, world, rank, local):
    import torch
    from kronecker_factored_gptq_gb300 import bakron as kb
    from kronecker_factored_gptq_gb300 import workloads as WL

    if not os.path.exists(kb.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WL.load(args.config, seed=args.seed, device=dev)
    m, n = w.m, w.n
    dW = torch.from_numpy(w.W).to(dev)
    dA = torch.from_numpy(w.A).to(dev)
    dB = torch.from_numpy(w.B).to(dev)
    opts = kb.default_opts()
    if args.simt:
        opts.use_3xtf32 = 0
    times = kb.PhaseTimes()
    solver = kb.Solver(m, n, bits=w.bits, opts=opts)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        solver.rowscale(dW)
        solver.prepare(dA, w.damp_A, dB, w.damp_B)
        if ev is not None:
            ev[1].record(stream)
        solver.quantize(dW)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()

    # Headline pass: K steps bracketed by a barrier and a synchronize, events
    # only around the phases on the caller's stream.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    launches0 = kb.kernel_launches()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = kb.kernel_launches() - launches0
    clocks = sampler.stop()
    barrier(world)
    total_s = max_over_ranks(t_start.elapsed_time(t_end) / 1e3, world, dev)

    # Roofline pass: the same K steps again with a CUDA event pair around
    # every launch of the solve on its own stream (bakron_opts.times).  The
    # events sit between the kernels of the critical stream, so they also
    # turn its programmatic dependent launches into plain ones: this pass is
    # slower than the headline pass and is reported separately.
    opts.times = kb.ctypes.pointer(times)
    solver.opts = opts
    phase = {"leaf_ms": 0.0, "prop1_ms": 0.0, "prop2_ms": 0.0, "other_ms": 0.0, "prop_flops": 0.0,
             "leaf_launches": 0, "prop_launches": 0, "other_launches": 0}
    torch.cuda.synchronize()
    barrier(world)
    r_start = torch.cuda.Event(enable_timing=True)
    r_end = torch.cuda.Event(enable_timing=True)
    r_start.record(stream)
    for k in range(args.steps):
        step()
        for key in phase:
            phase[key] += getattr(times, key)
    r_end.record(stream)
    torch.cuda.synchronize()
    instr_s = max_over_ranks(r_start.elapsed_time(r_end) / 1e3, world, dev)
    opts.times = None
    solver.opts = opts

    prep_ms = [e[0].elapsed_time(e[1]) for e in evs]
    solve_ms = [e[1].elapsed_time(e[2]) for e in evs]
    fl = flops_model(m, n)
    value = world * args.steps * fl / total_s / 1e12
    peaks = load_peaks()

    # roofline of the dominant kernel class (by device time in the timed region)
    prop_ms = phase["prop1_ms"] + phase["prop2_ms"]
    use_tc = opts.use_3xtf32 == 1
    if prop_ms >= phase["leaf_ms"]:
        kernel = "prop_tc_kernel (tcgen05 3xTF32)" if use_tc else "prop_simt_kernel (fp32 FMA)"
        per_launch_flops = phase["prop_flops"] / max(1, phase["prop_launches"])
        per_launch_ms = prop_ms / max(1, phase["prop_launches"])
        issued = 3.0 if use_tc else 1.0
        achieved = issued * per_launch_flops / (per_launch_ms / 1e3) / 1e12
        peak = peaks["tf32_tflops_sustained"] if use_tc else peaks["fp32_tflops"]
        bound = "tensor" if use_tc else "alu"
    else:
        kernel = "leaf_kernel"
        T = 128
        tiles = -(-m // T) * -(-n // T)
        per_launch_flops = 2.0 * T ** 3 * tiles * args.steps / max(1, phase["leaf_launches"])
        per_launch_ms = phase["leaf_ms"] / max(1, phase["leaf_launches"])
        achieved = per_launch_flops / (per_launch_ms / 1e3) / 1e12
        peak = peaks["fp32_tflops"]
        bound = "alu"
    roofline = {"bound": bound, "kernel": kernel, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_src": peaks["src"] + (" (bf16 x 1.1/2.25, sustained)" if bound == "tensor" else
                                             " (152 SMs x 128 FP32 lanes x 2 x max SM clock)"),
                "traffic": (traffic_per_launch("kronecker_factored_gptq_gb300/csrc/prop_tc.cu",
                                               "profiles/prop_tc_kernel_c8192_traffic.md")
                            if kernel != "leaf_kernel" and use_tc else None),
                "traffic_unit": "bytes per launch (ncu dram read + write, see profiles/)",
                "launches_per_step": (phase["leaf_launches"] if kernel == "leaf_kernel"
                                      else phase["prop_launches"]) / args.steps,
                "share_of_timed_region": (phase["leaf_ms"] if kernel == "leaf_kernel" else prop_ms)
                / (instr_s * 1e3),
                "timed_in": "roofline pass: %d steps with per-launch events, %.2f ms per step"
                            % (args.steps, 1e3 * instr_s / args.steps)}

    # End to end through the public API from pinned host buffers.  Copies run
    # on two copy streams, double-buffered: the inputs of step k+1 go up
    # while step k computes, and the result of step k comes down while step
    # k+1 runs its row grid and factor preparation (the solve writes V and the
    # codes only after that read has finished).
    e2e = None
    if not args.no_e2e:
        hW = torch.from_numpy(w.W).pin_memory()
        hA = torch.from_numpy(w.A).pin_memory()
        hB = torch.from_numpy(w.B).pin_memory()
        hV = torch.empty((m, n), dtype=torch.float32).pin_memory()
        hC = torch.empty((m, n), dtype=torch.int8).pin_memory()
        bufs = [(torch.empty_like(dW), torch.empty_like(dA), torch.empty_like(dB)) for _ in range(2)]
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_solved, ev_out = torch.cuda.Event(), torch.cuda.Event()

        def h2d(k):
            bW, bA, bB = bufs[k % 2]
            with torch.cuda.stream(up):
                bW.copy_(hW, non_blocking=True)
                bA.copy_(hA, non_blocking=True)
                bB.copy_(hB, non_blocking=True)
                ev_in[k % 2].record(up)

        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        up.wait_event(e0)
        h2d(0)
        for k in range(args.steps):
            if k + 1 < args.steps:
                h2d(k + 1)   # step k-1, the last reader of this buffer set, has finished
            stream.wait_event(ev_in[k % 2])
            bW, bA, bB = bufs[k % 2]
            solver.rowscale(bW)
            solver.prepare(bA, w.damp_A, bB, w.damp_B)
            if k > 0:
                stream.wait_event(ev_out)
            V, C = solver.quantize(bW)[:2]
            ev_solved.record(stream)
            down.wait_event(ev_solved)
            with torch.cuda.stream(down):
                hV.copy_(V, non_blocking=True)
                hC.copy_(C, non_blocking=True)
                ev_out.record(down)
        stream.wait_event(ev_out)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
        e2e = {"value": world * args.steps * fl / e2e_s / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": int(4 * (m * n + n * n + m * m)),
               "d2h_bytes_per_step": int(4 * m * n + m * n),
               "ms_per_step": 1e3 * e2e_s / args.steps,
               "copies": "pinned host buffers, two copy streams, double-buffered inputs"}

    # One-sided GPTQ (B = I) on the same W and A: the comparison the pages
    # quote (0.059 s for 8192 x 8192 on their GPU); context, not the metric.
    one_sided = None
    if not args.no_context:
        UA1 = torch.empty((n, n), dtype=torch.float32, device=dev)
        ws_p1 = torch.empty(kb.prepare_workspace_size(n, 0), dtype=torch.uint8, device=dev)
        ts = []
        for k in range(args.warmup + 5):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record(stream)
            solver.rowscale(dW)
            kb.bakron_prepare(dA, w.damp_A, workspace=ws_p1, out=(UA1, None))
            e[1].record(stream)
            kb.bakron_quantize(dW, UA1, None, solver.scale, solver.qmin, solver.qmax,
                               workspace=solver.ws_q, out=(solver.V, solver.codes))
            e[2].record(stream)
            torch.cuda.synchronize()
            if k >= args.warmup:
                ts.append((e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2])))
        prep1 = statistics.median(t[0] for t in ts)
        solve1 = statistics.median(t[1] for t in ts)
        one_sided = {"solve_s": solve1 / 1e3, "prepare_A_s": prep1 / 1e3,
                     "solve_tflops_mn2": float(m) * n * n / (solve1 / 1e3) / 1e12,
                     "pages_rtx_pro_6000_s": 0.059, "steps": len(ts)}

    # Kronecker-factor accumulation (K-FAC and one-step Shampoo) from a stream
    # of 16384 samples of both sides: the step before the solver; context.
    factors = None
    if not args.no_context:
        Ns = 16384
        Xs, Gs = WL.sample_stream(Ns, n, m, seed=args.seed)
        dXs, dGs = torch.from_numpy(Xs).to(dev), torch.from_numpy(Gs).to(dev)
        del Xs, Gs
        fws = torch.empty(kb.factors_workspace_size(Ns, n, m), dtype=torch.uint8, device=dev)
        factors = {"samples": Ns}
        for name, md in (("kfac", kb.FACTORS_KFAC), ("shampoo", kb.FACTORS_SHAMPOO)):
            ts = []
            for k in range(args.warmup + 3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                kb.bakron_factors(dXs, dGs, mode=md, workspace=fws)
                e1.record(stream)
                torch.cuda.synchronize()
                if k >= args.warmup:
                    ts.append(e0.elapsed_time(e1))
            t = statistics.median(ts) / 1e3
            # lower 128-tiles of both Gram matrices, 2 flops per multiply-add
            fl_f = 2.0 * Ns * (n * (n + 128) / 2 + m * (m + 128) / 2)
            factors[name + "_s"] = t
            factors[name + "_tflops"] = fl_f / t / 1e12
        del dXs, dGs, fws

    # Batched solves: the two MLP projection shapes (4096 x 14336 and its
    # transpose), one after the other and then together in one batch call
    # (each problem on its own stream set); context for throughput.
    batch = None
    if not args.no_context:
        probs = []
        for name in ("mlp4096x14336", "mlp14336x4096"):
            wb = WL.load(name, seed=args.seed, device=dev)
            bW, bA, bB = (torch.from_numpy(x).to(dev) for x in (wb.W, wb.A, wb.B))
            sb = kb.bakron_rowscale(bW, wb.qmax)
            UAb, UBb, _, _, _ = kb.bakron_prepare(bA, wb.damp_A, bB, wb.damp_B)
            del bA, bB
            probs.append(dict(W=bW, UA=UAb, UB=UBb, scale=sb, qmin=wb.qmin, qmax=wb.qmax))
        wsb = [torch.empty(kb.workspace_size(p_["W"].shape[0], p_["W"].shape[1]), dtype=torch.uint8,
                           device=dev) for p_ in probs]
        seq, bat = [], []
        for k in range(args.warmup + 3):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record(stream)
            for p_, wsp in zip(probs, wsb):
                kb.bakron_quantize(p_["W"], p_["UA"], p_["UB"], p_["scale"], p_["qmin"], p_["qmax"],
                                   workspace=wsp)
            e[1].record(stream)
            kb.bakron_quantize_batch(probs)
            e[2].record(stream)
            torch.cuda.synchronize()
            if k >= args.warmup:
                seq.append(e[0].elapsed_time(e[1]))
                bat.append(e[1].elapsed_time(e[2]))
        fl_b = sum(flops_model(*p_["W"].shape) for p_ in probs)
        batch = {"problems": "4096x14336 + 14336x4096", "sequential_s": statistics.median(seq) / 1e3,
                 "batched_s": statistics.median(bat) / 1e3,
                 "batched_tflops": fl_b / (statistics.median(bat) / 1e3) / 1e12}
        del probs, wsb

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t, f = oracle_sample(w, args.sample)
        cpu = {"value": f / t / 1e12, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
               "sample": "fp64 oracle prepare + BaKron solve of the leading %dx%d sub-problem of "
                         "the workload (%.1f s)" % (min(args.sample, m, n), min(args.sample, m, n), t)}

    if rank != 0:
        return
    solve_med = statistics.median(solve_ms)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "%s: %s" % (w.name, w.desc), "m": m, "n": n, "bits": w.bits,
                   "step": "rowscale + prepare(A, B) + quantize",
                   "l2": "inputs larger than L2 (W, A, B are 256 MiB each at 8192^2)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "propagation": "tcgen05 3xTF32" if use_tc else "fp32 FMA"},
        "solve_s": solve_med / 1e3,
        "solve_tflops": fl / (solve_med / 1e3) / 1e12,
        "solve_frac_of_tf32_peak": fl / (solve_med / 1e3) / 1e12 / peaks["tf32_tflops"],
        "solve_frac_of_fp32_peak": fl / (solve_med / 1e3) / 1e12 / peaks["fp32_tflops"],
        "prepare_s": statistics.median(prep_ms) / 1e3,
        "phases_ms_per_step": {k: (v / args.steps if k.endswith("_ms") else v)
                               for k, v in phase.items()},
        "executed_prop_flops_per_solve": phase["prop_flops"] / args.steps,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clocks,
        "one_sided_gptq": one_sided,
        "factor_accumulation": factors,
        "batched_solves": batch,
        "context": {"pages_rtx_pro_6000_solve_s": 1.839, "pages_yaqa_solve_s": 110.379,
                    "pages_gptq_solve_s": 0.059},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c8192")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--sample", type=int, default=1024,
                    help="edge of the leading sub-problem the CPU oracle times")
    ap.add_argument("--simt", action="store_true", help="fp32 FMA propagation instead of tcgen05")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-context", action="store_true",
                    help="skip the context timings (one-sided GPTQ, factor accumulation)")
    args = ap.parse_args()
    if args.impl == "reference":
        # the oracle runs on rank 0's host cores only; the other ranks exit at
        # once, so no process group is needed
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return
    world, rank, local = dist_setup()
    run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
