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
T = 128   # the solver's tile edge


def load_measured_peaks():
    """HBM copy bandwidth and cuBLAS bf16 rates measured by the pool's driver
    (MEASURED_PEAKS.json), else the recipe's fallback figures."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["src"] = "measured (MEASURED_PEAKS.json)"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "src": "fallback"}


def measure_peaks(kb, torch, dev, seconds=3.0):
    """The two roofline denominators, measured on this GPU in this run:
    TF32 tensor-core rate of cuBLAS (torch.matmul on 8192^3 fp32 operands
    with TF32 allowed; best of 10 launches, and back to back for `seconds`)
    and the FP32 FMA rate of the library's own probe (bakron_fma_probe)."""
    stream = torch.cuda.current_stream()
    out = {}
    old = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        n = 8192
        a = torch.randn(n, n, device=dev)
        b = torch.randn(n, n, device=dev)
        c = torch.empty(n, n, device=dev)
        fl = 2.0 * n ** 3
        for _ in range(3):
            torch.matmul(a, b, out=c)
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            torch.matmul(a, b, out=c)
            e1.record(stream)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) / 1e3)
        out["tf32_tflops"] = fl / best / 1e12
        k = max(1, int(seconds / best))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k):
            torch.matmul(a, b, out=c)
        e1.record(stream)
        torch.cuda.synchronize()
        out["tf32_tflops_sustained"] = k * fl / (e0.elapsed_time(e1) / 1e3) / 1e12
        del a, b, c
    finally:
        torch.backends.cuda.matmul.allow_tf32 = old
    sms = kb.sm_count()
    blocks = sms * 8
    buf = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    iters = 20000
    kb.fma_probe(buf, blocks, 200)
    torch.cuda.synchronize()
    best = 0.0
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fl = kb.fma_probe(buf, blocks, iters)
        e1.record(stream)
        torch.cuda.synchronize()
        best = max(best, fl / (e0.elapsed_time(e1) / 1e3) / 1e12)
    out["fp32_tflops"] = best
    out["sms"] = sms
    out["how"] = ("tf32: torch.matmul 8192^3 fp32 with allow_tf32 (cuBLAS), best of 10 and back to "
                  "back for %.0f s; fp32: bakron_fma_probe, %d CTAs x 256 threads x 8 FMA chains, "
                  "best of 5" % (seconds, blocks))
    return out


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

def oracle_solve(w, a, impl="rowacc"):
    """The fp64 oracle (prepare + solve) on the leading a x a sub-problem of
    workload w (the leading principal blocks of A and B; a >= m, n: the whole
    problem).  impl "rowacc": the C row-accumulator form on all host cores;
    "bakron": the numpy divide and conquer over anti-diagonals.  Returns
    (prepare seconds, solve seconds, flops under the mn(m+n) model)."""
    import oracle as O
    m, n = min(a, w.m), min(a, w.n)
    t0 = time.perf_counter()
    _, UA = O.prepare(w.A[:n, :n], w.damp_A)
    _, UB = O.prepare(w.B[:m, :m], w.damp_B)
    t1 = time.perf_counter()
    Wa = w.W[:m, :n]
    s = O.row_scale(Wa, w.qmax)
    if impl == "rowacc":
        O.rowacc(Wa, UA, UB, s, w.qmin, w.qmax)
    else:
        O.bakron(Wa, UA, UB, s, w.qmin, w.qmax)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1, flops_model(m, n)


def oracle_threads():
    try:
        from oracle import rowacc as R
        return R.threads()
    except Exception:
        return os.cpu_count()


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] or [os.cpu_count()])
    except Exception:
        return os.cpu_count()


# Oracle timing per workload: whole solves where the C oracle takes seconds,
# a named leading sub-problem for the three largest shapes.
ORACLE_SAMPLE = {"tiny64": None, "c1024": None, "c4096": None,
                 "mlp4096x14336": 2048, "mlp14336x4096": 2048, "c8192": 2048}


def oracle_report(w):
    a = ORACLE_SAMPLE.get(w.name)
    whole = a is None
    a = max(w.m, w.n) if whole else a
    tp, ts, fl = oracle_solve(w, a, "rowacc")
    r = {"impl": "rowacc (C, fp64, OpenMP)", "threads": oracle_threads(),
         "problem": "whole %dx%d" % (w.m, w.n) if whole else
                    "leading %dx%d sub-problem" % (min(a, w.m), min(a, w.n)),
         "prepare_s": tp, "solve_s": ts, "solve_tflops": fl / ts / 1e12}
    if w.m * w.n <= 1024 * 1024:
        tp2, ts2, fl2 = oracle_solve(w, a, "bakron")
        r["numpy_bakron"] = {"prepare_s": tp2, "solve_s": ts2, "solve_tflops": fl2 / ts2 / 1e12,
                             "blas_threads": blas_threads()}
    return r


def run_reference(args, world, rank):
    if rank != 0:
        return
    from kronecker_factored_gptq_gb300 import workloads as WL
    w = WL.load(args.config, seed=args.seed)
    a = args.sample
    for _ in range(args.warmup):
        oracle_solve(w, a)
    ts = []
    fl = 0.0
    for _ in range(args.steps):
        tp, tsolve, f = oracle_solve(w, a)
        ts.append(tp + tsolve)
        fl += f
    total = sum(ts)
    value = fl / total / 1e12
    cores = oracle_threads()
    sub = min(a, w.m, w.n)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "%s, leading %dx%d sub-problem per step" % (w.name, sub, sub),
                   "m": sub, "n": sub},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "fp64 oracle (C row-accumulator solve, %d threads) prepare + "
                                   "solve of the leading %dx%d sub-problem of %s, %d steps"
                                   % (cores, sub, sub, w.name, args.steps)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ metrics

def solve_metrics(torch, W, V, codes, scale, LA, LB, qmin, qmax, tol=1e-4):
    """fp64 metrics of a solve output on the GPU (measurement, not the solve):
    E = L_B (W - V) L_A^T, the proxy loss ||E||_F^2 (= vec(V - W)^T (A (x) B)
    vec(V - W)), and every rounding decision replayed from the output's own
    history, w~ = V + E / (l^B l^A^T) (the GPTQ identity W - V = U^T e):
    codes that differ from the replay, and how many of those are near ties
    (within `tol` grid units of a rounding boundary inside the clamp range)."""
    dt = torch.float64
    LA64, LB64 = LA.to(dt), LB.to(dt)
    E = LB64 @ (W.to(dt) - V.to(dt)) @ LA64.T
    loss = float((E * E).sum())
    wt = V.to(dt) + E / torch.outer(torch.diagonal(LB64), torch.diagonal(LA64))
    del E
    s32 = scale.to(torch.float32)[:, None]
    rep = torch.round(wt.to(torch.float32) / s32).to(dt)
    if qmin is not None:
        rep = rep.clamp(min=float(qmin), max=float(qmax))
    mism = rep != codes.to(dt)
    t = wt / scale.to(dt)[:, None]
    k = torch.floor(t)
    near = (t - (k + 0.5)).abs() < tol
    if qmin is not None:
        near &= (k >= qmin) & (k + 1 <= qmax)
    n_m = int(mism.sum())
    bad = int((mism & ~near).sum())
    return {"proxy_loss": loss, "cert_mismatch": n_m, "cert_not_near_tie": bad}


def config_report(kb, torch, dev, w, reps, peaks):
    """Solve and prepare times, TFLOP/s on the mn(m+n) model, fractions of
    the measured peaks, proxy loss, certificate counts and the Corollary 3.4
    bound on an unclamped unit-step run, for one workload."""
    stream = torch.cuda.current_stream()
    m, n = w.m, w.n
    dW = torch.from_numpy(w.W).to(dev)
    dA = torch.from_numpy(w.A).to(dev)
    dB = torch.from_numpy(w.B).to(dev)
    solver = kb.Solver(m, n, qmin=w.qmin, qmax=w.qmax)
    solver.rowscale(dW)
    solver.prepare(dA, w.damp_A, dB, w.damp_B)
    solver.quantize(dW)
    torch.cuda.synchronize()
    tp, tq = [], []
    for _ in range(reps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        solver.rowscale(dW)
        solver.prepare(dA, w.damp_A, dB, w.damp_B)
        e[1].record(stream)
        solver.quantize(dW)
        e[2].record(stream)
        torch.cuda.synchronize()
        tp.append(e[0].elapsed_time(e[1]) / 1e3)
        tq.append(e[1].elapsed_time(e[2]) / 1e3)
    solve_s, prep_s = statistics.median(tq), statistics.median(tp)
    fl = flops_model(m, n)
    r = {"m": m, "n": n, "bits": w.bits, "solve_s": solve_s, "prepare_s": prep_s,
         "solve_tflops": fl / solve_s / 1e12,
         "solve_frac_of_tf32_peak": fl / solve_s / 1e12 / peaks["tf32_tflops"],
         "solve_frac_of_fp32_peak": fl / solve_s / 1e12 / peaks["fp32_tflops"],
         "reps": reps}
    _, _, LA, LB, _ = kb.bakron_prepare(dA, w.damp_A, dB, w.damp_B, want_L=True)
    r.update(solve_metrics(torch, dW, solver.V, solver.codes, solver.scale, LA, LB, w.qmin, w.qmax))
    # Corollary 3.4 on an unclamped unit-step grid, input 10 W, same factors
    ones = torch.ones(m, dtype=torch.float32, device=dev)
    W10 = 10.0 * dW
    Vu, cu, _ = kb.bakron_quantize(W10, solver.UA, solver.UB, ones, kb.INT32_MIN, kb.INT32_MAX,
                                   workspace=solver.ws_q)
    u = solve_metrics(torch, W10, Vu, cu, ones, LA, LB, None, None)
    dt = torch.float64
    lA2 = float((torch.diagonal(LA.to(dt)) ** 2).sum())
    lB2 = float((torch.diagonal(LB.to(dt)) ** 2).sum())
    trA = float(torch.trace(dA.to(dt))) * (1.0 + w.damp_A)
    trB = float(torch.trace(dB.to(dt))) * (1.0 + w.damp_B)
    r["cor34_unclamped"] = {"proxy_loss": u["proxy_loss"], "bound_tight": 0.25 * lA2 * lB2,
                            "bound_trace": 0.25 * trA * trB,
                            "holds": u["proxy_loss"] <= 0.25 * lA2 * lB2 <= 0.25 * trA * trB * (1 + 1e-5),
                            "cert_mismatch": u["cert_mismatch"],
                            "cert_not_near_tie": u["cert_not_near_tie"]}
    del solver, dW, dA, dB, W10, Vu, cu, LA, LB
    torch.cuda.empty_cache()
    return r


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
    phase = {"leaf_ms": 0.0, "prop1_ms": 0.0, "prop2_ms": 0.0, "near_ms": 0.0, "other_ms": 0.0,
             "prop_flops": 0.0, "leaf_launches": 0, "prop_launches": 0, "near_launches": 0,
             "other_launches": 0}
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
    peaks = measure_peaks(kb, torch, dev)
    mp = load_measured_peaks()

    # Roofline of the dominant kernel class by event-summed device time in the
    # roofline pass.  The propagation product (prop_tc_kernel) counts in
    # algorithmic units: the method's mn(m+n) flops less the work done inside
    # the leaves' tiles (2 T^3 per tile, the in-tile row-accumulator form),
    # divided by the event-summed time of every propagation launch (the
    # off-path propagations and the near products between leaves), against the
    # TF32 rate measured in this run (sustained: the kernel runs inside a
    # seconds-long loop of steps).  The executed (dense 128-tile products) and
    # issued (3 MMAs per product with the 3xTF32 split) fractions stand beside
    # it.
    steps = args.steps
    tiles = -(-m // T) * -(-n // T)
    prop_ms = (phase["prop1_ms"] + phase["prop2_ms"] + phase["near_ms"]) / steps
    leaf_ms = phase["leaf_ms"] / steps
    prop_launches = (phase["prop_launches"] + phase["near_launches"]) / steps
    use_tc = opts.use_3xtf32 == 1
    alg_prop = fl - 2.0 * T ** 3 * tiles
    executed = phase["prop_flops"] / steps
    if prop_ms >= leaf_ms:
        kernel = "prop_tc_kernel (tcgen05 3xTF32)" if use_tc else "prop_simt_kernel (fp32 FMA)"
        per_launch = alg_prop / max(1.0, prop_launches)
        per_launch_ms = prop_ms / max(1.0, prop_launches)
        achieved = alg_prop / (prop_ms / 1e3) / 1e12
        peak = peaks["tf32_tflops_sustained"] if use_tc else peaks["fp32_tflops"]
        bound = "tensor" if use_tc else "alu"
        launches_per_step = prop_launches
        share = prop_ms * steps / (instr_s * 1e3)
        extra = {"executed_flops_per_solve": executed,
                 "executed_frac": executed / (prop_ms / 1e3) / 1e12 / peak,
                 "issued_frac": (3.0 if use_tc else 1.0) * executed / (prop_ms / 1e3) / 1e12 / peak,
                 "algorithmic_flops_per_solve": alg_prop,
                 "counting": "achieved = (m n (m+n) - 2 T^3 tiles) / event-summed propagation time; "
                             "executed: dense 128-tile products; issued: x3 (3xTF32)"}
    else:
        kernel = "leaf_kernel"
        per_launch = 2.0 * T ** 3 * tiles / max(1.0, phase["leaf_launches"] / steps)
        per_launch_ms = leaf_ms / max(1.0, phase["leaf_launches"] / steps)
        achieved = 2.0 * T ** 3 * tiles / (leaf_ms / 1e3) / 1e12
        peak = peaks["fp32_tflops"]
        bound = "alu"
        launches_per_step = phase["leaf_launches"] / steps
        share = leaf_ms * steps / (instr_s * 1e3)
        extra = {"counting": "2 T^3 flops per tile (in-tile row-accumulator form)"}
    roofline = {"bound": bound, "kernel": kernel, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_src": "measured in this run (%s)" % ("TF32 cuBLAS, sustained" if bound == "tensor"
                                                          else "bakron_fma_probe"),
                "algorithmic_flops_per_launch": per_launch, "avg_launch_ms": per_launch_ms,
                "traffic": (traffic_per_launch("kronecker_factored_gptq_gb300/csrc/prop_tc.cu",
                                               "profiles/prop_tc_kernel_c8192_traffic.md")
                            if kernel != "leaf_kernel" and use_tc else None),
                "traffic_unit": "bytes per launch (ncu dram read + write, see profiles/)",
                "launches_per_step": launches_per_step,
                "share_of_timed_region": share,
                "timed_in": "roofline pass: %d steps with per-launch events, %.2f ms per step"
                            % (steps, 1e3 * instr_s / steps)}
    roofline.update(extra)

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

    # Every workload: solve / prepare times, fractions of the measured peaks,
    # proxy loss, certificate counts and Corollary 3.4 (GPU, fp64 metrics),
    # and the fp64 oracle timed on the host cores (whole problems where the C
    # oracle takes seconds, a named leading sub-problem for the largest).
    per_config = None
    if rank == 0 and not args.no_per_config:
        per_config = {}
        del solver, dA, dB
        torch.cuda.empty_cache()
        for name in WL.CONFIGS:
            wc = w if name == args.config else WL.load(name, seed=args.seed, device=dev)
            reps = 3 if wc.m * wc.n >= 8192 * 4096 else 5
            r = config_report(kb, torch, dev, wc, reps, peaks)
            if not args.no_cpu_baseline:
                r["oracle"] = oracle_report(wc)
            per_config[name] = r

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tp, ts, f = oracle_solve(w, args.sample)
        sub = min(args.sample, m, n)
        cpu = {"value": f / (tp + ts) / 1e12, "unit": UNIT, "cores": oracle_threads(),
               "kind": "oracle",
               "sample": "fp64 oracle prepare + solve (C row-accumulator form) of the leading "
                         "%dx%d sub-problem of the workload (%.1f s)" % (sub, sub, tp + ts)}

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
        "peaks": dict(peaks, hbm_gbs=mp.get("hbm_gbs"), bf16_tflops=mp.get("bf16_tflops"),
                      hbm_bf16_src=mp.get("src")),
        "phases_ms_per_step": {k: (v / args.steps if k.endswith("_ms") else v)
                               for k, v in phase.items()},
        "executed_prop_flops_per_solve": phase["prop_flops"] / args.steps,
        "roofline": roofline,
        "per_config": per_config,
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


def run_profile_solve(args):
    """One warm-up step of the configuration, then one factor preparation in
    the NVTX range "prepare" and one solve in the range "solve" (for ncu's
    --nvtx-include); prints one line."""
    import torch
    from kronecker_factored_gptq_gb300 import bakron as kb
    from kronecker_factored_gptq_gb300 import workloads as WL
    if not os.path.exists(kb.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    w = WL.load(args.config, seed=args.seed, device="cuda")
    dW, dA, dB = (torch.from_numpy(x).cuda() for x in (w.W, w.A, w.B))
    solver = kb.Solver(w.m, w.n, bits=w.bits)
    solver.solve(dW, dA, w.damp_A, dB, w.damp_B)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("prepare")
    solver.prepare(dA, w.damp_A, dB, w.damp_B)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    n0 = kb.kernel_launches()
    torch.cuda.nvtx.range_push("solve")
    solver.quantize(dW)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    print(json.dumps({"profile_solve": w.name, "launches": kb.kernel_launches() - n0}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c8192")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--sample", type=int, default=None,
                    help="edge of the leading sub-problem the CPU oracle times (default 4096 for "
                         "the CPU baseline beside the GPU arm, 2048 per step of --impl reference)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload table (solve times, metrics, oracle timings)")
    ap.add_argument("--simt", action="store_true", help="fp32 FMA propagation instead of tcgen05")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-context", action="store_true",
                    help="skip the context timings (one-sided GPTQ, factor accumulation)")
    ap.add_argument("--profile-solve", action="store_true",
                    help="profiling helper: one warm-up step, then one preparation and one solve "
                         "in the NVTX ranges 'prepare' and 'solve'; no benchmark line")
    args = ap.parse_args()
    if args.profile_solve:
        run_profile_solve(args)
        return
    if args.sample is None:
        args.sample = 2048 if args.impl == "reference" else 4096
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
