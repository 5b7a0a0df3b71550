#!/usr/bin/env python
"""Benchmark of the IKBO hot path on one 1024-candidate, 15-user request.

One step = one request through the whole hot path:
  ikbo_plan         segment build from the candidate->user map
  ikbo_lce_forward  fused LCE  (n_cand 1024, n_users 15, K_u 381, K_c 243, D 256, N 192)
  ikbo_attn_forward broadcast attention (H 8, Lq 32, Lkv 2048, d 128) on the same map
Inputs are seeded synthetic tensors resident in HBM; the L2 is flushed
between steps, outside the per-step CUDA events: a 256 MiB memset (no input
survives in L2), then a 256 MiB read, which evicts the memset's dirty lines
so that their write-back does not land inside the next timed step.

Output: one JSON line (rank 0).  `value` = algorithmic TFLOP/s of the whole
step over all ranks (weak scaling: each rank runs its own request);
`roofline` is the attention kernel's tensor-core fraction, `roofline_lce`
the LCE kernel's HBM fraction; `cpu_baseline` is the fp64 oracle timed on
this host's cores on a bounded sample of the same request; `e2e` repeats the
step through the C ABI with host buffers (H2D of every input, D2H of Y and
O inside the timed region).

    python bench.py [--steps K] [--warmup W] [--impl ikbo|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LCE & broadcast-attn BF16 TFLOP/s, % of roofline; µs per 1024-cand request"
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Cold and clean L2 between timed steps: write a buffer larger than L2,
    then read another one (evicting the written lines; their write-back runs
    here, not in the next step's kernels)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.amax(self.r)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "source": "measured (MEASURED_PEAKS.json)"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback (no MEASURED_PEAKS.json)"}


def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "attn": ["broadcast_gemm_attention_gb300/csrc/attn.cu", "broadcast_gemm_attention_gb300/csrc/ptx.cuh",
             "broadcast_gemm_attention_gb300/csrc/ikbo_internal.h"],
    "lce": ["broadcast_gemm_attention_gb300/csrc/lce.cu", "broadcast_gemm_attention_gb300/csrc/ptx.cuh",
            "broadcast_gemm_attention_gb300/csrc/ikbo_internal.h"],
}


def recorded_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source is unchanged since the counters were taken; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            j = json.load(f)[kernel]
        if j.get("source_hash") == source_hash(KERNEL_SOURCES[kernel]):
            return float(j["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        self.dev = device_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.proc:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """Max of a per-rank float over the process group (identity when alone).
    Uses the group's own backend: a CUDA tensor for NCCL, a CPU one otherwise."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: every rank ran `steps` requests; time = slowest rank."""
    return world * flops_per_step * steps / (max_ms * 1e-3) / 1e12


# --------------------------------------------------------------- workload
def workload():
    from broadcast_gemm_attention_gb300 import inputs as gen
    x = gen.lce_70to1()
    a = gen.attn_70to1()
    assert x.map.tolist() == a.map.tolist()
    return x, a


def flops_bytes(x, a):
    from broadcast_gemm_attention_gb300 import accounting as acc
    lf = acc.lce_flops(x.n_cand, x.n_users, x.K_u, x.K_c, x.D, x.N)
    lb = acc.lce_bytes(x.n_cand, x.n_users, x.K_u, x.K_c, x.D, x.N)
    af = acc.attn_flops(a.H, a.Lq, a.d, [a.Lkv] * a.n_cand)
    ab = acc.attn_bytes(a.n_cand, a.H, a.Lq, a.d, a.n_users * a.Lkv)
    return lf, lb, af, ab


def config_dict(x, a):
    return {
        "workload": "request_70to1: plan + LCE + broadcast attention, 1024 candidates / 15 users (sorted "
                    "multinomial map)",
        "lce": {"n_cand": x.n_cand, "n_users": x.n_users, "K_u": x.K_u, "K_c": x.K_c, "D": x.D, "N": x.N},
        "attn": {"n_cand": a.n_cand, "n_users": a.n_users, "H": a.H, "Lq": a.Lq, "Lkv": a.Lkv, "d": a.d},
        "l2": "flushed between steps, outside the per-step events: 256 MiB memset, then a 256 MiB read that evicts its dirty lines (cold, clean L2); each step also streams ~490 MB",
    }


# ------------------------------------------------------------ CPU oracle
def cpu_oracle_sample(x, a, n: int, seed: int = 0):
    """The fp64 oracle on a bounded sample: n candidates' complete share of the
    request (their LCE rows and their attention over all heads).  Returns
    (seconds, algorithmic flops credited, description, threads)."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)
    cands = sorted(rng.choice(x.n_cand, size=n, replace=False).tolist())
    pairs = [(i, h) for i in cands for h in range(a.H)]
    per_cand = 2.0 * x.D * x.N * (x.K_c + x.K_u * x.n_users / x.n_cand)   # user GEMM amortised
    per_cand += a.H * 4.0 * a.Lq * a.Lkv * a.d
    t0 = time.perf_counter()
    oracle.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b, cands=cands)
    oracle.attn(a.map, a.Q, a.K, a.V, pairs=pairs)
    dt = time.perf_counter() - t0
    desc = (f"{n} of the 1024 candidates of the 70:1 request, each with its LCE rows and its attention over "
            f"all {a.H} heads; credited with the GPU path's algorithmic FLOPs for that share")
    return dt, n * per_cand, desc, oracle.max_threads()


def calibrate_oracle(x, a, seconds: float, lo: int = 1, hi: int = 1024):
    """Candidates per sample so that one sample takes about `seconds`.

    Two probes: a tiny one, then one of about a quarter of the target, whose
    per-candidate time reflects the thread parallelism the full sample gets
    (a 2-candidate probe on a many-core host overestimates it several-fold)."""
    n0 = 16
    dt, _, _, _ = cpu_oracle_sample(x, a, n0, seed=12345)
    n1 = max(n0, min(hi, int(round(0.25 * seconds / max(dt / n0, 1e-6)))))
    if n1 > n0:
        dt, _, _, _ = cpu_oracle_sample(x, a, n1, seed=12346)
        n0 = n1
    n = int(round(seconds / max(dt / n0, 1e-6)))
    return max(lo, min(hi, n))


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def oracle_time(run, total: int, unit: str, seconds: float = 2.0, probe: int = 32) -> dict:
    """Wall time of the fp64 oracle on a calibrated sample of `total` units
    (candidates, (candidate, head) pairs, ...): run(n) does n of them.  A
    probe of `probe` units (enough to keep every host thread busy) sizes the
    sample to about `seconds`; the full time is that sample's time scaled by
    total / n.  Returns the estimate, the sample and the host it ran on."""
    import oracle
    n0 = max(1, min(total, probe))
    t0 = time.perf_counter()
    run(n0)
    dt = time.perf_counter() - t0
    n = max(1, min(total, int(round(n0 * seconds / max(dt, 1e-6)))))
    if n > n0:
        t0 = time.perf_counter()
        run(n)
        dt = time.perf_counter() - t0
    else:
        n = n0
    return {"seconds_full_est": dt * total / n, "seconds_sample": dt, "sample": f"{n} of {total} {unit}",
            "full": n == total, "cores": oracle.max_threads(), "cpu_model": cpu_model(), "kind": "oracle"}


def oracle_lce_time(x, seconds=2.0, seed=0) -> dict:
    import numpy as np
    import oracle
    order = np.random.default_rng(seed).permutation(x.n_cand).tolist()
    return oracle_time(lambda n: oracle.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b, cands=sorted(order[:n])),
                       x.n_cand, "candidates (all their LCE rows)", seconds)


def oracle_attn_time(x, seconds=2.0, seed=0) -> dict:
    import numpy as np
    import oracle
    pairs = [(i, h) for i in range(x.n_cand) for h in range(x.H)]
    order = np.random.default_rng(seed).permutation(len(pairs)).tolist()
    offs = x.kv_offsets if x.jagged else None
    return oracle_time(lambda n: oracle.attn(x.map, x.Q, x.K, x.V, kv_offsets=offs, n_users=x.n_users,
                                             pairs=[pairs[k] for k in sorted(order[:n])]),
                       len(pairs), "(candidate, head) pairs", seconds)


def oracle_lce_backward_time(x, dY) -> dict:
    """The oracle's LCE backward, every gradient, once in full."""
    import oracle
    t0 = time.perf_counter()
    oracle.lce_backward(x.map, x.U, x.C, x.Wu, x.Wc, dY)
    dt = time.perf_counter() - t0
    return {"seconds_full_est": dt, "seconds_sample": dt, "sample": "the whole call (dU, dC, dWu, dWc, db)",
            "full": True, "cores": oracle.max_threads(), "cpu_model": cpu_model(), "kind": "oracle"}


def oracle_attn_backward_time(a, dO, seconds=2.0) -> dict:
    """The oracle's attention backward on two samples, dQ rows of (candidate,
    head) pairs and dK/dV of (user, head) pairs, each scaled to the full call."""
    q = oracle_time(lambda n: oracle_attn_bwd(a, dO, qpairs=[(i % a.n_cand, (i // a.n_cand) % a.H)
                                                              for i in range(0, n * 7, 7)], kvpairs=[]),
                    a.n_cand * a.H, "dQ (candidate, head) pairs", seconds / 2)
    kv = oracle_time(lambda n: oracle_attn_bwd(a, dO, qpairs=[], kvpairs=[(u % a.n_users, (u // a.n_users) % a.H)
                                                                          for u in range(n)]),
                     a.n_users * a.H, "dK/dV (user, head) pairs", seconds / 2, probe=16)
    return {"seconds_full_est": q["seconds_full_est"] + kv["seconds_full_est"],
            "seconds_sample": q["seconds_sample"] + kv["seconds_sample"],
            "sample": f"{q['sample']}; {kv['sample']}", "full": False, "cores": q["cores"],
            "cpu_model": q["cpu_model"], "kind": "oracle"}


def gen_grad_lce(x):
    from broadcast_gemm_attention_gb300 import inputs as gen
    return gen.make_lce_grad(1001, x.n_cand, x.N, x.D)


def gen_grad_attn(a):
    from broadcast_gemm_attention_gb300 import inputs as gen
    return gen.make_attn_grad(1003, tuple(a.Q.shape))


def oracle_attn_bwd(a, dO, qpairs, kvpairs):
    import oracle
    return oracle.attn_backward(a.map, a.Q, a.K, a.V, dO, qpairs=qpairs, kvpairs=kvpairs)


def run_reference(args):
    """The reference arm: the oracle, as it stands, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    x, a = workload()
    per_step = max(0.05, min(3.0, args.ref_budget / max(1, args.steps + args.warmup)))
    n = calibrate_oracle(x, a, per_step)
    for w in range(args.warmup):
        cpu_oracle_sample(x, a, n, seed=1000 + w)
    tot_t, tot_f = 0.0, 0.0
    desc, thr = "", 0
    for k in range(args.steps):
        dt, fl, desc, thr = cpu_oracle_sample(x, a, n, seed=k)
        tot_t += dt
        tot_f += fl
    v = tot_f / tot_t / 1e12
    out = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": config_dict(x, a),
           "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                            "sample": f"per step: {desc}"},
           "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ GPU
def run_gpu(args):
    import torch
    import __graft_entry__ as ge
    from broadcast_gemm_attention_gb300 import binding as B

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    ge.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    x, a = workload()
    lf, lb, af, ab = flops_bytes(x, a)
    step_flops = lf + af

    d = {k: v.to(dev) for k, v in dict(map=x.map, U=x.U, C=x.C, Wu=x.Wu, Wc=x.Wc, b=x.b, Q=a.Q, K=a.K, V=a.V).items()}
    Y = torch.empty(x.n_cand, x.N, x.D, dtype=torch.bfloat16, device=dev)
    O = torch.empty_like(d["Q"])
    flush = L2Flush(dev)
    plan = B.Plan(x.n_cand, max(x.n_users, x.n_cand), a.H)
    plan.set_lce_schedule(args.lce_schedule)

    def step():
        plan.plan(d["map"], x.n_users, a.H, a.Lq, stream)
        plan.lce_forward(d["U"], d["C"], d["Wu"], d["Wc"], d["b"], Y, stream)
        plan.attn_forward(d["Q"], d["K"], d["V"], None, O, None, stream)

    for _ in range(max(3, args.warmup)):
        flush()
        step()
    st = plan.status()
    if st != B.IKBO_OK:
        raise RuntimeError(f"device status after warm-up: {B.ikbo_status_string(st)}")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    launches0 = plan.launches()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        for k in range(K):
            flush()
            e = ev[k]
            e[0].record(stream)
            plan.plan(d["map"], x.n_users, a.H, a.Lq, stream)
            e[1].record(stream)
            plan.lce_forward(d["U"], d["C"], d["Wu"], d["Wc"], d["b"], Y, stream)
            e[2].record(stream)
            plan.attn_forward(d["Q"], d["K"], d["V"], None, O, None, stream)
            e[3].record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    gpu_launches = plan.launches() - launches0
    st = plan.status()
    if st != B.IKBO_OK:
        raise RuntimeError(f"device status after timing: {B.ikbo_status_string(st)}")
    plan_ms = [e[0].elapsed_time(e[1]) for e in ev]
    lce_ms = [e[1].elapsed_time(e[2]) for e in ev]
    attn_ms = [e[2].elapsed_time(e[3]) for e in ev]
    step_ms = [e[0].elapsed_time(e[3]) for e in ev]
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    ms_per_step = total_ms / K
    value = weak_scaling_value(step_flops, K, world, total_ms)

    pk = peaks()
    lce_s = statistics.mean(lce_ms) * 1e-3
    attn_s = statistics.mean(attn_ms) * 1e-3
    attn_tf = af / attn_s / 1e12
    lce_tf = lf / lce_s / 1e12
    lce_gbs = lb / lce_s / 1e9
    roofline = {"kernel": "attn_fwd_kernel (broadcast attention)", "bound": "tensor", "achieved": attn_tf,
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": attn_tf / pk["bf16_tflops"],
                "traffic": recorded_traffic("attn"),
                "peak_source": pk["source"] + ", bf16 burst (kernel timed alone in a short step)",
                "algorithmic": f"{af:.4g} FLOP per launch = 4*H*Lq*d*sum_i Lkv"}
    lce_launches = gpu_launches / K - 2  # a step is segment build + LCE + attention
    lce_kernel = {1: "lce_kernel (one launch)", 2: "lce_kernel (user-tile + candidate-tile launches)"}.get(
        round(lce_launches), "lce_kernel")
    if args.lce_schedule in (0, 3) and round(lce_launches) == 1 and x.N <= 192:
        lce_kernel = "lce_kernel (one launch: local user partials)"
    roofline_lce = {"kernel": lce_kernel, "bound": "hbm", "achieved": lce_gbs, "peak": pk["hbm_gbs"],
                    "unit": "GB/s", "frac": lce_gbs / pk["hbm_gbs"], "traffic": recorded_traffic("lce"),
                    "tflops": lce_tf, "algorithmic": f"{lb:.4g} bytes per launch (inputs once, Y once)"}

    # ---------------- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = e2e_run(plan, d, Y, O, x, a, step_flops, args, K, world, dist, dev)

    # ---------------- ablation: our kernels fed a materialised broadcast
    ablation = None
    if not args.no_ablation:
        ablation = ablation_run(plan, d, x, a, Y, O, flush, stream, dev)

    # ---------------- the pages' LCE stage ladder, rebuilt from our kernel
    lce_stages = None
    if not args.no_ablation:
        lce_stages = lce_stage_run(plan, d, Y, flush, stream)

    # ---------------- self + target attention in one launch vs two
    self_target = None
    if not args.no_self_target:
        self_target = self_target_run(plan, d, x, a, O, flush, stream, dev)
    lce_backward = None
    if not args.no_backward:
        lce_backward = lce_backward_run(plan, d, x, flush, stream, dev, peaks())
    attn_backward = None
    if not args.no_backward:
        attn_backward = attn_backward_run(plan, d, x, a, O, flush, stream, dev, peaks())

    plan.close()
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    cpu = None
    if (world == 1 or rank == 0) and args.cpu_seconds > 0:
        n = calibrate_oracle(x, a, args.cpu_seconds)
        dt, fl, desc, thr = cpu_oracle_sample(x, a, n)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": thr, "cpu_model": cpu_model(), "kind": "oracle",
               "sample": desc, "seconds": dt, "seconds_full_est": dt * x.n_cand / n}
        # the oracle's time for the backward passes of the same request
        if lce_backward is not None:
            lce_backward["cpu_oracle"] = oracle_lce_backward_time(x, gen_grad_lce(x))
        if attn_backward is not None:
            attn_backward["cpu_oracle"] = oracle_attn_backward_time(a, gen_grad_attn(a))

    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded bf16 N(0,1) activations, fan-in-scaled weights)",
        "config": config_dict(x, a),
        "us_per_request": 1e3 * ms_per_step,
        "us_per_request_forward_only": 1e3 * (statistics.mean(lce_ms) + statistics.mean(attn_ms)),
        "kernels": {"plan_us": 1e3 * statistics.mean(plan_ms), "lce_us": 1e3 * statistics.mean(lce_ms),
                    "attn_us": 1e3 * statistics.mean(attn_ms), "lce_tflops": lce_tf, "lce_gbs": lce_gbs,
                    "attn_tflops": attn_tf, "lce_us_median": 1e3 * statistics.median(lce_ms),
                    "attn_us_median": 1e3 * statistics.median(attn_ms)},
        "roofline": roofline, "roofline_lce": roofline_lce,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": gpu_launches,
        "clocks": clk.summary(), "ablation": ablation, "lce_stages": lce_stages, "self_target": self_target,
        "lce_backward": lce_backward, "attn_backward": attn_backward,
    }
    print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


def run_sweep(args):
    """Shape sweep (not the headline metric): the LCE over n_cand in
    {256, 1024, 4096} x ratio in {10, 70, 1000, 10000} and the attention ratio
    sweep (4096 candidates, Lq 16, Lkv 2048), each timed (median of flushed
    runs) and set against its own roofline.  One JSON line per point."""
    import statistics
    import torch
    import __graft_entry__ as ge
    from broadcast_gemm_attention_gb300 import accounting as acc
    from broadcast_gemm_attention_gb300 import binding as B
    from broadcast_gemm_attention_gb300 import inputs as gen
    ge.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(dev)
    pk = peaks()

    def timed(fn, iters=20):
        ts = []
        for k in range(iters + 3):
            flush()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            fn()
            e.record(stream)
            torch.cuda.synchronize()
            if k >= 3:
                ts.append(s.elapsed_time(e))
        return 1e3 * statistics.median(ts)

    for n, r, seed in gen.lce_sweep_points():
        x = gen.lce_sweep(n, r, seed)
        U, C, Wu, Wc, b, m = [t.to(dev) for t in (x.U, x.C, x.Wu, x.Wc, x.b, x.map)]
        Y = torch.empty(x.n_cand, x.N, x.D, dtype=torch.bfloat16, device=dev)
        sched = {}
        with B.Plan(x.n_cand, x.n_users, 1) as p:
            p.plan(m, x.n_users, 1, 8, stream)
            for name, code in (("two_launches", 1), ("one_launch", 2), ("local_partials", 3), ("auto", 0)):
                p.set_lce_schedule(code)
                sched[name] = timed(lambda: p.lce_forward(U, C, Wu, Wc, b, Y, stream))
            us = sched["auto"]
            st = p.status()
        # ablation: the same kernel fed the materialised broadcast U[map]
        # (identity map, n_users = n_cand), and the cost of building it
        idx = m.long()
        U_rep = torch.empty(x.n_cand, x.K_u, x.D, dtype=torch.bfloat16, device=dev)
        ident = torch.arange(x.n_cand, dtype=torch.int32, device=dev)
        mat_us = timed(lambda: torch.index_select(U, 0, idx, out=U_rep))
        with B.Plan(x.n_cand, x.n_cand, 1) as p2:
            p2.plan(ident, x.n_cand, 1, 8, stream)
            on_mat_us = timed(lambda: p2.lce_forward(U_rep, C, Wu, Wc, b, Y, stream))
            st2 = p2.status()
        del U_rep
        byt = acc.lce_bytes(x.n_cand, x.n_users, x.K_u, x.K_c, x.D, x.N)
        fl = acc.lce_flops(x.n_cand, x.n_users, x.K_u, x.K_c, x.D, x.N)
        t_roof = max(byt / (pk["hbm_gbs"] * 1e9), fl / (pk["bf16_tflops"] * 1e12))
        cpu = oracle_lce_time(x) if args.cpu_seconds > 0 else None
        print(json.dumps({"sweep": "lce", "n_cand": n, "ratio": r, "n_users": x.n_users, "us": us, "schedules_us": sched,
                          "cpu_oracle": cpu,
                          "roofline_us": t_roof * 1e6, "frac": t_roof * 1e6 / us, "gbs": byt / (us * 1e-6) / 1e9,
                          "materialised": {"build_us": mat_us, "lce_us": on_mat_us, "total_us": mat_us + on_mat_us,
                                           "ikbo_speedup": (mat_us + on_mat_us) / us,
                                           "status": B.ikbo_status_string(st2)},
                          "status": B.ikbo_status_string(st)}), flush=True)
        del U, C, Wu, Wc, b, m, Y
    for n, r, seed in gen.attn_ratio_sweep_points():
        x = gen.attn_ratio_sweep(n, r, seed)
        Q, K, V, m = [t.to(dev) for t in (x.Q, x.K, x.V, x.map)]
        O = torch.empty_like(Q)
        with B.Plan(x.n_cand, x.n_users, x.H) as p:
            p.plan(m, x.n_users, x.H, x.Lq, stream)
            us = timed(lambda: p.attn_forward(Q, K, V, None, O, None, stream))
            st = p.status()
        fl = acc.attn_flops(x.H, x.Lq, x.d, [x.Lkv] * x.n_cand)
        byt = acc.attn_bytes(x.n_cand, x.H, x.Lq, x.d, x.n_users * x.Lkv)
        t_roof = max(byt / (pk["hbm_gbs"] * 1e9), fl / (pk["bf16_tflops"] * 1e12))
        cpu = oracle_attn_time(x) if args.cpu_seconds > 0 else None
        print(json.dumps({"sweep": "attn", "n_cand": n, "ratio": r, "n_users": x.n_users, "us": us, "cpu_oracle": cpu,
                          "roofline_us": t_roof * 1e6, "frac": t_roof * 1e6 / us, "tflops": fl / (us * 1e-6) / 1e12,
                          "bound": "hbm" if byt / (pk["hbm_gbs"] * 1e9) > fl / (pk["bf16_tflops"] * 1e12) else "tensor",
                          "status": B.ikbo_status_string(st)}), flush=True)
        del Q, K, V, m, O
    # self + target attention: one launch against two, where the users' own
    # queries are a real share of the work (Lq_u up to 512 rows per user and
    # head) and at 4096 candidates of 59 users
    for x in (gen.attn_70to1(), gen.make_attn("attn_4096_59", 1044, n_cand=4096, n_users=59, H=8, Lq=16, d=128,
                                               Lkv=2048, map_kind="permuted")):
        Q, K, V, m = [t.to(dev) for t in (x.Q, x.K, x.V, x.map)]
        O = torch.empty_like(Q)
        with B.Plan(x.n_cand, x.n_users, x.H) as p:
            p.plan(m, x.n_users, x.H, x.Lq, stream)
            d = {"Q": Q, "K": K, "V": V}
            for Lq_u in (64, 128, 256, 512):
                res = self_target_run(p, d, x, x, O, flush, stream, dev, Lq_u=Lq_u)
                res.update({"sweep": "self_target", "n_cand": x.n_cand, "n_users": x.n_users, "Lq": x.Lq,
                            "Lkv": x.Lkv, "fused_over_separate": res["fused_us"] / res["separate_us"]})
                print(json.dumps(res), flush=True)
        del Q, K, V, m, O
    # the stress request: Zipf(1.1) candidates per user, permuted map, jagged
    # per-user histories packed with int32 offsets
    x = gen.attn_stress()
    Q, K, V, m, offs = [t.to(dev) for t in (x.Q, x.K, x.V, x.map, x.kv_offsets)]
    O = torch.empty_like(Q)
    with B.Plan(x.n_cand, x.n_users, x.H) as p:
        p.plan(m, x.n_users, x.H, x.Lq, stream)
        us = timed(lambda: p.attn_forward(Q, K, V, offs, O, None, stream))
        st = p.status()
    lens = (x.kv_offsets[1:] - x.kv_offsets[:-1]).long()
    fl = acc.attn_flops(x.H, x.Lq, x.d, lens[x.map.long()].tolist())
    byt = acc.attn_bytes(x.n_cand, x.H, x.Lq, x.d, int(x.kv_offsets[-1]))
    t_roof = max(byt / (pk["hbm_gbs"] * 1e9), fl / (pk["bf16_tflops"] * 1e12))
    cpu = oracle_attn_time(x) if args.cpu_seconds > 0 else None
    print(json.dumps({"sweep": "attn_stress", "n_cand": x.n_cand, "n_users": x.n_users, "Lq": x.Lq, "cpu_oracle": cpu,
                      "kv_rows": int(x.kv_offsets[-1]), "us": us, "roofline_us": t_roof * 1e6,
                      "frac": t_roof * 1e6 / us, "tflops": fl / (us * 1e-6) / 1e12,
                      "status": B.ikbo_status_string(st)}), flush=True)


CASES = ("attn_stress", "attn_ratio70", "lce_4096_70")


def run_case(args):
    """One forward workload alone, --warmup untimed and --steps timed calls
    with L2 flushed before each (events; median), for a profiler to capture
    one kernel at a shape other than the 70:1 request: the Zipf / jagged
    attention stress request, the attention ratio sweep at 4096 candidates
    and ratio 70, or the LCE sweep point of 4096 candidates and ratio 70.
    One JSON line; not the headline metric."""
    import statistics
    import torch
    import __graft_entry__ as ge
    from broadcast_gemm_attention_gb300 import binding as B
    from broadcast_gemm_attention_gb300 import inputs as gen
    ge.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(dev)
    if args.case == "lce_4096_70":
        n, r, seed = [t for t in gen.lce_sweep_points() if t[0] == 4096 and t[1] == 70][0]
        x = gen.lce_sweep(n, r, seed)
        U, C, Wu, Wc, b, m = [t.to(dev) for t in (x.U, x.C, x.Wu, x.Wc, x.b, x.map)]
        out = torch.empty(x.n_cand, x.N, x.D, dtype=torch.bfloat16, device=dev)
        p = B.Plan(x.n_cand, x.n_users, 1)
        p.plan(m, x.n_users, 1, 8, stream)
        call = lambda: p.lce_forward(U, C, Wu, Wc, b, out, stream)  # noqa: E731
    else:
        if args.case == "attn_stress":
            x = gen.attn_stress()
        else:
            n, r, seed = [t for t in gen.attn_ratio_sweep_points() if t[1] == 70][0]
            x = gen.attn_ratio_sweep(n, r, seed)
        Q, K, V, m = [t.to(dev) for t in (x.Q, x.K, x.V, x.map)]
        offs = None if x.kv_offsets is None else x.kv_offsets.to(dev)
        out = torch.empty_like(Q)
        p = B.Plan(x.n_cand, x.n_users, x.H)
        p.plan(m, x.n_users, x.H, x.Lq, stream)
        call = lambda: p.attn_forward(Q, K, V, offs, out, None, stream)  # noqa: E731
    ts = []
    for k in range(args.warmup + args.steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if k >= args.warmup:
            ts.append(e0.elapsed_time(e1) * 1e3)
    st = p.status()
    p.close()
    print(json.dumps({"case": args.case, "n_cand": x.n_cand, "n_users": x.n_users, "steps": args.steps,
                      "us_median": statistics.median(ts) if ts else None, "status": B.ikbo_status_string(st)}),
          flush=True)
    if st != B.IKBO_OK:
        raise SystemExit(1)


def e2e_run(plan, d, Y, O, x, a, step_flops, args, K, world, dist, dev):
    """End to end through the C ABI from pinned host memory, the way a server
    would run consecutive requests: request k's inputs go host -> device on a
    copy stream while request k-1 computes and request k-2's Y and O come back
    device -> host on a third stream (two device buffer sets; events order
    each request's copy-in, compute and copy-out).  Every request's copies
    are inside the timed region; ms per request = total time / requests."""
    import torch
    h_in = {k: v.cpu().pin_memory() for k, v in d.items()}
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = Y.numel() * 2 + O.numel() * 2
    dbuf = [d, {k: torch.empty_like(v) for k, v in d.items()}]
    ybuf, obuf = [Y, torch.empty_like(Y)], [O, torch.empty_like(O)]
    hy = [torch.empty(Y.shape, dtype=Y.dtype).pin_memory() for _ in range(2)]
    ho = [torch.empty(O.shape, dtype=O.dtype).pin_memory() for _ in range(2)]
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    n_e2e = max(3, min(args.e2e_steps, K))

    def request(k):
        b = k % 2
        di, yb, ob = dbuf[b], ybuf[b], obuf[b]
        if k >= 2:
            s_in.wait_event(comp_done[b])  # request k-2 has finished reading this buffer set
        for name, t in h_in.items():
            with torch.cuda.stream(s_in):
                di[name].copy_(t, non_blocking=True)
        in_done[b].record(s_in)
        s_comp.wait_event(in_done[b])
        if k >= 2:
            s_comp.wait_event(out_done[b])  # request k-2's Y and O have left this buffer set
        plan.plan(di["map"], x.n_users, a.H, a.Lq, s_comp)
        plan.lce_forward(di["U"], di["C"], di["Wu"], di["Wc"], di["b"], yb, s_comp)
        plan.attn_forward(di["Q"], di["K"], di["V"], None, ob, None, s_comp)
        comp_done[b].record(s_comp)
        s_out.wait_event(comp_done[b])
        with torch.cuda.stream(s_out):
            hy[b].copy_(yb, non_blocking=True)
            ho[b].copy_(ob, non_blocking=True)
        out_done[b].record(s_out)

    for k in range(2):  # warm-up: both buffer sets once
        request(k)
    torch.cuda.synchronize()
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_s.record(s_in)
    for st in (s_comp, s_out):
        st.wait_event(e_s)
    for k in range(n_e2e):
        request(k)
    s_in.wait_stream(s_out)
    e_e.record(s_in)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e_s.elapsed_time(e_e) / n_e2e, dist, dev)
    st = plan.status()
    # the plan borrows its map: bind it to the resident one again before
    # this function's second buffer set is freed (the later measurements
    # reuse the plan)
    plan.plan(d["map"], x.n_users, a.H, a.Lq, torch.cuda.current_stream(dev))
    torch.cuda.synchronize()
    return {"value": world * step_flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": n_e2e, "status": "ok" if st == 0 else st,
            "path": "pinned host -> device copies of every input, ikbo_plan + ikbo_lce_forward + ikbo_attn_forward, "
                    "device -> pinned host copies of Y and O; copy-in, compute and copy-out of consecutive requests "
                    "overlap on three streams (two device buffer sets)"}


def lce_stage_run(plan, d, Y, flush, stream, iters=20):
    """ikbo_lce_forward_staged at stages 1 (decomposed: user GEMM, candidate
    GEMM, separate broadcast add), 3 (fused epilogue, one accumulator) and 4
    (the full kernel), median µs over `iters` flushed runs each."""
    import statistics
    import torch
    res = {}
    for st in (1, 3, 4):
        ts = []
        for k in range(iters + 2):
            flush()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            plan.lce_forward_staged(d["U"], d["C"], d["Wu"], d["Wc"], d["b"], Y, st, stream)
            e.record(stream)
            torch.cuda.synchronize()
            if k >= 2:
                ts.append(s.elapsed_time(e))
        res[f"stage{st}_us"] = 1e3 * statistics.median(ts)
    res["note"] = ("stage 1: 3 launches, Y written then read back for the add; stage 3: add fused, one "
                   "accumulator; stage 4: = ikbo_lce_forward. The pages' stage 2 (pad K) is TMA's zero fill "
                   "in every stage")
    return res


def lce_backward_run(plan, d, x, flush, stream, dev, pk, iters=20):
    """ikbo_lce_backward at the request shape (every gradient: dU, dC, dW_u,
    dW_c, db) for a seeded upstream gradient dY, median and mean µs over
    `iters` flushed runs, against its HBM roofline."""
    import statistics
    import torch
    from broadcast_gemm_attention_gb300 import accounting as acc
    from broadcast_gemm_attention_gb300 import inputs as gen
    dY = gen.make_lce_grad(1001, x.n_cand, x.N, x.D).to(dev)
    out = dict(dU=torch.empty(x.n_users, x.K_u, x.D, dtype=torch.bfloat16, device=dev),
               dC=torch.empty(x.n_cand, x.K_c, x.D, dtype=torch.bfloat16, device=dev),
               dWu=torch.empty(x.K_u, x.N, dtype=torch.float32, device=dev),
               dWc=torch.empty(x.K_c, x.N, dtype=torch.float32, device=dev),
               db=torch.empty(x.N, dtype=torch.float32, device=dev))
    ts = []
    l0 = plan.launches()
    for k in range(iters + 3):
        flush()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        plan.lce_backward(d["U"], d["C"], d["Wu"], d["Wc"], dY, stream=stream, **out)
        e.record(stream)
        torch.cuda.synchronize()
        if k >= 3:
            ts.append(s.elapsed_time(e))
    launches = (plan.launches() - l0) / (iters + 3)
    us = 1e3 * statistics.median(ts)
    byt = acc.lce_backward_bytes(x.n_cand, x.n_users, x.K_u, x.K_c, x.D, x.N)
    fl = acc.lce_backward_flops(x.n_cand, x.n_users, x.K_u, x.K_c, x.D, x.N)
    gbs = byt / (us * 1e-6) / 1e9
    return {"us_median": us, "us_mean": 1e3 * statistics.mean(ts), "launches_per_call": launches,
            "tflops": fl / (us * 1e-6) / 1e12,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"],
                         "algorithmic": f"{byt:.4g} bytes per call (dY, U, C, W read once; dU, dC, dW, db written once)"},
            "note": "S = segment sum of dY (fp32; bf16 hi/lo pair for dU and dW_u); dC = W_c dY, dW_c = sum C dY^T; "
                    "dU = W_u S, dW_u = sum U S^T, db from S; one stream, L2 flushed before each call"}


def attn_backward_run(plan, d, x, a, O, flush, stream, dev, pk, iters=20):
    """ikbo_attn_backward at the request's attention shape (dQ for every
    candidate, dK / dV summed over each user's candidates) for a seeded
    upstream gradient dO, after one forward that provides O; median and mean
    µs over `iters` flushed runs, against the tensor roofline of the five
    products the backward needs."""
    import statistics
    import torch
    from broadcast_gemm_attention_gb300 import accounting as acc
    from broadcast_gemm_attention_gb300 import inputs as gen
    dO = gen.make_attn_grad(1003, tuple(a.Q.shape)).to(dev)
    dQ = torch.empty_like(d["Q"])
    dK = torch.empty_like(d["K"])
    dV = torch.empty_like(d["V"])
    lse = torch.empty(tuple(a.Q.shape[:3]), dtype=torch.float32, device=dev)
    plan.plan(d["map"], x.n_users, a.H, a.Lq, stream)
    plan.attn_forward_lse(d["Q"], d["K"], d["V"], None, O, lse, None, stream)

    def timed(with_lse):
        ts = []
        l0 = plan.launches()
        for k in range(iters + 3):
            flush()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            plan.attn_backward(d["Q"], d["K"], d["V"], O, dO, None, dQ, dK, dV, None, stream,
                               lse=lse if with_lse else None)
            e.record(stream)
            torch.cuda.synchronize()
            if k >= 3:
                ts.append(s.elapsed_time(e))
        return ts, (plan.launches() - l0) / (iters + 3)

    ts_re, _ = timed(False)
    ts, launches = timed(True)
    st = plan.status()
    us = 1e3 * statistics.median(ts)
    lens = [a.Lkv] * a.n_cand
    fl = acc.attn_backward_flops(a.H, a.Lq, a.d, lens)
    byt = acc.attn_backward_bytes(a.n_cand, a.H, a.Lq, a.d, a.n_users * a.Lkv)
    tf = fl / (us * 1e-6) / 1e12
    return {"us_median": us, "us_mean": 1e3 * statistics.mean(ts), "launches_per_call": launches,
            "us_median_recomputed_lse": 1e3 * statistics.median(ts_re),
            "tflops": tf, "gbs": byt / (us * 1e-6) / 1e9,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": tf / pk["bf16_tflops"],
                         "algorithmic": f"{fl:.4g} FLOP per call = 10*H*Lq*d*sum_i Lkv (S, dP, dV, dK, dQ)"},
            "status": "ok" if st == 0 else f"error {st}",
            "note": "given the forward's log-sum-exp (ikbo_attn_forward_lse): dQ kernel per forward work unit "
                    "(dS and dQ += dS K), dK/dV kernel per (user, head, 128-key block) over all of the user's "
                    "candidates; us_median_recomputed_lse: without it (one more pass over the keys); one "
                    "stream, L2 flushed before each call"}


def self_target_run(plan, d, x, a, O, flush, stream, dev, Lq_u=64, iters=20):
    """The request's target attention plus each user's own Lq_u queries over
    the same K/V: one launch (ikbo_attn_self_target_forward) against two
    (ikbo_attn_forward for the target part, then the self part alone:
    ikbo_attn_self_target_forward without Q and O)."""
    import statistics
    import torch
    from broadcast_gemm_attention_gb300 import binding as B
    from broadcast_gemm_attention_gb300 import inputs as gen
    Qu = gen.make_user_queries(1093, x.n_users, a.H, Lq_u, a.d).to(dev)
    Ou = torch.empty_like(Qu)
    Ou2 = torch.empty_like(Qu)

    def timed(fn):
        ts = []
        for k in range(iters + 2):
            flush()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            fn()
            e.record(stream)
            torch.cuda.synchronize()
            if k >= 2:
                ts.append(s.elapsed_time(e))
        return 1e3 * statistics.median(ts), 1e3 * statistics.mean(ts)

    fused, fused_mean = timed(lambda: plan.attn_self_target_forward(d["Q"], Qu, d["K"], d["V"], None, O, Ou, None,
                                                                    stream))
    sep, sep_mean = timed(lambda: (plan.attn_forward(d["Q"], d["K"], d["V"], None, O, None, stream),
                                   plan.attn_self_target_forward(None, Qu, d["K"], d["V"], None, None, Ou2, None,
                                                                 stream)))
    st = plan.status()
    same = bool(torch.equal(Ou, Ou2))
    flops = 4.0 * a.H * a.d * a.Lkv * (x.n_cand * a.Lq + x.n_users * Lq_u)
    return {"Lq_u": Lq_u, "fused_us": fused, "separate_us": sep, "fused_mean_us": fused_mean,
            "separate_mean_us": sep_mean, "fused_tflops": flops / (fused * 1e-6) / 1e12,
            "launches": {"fused": 1, "separate": 2}, "self_rows_identical": same,
            "status": "ok" if st == B.IKBO_OK else B.ikbo_status_string(st)}


def ablation_run(plan, d, x, a, Y, O, flush, stream, dev, iters=5):
    """Same kernels on the replicated tensors (identity map, n_users = n_cand),
    plus the cost of materialising them (torch index_select)."""
    import torch
    from broadcast_gemm_attention_gb300 import binding as B
    ident = torch.arange(x.n_cand, dtype=torch.int32, device=dev)
    idx = d["map"].long()
    res = {}

    def timed(fn):
        ts = []
        for _ in range(iters + 1):
            flush()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            fn()
            e.record(stream)
            torch.cuda.synchronize()
            ts.append(s.elapsed_time(e))
        return 1e3 * statistics.median(ts[1:])

    U_rep = torch.empty(x.n_cand, x.K_u, x.D, dtype=torch.bfloat16, device=dev)
    res["lce_materialise_us"] = timed(lambda: torch.index_select(d["U"], 0, idx, out=U_rep))
    p2 = B.Plan(x.n_cand, x.n_cand, a.H)
    p2.plan(ident, x.n_cand, a.H, a.Lq, stream)
    res["lce_on_materialised_us"] = timed(lambda: p2.lce_forward(U_rep, d["C"], d["Wu"], d["Wc"], d["b"], Y, stream))
    del U_rep
    K_rep = torch.empty(a.n_cand, a.H, a.Lkv, a.d, dtype=torch.bfloat16, device=dev)
    V_rep = torch.empty_like(K_rep)

    def mat():
        torch.index_select(d["K"], 0, idx, out=K_rep)
        torch.index_select(d["V"], 0, idx, out=V_rep)

    res["attn_materialise_us"] = timed(mat)
    res["attn_on_materialised_us"] = timed(lambda: p2.attn_forward(d["Q"], K_rep, V_rep, None, O, None, stream))
    st = p2.status()
    p2.close()
    del K_rep, V_rep
    torch.cuda.empty_cache()
    res["status"] = B.ikbo_status_string(st)
    res["note"] = "identity map with n_users = n_cand: the replicated user tensors are real inputs"
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ikbo", "reference"], default="ikbo")
    ap.add_argument("--no-ablation", action="store_true")
    ap.add_argument("--no-self-target", action="store_true", help="skip the self + target attention comparison")
    ap.add_argument("--no-backward", action="store_true", help="skip the LCE and attention backward measurements")
    ap.add_argument("--sweep", action="store_true", help="shape sweep (LCE and attention) instead of the benchmark")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--lce-schedule", type=int, default=0, choices=[0, 1, 2, 3],
                    help="LCE launch schedule: 0 plan-time choice, 1 two launches, 2 one launch, 3 local partials")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target length of the CPU-oracle baseline (0 skips it, e.g. under a profiler)")
    ap.add_argument("--ref-budget", type=float, default=120.0, help="reference arm: total seconds of oracle work")
    ap.add_argument("--case", choices=CASES, default=None,
                    help="run one forward workload alone (for a profiler) instead of the benchmark")
    args = ap.parse_args()
    if args.case:
        run_case(args)
    elif args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
