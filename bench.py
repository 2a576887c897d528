"""Benchmark of the causal linear-attention operator on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME] [--no-suite]

One step = one la_forward over the whole workload (every (b,h) sequence,
all chunks). The headline workload is the gated delta rule, B=2 H=16
T=8192 d_k=d_v=128, bf16 (the largest single-GPU prefill by FLOPs). The same
JSON line carries a suite of the other workloads measured the same way: the
normalized and per-channel gated prefills, the per-channel-decay delta rule,
and the 1024-step gated-delta decodes.

Timing: W untimed steps, then K steps bracketed by a barrier and a device
synchronize, timed with CUDA events on the launching stream. Each step reads
a different copy of the inputs from a rotating set larger than twice the L2
cache, so no step finds its inputs in L2. Under torchrun every rank runs its
own replica; the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

HEADLINE = W.GDN_B2H16_T8192_D128
SUITE = (W.NORM_B4H8_T2048_D64, W.GLA_B4H16_T4096_D128, W.GDN_DECODE_N256H16_D128, W.NORM_DECAY_B4H8_T2048_D64,
         W.KDA_B2H16_T8192_D128, W.KDA_DECODE_N256H16_D128)
BACKWARD = W.NORM_B4H8_T2048_D64   # the backward is timed on the normalized workload's shapes
GATED_BACKWARD = W.GDN_B2H16_T8192_D128   # and the gated delta rule's on the headline's
C_FLOPS = 64   # chunk size the algorithmic FLOP count is quoted at


# ------------------------------------------------------------------ algorithmic counts

def io_bytes(w: W.Workload) -> int:
    return 2 if w.io == "bf16" else 4


def state_elems(w: W.Workload) -> int:
    return w.dk * w.dv + (w.dk if w.variant in ("norm", "norm_decay") else 0)


def prefill_bytes(w: W.Workload) -> int:
    """q, k, v read and out written, gates read, final state written."""
    n = w.B * w.H * w.T
    b = n * (2 * w.dk + 2 * w.dv) * io_bytes(w)
    if w.variant == "gla":
        b += n * w.dk * 4
    elif w.variant == "gdn":
        b += n * 2 * 4
    elif w.variant == "kda":
        b += n * (w.dk + 1) * 4
    elif w.variant == "norm_decay":
        b += w.B * w.H * 4
    return b + w.B * w.H * state_elems(w) * 4


def backward_bytes(w: W.Workload) -> int:
    """la_backward: q, k, v and the outputs' gradient read; dq, dk, dv written."""
    return w.B * w.H * w.T * (4 * w.dk + 3 * w.dv) * io_bytes(w)


def gated_backward_bytes(w: W.Workload) -> int:
    """la_backward_gated: q, k, v, the outputs' gradient, gate and beta read;
    dq, dk, dv, dgate and dbeta written."""
    gate = w.dk if w.variant == "kda" else 1
    return w.B * w.H * w.T * ((4 * w.dk + 3 * w.dv) * io_bytes(w) + 2 * (gate + 1) * 4)


def prefill_flops(w: W.Workload) -> float:
    """Dense chunk contractions per sequence-head-token at C = 64."""
    C, dk, dv = C_FLOPS, w.dk, w.dv
    if w.variant in ("norm", "norm_decay"):
        per = 2 * C * (dk + dv + 1) + 4 * dk * (dv + 1)
    elif w.variant == "gla":
        per = 2 * C * (dk + dv) + 4 * dk * dv
    else:
        per = 10 * C * dk + 6 * dk * dk + C * C / 3
    return float(per) * w.B * w.H * w.T


def decode_step_bytes(w: W.Workload) -> int:
    n = w.B * w.H
    b = 2 * n * state_elems(w) * 4 + n * (2 * w.dk + 2 * w.dv) * io_bytes(w)
    b += n * 2 * 4 if w.variant == "gdn" else (n * w.dk * 4 if w.variant == "gla" else 0)
    b += n * (w.dk + 1) * 4 if w.variant == "kda" else 0
    return b


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons, every 200 ms."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.lines: list[str] = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        rows = [l.split(", ") for l in self.lines if l.count(",") >= 8]
        if self.uuid:
            mine = [r for r in rows if self.uuid in r[0]]
            rows = mine or rows
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ helpers

def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, dist, device: str) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_step: float, steps: int, n_ranks: int, max_ms: float) -> float:
    """Units all ranks processed (each rank runs the whole workload: replicas)
    per second of the slowest rank."""
    return units_per_step * steps * n_ranks / (max_ms * 1e-3)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def kernel_source_hash() -> str:
    """sha1 (12 hex) of the CUDA sources of the forward and decode paths
    (every file in csrc/ but the backward kernels, which none of the traffic
    keys covers) and the C header."""
    import glob
    import hashlib
    h = hashlib.sha1()
    files = sorted(f for f in glob.glob(os.path.join(ROOT, "gated_delta_rule_causal_gb300", "csrc", "*"))
                   if not os.path.basename(f).startswith("backward"))
    for f in files + [os.path.join(ROOT, "include", "la.h")]:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def all_source_hash() -> str:
    """sha1 (12 hex) of every CUDA source and the C header."""
    import glob
    import hashlib
    h = hashlib.sha1()
    files = sorted(glob.glob(os.path.join(ROOT, "gated_delta_rule_causal_gb300", "csrc", "*")))
    for f in files + [os.path.join(ROOT, "include", "la.h")]:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def traffic_from_profiles(key: str):
    """DRAM bytes (read + write) per unit from the committed ncu capture, or
    None when the kernels changed since the counters were taken (forward and
    decode keys: their sources; "backward/" keys: every source)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if key.startswith("backward/"):
        if d.get("all_source_hash") != all_source_hash():
            return None
    elif d.get("source_hash") != kernel_source_hash():
        return None
    return d.get(key)


# ------------------------------------------------------------------ GPU arm

class PrefillRunner:
    """Rotating device copies of one prefill workload's inputs."""

    def __init__(self, w: W.Workload, seed: int, l2_bytes: int, torch, la):
        self.w, self.torch, self.la = w, torch, la
        self.h = la.Handle(w.B, w.H, w.dk, w.dv, io=w.io)
        x = W.draw(w, seed)
        self.host = x
        in_bytes = prefill_bytes(w)
        self.copies = max(2, int(np.ceil(2.5 * l2_bytes / in_bytes)))
        dev = self.h.device
        mk = lambda a: None if a is None else self._dev(a, dev)
        base = [mk(x.q), mk(x.k), mk(x.v), mk(x.gate), mk(x.beta)]
        self.sets = [base] + [[None if t is None else t.clone() for t in base] for _ in range(self.copies - 1)]
        self.out = torch.empty((w.B, w.H, w.T, w.dv), dtype=self.h.dtype, device=dev)
        self.state = torch.empty((w.B, w.H, state_elems(w)), dtype=torch.float32, device=dev)
        self.i = 0

    @staticmethod
    def _dev(a, dev):
        import torch
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def step(self):
        q, k, v, g, b = self.sets[self.i % self.copies]
        self.i += 1
        self.h.forward(q, k, v, g, b, None, variant=self.w.variant, chunk=0, out=self.out, state_out=self.state)

    @property
    def launches_per_step(self):
        return self.h.last_launches()   # kernels the library enqueued for one forward


class GatedBackwardRunner:
    """The gated delta rule's inputs and an output gradient (two rotating
    device copies, each larger than L2); one la_backward_gated per step."""

    def __init__(self, w: W.Workload, seed: int, torch, la):
        self.w, self.torch = w, torch
        self.h = la.Handle(w.B, w.H, w.dk, w.dv, io=w.io)
        x = W.draw(w, seed)
        do = W.round_io(np.random.default_rng(seed + 1).standard_normal((w.B, w.H, w.T, w.dv)), w.io)
        dev = self.h.device
        base = [PrefillRunner._dev(a, dev) for a in (x.q, x.k, x.v, x.gate, x.beta, do)]
        self.sets = [base, [t.clone() for t in base]]
        self.i = 0

    def step(self):
        q, k, v, g, b, do = self.sets[self.i % 2]
        self.i += 1
        self.h.backward_gated(q, k, v, g, b, do, variant=self.w.variant, return_dstate=False)

    @property
    def launches_per_step(self):
        return self.h.last_launches()


class BackwardRunner:
    """Rotating device copies of the normalized workload's inputs and an
    output gradient; one la_backward per step."""

    def __init__(self, w: W.Workload, seed: int, l2_bytes: int, torch, la):
        self.w, self.torch = w, torch
        self.h = la.Handle(w.B, w.H, w.dk, w.dv, io=w.io)
        x = W.draw(w, seed)
        do = W.round_io(np.random.default_rng(seed + 1).standard_normal((w.B, w.H, w.T, w.dv)), w.io)
        self.copies = max(2, int(np.ceil(2.5 * l2_bytes / backward_bytes(w))))
        dev = self.h.device
        base = [PrefillRunner._dev(a, dev) for a in (x.q, x.k, x.v, do)]
        self.sets = [base] + [[t.clone() for t in base] for _ in range(self.copies - 1)]
        self.grads = [torch.empty_like(base[0]), torch.empty_like(base[1]), torch.empty_like(base[2])]
        self.i = 0

    def step(self):
        q, k, v, do = self.sets[self.i % self.copies]
        self.i += 1
        dq, dk, dv = self.grads
        self.h.backward(q, k, v, do, dq=dq, dk=dk, dv=dv, return_dstate=False)

    @property
    def launches_per_step(self):
        return self.h.last_launches()


class DecodeRunner:
    """A gated-delta decode workload (scalar or per-channel decay); inputs drawn on the device."""

    def __init__(self, w: W.Workload, seed: int, torch, la):
        self.w, self.torch, self.la = w, torch, la
        self.h = la.Handle(w.B, w.H, w.dk, w.dv, io=w.io)
        dev = self.h.device
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        S = w.decode_steps
        n = (S, w.B, w.H)
        self.q = torch.randn(n + (w.dk,), generator=g, device=dev).to(torch.bfloat16)
        k = torch.randn(n + (w.dk,), generator=g, device=dev)
        self.k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
        self.v = torch.randn(n + (w.dv,), generator=g, device=dev).to(torch.bfloat16)
        gshape = n + (w.dk,) if w.variant == "kda" else n   # kda: one decay per key channel
        self.gate = torch.sigmoid(torch.randn(gshape, generator=g, device=dev) + w.gate_mu)
        self.beta = torch.sigmoid(torch.randn(n, generator=g, device=dev) + w.beta_mu)
        self.state = torch.randn((w.B, w.H, state_elems(w)), generator=g, device=dev) * w.state_std
        self.out = torch.empty((w.B, w.H, w.dv), dtype=torch.bfloat16, device=dev)
        self.launches_per_step = S

    def step(self):
        for s in range(self.w.decode_steps):
            self.h.decode_step(self.q[s], self.k[s], self.v[s], self.gate[s], self.beta[s], self.state,
                               variant=self.w.variant, out=self.out, state_out=self.state)


def time_steps(runner, steps: int, warmup: int, torch, dist=None):
    """Returns (total_ms over `steps`, per-step event ms list)."""
    for _ in range(warmup):
        runner.step()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    # Hold the stream for ~0.5 ms before the timed region so that the host
    # has queued the first steps when it opens: the device clock then
    # measures the device's work, not the host's head start (the host-side
    # cost of a call is in the e2e figure).
    torch.cuda._sleep(1_000_000)
    t0.record(stream)
    for a, b in evs:
        a.record(stream)
        runner.step()
        b.record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return t0.elapsed_time(t1), [a.elapsed_time(b) for a, b in evs]


def measure_prefill(w, steps, warmup, torch, la, l2, dist=None):
    r = PrefillRunner(w, 0, l2, torch, la)
    total_ms, per = time_steps(r, steps, warmup, torch, dist)
    kern_ms = statistics.mean(per)
    return r, total_ms, kern_ms


def roofline_prefill(w, kern_ms, pk, key):
    """Roofline of one forward call (all the kernels it enqueues), timed with
    CUDA events around it."""
    byts = prefill_bytes(w)
    gbs = byts / (kern_ms * 1e-3) / 1e9
    t_hbm = byts / (pk["hbm_gbs"] * 1e9)
    t_tc = prefill_flops(w) / (pk["bf16_tflops"] * 1e12)
    return {"bound": "hbm" if t_hbm >= t_tc else "tensor", "achieved": round(gbs, 1),
            "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
            "traffic": traffic_from_profiles(key), "algorithmic_bytes": byts,
            "tflops": round(prefill_flops(w) / (kern_ms * 1e-3) / 1e12, 2),
            "kernel_ms": round(kern_ms, 4), "unit_timed": "one la_forward (all its kernels)",
            "peak_source": pk["source"] + " (burst copy bandwidth)"}


def e2e_prefill(r: PrefillRunner, steps: int, torch):
    """Same metric through the C ABI from pinned host buffers: every step is
    one la_forward_host call, which copies the step's inputs in, runs the
    kernels and copies output and final state out (the library overlaps the
    copies of one group of sequence-heads with the kernels of another); all
    of it inside the timing."""
    w, x = r.w, r.host

    def pinned(a):
        t = PrefillRunner._dev(a, "cpu") if a is not None else None
        return None if t is None else t.pin_memory()

    hq, hk, hv, hg, hb = (pinned(a) for a in (x.q, x.k, x.v, x.gate, x.beta))
    ho = torch.empty(r.out.shape, dtype=r.out.dtype).pin_memory()
    hs = torch.empty(r.state.shape, dtype=r.state.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hg, hb) if t is not None)
    d2h = ho.numel() * ho.element_size() + hs.numel() * hs.element_size()

    def one():
        r.h.forward_host(hq, hk, hv, hg, hb, None, variant=w.variant, chunk=0, out=ho, state_out=hs)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    for _ in range(steps):
        one()
    b.record(s)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    return {"value": round(w.tokens * steps / (ms * 1e-3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms / steps, 4)}


def cpu_oracle_baseline(w: W.Workload, budget_s: float = 2.0):
    """The float64 oracle as it stands, on this host's cores, on the whole
    workload repeated until `budget_s` of wall time has passed."""
    import oracle
    x = W.draw(w, 0)
    q, k, v = W.as_f64(x.q), W.as_f64(x.k), W.as_f64(x.v)
    g = None if x.gate is None else x.gate.astype(np.float64)
    b = None if x.beta is None else x.beta.astype(np.float64)
    cores = host_cores()
    oracle.run(w.variant, q[:1, :1, :64], k[:1, :1, :64], v[:1, :1, :64],
               None if g is None else g[:1, :1, :64], None if b is None else b[:1, :1, :64], nthreads=cores)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.run(w.variant, q, k, v, g, b, nthreads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": round(w.tokens * reps / el, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"whole workload ({w.B * w.H} sequence-heads x {w.T} tokens) x {reps}, "
                      f"{el:.2f} s wall, float64 C recurrence with OpenMP over sequence-heads"}


def gpu_arm(args):
    import torch
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
        dist = tdist
    import gated_delta_rule_causal_gb300 as la
    la.build()
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    uuid = str(getattr(props, "uuid", "")) or None
    pk = peaks()
    w = W.BY_NAME[args.workload] if args.workload else HEADLINE
    if w.decode_steps:
        raise SystemExit(f"{w.name} is a decode workload: it is measured in the suite entries of the default run "
                         "(or alone with --only-kernel)")

    sampler = ClockSampler(uuid)
    sampler.start()
    t_wall0 = time.perf_counter()
    r, total_ms, kern_ms = measure_prefill(w, args.steps, args.warmup, torch, la, l2, dist)
    # keep the same work running for >= 1.5 s so the clock sampler sees it
    t_s = time.perf_counter()
    while time.perf_counter() - t_s < 1.5:
        for _ in range(20):
            r.step()
        torch.cuda.synchronize()
    clocks = sampler.stop()
    max_ms = max_over_ranks(total_ms, dist, "cuda")
    n = ws
    value = job_throughput(w.tokens, args.steps, n, max_ms)
    line = {
        "metric": "prefill tokens/s (B*T)", "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": n, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded numpy PCG64, distributions of the workload)",
        "config": {"workload": w.name, "variant": w.variant, "B": w.B, "H": w.H, "T": w.T, "d_k": w.dk,
                   "d_v": w.dv, "chunk": 64, "parallelism": f"replicas x{n}",
                   "l2": f"{r.copies} rotating input copies, {r.copies * prefill_bytes(w) / 1e6:.0f} MB > 2x L2 "
                         f"({l2 / 1e6:.0f} MB)"},
        "roofline": roofline_prefill(w, kern_ms, pk, f"forward/{w.variant}"),
        "gpu_launches": args.steps * r.launches_per_step,
        "clocks": clocks,
    }
    if rank == 0 and ws == 1:
        line["e2e"] = e2e_prefill(r, args.steps, torch)
        line["cpu_baseline"] = cpu_oracle_baseline(w)
    elif rank == 0:
        line["e2e"] = e2e_prefill(r, args.steps, torch)
    if not args.no_suite:
        suite = []
        for sw in SUITE:
            if sw.decode_steps:
                dr = DecodeRunner(sw, 0, torch, la)
                steps = max(2, min(args.steps, 5))
                tot, per = time_steps(dr, steps, 1, torch, dist)
                ms_step = statistics.mean(per)
                launch_ms = ms_step / sw.decode_steps
                byts = decode_step_bytes(sw)
                gbs = byts / (launch_ms * 1e-3) / 1e9
                suite.append({"workload": sw.name, "metric": "decode sequence-tokens/s",
                              "value": round(sw.B * sw.decode_steps / (ms_step * 1e-3), 1),
                              "unit": "sequence-tokens/s", "ms_per_step": round(ms_step, 4),
                              "us_per_decode_launch": round(launch_ms * 1e3, 3),
                              "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"],
                                           "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                                           "traffic": traffic_from_profiles(f"decode_{sw.variant}"),
                                           "peak_source": pk["source"] + " (burst copy bandwidth)",
                                           "algorithmic_bytes": byts},
                              "gpu_launches": steps * dr.launches_per_step})
                del dr
            else:
                pr, tot, kms = measure_prefill(sw, args.steps, args.warmup, torch, la, l2, dist)
                suite.append({"workload": sw.name, "metric": "prefill tokens/s (B*T)",
                              "value": round(sw.tokens * args.steps / (tot * 1e-3), 1), "unit": "tokens/s",
                              "ms_per_step": round(tot / args.steps, 4),
                              "roofline": roofline_prefill(sw, kms, pk, f"forward/{sw.variant}"),
                              "gpu_launches": args.steps * pr.launches_per_step})
                del pr
            torch.cuda.empty_cache()
        # the backward of the normalized prefill on the normalized workload's shapes
        br = BackwardRunner(BACKWARD, 0, l2, torch, la)
        tot, per = time_steps(br, args.steps, args.warmup, torch, dist)
        kms = statistics.mean(per)
        byts = backward_bytes(BACKWARD)
        gbs = byts / (kms * 1e-3) / 1e9
        suite.append({"workload": "norm_backward_" + BACKWARD.name.split("_", 1)[1], "metric": "backward tokens/s (B*T)",
                      "value": round(BACKWARD.tokens * args.steps / (tot * 1e-3), 1), "unit": "tokens/s",
                      "ms_per_step": round(tot / args.steps, 4),
                      "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                                   "frac": round(gbs / pk["hbm_gbs"], 4),
                                   "traffic": traffic_from_profiles("backward/norm"), "algorithmic_bytes": byts,
                                   "kernel_ms": round(kms, 4),
                                   "peak_source": pk["source"] + " (burst copy bandwidth)",
                                   "note": "chunkwise tcgen05 chain (five launches per head group)"},
                      "gpu_launches": args.steps * br.launches_per_step})
        del br
        torch.cuda.empty_cache()
        # the gated delta rule's backward on the headline's shapes (chunkwise)
        gs = max(3, args.steps // 4)
        gr = GatedBackwardRunner(GATED_BACKWARD, 0, torch, la)
        tot, per = time_steps(gr, gs, args.warmup, torch)
        kms = statistics.mean(per)
        byts = gated_backward_bytes(GATED_BACKWARD)
        gbs = byts / (kms * 1e-3) / 1e9
        suite.append({"workload": "gdn_backward_" + GATED_BACKWARD.name.split("_", 1)[1],
                      "metric": "backward tokens/s (B*T)",
                      "value": round(GATED_BACKWARD.tokens * gs / (tot * 1e-3), 1), "unit": "tokens/s",
                      "ms_per_step": round(tot / gs, 4), "steps": gs,
                      "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                                   "frac": round(gbs / pk["hbm_gbs"], 4),
                                   "traffic": traffic_from_profiles("backward/gdn"), "algorithmic_bytes": byts,
                                   "kernel_ms": round(kms, 4),
                                   "peak_source": pk["source"] + " (burst copy bandwidth)",
                                   "note": "chunkwise: per-chunk prep, both chunk chains in one launch, two "
                                           "per-chunk gradient kernels; warp-level tf32 MMAs"},
                      "gpu_launches": gs * gr.launches_per_step})
        del gr
        torch.cuda.empty_cache()
        line["suite"] = suite
    line["wall_s"] = round(time.perf_counter() - t_wall0, 2)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def kernel_only(args):
    """Only the workload's launches (no suite, e2e, baseline or sampler)."""
    import torch
    import gated_delta_rule_causal_gb300 as la
    la.build()
    w = (BACKWARD if args.backward else GATED_BACKWARD if args.gated_backward
         else W.BY_NAME[args.workload] if args.workload else HEADLINE)
    if args.gated_backward and args.workload:
        w = W.BY_NAME[args.workload]   # a smaller gated workload, for ncu captures
    if args.seq_len:
        w = w.with_(T=args.seq_len)    # a shorter sequence of the same shapes, for ncu captures
    props = torch.cuda.get_device_properties(0)
    if args.backward:
        r = BackwardRunner(w, 0, int(getattr(props, "L2_cache_size", 126 * 2 ** 20)), torch, la)
    elif args.gated_backward:
        r = GatedBackwardRunner(w, 0, torch, la)
    elif w.decode_steps:
        r = DecodeRunner(w.with_(decode_steps=8), 0, torch, la)
    else:
        r = PrefillRunner(w, 0, int(getattr(props, "L2_cache_size", 126 * 2 ** 20)), torch, la)
    total_ms, per = time_steps(r, args.steps, args.warmup, torch)
    print(json.dumps({"workload": ("backward/" if args.backward or args.gated_backward else "") + w.name,
                      "steps": args.steps, "ms_per_step": round(total_ms / args.steps, 5),
                      "kernel_ms": [round(x, 5) for x in per]}), flush=True)


def cpu_model() -> str:
    """The host CPU's model name (/proc/cpuinfo; Arm hosts name the part)."""
    try:
        with open("/proc/cpuinfo") as f:
            txt = f.read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model", "CPU part"):
        for line in txt.splitlines():
            if line.startswith(key) and ":" in line:
                return line.split(":", 1)[1].strip()
    return "unknown"


def reference_arm(args):
    """The float64 CPU oracle, timed on the host cores (rank 0 only): every
    step runs the whole workload (all sequence-heads, all tokens) with OpenMP
    over the sequence-heads on every core the process may use."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = W.BY_NAME[args.workload] if args.workload else HEADLINE
    x = W.draw(w, 0)
    q, k, v = W.as_f64(x.q), W.as_f64(x.k), W.as_f64(x.v)
    g = None if x.gate is None else x.gate.astype(np.float64)
    b = None if x.beta is None else x.beta.astype(np.float64)
    cores = host_cores()
    # the whole workload is one step; keep the run within a few minutes
    t0 = time.perf_counter()
    oracle.run(w.variant, q, k, v, g, b, nthreads=cores)
    one = time.perf_counter() - t0
    steps = args.steps
    warm = max(0, args.warmup - 1)
    budget = 150.0
    if one * (steps + warm) > budget:
        steps = max(1, int(budget / one) - warm)
    for _ in range(warm):
        oracle.run(w.variant, q, k, v, g, b, nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.run(w.variant, q, k, v, g, b, nthreads=cores)
    el = time.perf_counter() - t0
    val = w.tokens * steps / el
    # one thread, on one sequence-head, scaled to the workload's tokens
    sel = lambda a: None if a is None else a.reshape((w.B * w.H,) + a.shape[2:])[:1][None]
    t1 = time.perf_counter()
    oracle.run(w.variant, sel(q), sel(k), sel(v), sel(g), sel(b), nthreads=1)
    # B*T tokens count one token of every head: one sequence-head's T tokens are T/H of them
    one_thread = w.T / w.H / (time.perf_counter() - t1)
    line = {"impl": "reference", "metric": "prefill tokens/s (B*T)", "value": round(val, 2), "unit": "tokens/s",
            "n_gpus": ws, "steps": steps, "warmup": args.warmup, "ms_per_step": round(el / steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy PCG64)",
            "config": {"workload": w.name, "variant": w.variant, "B": w.B, "H": w.H, "T": w.T, "d_k": w.dk,
                       "d_v": w.dv},
            "cpu_baseline": {"value": round(val, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "one_thread_tokens_per_s": round(one_thread, 2),
                             "sample": f"whole workload per step ({w.B * w.H} sequence-heads x {w.T} tokens), "
                                       f"{steps} steps; float64 C recurrence, OpenMP over sequence-heads"},
            "e2e": {"value": round(val, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None, choices=sorted(W.BY_NAME))
    ap.add_argument("--seq-len", type=int, default=0,
                    help="with --only-kernel: the workload at this T (small ncu captures)")
    ap.add_argument("--no-suite", action="store_true")
    ap.add_argument("--only-kernel", action="store_true",
                    help="run warmup + steps of the workload's kernel and nothing else (for ncu)")
    ap.add_argument("--backward", action="store_true",
                    help="with --only-kernel: the normalized backward on its workload's shapes")
    ap.add_argument("--gated-backward", action="store_true",
                    help="with --only-kernel: the gated delta rule's backward (headline shapes, or --workload)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        reference_arm(args)
    elif args.only_kernel:
        kernel_only(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
