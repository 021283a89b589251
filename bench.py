#!/usr/bin/env python
"""Benchmark of the speculative-decoding verification sampler on GB300.

A step is one call of the sampler over one batch (every step of the rule, all
of the call's kernel launches).  The headline workload is the largest
single-GPU one, the long ragged batch: B = 128 requests, K = 8, V = 128256,
f32 logits, draft lengths uniform in 1..8, constant-overlap pairs with alpha
0.5 / 0.8 / 0.95 (synthetic, seeded).  The same invocation also times the
other three workloads the HBM bar applies to (Llama-3-class, greedy,
DeepSeek-V3 MTP) and reports them under "workloads".

Metric: verified rows/s, rows = B*(K+1) per step, whole job (all ranks).
Timing: W eager warm-up steps, then a region of exactly K steps replayed from
CUDA graphs, bracketed by a barrier and a device synchronise and timed with
CUDA events on the launching stream (max over ranks).  The region is
repeated (at least 5 times and at least ~1 s of device time per workload);
ms_per_step is the median region / K, with the spread beside it.  Inputs
rotate over enough device copies to exceed 3x the L2 cache, so every step
streams its logits from HBM.

Also reported: the roofline of the call (algorithmic bytes per call / call
time vs the measured HBM copy bandwidth), acceptance statistics of the
outputs (mean accepted length; per-alpha acceptance rate on the ragged
batch), the same metric end to end through the host-buffer entry point
(pinned host inputs copied in, results copied out, every step; headline
only), SM clocks sampled during each workload's timed regions, and, in the
CPU-baseline leg (rank 0, N = 1), the CPU oracle timed on the host cores plus
the excused-mismatch counts of the GPU outputs against the oracle.

--impl reference times the CPU oracle instead (the only reference this
sampler has), rank 0 only, on bounded samples of the same workload.

Multi-GPU: requests are independent, so each rank runs its own batch (weak
scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "verify rows/s (B×(K+1) rows of V logits) and achieved HBM GB/s vs GB300 peak"
KERNEL_SRC = os.path.join(ROOT, "speculative_decoding_verify_sample_gb300", "csrc", "specverify.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "verify_kernel_traffic.json")
# A call launches four kernels (row statistics, decisions, residual piece
# sums with the bonus draws, residual searches) per sequence of at most 1024
# requests.
KERNELS_PER_SEQUENCE = 4
REQUESTS_PER_SEQUENCE = 1024
FALLBACK_HBM_GBS = 6800.0

WORKLOAD_TEXT = {
    "llama3": "Llama-3-class verify: B=32 K=4 V=128256 bf16, draft~N(0,3^2), target=draft+N(0,1), T=0.7",
    "greedy": "greedy verify: B=256 K=4 V=128256 bf16 N(0,3^2), T=0, target argmax = draft w.p. 0.8",
    "greedy_planted": "greedy verify, planted argmax: B=256 K=4 V=128256 bf16, T=0",
    "dsv3_mtp": "DeepSeek-V3 MTP: B=512 K=1 V=129280 bf16, 25% T=0, else T~U(0,1.2]",
    "ragged": "long ragged: B=128 K=8 V=128256 f32, draft_len~U{1..8}, constant overlap 0.5/0.8/0.95",
    "tiny": "tiny: B=4 K=4 V=1024 f32, T=1",
    "draft_sampler": "draft-side sampler, DeepSeek-class MTP draft step: R=512 rows V=129280 bf16, "
                     "T~U(0,1.2], 25% T=0",
    "onehot": "one-hot (top-token) draft verify: B=128 K=4 V=128256 bf16, T=0.7, 25% T=0",
    "tree_greedy": "greedy token-tree verify: 32 trees x 32 nodes, V=128256 bf16",
    "post_accept_insert": "post-accept insert: B=512 requests, K=4, history L=4096 int32",
}
# workloads of the steps around verification (timed by time_step_workload)
STEP_WORKLOADS = ("draft_sampler", "onehot", "tree_greedy", "post_accept_insert")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="ragged", choices=sorted(WORKLOAD_TEXT),
                    help="headline workload (the JSON line's top level)")
    ap.add_argument("--also", default="llama3,greedy,dsv3_mtp,draft_sampler,onehot,tree_greedy,"
                                      "post_accept_insert",
                    help="comma-separated workloads timed in the same run ('' for none)")
    ap.add_argument("--min-region-s", type=float, default=1.0,
                    help="device time per workload over the repeated K-step regions")
    ap.add_argument("--seed", type=int, default=None)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of CUDA graphs")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps is None:
        args.steps = 200 if args.impl == "ours" else 10
    args.also = [w for w in args.also.split(",") if w and w != args.workload]
    for w in args.also:
        if w not in WORKLOAD_TEXT:
            ap.error(f"unknown workload {w}")
    return args


# ---------------------------------------------------------------- helpers


def required_bytes(inp) -> int:
    """Logit bytes the rule must read: target rows t <= n_b of every request
    and draft rows t < n_b of every sampled request, once each."""
    from speculative_decoding_verify_sample_gb300 import synth
    rows_t, rows_d = synth.rows_needed(inp)
    elt = 2 if inp["dtype"] == "bf16" else 4
    return (rows_t + rows_d) * inp["V"] * elt


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    with open(KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, only if it was
    taken on the current kernel source and this workload."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(workload)
    if not entry or entry.get("source_sha256") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.window = None
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def wait_first(self, timeout=5.0):
        t0 = time.time()
        while self.proc and not self.samples and time.time() - t0 < timeout:
            time.sleep(0.02)

    def start(self):
        self.t0 = time.time()

    def stop(self):
        self.window = (self.t0, time.time())
        time.sleep(0.12)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.samples or self.window is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        lo, hi = self.window
        inside = [s for t, s in self.samples if lo - 0.05 <= t <= hi + 0.05]
        if not inside:   # a timed region shorter than the sampling period
            inside = [min(self.samples, key=lambda ts: abs(ts[0] - (lo + hi) / 2))[1]]
        sm, mx, reasons = [], [], set()
        for s in inside:
            try:
                sm.append(float(s[0]))
                mx.append(float(s[1]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(self.REASONS, s[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(inside)}


def gpu_id_for(torch, dev) -> str:
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:  # noqa: BLE001
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        idx = dev.index or 0
        return vis.split(",")[idx] if vis else str(idx)


# ---------------------------------------------------------------- distributed


def dist_setup(torch):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(torch, world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(torch, world, value: float, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base: int, rank: int) -> int:
    """Seed of a rank's own batch: every rank verifies different requests."""
    return base + rank


def job_rate(rows_per_rank: int, steps: int, world: int, seconds: float) -> float:
    """Whole-job rows/s: the rows every rank verified over the slowest
    rank's time (weak scaling: each rank holds a full batch)."""
    return rows_per_rank * steps * world / seconds


# ---------------------------------------------------------------- arms


def device_inputs(torch, inp, dev):
    def logits(a):
        if a is None:
            return None
        if inp["dtype"] == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)

    def small(a, dt):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dt)).to(dev)

    return dict(target=logits(inp["target"]), draft=logits(inp.get("draft")),
                draft_tokens=small(inp["draft_tokens"], np.int32),
                draft_len=small(inp.get("draft_len"), np.int32),
                temperature=small(inp["temperature"], np.float32),
                uniforms=small(inp["uniforms"], np.float32),
                uniforms_resample=small(inp["uniforms_resample"], np.float32))


def host_inputs(torch, d):
    return {k: (None if v is None else v.cpu().pin_memory()) for k, v in d.items()}


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (x86 "model name"; on Arm the
    implementer and part codes), else the machine type."""
    try:
        with open("/proc/cpuinfo") as f:
            lines = f.read().splitlines()
    except OSError:
        lines = []
    fields = {}
    for line in lines:
        if ":" in line:
            key, val = line.split(":", 1)
            fields.setdefault(key.strip(), val.strip())
    for key in ("model name", "Model", "Hardware"):
        if fields.get(key):
            return fields[key]
    if fields.get("CPU implementer") or fields.get("CPU part"):
        return (f"{platform.machine()} implementer {fields.get('CPU implementer', '?')} "
                f"part {fields.get('CPU part', '?')}")
    return platform.machine() or "unknown"


def cpu_oracle_single_thread_rate(inp, budget_s=0.5):
    """The oracle on one host thread: rows/s over at least one call on the
    first request of the batch."""
    rate, _, _ = cpu_oracle_rate(inp, budget_s=budget_s, nthreads=1, max_requests=1, min_reps=1)
    return rate


def cpu_oracle_rate(inp, budget_s=1.5, nthreads=None, max_requests=None, min_reps=3):
    """The oracle as it stands on the host cores: rows/s over repeated calls
    on a bounded sample (the first m requests of the batch)."""
    import oracle
    nthreads = nthreads or os.cpu_count() or 1
    B = inp["B"]
    m = B if max_requests is None else max(1, min(B, max_requests))
    sub = dict(inp)
    if m < B:
        sub["B"] = m
        for k in ("target", "draft", "draft_tokens", "draft_len", "temperature", "uniforms",
                  "uniforms_resample"):
            if sub.get(k) is not None:
                sub[k] = np.ascontiguousarray(np.asarray(inp[k])[:m])
    oracle.verify_sample(sub, nthreads=nthreads)          # untimed: build + page-in
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.verify_sample(sub, nthreads=nthreads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s and reps >= min_reps:
            break
    rows = reps * m * (inp["K"] + 1)
    return rows / el, nthreads, f"first {m} of {B} requests, {reps} repetitions, {el:.2f} s wall"


def acceptance_stats(inp, acc):
    """Acceptance statistics of one call's outputs (GPU results only): mean
    accepted length and emitted tokens; per constructed alpha, the empirical
    per-position acceptance rate (accepted drafts / accept tests taken)."""
    acc = np.asarray(acc)
    B, K = inp["B"], inp["K"]
    n = np.full(B, K) if inp.get("draft_len") is None else np.asarray(inp["draft_len"])
    ok = acc >= 0
    out = {"mean_accepted_len": round(float(acc[ok].mean()), 4),
           "mean_emitted": round(float(acc[ok].mean() + 1.0), 4),
           "bad_requests": int((~ok).sum())}
    T = np.asarray(inp["temperature"])
    if (T > 0).any() and (T == 0).any():
        for name, sel in (("sampled", T > 0), ("greedy", T == 0)):
            s = sel & ok
            out[f"mean_accepted_len_{name}"] = round(float(acc[s].mean()), 4)
    if inp.get("alpha") is not None:
        per = {}
        for a in sorted(set(np.asarray(inp["alpha"]).tolist())):
            s = (np.asarray(inp["alpha"]) == a) & ok
            tests = np.minimum(acc[s] + 1, n[s]).sum()
            per[str(a)] = {"constructed": a, "empirical": round(float(acc[s].sum() / tests), 4),
                           "accept_tests": int(tests),
                           "mean_emitted": round(float(acc[s].mean() + 1.0), 4),
                           "closed_form_mean_emitted": round(float(np.mean(
                               [(1 - a ** (k + 1)) / (1 - a) for k in n[s]])), 4)}
        out["per_alpha"] = per
    return out


def oracle_parity(inp, acc_g, out_g):
    """CPU-baseline leg: the oracle on the whole workload (untimed) against
    one call's GPU outputs; returns the mismatch counts under the parity rules
    (greedy bit-exact; sampled requests equal except at oracle-flagged
    near-ties, counted per flag)."""
    import oracle
    acc_o, out_o, flags_o = oracle.verify_sample(inp, nthreads=os.cpu_count() or 1)
    T = np.asarray(inp["temperature"])
    mism = (np.asarray(acc_g) != acc_o) | np.any(np.asarray(out_g) != out_o, axis=1)
    allowed = (flags_o & oracle.NEAR_TIE_MASK) != 0
    return {"compared": int(inp["B"]), "sampled": int((T > 0).sum()),
            "mismatched": int(mism.sum()),
            "unexcused": int((mism & (~allowed | (T == 0))).sum()),
            "excused": int((mism & allowed & (T > 0)).sum()),
            "flagged": {name: int(((flags_o & bit) != 0).sum())
                        for bit, name in oracle.FLAG_NAMES.items()}}


def time_workload(args, torch, sv, name, dev, world, rank):
    """Times one workload: W eager warm-ups, then the K-step region replayed
    from CUDA graphs, repeated; returns (summary dict, inp, device inputs,
    workspace, outputs of one call on the first copy)."""
    from speculative_decoding_verify_sample_gb300 import synth
    seed = rank_seed(args.seed if args.seed is not None else synth.DEFAULT_SEED[name], rank)
    inp = synth.make_inputs(name, seed)
    B, K, V = inp["B"], inp["K"], inp["V"]
    rows_per_step = B * (K + 1)
    req_bytes = required_bytes(inp)
    d0 = device_inputs(torch, inp, dev)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_copies = max(1, math.ceil(3 * l2 / max(req_bytes, 1)))
    copies = [d0]
    for _ in range(n_copies - 1):
        copies.append({k: (v.clone() if v is not None and k in ("target", "draft") else v)
                       for k, v in d0.items()})
    ws = sv.Workspace(B, K, V, inp["dtype"], dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty((B, K + 1), dtype=torch.int32, device=dev)

    def step(i):
        c = copies[i % n_copies]
        sv.spec_verify_sample(c["target"], c["draft"], c["draft_tokens"], c["draft_len"],
                              c["temperature"], c["uniforms"], c["uniforms_resample"],
                              workspace=ws, accepted_len=acc, out_tokens=out)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    status = ws.read_status()
    if status:
        raise RuntimeError(f"{name}: device status {status:#x} after warm-up")

    K_steps = args.steps
    stream = torch.cuda.current_stream(dev)
    graphs = []
    if not args.no_graph:
        cycle = n_copies * max(1, 64 // n_copies)
        full, rem = divmod(K_steps, cycle)

        def capture(nsteps):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in range(nsteps):
                    step(i)
            return g

        g_cycle = capture(cycle) if full else None
        g_rem = capture(rem) if rem else None
        graphs = [g_cycle] * full + ([g_rem] if g_rem else [])
        graphs[0].replay()      # one untimed replay of the captured graph
        torch.cuda.synchronize(dev)

    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)

    def region():
        """Exactly K steps between a barrier + synchronise on both sides."""
        barrier(torch, world)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        if graphs:
            for g in graphs:
                g.replay()
        else:
            for i in range(K_steps):
                step(i)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(torch, world)
        return max_over_ranks(torch, world, ev0.elapsed_time(ev1), dev)

    first = region()          # calibration (untimed): sets the repeat count
    reps = int(min(2000, max(5, math.ceil(args.min_region_s * 1e3 / max(first, 1e-3)))))
    reps = int(max_over_ranks(torch, world, float(reps), dev))
    clocks = None
    if not args.no_clocks:
        clocks = ClockSampler(gpu_id_for(torch, dev))
        clocks.wait_first()
        clocks.start()
    times = [region() for _ in range(reps)]
    if clocks:
        clocks.stop()
    status = ws.read_status()
    if status:
        raise RuntimeError(f"{name}: device status {status:#x} after the timed regions")

    # inputs that fit twice in L2: the same K steps on one copy of the
    # logits as well (L2-hot), reported beside the graded rotating number
    hot = None
    if req_bytes < 2 * l2 and graphs:
        def step_hot(i):
            c = copies[0]
            sv.spec_verify_sample(c["target"], c["draft"], c["draft_tokens"], c["draft_len"],
                                  c["temperature"], c["uniforms"], c["uniforms_resample"],
                                  workspace=ws, accepted_len=acc, out_tokens=out)
        g_hot = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_hot):
            for i in range(K_steps):
                step_hot(i)
        g_hot.replay()
        torch.cuda.synchronize(dev)
        hot_times = []
        for _ in range(max(5, min(reps, 200))):
            barrier(torch, world)
            torch.cuda.synchronize(dev)
            ev0.record(stream)
            g_hot.replay()
            ev1.record(stream)
            torch.cuda.synchronize(dev)
            barrier(torch, world)
            hot_times.append(max_over_ranks(torch, world, ev0.elapsed_time(ev1), dev))
        hot_ms = statistics.median(hot_times) / K_steps
        hot = {"ms_per_step": round(hot_ms, 6),
               "value": round(job_rate(rows_per_step, K_steps, world, hot_ms * K_steps / 1e3), 1),
               "unit": "rows/s", "inputs": "one device copy of the logits, L2-resident (not graded)"}
        del g_hot

    times.sort()
    ms = statistics.median(times)
    ms_per_step = ms / K_steps
    value = job_rate(rows_per_step, K_steps, world, ms / 1e3)
    achieved = req_bytes / (ms_per_step / 1e3) / 1e9
    peak, peak_src = measured_hbm_peak()

    # one more call on the first copy, for the outputs' statistics
    c = copies[0]
    acc1, out1 = sv.spec_verify_sample(c["target"], c["draft"], c["draft_tokens"], c["draft_len"],
                                       c["temperature"], c["uniforms"], c["uniforms_resample"],
                                       workspace=ws)
    torch.cuda.synchronize(dev)
    acc1, out1 = acc1.cpu().numpy(), out1.cpu().numpy()

    def pct(q):
        return round(times[min(len(times) - 1, int(q * (len(times) - 1) + 0.5))] / K_steps, 6)

    summary = {
        "workload": WORKLOAD_TEXT[name], "B": B, "K": K, "V": V, "logits_dtype": inp["dtype"],
        "value": round(value, 1), "unit": "rows/s", "ms_per_step": round(ms_per_step, 6),
        "ms_per_step_spread": {"min": pct(0.0), "p10": pct(0.1), "median": round(ms_per_step, 6),
                               "p90": pct(0.9), "max": pct(1.0), "regions": reps,
                               "steps_per_region": K_steps},
        "rows_per_step": rows_per_step, "required_bytes_per_step": req_bytes,
        "l2": f"rotating {n_copies} device copies of the logits "
              f"({n_copies * req_bytes / 1e6:.0f} MB read per cycle, L2 {l2 / 1e6:.0f} MB)",
        "launch": "CUDA graphs of the step launches" if graphs else "eager launches",
        "kernel_plan": sv.launch_plan(B, K, V, inp["dtype"], inp.get("draft") is not None),
        "roofline": {
            "kernel": "spec_verify_sample (stats_kernel + decide_kernel + residual_kernel + search_kernel, one call, timed together)",
            "bound": "hbm", "achieved": round(achieved, 1),
            "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic(name),
            "peak_source": f"{peak_src} HBM copy bandwidth ({'of measured' if peak_src == 'measured' else 'of fallback'})",
            "algorithmic_bytes_per_launch": req_bytes},
        "gpu_launches": K_steps * KERNELS_PER_SEQUENCE * math.ceil(B / REQUESTS_PER_SEQUENCE),
        "acceptance": acceptance_stats(inp, acc1),
    }
    if hot:
        summary["l2_hot"] = hot
    if clocks:
        summary["clocks"] = clocks.summary()
    del copies, graphs
    return summary, inp, d0, ws, (acc1, out1)


def time_graph_steps(args, torch, dev, world, step, n_copies):
    """W eager warm-ups of step(i), then the K-step region from CUDA graphs
    (rotating over n_copies inputs), repeated >= 5 times and ~min_region_s
    of device time; returns (sorted region times in ms, clock summary)."""
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    K_steps = args.steps
    stream = torch.cuda.current_stream(dev)
    cycle = n_copies * max(1, 64 // n_copies)
    full, rem = divmod(K_steps, cycle)

    def capture(nsteps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(nsteps):
                step(i)
        return g

    graphs = []
    if not args.no_graph:
        graphs = ([capture(cycle)] * full if full else []) + ([capture(rem)] if rem else [])
        graphs[0].replay()
        torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)

    def region():
        barrier(torch, world)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        if graphs:
            for g in graphs:
                g.replay()
        else:
            for i in range(K_steps):
                step(i)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(torch, world)
        return max_over_ranks(torch, world, ev0.elapsed_time(ev1), dev)

    first = region()
    reps = int(min(2000, max(5, math.ceil(args.min_region_s * 1e3 / max(first, 1e-3)))))
    reps = int(max_over_ranks(torch, world, float(reps), dev))
    clocks = None
    if not args.no_clocks:
        clocks = ClockSampler(gpu_id_for(torch, dev))
        clocks.wait_first()
        clocks.start()
    times = sorted(region() for _ in range(reps))
    if clocks:
        clocks.stop()
    return times, (clocks.summary() if clocks else None)


def summarize_times(times, K_steps):
    ms = statistics.median(times)

    def pct(q):
        return round(times[min(len(times) - 1, int(q * (len(times) - 1) + 0.5))] / K_steps, 6)

    return ms / K_steps, {"min": pct(0.0), "p10": pct(0.1), "median": round(ms / K_steps, 6),
                          "p90": pct(0.9), "max": pct(1.0), "regions": len(times),
                          "steps_per_region": K_steps}


def time_step_workload(args, torch, sv, name, dev, world, rank, cpu_leg):
    """The steps around verification: the draft-side sampler, the one-hot
    draft rule, greedy token trees, the post-accept insert.  Same timing as
    the verification workloads; parity against the oracle in the CPU leg."""
    from speculative_decoding_verify_sample_gb300 import synth
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    seed = rank_seed(args.seed if args.seed is not None else 7, rank)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)   # noqa: E731
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)  # noqa: E731

    def logits(a, dtype):
        return device_inputs(torch, {"dtype": dtype, "target": a, "draft": None,
                                     "draft_tokens": None, "draft_len": None, "temperature": None,
                                     "uniforms": None, "uniforms_resample": None}, dev)["target"]

    parity = None
    stats = {}
    if name == "draft_sampler":
        d = synth.draft_rows(seed, 512, 129280, "bf16")
        units, unit_name = d["R"], "rows/s"
        req = d["R"] * d["V"] * 2
        base = logits(d["logits"], "bf16")
        n_copies = max(1, math.ceil(3 * l2 / req))
        copies = [base] + [base.clone() for _ in range(n_copies - 1)]
        T, U = f32(d["temperature"]), f32(d["uniforms"])
        ws = sv.Workspace(d["R"], 0, d["V"], "bf16", dev, kind="sample")
        tok = torch.empty(d["R"], dtype=torch.int32, device=dev)

        def step(i):
            sv.sample_draft(copies[i % n_copies], T, U, workspace=ws, tokens=tok)

        def outputs():
            return sv.sample_draft(copies[0], T, U, workspace=ws).cpu().numpy()

        if cpu_leg:
            import oracle
            got = outputs()
            want, flags = oracle.sample_draft(d["logits"], "bf16", d["temperature"], d["uniforms"],
                                              nthreads=os.cpu_count() or 1)
            mism = got != want
            allowed = (flags & oracle.NEAR_TIE_MASK) != 0
            parity = {"compared": d["R"], "mismatched": int(mism.sum()),
                      "unexcused": int((mism & (~allowed | (d["temperature"] == 0))).sum())}
    elif name == "onehot":
        inp = synth.onehot_case(seed, 128, 4, 128256, "bf16", temperature=0.7, greedy_frac=0.25)
        units, unit_name = inp["B"] * (inp["K"] + 1), "rows/s"
        req = required_bytes(inp)
        d0 = device_inputs(torch, inp, dev)
        n_copies = max(1, math.ceil(3 * l2 / req))
        copies = [d0["target"]] + [d0["target"].clone() for _ in range(n_copies - 1)]
        ws = sv.Workspace(inp["B"], inp["K"], inp["V"], "bf16", dev)
        acc = torch.empty(inp["B"], dtype=torch.int32, device=dev)
        out = torch.empty((inp["B"], inp["K"] + 1), dtype=torch.int32, device=dev)

        def step(i):
            sv.spec_verify_sample_onehot(copies[i % n_copies], d0["draft_tokens"], d0["draft_len"],
                                         d0["temperature"], d0["uniforms"],
                                         d0["uniforms_resample"], workspace=ws, accepted_len=acc,
                                         out_tokens=out)

        step(0)
        torch.cuda.synchronize(dev)
        stats = {"acceptance": acceptance_stats(inp, acc.cpu().numpy())}
        if cpu_leg:
            import oracle
            a_o, o_o, fl = oracle.verify_onehot(inp, nthreads=os.cpu_count() or 1)
            a_g, o_g = acc.cpu().numpy(), out.cpu().numpy()
            mism = (a_g != a_o) | np.any(o_g != o_o, axis=1)
            allowed = (fl & oracle.NEAR_TIE_MASK) != 0
            parity = {"compared": inp["B"], "mismatched": int(mism.sum()),
                      "unexcused": int((mism & (~allowed | (inp["temperature"] == 0))).sum())}
    elif name == "tree_greedy":
        c = synth.tree_case(seed, 32, 32, 128256, "bf16")
        units, unit_name = c["B"] * c["N"], "rows/s"
        req = int(c["n_nodes"].sum()) * c["V"] * 2
        base = logits(c["target"], "bf16")
        n_copies = max(1, math.ceil(3 * l2 / req))
        copies = [base] + [base.clone() for _ in range(n_copies - 1)]
        par, tokn, nn = i32(c["parents"]), i32(c["tokens"]), i32(c["n_nodes"])
        ws = sv.Workspace(c["B"], c["N"], c["V"], "bf16", dev, kind="tree")
        acc = torch.empty(c["B"], dtype=torch.int32, device=dev)
        out = torch.empty((c["B"], c["N"]), dtype=torch.int32, device=dev)
        path = torch.empty((c["B"], c["N"]), dtype=torch.int32, device=dev)

        def step(i):
            sv.verify_tree_greedy(copies[i % n_copies], par, tokn, nn, workspace=ws,
                                  accepted_len=acc, out_tokens=out, path_nodes=path)

        step(0)
        torch.cuda.synchronize(dev)
        stats = {"acceptance": {"mean_accepted_len": round(float(acc.float().mean()), 4)}}
        if cpu_leg:
            import oracle
            a_o, o_o, p_o = oracle.tree_greedy(c["target"], "bf16", c["parents"], c["tokens"],
                                               c["n_nodes"], nthreads=os.cpu_count() or 1)
            mism = ((acc.cpu().numpy() != a_o) | np.any(out.cpu().numpy() != o_o, axis=1)
                    | np.any(path.cpu().numpy() != p_o, axis=1))
            parity = {"compared": c["B"], "mismatched": int(mism.sum()), "unexcused": int(mism.sum())}
    else:   # post_accept_insert
        rng = np.random.default_rng(seed)
        B, K, L = 512, 4, 4096
        acc_h = rng.integers(0, K + 1, size=B).astype(np.int32)
        out_h = rng.integers(0, 128256, size=(B, K + 1)).astype(np.int32)
        seq0 = rng.integers(0, 64, size=B).astype(np.int32)
        units, unit_name = B, "requests/s"
        req = B * 4 + B * (K + 1) * 4 + B * 8 + B * 4 * 3 + int((acc_h + 1).sum()) * 8 + (B + 1) * 4
        n_copies = 1
        acc_d, out_d = i32(acc_h), i32(out_h)
        seq_d = i32(seq0)
        hist = torch.zeros((B, L), dtype=torch.int32, device=dev)
        nxt = torch.empty(B, dtype=torch.int32, device=dev)
        cu = torch.empty(B + 1, dtype=torch.int32, device=dev)
        packed = torch.empty(B * (K + 1), dtype=torch.int32, device=dev)
        st = torch.empty(B, dtype=torch.int32, device=dev)

        def step(i):
            # the lengths rewind every 64 steps (inside a captured graph: a
            # device copy), so the histories never fill
            if i % 64 == 0:
                seq_d.fill_(0)
            sv.insert_accepted(acc_d, out_d, seq_d, hist, next_tokens=nxt, cu_emitted=cu,
                               packed=packed, status=st)

        if cpu_leg:
            import oracle
            seq_d.fill_(0)
            hist.zero_()
            sv.insert_accepted(acc_d, out_d, seq_d, hist, next_tokens=nxt, cu_emitted=cu,
                               packed=packed, status=st)
            torch.cuda.synchronize(dev)
            s_o, h_o, n_o, c_o, p_o, st_o = oracle.insert_accepted(
                acc_h, out_h, np.zeros(B, np.int32), np.zeros((B, L), np.int32))
            ok = (np.array_equal(hist.cpu().numpy(), h_o) and np.array_equal(nxt.cpu().numpy(), n_o)
                  and np.array_equal(cu.cpu().numpy(), c_o)
                  and np.array_equal(packed.cpu().numpy()[:c_o[-1]], p_o[:c_o[-1]]))
            parity = {"compared": B, "mismatched": 0 if ok else B, "unexcused": 0 if ok else B}
    times, clocks = time_graph_steps(args, torch, dev, world, step, n_copies)
    ms_per_step, spread = summarize_times(times, args.steps)
    peak, peak_src = measured_hbm_peak()
    achieved = req / (ms_per_step / 1e3) / 1e9
    out = {"workload": WORKLOAD_TEXT[name], "value": round(units / (ms_per_step / 1e3) * world, 1),
           "unit": unit_name, "ms_per_step": round(ms_per_step, 6), "ms_per_step_spread": spread,
           "required_bytes_per_step": req,
           "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(achieved / peak, 4),
                        "peak_source": f"{peak_src} HBM copy bandwidth",
                        "algorithmic_bytes_per_launch": req}}
    if name == "post_accept_insert":
        out["roofline"]["note"] = "one CTA, latency-bound: bytes moved are a few kB"
    out.update(stats)
    if clocks:
        out["clocks"] = clocks
    if parity is not None:
        out["parity"] = parity
    return out


def run_ours(args, torch, world, rank, local):
    import speculative_decoding_verify_sample_gb300 as sv

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sv.build()
    cpu_leg = rank == 0 and world == 1 and not args.no_cpu_baseline
    if args.workload in STEP_WORKLOADS:   # one of the steps around verification, alone
        summ = time_step_workload(args, torch, sv, args.workload, dev, world, rank, cpu_leg)
        line = {"metric": METRIC, "value": summ["value"], "unit": summ["unit"], "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": summ["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic (seeded; logits generated, no model weights)",
                "config": {"workload": summ["workload"],
                           "required_bytes_per_step": summ["required_bytes_per_step"]},
                "roofline": summ["roofline"], "ms_per_step_spread": summ["ms_per_step_spread"]}
        for k in ("clocks", "parity", "acceptance"):
            if k in summ:
                line[k] = summ[k]
        return line
    head, inp, d0, ws, outs = time_workload(args, torch, sv, args.workload, dev, world, rank)
    line = {
        "metric": METRIC, "value": head["value"], "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; logits generated, no model weights)",
        "config": {k: head[k] for k in ("workload", "B", "K", "V", "logits_dtype", "rows_per_step",
                                        "required_bytes_per_step", "l2", "launch", "kernel_plan")},
        "ms_per_step_spread": head["ms_per_step_spread"],
        "roofline": head["roofline"],
        "gpu_launches": head["gpu_launches"],
        "acceptance": head["acceptance"],
    }
    line["config"]["parallelism"] = f"{world} independent replica(s), requests sharded per rank"
    if "l2_hot" in head:
        line["l2_hot"] = head["l2_hot"]
    if "clocks" in head:
        line["clocks"] = head["clocks"]
    if not args.no_e2e:
        line["e2e"] = e2e_rate(args, torch, sv, inp, d0, dev, ws, head["rows_per_step"], world)
    if cpu_leg:
        v, cores, sample = cpu_oracle_rate(inp, budget_s=10.0)
        line["cpu_baseline"] = {"value": round(v, 1), "unit": "rows/s", "cores": cores,
                                "kind": "oracle", "sample": sample,
                                "single_thread_value": round(cpu_oracle_single_thread_rate(inp), 1),
                                "cpu_model": cpu_model()}
        line["parity"] = oracle_parity(inp, *outs)
    del d0, ws
    torch.cuda.empty_cache()
    extra = {}
    for name in args.also:
        if name in STEP_WORKLOADS:
            extra[name] = time_step_workload(args, torch, sv, name, dev, world, rank, cpu_leg)
            torch.cuda.empty_cache()
            continue
        summ, inp_w, d_w, ws_w, outs_w = time_workload(args, torch, sv, name, dev, world, rank)
        if cpu_leg:
            summ["parity"] = oracle_parity(inp_w, *outs_w)
        extra[name] = summ
        del inp_w, d_w, ws_w
        torch.cuda.empty_cache()
    if extra:
        line["workloads"] = extra
    return line


def e2e_rate(args, torch, sv, inp, d0, dev, ws, rows_per_step, world):
    """Same metric through the host-buffer entry point: every step copies
    that step's inputs from pinned host memory and reads the results back."""
    h = host_inputs(torch, d0)
    B, K, V = inp["B"], inp["K"], inp["V"]
    staging = sv.HostStaging(B, K, V, inp["dtype"], with_draft=h["draft"] is not None, device=dev)
    acc = torch.empty(B, dtype=torch.int32).pin_memory()
    out = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()

    def step():
        sv.spec_verify_sample_host(h["target"], h["draft"], h["draft_tokens"], h["draft_len"],
                                   h["temperature"], h["uniforms"], h["uniforms_resample"],
                                   staging=staging, workspace=ws, accepted_len=acc,
                                   out_tokens=out)

    for _ in range(3):
        step()
    n = max(1, min(args.e2e_steps, args.steps))
    barrier(torch, world)
    t0 = time.perf_counter()
    for _ in range(n):
        step()
    el = time.perf_counter() - t0
    el = max_over_ranks(torch, world, el, dev)
    # the library copies the logit rows the kernels read (required_bytes) and
    # every small input array whole
    h2d = required_bytes(inp) + sum(v.numel() * v.element_size() for k, v in h.items()
                                    if v is not None and k not in ("target", "draft"))
    d2h = acc.numel() * 4 + out.numel() * 4
    return {"value": round(job_rate(rows_per_step, n, world, el), 1), "unit": "rows/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": n,
            "path": "spec_verify_sample_host (pinned host buffers, synchronous per step)"}


def run_reference(args, world, rank):
    """The CPU oracle as it stands, timed on the host cores (rank 0 only)."""
    from speculative_decoding_verify_sample_gb300 import synth
    import oracle

    if rank != 0:
        return None
    seed = args.seed if args.seed is not None else synth.DEFAULT_SEED[args.workload]
    inp = synth.make_inputs(args.workload, seed)
    B, K, V = inp["B"], inp["K"], inp["V"]
    nthreads = os.cpu_count() or 1
    oracle.build()
    t0 = time.perf_counter()
    oracle.verify_sample(inp, nthreads=nthreads)               # calibration, untimed
    per_req = (time.perf_counter() - t0) / B
    budget = 90.0
    m = int(max(1, min(B, budget / max(per_req * (args.steps + args.warmup), 1e-9))))
    sub = dict(inp, B=m)
    for k in ("target", "draft", "draft_tokens", "draft_len", "temperature", "uniforms",
              "uniforms_resample"):
        if inp.get(k) is not None:
            sub[k] = np.ascontiguousarray(np.asarray(inp[k])[:m])
    for _ in range(args.warmup):
        oracle.verify_sample(sub, nthreads=nthreads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.verify_sample(sub, nthreads=nthreads)
    el = time.perf_counter() - t0
    rows = m * (K + 1) * args.steps
    value = rows / el
    sample = f"first {m} of {B} requests per step"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "rows/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; logits generated, no model weights)",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "B": B, "K": K, "V": V,
                   "logits_dtype": inp["dtype"], "rows_per_step": m * (K + 1),
                   "parallelism": "CPU oracle, rank 0 only"},
        "cpu_baseline": {"value": round(value, 1), "unit": "rows/s", "cores": nthreads,
                         "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 1), "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    import torch
    world, rank, local = dist_setup(torch)
    try:
        line = run_ours(args, torch, world, rank, local)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
