"""Throughput of batched speculative verification on GB300.

Default workload: block-diffusion verification, B=64 requests per GPU,
gamma=16 draft tokens, V=131072, bf16 logits, T=1 (synthetic, seeded).  One
step = one spec_verify call over the whole batch (plan, row statistics,
accept / first rejection, residual or bonus draw).  The JSON line also carries
the schedulers' per-call device times, a schedule-then-verify step on the
scheduled ragged workload, and the same step with D-cut, dense packing and
packed verification.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun every rank verifies its own
batch (weak scaling, no collective on the data path); the reported time is
the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified rows/sec at B=64,γ=16,V=128k bf16; achieved HBM GB/s as % of GB300 peak"
UNIT = "verified rows/s"
WORKLOAD = "block_diffusion"
SEED_OFFSET = 0           # --seed-offset
COST_READING = "Bprime"   # --cost-table
PROFILE_RECORD = os.path.join(ROOT, "profiles", "row_stats_block_diffusion.json")
KERNEL_SOURCES = ["speculative_decoding_verification_softmax_gb300/csrc/specv_rowstats.cuh",
                  "speculative_decoding_verification_softmax_gb300/csrc/specv_common.cuh"]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak_gbs():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def profiled_traffic():
    """DRAM bytes per launch of the row-statistics kernel from the committed
    ncu record, or None if the kernel source changed since the capture."""
    try:
        with open(PROFILE_RECORD) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha") != kernel_source_hash():
        return None
    return float(rec["traffic_bytes_per_launch"])


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------- distributed
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(x: float, world: int, device) -> float:
    """Max of x over all ranks (the slowest rank's time); device is where the
    collective's tensor lives (cuda for NCCL, cpu for gloo)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(ms_per_step_max: float, units_per_rank: int, world: int) -> float:
    """Whole-job throughput: units of all ranks over the slowest rank's time."""
    return units_per_rank * world / (ms_per_step_max / 1e3)


# -------------------------------------------------------------- CPU oracle
def time_oracle(case, requests: list[int], cores: int) -> float:
    """Wall time of the oracle over the given requests, split across threads."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    chunks = [requests[i::cores] for i in range(cores) if requests[i::cores]]

    def run(rs):
        for b in rs:
            oracle.verify(case.target, case.draft, case.dtype, case.draft_tokens, case.verify_len, case.T,
                          case.uniforms, b0=b, b1=b + 1)

    t0 = time.perf_counter()
    with ThreadPoolExecutor(len(chunks)) as ex:
        list(ex.map(run, chunks))
    return time.perf_counter() - t0


def cpu_baseline(case, cores: int) -> dict:
    reqs = list(range(case.B))
    # whole batches until about 10 s of CPU work (at most 20 batches)
    dt, reps = 0.0, 0
    while reps < 20 and (reps == 0 or dt * cores < 10.0):
        dt += time_oracle(case, reqs, cores)
        reps += 1
    dt /= reps
    # the oracle as defined, on one thread: four requests of the same batch
    one = list(range(min(4, case.B)))
    dt1 = time_oracle(case, one, 1)
    return {"value": len(reqs) * case.gamma / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"the full batch ({case.B} requests, {case.B * (2 * case.gamma + 1)} logit rows) "
                      f"of the {WORKLOAD} workload {reps} times, requests split across {cores} host "
                      f"threads; mean time per batch",
            "seconds": dt,
            "single_thread": {"value": len(one) * case.gamma / dt1, "unit": UNIT, "cores": 1,
                              "sample": f"requests 0..{len(one) - 1} of the same batch on one thread",
                              "seconds": dt1}}


# ------------------------------------------------------------------- main
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import specsynth
    o = SEED_OFFSET
    case = specsynth.make_verify_case(WORKLOAD, seed_logits=300 + o, seed_noise=301 + o, seed_tokens=302 + o,
                                      seed_uniforms=303 + o)
    cores = os.cpu_count() or 1
    per_step = min(case.B, cores)
    W = max(args.warmup, 0)
    for s in range(W):
        time_oracle(case, [(s * per_step + i) % case.B for i in range(per_step)], cores)
    t = 0.0
    for s in range(args.steps):
        t += time_oracle(case, [((W + s) * per_step + i) % case.B for i in range(per_step)], cores)
    ms = t / args.steps * 1e3
    value = per_step * case.gamma / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": W, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(case),
            "cpu_baseline": {"kind": "oracle", "cores": cores, "value": value, "unit": UNIT,
                             "sample": f"{per_step} requests of the {WORKLOAD} batch per step, "
                                       f"one host thread each"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(case):
    logit_bytes = case.B * (2 * case.gamma + 1) * case.V * 2
    return {"workload": f"{WORKLOAD} verify: B={case.B} per GPU, gamma={case.gamma}, V={case.V}, "
                        f"bf16 logits, T={case.T:g}, verify_len=gamma",
            "B_per_gpu": case.B, "gamma": case.gamma, "V": case.V, "storage": "bf16",
            "l2": f"inputs larger than L2 ({logit_bytes / 1e6:.1f} MB of logits read per step)"}


SCHED_REPLAYS = 200
PREROLL_STEPS = 20        # untimed calls right before the timed ones


def time_schedulers(sv, dev, stream, rank: int):
    """Device time per call of each scheduler on the scheduled workload
    (B=64, gamma=16 confidences, min_len=1): SCHED_REPLAYS calls captured in one
    CUDA graph, replayed, timed with CUDA events on the launching stream."""
    import torch
    import specsynth
    conf = specsynth.make_confidences(seed=specsynth.SCHED_SEED + 1000 * rank + SEED_OFFSET)
    B, gamma = conf.shape
    c = torch.from_numpy(conf).to(dev)
    out = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    cost = specsynth.COST_TABLES[COST_READING]
    ratios, rcost = [0.25, 0.5, 0.75, 1.0], [10.0, 13.0, 16.0, 19.0]
    sts = np.linspace(0.8, 1.6, gamma).astype(np.float32)
    ml = specsynth.SCHED_MIN_LEN
    modes = {
        "exact": lambda: sv.schedule(c, cost, ml, sv.SCHED_EXACT, out_verify_len=out, workspace=ws),
        "algorithm1": lambda: sv.schedule(c, cost, ml, sv.SCHED_ALGORITHM1, out_verify_len=out, workspace=ws),
        "dcut": lambda: sv.schedule(c, (ratios, rcost), ml, sv.SCHED_DCUT, out_verify_len=out, workspace=ws),
        "exact_sts": lambda: sv.schedule(c, cost, ml, sv.SCHED_EXACT, sts=sts, out_verify_len=out, workspace=ws),
        "static_threshold": lambda: sv.schedule_static(c, 0.6, gamma, ml, out_verify_len=out, workspace=ws),
        "static_threshold_sts": lambda: sv.schedule_static(c, 0.6, gamma, ml, sts=sts, out_verify_len=out,
                                                           workspace=ws),
    }
    res = {}
    for name, call in modes.items():
        for _ in range(3):
            call()
        torch.cuda.synchronize(dev)
        if sv.read_status(ws) != 0:
            raise RuntimeError(f"scheduler status ({name})")
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for _ in range(SCHED_REPLAYS):
                    call()
        stream.wait_stream(side)
        g.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(side):
            e0.record(side)
            for _ in range(5):
                g.replay()
            e1.record(side)
        torch.cuda.synchronize(dev)
        res[name] = {"us_per_call": e0.elapsed_time(e1) * 1e3 / (5 * SCHED_REPLAYS),
                     "mean_verify_len": float(out.float().mean().item())}
        if sv.read_status(ws) != 0:
            raise RuntimeError(f"scheduler status after replay ({name})")
    return {"workload": f"scheduled ragged: B={B}, gamma={gamma} confidences sigmoid(N(1.5, 1)), "
                        f"min_len={ml}; cost table reading {COST_READING} of 8 ms + 0.02 ms/token, +12 ms above 512 tokens; "
                        f"D-cut ratios {ratios} with costs {rcost} ms; STS temperatures 0.8..1.6",
            "timing": f"{SCHED_REPLAYS} calls per CUDA graph, 5 replays, CUDA events",
            "kernel_launches_per_call": 1, "modes": res}


def graph_us_per_call(dev, stream, call, n_calls: int = 50, reps: int = 5) -> float:
    """Device time per call: n_calls calls (call(i) for i in range(n_calls))
    captured in one CUDA graph on a side stream, replayed reps times between
    CUDA events."""
    import torch
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for i in range(n_calls):
                call(i)
    stream.wait_stream(side)
    g.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(side):
        e0.record(side)
        for _ in range(reps):
            g.replay()
        e1.record(side)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) * 1e3 / (reps * n_calls)


def head_start(n_calls: int, host_us_per_call: float = 100.0) -> None:
    """Keep the GPU busy (a device-side sleep, launched before any event of
    the loop that follows) while the host enqueues the next n_calls calls, so
    that those calls run back to back and no host launch gap falls inside an
    event bracket."""
    import torch
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:
        sleep(int(n_calls * host_us_per_call * 1e-6 * 2.2e9))  # cycles at up to 2.2 GHz


def event_floor_ms(dev, stream, n: int = 50) -> float | None:
    """Median time between the two events of a pair around an empty kernel,
    launched back to back: what an event bracket adds to any kernel's
    duration on this GPU (context for the event-bracketed kernel times)."""
    import torch
    sleep = getattr(torch.cuda, "_sleep", None)  # a private PyTorch helper: report nothing without it
    if sleep is None:
        return None
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize(dev)
    head_start(n, 20.0)
    for a, b in pairs:
        a.record(stream)
        sleep(0)
        b.record(stream)
    torch.cuda.synchronize(dev)
    return float(np.median([a.elapsed_time(b) for a, b in pairs]))


def row_stats_ms(sv, dev, stream, call, n: int) -> float:
    """Mean duration of the row-statistics kernel over n host-launched calls
    (call(i)), from an event pair recorded on the launching stream right
    before and after that kernel in each call (spec_profile_events)."""
    import torch
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in pairs:          # create the events before they are timed
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    head_start(n)
    for i, (a, b) in enumerate(pairs):
        sv.profile_events(a, b)
        call(i)
    torch.cuda.synchronize(dev)
    sv.profile_events(None, None)
    return sum(a.elapsed_time(b) for a, b in pairs) / n


def roofline_entry(alg_bytes: float, ms: float, launches: int, floor_ms: float | None = None) -> dict:
    peak, peak_kind = measured_peak_gbs()
    achieved = alg_bytes / (ms / 1e3) / 1e9
    return {"kernel": "k_row_stats", "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "algorithmic_bytes_per_launch": alg_bytes, "avg_launch_ms": ms,
            "launches_timed": launches, "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
            "event_pair_floor_ms": floor_ms}


def time_other_workloads(sv, specsynth, dev, stream, rank: int):
    """Device time per call of the other verification workloads (the small
    ones are latency-bound): 100 calls captured in a CUDA graph and replayed,
    inputs rotated over copies so that each call's working set exceeds twice
    the L2 where that takes at most 32 copies."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = {}
    for name in ("tiny", "mtp_chat", "greedy"):
        case = specsynth.make_verify_case(name)
        B, gamma, V = case.B, case.gamma, case.V
        bytes_call = case.target.nbytes + (case.draft.nbytes if case.T != 0 else 0)
        n_sets = max(1, min(32, -(-2 * l2 // bytes_call)))
        sets = [specsynth.to_device(case, dev) for _ in range(n_sets)]
        dt = sv.BF16 if case.dtype == "bf16" else sv.F32
        ws = sv.alloc_verify_workspace(B, gamma, V, dt, dev)
        ot = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
        on = torch.empty((B,), dtype=torch.int32, device=dev)

        def call(i):
            t, d, x, vl, u = sets[i % n_sets]
            sv.verify(t, d, x, vl, case.T, u if case.T != 0 else None, out_tokens=ot, out_accept_len=on,
                      workspace=ws)

        for i in range(3):
            call(i)
        torch.cuda.synchronize(dev)
        n_calls = 100
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for i in range(n_calls):
                    call(i)
        stream.wait_stream(side)
        g.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(side):
            e0.record(side)
            for _ in range(5):
                g.replay()
            e1.record(side)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / (5 * n_calls)
        if sv.read_status(ws) != 0:
            raise RuntimeError(f"device status on {name}")
        out[name] = {"shape": f"B={B}, gamma={gamma}, V={V}, {case.dtype}, T={case.T:g}",
                     "us_per_call": us, "verified_rows_per_s": B * gamma / (us / 1e6),
                     "logit_bytes_per_call": bytes_call, "input_copies": n_sets,
                     "l2_note": "working set > 2x L2" if n_sets * bytes_call > 2 * l2 else "L2-resident"}
        del sets
    return {"timing": "100 calls in a CUDA graph, 5 replays, CUDA events", "workloads": out}


def time_packed_step(sv, specsynth, case, t, d, x, u, dev, stream, rank: int, steps: int):
    """D-cut budget, dense packing and verification on packed logits: the
    deployed path of the scheduled workload.  The ratio costs C(B, rho) are the
    round-cost table at the budgets K_rho; the packed logits are gathered once
    from the padded batch (what the target model would write), outside the
    timed region."""
    import math
    import torch
    B, gamma, V = case.B, case.gamma, case.V
    conf = torch.from_numpy(specsynth.make_confidences(seed=specsynth.SCHED_SEED + 1000 * rank + SEED_OFFSET)).to(dev)
    kt, kc = specsynth.COST_TABLES[COST_READING]
    ratios = [0.25, 0.5, 0.75, 1.0]
    budgets = [max(B, math.ceil(r * B * (gamma + 1))) for r in ratios]
    costs = [float(np.interp(k, kt, kc)) for k in budgets]
    vl = torch.empty((B,), dtype=torch.int32, device=dev)
    sws = torch.zeros(256, dtype=torch.uint8, device=dev)
    tr = torch.empty((B,), dtype=torch.int32, device=dev)
    dr = torch.empty((B,), dtype=torch.int32, device=dev)
    tot = torch.empty((2,), dtype=torch.int32, device=dev)
    sv.schedule(conf, (ratios, costs), 0, sv.SCHED_DCUT, out_verify_len=vl, workspace=sws)
    sv.pack_rows(vl, gamma, target_row=tr, draft_row=dr, totals=tot)
    torch.cuda.synchronize(dev)
    vl_h, tr_h, dr_h = vl.cpu().numpy(), tr.cpu().numpy(), dr.cpu().numpy()
    Kt, Kd = (int(v) for v in tot.cpu().numpy())
    ti = np.concatenate([b * (gamma + 1) + np.arange(vl_h[b] + 1) for b in range(B)])
    di = np.concatenate([b * gamma + np.arange(vl_h[b]) for b in range(B)])
    tp = t.view(B * (gamma + 1), V)[torch.from_numpy(ti).to(dev)].contiguous()
    dp = d.view(B * gamma, V)[torch.from_numpy(di).to(dev)].contiguous()
    # copies of the packed logits, so that the graph-replayed steps' working
    # set exceeds twice the L2
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets = max(1, min(8, -(-2 * l2 // (tp.nbytes + dp.nbytes))))
    psets = [(tp, dp)] + [(tp.clone(), dp.clone()) for _ in range(n_sets - 1)]
    assert (tr_h == np.concatenate([[0], np.cumsum(vl_h + 1)[:-1]])).all()
    out_t = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = sv.alloc_verify_workspace(B, gamma, V, sv.BF16, dev)

    def step(i=0):
        ptp, pdp = psets[i % n_sets]
        sv.schedule(conf, (ratios, costs), 0, sv.SCHED_DCUT, out_verify_len=vl, workspace=sws)
        sv.pack_rows(vl, gamma, target_row=tr, draft_row=dr, totals=tot)
        sv.verify_packed(ptp, pdp, tr, dr, x, vl, case.T, u, out_tokens=out_t, out_accept_len=out_n, workspace=ws)

    for i in range(3):
        step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    host_ms = e0.elapsed_time(e1) / steps
    ms = graph_us_per_call(dev, stream, step) / 1e3
    rows = int(vl_h.sum())
    logit_bytes = (Kt + Kd) * V * 2
    k1 = row_stats_ms(sv, dev, stream, step, max(3, min(steps, 200)))
    floor_ms = event_floor_ms(dev, stream)
    if sv.read_status(ws) != 0 or sv.read_status(sws) != 0:
        raise RuntimeError("device status on the packed step")
    return {"workload": "D-cut budget (ratios 0.25..1, costs = the round-cost table at K_rho), dense packing, "
                        f"verify of the {WORKLOAD} logits packed as [{Kt}, V] target and [{Kd}, V] draft rows",
            "ms_per_step": ms, "verified_rows_per_step": rows, "verified_rows_per_s": rows / (ms / 1e3),
            "packed_logit_bytes": logit_bytes, "logit_gbs": logit_bytes / (ms / 1e3) / 1e9,
            "timing": f"50 steps in a CUDA graph, 5 replays; packed logits rotated over {n_sets} copies "
                      f"({n_sets * logit_bytes / 1e6:.0f} MB, L2 {l2 / 1e6:.0f} MB)",
            "host_launched_ms_per_step": host_ms, "host_launched_steps": steps,
            "kernel_launches_per_step": 2 + sv.kernel_count(B, case.T),
            "roofline": roofline_entry(logit_bytes, k1, max(3, min(steps, 200)), floor_ms)}


def run_ours(args):
    import torch
    import specsynth
    import speculative_decoding_verification_softmax_gb300 as sv

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sv.build()

    o = 1000 * rank + SEED_OFFSET
    case = specsynth.make_verify_case(WORKLOAD, seed_logits=300 + o, seed_noise=301 + o, seed_tokens=302 + o,
                                      seed_uniforms=303 + o)
    B, gamma, V = case.B, case.gamma, case.V
    t, d, x, vl, u = specsynth.to_device(case, dev)
    out_t = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = sv.alloc_verify_workspace(B, gamma, V, sv.BF16, dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        sv.verify(t, d, x, vl, case.T, u, out_tokens=out_t, out_accept_len=out_n, workspace=ws)

    W = max(args.warmup, 3)
    for _ in range(W):
        step()
    torch.cuda.synchronize(dev)
    if sv.read_status(ws) != 0:
        raise RuntimeError("device status after warm-up")

    # timed region 1: K steps back to back (the value); events on the
    # launching stream, synchronised on both sides
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    with ClockSampler(local) as clk:
        # an untimed burst first, so that the timed steps start on a busy GPU
        # with the host already ahead of it (not from the idle gap of the
        # clock sampler's start-up)
        for _ in range(PREROLL_STEPS):
            step()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    ms = ev0.elapsed_time(ev1) / args.steps
    ms_max = reduce_max(ms, world, dev)

    # timed region 2: the same K steps with the row-statistics kernel of each
    # step bracketed by its own event pair (the events sit between that kernel
    # and the next one, which then cannot overlap it: this region is used only
    # for the kernel's own duration)
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    for a, b in pairs:          # create the events before the timed region
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    head_start(min(args.steps, 1000))
    for a, b in pairs:
        sv.profile_events(a, b)
        step()
    torch.cuda.synchronize(dev)
    sv.profile_events(None, None)
    k1_ms = sum(a.elapsed_time(b) for a, b in pairs) / len(pairs)
    k1_list = sorted(a.elapsed_time(b) for a, b in pairs)
    floor_ms = event_floor_ms(dev, stream)  # reported beside the event-bracketed kernel times

    # timed region 3: each call bracketed by its own event pair (at call
    # boundaries, where nothing overlaps) for the latency distribution
    n_lat = min(args.steps, 1000)
    cpairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_lat)]
    torch.cuda.synchronize(dev)
    for a, b in cpairs:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    lat = sorted(a.elapsed_time(b) * 1e3 for a, b in cpairs)
    pct = lambda v, q: v[min(len(v) - 1, int(q * (len(v) - 1) + 0.5))]
    latency = {"unit": "us", "calls": n_lat, "p10": pct(lat, 0.1), "p50": pct(lat, 0.5), "p90": pct(lat, 0.9),
               "k1_p10": pct(k1_list, 0.1) * 1e3, "k1_p50": pct(k1_list, 0.5) * 1e3,
               "k1_p90": pct(k1_list, 0.9) * 1e3}
    status = sv.read_status(ws)
    n = out_n.cpu().numpy()

    # the whole path on the scheduled ragged workload: spec_schedule (exact
    # scan, cost table B', min_len 1) feeding spec_verify, back to back
    conf_s = torch.from_numpy(specsynth.make_confidences(seed=specsynth.SCHED_SEED + 1000 * rank + SEED_OFFSET)).to(dev)
    vl_s = torch.empty((B,), dtype=torch.int32, device=dev)
    ws_s = torch.zeros(256, dtype=torch.uint8, device=dev)
    cost_s = specsynth.COST_TABLES[COST_READING]

    # a second copy of the logits: the graph-replayed steps alternate between
    # the two, so the rows read in consecutive steps are not L2-resident
    ssets = [(t, d), (t.clone(), d.clone())]

    def sched_step(i=0):
        st_, sd_ = ssets[i % 2]
        sv.schedule(conf_s, cost_s, specsynth.SCHED_MIN_LEN, sv.SCHED_EXACT, out_verify_len=vl_s, workspace=ws_s)
        sv.verify(st_, sd_, x, vl_s, case.T, u, out_tokens=out_t, out_accept_len=out_n, workspace=ws)

    for i in range(3):
        sched_step(i)
    torch.cuda.synchronize(dev)
    s_steps = max(3, min(args.steps, 500))
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for i in range(s_steps):
        sched_step(i)
    s1.record(stream)
    torch.cuda.synchronize(dev)
    s_host_ms = s0.elapsed_time(s1) / s_steps
    s_ms = graph_us_per_call(dev, stream, sched_step) / 1e3
    vl_h = vl_s.cpu().numpy()
    s_rows = int(vl_h.sum())
    ragged_bytes = int((2 * vl_h + 1).sum()) * V * 2

    def ragged_verify(i=0):     # the verification alone, at the scheduled lengths
        st_, sd_ = ssets[i % 2]
        sv.verify(st_, sd_, x, vl_s, case.T, u, out_tokens=out_t, out_accept_len=out_n, workspace=ws)

    rv_ms = graph_us_per_call(dev, stream, ragged_verify) / 1e3
    n_rag = out_n.cpu().numpy()
    ragged_resid = int(((n_rag < vl_h) * 2 + (n_rag >= vl_h)).sum()) * V * 2
    # the streaming kernel of the verification alone at the scheduled lengths
    rk1 = row_stats_ms(sv, dev, stream, ragged_verify, max(3, min(args.steps, 200)))
    del ssets
    if sv.read_status(ws) != 0 or sv.read_status(ws_s) != 0:
        raise RuntimeError("device status on the scheduled workload")
    scheduled_step = {"workload": f"schedule (exact scan, cost table {COST_READING}, min_len 1) then verify of the "
                                  f"{WORKLOAD} logits at the scheduled lengths",
                      "ms_per_step": s_ms, "verified_rows_per_step": s_rows,
                      "verified_rows_per_s": s_rows / (s_ms / 1e3),
                      "timing": "50 steps in a CUDA graph, 5 replays; logits alternate between two copies",
                      "host_launched_ms_per_step": s_host_ms, "host_launched_steps": s_steps,
                      "kernel_launches_per_step": 1 + sv.kernel_count(B, case.T),
                      "logit_bytes_per_step": ragged_bytes,
                      "verify_only": {"ms_per_call": rv_ms, "bytes_per_call": ragged_bytes + ragged_resid,
                                      "gbs": (ragged_bytes + ragged_resid) / (rv_ms / 1e3) / 1e9,
                                      "pct_of_measured_peak": 100.0 * (ragged_bytes + ragged_resid)
                                      / (rv_ms / 1e3) / 1e9 / measured_peak_gbs()[0],
                                      "timing": "50 calls in a CUDA graph, 5 replays; logits alternate "
                                                "between two copies"},
                      "roofline": dict(roofline_entry(ragged_bytes, rk1, max(3, min(args.steps, 200)), floor_ms),
                                       calls="the verification alone at the scheduled lengths")}
    sched = time_schedulers(sv, dev, stream, rank)
    scheduled_step["scheduler_share"] = sched["modes"]["exact"]["us_per_call"] / 1e3 / s_ms
    packed_step = time_packed_step(sv, specsynth, case, t, d, x, u, dev, stream, rank, s_steps)
    others = time_other_workloads(sv, specsynth, dev, stream, rank)

    # end to end through the public API: pinned host inputs -> device -> verify -> host outputs
    h_t = torch.from_numpy(case.target.view(np.int16)).pin_memory()
    h_d = torch.from_numpy(case.draft.view(np.int16)).pin_memory()
    h_x = torch.from_numpy(case.draft_tokens).pin_memory()
    h_vl = torch.from_numpy(case.verify_len).pin_memory()
    h_u = torch.from_numpy(case.uniforms).pin_memory()
    h_ot = torch.empty((B, gamma + 1), dtype=torch.int32).pin_memory()
    h_on = torch.empty((B,), dtype=torch.int32).pin_memory()
    tv, dv = t.view(torch.int16), d.view(torch.int16)

    def e2e_step():
        tv.copy_(h_t, non_blocking=True)
        dv.copy_(h_d, non_blocking=True)
        x.copy_(h_x, non_blocking=True)
        vl.copy_(h_vl, non_blocking=True)
        u.copy_(h_u, non_blocking=True)
        step()
        h_ot.copy_(out_t, non_blocking=True)
        h_on.copy_(out_n, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 50))
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_serial_ms = reduce_max(e0.elapsed_time(e1) / e2e_steps, world, dev)

    # the same steps pipelined as a serving loop would run them: two device
    # input sets, step k+1's host-to-device copy (on a copy stream) overlapping
    # step k's verification and result read-back
    sets = [(t, d, x, vl, u), tuple(torch.empty_like(a) for a in (t, d, x, vl, u))]
    cstream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    freed = [torch.cuda.Event(), torch.cuda.Event()]

    def e2e_copy(k):
        bt, bd, bx, bvl, bu = sets[k % 2]
        with torch.cuda.stream(cstream):
            if k >= 2:
                cstream.wait_event(freed[k % 2])     # step k-2 has read this set
            bt.view(torch.int16).copy_(h_t, non_blocking=True)
            bd.view(torch.int16).copy_(h_d, non_blocking=True)
            bx.copy_(h_x, non_blocking=True)
            bvl.copy_(h_vl, non_blocking=True)
            bu.copy_(h_u, non_blocking=True)
            copied[k % 2].record(cstream)

    def e2e_verify(k):
        bt, bd, bx, bvl, bu = sets[k % 2]
        stream.wait_event(copied[k % 2])
        sv.verify(bt, bd, bx, bvl, case.T, bu, out_tokens=out_t, out_accept_len=out_n, workspace=ws)
        freed[k % 2].record(stream)
        h_ot.copy_(out_t, non_blocking=True)
        h_on.copy_(out_n, non_blocking=True)

    def e2e_pipelined(n_steps):
        cstream.wait_stream(stream)
        e2e_copy(0)
        for k in range(n_steps):
            if k + 1 < n_steps:
                e2e_copy(k + 1)
            e2e_verify(k)
        stream.wait_stream(cstream)

    e2e_pipelined(3)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    e2e_pipelined(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(e0.elapsed_time(e1) / e2e_steps, world, dev)
    if sv.read_status(ws) != 0:
        raise RuntimeError("device status after the end-to-end steps")
    h2d = sum(a.numel() * a.element_size() for a in (h_t, h_d, h_x, h_vl, h_u))
    d2h = h_ot.numel() * 4 + h_on.numel() * 4

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    rows_per_step = B * gamma
    value = aggregate(ms_max, rows_per_step, world)
    alg_bytes = B * (2 * gamma + 1) * V * 2                      # row-stats kernel, all rows needed
    rejected = int((n < gamma).sum())      # of the last verify-all call
    resid_bytes = (2 * rejected + (B - rejected)) * V * 2
    peak, peak_kind = measured_peak_gbs()
    achieved = alg_bytes / (k1_ms / 1e3) / 1e9
    step_gbs = (alg_bytes + resid_bytes) / (ms / 1e3) / 1e9
    traffic = profiled_traffic()
    cores = os.cpu_count() or 1
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": W, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": workload_config(case),
        "hbm": {"gbs_per_gpu": step_gbs, "pct_of_measured_peak": 100.0 * step_gbs / peak,
                "bytes_per_step": alg_bytes + resid_bytes, "peak_gbs": peak, "peak_kind": peak_kind,
                "vendor_nominal_gbs": 7900.0, "pct_of_vendor_nominal": 100.0 * step_gbs / 7900.0},
        "roofline": {"kernel": "k_row_stats", "bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": alg_bytes, "avg_launch_ms": k1_ms,
                     "launches_timed": args.steps,
                     "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
                     "event_pair_floor_ms": floor_ms},
        "cpu_baseline": cpu_baseline(case, cores),
        "e2e": {"value": aggregate(e2e_ms, rows_per_step, world), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "steps": e2e_steps,
                "pipeline": "two device input sets; step k+1's host-to-device copy runs on a copy "
                            "stream while step k verifies and reads its result back",
                "h2d_gbs": h2d / (e2e_ms / 1e3) / 1e9,
                "serial": {"ms_per_step": e2e_serial_ms,
                           "value": aggregate(e2e_serial_ms, rows_per_step, world)}},
        "gpu_launches": sv.kernel_count(B, case.T) * args.steps,
        "clocks": clk.summary(),
        "device_status": status,
        "latency": latency,
        "scheduled_step": scheduled_step,
        "schedule": sched,
        "scheduled_step_packed": packed_step,
        "other_workloads": others,
        "mean_accept_len": float(n.mean()),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_profile_case(args):
    """A small case for ncu captures: B requests of one workload (inputs still
    larger than L2), a few verification calls, nothing else.  --profile-packed
    verifies the block-diffusion rows at D-cut lengths packed as [K, V]."""
    import math
    import torch
    import specsynth
    import speculative_decoding_verification_softmax_gb300 as sv
    sv.build()
    name = args.profile_workload
    case = specsynth.make_verify_case(name, B=args.profile_batch)
    B, gamma, V = case.B, case.gamma, case.V
    t, d, x, vl, u = specsynth.to_device(case)
    dt = sv.BF16 if case.dtype == "bf16" else sv.F32
    ws = sv.alloc_verify_workspace(B, gamma, V, dt)
    uu = u if case.T != 0 else None
    if args.profile_packed:
        conf = torch.from_numpy(specsynth.make_confidences(B, gamma)).cuda()
        kt, kc = specsynth.COST_TABLES[COST_READING]
        ratios = [0.25, 0.5, 0.75, 1.0]
        costs = [float(np.interp(max(B, math.ceil(r * B * (gamma + 1))), kt, kc)) for r in ratios]
        vl, _ = sv.schedule(conf, (ratios, costs), 0, sv.SCHED_DCUT)
        tr, dr, tot = sv.pack_rows(vl, gamma)
        vl_h = vl.cpu().numpy()
        ti = np.concatenate([b * (gamma + 1) + np.arange(vl_h[b] + 1) for b in range(B)])
        di = np.concatenate([b * gamma + np.arange(vl_h[b]) for b in range(B)])
        tp = t.view(-1, V)[torch.from_numpy(ti).cuda()].contiguous()
        dp = d.view(-1, V)[torch.from_numpy(di).cuda()].contiguous()
        call = lambda: sv.verify_packed(tp, dp, tr, dr, x, vl, case.T, u, workspace=ws)
    else:
        call = lambda: sv.verify(t, d, x, vl, case.T, uu, workspace=ws)
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    st = sv.read_status(ws)
    print(json.dumps({"profile_case": name, "packed": bool(args.profile_packed), "B": B,
                      "calls": args.warmup + args.steps, "status": st}))
    if st != 0:
        raise SystemExit(1)


def run_profile_sched(args):
    """A case for ncu captures of the scheduler: spec_schedule (exact scan, cost
    table B', min_len 1) on the scheduled workload's 64 x 16 confidences, a few
    calls, nothing else."""
    import torch
    import specsynth
    import speculative_decoding_verification_softmax_gb300 as sv
    sv.build()
    conf = torch.from_numpy(specsynth.make_confidences()).cuda()
    out = torch.empty((conf.shape[0],), dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup + args.steps):
        sv.schedule(conf, specsynth.COST_TABLES[COST_READING], specsynth.SCHED_MIN_LEN, sv.SCHED_EXACT,
                    out_verify_len=out, workspace=ws)
    torch.cuda.synchronize()
    st = sv.read_status(ws)
    print(json.dumps({"profile_sched": "scheduled ragged", "calls": args.warmup + args.steps, "status": st,
                      "verified_rows": int(out.sum().item())}))
    if st != 0:
        raise SystemExit(1)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile-case", action="store_true",
                    help="run only a small case for ncu (B=--profile-batch)")
    ap.add_argument("--profile-batch", type=int, default=24)
    ap.add_argument("--profile-workload", default=WORKLOAD, choices=["block_diffusion", "greedy", "mtp_chat"],
                    help="workload of --profile-case")
    ap.add_argument("--profile-packed", action="store_true",
                    help="--profile-case on D-cut lengths with packed logits")
    ap.add_argument("--profile-sched", action="store_true",
                    help="run only the scheduler on the scheduled workload (for ncu)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed-offset", type=int, default=0,
                    help="added to every seed of the synthetic inputs (default 0: the stated recipe)")
    ap.add_argument("--cost-table", choices=["Bprime", "A", "C"], default="Bprime",
                    help="reading of the round-cost table used by the scheduled legs")
    args = ap.parse_args(argv)
    global SEED_OFFSET, COST_READING
    SEED_OFFSET, COST_READING = args.seed_offset, args.cost_table
    if args.profile_case:
        run_profile_case(args)
    elif args.profile_sched:
        run_profile_sched(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
