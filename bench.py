#!/usr/bin/env python3
"""Benchmark of the draft-verification step on GB300.

One step = one batched verification (target/draft logits in, tokens and
accept lengths out) of the concurrency-32 mixed workload: B=32 requests,
block 8 (gamma=7), V=248320, bf16 logits, temperatures cycling 0 (greedy) /
0.6 / 1.0, top-k 20, top-p 0.95. The metric is verified draft positions per
second (B * gamma per step) with the achieved HBM bandwidth in the roofline
block. Inputs rotate over 3 independently generated sets (each about 238 MB,
together well above the 129 MB L2), so no step finds its logits in L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload NAME] [--drafts sampled|det]

``--workload`` measures another of the step's workloads the same way (for
example b128_g15_fullvocab_f32: block 16, fp32, top-k off and top-p 1, where a
call is the stream plus the full-vocabulary draw's second pass); the default
is the headline above. ``--drafts det`` verifies deterministic drafts (each
draft row's argmax, as a greedy drafter proposes them) through
dflash_verify_det, which reads no draft logits.

N > 1 runs under torch.distributed.run: every rank verifies its own batch (the
step shards by request, no data exchange), timing is the max over ranks.
``--impl reference`` times the CPU oracle (fp64, host threads) on samples of
the same workload.

``--calls N`` makes no measurement: it runs N verification calls on one batch
of the workload (drafts = each draft row's argmax; ``--batch B`` for fewer
requests; ``--gpu-logits`` draws N(0, 2) target and target + N(0, 0.5) draft
logits on the GPU instead of the host) and exits, a short program for a
profiler's launch list or capture.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

WORKLOAD = "b32_mixed_v248320"
METRIC = "verified draft-positions/sec and achieved HBM GB/s (B=32, block 8, V=248320)"


def metric_for(workload: str, det: bool = False) -> str:
    if workload == WORKLOAD and not det:
        return METRIC
    w = synth.WORKLOADS[workload]
    return (f"verified draft-positions/sec and achieved HBM GB/s (B={w['B']}, block {w['gamma'] + 1}, "
            f"V={w['V']}" + (", deterministic drafts)" if det else ")"))


DET_DRAFTS = "deterministic: the argmax of each draft row (q = the point mass at the draft)"
UNIT = "verified draft positions/s"
N_SETS = 3
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "verify_sweep_b32_mixed_v248320.md")


def profile_summary(workload: str, det: bool = False) -> str:
    """The committed ncu summary of sweep_kernel on a workload (with
    deterministic drafts: the _det summary)."""
    return os.path.join(ROOT, "profiles", f"verify_sweep_{workload}{'_det' if det else ''}.md")
CSRC = os.path.join(ROOT, "speculative_decoding_verification_83_gb300", "csrc")


# the sources the profiled kernel (sweep_kernel) is built from
KERNEL_SOURCES = ("dflash_sweep.cu", "dflash_rule.cuh", "dflash_device.cuh", "dflash_internal.h")


def kernel_source_hash() -> str:
    """Hash of the profiled kernel's code: comments and the amount of white
    space do not count, so editing a comment keeps a profile valid."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(CSRC, f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(f.encode() + " ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(path: str = PROFILE_SUMMARY):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source."""
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != kernel_source_hash():
        return None
    return float(m.group(1))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0}, "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = f"/tmp/dflash_clocks_{os.getpid()}.csv"
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_index)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.remove(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- helpers
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def algorithmic_bytes(inp, accept_len=None, det=False) -> int:
    """Logit bytes one step must read: every target row, and the draft rows of
    requests that sample (greedy requests never read their draft rows, nor
    does the verification of deterministic drafts). Over the full vocabulary
    (top-k off) the residual or bonus draw reads its rows once more: two rows
    after a rejection, one for a bonus token (from the step's accept lengths).
    With top-p < 1 the passes that find each row's cut read the sampling rows
    again; they are counted as the path's overhead, not as algorithmic bytes
    (a cut that could be found inside the statistics pass would not need
    them)."""
    B, gamma, V = inp.shape
    es = 2 if inp.target.dtype == np.uint16 else 4
    samp = inp.temperature > 0
    rows = B * (gamma + 1) + (0 if det else int(np.sum(samp)) * gamma)
    if inp.top_k <= 0 and accept_len is not None:
        lens = np.asarray(accept_len)[samp]
        rows += int(np.sum(np.where(lens <= gamma, 2, 1)))
    return rows * V * es


def launches_per_step(top_k: int, top_p: float, bf16: bool = True) -> int:
    """Kernel launches of one verification call: the stream kernel, plus the
    full-vocabulary draw's two launches when top-k is off; with top-p < 1
    also the cut's rounds (a histogram and a select launch for the first
    round and for each refinement round: up to four for fp32 keys, two for
    bf16), its two tie launches and the accept launch."""
    if top_k > 0:
        return 1
    if top_p >= 1.0:
        return 3
    return 3 + 2 * (3 if bf16 else 5) + 3


def cpu_baseline(inp, d, workload, threads=None, det=False, min_s=10.0, max_batches=200):
    """The oracle (as it stands) on the host cores: whole batches of the
    workload, one seed each, until at least min_s seconds of work (at most
    max_batches batches)."""
    import oracle

    B, gamma, V = inp.shape
    threads = threads or oracle.default_threads()
    n = 0
    t0 = time.perf_counter()
    while n < max_batches and (n == 0 or time.perf_counter() - t0 < min_s):
        if det:
            oracle.verify_det(inp.target, d, inp.temperature, inp.top_k, inp.top_p, inp.seed + n,
                              threads=threads)
        else:
            oracle.verify(inp.target, inp.draft, d, inp.temperature, inp.top_k, inp.top_p, inp.seed + n,
                          threads=threads)
        n += 1
    dt = time.perf_counter() - t0
    return {"value": n * B * gamma / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n} whole {workload} batches of {B} requests, one seed each (fp64 C oracle, "
                      f"{threads} host threads), {dt:.1f} s"}


def accept_report(sets_np, lens_by_set, det=False):
    """Accept lengths of the timed steps (each input set's batch; its seed is
    fixed, so every step on it gives the same lengths): their histogram over
    1..gamma+1 and mean, next to the closed-form mean sum_i prod_{j<i} alpha_j
    with alpha_j = sum min(p_j, q_j) from the oracle's filtered distributions
    of the same rows (greedy requests enter with their own length, which is
    not random). With deterministic drafts q is the point mass at the draft,
    so alpha_j = p_j(d_j)."""
    import oracle

    B, gamma, V = sets_np[0].shape
    lens = np.concatenate(lens_by_set)
    hist = np.bincount(lens, minlength=gamma + 2)[1:gamma + 2]
    closed = []
    for inp, ln in zip(sets_np, lens_by_set):
        if det:
            return {"hist": hist.tolist(), "mean": float(lens.mean()), "closed_form_mean": None,
                    "requests": int(lens.size)}
        alpha = oracle.accept_rates(inp.target, inp.draft, inp.temperature, inp.top_k, inp.top_p)
        e = oracle.expected_accept_len(np.nan_to_num(alpha, nan=0.0))
        samp = inp.temperature > 0
        closed.append(np.where(samp, e, ln))
    closed = np.concatenate(closed)
    return {"hist": hist.tolist(), "mean": float(lens.mean()), "closed_form_mean": float(closed.mean()),
            "requests": int(lens.size),
            "note": "closed form over the drafts' distribution: the sampled drafts are one draw of it"}


def combine_over_ranks(region_ms: float, e2e_s: float, steps: int, per_rank_units: int, device=None):
    """Whole-job numbers from this rank's timings: the slowest rank's timed
    region and end-to-end step (max over ranks; every rank verifies its own
    batch, so the job is as slow as its slowest rank), and the units all
    ranks processed divided by that time. Needs the default process group
    when the world has more than one rank."""
    import torch

    world = 1
    t = torch.tensor([region_ms, e2e_s], dtype=torch.float64, device=device)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        world = torch.distributed.get_world_size()
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    region_ms, e2e_s = float(t[0].item()), float(t[1].item())
    return {"world": world, "region_ms": region_ms, "ms_per_step": region_ms / steps,
            "value": world * steps * per_rank_units / (region_ms / 1e3),
            "e2e_s": e2e_s, "e2e_value": world * per_rank_units / e2e_s}


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import oracle

    if args.workload == LMHEAD_WORKLOAD:
        return run_reference_lmhead(args)

    inp = synth.make_workload(args.workload, data_seed=0, seed=0)
    B, gamma, V = inp.shape
    det = args.drafts == "det"
    if det:
        d = np.argmax(synth.to_float(inp.draft), axis=-1).astype(np.int32)
    else:
        d, _, _ = oracle.sample_rows(inp.draft.reshape(B * gamma, V),
                                     synth.draft_sampling_temperatures(inp.temperature, gamma),
                                     inp.top_k, inp.top_p, 1000)
        d = d.reshape(B, gamma)
    threads = oracle.default_threads()

    def verify(seed, order):
        if det:
            Xs = np.ascontiguousarray(inp.target[order])
            return oracle.verify_det(Xs, d[order], inp.temperature[order], inp.top_k, inp.top_p,
                                     seed, threads=threads)
        return oracle.verify(inp.target, inp.draft, d, inp.temperature, inp.top_k, inp.top_p, seed,
                             threads=threads, requests=order)

    # size each step so that warmup + steps stay within about two minutes
    t0 = time.perf_counter()
    verify(0, [1])
    per_req = max(1e-3, time.perf_counter() - t0)
    budget = 120.0 / max(1, args.steps + args.warmup)
    n_req = int(max(1, min(B, budget / per_req)))
    order = [b % B for b in range(1, 1 + n_req)]  # starts with a sampling request
    for _ in range(args.warmup):
        verify(0, order)
    t0 = time.perf_counter()
    for s in range(args.steps):
        verify(s, order)
    dt = time.perf_counter() - t0
    value = args.steps * n_req * gamma / dt
    sample = f"{n_req} of the {B} requests per step (fp64 C oracle, {threads} host threads)"
    line = {
        "impl": "reference", "metric": metric_for(args.workload, det), "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": args.workload, "B": B, "gamma": gamma, "V": V,
                                        "top_k": inp.top_k, "top_p": inp.top_p,
                                        "drafts": DET_DRAFTS if det else "sampled from q"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def run_gpu(args):
    import torch

    import speculative_decoding_verification_83_gb300 as dv

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as tdist

        tdist.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    torch.cuda.set_device(local_rank)
    dev = torch.device(f"cuda:{local_rank}")
    dv.build()
    lib = dv.load()

    # ---- inputs: N_SETS independent batches, resident in HBM
    sets_np, sets_dev = [], []
    for s in range(N_SETS):
        sets_np.append(synth.make_workload(args.workload, data_seed=1000 * rank + s, seed=s))
    B, gamma, V = sets_np[0].shape
    bf16 = sets_np[0].target.dtype == np.uint16
    dt_code = dv.DFLASH_BF16 if bf16 else dv.DFLASH_F32
    es = 2 if bf16 else 4
    rows_ws = dv.Workspace(dv.rows_workspace_bytes(B * gamma, V, dt_code, sets_np[0].top_k,
                                                   sets_np[0].top_p), dev)
    for inp in sets_np:
        X = synth.to_torch(inp.target, dev)
        Y = synth.to_torch(inp.draft, dev)
        T = torch.from_numpy(inp.temperature).to(dev)
        # drafts: the library's own sampler on the draft rows (argmax for greedy requests)
        Trows = torch.from_numpy(synth.draft_sampling_temperatures(inp.temperature, gamma)).to(dev)
        d = dv.sample_rows(Y.view(B * gamma, V), Trows, inp.top_k, inp.top_p, 7 + inp.seed,
                           workspace=rows_ws).view(B, gamma).contiguous()
        sets_dev.append((X, Y, d, T))
    torch.cuda.synchronize()
    det = args.drafts == "det"
    if det:
        # a greedy drafter's proposals: each draft row's argmax (the sampler at T = 0)
        zeros = torch.zeros(B * gamma, dtype=torch.float32, device=dev)
        for s, (X, Y, d, T) in enumerate(sets_dev):
            d_det = dv.sample_rows(Y.view(B * gamma, V), zeros, sets_np[s].top_k, sets_np[s].top_p, 0,
                                   workspace=rows_ws).view(B, gamma).contiguous()
            sets_dev[s] = (X, Y, d_det, T)
        torch.cuda.synchronize()
    top_k, top_p = sets_np[0].top_k, sets_np[0].top_p
    ws = dv.Workspace(dv.workspace_bytes(B, gamma, V, dt_code, top_k, top_p), dev)
    out_tok = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    out_len = torch.empty((B,), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    calls = []
    for s, (X, Y, d, T) in enumerate(sets_dev):
        logits = (X.data_ptr(),) if det else (X.data_ptr(), Y.data_ptr())
        calls.append(logits + (d.data_ptr(), B, gamma, V, dt_code, T.data_ptr(),
                               top_k, top_p, s + 1, out_tok.data_ptr(), out_len.data_ptr(), ws.ptr,
                               ws.nbytes, status.data_ptr(), sp))
    fn = lib.dflash_verify_det if det else lib.dflash_verify

    def step(i):
        rc = fn(*calls[i % N_SETS])
        if rc:
            raise RuntimeError(lib.dflash_last_error().decode())

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"status word {int(status.item())} after warm-up")

    # ---- timed region: K steps back to back (no event between launches, so
    # each launch may overlap the end of the one before it: programmatic
    # dependent launch), bracketed by one event pair on the launching stream
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    time.sleep(0.3)
    # a spin kernel ahead of the start event keeps the device busy while the
    # host enqueues the K calls, so the region times the device, not the
    # host's first launch (it ends before the start event is recorded)
    torch.cuda._sleep(int(2e6))
    start.record(stream)
    for i in range(args.steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    region_ms = start.elapsed_time(end)

    # ---- roofline of the kernel: algorithmic bytes of one call over the
    # average call duration in the timed region (one call = one launch of the
    # stream kernel; plus the two draw launches over the full vocabulary)
    lens_by_set = []
    for s in range(N_SETS):  # the outputs of each input set (its seed is fixed, so every step on it gives these)
        step(s)
        torch.cuda.synchronize()
        lens_by_set.append(out_len.cpu().numpy().copy())
    alg = algorithmic_bytes(sets_np[(args.steps - 1) % N_SETS], lens_by_set[(args.steps - 1) % N_SETS], det)
    avg_launch_s = region_ms / args.steps / 1e3
    achieved = alg / avg_launch_s / 1e9
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    traffic = profiled_traffic(profile_summary(args.workload, det))
    # an isolated call (an event pair around each of a few launches, which
    # rules out overlap with the launch before): for reference, not timed above
    n_iso = min(200, max(20, args.steps))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_iso)]
    for i in range(n_iso):
        evs[i][0].record(stream)
        step(i)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    iso_ms = np.array([a.elapsed_time(b) for a, b in evs])
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
                "algorithmic_bytes_per_launch": alg,
                "avg_launch_us": avg_launch_s * 1e6,
                "isolated_launch_us_p50": float(np.median(iso_ms)) * 1e3}

    # ---- end to end through the host-buffer entry point (pinned host memory)
    inp = sets_np[0]

    def pin(a):
        return synth.to_torch(a, "cpu").pin_memory()

    hX, hY = pin(inp.target), pin(inp.draft)
    hd = sets_dev[0][2].cpu().pin_memory()
    hT = pin(inp.temperature)
    h_tok = torch.empty((B, gamma + 1), dtype=torch.int32).pin_memory()
    h_len = torch.empty((B,), dtype=torch.int32).pin_memory()
    h_st = torch.zeros((1,), dtype=torch.int32).pin_memory()
    staging = torch.empty(dv.host_staging_bytes(B, gamma, V, dt_code), dtype=torch.uint8,
                          device=dev)
    n_e2e = max(3, min(50, args.steps))
    if det:
        # through the Python binding: pinned inputs copied in, dflash_verify_det,
        # tokens and lengths copied back, on the bench stream
        eX = torch.empty_like(sets_dev[0][0])
        ed = torch.empty_like(sets_dev[0][2])
        eT = torch.empty_like(sets_dev[0][3])

        def e2e_step(i):
            eX.copy_(hX, non_blocking=True)
            ed.copy_(hd, non_blocking=True)
            eT.copy_(hT, non_blocking=True)
            t_, l_ = dv.verify_det(eX, ed, eT, top_k, top_p, i, out_tokens=out_tok, out_accept_len=out_len,
                                   workspace=ws, stream=stream)
            h_tok.copy_(t_, non_blocking=True)
            h_len.copy_(l_, non_blocking=True)
            stream.synchronize()
    else:
        def e2e_step(i):
            dv.verify_host(hX, hY, hd, hT, top_k, top_p, i, h_tok, h_len, h_st, staging, ws)
    for i in range(2):
        e2e_step(i)
    t0 = time.perf_counter()
    for i in range(n_e2e):
        e2e_step(i)
    e2e_s = (time.perf_counter() - t0) / n_e2e
    n_samp = 0 if det else int(np.sum(inp.temperature > 0))
    h2d = (B * (gamma + 1) + n_samp * gamma) * V * es + B * gamma * 4 + B * 4
    d2h = B * (gamma + 1) * 4 + B * 4 + (0 if det else 4)
    job = combine_over_ranks(region_ms, e2e_s, args.steps, B * gamma, dev)
    ms_per_step, value = job["ms_per_step"], job["value"]
    e2e = {"value": job["e2e_value"], "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": job["e2e_s"] * 1e3}

    if rank != 0:
        if world > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        return 0
    cpu, accept = None, None
    if world == 1:
        cpu = cpu_baseline(sets_np[0], sets_dev[0][2].cpu().numpy(), args.workload, det=det)
        cpu["single_core"] = cpu_baseline(sets_np[0], sets_dev[0][2].cpu().numpy(), args.workload, threads=1,
                                          det=det, min_s=5.0, max_batches=2)
        accept = accept_report(sets_np, lens_by_set, det)
    T0 = sets_np[0].temperature
    temps = ("cycling " + " / ".join(f"{t:g}" + (" (greedy)" if t == 0 else "")
                                     for t in dict.fromkeys(T0.tolist()))
             if len(set(T0.tolist())) > 1 else f"{T0[0]:g} for every request")
    line = {
        "metric": metric_for(args.workload, det), "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if bf16 else "f32", "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "gamma": gamma, "V": V, "top_k": top_k,
                   "top_p": top_p, "temperatures": temps,
                   "drafts": DET_DRAFTS if det else "sampled from q by the library's sampler",
                   "l2": f"inputs rotate over {N_SETS} sets of "
                         f"{(sets_np[0].target.nbytes + sets_np[0].draft.nbytes) / 1e6:.0f} MB "
                         "(larger than L2 together)",
                   "per_rank_batch": B},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_step(top_k, top_p, bf16),
        "clocks": clk,
        "accept_len": accept,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


# ---------------------------------------------------------------- LM head + verification
LMHEAD_WORKLOAD = "lmhead_b32_mixed_v248320_k5120"
LMHEAD_K = 5120


def lmhead_flops(M: int, V: int, K: int) -> int:
    """Dense flops of one LM-head product logits [M, V] = h [M, K] W^T."""
    return 2 * M * V * K


def run_lmhead(args):
    """The verification fused into the LM head's epilogue (dflash_lmhead_verify)
    at B = 32, block 8, hidden size 5120, V = 248320, against the same step
    unfused (dflash_lmhead_logits, then dflash_verify). W is a random
    bf16 matrix (no trained weights exist here); h and the draft tokens are
    drawn per input set. The roofline is the tensor cores': the product's
    dense flops over the step time against the measured bf16 peak."""
    import torch

    import speculative_decoding_verification_83_gb300 as dv

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as tdist

        tdist.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    torch.cuda.set_device(local_rank)
    dev = torch.device(f"cuda:{local_rank}")
    dv.build()
    lib = dv.load()
    B, gamma, V, K = 32, 7, 248320, LMHEAD_K
    M, Mt = B * (2 * gamma + 1), B * (gamma + 1)
    top_k, top_p = 20, 0.95
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + rank)
    w = (torch.randn((V, K), generator=g, device=dev) * (2.0 / K ** 0.5)).to(torch.bfloat16)
    T = torch.tensor([(0.0, 0.6, 1.0)[b % 3] for b in range(B)], dtype=torch.float32, device=dev)
    sets = []
    samp_ws = dv.Workspace(dv.rows_workspace_bytes(B * gamma, V, dv.DFLASH_BF16, top_k, top_p), dev)
    for s in range(2):
        h = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
        logits = dv.lmhead_logits(h, w)
        # drafts: the library's sampler on the draft rows (argmax for greedy requests)
        d = dv.sample_rows(logits[Mt:], T.repeat_interleave(gamma), top_k, top_p, 7 + s,
                           workspace=samp_ws).view(B, gamma).contiguous()
        sets.append((h, d, logits))
    torch.cuda.synchronize()
    ws = dv.Workspace(dv.workspace_bytes(B, gamma, V, dv.DFLASH_BF16, top_k, top_p), dev)
    out_tok = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    out_len = torch.empty((B,), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    row_bytes = V * 2

    def fused(i):
        h, d, logits = sets[i % 2]
        rc = lib.dflash_lmhead_verify(h.data_ptr(), w.data_ptr(), B, gamma, V, K, d.data_ptr(), T.data_ptr(),
                                      top_k, top_p, i + 1, logits.data_ptr(), out_tok.data_ptr(),
                                      out_len.data_ptr(), ws.ptr, ws.nbytes, status.data_ptr(), sp)
        if rc:
            raise RuntimeError(lib.dflash_last_error().decode())

    def unfused(i):
        h, d, logits = sets[i % 2]
        rc = lib.dflash_lmhead_logits(h.data_ptr(), w.data_ptr(), M, V, K, logits.data_ptr(), status.data_ptr(), sp)
        rc = rc or lib.dflash_verify(logits.data_ptr(), logits.data_ptr() + Mt * row_bytes, d.data_ptr(), B, gamma,
                                     V, dv.DFLASH_BF16, T.data_ptr(), top_k, top_p, i + 1, out_tok.data_ptr(),
                                     out_len.data_ptr(), ws.ptr, ws.nbytes, status.data_ptr(), sp)
        if rc:
            raise RuntimeError(lib.dflash_last_error().decode())

    def gemm_only(i):
        h, d, logits = sets[i % 2]
        rc = lib.dflash_lmhead_logits(h.data_ptr(), w.data_ptr(), M, V, K, logits.data_ptr(), status.data_ptr(), sp)
        if rc:
            raise RuntimeError(lib.dflash_last_error().decode())

    def timed(fn, steps):
        for i in range(max(3, args.warmup)):
            fn(i)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(int(2e6))
        a.record(stream)
        for i in range(steps):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    clocks = ClockSampler(local_rank)
    time.sleep(0.3)
    region_ms = timed(fused, args.steps)
    clk = clocks.stop()
    unfused_ms = timed(unfused, args.steps) / args.steps
    gemm_ms = timed(gemm_only, args.steps) / args.steps
    if int(status.item()) != 0:
        raise RuntimeError(f"status word {int(status.item())}")
    # the same outputs both ways, on the last input set
    fused(0)
    t_f, l_f = out_tok.clone(), out_len.clone()
    unfused(0)
    torch.cuda.synchronize()
    same = bool(torch.equal(t_f, out_tok) and torch.equal(l_f, out_len))

    # end to end through the binding: h from pinned host memory, the tokens back
    h_host = sets[0][0].cpu().pin_memory()
    d_host = sets[0][1].cpu().pin_memory()
    h_dev, d_dev = torch.empty_like(sets[0][0]), torch.empty_like(sets[0][1])
    tok_host = torch.empty((B, gamma + 1), dtype=torch.int32).pin_memory()
    len_host = torch.empty((B,), dtype=torch.int32).pin_memory()

    def e2e_step(i):
        h_dev.copy_(h_host, non_blocking=True)
        d_dev.copy_(d_host, non_blocking=True)
        t_, l_, _ = dv.lmhead_verify(h_dev, w, B, gamma, d_dev, T, top_k, top_p, i, logits=sets[0][2],
                                     workspace=ws, stream=stream)
        tok_host.copy_(t_, non_blocking=True)
        len_host.copy_(l_, non_blocking=True)
        stream.synchronize()

    for i in range(2):
        e2e_step(i)
    n_e2e = max(3, min(20, args.steps))
    t0 = time.perf_counter()
    for i in range(n_e2e):
        e2e_step(i)
    e2e_s = (time.perf_counter() - t0) / n_e2e
    job = combine_over_ranks(region_ms, e2e_s, args.steps, B * gamma, dev)
    if rank != 0:
        if world > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        return 0
    step_s = job["ms_per_step"] / 1e3
    flops = lmhead_flops(M, V, K)
    peaks, peak_kind = measured_peaks()
    # the timed region is a few tens of sub-millisecond steps at the maximum
    # SM clock: the burst figure of the cuBLAS GEMM is the comparison
    peak = float(peaks.get("bf16_tflops", 1900.0))
    cpu = None
    if world == 1:
        # the oracle's product on 1/64 of the vocabulary (scaled), and its
        # verification of one batch of the GPU's logits
        import oracle

        h0 = sets[0][0].view(torch.int16).cpu().numpy().view(np.uint16)
        w0 = w[: V // 64].view(torch.int16).cpu().numpy().view(np.uint16)
        L = sets[0][2].view(torch.int16).cpu().numpy().view(np.uint16)
        d0, T0 = sets[0][1].cpu().numpy(), T.cpu().numpy()
        c0 = time.perf_counter()
        oracle.lmhead_logits(h0, w0)
        t_gemm = (time.perf_counter() - c0) * 64
        c0 = time.perf_counter()
        oracle.verify(L[:Mt].reshape(B, gamma + 1, V), L[Mt:].reshape(B, gamma, V), d0, T0, top_k, top_p, 1)
        t_ver = time.perf_counter() - c0
        cpu = {"value": B * gamma / (t_gemm + t_ver), "unit": UNIT, "cores": oracle.default_threads(),
               "kind": "oracle",
               "sample": f"the fp64 product on {V // 64} of {V} vocabulary rows (x64) and the verification of "
                         f"one batch: {t_gemm:.1f} s + {t_ver:.1f} s"}
    line = {
        "metric": "verified draft-positions/sec of the LM head with the verification in its epilogue "
                  "(B=32, block 8, K=5120, V=248320)",
        "value": job["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": job["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (random-init W and h)",
        "config": {"workload": LMHEAD_WORKLOAD, "B": B, "gamma": gamma, "V": V, "K": K, "M": M,
                   "top_k": top_k, "top_p": top_p, "temperatures": "cycling 0 (greedy) / 0.6 / 1",
                   "l2": f"W ({V * K * 2 / 1e9:.2f} GB) is read once per step, larger than L2",
                   "per_rank_batch": B},
        "roofline": {"bound": "tensor", "achieved": flops / step_s / 1e12, "peak": peak, "unit": "TFLOP/s",
                     "frac": flops / step_s / 1e12 / peak, "traffic": None,
                     "peak_source": f"{peak_kind} bf16_tflops (cuBLAS 8192^3, burst)",
                     "peak_sustained": peaks.get("bf16_tflops_sustained"),
                     "achieved_over": "the fused step (GEMM with the statistics in its epilogue, then the "
                                      "verification's finals)",
                     "flops_per_step": flops, "w_bytes_per_step": V * K * 2,
                     "w_read_gbs": V * K * 2 / step_s / 1e9,
                     "logits_only_kernel_ms": gemm_ms,
                     "logits_only_kernel_tflops": flops / (gemm_ms / 1e3) / 1e12},
        "unfused_ms_per_step": unfused_ms,
        "fused_equals_unfused": same,
        "cpu_baseline": cpu,
        "e2e": {"value": job["e2e_value"], "unit": UNIT, "h2d_bytes_per_step": M * K * 2 + B * gamma * 4,
                "d2h_bytes_per_step": B * (gamma + 1) * 4 + B * 4, "ms_per_step": job["e2e_s"] * 1e3},
        "gpu_launches": args.steps * 2,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def run_reference_lmhead(args):
    """The oracle on the fused LM-head workload: its fp64 product on 1/64 of
    the vocabulary (scaled to all of it) plus its verification of one
    headline batch, per step."""
    import oracle

    B, gamma, V, K = 32, 7, 248320, LMHEAD_K
    M = B * (2 * gamma + 1)
    rng = np.random.default_rng(0)
    h = synth.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    w = synth.f32_to_bf16_bits((rng.standard_normal((V // 64, K)) * (2.0 / K ** 0.5)).astype(np.float32))
    inp = synth.make_workload(WORKLOAD, data_seed=0, seed=0)
    d, _, _ = oracle.sample_rows(inp.draft.reshape(B * gamma, V),
                                 synth.draft_sampling_temperatures(inp.temperature, gamma), 20, 0.95, 7)
    d = d.reshape(B, gamma)
    times = []
    for i in range(max(1, args.warmup) + max(1, args.steps)):
        c0 = time.perf_counter()
        oracle.lmhead_logits(h, w)
        t_gemm = (time.perf_counter() - c0) * 64
        c0 = time.perf_counter()
        oracle.verify(inp.target, inp.draft, d, inp.temperature, 20, 0.95, i)
        times.append(t_gemm + time.perf_counter() - c0)
    step_s = float(np.mean(times[max(1, args.warmup):]))
    value = B * gamma / step_s
    print(json.dumps({
        "impl": "reference", "metric": "verified draft-positions/sec of the LM head with the verification in its "
                                       "epilogue (B=32, block 8, K=5120, V=248320)",
        "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (random-init W and h)",
        "config": {"workload": LMHEAD_WORKLOAD, "B": B, "gamma": gamma, "V": V, "K": K},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.default_threads(), "kind": "oracle",
                         "sample": f"per step: the fp64 product on {V // 64} of {V} vocabulary rows (x64) and "
                                   "the verification of one B=32 batch"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)
    return 0


def run_calls(args):
    """--calls N: N verification calls on one batch of the workload and nothing
    else (no timing, no oracle), for a profiler."""
    import torch

    import speculative_decoding_verification_83_gb300 as dv

    dv.build()
    dv.load()
    w = synth.WORKLOADS[args.workload]
    B = args.batch or w["B"]
    t = w["temperature"]
    temps = synth.cycle_temperatures(B, t) if isinstance(t, tuple) else np.full(B, t, np.float32)
    if args.gpu_logits:
        gamma, V = w["gamma"], w["V"]
        g = torch.Generator(device="cuda")
        g.manual_seed(0)
        X = torch.randn((B, gamma + 1, V), generator=g, device="cuda") * 2.0
        Y = (X[:, :gamma] + 0.5 * torch.randn((B, gamma, V), generator=g, device="cuda")).contiguous()
        d = Y.argmax(-1).to(torch.int32).contiguous()
        if w["dtype"] == synth.BF16:
            X, Y = X.to(torch.bfloat16), Y.to(torch.bfloat16)
    else:
        inp = synth.make_workload(args.workload, data_seed=0, seed=0, B=B)
        X, Y = synth.to_torch(inp.target, "cuda"), synth.to_torch(inp.draft, "cuda")
        d = torch.from_numpy(np.argmax(synth.to_float(inp.draft), -1).astype(np.int32)).cuda()
    T = torch.from_numpy(np.asarray(temps, np.float32)).cuda()
    ln = None
    for i in range(args.calls):
        _, ln = dv.verify(X, Y, d, T, w["top_k"], w["top_p"], i)
    torch.cuda.synchronize()
    print(json.dumps({"workload": args.workload, "B": B, "calls": args.calls,
                      "accept_len": ln.cpu().numpy()[:8].tolist() if ln is not None else []}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(synth.WORKLOADS) + [LMHEAD_WORKLOAD])
    ap.add_argument("--drafts", default="sampled", choices=["sampled", "det"])
    ap.add_argument("--calls", type=int, default=0, help="run this many calls for a profiler and exit")
    ap.add_argument("--batch", type=int, default=0, help="with --calls: requests per call (default: the workload's)")
    ap.add_argument("--gpu-logits", action="store_true", help="with --calls: draw the logits on the GPU")
    args = ap.parse_args()
    if args.calls > 0:
        if args.workload == LMHEAD_WORKLOAD:
            ap.error("--calls runs a verification workload")
        return run_calls(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == LMHEAD_WORKLOAD:
        return run_lmhead(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
