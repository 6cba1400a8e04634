#!/usr/bin/env python3
"""Benchmark of the KDA hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one kda_chunk_fwd over the prefill workload B=8, T=8192, H=32,
dk=dv=128 (bf16 q/k/v/o, fp32 g/beta/states, h0 ~ N(0, 0.02^2), hT returned).
The same run also times the batched decode workload (256 sequences x H=32,
128x128 fp32 state updated in place, 1000 consecutive steps) and reports it
in the "decode" object, and a speculative-decoding round (verify + commit of 4
draft tokens) in "spec_decode", and the long-context workload (B=1, T=2^20,
H=32) single-pass and split in time into parallel segments in "prefill_long"
(--no-long skips it; the split by the shape-only segment hint, and as planned
from a sampled decay statistic of g, probe and plan timed with the call), and
the workload B=1, T=4096, H=32 (half the heads at g = -4.99) the same three
ways in "prefill_t4k". Inputs are synthetic (seeded), already
resident in HBM for `value`; `e2e` repeats the prefill step through the same
C-ABI call from pinned host buffers, every input uploaded and o, hT read back
inside the timed region, pipelined by batch row over copy and compute streams;
its "host_link" object times the step's input bytes going up as one copy and
its output bytes coming down as another, at the same time, nothing else: the
least time any step that moves them can take. The e2e figure is the median
over the timed steps of the pipeline's step period; every run is listed too.

The cpu_baseline sample doubles as a parity check ("parity"): the kernel runs
on every batch row the oracle timed and the errors against it are reported.

Prints ONE JSON line (rank 0). Under torchrun (N > 1) every rank runs its own
independent batch on its own GPU (data-parallel sequences, no collective on
the data path): `value` = tokens of all ranks / max over ranks of the time.

`--impl reference` times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gated_delta_rule_57_gb300 import inputs  # noqa: E402

METRIC = "KDA prefill tokens/s (B=8,T=8192,H=32,d=128,bf16) & decode GB/s; % of roofline"
PREFILL = inputs.PREFILL_B8_T8K
DECODE = inputs.DECODE_N256
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
KERNEL_SOURCES = {
    "prefill": "gated_delta_rule_57_gb300/csrc/kda_chunk_tc.cu",
    "decode": "gated_delta_rule_57_gb300/csrc/kda_decode.cu",
}


# --------------------------------------------------------------------------
# algorithmic traffic (bytes the method must move, nothing more)
# --------------------------------------------------------------------------
def prefill_bytes(w, B=None):
    B = w.B if B is None else B
    th = B * w.T * w.H
    esz = 2 if w.io == "bf16" else 4
    per_th = esz * (2 * w.dk + 2 * w.dv) + 4 * w.dk + 4  # q, k, v, o + g + beta
    states = 2 * B * w.H * w.dk * w.dv * 4 if w.h0_std is not None else B * w.H * w.dk * w.dv * 4
    return th * per_th + states


def decode_bytes(w):
    nh = w.N * w.H
    esz = 2 if w.io == "bf16" else 4
    return nh * (2 * w.dk * w.dv * 4 + esz * (2 * w.dk + 2 * w.dv) + 4 * w.dk + 4)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def file_sha(rel):
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(which):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source is unchanged since the capture; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(which)
    if not d or d.get("source_sha256_16") != file_sha(KERNEL_SOURCES[which]):
        return None
    return d.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, smax, reasons = [], None, set()
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# distributed helpers (weak scaling: one independent batch per rank)
# --------------------------------------------------------------------------
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist.get_rank(), world, int(os.environ.get("LOCAL_RANK", "0"))
    return 0, 1, 0


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base, rank):
    return base + 7919 * rank


def job_value(units_per_rank, ms_per_step_max, world):
    """Whole-job throughput: every rank processes its own units in a step that
    takes the slowest rank's time."""
    return world * units_per_rank / (ms_per_step_max * 1e-3)


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------
def time_prefill(x, steps, warmup, world, device):
    from gated_delta_rule_57_gb300 import kda
    w = PREFILL
    o = torch.empty_like(x["v"])
    hT = torch.empty(w.B, w.H, w.dk, w.dv, dtype=torch.float32, device=device)
    # the prefill's workspace (state handoffs of the balanced schedule), allocated once
    ws = torch.empty(max(16, kda.kda_chunk_fwd_workspace_size(w.B, w.T, w.H, w.dk, w.dv,
                                                             x["q"].dtype)),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def step():
        kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], o=o, hT=hT,
                          workspace=ws, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    total_ms = start.elapsed_time(end)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    return total_ms, launch_ms, o, hT


def time_prefill_e2e(xh, steps, warmup, device):
    """The same step through the public call, from pinned host memory and back.

    Batch rows are independent sequences, so the step is pipelined by row: row
    b's inputs go up on a copy stream, its kda_chunk_fwd runs on one of four
    compute streams as soon as they land, and its o and hT come back on a third
    stream, overlapping the upload of row b + 1. Every byte of every step still
    crosses the host link inside the timed region."""
    from gated_delta_rule_57_gb300 import kda
    w = PREFILL
    names = ("q", "k", "v", "g", "beta", "h0")
    xd = {n: torch.empty_like(xh[n], device=device) for n in names}
    o_d = torch.empty_like(xd["v"])
    hT_d = torch.empty(w.B, w.H, w.dk, w.dv, dtype=torch.float32, device=device)
    o_h = torch.empty_like(o_d, device="cpu").pin_memory()
    hT_h = torch.empty_like(hT_d, device="cpu").pin_memory()
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    s_c = [torch.cuda.Stream(device) for _ in range(4)]
    h2d = sum(xh[n].numel() * xh[n].element_size() for n in names)
    d2h = o_h.numel() * o_h.element_size() + hT_h.numel() * hT_h.element_size()

    # Per-row events of the previous step: a row's inputs are not overwritten
    # before its kernel has read them, nor its outputs before they went out.
    done_c = [None] * w.B
    done_out = [None] * w.B

    def step():
        for b in range(w.B):
            e_in = torch.cuda.Event()
            if done_c[b] is not None:
                s_in.wait_event(done_c[b])
            with torch.cuda.stream(s_in):
                for n in names:
                    xd[n][b].copy_(xh[n][b], non_blocking=True)
                e_in.record(s_in)
            sc = s_c[b % len(s_c)]
            sc.wait_event(e_in)
            if done_out[b] is not None:
                sc.wait_event(done_out[b])
            kda.kda_chunk_fwd(xd["q"][b:b + 1], xd["k"][b:b + 1], xd["v"][b:b + 1],
                              xd["g"][b:b + 1], xd["beta"][b:b + 1], xd["h0"][b:b + 1],
                              o=o_d[b:b + 1], hT=hT_d[b:b + 1], stream=sc)
            done_c[b] = torch.cuda.Event()
            done_c[b].record(sc)
            s_out.wait_event(done_c[b])
            with torch.cuda.stream(s_out):
                o_h[b].copy_(o_d[b], non_blocking=True)
                hT_h[b].copy_(hT_d[b], non_blocking=True)
            done_out[b] = torch.cuda.Event()
            done_out[b].record(s_out)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    # The host link alone: the step's input bytes up as one copy from one
    # pinned buffer and its output bytes down as one copy into another, at
    # the same time on two streams, nothing else. Copy engines and SM loads of
    # mapped host memory top out at the same rate on this link, so no step
    # that moves these bytes can take less.
    hb_in = torch.empty(h2d, dtype=torch.uint8).pin_memory()
    db_in = torch.empty(h2d, dtype=torch.uint8, device=device)
    hb_out = torch.empty(d2h, dtype=torch.uint8).pin_memory()
    db_out = torch.empty(d2h, dtype=torch.uint8, device=device)

    def link():
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t2 = torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        s_out.wait_event(t0)
        with torch.cuda.stream(s_in):
            db_in.copy_(hb_in, non_blocking=True)
        with torch.cuda.stream(s_out):
            hb_out.copy_(db_out, non_blocking=True)
        t1.record(s_in)
        t2.record(s_out)
        torch.cuda.synchronize()
        return max(t0.elapsed_time(t1), t0.elapsed_time(t2))

    link()
    # Nine timed runs of `steps` pipelined steps, each right after one timing
    # of the link alone. Inside a run every step is timed too: an event on the
    # upload stream before each step's first copy, so the interval between two
    # marks is the pipeline's period (uploads of one step, overlapped with the
    # compute and downloads of the step before). The median step is the
    # number; every run, its link time and the step spread are reported. (On a
    # shared machine the host link itself slows down for ~180 ms in every
    # ~480 ms or so: a run of ten steps overlaps such a window more often than
    # not, a single step much less often, so the median step resolves the
    # undisturbed rate that the median run only hits by chance.)
    runs, links, step_ms = [], [], []
    for _ in range(9):
        links.append(link())
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        start.record(s_in)
        for i in range(steps):
            marks[i].record(s_in)
            step()
        marks[steps].record(s_in)
        end.record(s_out)
        torch.cuda.synchronize()
        runs.append(start.elapsed_time(end) / steps)
        step_ms += [marks[i].elapsed_time(marks[i + 1]) for i in range(steps)]
    e2e_ms = statistics.median(step_ms)
    del hb_in, db_in, hb_out, db_out
    return e2e_ms, links, h2d, d2h, o_h, hT_h, runs, step_ms


def time_decode(device, seed, warmup=10):
    from gated_delta_rule_57_gb300 import kda
    w = DECODE
    x = inputs.decode_inputs(w, device, seed=seed)
    S = x["S"]
    o = torch.empty(w.N, w.H, w.dv, dtype=inputs.io_dtype(w.io), device=device)
    stream = torch.cuda.current_stream()
    for s in range(warmup):
        kda.kda_decode_step(x["q"][s], x["k"][s], x["v"][s], x["g"][s], x["beta"][s], S, o=o,
                            stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(w.steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for s in range(w.steps):
        ev[s][0].record(stream)
        kda.kda_decode_step(x["q"][s], x["k"][s], x["v"][s], x["g"][s], x["beta"][s], S, o=o,
                            stream=stream)
        ev[s][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    total = start.elapsed_time(end)
    per = [a.elapsed_time(b) for a, b in ev]
    return total / w.steps, statistics.mean(per), w.steps


def spec_bytes(w, K):
    """Algorithmic bytes of one verify (state read, K tokens in, K outputs) plus
    one commit of all K tokens (state read and written, K tokens in)."""
    nh = w.N * w.H
    esz = 2 if w.io == "bf16" else 4
    state = w.dk * w.dv * 4
    tok_in = esz * (2 * w.dk + w.dv) + 4 * w.dk + 4
    verify = nh * (state + K * (tok_in + esz * w.dv))
    commit = nh * (2 * state + K * tok_in)
    return verify + commit


def time_spec_decode(device, seed, K=4, iters=50, warmup=5):
    """Speculative decoding round: verify K draft tokens, then commit them all."""
    from gated_delta_rule_57_gb300 import kda
    w = DECODE
    x = inputs.prefill_inputs(
        inputs.PrefillWorkload("draft", w.N, K, w.H, w.dk, w.dv, w.io, seed, h0_std=w.S_std),
        device)
    S = x["h0"]
    o = torch.empty_like(x["v"])
    stream = torch.cuda.current_stream()

    def rnd():
        kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S, o=o, stream=stream)
        kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S, commit=True,
                             want_o=False, stream=stream)

    for _ in range(warmup):
        rnd()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(iters):
        rnd()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters, iters * 2


def time_single_and_segmented(w, device, seed, iters, warmup, flush_l2=False):
    """A workload with few sequences (B*H well below the SM count), timed in
    one pass (kda_chunk_fwd), split in time into the segment count
    kda_chunk_fwd_segments_hint picks (kda_chunk_fwd_segmented: segment
    pass, scan, correction), and split as planned on the device from the
    decay statistic (kda_chunk_fwd_segmented with nseg = 0: the probe and
    planning kernels, then the three passes reading the plan; all of it inside
    each timed step, no host round trip). Each call is timed alone
    with CUDA events; with flush_l2 a 256 MB buffer is written before each
    timed call, so inputs that fit in part in L2 start cold. Returns
    (single-pass ms, segmented ms, nseg, launches per segmented call,
    decay-planned ms, its (nseg, lead) in the last timed step)."""
    from gated_delta_rule_57_gb300 import kda
    x = inputs.prefill_inputs(w, device, seed=seed)
    o = torch.empty_like(x["v"])
    hT = torch.empty(w.B, w.H, w.dk, w.dv, dtype=torch.float32, device=device)
    nseg = kda.kda_chunk_fwd_segments_hint(w.B, w.T, w.H, w.dk, w.dv)
    ws = torch.empty(max(1, kda.kda_chunk_fwd_segmented_workspace_size(
        w.B, w.T, w.H, w.dk, w.dv, nseg=nseg)), dtype=torch.uint8, device=device)
    ws_plan = torch.empty(max(1, kda.kda_chunk_fwd_segmented_workspace_size(
        w.B, w.T, w.H, w.dk, w.dv, nseg=0)), dtype=torch.uint8, device=device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device) if flush_l2 else None
    stream = torch.cuda.current_stream()

    def single():
        kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], o=o, hT=hT,
                          stream=stream)

    def segmented():
        kda.kda_chunk_fwd_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                    nseg=nseg, o=o, hT=hT, workspace=ws, stream=stream)

    def decay_planned():
        kda.kda_chunk_fwd_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                    nseg=0, o=o, hT=hT, workspace=ws_plan, stream=stream)

    res = []
    for f in (single, segmented, decay_planned):
        for _ in range(warmup):
            f()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(iters)]
        for i in range(iters):
            if flush is not None:
                flush.fill_(i & 0xff)
            ev[i][0].record(stream)
            f()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        res.append(statistics.mean(a.elapsed_time(b) for a, b in ev))
    # the plan the device chose, recomputed by the host's copy of the planner
    planned = kda.kda_chunk_fwd_segments_hint_decay(
        w.B, w.T, w.H, w.dk, w.dv, probe=kda.kda_chunk_fwd_decay_probe(x["g"]))
    del x, o, ws, ws_plan, flush
    torch.cuda.empty_cache()
    return res[0], res[1], nseg, (3 if nseg > 1 else 1), res[2], planned


def few_sequences_obj(w, device, rank, world, peaks, iters, warmup, flush_l2):
    """JSON object of time_single_and_segmented for workload w."""
    t1, ts, nseg, launches, td, (nd, ld) = time_single_and_segmented(
        w, device, rank_seed(w.seed, rank), iters, warmup, flush_l2)
    t1 = max_over_ranks(t1, world, device)
    ts = max_over_ranks(ts, world, device)
    td = max_over_ranks(td, world, device)
    nbytes = prefill_bytes(w)
    tok = w.B * w.T
    return {
        "workload": w.name, "B": w.B, "T": w.T, "H": w.H,
        "single_pass": {"ms_per_step": t1, "value": job_value(tok, t1, world),
                        "unit": "tokens/s",
                        "frac_of_peak_hbm": nbytes / (t1 * 1e-3) / 1e9 / peaks["hbm_gbs"]},
        "segmented": {"nseg": nseg, "ms_per_step": ts, "value": job_value(tok, ts, world),
                      "unit": "tokens/s",
                      "frac_of_peak_hbm": nbytes / (ts * 1e-3) / 1e9 / peaks["hbm_gbs"],
                      "launches_per_step": launches},
        "segmented_decay_planned": {
            "nseg": nd, "lead": ld, "ms_per_step": td, "value": job_value(tok, td, world),
            "unit": "tokens/s",
            "frac_of_peak_hbm": nbytes / (td * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "launches_per_step": 5,
            "what": "kda_chunk_fwd_segmented with nseg = 0: decay probe of g and planning "
                    "kernel, then the passes reading the plan, all inside the timed step; "
                    "nseg and lead as the host's copy of the planner gives them"},
        "speedup": t1 / ts,
        "speedup_decay_planned": t1 / td,
        "algorithmic_bytes_per_step": nbytes,
        "l2": ("256 MB written between timed calls" if flush_l2
               else f"inputs larger than L2 ({nbytes / 1e9:.1f} GB per step)"),
    }


def oracle_sample(budget_s, max_b=None, check=None):
    """Oracle on whole batch rows of the prefill workload until ~budget_s;
    check(x, o_ref, hT_ref), when given, sees every row (outside the timing)."""
    import oracle
    w = PREFILL
    rows = w.B if max_b is None else max_b
    tokens, elapsed, done = 0, 0.0, 0
    for b in range(rows):
        x = inputs.prefill_inputs(w, "cpu", B=1, seed=w.seed + 101 * b)
        t0 = time.perf_counter()
        o_ref, h_ref = oracle.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
        elapsed += time.perf_counter() - t0
        if check is not None:
            check(x, o_ref, h_ref)
        tokens += w.T
        done += 1
        if elapsed >= budget_s:
            break
    return tokens, elapsed, done


def run_ours(args):
    rank, world, local = dist_setup(args.gpus)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from gated_delta_rule_57_gb300 import kda
    kda.lib()  # fail loudly now if the CUDA library is missing
    w = PREFILL
    x = inputs.prefill_inputs(w, device, seed=rank_seed(w.seed, rank))
    torch.cuda.synchronize()

    with ClockSampler(local) as clk:
        total_ms, launch_ms, o_dev, hT_dev = time_prefill(x, args.steps, args.warmup, world,
                                                          device)
    clocks = clk.summary()
    ms_step = max_over_ranks(total_ms / args.steps, world, device)
    tokens_per_rank = w.B * w.T
    value = job_value(tokens_per_rank, ms_step, world)

    peaks, peak_src = load_peaks()
    alg_bytes = prefill_bytes(w)
    launch_avg = statistics.mean(launch_ms)
    achieved = alg_bytes / (launch_avg * 1e-3) / 1e9
    traffic = recorded_traffic("prefill")

    # end to end through the same call, pinned host buffers, copies timed
    xh = {n: x[n].cpu().pin_memory() for n in ("q", "k", "v", "g", "beta", "h0")}
    e2e_ms, e2e_links, h2d, d2h, o_host, hT_host, e2e_runs, e2e_steps = time_prefill_e2e(
        xh, max(3, min(args.steps, 10)), 2, device)
    link_ms = statistics.median(e2e_links)
    link_frac = link_ms / e2e_ms
    # the pipelined host round trip must reproduce the device-resident result exactly
    e2e_exact = bool(torch.equal(o_host, o_dev.cpu()) and torch.equal(hT_host, hT_dev.cpu()))
    link_ms = max_over_ranks(link_ms, world, device)
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    del xh

    dec_ms, dec_launch_ms, dec_steps = time_decode(device, rank_seed(DECODE.seed, rank))
    dec_bytes = decode_bytes(DECODE)
    dec_gbs = job_value(dec_bytes, max_over_ranks(dec_ms, world, device), world) / 1e9
    dec_ach = dec_bytes / (dec_launch_ms * 1e-3) / 1e9
    dec_traffic = recorded_traffic("decode")

    spec_ms, spec_launches = time_spec_decode(device, rank_seed(DECODE.seed + 1, rank))
    spec_b = spec_bytes(DECODE, 4)
    spec_gbs = job_value(spec_b, max_over_ranks(spec_ms, world, device), world) / 1e9

    t4k_obj = few_sequences_obj(inputs.PREFILL_T4K, device, rank, world, peaks, iters=20,
                                warmup=3, flush_l2=True)
    long_obj = None
    if not args.no_long:
        long_obj = few_sequences_obj(inputs.PREFILL_T1M, device, rank, world, peaks, iters=3,
                                     warmup=1, flush_l2=False)

    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        errs = []

        def check(xr, o_ref, h_ref):
            # the kernel on the same batch row, against the oracle's output
            xd = {n: t.to(device) for n, t in xr.items()}
            o, hT = kda.kda_chunk_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], xd["h0"])
            torch.cuda.synchronize()
            od = o.double().cpu().numpy()
            eo = float(abs(od - o_ref).max() / abs(o_ref).max())
            hd = hT.double().cpu().numpy()
            eh = float(((hd - h_ref) ** 2).sum() ** 0.5 / (h_ref ** 2).sum() ** 0.5)
            errs.append((eo, eh))

        tok, el, rows = oracle_sample(args.cpu_budget, check=check)
        cpu = {"value": tok / el, "unit": "tokens/s", "cores": oracle.max_threads(),
               "kind": "oracle",
               "sample": f"{rows} of {w.B} batch rows x T={w.T} x H={w.H} (fp64 token loop, "
                         f"{el:.1f} s wall)"}
        parity = {"sample": f"{rows} batch rows of the workload (T={w.T} x H={w.H} each, own "
                            f"seeds) through kda_chunk_fwd against the fp64 oracle",
                  "o_max_rel_err": max(e[0] for e in errs),
                  "hT_rel_frobenius_err": max(e[1] for e in errs),
                  "tolerance": {"o": 2e-2, "hT": 1e-2}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "dk": w.dk,
                       "dv": w.dv, "io": "bf16 q/k/v/o, fp32 g/beta/h0/hT",
                       "global_batch": world * w.B, "seq_len": w.T,
                       "parallelism": f"dp{world} (independent sequences per GPU)",
                       "l2": f"inputs larger than L2 ({alg_bytes / 1e9:.2f} GB per step)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "traffic": traffic, "peak_source": peak_src,
                         "algorithmic_bytes_per_launch": alg_bytes,
                         "kernel": "kda_chunk_fwd (prefill)"},
            "cpu_baseline": cpu,
            "parity": parity,
            "e2e": {"value": job_value(tokens_per_rank, e2e_ms, world), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "pipelined_by_batch_row": True,
                    "what": "median over the timed steps of the step period (an event on the "
                            "upload stream before each step); runs_ms_per_step: each run of "
                            "consecutive steps, start of its first upload to end of its last "
                            "download, per step",
                    "steps_timed": len(e2e_steps),
                    "steps_slower_than_median_by_10pct": sum(t > 1.1 * e2e_ms for t in e2e_steps),
                    "median_run_ms_per_step": statistics.median(e2e_runs),
                    "runs_ms_per_step": e2e_runs,
                    "best_run_ms_per_step": min(e2e_runs),
                    "runs_slower_than_best_by_10pct": sum(r > 1.1 * min(e2e_runs)
                                                          for r in e2e_runs),
                    "matches_device_result": e2e_exact,
                    "host_link": {"ms_per_step": link_ms,
                                  "gbs_up": h2d / (link_ms * 1e-3) / 1e9,
                                  "frac": link_frac,
                                  "runs_ms": e2e_links,
                                  "what": "the step's input bytes up as one copy and its "
                                          "output bytes down as another, concurrently, nothing "
                                          "else: the floor of any step that moves them, timed "
                                          "before each e2e run; frac = its median / the median "
                                          "step"}},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "decode": {"workload": DECODE.name, "value": dec_gbs, "unit": "GB/s",
                       "ms_per_step": dec_ms, "steps": dec_steps,
                       "roofline": {"bound": "hbm", "achieved": dec_ach,
                                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                    "frac": dec_ach / peaks["hbm_gbs"],
                                    "traffic": dec_traffic,
                                    "algorithmic_bytes_per_launch": dec_bytes},
                       "gpu_launches": dec_steps,
                       "l2": f"state larger than L2 ({dec_bytes / 1e9:.2f} GB per step)"},
            "spec_decode": {"workload": DECODE.name + ", 4 draft tokens",
                            "round": "verify 4 tokens (state read) + commit 4 tokens (state "
                                     "read and written in place)",
                            "ms_per_round": spec_ms, "value": spec_gbs, "unit": "GB/s",
                            "frac_of_peak_hbm": spec_gbs / peaks["hbm_gbs"],
                            "algorithmic_bytes_per_round": spec_b,
                            "tokens_per_s": world * DECODE.N * 4 / (spec_ms * 1e-3),
                            "gpu_launches": spec_launches},
            "prefill_t4k": t4k_obj,
            "prefill_long": long_obj,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# --------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# --------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    w = PREFILL
    per_step_rows = 1  # one batch row (8192 tokens x 32 heads) per step
    for i in range(args.warmup):
        oracle_sample(0.0, max_b=per_step_rows)
    times = []
    for i in range(args.steps):
        tok, el, _ = oracle_sample(0.0, max_b=per_step_rows)
        times.append(el)
    ms = 1e3 * statistics.mean(times)
    val = w.T * per_step_rows / (ms * 1e-3)
    cores = oracle.max_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: 1 of {w.B} batch rows x T={w.T} x H={w.H}"},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-long", action="store_true",
                    help="skip the T = 2^20 long-context measurement (52 GB of inputs)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # timing rule: at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
