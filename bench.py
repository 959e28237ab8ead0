#!/usr/bin/env python
"""Throughput of KV² compression on GB300: compressed context tokens/s over
all layers, with the roofline fraction of the dominant kernel.

One step = the whole hot path on one synthetic cache (Llama-3.1-8B shape,
16K context by default): KeyDiff proxy -> per-chunk query selection ->
tensor-core reconstruction scoring (row LSE pass + chunk column-max pass) ->
sink pinning + eviction -> headwise compaction, through kvc_compress.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank compresses its own cache (independent problems, no
collective on the data path); rank 0 prints one JSON line with the job-wide
throughput (max time over ranks).  `--impl reference` times the float64 CPU
oracle on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import kv_synth as ks  # noqa: E402

METRIC = "compressed ctx tokens/s (all layers) at Llama-8B-shape 16K; % of roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=ks.LLAMA_16K.name, choices=list(ks.KV2_CONFIGS))
    ap.add_argument("--e2e-steps", type=int, default=12)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="use only this many layers (profiling cases)")
    ap.add_argument("--proxy", choices=["keydiff", "knorm"], default="keydiff", help="stage-1 proxy")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of the step captured in a CUDA graph (launch-bound small workloads)")
    ap.add_argument("--op", choices=["compress", "decode", "episode", "q4", "epicache", "rho"], default="compress",
                    help="compress: the KV² compression step; decode: attention over the compacted cache; "
                         "episode: EpiCache per-turn match + episode cache swap; q4: Q4 codec of the cache; "
                         "epicache: EpiCache block prefill of every episode; rho: the compression step at "
                         "several reconstruction ratios")
    ap.add_argument("--decode-config", default=ks.DECODE_128K.name, choices=list(ks.DECODE_CONFIGS))
    ap.add_argument("--epi-layout", choices=["two-slab", "one-slab"], default="one-slab",
                    help="EpiCache block state: kept rows compacted into the other slab every step, or kept in "
                         "place with the kept block rows moved into evicted rows")
    return ap.parse_args()


# ---------------------------------------------------------------- workload arithmetic
def plan_of(cfg):
    """(chunk sizes, n_q per chunk) by the chunking rule of the KV² page."""
    sizes, nqs = [], []
    lo = cfg.sinks
    while lo < cfg.N:
        hi = min(lo + cfg.m, cfg.N)
        sizes.append(hi - lo)
        nqs.append(max(int(math.floor(cfg.rho * (hi - lo) + 1e-9)), 1))
        lo = hi
    return sizes, nqs


def algorithmic_work(cfg):
    """Per-step algorithmic FLOPs of the two scoring passes and bytes of the
    bandwidth-bound stages (see the design notes)."""
    sizes, nqs = plan_of(cfg)
    d, L, Hq, Hkv, N = cfg.d, cfg.L, cfg.Hq, cfg.Hkv, cfg.N
    Q = sum(nqs)
    f_lse = L * Hq * 2 * d * sum(n * (N + (n + 1) / 2) for n in nqs)
    f_col = L * Hq * 2 * d * sum(n * c for n, c in zip(nqs, sizes))
    k = int(math.floor(cfg.budget * N + 1e-9))
    b_k = L * Hkv * N * d * 2                       # one read of K
    b = {
        "keydiff": b_k + L * Hkv * N * 4,           # read K, write s
        "knorm": b_k + L * Hkv * N * 4,             # read K, write s
        "recon_gather": L * Hq * Q * d * 2 * 2 + L * Hkv * Q * d * 2 * 2,
        "evict_topk": L * Hkv * N * 4 + L * Hkv * k * 4,
        "compact": 2 * 2 * L * Hkv * k * d * 2,     # read + write kept K and V
    }
    # eviction and compaction fused into one launch
    b["evict_compact"] = b["evict_topk"] + b["compact"]
    return {"flops_lse": f_lse * cfg.passes, "flops_colmax": f_col * cfg.passes, "Q": Q, "k": k,
            "bytes": b, "flops_lse_per_launch": f_lse, "flops_colmax_per_launch": f_col}


# DRAM bytes per launch of the row-LSE kernel as ncu counted them (one pass,
# no replay) on the 4-layer case of the 16K workload, the mean of three
# launches in two captures: dram__bytes_read + dram__bytes_write = 202.58 +
# 6.12 MB (the writes are the 32-byte lse rows the column-max pass reads,
# part of them still in L2 when the kernel ends); the traffic grows with the
# number of (layer, KV head) pairs.  Reset to None whenever the kernel
# changes until it is captured again.
LSE_TRAFFIC_PER_LAYER = (202.58e6 + 6.12e6) / 4


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None

    def start(self, settle_s: float = 0.5):
        """Start sampling; returns once the first sample has arrived and the
        sampler has settled (its start-up briefly slows the GPU's host link)."""
        self.first = ""
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        import select
        r, _, _ = select.select([self.proc.stdout], [], [], 15.0)
        if r:
            self.first = self.proc.stdout.readline()
        time.sleep(settle_s)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        out = self.first + out
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        rows = [[c.strip() for c in r] for r in rows]
        if self.uuid:
            mine = [r for r in rows if r[0] == self.uuid]
            rows = mine or rows
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for nm, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle timing
class OracleSample:
    """Times the float64 oracle on a bounded sample of the workload and
    scales it to one full step.  Sample units: the KeyDiff proxy and the
    eviction of one (layer, KV head), the selection over all chunks, and the
    reconstruction scoring of one (query head, chunk) -- the oracle's
    per-head work is the same for every head, so a full step costs
    L*Hkv*(proxy + evict) + L*Hq*M*(one scoring unit) + selection."""

    def __init__(self, cfg):
        from oracle import kv2
        self.kv2 = kv2
        self.cfg = cfg
        dr = ks.gen_layer(cfg, 0, with_values=False)
        self.K0 = kv2.bf16_to_f64(dr.K[0])
        self.Q0 = kv2.bf16_to_f64(dr.Q[0])
        self.s = kv2.keydiff_head(self.K0)
        self.sel, self.chunks = kv2.select_queries(self.s, cfg.N, cfg.sinks, cfg.m, cfg.rho)
        self.k = int(math.floor(cfg.budget * cfg.N + 1e-9))
        self.unit = 0

    def per_head(self):
        kv2, cfg = self.kv2, self.cfg
        a = time.perf_counter()
        kv2.keydiff_head(self.K0)
        sc = np.random.default_rng(0).random((1, 1, cfg.N))
        kv2.evict(sc, cfg.sinks, [self.k])
        b = time.perf_counter()
        kv2.select_queries(self.s, cfg.N, cfg.sinks, cfg.m, cfg.rho)
        c = time.perf_counter()
        return b - a, c - b

    def scoring_unit(self):
        kv2 = self.kv2
        c = self.chunks[self.unit % len(self.chunks)]
        self.unit += 1
        idx = self.sel[c.off:c.off + c.nq]
        one = kv2.Chunk(c.lo, c.hi, 0, c.nq)
        a = time.perf_counter()
        kv2.recon_head(self.K0, self.Q0[idx][None], self.K0[idx], [one])
        return time.perf_counter() - a

    def full_step(self, t_head, t_sel, t_unit):
        cfg = self.cfg
        return cfg.passes * (cfg.L * cfg.Hkv * t_head + cfg.L * cfg.Hq * len(self.chunks) * t_unit + t_sel)

    def describe(self, units):
        cfg = self.cfg
        return (f"oracle on {units} (query head, chunk) scoring unit(s) of {cfg.L * cfg.Hq * len(self.chunks)} "
                f"plus KeyDiff+eviction of 1 of {cfg.L * cfg.Hkv} heads and the selection, "
                f"{cfg.name}; scaled to the full step")


def time_oracle_sample(cfg, budget_s=20.0, sampler=None):
    """(seconds per full step, description): scoring units until `budget_s`
    of CPU time (at least one)."""
    smp = sampler or OracleSample(cfg)
    t_head, t_sel = smp.per_head()
    times = []
    t0 = time.perf_counter()
    while True:
        times.append(smp.scoring_unit())
        if time.perf_counter() - t0 >= budget_s or len(times) >= 64:
            break
    t_unit = statistics.median(times)
    return smp.full_step(t_head, t_sel, t_unit), smp.describe(len(times))


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- reference arm
def run_reference(args, cfg, rank, world):
    if rank != 0:
        return
    smp = OracleSample(cfg)
    sample = []
    for _ in range(args.warmup):
        time_oracle_sample(cfg, budget_s=0.0, sampler=smp)
    desc = ""
    timed = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        full, desc = time_oracle_sample(cfg, budget_s=0.0, sampler=smp)
        timed.append(time.perf_counter() - t0)
        sample.append(full)
    t = statistics.median(sample)
    value = cfg.N / t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(cfg),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores(), "kind": "oracle",
                         "sample": "per step: " + desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        # each step times a bounded sample of the workload and scales it to
        # the full step: ms_per_step and value are extrapolated, not timed
        "extrapolated": True,
        "timed_s_per_step": statistics.median(timed),
    }
    print(json.dumps(line), flush=True)


def config_of(cfg, proxy="keydiff"):
    return {"workload": cfg.name, "proxy": proxy, "L": cfg.L, "Hkv": cfg.Hkv, "Hq": cfg.Hq, "d": cfg.d, "N": cfg.N,
            "sinks": cfg.sinks, "m": cfg.m, "rho": cfg.rho, "budget": cfg.budget, "passes": cfg.passes,
            "needle_clusters_per_layer": cfg.needles_per_layer,
            "l2": "inputs larger than L2 (K alone exceeds the 129 MB L2); no flush between steps",
            "parallelism": "independent cache per GPU"}


# ---------------------------------------------------------------- our arm
def run_ours(args, cfg, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import query_agnostic_kv_gb300 as qk
    from query_agnostic_kv_gb300 import _build

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    _build.build_library()
    qk.kvc_device_check()
    # each rank compresses its own cache
    cfg_r = ks.scaled(cfg, seed=cfg.seed + rank)
    x = ks.gen_kv2(cfg_r)
    L, H, Hq, N, S, d = cfg.L, cfg.Hkv, cfg.Hq, cfg.N, cfg.sinks, cfg.d

    def dev_bf16(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)

    K, V, Q = dev_bf16(x.K), dev_bf16(x.V), dev_bf16(x.Q)
    shape = (L, H, Hq, d, N)
    k = qk.kvc_budget_count(cfg.budget, N, S)
    kl = [k] * L
    ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, cfg.rho), dtype=torch.uint8, device=dev)
    kept = torch.empty(L * H * k, dtype=torch.int32, device=dev)
    Kc = torch.empty(L * H * k * d, dtype=torch.bfloat16, device=dev)
    Vc = torch.empty_like(Kc)
    stream = torch.cuda.current_stream()

    def step():
        qk.kvc_compress_ex(shape, args.proxy, K, V, Q, S, cfg.m, cfg.rho, cfg.passes, kl, kept, Kc, Vc, ws=ws,
                           stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    st = qk.kvc_stream_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {qk.kvc_status_string(st)}")

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    qk.kvc_profile_begin()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    prof = qk.kvc_profile_end()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1)
    st = qk.kvc_stream_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {qk.kvc_status_string(st)}")
    t_max = ms
    if world > 1:
        t = torch.tensor([ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        t_max = float(t.item())
    ms_per_step = t_max / args.steps
    value = world * N * args.steps / (t_max / 1e3)

    # ---- per-kernel breakdown and roofline of the dominant kernel
    work = algorithmic_work(cfg)
    peaks, peak_src = load_peaks()
    launches = sum(v[0] for v in prof.values())
    total_k = sum(v[1] for v in prof.values())
    kernels = {n: {"launches": v[0], "avg_ms": v[1] / v[0], "share": v[1] / total_k if total_k else None}
               for n, v in prof.items()}
    lse_avg_s = prof["recon_lse"][1] / prof["recon_lse"][0] / 1e3
    col_avg_s = prof["recon_colmax"][1] / prof["recon_colmax"][0] / 1e3
    # The timed region is a short burst (well under a second of tensor work
    # at the clocks sampled), so the burst bf16 peak is the denominator; the
    # ratio to the power-capped sustained peak is reported beside it.
    peak_tf = peaks.get("bf16_tflops")
    peak_sus = peaks.get("bf16_tflops_sustained", peak_tf)
    ach_lse = work["flops_lse_per_launch"] / lse_avg_s / 1e12
    ach_col = work["flops_colmax_per_launch"] / col_avg_s / 1e12
    traffic = None
    if LSE_TRAFFIC_PER_LAYER is not None and cfg.N == ks.LLAMA_16K.N and cfg.Hkv == ks.LLAMA_16K.Hkv:
        traffic = LSE_TRAFFIC_PER_LAYER * cfg.L
    roof = {"kernel": "recon_lse (tcgen05 row-LSE pass)", "bound": "tensor", "achieved": ach_lse,
            "peak": peak_tf, "unit": "TFLOP/s", "frac": ach_lse / peak_tf, "traffic": traffic,
            "traffic_source": "ncu dram bytes (read + write, one pass) of the 4-layer case on the current "
                              "kernel, scaled by layers",
            "peak_source": f"bf16_tflops (burst) of {peak_src} peaks",
            "frac_of_sustained": ach_lse / peak_sus,
            "algorithmic_flops_per_launch": work["flops_lse_per_launch"],
            "colmax": {"achieved": ach_col, "frac": ach_col / peak_tf}}
    hbm = peaks.get("hbm_gbs")
    bw = {}
    for name, b in work["bytes"].items():
        if name in prof:
            avg = prof[name][1] / prof[name][0] / 1e3
            bw[name] = {"GB/s": b / avg / 1e9, "frac_of_hbm": b / avg / 1e9 / hbm}
    # whole-step roofline (slower of tensor FLOPs and HBM bytes)
    f_all = work["flops_lse"] + work["flops_colmax"]
    b_all = sum(work["bytes"].values())
    t_roof = max(f_all / (peak_tf * 1e12), b_all / (hbm * 1e9))
    t_roof_sus = max(f_all / (peak_sus * 1e12), b_all / (hbm * 1e9))
    step_roof = {"t_roof_ms": t_roof * 1e3, "frac": t_roof / (ms_per_step / 1e3),
                 "tokens_per_s_at_roof": N / t_roof, "peak": "bf16_tflops (burst) and hbm_gbs",
                 "frac_of_sustained": t_roof_sus / (ms_per_step / 1e3)}

    # ---- end to end through the public API with host buffers
    e2e = None
    if args.e2e_steps > 0:
        kept_ref = kept.cpu()              # the device-resident run's result, for the check below
        hK = torch.from_numpy(x.K.view(np.int16)).view(torch.bfloat16).pin_memory()
        hV = torch.from_numpy(x.V.view(np.int16)).view(torch.bfloat16).pin_memory()
        hQ = torch.from_numpy(x.Q.view(np.int16)).view(torch.bfloat16).pin_memory()
        hkept = [torch.empty(kept.shape, dtype=torch.int32).pin_memory() for _ in range(2)]
        hKc = [torch.empty(Kc.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        hVc = [torch.empty(Vc.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        kept2 = [kept, torch.empty_like(kept)]
        Kc2 = [Kc, torch.empty_like(Kc)]
        Vc2 = [Vc, torch.empty_like(Vc)]

        # K is copied whole (the proxy and the scoring read all of it) into
        # one of two device buffers on a copy stream; V and the query pool stay
        # in pinned host memory, mapped into the device address space, and the
        # gather / compaction kernels read only the selected query rows and the
        # kept value rows across the link.  The next step's K copy starts once
        # this step's query gather has been issued (kvc_compress_ex records an
        # event there), so the two do not share the link and the copy runs
        # under the scoring passes.  Results go back to pinned host memory on a
        # third stream from double-buffered outputs.
        Kbuf = [K, torch.empty_like(K)]
        copy_stream = torch.cuda.Stream(device=dev)
        d2h_stream = torch.cuda.Stream(device=dev)
        ev_copied = [torch.cuda.Event(), torch.cuda.Event()]
        ev_free = [torch.cuda.Event(), torch.cuda.Event()]
        ev_out = [torch.cuda.Event(), torch.cuda.Event()]
        gather_done = [torch.cuda.Event(), torch.cuda.Event()]
        for evs in (ev_copied, ev_free, ev_out, gather_done):
            for ev in evs:
                ev.record(stream)       # create the events
        torch.cuda.synchronize()

        def e2e_steps(n, start_event=None):
            for i in range(n):
                bsel = i % 2
                with torch.cuda.stream(copy_stream):
                    if i == 0 and start_event is not None:
                        copy_stream.wait_event(start_event)
                    if i > 0:
                        copy_stream.wait_event(gather_done[(i - 1) % 2])
                    copy_stream.wait_event(ev_free[bsel])
                    Kbuf[bsel].copy_(hK, non_blocking=True)
                    ev_copied[bsel].record(copy_stream)
                stream.wait_event(ev_copied[bsel])
                stream.wait_event(ev_out[bsel])
                qk.kvc_compress_ex(shape, args.proxy, Kbuf[bsel], hV, hQ, S, cfg.m, cfg.rho, cfg.passes, kl,
                                   kept2[bsel], Kc2[bsel], Vc2[bsel], ws=ws, stream=stream,
                                   gather_done=gather_done[bsel])
                ev_free[bsel].record(stream)
                with torch.cuda.stream(d2h_stream):
                    d2h_stream.wait_event(ev_free[bsel])
                    hkept[bsel].copy_(kept2[bsel], non_blocking=True)
                    hKc[bsel].copy_(Kc2[bsel], non_blocking=True)
                    hVc[bsel].copy_(Vc2[bsel], non_blocking=True)
                    ev_out[bsel].record(d2h_stream)
            stream.wait_stream(d2h_stream)

        # Single-pass steps run through the three scoring phases instead, so
        # that consecutive steps overlap: while step i's row pass runs, step
        # i+1's K copy finishes; step i+1's proxy and selection then run (the
        # whole GPU), and its query gather -- reads across the host link --
        # runs beside step i's column pass (its blocks fit beside the
        # column-max CTAs); step i+2's K copy follows that gather.  Each step
        # alternates between two workspaces and output sets.  The host
        # enqueues in dependency order, so every event a stream waits on has
        # already been recorded for that step.
        if cfg.passes == 1:
            wsb = [ws, torch.empty_like(ws)]
            pb = [torch.empty(N, dtype=torch.float32, device=dev) for _ in range(2)]
            selb = [torch.empty(work["Q"], dtype=torch.int32, device=dev) for _ in range(2)]
            scoreb = [torch.empty(L * H * N, dtype=torch.float32, device=dev) for _ in range(2)]
            prep_stream = torch.cuda.Stream(device=dev)
            ev_sel = [torch.cuda.Event(), torch.cuda.Event()]
            ev_gath = [torch.cuda.Event(), torch.cuda.Event()]
            ev_done = [torch.cuda.Event(), torch.cuda.Event()]
            for evs in (ev_sel, ev_gath, ev_done):
                for ev in evs:
                    ev.record(stream)
            torch.cuda.synchronize()

            def copy_k(i, after):
                with torch.cuda.stream(copy_stream):
                    for ev in after:
                        copy_stream.wait_event(ev)
                    Kbuf[i % 2].copy_(hK, non_blocking=True)
                    ev_copied[i % 2].record(copy_stream)

            def prep_front(i):        # proxy and selection of step i
                b = i % 2
                with torch.cuda.stream(prep_stream):
                    prep_stream.wait_event(ev_copied[b])
                    if i >= 2:
                        prep_stream.wait_event(ev_done[b])   # workspace b: step i-2 is done with it
                    qk.kvc_proxy_score_kind(shape, args.proxy, Kbuf[b], pb[b], ws=wsb[b], stream=prep_stream)
                    qk.kvc_select_queries(N, S, cfg.m, cfg.rho, pb[b], selb[b], stream=prep_stream)
                    ev_sel[b].record(prep_stream)

            def prep_back(i):         # query gather of step i
                b = i % 2
                with torch.cuda.stream(prep_stream):
                    qk.kvc_recon_gather(shape, Kbuf[b], hQ, selb[b], S, cfg.m, cfg.rho, ws=wsb[b],
                                        stream=prep_stream)
                    ev_gath[b].record(prep_stream)

            def e2e_steps(n, start_event=None):
                copy_k(0, [start_event] if start_event is not None else [])
                prep_front(0)
                prep_back(0)
                if n > 1:
                    copy_k(1, [ev_gath[0]])
                for i in range(n):
                    b = i % 2
                    stream.wait_event(ev_gath[b])
                    qk.kvc_recon_rows(shape, Kbuf[b], S, cfg.m, cfg.rho, ws=wsb[b], stream=stream)
                    if i + 1 < n:
                        prep_front(i + 1)
                        stream.wait_event(ev_sel[(i + 1) % 2])
                    qk.kvc_recon_cols(shape, Kbuf[b], S, cfg.m, cfg.rho, scoreb[b], ws=wsb[b], stream=stream)
                    if i + 1 < n:
                        prep_back(i + 1)
                    stream.wait_event(ev_out[b])                 # host copies of step i-2 are done
                    qk.kvc_evict_compact(shape, scoreb[b], S, kl, kept2[b], Kbuf[b], hV, Kc2[b], Vc2[b], ws=wsb[b],
                                         stream=stream)
                    ev_done[b].record(stream)
                    if i + 2 < n:
                        copy_k(i + 2, [ev_gath[(i + 1) % 2], ev_done[b]])
                    with torch.cuda.stream(d2h_stream):
                        d2h_stream.wait_event(ev_done[b])
                        hkept[b].copy_(kept2[b], non_blocking=True)
                        hKc[b].copy_(Kc2[b], non_blocking=True)
                        hVc[b].copy_(Vc2[b], non_blocking=True)
                        ev_out[b].record(d2h_stream)
                stream.wait_stream(d2h_stream)

        e2e_steps(2)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_steps(args.e2e_steps, start_event=a)
        b.record(stream)
        torch.cuda.synchronize()
        e_ms = a.elapsed_time(b)
        if world > 1:
            t = torch.tensor([e_ms], device=dev, dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e_ms = float(t.item())
        st = qk.kvc_stream_status(stream)
        if st != 0:
            raise RuntimeError(f"device status after e2e steps: {qk.kvc_status_string(st)}")
        # every step compresses the same inputs: the last one must match the device-resident run
        if not torch.equal(hkept[(args.e2e_steps - 1) % 2], kept_ref):
            raise RuntimeError("end-to-end steps kept other positions than the device-resident run")
        # bytes crossing host -> device per step: K copied, plus the query rows
        # and kept V rows the kernels read from mapped host memory
        h2d = hK.numel() * 2 + cfg.passes * L * Hq * work["Q"] * d * 2 + L * H * k * d * 2
        d2h = hkept[0].numel() * 4 + (hKc[0].numel() + hVc[0].numel()) * 2
        e2e = {"value": world * N * args.e2e_steps / (e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms / args.e2e_steps,
               "how": ("pinned host inputs: K copied each step on a copy stream into one of two device buffers; "
                       "query rows and kept V rows read in place; kept indices and compacted K/V copied back to "
                       "pinned host memory on another stream; " +
                       ("the scoring phases of consecutive steps overlap: the next step's proxy, selection and "
                        "query gather run on a second stream, the gather beside this step's column-max pass, and "
                        "the K copy after that gather, under the next row pass"
                        if cfg.passes == 1 else
                        "each K copy starts after the previous step's query gather, under its scoring passes") +
                       "; the first step's K copy and preparation have nothing to overlap and are inside the timed "
                       "region")}

    # ---- CPU oracle baseline (rank 0, one GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        full, desc = time_oracle_sample(cfg, budget_s=20.0)
        cpu = {"value": N / full, "unit": UNIT, "cores": cores(), "kind": "oracle", "sample": desc,
               "extrapolated": True, "extrapolated_s_per_step": full}

    graph = None
    if args.graph:
        # the same step captured once into a CUDA graph, replayed; the eager
        # per-kernel profile above stays the source of the roofline figures
        gs = torch.cuda.Stream(device=dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            qk.kvc_compress_ex(shape, args.proxy, K, V, Q, S, cfg.m, cfg.rho, cfg.passes, kl, kept, Kc, Vc, ws=ws,
                               stream=torch.cuda.current_stream())
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        ga = torch.cuda.Event(enable_timing=True)
        gb = torch.cuda.Event(enable_timing=True)
        ga.record(gs)
        with torch.cuda.stream(gs):
            for _ in range(args.steps):
                g.replay()
        gb.record(gs)
        torch.cuda.synchronize()
        st = qk.kvc_stream_status(gs)
        if st != 0:
            raise RuntimeError(f"device status after graph replays: {qk.kvc_status_string(st)}")
        g_ms = ga.elapsed_time(gb) / args.steps
        graph = {"ms_per_step": g_ms, "eager_ms_per_step": ms_per_step,
                 "eager_value": value}
        ms_per_step = g_ms
        value = world * N / (g_ms / 1e3)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_of(cfg, args.proxy),
            "roofline": roof, "step_roofline": step_roof, "bandwidth": bw, "kernels": kernels,
            "gpu_launches": launches, "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu,
        }
        if graph is not None:
            line["cuda_graph"] = graph
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- decode attention leg
DECODE_METRIC = "decode attention over compacted KV caches: algorithmic HBM GB/s"


def decode_bytes(cfg):
    """Algorithmic bytes of one decode launch: every kept K and V row once,
    the queries, the outputs and their lse."""
    rows = cfg.n_seg * cfg.kept
    return rows * 128 * 2 * 2 + cfg.n_seg * cfg.G * (128 * 2 + 128 * 4 + 4)


# DRAM bytes per launch per sequence of decode_kernel as ncu counted them on the
# 16-sequence case (dram__bytes_read + dram__bytes_write = 867.78 MB / 16); the
# kernel's traffic grows in proportion to the rows.  Reset to None whenever the
# kernel changes until it is captured again.
DECODE_TRAFFIC_PER_SEQ = 867.78e6 / 16


def decode_config_of(cfg):
    return {"workload": cfg.name, "seqs": cfg.seqs, "Hkv": cfg.Hkv, "G": cfg.G, "kept_rows_per_head": cfg.kept,
            "d": 128, "layers_per_step": 1,
            "l2": "inputs larger than L2 (3.4 GB of K and V); no flush between steps",
            "parallelism": "independent batch per GPU"}


def time_decode_oracle(cfg, x, budget_s=15.0):
    """Oracle on whole sampled segments (host copies), scaled to a full launch."""
    from oracle import decode
    K = x["K"]
    rng = np.random.default_rng(1)
    t_used, done = 0.0, 0
    while done == 0 or (t_used < budget_s and done < cfg.n_seg):
        s = int(rng.integers(cfg.n_seg))
        o, n = int(x["seg_off"][s]), int(x["seg_len"][s])
        Ks = K[o:o + n].double().cpu().numpy()
        Vs = x["V"][o:o + n].double().cpu().numpy()
        q = x["q"][s:s + 1].double().cpu().numpy()
        a = time.perf_counter()
        decode.decode_attention(Ks, Vs, [0], [n], q)
        t_used += time.perf_counter() - a
        done += 1
    per_launch = t_used / done * cfg.n_seg
    return per_launch, f"{done} whole segments of {cfg.kept} rows (G={cfg.G}) timed, scaled x{cfg.n_seg / done:.1f}"


def run_decode(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import query_agnostic_kv_gb300 as qk
    from query_agnostic_kv_gb300 import _build

    cfg = ks.DECODE_CONFIGS[args.decode_config]
    if args.impl == "reference":
        if rank != 0:
            return
        x = ks.gen_decode(ks.DecodeConfig(**{**cfg.__dict__, "seed": cfg.seed}), "cpu")
        for _ in range(args.warmup):
            time_decode_oracle(cfg, x, budget_s=0.0)
        samples, desc = [], ""
        for _ in range(args.steps):
            t, desc = time_decode_oracle(cfg, x, budget_s=2.0)
            samples.append(t)
        t = statistics.median(samples)
        v = decode_bytes(cfg) / t / 1e9
        print(json.dumps({
            "impl": "reference", "metric": DECODE_METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": decode_config_of(cfg),
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores(), "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)
        return

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    _build.build_library()
    qk.kvc_device_check()
    x = ks.gen_decode(ks.DecodeConfig(**{**cfg.__dict__, "seed": cfg.seed + rank}), dev)
    n_seg, G = cfg.n_seg, cfg.G
    ws = torch.empty(qk.kvc_decode_workspace_size(n_seg, G, cfg.kept), dtype=torch.uint8, device=dev)
    out = torch.empty(n_seg, G, 128, dtype=torch.float32, device=dev)
    lse = torch.empty(n_seg, G, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(q=None):
        qk.kvc_decode_attention(x["K"], x["V"], x["seg_off"], x["seg_len"], cfg.kept, x["q"] if q is None else q,
                                out, lse, ws=ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    st = qk.kvc_stream_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {qk.kvc_status_string(st)}")
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    qk.kvc_profile_begin()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    prof = qk.kvc_profile_end()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1)
    st = qk.kvc_stream_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {qk.kvc_status_string(st)}")
    if world > 1:
        t = torch.tensor([ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    B = decode_bytes(cfg)
    value = world * B * args.steps / (ms / 1e3) / 1e9
    peaks, peak_src = load_peaks()
    hbm = peaks.get("hbm_gbs")
    n_l, tot = prof["decode_attn"]
    ach = B / (tot / n_l / 1e3) / 1e9
    roof = {"kernel": "decode_attn (bulk-copy ring, CUDA-core f32x2)", "bound": "hbm", "achieved": ach,
            "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
            "traffic": None if DECODE_TRAFFIC_PER_SEQ is None else DECODE_TRAFFIC_PER_SEQ * cfg.seqs,
            "traffic_source": "ncu dram bytes of the 16-sequence case, scaled by sequences",
            "peak_source": f"hbm_gbs of {peak_src} peaks", "algorithmic_bytes_per_launch": B}
    kernels = {n: {"launches": v[0], "avg_ms": v[1] / v[0]} for n, v in prof.items()}

    # end to end: this step's queries from pinned host memory in, outputs and lse back out
    e2e = None
    if args.e2e_steps > 0:
        hq = x["q"].cpu().pin_memory()
        dq = torch.empty_like(x["q"])
        hout = torch.empty(out.shape, dtype=torch.float32).pin_memory()
        hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()

        def e2e_step():
            dq.copy_(hq, non_blocking=True)
            step(dq)
            hout.copy_(out, non_blocking=True)
            hlse.copy_(lse, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e_ms = a.elapsed_time(b)
        if world > 1:
            t = torch.tensor([e_ms], device=dev, dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e_ms = float(t.item())
        e2e = {"value": world * B * args.e2e_steps / (e_ms / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": hq.numel() * 2, "d2h_bytes_per_step": (hout.numel() + hlse.numel()) * 4,
               "ms_per_step": e_ms / args.e2e_steps,
               "how": "the compacted cache is resident (serving state); each step copies its queries from pinned "
                      "host memory and its outputs and lse back to pinned host memory"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        xh = {k: (v.cpu() if hasattr(v, "cpu") else v) for k, v in x.items()}
        t, desc = time_decode_oracle(cfg, xh)
        cpu = {"value": B / t / 1e9, "unit": "GB/s", "cores": cores(), "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps({
            "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": decode_config_of(cfg),
            "roofline": roof, "kernels": kernels, "gpu_launches": sum(v[0] for v in prof.values()),
            "clocks": clocks, "e2e": e2e,
            "cpu_baseline": cpu}), flush=True)


# ---------------------------------------------------------------- EpiCache per-turn leg
EPISODE_METRIC = ("EpiCache turn (match + write back and load of one compressed episode cache): "
                  "GB/s over the host link")


def episode_oracle_turn(cfg, De, warmup, steps):
    """One turn on the host with the oracle: match, pack one episode, and the
    two host copies standing for the write-back and the load."""
    from oracle import episode, kv2
    E, H = cfg.episodes, cfg.Hkv
    budgets = [int(x) for x in kv2.layer_budgets(ks.gen_sensitivity(cfg).astype(np.float64), cfg.alpha,
                                                  cfg.mean_budget, cfg.sinks)]
    rng = np.random.default_rng(0)
    layers = [rng.integers(0, 1 << 15, size=(H, b, 128), dtype=np.int16) for b in budgets]
    pos = [np.tile(np.arange(b, dtype=np.int32), (H, 1)) for b in budgets]
    C, Q = ks.gen_turn_embeddings(E, De, 1)
    samples = []
    for i in range(warmup + steps):
        a = time.perf_counter()
        episode.nearest_episode(Q.astype(np.float64), C.astype(np.float64))
        K, V, P, _ = episode.pack_cache(layers, layers, pos)
        out = np.empty_like(K)
        np.copyto(out, K)                 # write back
        np.copyto(out, V)                 # load
        if i >= warmup:
            samples.append(time.perf_counter() - a)
    t = statistics.median(samples)
    return 2 * 2 * K.nbytes / t / 1e9, t, "one turn: oracle match (E=4, De=1024) + pack of one episode + two host copies"


def run_episode(args, rank, world, local_rank):
    import torch
    import query_agnostic_kv_gb300 as qk
    from query_agnostic_kv_gb300 import _build

    cfg = ks.EPI_3B
    E, De = cfg.episodes, 1024
    L, H = cfg.L, cfg.Hkv
    if args.impl == "reference":
        if rank != 0:
            return
        v, t, desc = episode_oracle_turn(cfg, De, args.warmup, args.steps)
        print(json.dumps({
            "impl": "reference", "metric": EPISODE_METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "epicache-llama3.2-3b-M8k-swap", "L": L, "Hkv": H, "mean_budget": cfg.mean_budget,
                       "alpha": cfg.alpha},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores(), "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)
        return

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    _build.build_library()
    qk.kvc_device_check()
    budgets = qk.kvc_layer_budgets(ks.gen_sensitivity(cfg).tolist(), cfg.alpha, cfg.mean_budget, cfg.sinks)
    cap = max(budgets)
    # a block state holding each layer's full budget (as at the end of an episode's block prefill)
    g = torch.Generator(device=dev).manual_seed(5)
    slabs = [torch.randn(L * H * cap * 128, generator=g, device=dev).to(torch.bfloat16) for _ in range(2)]
    slabs += [torch.empty_like(slabs[0]) for _ in range(2)]
    pos = [torch.arange(L * H * cap, dtype=torch.int32, device=dev) for _ in range(2)]
    st = qk.kvc_block_state_init(L, H, H * 3, cap, cfg.sinks, budgets, slabs[0], slabs[1], pos[0], slabs[2],
                                 slabs[3], pos[1])
    for l in range(L):
        st.len[l] = budgets[l]
    R = qk.kvc_episode_rows(st)
    img = [torch.empty(2 * R, 128, dtype=torch.bfloat16, device=dev) for _ in range(2)]   # [K rows; V rows]
    img_pos = torch.empty(R, dtype=torch.int32, device=dev)
    host = [torch.empty(2 * R, 128, dtype=torch.bfloat16).pin_memory() for _ in range(E)]
    stream = torch.cuda.current_stream()
    s_out, s_in = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def pack(i=0):
        qk.kvc_episode_pack(st, img[i][:R], img[i][R:], img_pos, stream=stream)

    for _ in range(3):
        pack()
    qk.kvc_episode_swap(img[0], host[0], host[1], img[1], out_stream=s_out, in_stream=s_in)
    torch.cuda.synchronize()
    assert qk.kvc_stream_status() == 0

    def timed(fn, n):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(n):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    C, Qb = ks.gen_turn_embeddings(E, De, 4096)
    c_d, q_d = torch.from_numpy(C).to(dev), torch.from_numpy(Qb).to(dev)
    ep = torch.empty(4096, dtype=torch.int32, device=dev)

    def swap_step(i, match=True):
        if match:
            qk.kvc_episode_match(q_d[:1], c_d, ep[:1], stream=stream)
        ev = torch.cuda.Event()
        ev.record(stream)
        s_out.wait_event(ev)
        s_in.wait_event(ev)
        qk.kvc_episode_swap(img[i % 2], host[i % E], host[(i + 1) % E], img[(i + 1) % 2], out_stream=s_out,
                            in_stream=s_in)
        stream.wait_stream(s_out)
        stream.wait_stream(s_in)

    def load_only(i):
        qk.kvc_episode_swap(host_in=host[i % E], dev_in=img[i % 2], in_stream=stream)

    def store_only(i):
        qk.kvc_episode_swap(img[i % 2], host[i % E], out_stream=stream)

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    for _ in range(args.warmup):
        swap_step(0)

    def one(fn, i):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn(i)
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b)

    # The host link is shared with other work on the machine, so the kinds of
    # copy are interleaved step by step and each reported as a median.
    # nvidia-smi queries stall host-link copies for tens of milliseconds, so
    # the turns are timed without the clock sampler; the clocks come from a
    # second, identical pass whose times are reported beside it.
    torch.cuda.synchronize()
    t_turn, t_swap, t_load, t_store, t_sampled = [], [], [], [], []
    qk.kvc_profile_begin()
    for i in range(args.steps):
        t_turn.append(one(swap_step, i))
    prof = qk.kvc_profile_end()
    sampler = ClockSampler(uuid)
    sampler.start()
    for i in range(args.steps):
        t_sampled.append(one(swap_step, i))
    clocks = sampler.stop()
    clocks["note"] = ("sampled during a second pass of the same turns (median %.2f ms per turn while sampling); "
                      "nvidia-smi queries stall host-link copies" % statistics.median(t_sampled))
    for i in range(args.steps):
        t_swap.append(one(lambda k: swap_step(k, match=False), i))
        t_load.append(one(load_only, i))
        t_store.append(one(store_only, i))
    ms_swap, ms_swap_only = statistics.median(t_turn), statistics.median(t_swap)
    ms_load, ms_store = statistics.median(t_load), statistics.median(t_store)
    img_bytes = img[0].numel() * 2
    moved = 2 * img_bytes
    value = moved / (ms_swap / 1e3) / 1e9
    # pack kernel (HBM): reads and writes every kept K and V row and position
    qk.kvc_profile_begin()
    ms_pack = timed(lambda i: pack(), max(5, args.steps))
    prof_pack = qk.kvc_profile_end()
    pack_bytes = 2 * (img_bytes + R * 4)
    pk = prof_pack["episode_pack"]
    pack_gbs = pack_bytes / (pk[1] / pk[0] / 1e3) / 1e9
    # match: one question per turn (latency) and a batch of 4096 questions
    for _ in range(5):
        qk.kvc_episode_match(q_d[:1], c_d, ep[:1])
    ms_m1 = timed(lambda i: qk.kvc_episode_match(q_d[:1], c_d, ep[:1]), 200)
    ms_mb = timed(lambda i: qk.kvc_episode_match(q_d, c_d, ep), 50)
    # end to end of one turn through the public API: the question embedding in
    # from pinned host memory, match, episode id back to the host, then the swap
    hq = torch.from_numpy(Qb[:1].copy()).pin_memory()
    hep = torch.empty(1, dtype=torch.int32).pin_memory()

    def turn(i):
        q_d[:1].copy_(hq, non_blocking=True)
        qk.kvc_episode_match(q_d[:1], c_d, ep[:1])
        hep.copy_(ep[:1], non_blocking=True)
        swap_step(i)

    ms_turn = timed(turn, max(3, args.steps // 2))
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, _, desc = episode_oracle_turn(cfg, De, 1, 3)
        cpu = {"value": v, "unit": "GB/s", "cores": cores(), "kind": "oracle", "sample": desc}
    hbm = load_peaks()[0].get("hbm_gbs")
    ach = value
    link_peak = img_bytes / (ms_load / 1e3) / 1e9 + img_bytes / (ms_store / 1e3) / 1e9
    print(json.dumps({
        "metric": EPISODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_swap, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "epicache-llama3.2-3b-M8k-swap", "L": L, "Hkv": H, "mean_budget": cfg.mean_budget,
                   "alpha": cfg.alpha, "episode_image_bytes": img_bytes, "episodes_in_host_memory": E,
                   "l2": "each copy moves 0.94 GB (above L2)"},
        "roofline": {"kernel": "episode swap (copy engines, both directions)", "bound": "host-link",
                     "achieved": ach, "peak": link_peak, "unit": "GB/s", "frac": ach / link_peak,
                     "traffic": None,
                     "peak_source": "sum of the one-direction copy rates measured in this run (load alone + "
                                    "write-back alone); no measured peak file entry covers the host link"},
        "turn_ms": ms_swap, "swap_only_ms": ms_swap_only, "load_only_ms": ms_load, "store_only_ms": ms_store,
        "load_gbs": img_bytes / (ms_load / 1e3) / 1e9, "store_gbs": img_bytes / (ms_store / 1e3) / 1e9,
        "pack": {"ms": pk[1] / pk[0], "GB/s": pack_gbs, "frac_of_hbm": pack_gbs / hbm},
        "match": {"E": E, "De": De, "one_question_us": ms_m1 * 1e3, "batch4096_us": ms_mb * 1e3,
                  "questions_per_s": 4096 / (ms_mb / 1e3)},
        "pages_context": {"match_s": 0.04, "swap_s": 0.3, "note": "the page's per-turn figures, other hardware"},
        "kernels": {n: {"launches": v[0], "avg_ms": v[1] / v[0]} for n, v in {**prof, **prof_pack}.items()},
        "gpu_launches": sum(v[0] for v in prof.values()), "clocks": clocks,
        "e2e": {"value": moved / (ms_turn / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": img_bytes + De * 4,
                "d2h_bytes_per_step": img_bytes + 4, "ms_per_step": ms_turn,
                "how": "one turn: question embedding in from pinned memory, match, episode id back, then the "
                       "duplex swap of the episode images"},
        "cpu_baseline": cpu}), flush=True)


# ---------------------------------------------------------------- Q4 codec leg
Q4_METRIC = "Q4 codec of a compacted KV cache: bf16 bytes encoded or restored per second"


def q4_oracle_sample(cfg, warmup, steps):
    """The float64 oracle's Q4 encode + decode of one segment (at most 65536
    rows) of the workload: GB/s of bf16 rows (read and written), seconds per
    repetition (median) and a description of the sample."""
    from oracle import q4
    x = ks.gen_decode(cfg, "cpu", lens=[min(cfg.kept, 65536)])
    X = x["K"].float().numpy()
    samples = []
    for i in range(warmup + steps):
        a = time.perf_counter()
        c, sc, lo = q4.encode(X)
        q4.decode(c, sc, lo)
        if i >= warmup:
            samples.append(time.perf_counter() - a)
    t = statistics.median(samples)
    return 2 * X.shape[0] * 256 / t / 1e9, t, f"encode + decode of {X.shape[0]} rows"


# DRAM bytes per launch of the Q4 decode kernel as ncu counted them on the
# 16-sequence Llama-3.1-8B 128K/10% workload (dram__bytes_read + write =
# 241.6 + 799.3 MB); the traffic grows with the rows.  Reset to None when the
# kernel changes until it is captured again.
Q4_DECODE_TRAFFIC_PER_SEQ = (241.6e6 + 799.3e6) / 16


def run_q4(args, rank, world, local_rank):
    import torch
    import query_agnostic_kv_gb300 as qk
    from query_agnostic_kv_gb300 import _build

    cfg = ks.DECODE_CONFIGS[args.decode_config]
    if args.impl == "reference":
        if rank != 0:
            return
        v, t, desc = q4_oracle_sample(cfg, args.warmup, args.steps)
        print(json.dumps({
            "impl": "reference", "metric": Q4_METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u4", "data": "synthetic",
            "config": {"workload": cfg.name + "-q4"},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores(), "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)
        return

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    _build.build_library()
    qk.kvc_device_check()
    x = ks.gen_decode(cfg, dev)
    X = torch.cat([x["K"], x["V"]])                      # every kept K and V row of one layer of the batch
    rows = X.shape[0]
    codes = torch.empty(rows, 64, dtype=torch.uint8, device=dev)
    params = torch.empty(rows, 2, 2, dtype=torch.bfloat16, device=dev)
    Y = torch.empty_like(X)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        qk.kvc_q4_encode(X, codes, params)
        qk.kvc_q4_decode(codes, params, Y)
    hc, hp = codes.cpu().pin_memory(), params.cpu().pin_memory()
    assert qk.kvc_stream_status() == 0
    bf16_bytes = rows * 256
    q4_bytes = rows * 72

    def timed(fn, n):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    qk.kvc_profile_begin()
    ms_enc = timed(lambda: qk.kvc_q4_encode(X, codes, params), args.steps)
    ms_dec = timed(lambda: qk.kvc_q4_decode(codes, params, Y), args.steps)
    prof = qk.kvc_profile_end()
    clocks = sampler.stop()
    # restore from page-locked host memory: the kernel reads the Q4 image in place
    # across the host link (the sampler is off: its queries stall host-link traffic)
    ms_rest = timed(lambda: qk.kvc_q4_decode(hc, hp, Y), max(3, args.steps // 4))
    hX = torch.empty(X.shape, dtype=torch.bfloat16).pin_memory()
    ms_h2d = timed(lambda: Y.copy_(hX, non_blocking=True), max(3, args.steps // 4))
    assert qk.kvc_stream_status() == 0
    hbm = load_peaks()[0].get("hbm_gbs")
    enc_l, enc_t = prof["q4_encode"]
    dec_l, dec_t = prof["q4_decode"]
    traffic = bf16_bytes + q4_bytes                      # one read and one write per row, either direction
    ach_enc = traffic / (enc_t / enc_l / 1e3) / 1e9
    ach_dec = traffic / (dec_t / dec_l / 1e3) / 1e9
    value = 2 * bf16_bytes / ((ms_enc + ms_dec) / 1e3) / 1e9
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, _, desc = q4_oracle_sample(cfg, 1, 3)
        cpu = {"value": v, "unit": "GB/s", "cores": cores(), "kind": "oracle", "sample": desc}
    print(json.dumps({
        "metric": Q4_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_enc + ms_dec, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u4", "data": "synthetic",
        "config": {"workload": cfg.name + "-q4", "rows": rows, "bf16_bytes": bf16_bytes, "q4_bytes": q4_bytes,
                   "l2": "inputs larger than L2; no flush between steps", "step": "one encode + one decode"},
        "roofline": {"kernel": "q4_decode", "bound": "hbm", "achieved": ach_dec, "peak": hbm, "unit": "GB/s",
                     "frac": ach_dec / hbm,
                     "traffic": None if Q4_DECODE_TRAFFIC_PER_SEQ is None else Q4_DECODE_TRAFFIC_PER_SEQ * cfg.seqs,
                     "traffic_source": "ncu dram bytes of the 16-sequence case, scaled by sequences",
                     "peak_source": "hbm_gbs of measured peaks", "algorithmic_bytes_per_launch": traffic},
        "encode": {"ms": enc_t / enc_l, "GB/s": ach_enc, "frac_of_hbm": ach_enc / hbm},
        "decode": {"ms": dec_t / dec_l, "GB/s": ach_dec, "frac_of_hbm": ach_dec / hbm},
        "restore_from_host": {"ms": ms_rest, "bf16_GB/s": bf16_bytes / (ms_rest / 1e3) / 1e9,
                              "link_GB/s": q4_bytes / (ms_rest / 1e3) / 1e9,
                              "bf16_h2d_copy_ms": ms_h2d,
                              "speedup_vs_bf16_copy": ms_h2d / ms_rest},
        "kernels": {n: {"launches": v[0], "avg_ms": v[1] / v[0]} for n, v in prof.items()},
        "gpu_launches": enc_l + dec_l, "clocks": clocks,
        "e2e": {"value": bf16_bytes / (ms_rest / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": q4_bytes,
                "d2h_bytes_per_step": 0, "ms_per_step": ms_rest,
                "how": "restore: the Q4 image in page-locked host memory decoded in place into device bf16 rows"},
        "cpu_baseline": cpu}), flush=True)


# ---------------------------------------------------------------- EpiCache block prefill leg
EPI_METRIC = "EpiCache block prefill: history tokens/s over all episodes (E * N_hist / T)"


def epi_oracle_sample(cfg):
    """The float64 oracle's block prefill on one KV head of layer 0 over the
    first 8 blocks, scaled to all layers, heads and history tokens: seconds
    per episode and a description of the sample."""
    from oracle import kv2
    B, S = cfg.block, cfg.sinks
    budgets = kv2.layer_budgets(ks.gen_sensitivity(cfg).astype(np.float64), cfg.alpha, cfg.mean_budget, S)
    Kh, Vh = ks.gen_epi_history_layer(cfg, 0)
    Qp, Kp = ks.gen_epi_prompt_layer(cfg, 0, 0)
    n = min(cfg.n_hist, 8 * B)
    a = time.perf_counter()
    kv2.block_prefill_layer(kv2.bf16_to_f64(Kh[:1, :n]), kv2.bf16_to_f64(Vh[:1, :n]),
                            kv2.bf16_to_f64(Qp[:cfg.G]), kv2.bf16_to_f64(Kp[:1]), B, int(budgets[0]), S)
    t = (time.perf_counter() - a) * (cfg.n_hist / n) * cfg.L * cfg.Hkv
    return t, (f"layer 0, KV head 0, first {n} history tokens, scaled to {cfg.L} layers x {cfg.Hkv} heads x "
               f"{cfg.n_hist} tokens")


def epi_evict_compact_bytes(cfg, budgets):
    """Algorithmic bytes of the block step's eviction + compaction launches
    over one episode: an over-budget layer reads the n scores of each KV head,
    writes its k_l kept indices, and moves the k_l kept K and V rows (read +
    write) with their int32 positions."""
    B, S = cfg.block, cfg.sinks
    nb = (cfg.n_hist + B - 1) // B
    length = [0] * cfg.L
    total = 0
    for b in range(nb):
        blk = min(B, cfg.n_hist - b * B)
        for l in range(cfg.L):
            n = length[l] + blk
            if n > budgets[l] and n > S:
                total += cfg.Hkv * (n * 4 + budgets[l] * 4 + budgets[l] * (2 * 2 * 128 * 2 + 2 * 4))
                length[l] = budgets[l]
            else:
                length[l] = n
    return total


def epi_in_place_bytes(qk, cfg, budgets, new_state, blocks, prompt, ws, stream, pos0, cap):
    """Algorithmic bytes of the one-slab eviction launches over one episode,
    replayed untimed: an over-budget layer reads the n scores of each KV head
    and moves each kept block row that was appended at or above its budget
    into an evicted row (K and V rows read and written, positions read and
    written).  Such a row has position >= t0 + M_l - len_l."""
    import torch
    B, S, L, H = cfg.block, cfg.sinks, cfg.L, cfg.Hkv
    st = new_state()
    dq, dk = prompt
    total = 0
    t0 = 0
    for kb, vb, n in blocks:
        old = [st.len[l] for l in range(L)]
        qk.kvc_block_prefill_step(st, kb, vb, n, dq, dk, cfg.prompt_len, ws=ws, stream=stream)
        P = pos0.view(L, H, cap)
        for l in range(L):
            if old[l] + n > budgets[l] and old[l] + n > S:
                first = t0 + max(budgets[l] - old[l], 0)
                p = P[l, :, :budgets[l]]
                moved = int(((p >= first) & (p < t0 + n)).sum())
                total += H * (old[l] + n) * 4 + moved * (2 * 2 * 128 * 2 + 2 * 4)
        t0 += n
    torch.cuda.synchronize()
    return total


# DRAM bytes (read + write) per launch of the EpiCache block step's in-place
# eviction (one-slab state), from a one-pass ncu capture of one episode's 44
# launches: 52.21 + 8.71 MB on average.  Reset to None whenever the kernel
# changes until it is captured again.
EPI_EVICT_TRAFFIC_PER_LAUNCH = (52.21e6 + 8.71e6)


def run_epicache(args, rank, world, local_rank):
    import torch
    import query_agnostic_kv_gb300 as qk
    from query_agnostic_kv_gb300 import _build

    cfg = ks.EPI_3B
    L, H, Hq, B, P, S = cfg.L, cfg.Hkv, cfg.Hq, cfg.block, cfg.prompt_len, cfg.sinks
    if args.impl == "reference":
        if rank != 0:
            return
        t, sample = epi_oracle_sample(cfg)
        v = cfg.episodes * cfg.n_hist / (t * cfg.episodes)
        print(json.dumps({
            "impl": "reference", "metric": EPI_METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": 1, "warmup": 0, "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": {"workload": cfg.name},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores(), "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)
        return

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    _build.build_library()
    qk.kvc_device_check()
    budgets = qk.kvc_layer_budgets(ks.gen_sensitivity(cfg).tolist(), cfg.alpha, cfg.mean_budget, S)
    nb = (cfg.n_hist + B - 1) // B
    # history, block-major on the device: blocks[b] = [L][H][B][d] (last block ragged)
    Kblk = torch.zeros(nb, L, H, B, 128, dtype=torch.bfloat16, device=dev)
    Vblk = torch.zeros_like(Kblk)
    for l in range(L):
        kh, vh = ks.gen_epi_history_layer(cfg, l)
        for src, dst in ((kh, Kblk), (vh, Vblk)):
            t = torch.from_numpy(src.view(np.int16)).view(torch.bfloat16)        # [H][n_hist][d]
            pad = torch.zeros(H, nb * B - cfg.n_hist, 128, dtype=torch.bfloat16)
            t = torch.cat([t, pad], dim=1).view(H, nb, B, 128).permute(1, 0, 2, 3)
            dst[:, l] = t.to(dev)
    prompts = []
    for e in range(cfg.episodes):
        prm = [ks.gen_epi_prompt_layer(cfg, e, l) for l in range(L)]
        dq = torch.from_numpy(np.stack([p[0] for p in prm]).view(np.int16)).view(torch.bfloat16).to(dev)
        dk = torch.from_numpy(np.stack([p[1] for p in prm]).view(np.int16)).view(torch.bfloat16).to(dev)
        prompts.append((dq, dk))
    cap = max(budgets) + B
    torch.cuda.synchronize()
    mem0 = torch.cuda.memory_allocated(dev)
    n_slab = 2 if args.epi_layout == "two-slab" else 1
    slabs = [torch.zeros(L * H * cap * 128, dtype=torch.bfloat16, device=dev) for _ in range(2 * n_slab)]
    pos = [torch.zeros(L * H * cap, dtype=torch.int32, device=dev) for _ in range(n_slab)]

    def new_state():
        if n_slab == 2:
            return qk.kvc_block_state_init(L, H, Hq, cap, S, budgets, slabs[0], slabs[1], pos[0], slabs[2],
                                           slabs[3], pos[1])
        return qk.kvc_block_state_init(L, H, Hq, cap, S, budgets, slabs[0], slabs[1], pos[0])

    stream = torch.cuda.current_stream()
    blocks = [(Kblk[b] if b < nb - 1 or cfg.n_hist % B == 0 else Kblk[b, :, :, :cfg.n_hist - b * B].contiguous(),
               Vblk[b] if b < nb - 1 or cfg.n_hist % B == 0 else Vblk[b, :, :, :cfg.n_hist - b * B].contiguous(),
               min(B, cfg.n_hist - b * B)) for b in range(nb)]

    last_state = []

    def episode(e, ws=None):
        st = new_state()
        if ws is None:
            ws = torch.empty(qk.kvc_block_workspace_size(st, B, P), dtype=torch.uint8, device=dev)
        dq, dk = prompts[e]
        for kb, vb, n in blocks:
            qk.kvc_block_prefill_step(st, kb, vb, n, dq, dk, P, ws=ws, stream=stream)
        last_state[:] = [st]
        return ws

    n_warm = max(3, args.warmup)
    ws = episode(0)
    torch.cuda.synchronize()
    memory = {
        "layout": args.epi_layout,
        "block_state_and_workspace_bytes": torch.cuda.memory_allocated(dev) - mem0,
        "workspace_bytes": ws.numel(),
        "full_kv_cache_of_history_bytes": 2 * L * H * cfg.n_hist * 128 * 2,
        "how": "device bytes allocated for the K/V slabs, the position arrays and the step workspace (torch "
               "allocator, measured), against the K and V of the whole history (computed from its shape); the "
               "model weights and the history blocks themselves are not counted",
    }
    for w in range(1, n_warm):
        episode(w % cfg.episodes, ws)
    torch.cuda.synchronize()
    assert qk.kvc_stream_status() == 0
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    qk.kvc_profile_begin()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for e in range(cfg.episodes):
        episode(e, ws)
    b.record(stream)
    torch.cuda.synchronize()
    prof = qk.kvc_profile_end()
    clocks = sampler.stop()
    assert qk.kvc_stream_status() == 0
    ms = a.elapsed_time(b)
    value = world * cfg.episodes * cfg.n_hist / (ms / 1e3)
    total = sum(v[1] for v in prof.values())
    kernels = {n: {"launches": v[0], "avg_ms": v[1] / v[0], "share": v[1] / total} for n, v in prof.items()}

    # roofline of eviction + compaction, bound by HBM.  Two slabs: one fused
    # launch when the kept lists are short, else the eviction launch and one
    # tiled compaction launch.  One slab: one launch moving the kept block
    # rows into evicted rows; how many rows moved is counted in an untimed
    # replay of the same episodes.
    peaks, peak_src = load_peaks()
    hbm = peaks.get("hbm_gbs")
    if n_slab == 2:
        cbytes = epi_evict_compact_bytes(cfg, budgets) * cfg.episodes
        parts = [n for n in ("evict_compact", "evict_topk", "compact") if n in prof]
        what = "top-M_l per KV head, kept rows into the other slab"
    else:
        cbytes = sum(epi_in_place_bytes(qk, cfg, budgets, new_state, blocks, prompts[e], ws, stream, pos[0], cap)
                     for e in range(cfg.episodes))
        parts = ["evict_in_place"]
        what = "top-M_l per KV head, kept block rows into evicted rows"
    ctime = sum(prof[n][1] for n in parts) / 1e3
    steps_scored = sum(prof[n][0] for n in ("evict_compact", "evict_topk", "evict_in_place") if n in prof)
    ach = cbytes / ctime / 1e9
    roof = {"kernel": " + ".join(parts) + f" ({what})", "bound": "hbm",
            "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
            "traffic": EPI_EVICT_TRAFFIC_PER_LAUNCH if n_slab == 1 else None,
            "traffic_source": "ncu dram bytes per launch, mean over one episode (one-slab layout; null for the "
                              "two-slab kernels, not captured)",
            "peak_source": f"hbm_gbs of {peak_src} peaks",
            "algorithmic_bytes_per_step": cbytes / steps_scored}

    # the episode's packed image (kvc_episode_pack): one contiguous copy of the
    # kept rows in ascending position order per (layer, KV head); for the
    # one-slab state this is where the position order is restored
    st_last = last_state[0]
    R = qk.kvc_episode_rows(st_last)
    Kp = torch.empty(R * 128, dtype=torch.bfloat16, device=dev)
    Vp = torch.empty_like(Kp)
    Pp = torch.empty(R, dtype=torch.int32, device=dev)
    for _ in range(3):
        qk.kvc_episode_pack(st_last, Kp, Vp, Pp, stream=stream)
    torch.cuda.synchronize()
    pa = torch.cuda.Event(enable_timing=True)
    pb = torch.cuda.Event(enable_timing=True)
    pa.record(stream)
    for _ in range(20):
        qk.kvc_episode_pack(st_last, Kp, Vp, Pp, stream=stream)
    pb.record(stream)
    torch.cuda.synchronize()
    assert qk.kvc_stream_status() == 0
    pack_ms = pa.elapsed_time(pb) / 20
    pack_bytes = R * (2 * 2 * 128 * 2 + 2 * 4)      # K and V rows read and written, positions
    pack = {"ms": pack_ms, "rows": R, "GB/s": pack_bytes / (pack_ms / 1e3) / 1e9,
            "frac_of_hbm": pack_bytes / (pack_ms / 1e3) / 1e9 / hbm if hbm else None,
            "ordered": n_slab == 1,
            "how": "kvc_episode_pack of the last timed episode's state, 20 back-to-back calls (CUDA events); algorithmic "
                   "bytes = every kept K and V row read and written plus its position"}

    # end to end: the history streamed from pinned host memory; block b is
    # copied on a copy stream into one of two device buffers while the step
    # of block b - 1 runs
    e2e = None
    if args.e2e_steps > 0:
        hblocks = [(kb.cpu().pin_memory(), vb.cpu().pin_memory(), n) for kb, vb, n in blocks]
        dK = [torch.empty(L * H * B * 128, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        dV = [torch.empty_like(dK[0]) for _ in range(2)]
        cps = torch.cuda.Stream(device=dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        free = [torch.cuda.Event() for _ in range(2)]
        for ev in copied + free:
            ev.record(stream)
        torch.cuda.synchronize()

        def episode_host(e, start=None):
            st = new_state()
            dq, dk = prompts[e]
            for i, (hk, hv, n) in enumerate(hblocks):
                j = i % 2
                kb = dK[j][:L * H * n * 128].view(L, H, n, 128)
                vb = dV[j][:L * H * n * 128].view(L, H, n, 128)
                with torch.cuda.stream(cps):
                    if start is not None and i == 0:
                        cps.wait_event(start)
                    cps.wait_event(free[j])
                    kb.copy_(hk, non_blocking=True)
                    vb.copy_(hv, non_blocking=True)
                    copied[j].record(cps)
                stream.wait_event(copied[j])
                qk.kvc_block_prefill_step(st, kb, vb, n, dq, dk, P, ws=ws, stream=stream)
                free[j].record(stream)

        for w in range(n_warm):
            episode_host(w % cfg.episodes)
        torch.cuda.synchronize()
        a2 = torch.cuda.Event(enable_timing=True)
        b2 = torch.cuda.Event(enable_timing=True)
        a2.record(stream)
        for e in range(cfg.episodes):
            episode_host(e, start=a2 if e == 0 else None)
        b2.record(stream)
        torch.cuda.synchronize()
        assert qk.kvc_stream_status() == 0
        e_ms = a2.elapsed_time(b2)
        h2d = sum(hk.numel() + hv.numel() for hk, hv, _ in hblocks) * 2
        e2e = {"value": world * cfg.episodes * cfg.n_hist / (e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 0, "ms_per_step": e_ms / cfg.episodes,
               "how": "history K/V blocks in pinned host memory, each copied on a copy stream into one of two device "
                      "buffers while the previous block's step runs; the compressed cache stays on the device"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t, sample = epi_oracle_sample(cfg)
        cpu = {"value": cfg.n_hist / t, "unit": "tokens/s", "cores": cores(), "kind": "oracle", "sample": sample}
    print(json.dumps({
        "metric": EPI_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": cfg.episodes,
        "warmup": n_warm, "ms_per_step": ms / cfg.episodes, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "layout": args.epi_layout, "L": L, "Hkv": H, "Hq": Hq,
                   "n_hist": cfg.n_hist, "block": B, "episodes": cfg.episodes, "prompt_queries": P, "mean_budget": cfg.mean_budget, "alpha": cfg.alpha,
                   "step": "one episode (all history blocks)", "l2": "history 10 GB on the device"},
        "roofline": roof, "kernels": kernels, "gpu_launches": sum(v[0] for v in prof.values()), "clocks": clocks,
        "memory": memory, "pack": pack, "e2e": e2e, "cpu_baseline": cpu}), flush=True)


# ---------------------------------------------------------------- reconstruction-ratio sweep
RHO_METRIC = "compression step time and workspace vs reconstruction ratio rho (Llama-8B shape, 16K)"
RHO_SWEEP = (0.05, 0.1, 0.25, 0.5)


def run_rho_sweep(args, rank, world, local_rank):
    """KV² page, "무엇과 다른가": the method's runtime and peak activation
    memory grow with the reconstruction ratio rho.  The 16K workload is
    compressed at each rho of RHO_SWEEP (same cache, budget and sinks)."""
    base = ks.LLAMA_16K
    if args.impl == "reference":
        if rank != 0:
            return
        pts = []
        for rho in RHO_SWEEP:
            cfg = ks.scaled(base, rho=rho)
            t, desc = time_oracle_sample(cfg, budget_s=2.0)
            pts.append({"rho": rho, "ms_per_step": t * 1e3, "sample": desc})
        v = base.N / (pts[1]["ms_per_step"] / 1e3)
        print(json.dumps({"impl": "reference", "metric": RHO_METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
                          "steps": 1, "warmup": 0, "ms_per_step": pts[1]["ms_per_step"], "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                          "config": {"workload": base.name + "-rho-sweep"}, "sweep": pts, "extrapolated": True,
                          "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores(), "kind": "oracle",
                                           "sample": "per rho: " + pts[1]["sample"]},
                          "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return
    import torch
    import query_agnostic_kv_gb300 as qk
    from query_agnostic_kv_gb300 import _build

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    _build.build_library()
    qk.kvc_device_check()
    x = ks.gen_kv2(base)
    L, H, Hq, N, S, d = base.L, base.Hkv, base.Hq, base.N, base.sinks, base.d

    def dev_bf16(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)

    K, V, Q = dev_bf16(x.K), dev_bf16(x.V), dev_bf16(x.Q)
    shape = (L, H, Hq, d, N)
    k = qk.kvc_budget_count(base.budget, N, S)
    kept = torch.empty(L * H * k, dtype=torch.int32, device=dev)
    Kc = torch.empty(L * H * k * d, dtype=torch.bfloat16, device=dev)
    Vc = torch.empty_like(Kc)
    stream = torch.cuda.current_stream()
    peaks, peak_src = load_peaks()
    pts = []
    steps = max(1, min(args.steps, 50))
    for rho in RHO_SWEEP:
        cfg = ks.scaled(base, rho=rho)
        work = algorithmic_work(cfg)
        ws = torch.empty(qk.kvc_workspace_size(shape, S, cfg.m, rho), dtype=torch.uint8, device=dev)

        def step():
            qk.kvc_compress_ex(shape, "keydiff", K, V, Q, S, cfg.m, rho, 1, [k] * L, kept, Kc, Vc, ws=ws,
                               stream=stream)

        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize()
        assert qk.kvc_stream_status(stream) == 0
        qk.kvc_profile_begin()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        prof = qk.kvc_profile_end()
        ms = a.elapsed_time(b) / steps
        lse = prof["recon_lse"][1] / prof["recon_lse"][0]
        col = prof["recon_colmax"][1] / prof["recon_colmax"][0]
        f_step = work["flops_lse"] + work["flops_colmax"]
        pts.append({"rho": rho, "ms_per_step": ms, "tokens_per_s": N / (ms / 1e3),
                    "recon_lse_ms": lse, "recon_colmax_ms": col, "reconstruction_queries": work["Q"],
                    "scoring_flops": f_step, "scoring_tflops": f_step / ((lse + col) / 1e3) / 1e12,
                    "lse_frac_of_burst": work["flops_lse_per_launch"] / (lse / 1e3) / 1e12 / peaks["bf16_tflops"],
                    "workspace_bytes": ws.numel()})
        del ws
        torch.cuda.empty_cache()
    if rank == 0:
        mid = pts[1]
        print(json.dumps({
            "metric": RHO_METRIC, "value": mid["tokens_per_s"], "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": max(3, args.warmup), "ms_per_step": mid["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": base.name + "-rho-sweep", "rho": list(RHO_SWEEP), "budget": base.budget,
                       "m": base.m, "value_at_rho": 0.1}, "sweep": pts,
            "peak_source": f"bf16_tflops of {peak_src} peaks"}), flush=True)


def main():
    args = parse()
    cfg = ks.KV2_CONFIGS[args.config]
    if args.layers:
        cfg = ks.scaled(cfg, name=f"{cfg.name}-{args.layers}layers", L=args.layers)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.op == "decode" and args.impl == "reference":
        run_decode(args, rank, world, local_rank)
        return
    if args.op == "episode":
        run_episode(args, rank, world, local_rank)
        return
    if args.op == "q4":
        run_q4(args, rank, world, local_rank)
        return
    if args.op == "epicache":
        run_epicache(args, rank, world, local_rank)
        return
    if args.op == "rho":
        run_rho_sweep(args, rank, world, local_rank)
        return
    if args.impl == "reference":
        run_reference(args, cfg, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        if args.op == "decode":
            run_decode(args, rank, world, local_rank)
        else:
            run_ours(args, cfg, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
