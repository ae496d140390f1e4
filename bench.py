#!/usr/bin/env python
"""Benchmark of the DSA indexer decode step on GB300.

A step is one pass of the whole hot path over one batch of synthetic input
(DecodePlan): paged MQA logits with the fused coarse histogram, the
histogram-driven exact top-2048, block amax8, block top-512, the sorted block
table, sparse logits over the chosen blocks (FP16) and the FP16 top-2048.

Default workload: B=32 requests, next_n=1, L=131072 keys each, page size 64,
'mixed' score distribution (heads 16..31 weighted x20) -- the configuration
the >= 70 % HBM target of the logits kernel is stated on.  Inputs are resident
in HBM and larger than L2: each step streams the whole K cache (554 MB at
this size) through the 129 MB L2 with an evict-first policy, so no step finds
the previous step's K lines; L2 is not flushed between steps.  The timed
loop replays the step's CUDA graph (DecodePlan.capture / replay), every 16th
step run eagerly with events around the dense logits launch for the roofline.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the plain CPU
oracle on the host cores instead (the reference arm of this comparison).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "indexer decode keys scored/s and HBM GB/s (% of peak); top-2048 rows/s"
KEY_BYTES = 132  # 128 FP8 bytes of K + 4 bytes of kscale per key
NOMINAL_GBS = 8000.0  # the ~8 TB/s nominal HBM3e figure the target is stated against
PER_WORKLOADS = ("c0", "c1", "c3", "c3u", "c4")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="c2")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-budget", type=float, default=12.0)
    p.add_argument("--no-per-workload", action="store_true",
                   help="skip the per-workload table (c0, c1, c3, c3u, c4)")
    p.add_argument("--no-mx", action="store_true", help="skip the MXFP4-key logits timing")
    p.add_argument("--mx-only", action="store_true",
                   help="only the MXFP4-key logits launch (warm-up + steps), one JSON object")
    return p.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    lrank = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, lrank


def max_over_ranks(x: float, dist, device) -> float:
    """The slowest rank's time (weak scaling: every rank runs one replica)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step: int, world: int, steps: int, t_max: float) -> float:
    """Units all ranks processed / the slowest rank's time."""
    return world * units_per_rank_step * steps / t_max


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def traffic_record(kernel_src):
    """Per-launch DRAM bytes of the logits kernel from the committed ncu record
    (profiles/logits_fused_hist_c2.json), valid only while the kernel source
    (the kernel file and the device header it includes) is unchanged: the
    sha256 of the two, in that order, is stored beside the number; None
    otherwise."""
    path = os.path.join(ROOT, "profiles", "logits_fused_hist_c2.json")
    try:
        h = hashlib.sha256()
        for src in (kernel_src, os.path.join(os.path.dirname(kernel_src), "dsa_device.cuh")):
            h.update(open(src, "rb").read())
        sha = h.hexdigest()
        with open(path) as f:
            rec = json.load(f)
        if rec.get("source_sha256") == sha:
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class Clocks:
    Q = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            if self.uuid and self.uuid not in f[0]:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_step_sample(case, nn, ps, b, k=2048, kb=512, max_keys=None):
    """The oracle's whole step for request b (all its rows), optionally on the
    first ``max_keys`` keys of the request only: returns keys scored."""
    from oracle import oracle as O
    r0, r1 = b * nn, (b + 1) * nn
    ctx = case["context_lens"][b:b + 1].copy()
    if max_keys is not None:
        ctx = np.minimum(ctx, np.int32(max_keys))
    pt = case["page_table"][b:b + 1]
    q = case["q"][r0:r1]
    w = case["weights"][r0:r1]
    L = O.paged_mqa_logits(q, case["kv"], case["kscale"], w, pt, ctx, nn, ps)
    rl = O.row_lens(ctx, nn)
    O.histogram(L, rl)
    O.topk(L, rl, k)
    A = O.block_amax8(L, rl, skip_le=kb)
    t, _, vl = O.block_table(A, rl, np.zeros(nn, np.int32), kb, pt, ps)
    sp = O.sparse_logits(q, case["kv"], case["kscale"], w, pt, rl, np.zeros(nn, np.int32), ps, t)
    O.topk_fp16(O.fp16_rn_array(sp), vl, k, t)
    return int(rl.sum())


def run_reference(args, ws_, rank):
    import synthetic as S
    if rank != 0:
        return
    w = S.named(args.workload)
    case = S.generate(w)
    # size each step's sample so the whole run stays near two minutes
    t0 = time.perf_counter()
    full = oracle_step_sample(case, w.next_n, w.page_size, 0)
    t_full = time.perf_counter() - t0
    budget = 120.0 / max(1, args.steps + args.warmup)
    max_keys = None
    if t_full > budget:
        max_keys = max(4096, int(max(w.context_lens) * budget / t_full))
    for i in range(args.warmup):
        oracle_step_sample(case, w.next_n, w.page_size, i % w.B, max_keys=max_keys)
    t0 = time.perf_counter()
    keys = 0
    for i in range(args.steps):
        keys += oracle_step_sample(case, w.next_n, w.page_size, i % w.B, max_keys=max_keys)
    dt = time.perf_counter() - t0
    sample = ("one request (all its rows) per step" if max_keys is None else
              f"the first {max_keys} keys of one request per step (full request: "
              f"{full} keys in {t_full:.2f} s)")
    v = keys / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "keys/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample": sample},
            "cpu_baseline": {"value": v, "unit": "keys/s", "cores": 1, "kind": "oracle",
                             "sample": "each step: " + sample + " through the whole oracle "
                                       "step (logits, histogram, top-2048, amax8, block "
                                       "table, sparse logits, FP16 top-2048)"},
            "e2e": {"value": v, "unit": "keys/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure_workload(name, dev, steps=200, warmup=5):
    """Per-workload timings of the same step (outside the headline's timed
    region): the logits launch alone (a CUDA graph of back-to-back launches),
    the eager step (events around the whole step only) and the CUDA-graph
    replay of the step."""
    import torch
    import synthetic as S
    from dsa_sparse_attention_paged_gb300.pipeline import DecodePlan
    w = S.named(name)
    case = S.generate(w)
    nn = w.next_n
    d = {k: (torch.from_numpy(v).to(dev) if isinstance(v, np.ndarray) else v)
         for k, v in case.items()}
    plan = DecodePlan(w.B, nn, max(w.context_lens), w.page_size, k=2048, kb=512,
                      two_level=True, device=dev)
    inputs = (d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"], d["context_lens"])
    ctx = np.asarray(w.context_lens, dtype=np.int64)
    keys = int((ctx[:, None] - (nn - 1 - np.arange(nn))[None, :]).sum())
    kv_bytes = int(ctx.sum()) * KEY_BYTES

    def ev():
        return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    for _ in range(warmup):
        plan.step(*inputs)
    torch.cuda.synchronize()
    steps_ev = [ev() for _ in range(steps)]
    for a, b in steps_ev:
        a.record()
        plan.step(*inputs)
        b.record()
    torch.cuda.synchronize()
    step_us = 1e3 * statistics.median(a.elapsed_time(b) for a, b in steps_ev)
    # the logits launch alone, from a CUDA graph of back-to-back launches (an
    # eager launch of a few-microsecond kernel would time the host's launch)
    import dsa_sparse_attention_paged_gb300 as D
    hist = torch.zeros((w.R, 1024), dtype=torch.int32, device=dev)
    reps = 20

    def logits_only():
        D.paged_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                           d["context_lens"], nn, plan.ws, logits=plan.logits, histogram=hist)

    logits_only()
    torch.cuda.synchronize()
    gl = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gl):
        for _ in range(reps):
            logits_only()
    gl.replay()
    torch.cuda.synchronize()
    lg = []
    for _ in range(10):
        a, b = ev()
        a.record()
        gl.replay()
        b.record()
        torch.cuda.synchronize()
        lg.append(a.elapsed_time(b) / reps)
    lg_us = 1e3 * statistics.median(lg)
    plan.capture(*inputs)
    plan.replay()
    torch.cuda.synchronize()
    gs, ge = ev()
    gs.record()
    for _ in range(steps):
        plan.replay()
    ge.record()
    torch.cuda.synchronize()
    graph_us = 1e3 * gs.elapsed_time(ge) / steps
    if plan.ws.status() != 0:
        raise RuntimeError(f"{name}: device status {plan.ws.status():#x}")
    peak, kind = peaks()
    gbs = kv_bytes / (lg_us * 1e-6) / 1e9
    out = {"workload": w.name, "keys_per_step": keys, "kstream_bytes": kv_bytes,
           "logits_us": lg_us, "kstream_gbs": gbs, "frac_of_measured_peak": gbs / peak,
           "frac_of_8tbs_nominal": gbs / NOMINAL_GBS, "step_us_eager": step_us,
           "step_us_graph": graph_us, "keys_per_s_eager": keys / (step_us * 1e-6),
           "keys_per_s_graph": keys / (graph_us * 1e-6)}
    del plan, d
    torch.cuda.empty_cache()
    return out


MX_KEY_BYTES = 68  # 64 bytes of E2M1 codes + 4 UE8M0 block exponents per key
LOGITS_EVERY = 16  # steps per event-bracketed logits launch in the timed loop


def measure_mx_logits(case, w, d, dev, steps=200, warmup=5):
    """The MXFP4-key logits launch (with the fused histogram) at this
    workload's shape and page pool: seeded E2M1 codes and exponents, timed
    like the per-workload logits: a CUDA graph of 20 launches back to back
    (the 68-byte-a-key stream is larger than L2), CUDA events around its
    replays."""
    import torch
    import dsa_sparse_attention_paged_gb300 as D
    g = torch.Generator().manual_seed(w.seed + 1000)
    P, ps = case["num_pages"], w.page_size
    codes = torch.randint(0, 256, (P, ps, 64), generator=g, dtype=torch.uint8).to(dev)
    exps = torch.randint(125, 130, (P, ps, 4), generator=g, dtype=torch.uint8).to(dev)
    nn = w.next_n
    ctx = np.asarray(w.context_lens, dtype=np.int64)
    stride = (int(ctx.max()) + 7) // 8 * 8
    ws = D.Workspace(w.R, device=dev)
    logits = torch.empty((w.R, stride), dtype=torch.float32, device=dev)
    hist = torch.zeros((w.R, 1024), dtype=torch.int32, device=dev)

    def launch():
        D.paged_mqa_logits_mx(d["q"], codes, exps, d["weights"], d["page_table"],
                              d["context_lens"], nn, ws, logits=logits, histogram=hist)

    for _ in range(warmup):
        launch()
    torch.cuda.synchronize()
    gl = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gl):
        for _ in range(20):
            launch()
    gl.replay()
    torch.cuda.synchronize()
    reps = max(1, min(10, steps // 20))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        gl.replay()
    e1.record()
    torch.cuda.synchronize()
    if ws.status() != 0:
        raise RuntimeError(f"MXFP4 logits: device status {ws.status():#x}")
    us = 1e3 * e0.elapsed_time(e1) / (20 * reps)
    keys = int(ctx.sum())
    kbytes = keys * MX_KEY_BYTES
    peak, kind = peaks()
    gbs = kbytes / (us * 1e-6) / 1e9
    del codes, exps, logits, hist
    torch.cuda.empty_cache()
    return {"kernel": f"logits_kernel<next_n={nn}, MXFP4 keys, histogram>",
            "logits_us": us, "kstream_bytes": kbytes, "key_bytes": MX_KEY_BYTES,
            "kstream_gbs": gbs, "frac_of_measured_peak": gbs / peak,
            "frac_of_8tbs_nominal": gbs / NOMINAL_GBS,
            "keys_per_s": keys * nn / (us * 1e-6)}


def cpu_baseline(case, w, budget):
    t0 = time.perf_counter()
    keys, n = 0, 0
    while time.perf_counter() - t0 < budget and n < w.B:
        keys += oracle_step_sample(case, w.next_n, w.page_size, n)
        n += 1
    dt = time.perf_counter() - t0
    return {"value": keys / dt, "unit": "keys/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} request(s) of the workload ({keys} keys) through the whole "
                      f"oracle step, {dt:.1f} s single-threaded"}


def main():
    args = parse()
    world, rank, lrank = dist_env()
    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    if args.impl == "reference":
        run_reference(args, world, rank)
        if dist is not None:
            dist.destroy_process_group()
        return

    import synthetic as S
    import dsa_sparse_attention_paged_gb300 as D
    from dsa_sparse_attention_paged_gb300.pipeline import DecodePlan, HostStepPipeline

    torch.cuda.set_device(lrank)
    dev = torch.device("cuda", lrank)
    w = S.named(args.workload)
    case = S.generate(w)
    nn, ps = w.next_n, w.page_size
    d = {k: (torch.from_numpy(v).to(dev) if isinstance(v, np.ndarray) else v)
         for k, v in case.items()}
    if args.mx_only:
        print(json.dumps(measure_mx_logits(case, w, d, dev, steps=max(1, args.steps),
                                           warmup=args.warmup)), flush=True)
        return
    plan = DecodePlan(w.B, nn, max(w.context_lens), ps, k=2048, kb=512, two_level=True,
                      device=dev)
    inputs = (d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"], d["context_lens"])

    ctx = np.asarray(w.context_lens, dtype=np.int64)
    rl = ctx[:, None] - (nn - 1 - np.arange(nn))[None, :]
    keys_per_step = int(rl.sum())
    logits_bytes = int(ctx.sum()) * KEY_BYTES + keys_per_step * 4 + w.R * 32 * (128 + 4)
    kv_bytes = int(ctx.sum()) * KEY_BYTES

    for _ in range(args.warmup):
        plan.step(*inputs)
    torch.cuda.synchronize()
    if plan.ws.status() != 0:
        raise RuntimeError(f"device status {plan.ws.status():#x} after warm-up")

    # The timed loop replays the step captured as a CUDA graph
    # (DecodePlan.capture / replay: the same four kernels, no host launch
    # cost between them), except every LOGITS_EVERY-th step, which runs
    # eagerly with the dense logits kernel bracketed by CUDA events (the
    # roofline's launch duration; an event record between two kernels holds
    # back the programmatic launch of the second, so the other steps run
    # without them).  The per-stage split is taken in a separate, untimed loop
    # below.  One pair of events brackets all K steps.
    names = ["logits"]
    K = args.steps
    every = max(1, min(LOGITS_EVERY, K // 4))  # at least four bracketed launches
    ev_k = [{n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for n in names} if i % every == every - 1 else None
            for i in range(K)]
    plan.capture(*inputs)
    plan.replay()
    torch.cuda.synchronize()
    t_rep = time.perf_counter()
    plan.replay()
    torch.cuda.synchronize()
    t_rep = time.perf_counter() - t_rep
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clk = Clocks(uuid)

    t0_ev, t1_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clk.start()
    # about 0.2 s of untimed replays while the clock sampler starts: the GPU
    # enters the timed loop busy rather than after an idle gap
    for _ in range(max(10, min(4000, int(0.2 / max(t_rep, 1e-5))))):
        plan.replay()
    torch.cuda.synchronize()
    t0_ev.record()
    for i in range(K):
        if ev_k[i] is not None:
            plan.step(*inputs, events=ev_k[i])
        else:
            plan.replay()
    t1_ev.record()
    torch.cuda.synchronize()
    clocks = clk.stop()
    if dist is not None:
        dist.barrier()
    kern_ms = {n: [e[n][0].elapsed_time(e[n][1]) for e in ev_k if e is not None]
               for n in names}
    t_total = max_over_ranks(t0_ev.elapsed_time(t1_ev) / 1e3, dist, dev)
    if plan.ws.status() != 0:
        raise RuntimeError(f"device status {plan.ws.status():#x} after timing")

    # e2e through the public API with host buffers: per step, H2D of the
    # step's decode inputs (q, weights, context lens, page table) from pinned
    # memory, the step, D2H of both top-2048 index sets.  HostStepPipeline
    # keeps two steps in flight (two slots, each replaying one CUDA graph of
    # copies + kernels + copies on its own stream); every step's copies stay
    # inside the timed region, which runs from an event before the first H2D
    # to the end of the last D2H.
    slots = []
    for _ in range(2):
        hin = {k: torch.from_numpy(case[k]).pin_memory()
               for k in ("q", "weights", "context_lens", "page_table")}
        hout = [torch.empty_like(plan.topk_idx, device="cpu").pin_memory(),
                torch.empty_like(plan.sparse_idx, device="cpu").pin_memory()]
        slots.append((hin, hout))
    host_in, host_out = slots[0]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out)
    Ke = max(200, min(K, 1000))  # long enough that pipeline fill and drain do not dominate
    pipe = HostStepPipeline(w.B, nn, max(w.context_lens), ps, d["kv"], d["kscale"], k=2048,
                            kb=512, device=dev)

    def submit(j):
        hin, hout = slots[j % 2]
        pipe.submit(hin["q"], hin["weights"], hin["context_lens"], hin["page_table"],
                    hout[0], hout[1])

    for j in range(max(4, args.warmup)):
        submit(j)
    pipe.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e_start.record()
    pipe.start_after(e_start)
    for j in range(Ke):
        submit(j)
    for e in pipe.record_all():
        torch.cuda.current_stream().wait_event(e)
    e_end.record()
    torch.cuda.synchronize()
    pipe.synchronize()
    e2e_s = max_over_ranks(e_start.elapsed_time(e_end) / 1e3, dist, dev)
    for p2 in pipe.plans:
        if p2.ws.status() != 0:
            raise RuntimeError(f"device status {p2.ws.status():#x} after the e2e loop")
    # the same copies and step issued back to back on one stream (diagnostic)
    Ks = max(1, min(K, 200))
    s_start, s_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s_start.record()
    for _ in range(Ks):
        for k2, v in host_in.items():
            d[k2].copy_(v, non_blocking=True)
        a, b = plan.step(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                         d["context_lens"])
        host_out[0].copy_(a, non_blocking=True)
        host_out[1].copy_(b, non_blocking=True)
    s_end.record()
    torch.cuda.synchronize()
    e2e_serial_us = 1e3 * s_start.elapsed_time(s_end) / Ks
    del pipe

    # per-stage split (diagnostic, outside the timed region): events between
    # the stages, so the stages sum to more than a step
    stages = ["logits", "select", "publish", "consume"]
    Kd = max(1, min(K, 200))
    ev_d = [{n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for n in stages} for _ in range(Kd)]
    for i in range(Kd):
        plan.step(*inputs, events=ev_d[i])
    torch.cuda.synchronize()
    stage_us_eager = {n: 1e3 * statistics.mean(e[n][0].elapsed_time(e[n][1]) for e in ev_d)
                      for n in stages}
    # the same split from a CUDA graph of the step whose timing events are
    # graph nodes, as the timed loop runs it: no host launch gaps between the
    # stages (an event between two kernels still holds back the second's
    # programmatic launch, so these stages too sum to more than a step)
    stage_us = None
    try:
        evg = {n: (torch.cuda.Event(enable_timing=True, external=True),
                   torch.cuda.Event(enable_timing=True, external=True)) for n in stages}
        gst = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gst):
            plan.step(*inputs, events=evg)
        acc = {n: [] for n in stages}
        for i in range(Kd + 3):
            gst.replay()
            torch.cuda.synchronize()
            if i >= 3:
                for n in stages:
                    acc[n].append(1e3 * evg[n][0].elapsed_time(evg[n][1]))
        stage_us = {n: statistics.mean(v) for n, v in acc.items()}
        del gst
    except Exception as exc:  # a torch without graph-node timing events
        print(f"[bench] graph-timed stage split unavailable: {exc}", file=sys.stderr)
    stage_note = ("stage_us: CUDA-graph replays of the step with timing events as graph nodes "
                  "between the stages; stage_us_eager: the same split from eager steps. "
                  "Each stage includes its kernels' set-up without programmatic overlap and "
                  "the event pair's own cost: 'publish' holds no launch in the fused-table "
                  "plan and reads that cost alone")
    if stage_us is None:
        stage_us = stage_us_eager
        stage_note = "stages timed in eager steps with events between them"
    # the step replayed from its CUDA graph alone (diagnostic, untimed region)
    Kg = max(1, min(K, 200))
    gs, ge = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    plan.replay()
    torch.cuda.synchronize()
    gs.record()
    for _ in range(Kg):
        plan.replay()
    ge.record()
    torch.cuda.synchronize()
    graph_us = 1e3 * gs.elapsed_time(ge) / Kg

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    peak, peak_kind = peaks()
    lg_ms = statistics.mean(kern_ms["logits"])
    achieved = logits_bytes / (lg_ms * 1e-3) / 1e9
    ms_step = 1e3 * t_total / K
    value = whole_job_rate(keys_per_step, world, K, t_total)
    cb = None
    if not args.no_cpu_baseline:
        cb = cpu_baseline(case, w, args.cpu_budget)
    mx = None if args.no_mx else measure_mx_logits(case, w, d, dev)
    per_workload = None
    if not args.no_per_workload:
        per_workload = {nm: measure_workload(nm, dev) for nm in PER_WORKLOADS
                        if nm != args.workload}
    kstream_gbs = kv_bytes / (lg_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "keys/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8e4m3 x fp8e4m3 -> f32", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "next_n": nn, "context_len": int(ctx.max()),
                   "page_size": ps, "H": 32, "D": 128, "k": 2048, "k_blocks": 512,
                   "dist": w.dist, "seed": w.seed, "parallelism": f"replicas x{world}",
                   "l2": (f"not flushed: inputs larger than L2 (each step streams "
                          f"{kv_bytes / 1e6:.0f} MB of K cache and scales, L2 129 MB)")},
        "hbm_gbs_logits": achieved,
        "kstream_gbs": kstream_gbs,
        "kstream_frac_of_measured_peak": kstream_gbs / peak,
        "kstream_frac_of_8tbs_nominal": kstream_gbs / NOMINAL_GBS,
        "top2048_rows_per_s": world * 2 * w.R * K / t_total,
        "logits_us": 1e3 * lg_ms,
        "logits_launches_timed": len(kern_ms["logits"]),
        "stage_us": stage_us,
        "stage_us_eager": stage_us_eager,
        "stage_note": stage_note,
        "timed_loop": "CUDA-graph replays of the step; every %d-th step eager with the "
                      "dense logits launch bracketed by events" % every,
        "graph_us_per_step": graph_us,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "kernel": "logits_kernel<next_n=1, histogram>",
                     "algorithmic_bytes_per_launch": logits_bytes,
                     "traffic": traffic_record(os.path.join(
                         ROOT, "dsa_sparse_attention_paged_gb300", "csrc", "logits.cu"))},
        "cpu_baseline": cb,
        "e2e": {"value": whole_job_rate(keys_per_step, world, Ke, e2e_s), "unit": "keys/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": 1e3 * e2e_s / Ke, "steps": Ke,
                "overlap": "two slots in flight, each a CUDA graph of H2D + step + D2H",
                "serial_one_stream_us_per_step": e2e_serial_us},
        "gpu_launches": plan.launches_per_step * K,
        "clocks": clocks,
        "mxfp4_logits": mx,
        "per_workload": per_workload,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
