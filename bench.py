"""Benchmark of the chunked Gated DeltaNet on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--mode exact|truncate]

Workload: one 32768-token sequence, 8 value heads over 2 key heads, head dimension
128, chunk 64 (the 32K prefill at a TP8-style per-GPU shape of "How to Speed Up GDN
Kernels for Qwen Models", sections "The real enemy: an idle GPU" and "What it adds
up to"); seeded synthetic inputs (synth.workload_long). A step is one pass of the
library's forward (and backward, when the library provides it) over that batch.

Prints ONE JSON line (rank 0). `value` is Mtokens/s over all ranks; `roofline`
describes the dominant kernel (achieved algorithmic bytes / its CUDA-event time);
`cpu_baseline` is the fp64 oracle timed on this host's cores; `e2e` is the same
metric through the public API with host buffers and host<->device copies inside
the timed region. N > 1 runs independent replicas (one per GPU, no collective on
the data path) launched by torchrun.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN fwd/bwd Mtokens/s at 32K x 8 heads; % of binding bf16-TC/HBM roofline"
UNIT = "Mtokens/s"
# Context only (another machine): FlashQLA forward, 32K prefill at TP8 on H200, 0.31 ms.
PAGE_FWD_MTOK_S = 32768 / 0.31e-3 / 1e6
# Algorithmic counts per token at H_v = 8, H_k = 2, d = 128 (inputs read once, outputs written once;
# FLOPs of the chunked method with K K^T / Q K^T shared across a key-head group).
D = 128


def algorithmic_fwd(T, Hk, Hv, N):
    bytes_ = T * (2 * Hk * D * 2 + Hv * D * 2 + 2 * Hv * 4 + Hv * D * 2) + N * Hv * D * D * 4
    flops = T * (Hk * 4 * 64 * D + Hv * (6 * 64 * D + 6 * D * D))
    return bytes_, flops


def algorithmic_bwd(T, Hk, Hv, N):
    # read q, k, v, g, beta, dO; write dq, dk, dv (fp32), dg, dbeta
    bytes_ = T * (2 * Hk * D * 2 + 2 * Hv * D * 2 + 2 * Hv * 4) + T * (2 * Hk * D * 4 + Hv * D * 4 + 2 * Hv * 4)
    flops = T * (Hk * 4 * 64 * D + Hv * (14 * D * D + 26 * 64 * D))
    return bytes_, flops


def kernel_counts(T, Hk, Hv, N):
    """Algorithmic (bytes, FLOPs) per launch of the kernels that can dominate a step: inputs a
    kernel must read and outputs it must write (no intermediates), and the FLOPs of the matrix
    products its math needs (compensation products not counted)."""
    C = 64
    n_ch = T / C
    fb, ff = algorithmic_fwd(T, Hk, Hv, N)
    # chain (forward output pass): q, k, v in; o, final state out; W S, K~^T V', Q S, P V'
    chain = (fb - T * 2 * Hv * 4, n_ch * Hv * 2 * (3 * C * D * D + C * C * D))
    # grad_kernel: q, k, v, dO, g, beta in; dk, dv, dg, dbeta out (fp32)
    grad_b = T * (2 * Hk * D * 2 + 2 * Hv * D * 2 + 2 * Hv * 4) + T * (Hk * D * 4 + Hv * D * 4 + 2 * Hv * 4)
    # per value head: K dS, dV' S^T, V'_s dS^T (C D^2 each); dO V'^T, dV' V^T, dW K^T, P Q,
    # T_u^T dV', T_w^T dW, dKK K (C^2 D each); dT T^T, T^T R (C^3 each); per key head K K^T, Q K^T.
    # The term of dgamma through q S dO needs no product of its own: dq_kernel forms it from dO S^T.
    grad_f = n_ch * (Hk * 2 * 2 * C * C * D + Hv * 2 * (3 * C * D * D + 7 * C * C * D + 2 * C * C * C))
    # dq_kernel: q, k, dO, g in; dq out (fp32); dO S^T, dO V'^T, (dQK o E) K
    dq_b = T * (2 * Hk * D * 2 + Hv * D * 2 + Hv * 4) + T * Hk * D * 4
    dq_f = n_ch * Hv * 2 * (C * D * D + 2 * C * C * D)
    # reverse chain: k, q, dO in; K~ dS, P^T dO, Q~^T dO, W^T dV'
    rev_b = T * (2 * Hk * D * 2 + Hv * D * 2)
    rev_f = n_ch * Hv * 2 * (3 * C * D * D + C * C * D)
    # kkt_solve: k, g, beta in; K K^T and the 64x64 solve per value head
    kkt_b = T * (Hk * D * 2 + 2 * Hv * 4)
    kkt_f = n_ch * (Hk * 2 * C * C * D + Hv * C * C * C / 3)
    # out_kernel (o from the records of a training forward): q in, o out; Q S, P V' per value head
    out_b = T * (Hk * D * 2 + Hv * D * 2)
    out_f = n_ch * Hv * 2 * (C * D * D + C * C * D)
    return {"chain_kernel<out>": chain, "chain_kernel<out,record>": chain, "grad_kernel": (grad_b, grad_f),
            "dq_kernel": (dq_b, dq_f), "rev_chain_kernel": (rev_b, rev_f), "kkt_solve_kernel": (kkt_b, kkt_f),
            "kkt_solve_kernel<record>": (kkt_b, kkt_f), "out_kernel": (out_b, out_f)}


def whole_job(ms, tokens_per_rank, world, device=None):
    """Replicas: the slowest rank's mean step time (max over ranks) and the whole-job rate in
    Mtokens/s (every rank's tokens over that time). One process per GPU, no collective on the
    data path; this reduction runs once, after the timed steps."""
    if world > 1:
        import torch
        t = torch.tensor([float(ms)], device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    return ms, tokens_per_rank * world / (ms * 1e-3) / 1e6


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return dict(hbm=float(pk["hbm_gbs"]), tc=float(pk["bf16_tflops"]), tc_sus=float(pk.get(
            "bf16_tflops_sustained", pk["bf16_tflops"])), src="measured")
    return dict(hbm=6800.0, tc=1900.0, tc_sus=1700.0, src="fallback")


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
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
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- reference arm (fp64 oracle)


def _oracle_step(p, f, cores):
    """One forward + backward of the fp64 oracle on problem p (the bench step's work)."""
    import oracle
    oracle.fwd(f["q"], f["k"], f["v"], f["g"], f["beta"], p.cu_seqlens, threads=cores)
    oracle.bwd(f["q"], f["k"], f["v"], f["g"], f["beta"], p.cu_seqlens, f["dout"], threads=cores)


def workload_config(T, Hv, Hk, mode, has_bwd, train):
    """The `config` object of the bench line; the reference arm reports the same one."""
    return {"workload": "GDN " + ("fwd+bwd" if has_bwd else "fwd") + f", one {T}-token sequence, H_v={Hv}, "
            f"H_k={Hk}, d_k=d_v=128, chunk 64, " + mode + " mode", "T": T, "H_v": Hv, "H_k": Hk,
            "mode": mode, "pass": "fwd+bwd" if has_bwd else "fwd",
            "step": ("training step: forward keeping its records (save_for_backward), backward reusing "
                     "them (reuse_forward)" if train else
                     ("forward, then a backward that recomputes the forward" if has_bwd else "forward")),
            "l2": "flushed between timed steps (512 MiB write outside the timed events)"}


def run_reference(args, rank):
    if rank != 0:
        return None
    import numpy as np

    import oracle
    import synth
    oracle.build()
    T_sample = 1024
    p = synth.make_problem(f"long_sample_T{T_sample}", synth.SEEDS[2], [T_sample], 2, 8, with_dout=True)
    f = p.as_f64()
    cores = oracle.hw_threads()
    for _ in range(args.warmup):
        _oracle_step(p, f, cores)
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _oracle_step(p, f, cores)
        ts.append(time.perf_counter() - t0)
    sec = float(np.mean(ts))
    value = T_sample / sec / 1e6
    sample = (f"a {T_sample}-token single sequence with the 32768-token workload's shapes and distributions "
              f"(H_v=8, H_k=2), fp64 oracle forward + backward per step")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(workload_config(args.tokens, 8, 2, args.mode, True, args.mode == "exact"),
                       l2="not applicable: the fp64 oracle on the host cores, one sample per step",
                       sample_tokens_per_step=T_sample,
                       sample=f"each step runs the oracle on the first {T_sample} tokens' worth of the workload "
                              f"(same shapes and distributions); Mtokens/s of the token-by-token recurrence is "
                              f"independent of the sequence length"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def cpu_baseline(T_full):
    """The fp64 oracle's forward + backward on a bounded sample of the workload (the first 4096
    tokens' shape), repeated until about 10 s of CPU work."""
    import oracle
    import synth
    oracle.build()
    T_s = min(4096, T_full)
    p = synth.make_problem(f"long_sample_T{T_s}", synth.SEEDS[2], [T_s], 2, 8, with_dout=True)
    f = p.as_f64()
    cores = oracle.hw_threads()
    total, runs = 0.0, 0
    while runs < 1 or (total < 10.0 and runs < 200):
        t0 = time.perf_counter()
        _oracle_step(p, f, cores)
        total += time.perf_counter() - t0
        runs += 1
    return {"value": p.T * runs / total / 1e6, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{T_s}-token single sequence, 8 value heads over 2 key heads, forward + backward, "
                      f"{runs} run(s), {total:.1f} s"}


# ----------------------------------------------------------------------------- our arm


def traffic_record(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summaries (profiles/traffic.json:
    one record per kernel), if the record was taken on the current source of that kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        recs = json.load(open(path))
        rec = recs.get(kernel) if isinstance(recs, dict) else None
        if not rec:
            return None
        sha = hashlib.sha256(open(os.path.join(ROOT, rec["source"]), "rb").read()).hexdigest()
        if rec.get("source_sha256") == sha:
            return rec
    except (OSError, ValueError, KeyError):
        pass
    return None


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import linear_attention_varlen_gb300 as gdn
    import synth
    from linear_attention_varlen_gb300 import build as gdn_build
    from synth import to_device

    gdn_build.build()
    gdn.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    p = synth.workload_long(T=args.tokens)
    d = to_device(p, dev)
    T, Hk, Hv, N = p.T, p.Hk, p.Hv, p.N
    stream = torch.cuda.current_stream()
    ev_f = [torch.cuda.Event(enable_timing=True) for _ in range(2 * gdn.NUM_STAGES)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(2 * gdn.NUM_STAGES)]
    for e in ev_f + ev_b:
        e.record(stream)
    opts = gdn.Options(mode=args.mode)
    ws = torch.empty(max(gdn.fwd_workspace_size(N, T, Hk, Hv, opts), gdn.bwd_workspace_size(N, T, Hk, Hv, opts)),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((T, Hv, D), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((N, Hv, D, D), dtype=torch.float32, device=dev)
    dout = torch.randn((T, Hv, D), device=dev).to(torch.bfloat16)

    def fwd(o):
        gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], None, None, options=o, out=out,
                      final_state=fin, workspace=ws)

    has_bwd = True
    try:
        gdn.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], dout, options=opts, workspace=ws)
    except gdn.GdnError as e:
        if e.status != gdn.GDN_ERR_UNSUPPORTED:
            raise
        has_bwd = False

    # A training step (exact mode) keeps the forward's records for its backward: the forward runs the
    # backward's recompute and forms o from the records, the backward skips the recompute.
    train = has_bwd and args.mode == "exact"
    o_fwd = gdn.Options(mode=args.mode, save_for_backward=train)
    o_bwd = gdn.Options(mode=args.mode, reuse_forward=train)

    def step(of, ob):
        fwd(of)
        if has_bwd:
            gdn.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], dout, options=ob, workspace=ws)

    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)  # > 129 MB L2
    for _ in range(args.warmup):
        step(o_fwd, o_bwd)
    torch.cuda.synchronize()
    st = gdn.workspace_status(ws)
    if st != gdn.GDN_OK:
        raise RuntimeError(f"device status after warm-up: {gdn.status_string(st)}")
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    split_launched = args.mode == "exact" and N * Hv < 2 * n_sm  # pass 1 of the exact split runs

    infer_f = {gdn.STAGE_PLAN: "plan_kernel", gdn.STAGE_KKT_SOLVE: "kkt_solve_kernel",
               gdn.STAGE_SPLIT: "chain_kernel<pass1>", gdn.STAGE_CHAIN: "chain_kernel<out>"}
    recomp_b = {gdn.STAGE_PLAN: "plan_kernel", gdn.STAGE_KKT_SOLVE: "kkt_solve_kernel<record>",
                gdn.STAGE_SPLIT: "chain_kernel<pass1,record>", gdn.STAGE_CHAIN: "chain_kernel<out,record>",
                gdn.STAGE_REV_CHAIN: "rev_chain_kernel", gdn.STAGE_GRADS: "grad_kernel",
                gdn.STAGE_DQ: "dq_kernel", gdn.STAGE_DINIT: "dinit_reduce_kernel"}
    if train:
        fnames = {gdn.STAGE_PLAN: "plan_kernel", gdn.STAGE_KKT_SOLVE: "kkt_solve_kernel<record>",
                  gdn.STAGE_SPLIT: "chain_kernel<pass1,record>", gdn.STAGE_CHAIN: "chain_kernel<out,record>",
                  gdn.STAGE_OUT: "out_kernel"}
        bnames = {gdn.STAGE_PLAN: "plan_kernel", gdn.STAGE_REV_CHAIN: "rev_chain_kernel",
                  gdn.STAGE_GRADS: "grad_kernel", gdn.STAGE_DQ: "dq_kernel", gdn.STAGE_DINIT: "dinit_reduce_kernel"}
    else:
        fnames, bnames = infer_f, recomp_b
    counts = kernel_counts(T, Hk, Hv, N)

    def new_events(n):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in ev:  # creates the CUDA events (the library records them again inside each call)
            e.record(stream)
        return ev

    # Stage breakdown: untimed steps with every stage event (each recorded event costs about two
    # microseconds of stream time, so the timed steps below record only the dominant kernel's pair)
    diag_n = max(3, min(args.steps, 10))
    dev_ = [(new_events(2 * gdn.NUM_STAGES), new_events(2 * gdn.NUM_STAGES)) for _ in range(diag_n)]
    torch.cuda.synchronize()
    for i in range(diag_n):
        flush.zero_()
        step(dataclasses.replace(o_fwd, stage_events=dev_[i][0]), dataclasses.replace(o_bwd, stage_events=dev_[i][1]))
    torch.cuda.synchronize()
    stage_f = np.zeros((diag_n, gdn.NUM_STAGES))
    stage_b = np.zeros((diag_n, gdn.NUM_STAGES))
    for i in range(diag_n):
        ef, eb = dev_[i]
        for s_ in range(gdn.NUM_STAGES):
            stage_f[i, s_] = ef[2 * s_].elapsed_time(ef[2 * s_ + 1])
            if has_bwd:
                stage_b[i, s_] = eb[2 * s_].elapsed_time(eb[2 * s_ + 1])
    avg = stage_f.mean(axis=0)
    bavg = stage_b.mean(axis=0)
    # the dominant kernel of the step (one launch per stage, except the two-pass reverse chain)
    cands = [(avg[s_], fnames[s_], 0, s_) for s_ in fnames]
    if has_bwd:
        cands += [(bavg[s_], bnames[s_], 1, s_) for s_ in bnames]
    _, dom, dom_call, dom_stage = max((c for c in cands if c[1] in counts), key=lambda c: c[0])

    clocks = ClockSampler(local_rank) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    # the dominant kernel's own events in every timed step; steps enqueued back to back (the host
    # runs ahead of the device), events read once all steps have run
    dom_ev = [new_events(2) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        sev = [None] * (2 * gdn.NUM_STAGES)
        sev[2 * dom_stage], sev[2 * dom_stage + 1] = dom_ev[i]
        of = dataclasses.replace(o_fwd, stage_events=sev) if dom_call == 0 else o_fwd
        ob = dataclasses.replace(o_bwd, stage_events=sev) if dom_call == 1 else o_bwd
        flush.zero_()
        starts[i].record(stream)
        step(of, ob)
        stops[i].record(stream)
    torch.cuda.synchronize()
    dom_ms = float(np.mean([a_.elapsed_time(b_) for a_, b_ in dom_ev]))
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop() if clocks else None
    step_ms = np.array([a.elapsed_time(b) for a, b in zip(starts, stops)])
    ms, value = whole_job(float(step_ms.mean()), T, world, dev)

    # context, outside the timed region: the inference forward and the backward that recomputes
    ctx = None
    if train:
        ctx_n = max(3, min(args.steps, 10))
        ctx_f = np.zeros((ctx_n, gdn.NUM_STAGES))
        ctx_b = np.zeros((ctx_n, gdn.NUM_STAGES))
        for i in range(ctx_n):
            flush.zero_()
            torch.cuda.nvtx.range_push("fwd_inference")  # a marker for profiler filters (no-op otherwise)
            fwd(dataclasses.replace(opts, stage_events=ev_f))
            torch.cuda.nvtx.range_pop()
            gdn.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], dout,
                          options=dataclasses.replace(opts, stage_events=ev_b), workspace=ws)
            torch.cuda.synchronize()
            for s_ in range(gdn.NUM_STAGES):
                ctx_f[i, s_] = ev_f[2 * s_].elapsed_time(ev_f[2 * s_ + 1])
                ctx_b[i, s_] = ev_b[2 * s_].elapsed_time(ev_b[2 * s_ + 1])
        ctx = (ctx_f.mean(axis=0), ctx_b.mean(axis=0))

    # e2e: the same step through the public API from pinned host buffers, every step's copies inside
    # the timed region: its inputs (and the output gradient) host->device, its outputs (o, final
    # state, gradients) device->host. Copies run on their own streams with two device buffer sets,
    # so that step i + 1's inputs come in and step i - 1's outputs go out while step i computes.
    host = {k: v.detach().cpu().pin_memory() for k, v in d.items() if v is not None}
    if has_bwd:
        host["dout"] = dout.cpu().pin_memory()
    gshapes = {"dq": d["q"].shape, "dk": d["k"].shape, "dv": d["v"].shape, "dg": (T, Hv), "dbeta": (T, Hv)}
    host_out = {"out": torch.empty(out.shape, dtype=out.dtype, pin_memory=True),
                "fin": torch.empty(fin.shape, dtype=fin.dtype, pin_memory=True)}
    if has_bwd:
        host_out.update({k2: torch.empty(sh, dtype=torch.float32, pin_memory=True) for k2, sh in gshapes.items()})
    dev_in = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    dev_out = [{"out": torch.empty_like(out), "fin": torch.empty_like(fin)} for _ in range(2)]
    if has_bwd:
        for b_ in dev_out:
            b_.update({k2: torch.empty(sh, dtype=torch.float32, device=dev) for k2, sh in gshapes.items()})
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    e2e_steps = max(3, min(args.steps, 50))
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    ev_in, ev_comp, ev_out = ([ev() for _ in range(e2e_steps)] for _ in range(3))
    torch.cuda.synchronize()
    ea = ev()
    ea.record(s_in)
    for i in range(e2e_steps):
        bi, bo = dev_in[i % 2], dev_out[i % 2]
        if i >= 2:
            s_in.wait_event(ev_comp[i - 2])  # step i - 2 has read this input set
        with torch.cuda.stream(s_in):
            for k2, v2 in host.items():
                bi[k2].copy_(v2, non_blocking=True)
        ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        if i >= 2:
            stream.wait_event(ev_out[i - 2])  # step i - 2's outputs have left this output set
        gdn.chunk_fwd(bi["q"], bi["k"], bi["v"], bi["g"], bi["beta"], bi["cu_seqlens"], None, None, options=o_fwd,
                      out=bo["out"], final_state=bo["fin"], workspace=ws, stream=stream)
        if has_bwd:
            gdn.chunk_bwd(bi["q"], bi["k"], bi["v"], bi["g"], bi["beta"], bi["cu_seqlens"], bi["dout"],
                          options=o_bwd, workspace=ws, stream=stream, grads=bo)
        ev_comp[i].record(stream)
        s_out.wait_event(ev_comp[i])
        with torch.cuda.stream(s_out):
            for k2, v2 in host_out.items():
                v2.copy_(bo[k2], non_blocking=True)
        ev_out[i].record(s_out)
    torch.cuda.synchronize()
    e2e_ms = ea.elapsed_time(ev_out[-1]) / e2e_steps
    e2e_value = T * world / (e2e_ms * 1e-3) / 1e6

    # The inference forward alone (exact mode, the 32K x 8-head prefill) and the truncation mode, each
    # timed with one event pair around the whole call (L2 flushed before each), outside the step
    # loop; truncation's deviation from the exact forward on the same inputs.
    def time_forward(mode, reps):
        of = gdn.Options(mode=mode)
        for _ in range(3):
            fwd(of)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for a_, b_ in evs:
            flush.zero_()
            a_.record(stream)
            fwd(of)
            b_.record(stream)
        torch.cuda.synchronize()
        return float(np.median([a_.elapsed_time(b_) for a_, b_ in evs]))

    fwd_reps = max(10, min(args.steps, 50))
    fwd_exact_ms = time_forward("exact", fwd_reps)
    o_exact, f_exact = out.double().clone(), fin.double().clone()
    fwd_trunc_ms = time_forward("truncate", fwd_reps)
    o_trunc, f_trunc = out.double().clone(), fin.double().clone()

    def deviation(a_, b_):
        n_ = float(torch.linalg.vector_norm(b_))
        return {"rel_l2": float(torch.linalg.vector_norm(a_ - b_)) / n_ if n_ > 0 else 0.0,
                "max_abs": float((a_ - b_).abs().max())}
    trunc_dev = {"out": deviation(o_trunc, o_exact), "final_state": deviation(f_trunc, f_exact)}

    # q / k normalisation (GDN_FLAG_L2NORM_QK) on the inference forward: the whole call, and the
    # normalisation pass alone (its stage events), both with L2 flushed before each call
    l2_reps = max(10, min(args.steps, 50))
    l2_ws = torch.empty(gdn.fwd_workspace_size(N, T, Hk, Hv, gdn.Options(l2norm_qk=True)), dtype=torch.uint8,
                        device=dev)
    l2_stage = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(l2_reps)]
    l2_call = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(l2_reps)]
    for e_ in [e for pr in l2_stage for e in pr]:
        e_.record(stream)
    for _ in range(3):
        gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], options=gdn.Options(l2norm_qk=True),
                      out=out, final_state=fin, workspace=l2_ws)
    torch.cuda.synchronize()
    for (a_, b_), (sa, sb) in zip(l2_call, l2_stage):
        sev = [None] * (2 * gdn.NUM_STAGES)
        sev[2 * gdn.STAGE_L2NORM], sev[2 * gdn.STAGE_L2NORM + 1] = sa, sb
        flush.zero_()
        a_.record(stream)
        gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                      options=gdn.Options(l2norm_qk=True, stage_events=sev), out=out, final_state=fin, workspace=l2_ws)
        b_.record(stream)
    torch.cuda.synchronize()
    l2_fwd_ms = float(np.median([a_.elapsed_time(b_) for a_, b_ in l2_call]))
    l2_pass_ms = float(np.median([a_.elapsed_time(b_) for a_, b_ in l2_stage]))
    l2_bytes = 2 * (2 * T * Hk * D * 2)  # q and k read once, their normalised copies written once
    del l2_ws

    # The width-4 causal convolution in front of the recurrence, over the packed training layout (four
    # 16384-token documents) with the channels of q, k and v at these heads
    CONV_T, CONV_C = 65536, 2 * Hk * D + Hv * D
    cvx = torch.randn((CONV_T, CONV_C), device=dev).to(torch.bfloat16)
    cvdy = torch.randn((CONV_T, CONV_C), device=dev).to(torch.bfloat16)
    cvw = 0.5 * torch.randn((CONV_C, 4), device=dev)
    cvb = 0.1 * torch.randn((CONV_C,), device=dev)
    cvcu = torch.arange(0, CONV_T + 1, 16384, dtype=torch.int32, device=dev)
    cvws = torch.empty(gdn.conv_workspace_size(4, CONV_T, CONV_C, True), dtype=torch.uint8, device=dev)
    conv_reps = max(10, min(args.steps, 50))

    def time_conv(fn):
        for _ in range(3):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(conv_reps)]
        torch.cuda.synchronize()
        for a_, b_ in evs:
            flush.zero_()
            a_.record(stream)
            fn()
            b_.record(stream)
        torch.cuda.synchronize()
        return float(np.median([a_.elapsed_time(b_) for a_, b_ in evs]))
    conv_f_ms = time_conv(lambda: gdn.conv_fwd(cvx, cvw, cvcu, cvb, workspace=cvws))
    conv_b_ms = time_conv(lambda: gdn.conv_bwd(cvx, cvw, cvcu, cvdy, cvb, workspace=cvws))
    conv_f_bytes = CONV_T * CONV_C * (2 + 2)          # x read, y written (bf16)
    conv_b_bytes = CONV_T * CONV_C * (2 + 2 + 4)      # x, dy read, dx written (fp32)
    del cvx, cvdy, cvws

    # Decode: one token for each of DEC_B sequences at the same heads, in place on a pool of states
    # (one entry per sequence); bound by reading and writing every state once.
    DEC_B = 256
    pdec = synth.make_problem("decode_bench", 2024, [1] * DEC_B, Hk, Hv, init_idx=list(range(DEC_B)), n_init=DEC_B)
    ddec = to_device(pdec, dev)
    dec_in = [ddec[x] for x in ("q", "k", "v", "g", "beta")]
    dec_pool, dec_idx = ddec["initial_state"], ddec["init_idx"]
    dec_out = torch.empty((DEC_B, Hv, D), dtype=torch.bfloat16, device=dev)
    for _ in range(3):
        gdn.decode_step(*dec_in, dec_pool, dec_idx, out=dec_out)
    dec_reps = max(10, min(args.steps, 50))
    dec_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(dec_reps)]
    torch.cuda.synchronize()
    for a_, b_ in dec_ev:
        flush.zero_()
        a_.record(stream)
        gdn.decode_step(*dec_in, dec_pool, dec_idx, out=dec_out)
        b_.record(stream)
    torch.cuda.synchronize()
    dec_ms = float(np.median([a_.elapsed_time(b_) for a_, b_ in dec_ev]))
    dec_bytes = DEC_B * (Hv * 2 * D * D * 4 + Hk * 2 * D * 2 + Hv * 2 * D * 2 + Hv * 2 * 4 + 4)
    if world > 1:
        torch.distributed.barrier()

    if rank != 0:
        return None
    peaks = load_peaks()
    fwd_ms = float(sum(avg[s_] for s_ in fnames))
    bwd_ms = float(sum(bavg[s_] for s_ in bnames)) if has_bwd else 0.0
    kb, kf = counts[dom]
    kern_s = dom_ms * 1e-3
    # binding roofline of that kernel at the measured peaks (sustained TC: it runs inside a long step)
    if kb / (peaks["hbm"] * 1e9) >= kf / (peaks["tc_sus"] * 1e12):
        bound, achieved, peak, unit_r = "hbm", kb / kern_s / 1e9, peaks["hbm"], "GB/s"
    else:
        bound, achieved, peak, unit_r = "tensor", kf / kern_s / 1e12, peaks["tc_sus"], "TFLOP/s"
    tr = traffic_record(dom)
    launches_per_step = 3 + (1 if split_launched else 0)
    if train:  # + o from the records; backward: plan, two reverse passes (one unsplit), grad, dq
        launches_per_step += 1 + 1 + (2 if split_launched else 1) + 2
    elif has_bwd:  # recompute (same launches as the forward) + two reverse passes (one unsplit), grad, dq
        launches_per_step += 3 + (1 if split_launched else 0) + (2 if split_launched else 1) + 2
    fb, ff = algorithmic_fwd(T, Hk, Hv, N)
    bb, bf = algorithmic_bwd(T, Hk, Hv, N) if has_bwd else (0, 0)
    step_alg_s = max(fb / (peaks["hbm"] * 1e9), ff / (peaks["tc_sus"] * 1e12))
    if has_bwd:
        step_alg_s += max(bb / (peaks["hbm"] * 1e9), bf / (peaks["tc_sus"] * 1e12))
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / PAGE_FWD_MTOK_S if not has_bwd else None,
        "dtype": "bf16", "data": "synthetic",
        "config": workload_config(T, Hv, Hk, args.mode, has_bwd, train),
        "roofline": {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak, "unit": unit_r,
                     "frac": achieved / peak, "traffic": (tr["bytes_per_launch"] if tr else None),
                     "peak_source": peaks["src"] + (" hbm_gbs" if bound == "hbm" else " bf16_tflops_sustained"),
                     "algorithmic_bytes": kb, "algorithmic_flops": kf, "ms_per_launch": dom_ms},
        "step_roofline": {"frac": step_alg_s / (ms * 1e-3),
                          "note": "sum over forward and backward of max(algorithmic bytes / HBM peak, algorithmic "
                                  "FLOPs / sustained bf16 peak), divided by the measured step time"},
        "stages_note": f"stage times from {diag_n} untimed steps with every stage event recorded; the timed "
                       "steps record only the dominant kernel's pair",
        "stages_ms": {fnames[s_]: float(avg[s_]) for s_ in fnames},
        "bwd_stages_ms": ({bnames[s_]: float(bavg[s_]) for s_ in bnames} if has_bwd else None),
        "fwd_ms": fwd_ms, "bwd_ms": (bwd_ms if has_bwd else None),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "note": "public API from pinned host buffers; each step copies its inputs in and its outputs and "
                        "gradients out, on copy streams overlapping the neighbouring steps' compute"},
        "gpu_launches": int(launches_per_step * args.steps),
        "clocks": clk,
    }
    if ctx is not None:
        res["context"] = {
            "note": "outside the timed region: the inference forward and the backward that recomputes the forward",
            "fwd_inference_ms": float(sum(ctx[0][s_] for s_ in infer_f)),
            "bwd_recompute_ms": float(sum(ctx[1][s_] for s_ in recomp_b)),
            "fwd_inference_stages_ms": {infer_f[s_]: float(ctx[0][s_]) for s_ in infer_f},
            "bwd_recompute_stages_ms": {recomp_b[s_]: float(ctx[1][s_]) for s_ in recomp_b}}
    fb_inf, ff_inf = algorithmic_fwd(T, Hk, Hv, N)

    def fwd_object(ms_):
        t_ = ms_ * 1e-3
        hbm_t, tc_t = fb_inf / (peaks["hbm"] * 1e9), ff_inf / (peaks["tc"] * 1e12)
        bound_ = "hbm" if hbm_t >= tc_t else "tensor"
        ach = fb_inf / t_ / 1e9 if bound_ == "hbm" else ff_inf / t_ / 1e12
        pk = peaks["hbm"] if bound_ == "hbm" else peaks["tc"]
        return {"ms": ms_, "value": T / t_ / 1e6, "unit": UNIT,
                "roofline": {"bound": bound_, "achieved": ach, "peak": pk, "unit": "GB/s" if bound_ == "hbm" else
                             "TFLOP/s", "frac": ach / pk, "algorithmic_bytes": fb_inf, "algorithmic_flops": ff_inf,
                             "peak_source": peaks["src"] + (" hbm_gbs" if bound_ == "hbm" else " bf16_tflops")}}
    fwd_tr = [traffic_record(k_) for k_ in ("kkt_solve_kernel", "chain_kernel<out>")]
    fwd_traffic = sum(r_["bytes_per_launch"] for r_ in fwd_tr) if all(fwd_tr) else None
    res["fwd"] = dict(fwd_object(fwd_exact_ms), mode="exact", traffic=fwd_traffic,
                      traffic_note="DRAM bytes of kkt_solve + the chain output pass (profiles/traffic.json, ncu, "
                                   "scaled from 16384 tokens), null once either kernel's source has changed",
                      note=f"inference forward alone (o and final state), {T} tokens x {Hv} value heads, median of "
                           f"{fwd_reps} calls with one event pair around each and L2 flushed before it; roofline "
                           f"over the whole call (q, k, v, g, beta read once, o and the final state written once)")
    res["truncate"] = dict(fwd_object(fwd_trunc_ms), mode="truncate",
                           threshold=float(opts.trunc_log_threshold),
                           deviation_from_exact=trunc_dev,
                           note="the opt-in truncation mode (segment carries rebuilt from a window whose summed "
                                "log-decay is below the threshold), timed like `fwd`; deviation_from_exact compares "
                                "its o and final state with the exact forward's on the same inputs (the tests bound "
                                "both modes against the fp64 oracle)")
    l2_ach = l2_bytes / (l2_pass_ms * 1e-3) / 1e9
    res["l2norm"] = {"fwd_ms": l2_fwd_ms, "fwd_value": T / (l2_fwd_ms * 1e-3) / 1e6, "unit": UNIT,
                     "pass_ms": l2_pass_ms,
                     "roofline": {"bound": "hbm", "achieved": l2_ach, "peak": peaks["hbm"], "unit": "GB/s",
                                  "frac": l2_ach / peaks["hbm"], "algorithmic_bytes": l2_bytes,
                                  "peak_source": peaks["src"] + " hbm_gbs"},
                     "note": "inference forward with GDN_FLAG_L2NORM_QK (q, k unnormalised): the whole call, and "
                             "the normalisation pass alone between its stage events (a recorded event costs about "
                             "two microseconds, so pass_ms is an upper bound); roofline of the pass: q and k read, "
                             "their normalised copies written"}
    def hbm_obj(bytes_, ms_):
        ach = bytes_ / (ms_ * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm"], "unit": "GB/s", "frac": ach / peaks["hbm"],
                "algorithmic_bytes": bytes_, "peak_source": peaks["src"] + " hbm_gbs"}
    res["conv"] = {"fwd_ms": conv_f_ms, "bwd_ms": conv_b_ms, "T": CONV_T, "C": CONV_C,
                   "fwd_value": CONV_T / (conv_f_ms * 1e-3) / 1e6, "bwd_value": CONV_T / (conv_b_ms * 1e-3) / 1e6,
                   "unit": UNIT, "fwd_roofline": hbm_obj(conv_f_bytes, conv_f_ms),
                   "bwd_roofline": hbm_obj(conv_b_bytes, conv_b_ms),
                   "note": "width-4 causal convolution (gdn_conv_fwd / gdn_conv_bwd) over four 16384-token "
                           "documents, channels of q, k and v; one event pair around each call, L2 flushed "
                           "before it"}
    dec_ach = dec_bytes / (dec_ms * 1e-3) / 1e9
    res["decode"] = {"ms": dec_ms, "value": DEC_B / (dec_ms * 1e-3) / 1e6, "unit": "Msequence-steps/s",
                     "batch": DEC_B, "H_v": Hv, "H_k": Hk,
                     "roofline": {"bound": "hbm", "achieved": dec_ach, "peak": peaks["hbm"], "unit": "GB/s",
                                  "frac": dec_ach / peaks["hbm"], "algorithmic_bytes": dec_bytes,
                                  "peak_source": peaks["src"] + " hbm_gbs"},
                     "note": f"gdn_decode_step: one token for each of {DEC_B} sequences, in place on a pool of "
                             f"{DEC_B} states (each read and written once), median of {dec_reps} steps with one "
                             f"event pair around each and L2 flushed before it"}
    if not has_bwd:
        res["vs_baseline_note"] = "value / FlashQLA forward on H200 (0.31 ms for 32K at TP8), context only"
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(T)
    return res


def profile_fwd(T, g_mean):
    """The inference forward alone on one T-token sequence (H_v=8, H_k=2) with gates
    u ~ N(g_mean, 1), for ncu captures of its kernels (g_mean 6: no exact-split boundary can warm
    up, so pass 1 computes every transition and walks them)."""
    import torch

    import linear_attention_varlen_gb300 as gdn
    import synth
    from synth import to_device
    p = synth.make_problem(f"profile_T{T}_g{g_mean}", synth.SEEDS[2], [T], 2, 8, g_mean=g_mean)
    d = to_device(p)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"])
    for _ in range(3):
        gdn.chunk_fwd(*args)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("profile_fwd")
    for _ in range(2):
        gdn.chunk_fwd(*args)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--mode", choices=["exact", "truncate"], default="exact")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=32768,
                    help="sequence length (32768 = the benchmark; smaller only for profiler captures)")
    ap.add_argument("--profile-fwd", type=float, default=None, metavar="G_MEAN",
                    help="for profiler captures only: run the inference forward alone (3 calls, then 2 in the "
                         "NVTX range 'profile_fwd') with gates u ~ N(G_MEAN, 1), print nothing else, exit")
    args = ap.parse_args()
    if args.profile_fwd is not None:
        profile_fwd(args.tokens, args.profile_fwd)
        return
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
