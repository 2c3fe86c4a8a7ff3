"""Helpers for the GPU parity tests: move a synth.Problem to the device, run the
library through its C ABI binding, and compare against the fp64 oracle with the
stated tolerances (relative L2 <= 1e-2 and max-abs <= 2e-2 per output tensor)."""
from __future__ import annotations

import numpy as np

import synth

REL_L2 = 1e-2
MAX_ABS = 2e-2


to_device = synth.to_device  # the problem's arrays on the device (plain copies)


def bf16_to_f64(t):
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def with_dtype(p: synth.Problem, options):
    """The options with the input format of the problem (fp16 inputs need their workspace copies)."""
    import dataclasses

    import linear_attention_varlen_gb300 as gdn
    return dataclasses.replace(options or gdn.Options(), fp16_inputs=(p.dtype == "f16"))


def run_fwd(p: synth.Problem, options=None):
    import linear_attention_varlen_gb300 as gdn
    import torch
    options = with_dtype(p, options)
    d = to_device(p)
    ws = torch.empty(gdn.fwd_workspace_size(p.N, p.T, p.Hk, p.Hv, options), dtype=torch.uint8, device="cuda")
    out, fin = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_idx"],
                             d["initial_state"], options=options, workspace=ws)
    st = gdn.workspace_status(ws)
    assert st == 0, f"device status {gdn.status_string(st)}"
    return bf16_to_f64(out), fin.double().cpu().numpy()


def errors(got, ref):
    diff = got - ref
    n = np.linalg.norm(ref)
    rel = np.linalg.norm(diff) / n if n > 0 else np.linalg.norm(diff)
    return float(rel), float(np.abs(diff).max()) if diff.size else 0.0


def assert_close(name, got, ref, rel_l2=REL_L2, max_abs=MAX_ABS):
    assert got.shape == ref.shape, f"{name}: shape {got.shape} vs {ref.shape}"
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    rel, mx = errors(got, ref)
    assert rel <= rel_l2 and mx <= max_abs, f"{name}: rel-L2 {rel:.3e} (<= {rel_l2}), max-abs {mx:.3e} (<= {max_abs})"
    return rel, mx


def head_slice(p: synth.Problem, heads):
    """The sub-problem of the given value heads (all in one GQA group) with its key head.
    Value heads are independent given their key head, so the oracle can check a sample
    of heads of a full-size workload one head at a time."""
    G = p.Hv // p.Hk
    hk = heads[0] // G
    assert all(h // G == hk for h in heads)
    q = synth.Problem(name=p.name + f"_h{heads}", q=p.q[:, hk:hk + 1], k=p.k[:, hk:hk + 1],
                      v=p.v[:, heads], g=p.g[:, heads], beta=p.beta[:, heads], cu_seqlens=p.cu_seqlens,
                      Hk=1, Hv=len(heads), Dk=p.Dk, Dv=p.Dv, init_idx=p.init_idx,
                      initial_state=None if p.initial_state is None else p.initial_state[:, heads])
    q.q = np.ascontiguousarray(q.q)
    q.k = np.ascontiguousarray(q.k)
    q.v = np.ascontiguousarray(q.v)
    q.g = np.ascontiguousarray(q.g)
    q.beta = np.ascontiguousarray(q.beta)
    if q.initial_state is not None:
        q.initial_state = np.ascontiguousarray(q.initial_state)
    return q


def run_bwd(p: synth.Problem, options=None):
    """Backward through the library; returns fp64 numpy dq, dk, dv, dg, dbeta, dinit."""
    import linear_attention_varlen_gb300 as gdn
    import torch
    options = with_dtype(p, options)
    d = to_device(p)
    ws = torch.empty(gdn.bwd_workspace_size(p.N, p.T, p.Hk, p.Hv, options), dtype=torch.uint8, device="cuda")
    gr = gdn.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["dout"], d.get("dfinal_state"),
                       d["init_idx"], d["initial_state"], options=options, workspace=ws)
    st = gdn.workspace_status(ws)
    assert st == 0, f"device status {gdn.status_string(st)}"
    out = {k: gr[k].double().cpu().numpy() for k in ("dq", "dk", "dv", "dg", "dbeta")}
    out["dinit"] = None if gr["dinit"] is None else gr["dinit"].double().cpu().numpy()
    return out


def run_train(p: synth.Problem, options=None):
    """Training step through the library: a forward that keeps its records (save_for_backward),
    then the backward on the same workspace (reuse_forward). Returns (out, final_state, grads) as
    fp64 numpy arrays."""
    import dataclasses

    import linear_attention_varlen_gb300 as gdn
    import torch
    base = with_dtype(p, options)
    fo = dataclasses.replace(base, save_for_backward=True, reuse_forward=False)
    bo = dataclasses.replace(base, save_for_backward=False, reuse_forward=True)
    d = to_device(p)
    ws = torch.empty(gdn.fwd_workspace_size(p.N, p.T, p.Hk, p.Hv, fo), dtype=torch.uint8, device="cuda")
    assert ws.numel() == gdn.bwd_workspace_size(p.N, p.T, p.Hk, p.Hv, base)
    out, fin = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_idx"],
                             d["initial_state"], options=fo, workspace=ws)
    st = gdn.workspace_status(ws)
    assert st == 0, f"device status {gdn.status_string(st)}"
    gr = gdn.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["dout"], d.get("dfinal_state"),
                       d["init_idx"], d["initial_state"], options=bo, workspace=ws)
    st = gdn.workspace_status(ws)
    assert st == 0, f"device status {gdn.status_string(st)}"
    grads = {k: gr[k].double().cpu().numpy() for k in ("dq", "dk", "dv", "dg", "dbeta")}
    grads["dinit"] = None if gr["dinit"] is None else gr["dinit"].double().cpu().numpy()
    return bf16_to_f64(out), fin.double().cpu().numpy(), grads


def mixed_decay_problem(name, seed, nchunks=30, Hk=1, Hv=2, with_dout=False, beta_boost=None):
    """One document whose gates change regime along it: slow decay (u ~ N(6, 1)) in its first
    third, fast (u ~ N(-3, 1)) in the second, the workloads' (u ~ N(2, 1)) in the last. With
    beta_boost, beta in the middle third is multiplied by it, so that beta |k|^2 exceeds 2 there:
    chunks whose token transitions do not contract."""
    T = 64 * nchunks + 5
    p = synth.make_problem(name, seed, [T], Hk, Hv, with_dout=with_dout, g_mean=6.0)
    fast = synth.make_problem(name, seed + 1, [T], Hk, Hv, g_mean=-3.0)
    mid = synth.make_problem(name, seed + 2, [T], Hk, Hv, g_mean=2.0)
    a, b = T // 3, 2 * T // 3
    g = p.g.copy()
    g[a:b] = fast.g[a:b]
    g[b:] = mid.g[b:]
    p.g = g.astype(np.float32)
    if beta_boost:
        beta = p.beta.copy()
        beta[a:b] *= beta_boost
        p.beta = beta.astype(np.float32)
    return p


def fast_then_slow_problem(name, seed, fast_chunks=8, slow_chunks=40, Hk=1, Hv=2, with_dout=False):
    """One document: fast decay (u ~ N(-3, 1)) over its first chunks, then slow decay (u ~ N(6, 1))
    for longer than a warm-up window can reach back. With short segments, a segment a little
    under a window after the fast stretch warms up while the next one cannot and waits for the
    state it publishes."""
    T = 64 * (fast_chunks + slow_chunks) + 5
    p = synth.make_problem(name, seed, [T], Hk, Hv, with_dout=with_dout, g_mean=6.0)
    fast = synth.make_problem(name, seed + 1, [T], Hk, Hv, g_mean=-3.0)
    g = p.g.copy()
    g[:64 * fast_chunks] = fast.g[:64 * fast_chunks]
    p.g = g.astype(np.float32)
    return p
