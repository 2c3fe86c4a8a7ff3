"""The allocation-free forward entry point (gdn_chunk_fwd_noalloc), called through the C ABI.

It exists for callers that cannot allocate device memory themselves (a host program without a
device allocator, or a plugin inside a framework whose pool owns all device memory): it takes no
workspace and uses a fixed array compiled into the library. Its output must match gdn_chunk_fwd
(which takes a caller workspace) and the fp64 oracle within the tolerances the other GPU tests use,
on two calls in a row (the second call finds the first call's leftovers in the shared array).
Errors found on the device are read back with gdn_noalloc_status.

This file sorts last so that a failure here does not stop the rest of the GPU suite."""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, bf16_to_f64, head_slice, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import linear_attention_varlen_gb300 as gdn  # noqa: E402


def _call_noalloc(lib, d, N, T, Hk, Hv, out, fin):
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    o = gdn.Options().c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    n_init = 0 if d.get("initial_state") is None else d["initial_state"].shape[0]
    return lib.gdn_chunk_fwd_noalloc(P(d["q"]), P(d["k"]), P(d["v"]), P(d["g"]), P(d["beta"]), P(d["cu_seqlens"]),
                                     N, T, Hk, Hv, 128, P(d.get("init_idx")), P(d.get("initial_state")), n_init,
                                     P(out), P(fin), ctypes.byref(o), stream)


def _status(lib):
    return lib.gdn_noalloc_status(torch.cuda.current_device(),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _run_twice(lib, p, d):
    res = []
    for _ in range(2):
        out = torch.full((p.T, p.Hv, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        fin = torch.full((p.N, p.Hv, 128, 128), float("nan"), dtype=torch.float32, device="cuda")
        rc = _call_noalloc(lib, d, p.N, p.T, p.Hk, p.Hv, out, fin)
        assert rc == gdn.GDN_OK, gdn.status_string(rc)
        torch.cuda.synchronize()
        assert _status(lib) == gdn.GDN_OK
        res.append((bf16_to_f64(out), fin.double().cpu().numpy()))
    return res


def test_noalloc_forward_matches_workspace_forward_and_oracle_twice():
    lib = gdn.load()
    assert lib.gdn_noalloc_scratch_bytes() > 0
    # pool entry, empty document and two in-call forks (n_init = 1: x >= 1 forks document x - 1)
    problems = [synth.make_problem("noalloc_a", 901, [300, 0, 129, 64], 2, 8, init_idx=[-1, 0, 1, 2], n_init=1),
                synth.workload_single()]
    for p in problems:
        d = to_device(p)
        ws = torch.empty(gdn.fwd_workspace_size(p.N, p.T, p.Hk, p.Hv), dtype=torch.uint8, device="cuda")
        ref_out, ref_fin = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_idx"],
                                         d["initial_state"], workspace=ws)
        assert gdn.workspace_status(ws) == gdn.GDN_OK
        ro, rf = oracle.fwd_problem(p)
        assert np.abs(ro).max() > 0
        for out, fin in _run_twice(lib, p, d):
            assert_close(f"{p.name} out vs gdn_chunk_fwd", out, bf16_to_f64(ref_out))
            assert_close(f"{p.name} final_state vs gdn_chunk_fwd", fin, ref_fin.double().cpu().numpy())
            assert_close(f"{p.name} out vs oracle", out, ro)
            assert_close(f"{p.name} final_state vs oracle", fin, rf)


def test_noalloc_runs_the_32k_prefill():
    """One 32768-token document at 8 value heads over 2 key heads fits the array; two value heads
    of one key head are checked against the oracle, the rest against gdn_chunk_fwd."""
    lib = gdn.load()
    p = synth.workload_long()
    assert gdn.fwd_workspace_size(p.N, p.T, p.Hk, p.Hv) <= lib.gdn_noalloc_scratch_bytes()
    d = to_device(p)
    ref_out, ref_fin = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"])
    sub = head_slice(p, [4, 5])
    ro, rf = oracle.fwd_problem(sub)
    for out, fin in _run_twice(lib, p, d):
        assert_close("32k out vs gdn_chunk_fwd", out, bf16_to_f64(ref_out))
        assert_close("32k final_state vs gdn_chunk_fwd", fin, ref_fin.double().cpu().numpy())
        assert_close("32k out heads 4-5 vs oracle", out[:, 4:6], ro)
        assert_close("32k final_state heads 4-5 vs oracle", fin[:, 4:6], rf)


def test_noalloc_reports_device_errors():
    """cu_seqlens that decrease are only visible on the device: the call returns GDN_OK, the
    status read reports GDN_ERR_INVALID_ARG; the next valid call clears it."""
    lib = gdn.load()
    p = synth.make_problem("noalloc_bad", 903, [100, 50], 1, 2)
    d = to_device(p)
    d["cu_seqlens"] = torch.tensor([0, 120, 150], dtype=torch.int32, device="cuda")  # fine on the host side
    bad = dict(d)
    bad["cu_seqlens"] = torch.tensor([0, 160, 150], dtype=torch.int32, device="cuda")  # decreasing: device-side error
    out = torch.zeros((p.T, 2, 128), dtype=torch.bfloat16, device="cuda")
    fin = torch.zeros((2, 2, 128, 128), dtype=torch.float32, device="cuda")
    assert _call_noalloc(lib, bad, 2, p.T, 1, 2, out, fin) == gdn.GDN_OK
    assert _status(lib) == gdn.GDN_ERR_INVALID_ARG
    assert _call_noalloc(lib, d, 2, p.T, 1, 2, out, fin) == gdn.GDN_OK
    assert _status(lib) == gdn.GDN_OK


def test_noalloc_rejects_problems_beyond_the_array():
    """A problem just over the array's size is refused before anything runs. Its tensors are real
    and of full size, so that even a launch would stay inside them."""
    lib = gdn.load()
    cap = lib.gdn_noalloc_scratch_bytes()
    Hk, Hv = 2, 8
    T = 32768
    while gdn.fwd_workspace_size(1, T, Hk, Hv) <= cap:
        T += 2048
    assert gdn.fwd_workspace_size(1, T - 2048, Hk, Hv) <= cap < gdn.fwd_workspace_size(1, T, Hk, Hv)
    dev = "cuda"
    d = dict(q=torch.zeros((T, Hk, 128), dtype=torch.bfloat16, device=dev),
             k=torch.zeros((T, Hk, 128), dtype=torch.bfloat16, device=dev),
             v=torch.zeros((T, Hv, 128), dtype=torch.bfloat16, device=dev),
             g=torch.zeros((T, Hv), dtype=torch.float32, device=dev),
             beta=torch.zeros((T, Hv), dtype=torch.float32, device=dev),
             cu_seqlens=torch.tensor([0, T], dtype=torch.int32, device=dev))
    out = torch.full((T, Hv, 128), 3.0, dtype=torch.bfloat16, device=dev)
    fin = torch.full((1, Hv, 128, 128), 3.0, dtype=torch.float32, device=dev)
    rc = _call_noalloc(lib, d, 1, T, Hk, Hv, out, fin)
    assert rc == gdn.GDN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 3.0).all()) and bool((fin == 3.0).all())
