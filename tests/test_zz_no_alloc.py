"""The allocation-free forward entry point (gdn_chunk_fwd_noalloc), called through the C ABI.

It exists for callers that cannot allocate device memory themselves (a host program without a
device allocator, or a plugin inside a framework whose pool owns all device memory): it takes no
workspace and uses a fixed array compiled into the library. Its output must match gdn_chunk_fwd
(which takes a caller workspace) within the tolerances the other GPU tests use, on two calls in a
row (the second call finds the first call's leftovers in the shared array).

This file sorts last so that a failure here does not stop the rest of the GPU suite."""
import ctypes

import numpy as np
import pytest

import synth
from tests.gpu_util import assert_close, bf16_to_f64, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import linear_attention_varlen_gb300 as gdn  # noqa: E402


def _call_noalloc(lib, d, p, out, fin):
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    o = gdn.Options().c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    n_init = 0 if d["initial_state"] is None else d["initial_state"].shape[0]
    return lib.gdn_chunk_fwd_noalloc(P(d["q"]), P(d["k"]), P(d["v"]), P(d["g"]), P(d["beta"]), P(d["cu_seqlens"]),
                                     p.N, p.T, p.Hk, p.Hv, 128, P(d["init_idx"]), P(d["initial_state"]), n_init,
                                     P(out), P(fin), ctypes.byref(o), stream)


def test_noalloc_forward_matches_workspace_forward_twice():
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
        assert np.abs(bf16_to_f64(ref_out)).max() > 0
        for _ in range(2):
            out = torch.full((p.T, p.Hv, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
            fin = torch.full((p.N, p.Hv, 128, 128), float("nan"), dtype=torch.float32, device="cuda")
            rc = _call_noalloc(lib, d, p, out, fin)
            assert rc == gdn.GDN_OK, gdn.status_string(rc)
            torch.cuda.synchronize()
            assert_close(f"{p.name} out", bf16_to_f64(out), bf16_to_f64(ref_out))
            assert_close(f"{p.name} final_state", fin.double().cpu().numpy(), ref_fin.double().cpu().numpy())


def test_noalloc_rejects_problems_beyond_the_array():
    lib = gdn.load()
    cap = lib.gdn_noalloc_scratch_bytes()
    T = 1 << 21  # 2M tokens x 8 heads needs far more scratch than the array holds
    assert gdn.fwd_workspace_size(1, T, 2, 8) > cap
    d = {k: torch.zeros(1, dtype=torch.int32, device="cuda") for k in ("q", "k", "v", "g", "beta", "cu_seqlens")}
    d["init_idx"] = None
    d["initial_state"] = None
    out = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    fin = torch.zeros(1, dtype=torch.float32, device="cuda")

    class P:
        N, T_, Hk, Hv = 1, T, 2, 8
    P.T = T
    rc = _call_noalloc(lib, d, P, out, fin)
    assert rc == gdn.GDN_ERR_WORKSPACE
