"""Host-side argument checks of the C ABI on a machine with a GPU, through the exported check
functions (gdn_fwd_check_args / gdn_bwd_check_args run every check the entry points make before
their first launch, and launch nothing): every pointer must be device memory of the workspace's
GPU, so a host or pinned-host buffer among device buffers is refused without any kernel ever
seeing it; a short workspace is reported; and no entry point changes the caller's current
device."""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import linear_attention_varlen_gb300 as gdn  # noqa: E402

P = ctypes.c_void_p


def _p(x):
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        return P(x.ctypes.data)
    return P(x.data_ptr())


@pytest.fixture(scope="module")
def setup():
    lib = gdn.load()
    p = synth.make_problem("abi", 5, [70, 30], 1, 2, with_dout=True)
    d = synth.to_device(p)
    T, N = p.T, p.N
    out = torch.empty((T, 2, 128), dtype=torch.bfloat16, device="cuda")
    fin = torch.empty((N, 2, 128, 128), dtype=torch.float32, device="cuda")
    need_f = gdn.fwd_workspace_size(N, T, 1, 2)
    need_b = gdn.bwd_workspace_size(N, T, 1, 2)
    ws = torch.empty(max(need_f, need_b), dtype=torch.uint8, device="cuda")
    grads = {k: torch.empty(s, dtype=torch.float32, device="cuda") for k, s in
             dict(dq=(T, 1, 128), dk=(T, 1, 128), dv=(T, 2, 128), dg=(T, 2), dbeta=(T, 2)).items()}
    return lib, p, d, out, fin, ws, need_f, need_b, grads


def fwd_check(lib, p, t, ws_bytes, opts=None):
    o = (opts or gdn.Options()).c()
    return lib.gdn_fwd_check_args(_p(t["q"]), _p(t["k"]), _p(t["v"]), _p(t["g"]), _p(t["beta"]), _p(t["cu"]), p.N,
                                  p.T, 1, 2, 128, None, None, 0, _p(t["out"]), _p(t["fin"]), _p(t["ws"]), ws_bytes,
                                  ctypes.byref(o))


def bwd_check(lib, p, t, ws_bytes):
    o = gdn.Options().c()
    return lib.gdn_bwd_check_args(_p(t["q"]), _p(t["k"]), _p(t["v"]), _p(t["g"]), _p(t["beta"]), _p(t["cu"]), p.N,
                                  p.T, 1, 2, 128, None, None, 0, _p(t["dout"]), None, _p(t["dq"]), _p(t["dk"]),
                                  _p(t["dv"]), _p(t["dg"]), _p(t["dbeta"]), None, _p(t["ws"]), ws_bytes,
                                  ctypes.byref(o))


def tensors(d, out, fin, ws, grads):
    t = dict(q=d["q"], k=d["k"], v=d["v"], g=d["g"], beta=d["beta"], cu=d["cu_seqlens"], out=out, fin=fin, ws=ws,
             dout=d["dout"])
    t.update(grads)
    return t


def test_all_device_buffers_pass(setup):
    lib, p, d, out, fin, ws, need_f, need_b, grads = setup
    t = tensors(d, out, fin, ws, grads)
    assert fwd_check(lib, p, t, need_f) == gdn.GDN_OK
    assert bwd_check(lib, p, t, need_b) == gdn.GDN_OK
    assert fwd_check(lib, p, t, need_f - 256) == gdn.GDN_ERR_WORKSPACE
    assert bwd_check(lib, p, t, need_b - 256) == gdn.GDN_ERR_WORKSPACE


@pytest.mark.parametrize("name", ["q", "k", "v", "g", "beta", "cu", "out", "fin"])
@pytest.mark.parametrize("kind", ["host", "pinned"])
def test_one_host_buffer_among_device_buffers_is_refused(setup, name, kind):
    lib, p, d, out, fin, ws, need_f, need_b, grads = setup
    t = tensors(d, out, fin, ws, grads)
    src = t[name]
    if kind == "host":
        t[name] = np.zeros(src.numel() * src.element_size() // 4 + 8, dtype=np.float32)
        assert t[name].ctypes.data % 16 == 0
    else:
        t[name] = torch.empty(src.shape, dtype=src.dtype, pin_memory=True)
    assert fwd_check(lib, p, t, need_f) == gdn.GDN_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["dout", "dq", "dk", "dv", "dg", "dbeta", "ws"])
def test_backward_host_buffer_is_refused(setup, name):
    lib, p, d, out, fin, ws, need_f, need_b, grads = setup
    t = tensors(d, out, fin, ws, grads)
    src = t[name]
    t[name] = torch.empty(src.shape, dtype=src.dtype, pin_memory=True)
    assert bwd_check(lib, p, t, need_b) == gdn.GDN_ERR_INVALID_ARG


def test_entry_points_keep_the_callers_device(setup):
    lib, p, d, out, fin, ws, need_f, need_b, grads = setup
    before = torch.cuda.current_device()
    gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], out=out, final_state=fin, workspace=ws)
    gdn.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["dout"], workspace=ws)
    torch.cuda.synchronize()
    assert gdn.workspace_status(ws) == gdn.GDN_OK
    assert torch.cuda.current_device() == before
