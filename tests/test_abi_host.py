"""Host-side checks of the C ABI (no GPU needed): the library builds and loads, it
exports every entry point include/gdn.h declares, host argument checks reject bad
calls before any launch, and the exported host planner produces the chunk and
segment maps a plain restatement of the packing rules gives (bit-exact)."""
import ctypes
import os
import re

import numpy as np
import pytest

import linear_attention_varlen_gb300 as gdn
from linear_attention_varlen_gb300 import build as gdn_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gdn_build.build()
    return gdn.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), f"missing export {n}"
    assert set(names) == set(gdn.EXPORTS)


def test_status_strings(lib):
    for code, name in [(0, "GDN_OK"), (-1, "GDN_ERR_INVALID_ARG"), (-2, "GDN_ERR_UNSUPPORTED"), (-3, "GDN_ERR_CUDA"),
                       (-4, "GDN_ERR_TIMEOUT"), (-5, "GDN_ERR_WORKSPACE"), (7, "GDN_ERR_UNKNOWN")]:
        assert gdn.status_string(code) == name


def test_default_options(lib):
    o = gdn.COptions()
    lib.gdn_default_options(ctypes.byref(o))
    assert (o.mode, o.trunc_log_threshold, o.segment_chunks, o.scale, o.flags, o.flag_wait_us) == (0, -10.0, 0, 1.0, 0, 0)
    assert o.stage_events is None


def test_workspace_size_queries(lib):
    a = gdn.fwd_workspace_size(1, 512, 2, 2)
    b = gdn.fwd_workspace_size(1, 32768, 2, 8)
    assert a > 0 and b > a
    assert gdn.fwd_workspace_size(0, 512, 2, 2) == 0          # no documents
    assert gdn.fwd_workspace_size(1, 512, 2, 3) == 0          # Hv not a multiple of Hk
    assert gdn.bwd_workspace_size(4, 65536, 2, 8) > 0


def _fwd_raw(lib, mode=0, flags=0, **kw):
    args = dict(q=1 << 20, k=1 << 20, v=1 << 20, g=1 << 20, beta=1 << 20, cu=1 << 20, N=1, T=64, Hk=1, Hv=1, D=128,
                init=None, h0=None, n_init=0, out=1 << 20, fin=1 << 20, ws=1 << 20, ws_bytes=1 << 30)
    args.update(kw)
    o = gdn.COptions(mode, -10.0, 0, 1.0, flags, None)
    P = ctypes.c_void_p
    return lib.gdn_chunk_fwd(P(args["q"]), P(args["k"]), P(args["v"]), P(args["g"]), P(args["beta"]), P(args["cu"]),
                             args["N"], args["T"], args["Hk"], args["Hv"], args["D"], P(args["init"]), P(args["h0"]),
                             args["n_init"], P(args["out"]), P(args["fin"]), P(args["ws"]), args["ws_bytes"],
                             ctypes.byref(o), None)


def test_host_argument_checks(lib):
    # every rejection below happens before the library touches the GPU
    assert _fwd_raw(lib, D=64) == gdn.GDN_ERR_UNSUPPORTED
    assert _fwd_raw(lib, N=0) == gdn.GDN_ERR_INVALID_ARG
    assert _fwd_raw(lib, Hk=2, Hv=3) == gdn.GDN_ERR_INVALID_ARG
    assert _fwd_raw(lib, q=None) == gdn.GDN_ERR_INVALID_ARG
    assert _fwd_raw(lib, cu=None) == gdn.GDN_ERR_INVALID_ARG
    assert _fwd_raw(lib, n_init=1, h0=None) == gdn.GDN_ERR_INVALID_ARG
    assert _fwd_raw(lib, q=(1 << 20) + 8) == gdn.GDN_ERR_INVALID_ARG      # 16-byte alignment
    assert _fwd_raw(lib, ws=(1 << 20) + 128) == gdn.GDN_ERR_INVALID_ARG   # 256-byte workspace alignment
    assert _fwd_raw(lib, T=-1) == gdn.GDN_ERR_INVALID_ARG


def _bwd_raw(lib, flags=0):
    P, a = ctypes.c_void_p, 1 << 20
    o = gdn.COptions(0, -10.0, 0, 1.0, flags, None)
    return lib.gdn_chunk_bwd(P(a), P(a), P(a), P(a), P(a), P(a), 1, 64, 1, 1, 128, None, None, 0, P(a), None,
                             P(a), P(a), P(a), P(a), P(a), None, P(a), 1 << 30, ctypes.byref(o), None)


def test_training_flags_host_checks(lib):
    # rejected before the library touches the GPU
    assert _fwd_raw(lib, flags=gdn.FLAG_REUSE_FWD) == gdn.GDN_ERR_INVALID_ARG       # a backward flag
    assert _fwd_raw(lib, flags=gdn.FLAG_SAVE_FOR_BWD, mode=1) == gdn.GDN_ERR_INVALID_ARG  # exact mode only
    assert _fwd_raw(lib, flags=4) == gdn.GDN_ERR_INVALID_ARG                         # unknown bit
    assert _bwd_raw(lib, flags=gdn.FLAG_SAVE_FOR_BWD) == gdn.GDN_ERR_INVALID_ARG     # a forward flag
    assert _bwd_raw(lib, flags=8) == gdn.GDN_ERR_INVALID_ARG
    # a forward that keeps its records needs the backward's workspace
    save = gdn.Options(save_for_backward=True)
    for N, T, Hk, Hv in [(1, 512, 2, 2), (1, 32768, 2, 8), (12, 16384, 2, 8)]:
        assert gdn.fwd_workspace_size(N, T, Hk, Hv, save) == gdn.bwd_workspace_size(N, T, Hk, Hv)
        assert gdn.fwd_workspace_size(N, T, Hk, Hv, save) > gdn.fwd_workspace_size(N, T, Hk, Hv)
    P = ctypes.c_void_p
    o = gdn.COptions(0, -10.0, 0, 1.0, gdn.FLAG_SAVE_FOR_BWD, None)
    assert lib.gdn_chunk_fwd_noalloc(P(1 << 20), P(1 << 20), P(1 << 20), P(1 << 20), P(1 << 20), P(1 << 20), 1, 64, 1,
                                     1, 128, None, None, 0, P(1 << 20), P(1 << 20), ctypes.byref(o),
                                     None) == gdn.GDN_ERR_INVALID_ARG


def test_reuse_needs_the_forward_workspace():
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):
        z = torch.zeros(1)
        gdn.chunk_bwd(z, z, z, z, z, z, z, options=gdn.Options(reuse_forward=True))


# ----------------------------------------------------------------------------- planner


def plan_reference(cu, Hv, init_idx, n_init, seg_override, num_sms):
    """Plain restatement of the packing rules: 64-token chunks from each document's first
    token, last chunk partial; segments of L chunks when the documents cannot fill the SMs."""
    N = len(cu) - 1
    lens = [cu[i + 1] - cu[i] for i in range(N)]
    nch = [(L + 63) // 64 for L in lens]
    total, longest = sum(nch), max(nch)
    if seg_override < 0:
        L = 0
    elif seg_override > 0:
        L = seg_override if longest > seg_override else 0
    elif N * Hv >= 2 * num_sms:
        L = 0
    else:
        L = max(4, -(-total * Hv // num_sms))
        L = L if longest > L else 0
    chunks = []
    for i in range(N):
        for c in range(nch[i]):
            t0 = cu[i] + 64 * c
            chunks.append((i, t0, min(64, cu[i + 1] - t0)))
    segs = []
    first_chunk = np.concatenate([[0], np.cumsum(nch)])
    for i in range(N):
        nseg = -(-nch[i] // L) if (L > 0 and nch[i] > L) else 1
        for k in range(nseg):
            c0 = k * L if nseg > 1 else 0
            cnt = min(L, nch[i] - c0) if nseg > 1 else nch[i]
            if k > 0:
                dep = len(segs) - 1
            else:
                x = -1 if init_idx is None else init_idx[i]
                dep = -(x - n_init) - 2 if x >= n_init else -1
            segs.append((i, int(first_chunk[i]) + c0, cnt, dep))
    return np.array(chunks, dtype=np.int32).reshape(-1, 3), np.array(segs, dtype=np.int32).reshape(-1, 4), L


CASES = [
    ([0, 512], 2, None, 0, 0),
    ([0, 1769, 5709, 6376, 16384], 8, None, 0, 0),
    ([0, 32768], 8, None, 0, 0),
    ([0, 32768], 8, None, 0, 7),
    ([0, 0, 1, 64, 65, 65, 200], 4, [-1, 0, 2, -1, 5, 3], 2, 0),
    ([0, 8192, 10000, 16000], 64, [-1, 0, 0], 0, 0),
    ([0, 100, 300, 1000], 2, [0, 0, 2], 1, 2),
    ([0, 640, 1280], 1, None, 0, -1),
]


@pytest.mark.parametrize("cu,Hv,init,n_init,seg", CASES)
def test_host_planner_matches_restatement(lib, cu, Hv, init, n_init, seg):
    opts = gdn.Options(segment_chunks=seg)
    chunks, segs, L = gdn.plan_host(cu, Hv, init, n_init, opts, num_sms=152)
    rc, rs, rL = plan_reference(cu, Hv, init, n_init, seg, 152)
    assert L == rL
    np.testing.assert_array_equal(chunks, rc)
    np.testing.assert_array_equal(segs, rs)
    # every token covered exactly once, in order
    covered = np.concatenate([np.arange(t0, t0 + n) for _, t0, n in chunks]) if len(chunks) else np.zeros(0)
    np.testing.assert_array_equal(covered, np.arange(cu[-1]))


def test_host_planner_rejects_bad_layouts(lib):
    with pytest.raises(gdn.GdnError):
        gdn.plan_host([0, 10, 5, 20], 2)         # decreasing
    with pytest.raises(gdn.GdnError):
        gdn.plan_host([0, 10, 20], 2, [-1, 3], 2)  # fork into a later document (x - n_init = 1 >= i)
    with pytest.raises(gdn.GdnError):
        gdn.plan_host([0, 10, 20], 2, [-2, -1], 0)


def test_split_layout_fills_the_sms(lib):
    """32K tokens, 8 heads, 152 SMs: segments x heads close to the SM count, floor 4 chunks."""
    _, segs, L = gdn.plan_host([0, 32768], 8, num_sms=152)
    assert L == 27 and len(segs) * 8 >= 152 - 8 and len(segs) * 8 <= 152 + 8
    _, segs, L = gdn.plan_host([0, 2048], 8, num_sms=152)
    assert L == 4


def test_stage_events_allow_skipped_entries():
    n = 2 * gdn.NUM_STAGES
    o = gdn.Options(stage_events=[None] * n).c()  # every entry skipped
    arr = ctypes.cast(o.stage_events, ctypes.POINTER(ctypes.c_void_p))
    assert all(arr[i] is None for i in range(n))
    with pytest.raises(ValueError):
        gdn.Options(stage_events=[None] * (n - 1)).c()


def test_no_cpu_fallback(lib):
    """Host memory is refused, never computed on: the binding rejects host tensors, the C ABI
    returns an error for host buffers and leaves the outputs untouched, and a missing library
    raises instead of falling back."""
    torch = pytest.importorskip("torch")
    import synth
    from tests.gpu_util import to_device
    p = synth.make_problem("host", 3, [70], 1, 2, with_dout=True)
    d = to_device(p, "cpu")
    with pytest.raises(ValueError):
        gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"])
    with pytest.raises(ValueError):
        gdn.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["dout"])
    # the C ABI on host buffers (aligned, well-formed): an argument error before any launch
    T, N = p.T, p.N
    need = gdn.fwd_workspace_size(N, T, 1, 2)
    raw = np.zeros(need + 256, dtype=np.uint8)
    ws = raw[(-raw.ctypes.data) % 256:][:need]
    out = np.full((T, 2, 128), 0x7FC0, dtype=np.uint16)
    fin = np.full((N, 2, 128, 128), 7.0, dtype=np.float32)
    o = gdn.COptions(0, -10.0, 0, 1.0, 0, None)
    P = ctypes.c_void_p
    rc = lib.gdn_chunk_fwd(P(p.q.ctypes.data), P(p.k.ctypes.data), P(p.v.ctypes.data), P(p.g.ctypes.data),
                           P(p.beta.ctypes.data), P(p.cu_seqlens.ctypes.data), N, T, 1, 2, 128, None, None, 0,
                           P(out.ctypes.data), P(fin.ctypes.data), P(ws.ctypes.data), need, ctypes.byref(o), None)
    assert rc == gdn.GDN_ERR_INVALID_ARG
    assert (out == 0x7FC0).all() and (fin == 7.0).all()
    with pytest.raises(RuntimeError):
        gdn.load("/nonexistent/libgdn_gb300.so")
