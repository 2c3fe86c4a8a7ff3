"""Chunked Gated DeltaNet over packed varlen batches on GB300 (sm_103a).

A thin binding over the C ABI declared in include/gdn.h: argument marshalling
only. Every step of the computation runs in the CUDA library
`_build/libgdn_gb300.so`; if that library is missing, every call raises.
PyTorch is used for device memory and streams.

    import linear_attention_varlen_gb300 as gdn
    out, final_state = gdn.chunk_fwd(q, k, v, g, beta, cu_seqlens)
    grads = gdn.chunk_bwd(q, k, v, g, beta, cu_seqlens, dout)
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libgdn_gb300.so")

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA, GDN_ERR_TIMEOUT, GDN_ERR_WORKSPACE = 0, -1, -2, -3, -4, -5
MODE_EXACT, MODE_TRUNCATE = 0, 1
HEAD_DIM = 128
CHUNK = 64

# Every symbol include/gdn.h declares.
EXPORTS = ("gdn_default_options", "gdn_fwd_workspace_size", "gdn_bwd_workspace_size", "gdn_chunk_fwd",
           "gdn_chunk_bwd", "gdn_workspace_status", "gdn_status_string", "gdn_plan_host", "gdn_chunk_fwd_noalloc",
           "gdn_noalloc_scratch_bytes", "gdn_noalloc_status", "gdn_fwd_check_args", "gdn_bwd_check_args",
           "gdn_decode_step", "gdn_conv_workspace_size", "gdn_conv_fwd", "gdn_conv_bwd")


class GdnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class COptions(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("trunc_log_threshold", ctypes.c_float),
                ("segment_chunks", ctypes.c_int32), ("scale", ctypes.c_float), ("flags", ctypes.c_int32),
                ("stage_events", ctypes.c_void_p), ("flag_wait_us", ctypes.c_int32)]


NUM_STAGES = 11
(STAGE_PLAN, STAGE_KKT_SOLVE, STAGE_SPLIT, STAGE_CHAIN, STAGE_REV_CHAIN, STAGE_GRADS, STAGE_DINIT, STAGE_DQ,
 STAGE_OUT, STAGE_L2NORM, STAGE_L2NORM_BWD) = range(11)
FLAG_SAVE_FOR_BWD = 1  # forward of a training step: keep the records for the backward
FLAG_REUSE_FWD = 2     # backward: use the records of a FLAG_SAVE_FOR_BWD forward instead of recomputing
FLAG_TEST_WITHHOLD_FORK = 4  # forward, tests of the bounded waits only: forked documents never get their start
FLAG_L2NORM_QK = 8     # q and k come unnormalised: the library scales each row to unit L2 norm (both directions)
FLAG_FP16_INPUTS = 16  # q, k, v (and dout) are fp16; set by the calls below when the tensors are float16


@dataclass
class Options:
    """Mirror of gdn_options. mode: "exact" (default) or "truncate". save_for_backward (forward) and
    reuse_forward (backward) set the two gdn_flags of a training step that shares one workspace."""
    mode: str = "exact"
    trunc_log_threshold: float = -10.0
    segment_chunks: int = 0
    scale: float = 1.0
    stage_events: Optional[object] = None  # optional list of 2 * NUM_STAGES timing torch.cuda.Event (or None)
    save_for_backward: bool = False
    reuse_forward: bool = False
    l2norm_qk: bool = False          # q and k unnormalised: normalise each row first (forward and backward)
    fp16_inputs: bool = False        # q, k, v (and dout) in fp16 (the tensor calls below set it from the dtype)
    flag_wait_us: int = 0            # limit of a wait for another item's published state (0 = about 2 s)
    test_withhold_fork: bool = False  # tests only: make the waits of forked documents run out

    def c(self) -> COptions:
        m = {"exact": MODE_EXACT, "truncate": MODE_TRUNCATE}[self.mode]
        ev = None
        if self.stage_events is not None:
            # None entries are not recorded (each recorded event costs a few microseconds of stream time)
            handles = [0 if e is None else int(e.cuda_event) for e in self.stage_events]
            given = [e for e in self.stage_events if e is not None]
            if len(handles) != 2 * NUM_STAGES or not all(int(e.cuda_event) for e in given):
                raise ValueError("stage_events: 2 * NUM_STAGES entries, each None or a recorded timing event")
            self._ev_array = (ctypes.c_void_p * len(handles))(*handles)
            ev = ctypes.cast(self._ev_array, ctypes.c_void_p)
        flags = ((FLAG_SAVE_FOR_BWD if self.save_for_backward else 0) | (FLAG_REUSE_FWD if self.reuse_forward else 0)
                 | (FLAG_TEST_WITHHOLD_FORK if self.test_withhold_fork else 0)
                 | (FLAG_L2NORM_QK if self.l2norm_qk else 0)
                 | (FLAG_FP16_INPUTS if self.fp16_inputs else 0))
        return COptions(m, float(self.trunc_log_threshold), int(self.segment_chunks), float(self.scale), flags, ev,
                        int(self.flag_wait_us))


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return LIB_PATH


def load(path: Optional[str] = None):
    """Open the compiled library (no fallback: raises if it is missing) and declare signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"GDN CUDA library not built: {p} is missing (run linear_attention_varlen_gb300.build)")
        lib = ctypes.CDLL(p)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        OP = ctypes.POINTER(COptions)
        lib.gdn_default_options.argtypes = [OP]
        lib.gdn_default_options.restype = None
        lib.gdn_fwd_workspace_size.argtypes = [I, I, I, I, OP]
        lib.gdn_fwd_workspace_size.restype = Z
        lib.gdn_bwd_workspace_size.argtypes = [I, I, I, I, OP]
        lib.gdn_bwd_workspace_size.restype = Z
        lib.gdn_chunk_fwd.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, I, P, P, P, Z, OP, P]
        lib.gdn_chunk_fwd.restype = I
        lib.gdn_chunk_bwd.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, I, P, P, P, P, P, P, P, P, P, Z, OP, P]
        lib.gdn_chunk_bwd.restype = I
        lib.gdn_workspace_status.argtypes = [P, P]
        lib.gdn_workspace_status.restype = I
        lib.gdn_status_string.argtypes = [I]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_plan_host.argtypes = [P, I, I, I, P, I, OP, I, P, P, P, I, P, I, P]
        lib.gdn_plan_host.restype = I
        lib.gdn_chunk_fwd_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, I, P, P, OP, P]
        lib.gdn_chunk_fwd_noalloc.restype = I
        lib.gdn_noalloc_scratch_bytes.argtypes = []
        lib.gdn_noalloc_scratch_bytes.restype = Z
        lib.gdn_noalloc_status.argtypes = [I, P]
        lib.gdn_noalloc_status.restype = I
        lib.gdn_fwd_check_args.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, I, P, P, P, Z, OP]
        lib.gdn_fwd_check_args.restype = I
        lib.gdn_bwd_check_args.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, I, P, P, P, P, P, P, P, P, P, Z, OP]
        lib.gdn_bwd_check_args.restype = I
        lib.gdn_decode_step.argtypes = [P, P, P, P, P, I, I, I, I, P, P, I, P, P, OP, P]
        lib.gdn_decode_step.restype = I
        lib.gdn_conv_workspace_size.argtypes = [I, I, I, I]
        lib.gdn_conv_workspace_size.restype = Z
        lib.gdn_conv_fwd.argtypes = [P, P, P, P, I, I, I, P, P, I, P, P, P, Z, P]
        lib.gdn_conv_fwd.restype = I
        lib.gdn_conv_bwd.argtypes = [P, P, P, P, I, I, I, P, P, I, P, P, P, P, P, P, P, Z, P]
        lib.gdn_conv_bwd.restype = I
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load().gdn_status_string(int(status)).decode()
    except RuntimeError:
        return {0: "GDN_OK", -1: "GDN_ERR_INVALID_ARG", -2: "GDN_ERR_UNSUPPORTED", -3: "GDN_ERR_CUDA",
                -4: "GDN_ERR_TIMEOUT", -5: "GDN_ERR_WORKSPACE"}.get(int(status), "GDN_ERR_UNKNOWN")


def _opts(options: Optional[Options]) -> COptions:
    return (options or Options()).c()


def _half_dtype(q):
    """bf16 or fp16 inputs: the dtype of q decides, k and v (and dout) must match it."""
    torch = _torch()
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q: expected a bfloat16 or float16 tensor")
    return q.dtype


def _with_dtype(options: Optional[Options], half) -> Options:
    import dataclasses
    torch = _torch()
    base = options or Options()
    return dataclasses.replace(base, fp16_inputs=(half == torch.float16))


def fwd_workspace_size(N: int, T: int, H_k: int, H_v: int, options: Optional[Options] = None) -> int:
    o = _opts(options)
    return int(load().gdn_fwd_workspace_size(N, T, H_k, H_v, ctypes.byref(o)))


def bwd_workspace_size(N: int, T: int, H_k: int, H_v: int, options: Optional[Options] = None) -> int:
    o = _opts(options)
    return int(load().gdn_bwd_workspace_size(N, T, H_k, H_v, ctypes.byref(o)))


def plan_host(cu_seqlens, H_v: int, init_idx=None, n_init: int = 0, options: Optional[Options] = None,
              num_sms: int = 152):
    """Run the exported host planner on host arrays; returns (chunks [n,3], segments [s,4], seg_len)."""
    import numpy as np
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    N = cu.shape[0] - 1
    T = int(cu[-1])
    ii = None if init_idx is None else np.ascontiguousarray(init_idx, dtype=np.int32)
    mc = T // CHUNK + N + 1
    ms = mc + N + 1
    cs, ct, cl = (np.zeros(mc, np.int32) for _ in range(3))
    si = np.zeros(4 * ms, np.int32)
    cnt = np.zeros(3, np.int32)
    o = _opts(options)
    ptr = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    rc = load().gdn_plan_host(ptr(cu), N, T, H_v, ptr(ii), n_init, ctypes.byref(o), num_sms, ptr(cs), ptr(ct),
                              ptr(cl), mc, ptr(si), ms, ptr(cnt))
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_plan_host")
    nc, ns, L = int(cnt[0]), int(cnt[1]), int(cnt[2])
    chunks = np.stack([cs[:nc], ct[:nc], cl[:nc]], axis=1)
    return chunks, si[:4 * ns].reshape(ns, 4), L


# ----------------------------------------------------------------------------- torch-facing calls


def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(t, name, dtype, shape=None):
    torch = _torch()
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def chunk_fwd(q, k, v, g, beta, cu_seqlens, init_idx=None, initial_state=None, options: Optional[Options] = None,
              out=None, final_state=None, workspace=None, stream=None):
    """Forward over a packed batch. Shapes: q, k [T, Hk, 128] bf16; v [T, Hv, 128] bf16;
    g, beta [T, Hv] fp32; cu_seqlens [N+1] int32 (device); init_idx [N] int32 or None;
    initial_state [n_init, Hv, 128, 128] fp32 or None. Returns (out, final_state).
    With options.save_for_backward the workspace (allocated here when not given, of the backward's
    size) keeps the records for chunk_bwd(..., options with reuse_forward, workspace=the same)."""
    torch = _torch()
    T, Hk, D = q.shape
    Hv = v.shape[1]
    N = cu_seqlens.shape[0] - 1
    half = _half_dtype(q)
    options = _with_dtype(options, half)
    _check(q, "q", half, (T, Hk, D))
    _check(k, "k", half, (T, Hk, D))
    _check(v, "v", half, (T, Hv, D))
    _check(g, "g", torch.float32, (T, Hv))
    _check(beta, "beta", torch.float32, (T, Hv))
    _check(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,))
    n_init = 0
    if initial_state is not None:
        _check(initial_state, "initial_state", torch.float32)
        n_init = initial_state.shape[0]
    if init_idx is not None:
        _check(init_idx, "init_idx", torch.int32, (N,))
    dev = q.device
    if out is None:
        out = torch.empty((T, Hv, D), dtype=torch.bfloat16, device=dev)
    if final_state is None:
        final_state = torch.empty((N, Hv, D, D), dtype=torch.float32, device=dev)
    o = _opts(options)
    need = int(load().gdn_fwd_workspace_size(N, T, Hk, Hv, ctypes.byref(o)))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    rc = load().gdn_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, Hk, Hv, D,
                              _ptr(init_idx), _ptr(initial_state), n_init, _ptr(out), _ptr(final_state),
                              _ptr(workspace), workspace.numel(), ctypes.byref(o), _stream_handle(stream))
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_chunk_fwd")
    return out, final_state


def chunk_bwd(q, k, v, g, beta, cu_seqlens, dout, dfinal_state=None, init_idx=None, initial_state=None,
              options: Optional[Options] = None, workspace=None, stream=None, grads=None):
    """Backward. Returns dict of fp32 gradients dq, dk, dv, dg, dbeta and dinit (None without a pool).
    With options.reuse_forward, `workspace` must be the one a save_for_backward forward of the same
    inputs used. `grads` may hold preallocated fp32 outputs (keys dq, dk, dv, dg, dbeta, dinit)."""
    torch = _torch()
    if options is not None and options.reuse_forward and workspace is None:
        raise ValueError("reuse_forward needs the workspace of the save_for_backward forward")
    T, Hk, D = q.shape
    Hv = v.shape[1]
    N = cu_seqlens.shape[0] - 1
    half = _half_dtype(q)
    options = _with_dtype(options, half)
    _check(q, "q", half, (T, Hk, D))
    _check(k, "k", half, (T, Hk, D))
    _check(v, "v", half, (T, Hv, D))
    _check(dout, "dout", half, (T, Hv, D))
    if dfinal_state is not None:
        _check(dfinal_state, "dfinal_state", torch.float32, (N, Hv, D, D))
    n_init = 0 if initial_state is None else initial_state.shape[0]
    dev = q.device
    grads = grads or {}
    f32 = torch.float32

    def out_buf(key, shape):
        t = grads.get(key)
        if t is None:
            return torch.empty(shape, dtype=f32, device=dev)
        return _check(t, key, f32, shape)
    dq = out_buf("dq", q.shape)
    dk = out_buf("dk", k.shape)
    dv = out_buf("dv", v.shape)
    dg = out_buf("dg", (T, Hv))
    db = out_buf("dbeta", (T, Hv))
    dinit = out_buf("dinit", initial_state.shape) if n_init > 0 else None
    o = _opts(options)
    need = int(load().gdn_bwd_workspace_size(N, T, Hk, Hv, ctypes.byref(o)))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    rc = load().gdn_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, Hk, Hv, D,
                              _ptr(init_idx), _ptr(initial_state), n_init, _ptr(dout), _ptr(dfinal_state),
                              _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(db), _ptr(dinit), _ptr(workspace),
                              workspace.numel(), ctypes.byref(o), _stream_handle(stream))
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_chunk_bwd")
    return dict(dq=dq, dk=dk, dv=dv, dg=dg, dbeta=db, dinit=dinit)


def decode_step(q, k, v, g, beta, state_pool, state_idx, options: Optional[Options] = None, out=None, status=None,
                stream=None):
    """One decode token per sequence, in place on the state pool. Shapes: q, k [B, Hk, 128] bf16;
    v [B, Hv, 128] bf16; g, beta [B, Hv] fp32; state_pool [n_pool, Hv, 128, 128] fp32 (updated);
    state_idx [B] int32 (distinct entries of the pool). Returns out [B, Hv, 128] bf16. `status`: an
    optional int32 device tensor of one element that receives GDN_ERR_INVALID_ARG for out-of-range
    indices (not cleared here)."""
    torch = _torch()
    B, Hk, D = q.shape
    Hv = v.shape[1]
    half = _half_dtype(q)
    options = _with_dtype(options, half)
    _check(q, "q", half, (B, Hk, D))
    _check(k, "k", half, (B, Hk, D))
    _check(v, "v", half, (B, Hv, D))
    _check(g, "g", torch.float32, (B, Hv))
    _check(beta, "beta", torch.float32, (B, Hv))
    _check(state_idx, "state_idx", torch.int32, (B,))
    _check(state_pool, "state_pool", torch.float32)
    if state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (Hv, D, D):
        raise ValueError("state_pool: expected [n_pool, Hv, 128, 128]")
    if status is not None:
        _check(status, "status", torch.int32, (1,))
    if out is None:
        out = torch.empty((B, Hv, D), dtype=torch.bfloat16, device=q.device)
    o = _opts(options)
    rc = load().gdn_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), B, Hk, Hv, D, _ptr(state_idx),
                                _ptr(state_pool), state_pool.shape[0], _ptr(out), _ptr(status), ctypes.byref(o),
                                _stream_handle(stream))
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_decode_step")
    return out


def conv_workspace_size(N: int, T: int, C: int, backward: bool = False) -> int:
    return int(load().gdn_conv_workspace_size(N, T, C, 1 if backward else 0))


def conv_fwd(x, w, cu_seqlens, bias=None, init_idx=None, conv_init=None, y=None, final_tail=None, workspace=None,
             stream=None):
    """Width-4 causal convolution over packed documents. x [T, C] bf16; w [C, 4] fp32; bias [C] fp32 or
    None; cu_seqlens [N+1] int32; init_idx [N] int32 or None; conv_init [n_init, 3, C] bf16 or None.
    Returns (y [T, C] bf16, final_tail [N, 3, C] bf16)."""
    torch = _torch()
    T, C = x.shape
    N = cu_seqlens.shape[0] - 1
    _check(x, "x", torch.bfloat16, (T, C))
    _check(w, "w", torch.float32, (C, 4))
    _check(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,))
    if bias is not None:
        _check(bias, "bias", torch.float32, (C,))
    if init_idx is not None:
        _check(init_idx, "init_idx", torch.int32, (N,))
    n_init = 0
    if conv_init is not None:
        _check(conv_init, "conv_init", torch.bfloat16)
        n_init = conv_init.shape[0]
    if y is None:
        y = torch.empty((T, C), dtype=torch.bfloat16, device=x.device)
    if final_tail is None:
        final_tail = torch.empty((N, 3, C), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = torch.empty(conv_workspace_size(N, T, C), dtype=torch.uint8, device=x.device)
    rc = load().gdn_conv_fwd(_ptr(x), _ptr(w), _ptr(bias), _ptr(cu_seqlens), N, T, C, _ptr(init_idx), _ptr(conv_init),
                             n_init, _ptr(y), _ptr(final_tail), _ptr(workspace), workspace.numel(),
                             _stream_handle(stream))
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_conv_fwd")
    return y, final_tail


def conv_bwd(x, w, cu_seqlens, dy, bias=None, init_idx=None, conv_init=None, dfinal_tail=None, workspace=None,
             stream=None):
    """Backward of conv_fwd. Returns dict dx [T, C], dw [C, 4], dbias [C] (None without bias),
    dconv_init [n_init, 3, C] (None without a pool), all fp32."""
    torch = _torch()
    T, C = x.shape
    N = cu_seqlens.shape[0] - 1
    _check(dy, "dy", torch.bfloat16, (T, C))
    if dfinal_tail is not None:
        _check(dfinal_tail, "dfinal_tail", torch.float32, (N, 3, C))
    n_init = 0 if conv_init is None else conv_init.shape[0]
    f32 = dict(dtype=torch.float32, device=x.device)
    dx = torch.empty((T, C), **f32)
    dw = torch.empty((C, 4), **f32)
    dbias = torch.empty((C,), **f32) if bias is not None else None
    dci = torch.empty((n_init, 3, C), **f32) if n_init > 0 else None
    if workspace is None:
        workspace = torch.empty(conv_workspace_size(N, T, C, True), dtype=torch.uint8, device=x.device)
    rc = load().gdn_conv_bwd(_ptr(x), _ptr(w), _ptr(bias), _ptr(cu_seqlens), N, T, C, _ptr(init_idx), _ptr(conv_init),
                             n_init, _ptr(dy), _ptr(dfinal_tail), _ptr(dx), _ptr(dw), _ptr(dbias), _ptr(dci),
                             _ptr(workspace), workspace.numel(), _stream_handle(stream))
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_conv_bwd")
    return dict(dx=dx, dw=dw, dbias=dbias, dconv_init=dci)


def workspace_status(workspace, stream=None) -> int:
    """Device status word of the last call that used `workspace` (synchronises the stream)."""
    return int(load().gdn_workspace_status(_ptr(workspace), _stream_handle(stream)))
