"""fp64 oracle for the gated delta rule over packed varlen batches.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
benchmark's CPU-baseline leg. The product path never imports it. The width-4
causal convolution's oracle is oracle/conv.py (numpy, fp64).

`gdn_oracle.cpp` holds the token-by-token recurrence and its hand-written
reverse mode (fp64, std::thread); this module compiles it with the host C++
compiler into `_build/libgdn_oracle.so` and wraps it with ctypes.
See the C++ file for the definition and the passages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (host C++ compiler, no GPU)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def load_library(path: str):
    """Open a compiled oracle library at `path` and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    lib.gdn_oracle_fwd.argtypes = [P, P, P, P, P, P, i32, i64, i32, i32, i32, i32, P, P, i32, P, P, i32]
    lib.gdn_oracle_fwd.restype = ctypes.c_int
    lib.gdn_oracle_bwd.argtypes = [P, P, P, P, P, P, i32, i64, i32, i32, i32, i32, P, P, i32,
                                   P, P, P, P, P, P, P, P, i32]
    lib.gdn_oracle_bwd.restype = ctypes.c_int
    lib.gdn_oracle_hw_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def hw_threads() -> int:
    return int(_load().gdn_oracle_hw_threads())


def _f64(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.float64)


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def _check_shapes(q, k, v, g, beta, cu):
    T, Hk, Dk = q.shape
    assert k.shape == (T, Hk, Dk), "k shape"
    Tv, Hv, Dv = v.shape
    assert Tv == T and g.shape == (T, Hv) and beta.shape == (T, Hv), "v/g/beta shape"
    assert cu.ndim == 1 and cu.shape[0] >= 1
    return T, Hk, Dk, Hv, Dv


def fwd(q, k, v, g, beta, cu_seqlens, init_idx=None, initial_state=None, threads: Optional[int] = None):
    """Forward recurrence. Returns (out [T,Hv,Dv], final_state [N,Hv,Dk,Dv]) in fp64."""
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T, Hk, Dk, Hv, Dv = _check_shapes(q, k, v, g, beta, cu)
    N = cu.shape[0] - 1
    ii = None if init_idx is None else np.ascontiguousarray(init_idx, dtype=np.int32)
    h0 = _f64(initial_state)
    n_init = 0 if h0 is None else h0.shape[0]
    out = np.zeros((T, Hv, Dv))
    fin = np.zeros((N, Hv, Dk, Dv))
    nt = threads if threads is not None else (os.cpu_count() or 1)
    rc = _load().gdn_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu), N, T, Hk, Hv, Dk, Dv,
                                _ptr(ii), _ptr(h0), n_init, _ptr(out), _ptr(fin), nt)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return out, fin


def bwd(q, k, v, g, beta, cu_seqlens, dout, dfinal=None, init_idx=None, initial_state=None,
        threads: Optional[int] = None):
    """Reverse mode. Returns dict dq, dk [T,Hk,Dk]; dv [T,Hv,Dv]; dg, dbeta [T,Hv];
    dinit [n_init,Hv,Dk,Dv] (None without a pool)."""
    q, k, v, g, beta, dout, dfinal = map(_f64, (q, k, v, g, beta, dout, dfinal))
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T, Hk, Dk, Hv, Dv = _check_shapes(q, k, v, g, beta, cu)
    N = cu.shape[0] - 1
    ii = None if init_idx is None else np.ascontiguousarray(init_idx, dtype=np.int32)
    h0 = _f64(initial_state)
    n_init = 0 if h0 is None else h0.shape[0]
    dq = np.zeros((T, Hk, Dk))
    dk = np.zeros((T, Hk, Dk))
    dv = np.zeros((T, Hv, Dv))
    dg = np.zeros((T, Hv))
    db = np.zeros((T, Hv))
    dh0 = np.zeros((n_init, Hv, Dk, Dv)) if n_init > 0 else None
    nt = threads if threads is not None else (os.cpu_count() or 1)
    rc = _load().gdn_oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu), N, T, Hk, Hv, Dk, Dv,
                                _ptr(ii), _ptr(h0), n_init, _ptr(dout), _ptr(dfinal), _ptr(dq), _ptr(dk), _ptr(dv),
                                _ptr(dg), _ptr(db), _ptr(dh0), nt)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return dict(dq=dq, dk=dk, dv=dv, dg=dg, dbeta=db, dinit=dh0)


def fwd_problem(p, threads: Optional[int] = None):
    """Run the forward on a synth.Problem (exact fp64 upcasts of its inputs)."""
    f = p.as_f64()
    return fwd(f["q"], f["k"], f["v"], f["g"], f["beta"], p.cu_seqlens, p.init_idx, f.get("initial_state"),
               threads=threads)


def bwd_problem(p, threads: Optional[int] = None):
    f = p.as_f64()
    return bwd(f["q"], f["k"], f["v"], f["g"], f["beta"], p.cu_seqlens, f["dout"], f.get("dfinal"), p.init_idx,
               f.get("initial_state"), threads=threads)


# ----------------------------------------------------------------------------- q / k normalisation

L2NORM_EPS = 1e-6


def l2norm_rows(x, eps: float = L2NORM_EPS):
    """y = x / sqrt(x . x + eps) over the last axis, in fp64: the unit-norm scaling of each (token,
    head) row of q and k that the model applies right before the recurrence ("Musings on long-context
    fine-tuning", section "Triton autotuning in the first backward pass"; the workloads' recipe
    normalises q and k per token and head). eps guards a zero row."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def l2norm_rows_bwd(x, dy, eps: float = L2NORM_EPS):
    """Gradient with respect to x of sum(dy * l2norm_rows(x)), in fp64. With r = (x . x + eps)^{-1/2}
    and y = r x, the derivative of y is r I - r^3 x x^T, so dx = r dy - r^3 (x . dy) x = r (dy - (y . dy) y)."""
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    r = 1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)
    y = r * x
    return r * (dy - np.sum(y * dy, axis=-1, keepdims=True) * y)

