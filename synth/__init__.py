"""Seeded synthetic inputs for the chunked Gated DeltaNet path.

This module is shared by the tests, the benchmark and the smoke check, and it
feeds both the CUDA library and the fp64 oracle. It holds no part of the
method's arithmetic: it only draws random numbers, shapes them into the input
distributions and packs documents into one token buffer.

Random numbers come from a counter-based splitmix64 stream (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", 2014) turned into
normals with the Box-Muller transform. Every draw is a pure function of
(seed, stream, index), so a given seed gives the same bits on any machine
whose libm rounds log/cos/sin the same way; the tests never compare stored
values across machines, only values produced in the same process.

Input recipe (the workloads on "How to Speed Up GDN Kernels for Qwen Models",
section "The real enemy: an idle GPU", a 32K-token prefill with 8 heads per
GPU, head dimension 128; and the packed and shared-prefix layouts of "Musings
on long-context fine-tuning", section "Isolating the recurrent layers"):
  * q, k ~ N(0, 1) per element, L2-normalised per (token, head) in fp64,
    q multiplied by 1/sqrt(d_k), then rounded once to bf16 (RNE);
  * v ~ N(0, 1) rounded to bf16;
  * g = log(sigmoid(u)), u ~ N(2, 1), stored as fp32 (so g < 0);
  * beta = sigmoid(w), w ~ N(0, 1), stored as fp32;
  * dO ~ N(0, 1) rounded to bf16 (backward workloads).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1


def _mix_seed(seed: int, stream: int) -> np.uint64:
    """Derive a per-stream 64-bit key from (seed, stream) with one splitmix64 round."""
    z = (seed * 0x9E3779B97F4A7C15 + stream * 0xD1B54A32D192ED03 + 0x632BE59BD9B4E019) & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return np.uint64(z ^ (z >> 31))


def splitmix64(seed: int, stream: int, n: int) -> np.ndarray:
    """n uint64 outputs of the splitmix64 sequence keyed by (seed, stream)."""
    key = _mix_seed(seed, stream)
    with np.errstate(over="ignore"):
        z = key + (np.arange(1, n + 1, dtype=np.uint64) * _GOLDEN)
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, stream: int, n: int) -> np.ndarray:
    """n doubles in (0, 1): the top 53 bits of splitmix64, offset by half a step."""
    u = splitmix64(seed, stream, n) >> np.uint64(11)
    return (u.astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """n standard normals (fp64) by Box-Muller on pairs of uniforms."""
    m = (n + 1) // 2
    u = uniform01(seed, stream, 2 * m)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    th = 2.0 * math.pi * u[1::2]
    out = np.empty(2 * m, dtype=np.float64)
    out[0::2] = r * np.cos(th)
    out[1::2] = r * np.sin(th)
    return out[:n]


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round to bf16 (round-to-nearest-even via fp32) and return the uint16 bit patterns."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = (b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16).reshape(f.shape)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact fp32 values of bf16 bit patterns."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round to IEEE fp16 (numpy's round-to-nearest-even) and return the uint16 bit patterns."""
    return np.ascontiguousarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def f16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact fp32 values of fp16 bit patterns."""
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


_ROUND = {"bf16": to_bf16_bits, "f16": to_f16_bits}
_DECODE = {"bf16": bf16_bits_to_f32, "f16": f16_bits_to_f32}


# ----------------------------------------------------------------------------- problems


@dataclass
class Problem:
    """One packed varlen problem: token-major tensors plus the document layout.

    Layouts (T tokens, N documents):
      q, k  : bf16 (or fp16, see dtype) bits uint16 [T, Hk, Dk]
      v     : bf16 (or fp16) bits uint16 [T, Hv, Dv]
      g, beta : float32 [T, Hv]
      cu_seqlens : int32 [N + 1]
      init_idx : int32 [N] (-1 zero, 0..n_init-1 pool, n_init + j fork from document j < i) or None
      initial_state : float32 [n_init, Hv, Dk, Dv] or None
      dout : bf16 (or fp16) bits [T, Hv, Dv] or None ; dfinal : float32 [N, Hv, Dk, Dv] or None
      dtype : "bf16" or "f16", the format of q, k, v and dout
    """
    name: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    beta: np.ndarray
    cu_seqlens: np.ndarray
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    init_idx: Optional[np.ndarray] = None
    initial_state: Optional[np.ndarray] = None
    dout: Optional[np.ndarray] = None
    dfinal: Optional[np.ndarray] = None
    meta: dict = field(default_factory=dict)
    dtype: str = "bf16"

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def N(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)

    @property
    def n_init(self) -> int:
        return 0 if self.initial_state is None else int(self.initial_state.shape[0])

    def as_f64(self):
        """Exact fp64 upcasts of every input (what the oracle consumes)."""
        dec = _DECODE[self.dtype]
        d = dict(
            q=dec(self.q).astype(np.float64),
            k=dec(self.k).astype(np.float64),
            v=dec(self.v).astype(np.float64),
            g=self.g.astype(np.float64),
            beta=self.beta.astype(np.float64),
        )
        if self.initial_state is not None:
            d["initial_state"] = self.initial_state.astype(np.float64)
        if self.dout is not None:
            d["dout"] = dec(self.dout).astype(np.float64)
        if self.dfinal is not None:
            d["dfinal"] = self.dfinal.astype(np.float64)
        return d


_STREAM_Q, _STREAM_K, _STREAM_V, _STREAM_G, _STREAM_B, _STREAM_DO, _STREAM_H0, _STREAM_DHT = range(1, 9)
_STREAM_LEN = 100


def _unit_rows(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.maximum(n, 1e-30)


def make_problem(name: str, seed: int, lengths: List[int], Hk: int, Hv: int, Dk: int = 128, Dv: int = 128,
                 init_idx: Optional[List[int]] = None, n_init: int = 0, with_dout: bool = False,
                 with_dfinal: bool = False, q_scale: Optional[float] = None,
                 g_mean: float = 2.0, dtype: str = "bf16") -> Problem:
    """Draw one problem with the recipe in the module docstring.

    `g_mean` is the mean of u in g = log sigmoid(u); 2.0 is the workload value. `dtype` "f16" rounds
    q, k, v and dO to IEEE fp16 instead of bf16 (the same draws).
    Pool initial states (n_init > 0) are N(0, 1) scaled by 0.1 in fp32.
    """
    if Hv % Hk != 0:
        raise ValueError("Hv must be a multiple of Hk")
    lengths = [int(x) for x in lengths]
    T = int(sum(lengths))
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    qs = (1.0 / math.sqrt(Dk)) if q_scale is None else q_scale
    q = _unit_rows(normal(seed, _STREAM_Q, T * Hk * Dk).reshape(T, Hk, Dk)) * qs
    k = _unit_rows(normal(seed, _STREAM_K, T * Hk * Dk).reshape(T, Hk, Dk))
    v = normal(seed, _STREAM_V, T * Hv * Dv).reshape(T, Hv, Dv)
    u = normal(seed, _STREAM_G, T * Hv).reshape(T, Hv) + g_mean
    g = -np.logaddexp(0.0, -u)  # log(sigmoid(u))
    w = normal(seed, _STREAM_B, T * Hv).reshape(T, Hv)
    beta = 1.0 / (1.0 + np.exp(-w))
    rnd = _ROUND[dtype]
    p = Problem(name=name, q=rnd(q), k=rnd(k), v=rnd(v),
                g=g.astype(np.float32), beta=beta.astype(np.float32), cu_seqlens=cu,
                Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, dtype=dtype)
    if init_idx is not None:
        p.init_idx = np.asarray(init_idx, dtype=np.int32)
    if n_init > 0:
        p.initial_state = (0.1 * normal(seed, _STREAM_H0, n_init * Hv * Dk * Dv)).astype(
            np.float32).reshape(n_init, Hv, Dk, Dv)
    if with_dout:
        p.dout = rnd(normal(seed, _STREAM_DO, T * Hv * Dv).reshape(T, Hv, Dv))
    if with_dfinal:
        p.dfinal = normal(seed, _STREAM_DHT, len(lengths) * Hv * Dk * Dv).astype(
            np.float32).reshape(len(lengths), Hv, Dk, Dv)
    p.meta = dict(seed=seed, lengths=lengths)
    return p


# ----------------------------------------------------------------------------- document lengths


def lognormal_lengths(seed: int, n_docs: int, total: int, mu: float = 7.0, sigma: float = 0.8,
                      lo: int = 64, hi: int = 4096) -> List[int]:
    """Packed-document lengths: lognormal(mu, sigma) draws, each clipped to [lo, hi],
    then rescaled so they fill exactly `total` tokens.

    The draws alone rarely sum to `total`, so they are scaled by total/sum,
    rounded and clipped again, and the remainder is added or removed one token
    at a time, round-robin, without leaving [lo, hi].
    """
    if not (n_docs * lo <= total <= n_docs * hi):
        raise ValueError("total tokens cannot be met within the length bounds")
    z = normal(seed, _STREAM_LEN, n_docs)
    raw = np.clip(np.rint(np.exp(mu + sigma * z)), lo, hi)
    scaled = np.clip(np.rint(raw * (total / raw.sum())), lo, hi).astype(np.int64)
    rem = int(total - scaled.sum())
    i = 0
    while rem != 0:
        step = 1 if rem > 0 else -1
        j = i % n_docs
        if lo <= scaled[j] + step <= hi:
            scaled[j] += step
            rem -= step
        i += 1
    return [int(x) for x in scaled]


def uniform_int_lengths(seed: int, n: int, lo: int, hi: int) -> List[int]:
    """n integers uniform in [lo, hi] (inclusive)."""
    u = uniform01(seed, _STREAM_LEN + 1, n)
    return [int(lo + min(hi - lo, int(math.floor(x * (hi - lo + 1))))) for x in u]


# ----------------------------------------------------------------------------- the five workloads

SEEDS = (1001, 1002, 1003, 1004, 1005)


def workload_single(T: int = 512, Hk: int = 2, Hv: int = 2, seed: int = SEEDS[0]) -> Problem:
    """One sequence, zero initial state (T=512, Hv=Hk=2 at full size)."""
    return make_problem(f"single_T{T}_H{Hv}", seed, [T], Hk, Hv)


def workload_packed(total: int = 16384, n_docs: int = 12, Hk: int = 2, Hv: int = 8,
                    seed: int = SEEDS[1]) -> Problem:
    """Packed documents with lognormal lengths; state resets at each boundary."""
    lo, hi = 64, 4096
    if total < n_docs * lo:
        raise ValueError("too few tokens for the document count")
    hi = max(hi, -(-total // n_docs))
    lens = lognormal_lengths(seed, n_docs, total, lo=lo, hi=hi)
    return make_problem(f"packed_T{total}_N{n_docs}_H{Hv}", seed, lens, Hk, Hv)


def workload_long(T: int = 32768, Hk: int = 2, Hv: int = 8, seed: int = SEEDS[2]) -> Problem:
    """Long single-sequence prefill (T=32768, 8 value heads over 2 key heads at full size)."""
    return make_problem(f"long_T{T}_H{Hv}", seed, [T], Hk, Hv)


def workload_fork(prefix: int = 8192, n_branch: int = 16, lo: int = 2048, hi: int = 6144,
                  Hk: int = 16, Hv: int = 64, seed: int = SEEDS[3]) -> Problem:
    """Shared prefix (document 0) forked as the initial state of n_branch documents.

    init_idx = [-1, 0, 0, ...] with an empty pool: every branch starts from the
    final state of document 0 of the same call.
    """
    lens = [prefix] + uniform_int_lengths(seed, n_branch, lo, hi)
    init = [-1] + [0] * n_branch
    return make_problem(f"fork_P{prefix}_B{n_branch}_H{Hv}", seed, lens, Hk, Hv, init_idx=init)


def workload_train(n_docs: int = 4, doc_len: int = 16384, Hk: int = 2, Hv: int = 8,
                   seed: int = SEEDS[4]) -> Problem:
    """Forward + backward training step over equal-length packed documents, with dO."""
    return make_problem(f"train_{n_docs}x{doc_len}_H{Hv}", seed, [doc_len] * n_docs, Hk, Hv, with_dout=True)


# ----------------------------------------------------------------------------- device copies


def to_device(p: Problem, device="cuda"):
    """The problem's arrays as torch tensors on `device` (bf16 or fp16 bit patterns viewed as
    bfloat16 or float16, fp32 and int32 as they are): plain copies, no arithmetic."""
    import torch
    half = torch.bfloat16 if p.dtype == "bf16" else torch.float16
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(half).to(device)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)
    d = dict(q=bf(p.q), k=bf(p.k), v=bf(p.v), g=f32(p.g), beta=f32(p.beta),
             cu_seqlens=torch.from_numpy(p.cu_seqlens.astype(np.int32)).to(device))
    d["init_idx"] = None if p.init_idx is None else torch.from_numpy(p.init_idx.astype(np.int32)).to(device)
    d["initial_state"] = None if p.initial_state is None else f32(p.initial_state)
    if p.dout is not None:
        d["dout"] = bf(p.dout)
    if p.dfinal is not None:
        d["dfinal_state"] = f32(p.dfinal)
    return d
