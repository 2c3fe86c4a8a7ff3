"""fp64 oracle of the width-4 causal convolution over packed documents.

TEST INFRASTRUCTURE ONLY (like the rest of oracle/): imported by tests/ and the benchmark's CPU
baseline; the product path never imports it.

What it computes ("Musings on long-context fine-tuning", section "Isolating the recurrent layers":
a width-4 causal convolution reads the current input and three preceding inputs; each
continuation gets the shared prefix's final three inputs in front of it, seq_idx keeps documents
from reading each other; section "Backward through P": the gradients through that tail sum into the
prefix). Per channel c (depthwise), for document i with tokens x_i[0 .. n-1]:
    E_i = (init_i[0], init_i[1], init_i[2], x_i[0], ..., x_i[n-1])      (the extended input)
    y_i[p] = bias[c] + sum_{m=0..3} w[c, m] * E_i[p + m]                (p = 0 .. n-1)
    tail_i = (E_i[n], E_i[n + 1], E_i[n + 2])                           (its last three inputs)
init_i is zero (init_idx -1), a pool entry conv_init[x] (0 <= x < n_init), or tail_j of an earlier
document j of the same call (init_idx = n_init + j): the fork. Documents run in order.
The backward is the hand-written reverse of the same loops.
"""
from __future__ import annotations

import numpy as np

W = 4  # taps: the current input and three preceding ones


def conv_fwd(x, w, bias, cu_seqlens, init_idx=None, conv_init=None):
    """x [T, C], w [C, 4], bias [C] or None, conv_init [n_init, 3, C] or None.
    Returns y [T, C] and the final tails [N, 3, C], in fp64."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, C = x.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    n_init = 0 if conv_init is None else conv_init.shape[0]
    b = np.zeros(C) if bias is None else np.asarray(bias, dtype=np.float64)
    y = np.zeros((T, C))
    tails = np.zeros((N, 3, C))
    for i in range(N):
        s = int(init_idx[i]) if init_idx is not None else -1
        if s < 0:
            init = np.zeros((3, C))
        elif s < n_init:
            init = np.asarray(conv_init[s], dtype=np.float64)
        else:
            assert s - n_init < i, "a fork reads an earlier document"
            init = tails[s - n_init]
        E = np.concatenate([init, x[cu[i]:cu[i + 1]]], axis=0)
        n = cu[i + 1] - cu[i]
        for p in range(n):
            acc = b.copy()
            for m in range(W):
                acc += w[:, m] * E[p + m]
            y[cu[i] + p] = acc
        tails[i] = E[n:n + 3]
    return y, tails


def conv_bwd(x, w, bias, cu_seqlens, dy, dtail=None, init_idx=None, conv_init=None):
    """Reverse mode of conv_fwd for the loss sum(dy * y) + sum(dtail * tails).
    Returns dict dx [T, C], dw [C, 4], dbias [C], dinit [n_init, 3, C] (None without a pool)."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    T, C = x.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    n_init = 0 if conv_init is None else conv_init.shape[0]
    # forward sweep: every document's extended input
    Es = []
    tails = np.zeros((N, 3, C))
    for i in range(N):
        s = int(init_idx[i]) if init_idx is not None else -1
        init = (np.zeros((3, C)) if s < 0 else np.asarray(conv_init[s], dtype=np.float64) if s < n_init
                else tails[s - n_init])
        E = np.concatenate([init, x[cu[i]:cu[i + 1]]], axis=0)
        Es.append(E)
        n = cu[i + 1] - cu[i]
        tails[i] = E[n:n + 3]
    dx = np.zeros((T, C))
    dw = np.zeros((C, W))
    db = np.zeros(C)
    dinit = np.zeros((n_init, 3, C)) if n_init else None
    dtl = np.zeros((N, 3, C)) if dtail is None else np.array(dtail, dtype=np.float64)
    for i in range(N - 1, -1, -1):  # forks point backwards: their gradients arrive before i is reached
        E = Es[i]
        n = cu[i + 1] - cu[i]
        dE = np.zeros_like(E)
        dE[n:n + 3] += dtl[i]  # tail_i = E[n .. n + 2]
        for p in range(n):
            g = dy[cu[i] + p]
            db += g
            for m in range(W):
                dw[:, m] += g * E[p + m]
                dE[p + m] += w[:, m] * g
        dx[cu[i]:cu[i + 1]] += dE[3:]
        s = int(init_idx[i]) if init_idx is not None else -1
        if 0 <= s < n_init:
            dinit[s] += dE[:3]
        elif s >= n_init:
            dtl[s - n_init] += dE[:3]
    return dict(dx=dx, dw=dw, dbias=db, dinit=dinit)
