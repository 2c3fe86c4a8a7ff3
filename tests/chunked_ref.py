"""fp64 chunked restatement of the gated delta rule (test helper, numpy).

The CUDA library computes the recurrence chunk by chunk. This module writes the
same chunk algebra in plain numpy so that the tests can check the algebra itself
against the token-by-token oracle before trusting any kernel; it also exposes
the per-chunk intermediates the kernels hold (T, w, u, the chunk-start states)
for debugging. It shares no code with the CUDA path.

Chunk algebra for one value head, chunk of n <= C tokens, start state S0
(derived by unrolling the recurrence of "How to Speed Up GDN Kernels for Qwen
Models", section "What GDN actually computes"; the chunked layout, the per-chunk
triangular system and the reuse of its solution by both the output and the
state update follow the same page, sections "What GDN actually computes" and
"Lever 2: do less arithmetic, not just faster arithmetic"):
    gamma_i = sum_{j<=i} g_j,  Gam_i = e^{gamma_i}
    A[i, j] = beta_i e^{gamma_i - gamma_j} k_i.k_j            (j < i)
    T = (I + A)^{-1}
    W = T diag(beta Gam) K,   U = T diag(beta) V
    V' = U - W S0                                             (the corrections d_i)
    O  = diag(Gam) Q S0 + ((Q K^T) o E) V',  E[i, j] = e^{gamma_i - gamma_j} (j <= i)
    S1 = Gam_n S0 + Kt^T V',  Kt_j = e^{gamma_n - gamma_j} k_j
which is the affine map S1 = Phi S0 + Kt^T U with Phi = Gam_n I - Kt^T W.
"""
from __future__ import annotations

import numpy as np


def chunk_quantities(q, k, v, g, beta):
    n = q.shape[0]
    gam = np.cumsum(g)
    Gam = np.exp(gam)
    E = np.exp(gam[:, None] - gam[None, :])
    A = np.tril(beta[:, None] * E * (k @ k.T), -1)
    Tm = np.linalg.inv(np.eye(n) + A)
    W = Tm @ ((beta * Gam)[:, None] * k)
    U = Tm @ (beta[:, None] * v)
    P = (q @ k.T) * np.tril(E)
    Kt = np.exp(gam[-1] - gam)[:, None] * k
    return dict(gam=gam, Gam=Gam, A=A, T=Tm, W=W, U=U, P=P, Kt=Kt, E=E)


def chunk_step(q, k, v, g, beta, S0):
    c = chunk_quantities(q, k, v, g, beta)
    Vp = c["U"] - c["W"] @ S0
    O = c["Gam"][:, None] * (q @ S0) + c["P"] @ Vp
    S1 = c["Gam"][-1] * S0 + c["Kt"].T @ Vp
    return O, S1, c


def chunk_affine(q, k, v, g, beta):
    """(Phi, B) with S1 = Phi S0 + B for this chunk."""
    c = chunk_quantities(q, k, v, g, beta)
    Phi = c["Gam"][-1] * np.eye(k.shape[1]) - c["Kt"].T @ c["W"]
    B = c["Kt"].T @ c["U"]
    return Phi, B


def doc_fwd(q, k, v, g, beta, S0, C=64):
    """One document, one value head. Returns (O, S_end, chunk start states)."""
    L = q.shape[0]
    O = np.zeros((L, v.shape[1]))
    S = S0.copy()
    starts = []
    for s in range(0, L, C):
        e = min(L, s + C)
        starts.append(S.copy())
        O[s:e], S, _ = chunk_step(q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e], S)
    return O, S, starts


def doc_fwd_split(q, k, v, g, beta, S0, seg_chunks, C=64):
    """Exact segment split: per segment, the local end state from zero (B_j) and the
    transition M_j = product of the chunk maps; an affine scan gives every
    segment's true start state; each segment then reruns with outputs."""
    L = q.shape[0]
    Dk = k.shape[1]
    bounds = list(range(0, L, C * seg_chunks)) + [L]
    segs = list(zip(bounds[:-1], bounds[1:]))
    maps = []
    for s, e in segs:
        M = np.eye(Dk)
        B = np.zeros((Dk, v.shape[1]))
        for cs in range(s, e, C):
            ce = min(e, cs + C)
            Phi, Bc = chunk_affine(q[cs:ce], k[cs:ce], v[cs:ce], g[cs:ce], beta[cs:ce])
            M = Phi @ M
            B = Phi @ B + Bc
        maps.append((M, B))
    # inclusive scan of affine maps: (M, B) o (M', B') = (M M', M B' + B)
    starts = [S0]
    for M, B in maps[:-1]:
        starts.append(M @ starts[-1] + B)
    O = np.zeros((L, v.shape[1]))
    S = None
    for (s, e), St in zip(segs, starts):
        O[s:e], S, _ = doc_fwd(q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e], St, C)
    return O, S


def doc_fwd_truncated(q, k, v, g, beta, S0, seg_chunks, C=64, log_threshold=-10.0):
    """Truncation mode: each segment start recomputes its carry from zero over the
    fewest preceding whole chunks whose summed log-decay is below the threshold
    (or from the document start, with S0, if the window reaches it)."""
    L = q.shape[0]
    bounds = list(range(0, L, C * seg_chunks)) + [L]
    O = np.zeros((L, v.shape[1]))
    S_end = None
    n_warm = []
    for s, e in zip(bounds[:-1], bounds[1:]):
        w = s
        acc = 0.0
        while w > 0 and acc >= log_threshold:
            w -= C
            acc += float(np.sum(g[w:w + C]))
        if w == 0 and acc >= log_threshold:
            start = S0.copy()
        else:
            start = np.zeros_like(S0)
        if w < s:
            _, start, _ = doc_fwd(q[w:s], k[w:s], v[w:s], g[w:s], beta[w:s], start, C)
        n_warm.append((s - w) // C)
        O[s:e], S_end, _ = doc_fwd(q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e], start, C)
    return O, S_end, n_warm


def chunk_bwd(q, k, v, g, beta, S0, dO, dS1):
    """Reverse mode of chunk_step. Returns dS0 and the chunk's dq, dk, dv, dg, dbeta."""
    c = chunk_quantities(q, k, v, g, beta)
    gam, Gam, Tm, W, U, Kt, E = c["gam"], c["Gam"], c["T"], c["W"], c["U"], c["Kt"], c["E"]
    n = q.shape[0]
    Vp = U - W @ S0
    P = c["P"]
    QK = q @ k.T
    lowc = np.tril(np.ones((n, n)))
    lows = np.tril(np.ones((n, n)), -1)
    dgam = np.zeros(n)
    # S1 = Gam_n S0 + Kt^T Vp
    dVp = Kt @ dS1 + P.T @ dO
    dS0 = Gam[-1] * dS1 + (Gam[:, None] * q).T @ dO
    dgam[-1] += Gam[-1] * np.sum(dS1 * S0)
    dKt = Vp @ dS1.T
    dk = np.exp(gam[-1] - gam)[:, None] * dKt
    kt_dot = np.sum(dKt * Kt, axis=1)
    dgam[-1] += kt_dot.sum()
    dgam -= kt_dot
    # O = diag(Gam) Q S0 + (QK o E) Vp
    QS = q @ S0
    dq = Gam[:, None] * (dO @ S0.T)
    dgam += Gam * np.sum(dO * QS, axis=1)
    dP = (dO @ Vp.T) * lowc
    dQK = dP * E
    dq += dQK @ k
    dk += dQK.T @ q
    dEg = dP * QK * E
    dgam += dEg.sum(axis=1) - dEg.sum(axis=0)
    # Vp = U - W S0
    dU = dVp
    dW = -dVp @ S0.T
    dS0 -= W.T @ dVp
    # U = T diag(beta) V ; W = T diag(beta Gam) K
    bV = beta[:, None] * v
    bGK = (beta * Gam)[:, None] * k
    dT = dU @ bV.T + dW @ bGK.T
    Y = Tm.T @ dU
    dv = beta[:, None] * Y
    dbeta = np.sum(v * Y, axis=1)
    X = Tm.T @ dW
    dk += (beta * Gam)[:, None] * X
    kx = np.sum(k * X, axis=1)
    dbeta += Gam * kx
    dgam += beta * Gam * kx
    # T = (I + A)^{-1}
    dA = -(Tm.T @ dT @ Tm.T) * lows
    # A = diag(beta) (E o KK^T), strictly lower
    KK = k @ k.T
    dKK = dA * beta[:, None] * E
    dk += (dKK + dKK.T) @ k
    dbeta += np.sum(dA * E * KK, axis=1)
    dAg = dA * c["A"]
    dgam += dAg.sum(axis=1) - dAg.sum(axis=0)
    dg = np.cumsum(dgam[::-1])[::-1]
    return dS0, dict(dq=dq, dk=dk, dv=dv, dg=dg, dbeta=dbeta)


def doc_bwd(q, k, v, g, beta, S0, dO, dS_end, C=64):
    """Reverse over the chunks of one document. Returns dS0 and the per-token grads."""
    L = q.shape[0]
    _, _, starts = doc_fwd(q, k, v, g, beta, S0, C)
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v), dg=np.zeros(L), dbeta=np.zeros(L))
    dS = dS_end.copy()
    chunks = list(range(0, L, C))
    for ci in reversed(range(len(chunks))):
        s = chunks[ci]
        e = min(L, s + C)
        dS, gr = chunk_bwd(q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e], starts[ci], dO[s:e], dS)
        for key in out:
            out[key][s:e] = gr[key]
    return dS, out
