"""Pins for the fp64 oracle: checks against facts fixed outside it.

Each check is chosen so that a plausible slip in the oracle (a dropped decay,
a sign, a transposed state, a wrong head map, a lost reset) fails at least one:
  * hand-worked cases (tests/golden/hand_worked.json);
  * the brute-force quadratic form: the whole document as ONE dense linear
    system solved by LU (different arithmetic, same mathematics);
  * closed forms: beta = 0 is pure decay; g = 0, beta = 1 with orthonormal keys
    stores every value exactly (S^T k_i = v_i);
  * packing invariants: a state reset at each cu_seqlens boundary equals
    separate runs, and an in-call fork equals two calls ("Musings on
    long-context fine-tuning", sections "Isolating the recurrent layers" and
    "Checking the packed computation");
  * the backward against central finite differences of the forward, and the
    gradient-sum rule at a shared initial state (same page, section "Backward
    through P").
Dk != Dv everywhere a transposed state could hide.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng


def rand_problem(seed, lengths, Hk, Hv, Dk, Dv, n_init=0, init_idx=None, g_lo=-0.6, g_hi=-0.01):
    r = rng(seed)
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q = r.standard_normal((T, Hk, Dk)) / np.sqrt(Dk)
    k = r.standard_normal((T, Hk, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((T, Hv, Dv))
    g = r.uniform(g_lo, g_hi, (T, Hv))
    beta = r.uniform(0.05, 0.95, (T, Hv))
    h0 = r.standard_normal((n_init, Hv, Dk, Dv)) if n_init else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, cu_seqlens=cu, init_idx=init_idx, initial_state=h0)


# ----------------------------------------------------------------------------- hand-worked cases


def test_hand_worked_cases():
    cases = json.load(open(os.path.join(GOLD, "hand_worked.json")))["cases"]
    for c in cases:
        q = np.array(c["q"])[:, None, :]
        k = np.array(c["k"])[:, None, :]
        v = np.array(c["v"])[:, None, :]
        g = np.array(c["g"])[:, None]
        b = np.array(c["beta"])[:, None]
        T = q.shape[0]
        S0 = np.array(c["S0"])[None, None]
        out, fin = oracle.fwd(q, k, v, g, b, [0, T], init_idx=[0], initial_state=S0)
        np.testing.assert_allclose(out[:, 0, :], np.array(c["o"]), rtol=0, atol=1e-14, err_msg=c["name"])
        np.testing.assert_allclose(fin[0, 0], np.array(c["S"]), rtol=0, atol=1e-14, err_msg=c["name"])


# ----------------------------------------------------------------------------- brute-force quadratic form


def dense_solution(q, k, v, g, beta, S0):
    """One document, one value head, as a single dense system.

    Unrolling the recurrence with gamma_t = sum_{j<=t} g_j gives, for the
    corrections d_t = beta_t (v_t - e^{g_t} S_{t-1}^T k_t),
        (I + A) D = diag(beta) V - diag(beta e^gamma) K S0,
        A[t, j] = beta_t e^{gamma_t - gamma_j} k_t.k_j   (j < t),
    then O = diag(e^gamma) Q S0 + ((Q K^T) o Mask) D with Mask[t, j] = e^{gamma_t - gamma_j}
    (j <= t), and S_T = e^{gamma_T} S0 + sum_j e^{gamma_T - gamma_j} k_j d_j^T.
    Solved with LU (numpy.linalg.solve) over the full T x T system.
    """
    T = q.shape[0]
    gam = np.cumsum(g)
    E = np.exp(gam[:, None] - gam[None, :])
    low = np.tril(np.ones((T, T)), -1)
    A = beta[:, None] * E * (k @ k.T) * low
    rhs = beta[:, None] * v - (beta * np.exp(gam))[:, None] * (k @ S0)
    D = np.linalg.solve(np.eye(T) + A, rhs)
    M = E * np.tril(np.ones((T, T)))
    O = np.exp(gam)[:, None] * (q @ S0) + ((q @ k.T) * M) @ D
    S = np.exp(gam[-1]) * S0 + (np.exp(gam[-1] - gam)[:, None] * k).T @ D
    return O, S


@pytest.mark.parametrize("T,Dk,Dv", [(1, 4, 3), (17, 8, 5), (64, 16, 16), (200, 8, 12), (256, 128, 128)])
def test_brute_force_quadratic_form(T, Dk, Dv):
    Hk, Hv = 1, 2
    p = rand_problem(7 + T, [T], Hk, Hv, Dk, Dv, n_init=1, init_idx=[0])
    out, fin = oracle.fwd(**p)
    for h in range(Hv):
        O, S = dense_solution(p["q"][:, 0], p["k"][:, 0], p["v"][:, h], p["g"][:, h], p["beta"][:, h],
                              p["initial_state"][0, h])
        scale = max(1.0, np.abs(O).max())
        np.testing.assert_allclose(out[:, h], O, rtol=0, atol=1e-11 * scale)
        np.testing.assert_allclose(fin[0, h], S, rtol=0, atol=1e-11 * max(1.0, np.abs(S).max()))


def test_gqa_head_map_contiguous_groups():
    """Value head h reads key head h // (Hv/Hk): each value head must match a single-head
    run that uses that key head alone."""
    Hk, Hv, Dk, Dv = 2, 6, 8, 4
    p = rand_problem(11, [40], Hk, Hv, Dk, Dv)
    out, fin = oracle.fwd(**p)
    for h in range(Hv):
        hk = h // (Hv // Hk)
        O, S = dense_solution(p["q"][:, hk], p["k"][:, hk], p["v"][:, h], p["g"][:, h], p["beta"][:, h],
                              np.zeros((Dk, Dv)))
        np.testing.assert_allclose(out[:, h], O, atol=1e-12)
        np.testing.assert_allclose(fin[0, h], S, atol=1e-12)


# ----------------------------------------------------------------------------- closed forms


def test_beta_zero_is_pure_decay():
    Hk, Hv, Dk, Dv = 1, 3, 8, 6
    p = rand_problem(3, [50], Hk, Hv, Dk, Dv, n_init=1, init_idx=[0])
    p["beta"][:] = 0.0
    out, fin = oracle.fwd(**p)
    gam = np.cumsum(p["g"], axis=0)  # [T, Hv]
    for h in range(Hv):
        S0 = p["initial_state"][0, h]
        expect = np.exp(gam[:, h])[:, None] * (p["q"][:, 0] @ S0)
        np.testing.assert_allclose(out[:, h], expect, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(fin[0, h], np.exp(gam[-1, h]) * S0, rtol=1e-13, atol=1e-15)


def test_orthonormal_keys_store_values_exactly():
    """g = 0, beta = 1, orthonormal keys: each token overwrites its own direction,
    so S^T k_i = v_i for every i and o_t = sum_{i<=t} (q_t.k_i) v_i."""
    T, Dk, Dv = 12, 16, 7
    r = rng(5)
    Qm, _ = np.linalg.qr(r.standard_normal((Dk, Dk)))
    k = Qm[:T][:, None, :]
    q = r.standard_normal((T, 1, Dk))
    v = r.standard_normal((T, 1, Dv))
    g = np.zeros((T, 1))
    b = np.ones((T, 1))
    out, fin = oracle.fwd(q, k, v, g, b, [0, T])
    S = fin[0, 0]
    np.testing.assert_allclose(k[:, 0] @ S, v[:, 0], atol=1e-13)
    qk = q[:, 0] @ k[:, 0].T
    expect = np.tril(qk) @ v[:, 0]
    np.testing.assert_allclose(out[:, 0], expect, atol=1e-13)


def test_empty_documents_pass_the_state_through():
    Hk, Hv, Dk, Dv = 1, 2, 4, 4
    p = rand_problem(9, [0, 5, 0], Hk, Hv, Dk, Dv, n_init=2, init_idx=[1, 0, 0])
    out, fin = oracle.fwd(**p)
    np.testing.assert_array_equal(fin[0], p["initial_state"][1])
    np.testing.assert_array_equal(fin[2], p["initial_state"][0])


# ----------------------------------------------------------------------------- packing invariants


def test_reset_at_boundaries_equals_separate_runs():
    Hk, Hv, Dk, Dv = 2, 4, 8, 6
    lens = [13, 1, 30, 7]
    p = rand_problem(21, lens, Hk, Hv, Dk, Dv)
    out, fin = oracle.fwd(**p)
    cu = p["cu_seqlens"]
    for i, L in enumerate(lens):
        sl = slice(cu[i], cu[i + 1])
        o1, f1 = oracle.fwd(p["q"][sl], p["k"][sl], p["v"][sl], p["g"][sl], p["beta"][sl], [0, L])
        np.testing.assert_array_equal(out[sl], o1)
        np.testing.assert_array_equal(fin[i], f1[0])


def test_contamination_probe():
    """Changing document A must leave document B's outputs untouched (block-diagonal)."""
    Hk, Hv, Dk, Dv = 1, 2, 8, 4
    p = rand_problem(22, [20, 20], Hk, Hv, Dk, Dv)
    out, _ = oracle.fwd(**p)
    p2 = {kk: (vv.copy() if isinstance(vv, np.ndarray) else vv) for kk, vv in p.items()}
    p2["v"][:20] += 5.0
    p2["k"][:20] = -p2["k"][:20]
    out2, _ = oracle.fwd(**p2)
    np.testing.assert_array_equal(out[20:], out2[20:])
    assert np.abs(out[:20] - out2[:20]).max() > 1e-3


def test_in_call_fork_equals_two_calls():
    Hk, Hv, Dk, Dv = 1, 2, 8, 5
    lens = [25, 10, 17, 9]
    p = rand_problem(31, lens, Hk, Hv, Dk, Dv, init_idx=[-1, 0, 0, 1])  # n_init = 0: x = j
    out, fin = oracle.fwd(**p)
    cu = p["cu_seqlens"]

    def seg(i):
        return slice(cu[i], cu[i + 1])

    o0, f0 = oracle.fwd(*(p[x][seg(0)] for x in ("q", "k", "v", "g", "beta")), [0, lens[0]])
    o1, f1 = oracle.fwd(*(p[x][seg(1)] for x in ("q", "k", "v", "g", "beta")), [0, lens[1]], [0], f0)
    o2, f2 = oracle.fwd(*(p[x][seg(2)] for x in ("q", "k", "v", "g", "beta")), [0, lens[2]], [0], f0)
    o3, f3 = oracle.fwd(*(p[x][seg(3)] for x in ("q", "k", "v", "g", "beta")), [0, lens[3]], [0], f1)
    for i, (o, f) in enumerate([(o0, f0), (o1, f1), (o2, f2), (o3, f3)]):
        np.testing.assert_array_equal(out[seg(i)], o)
        np.testing.assert_array_equal(fin[i], f[0])


def test_thread_count_does_not_change_bits():
    p = rand_problem(41, [33, 64, 5], 2, 4, 16, 16)
    a = oracle.fwd(**p, threads=1)
    b = oracle.fwd(**p, threads=7)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_invalid_layouts_are_rejected():
    p = rand_problem(1, [4, 4], 1, 1, 4, 4)
    bad = dict(p)
    bad["cu_seqlens"] = np.array([0, 5, 4], dtype=np.int32)
    with pytest.raises(ValueError):
        oracle.fwd(**bad)
    bad = dict(p)
    bad["init_idx"] = [-1, 1]  # fork must point to an earlier document
    with pytest.raises(ValueError):
        oracle.fwd(**bad)


# ----------------------------------------------------------------------------- backward


def _loss(p, dout, dfinal):
    out, fin = oracle.fwd(**p)
    return float(np.sum(out * dout) + np.sum(fin * dfinal))


def test_backward_matches_finite_differences():
    """Tiny problem with GQA 4:2, a pool initial state shared by two documents, an
    in-call fork and a one-token document; every gradient against central differences."""
    Hk, Hv, Dk, Dv = 2, 4, 5, 3
    lens = [6, 1, 5, 4]
    p = rand_problem(51, lens, Hk, Hv, Dk, Dv, n_init=1, init_idx=[0, 0, 1, -1])  # doc 2 forks doc 0
    r = rng(52)
    T = sum(lens)
    dout = r.standard_normal((T, Hv, Dv))
    dfinal = r.standard_normal((len(lens), Hv, Dk, Dv))
    gr = oracle.bwd(p["q"], p["k"], p["v"], p["g"], p["beta"], p["cu_seqlens"], dout, dfinal,
                    p["init_idx"], p["initial_state"])
    eps = 1e-6
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", initial_state="dinit")
    for name, gname in names.items():
        x = p[name]
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(p, dout, dfinal)
            x[idx] = old - eps
            lm = _loss(p, dout, dfinal)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        ana = gr[gname]
        err = np.abs(ana - num).max() / max(1.0, np.abs(num).max())
        assert err < 1e-6, f"{gname}: rel err {err:.3e}"


def test_backward_finite_differences_across_checkpoints():
    """The oracle's backward rebuilds each document in 64-token blocks from saved states; here
    documents of 130 and 70 tokens cross that interval (the 130-token one twice, the second one
    forked from the first), with a slow decay so that the state carries across the block edges.
    Central differences on a seeded sample of entries of every input, always including the tokens
    on both sides of each block edge, must match the hand-written reverse mode."""
    Hk, Hv, Dk, Dv = 1, 2, 3, 2
    lens = [130, 70]
    p = rand_problem(61, lens, Hk, Hv, Dk, Dv, n_init=1, init_idx=[0, 1], g_lo=-0.08, g_hi=-0.002)
    r = rng(62)
    T = sum(lens)
    dout = r.standard_normal((T, Hv, Dv))
    dfinal = r.standard_normal((len(lens), Hv, Dk, Dv))
    gr = oracle.bwd(p["q"], p["k"], p["v"], p["g"], p["beta"], p["cu_seqlens"], dout, dfinal,
                    p["init_idx"], p["initial_state"])
    edges = [0, 63, 64, 65, 127, 128, 129, 130, 130 + 63, 130 + 64, T - 1]  # block edges of both documents
    eps = 1e-6
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", initial_state="dinit")
    for name, gname in names.items():
        x = p[name]
        if name == "initial_state":
            picks = [tuple(i) for i in np.ndindex(x.shape)]
        else:
            rest = x.shape[1:]
            picks = [(t,) + tuple(i) for t in edges for i in np.ndindex(rest)]
            flat = r.choice(x.size, size=min(40, x.size), replace=False)
            picks += [tuple(int(c) for c in np.unravel_index(f, x.shape)) for f in flat]
        ana = gr[gname]
        num = np.array([0.0] * len(picks))
        for n_, idx in enumerate(picks):
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(p, dout, dfinal)
            x[idx] = old - eps
            lm = _loss(p, dout, dfinal)
            x[idx] = old
            num[n_] = (lp - lm) / (2 * eps)
        got = np.array([ana[idx] for idx in picks])
        err = np.abs(got - num).max() / max(1.0, np.abs(num).max())
        assert err < 1e-6, f"{gname}: rel err {err:.3e}"


def test_backward_gradient_sums_at_shared_state():
    """d(shared initial state) = sum over the documents that start from it."""
    Hk, Hv, Dk, Dv = 1, 2, 6, 4
    lens = [9, 14]
    p = rand_problem(61, lens, Hk, Hv, Dk, Dv, n_init=1, init_idx=[0, 0])
    r = rng(62)
    dout = r.standard_normal((sum(lens), Hv, Dv))
    full = oracle.bwd(p["q"], p["k"], p["v"], p["g"], p["beta"], p["cu_seqlens"], dout, None, p["init_idx"],
                      p["initial_state"])
    parts = []
    cu = p["cu_seqlens"]
    for i, L in enumerate(lens):
        sl = slice(cu[i], cu[i + 1])
        parts.append(oracle.bwd(p["q"][sl], p["k"][sl], p["v"][sl], p["g"][sl], p["beta"][sl], [0, L], dout[sl],
                                None, [0], p["initial_state"])["dinit"])
    np.testing.assert_allclose(full["dinit"], parts[0] + parts[1], rtol=1e-13, atol=1e-13)


def test_backward_fork_equals_two_calls():
    """Gradient into a forked prefix = its own gradient with dfinal set to the
    branch's d(initial state) (same page, section "Backward through P")."""
    Hk, Hv, Dk, Dv = 1, 2, 6, 5
    lens = [12, 8]
    p = rand_problem(71, lens, Hk, Hv, Dk, Dv, init_idx=[-1, 0])
    r = rng(72)
    T = sum(lens)
    dout = r.standard_normal((T, Hv, Dv))
    full = oracle.bwd(p["q"], p["k"], p["v"], p["g"], p["beta"], p["cu_seqlens"], dout, None, p["init_idx"])
    sa, sb = slice(0, 12), slice(12, 20)
    _, f0 = oracle.fwd(*(p[x][sa] for x in ("q", "k", "v", "g", "beta")), [0, 12])
    br = oracle.bwd(*(p[x][sb] for x in ("q", "k", "v", "g", "beta")), [0, 8], dout[sb], None, [0], f0)
    pre = oracle.bwd(*(p[x][sa] for x in ("q", "k", "v", "g", "beta")), [0, 12], dout[sa], br["dinit"])
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        np.testing.assert_allclose(full[key][sa], pre[key], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(full[key][sb], br[key], rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------- q / k normalisation


def test_l2norm_rows_closed_forms():
    """Rows come out with norm sqrt(s / (s + eps)) (1 up to eps), parallel to the input; a row that is
    already a unit vector times c > 0 maps to (almost) the unit vector; a zero row stays zero."""
    r = rng(81)
    x = r.standard_normal((7, 3, 16)) * r.uniform(0.1, 5.0, (7, 3, 1))
    y = oracle.l2norm_rows(x)
    s_ = np.sum(x * x, axis=-1)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.sqrt(s_ / (s_ + oracle.L2NORM_EPS)), rtol=1e-14)
    cos = np.sum(x * y, axis=-1) / (np.linalg.norm(x, axis=-1) * np.linalg.norm(y, axis=-1))
    np.testing.assert_allclose(cos, 1.0, rtol=1e-14)
    u = np.zeros((1, 1, 4))
    u[0, 0, 2] = 3.0
    np.testing.assert_allclose(oracle.l2norm_rows(u)[0, 0], [0, 0, 3.0 / np.sqrt(9.0 + 1e-6), 0], rtol=1e-15)
    assert not np.any(oracle.l2norm_rows(np.zeros((2, 5))))


def test_l2norm_rows_bwd_matches_finite_differences():
    r = rng(82)
    x = r.standard_normal((3, 2, 6)) * r.uniform(0.2, 3.0, (3, 2, 1))
    dy = r.standard_normal(x.shape)
    dx = oracle.l2norm_rows_bwd(x, dy)
    eps = 1e-6
    num = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        old = x[idx]
        x[idx] = old + eps
        lp = np.sum(dy * oracle.l2norm_rows(x))
        x[idx] = old - eps
        lm = np.sum(dy * oracle.l2norm_rows(x))
        x[idx] = old
        num[idx] = (lp - lm) / (2 * eps)
    np.testing.assert_allclose(dx, num, rtol=0, atol=1e-8)
    # the gradient is orthogonal to the row (scaling a row leaves the output unchanged, up to eps)
    np.testing.assert_allclose(np.sum(dx * x, axis=-1), 0.0, atol=1e-6 * np.abs(dx).max())


def test_normalised_recurrence_gradient_chain_rule():
    """Through the recurrence: the gradient with respect to raw q and k, formed as l2norm_rows_bwd of
    the oracle's gradient at the normalised inputs, matches central differences of the composed
    forward."""
    Hk, Hv, Dk, Dv = 1, 2, 4, 3
    lens = [5, 3]
    p = rand_problem(83, lens, Hk, Hv, Dk, Dv)
    r = rng(84)
    q_raw = p["q"] * r.uniform(0.5, 2.0, (sum(lens), Hk, 1))
    k_raw = p["k"] * r.uniform(0.5, 2.0, (sum(lens), Hk, 1))
    dout = r.standard_normal((sum(lens), Hv, Dv))

    def loss(qr, kr):
        out, _ = oracle.fwd(oracle.l2norm_rows(qr), oracle.l2norm_rows(kr), p["v"], p["g"], p["beta"],
                            p["cu_seqlens"])
        return float(np.sum(out * dout))

    gr = oracle.bwd(oracle.l2norm_rows(q_raw), oracle.l2norm_rows(k_raw), p["v"], p["g"], p["beta"],
                    p["cu_seqlens"], dout)
    dq = oracle.l2norm_rows_bwd(q_raw, gr["dq"])
    dk = oracle.l2norm_rows_bwd(k_raw, gr["dk"])
    eps = 1e-6
    for x, ana in ((q_raw, dq), (k_raw, dk)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            lp = loss(q_raw, k_raw)
            x[idx] = old - eps
            lm = loss(q_raw, k_raw)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        assert np.abs(ana - num).max() / max(1.0, np.abs(num).max()) < 1e-6

