"""Pins for the fp64 oracle of the width-4 causal convolution (oracle/conv.py), fixed outside it:
  * a library convolution (numpy.convolve) on one document from zero;
  * closed form: a one-hot filter tap m copies the input shifted by 3 - m;
  * packing: documents never read each other (packed = separate runs; the contamination probe);
  * the fork of "Musings on long-context fine-tuning" ("Isolating the recurrent layers"): a
    continuation forked from P equals a second call whose initial inputs are P's final three, and
    ("Backward through P") the gradient through that tail sums into P;
  * the backward against central differences, with a pool entry, forks, documents shorter than
    the tail and a gradient on the final tails;
  * mutants of the oracle (substituted functions) that these pins reject."""
import numpy as np
import pytest

import oracle.conv as oc

rng = np.random.default_rng


def rand_case(seed, lengths, C, n_init=0):
    r = rng(seed)
    T = sum(lengths)
    return dict(x=r.standard_normal((T, C)), w=r.standard_normal((C, 4)), bias=r.standard_normal(C),
                cu=np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64),
                conv_init=r.standard_normal((n_init, 3, C)) if n_init else None)


def test_matches_numpy_convolve_on_one_document():
    c = rand_case(1, [57], 5)
    y, tails = oc.conv_fwd(c["x"], c["w"], c["bias"], c["cu"])
    for ch in range(5):
        # y[t] = b + sum_m w[m] x[t - 3 + m]: the full convolution with the reversed taps, first T outputs
        ref = np.convolve(c["x"][:, ch], c["w"][ch, ::-1])[:57] + c["bias"][ch]
        np.testing.assert_allclose(y[:, ch], ref, rtol=0, atol=1e-13)
    np.testing.assert_array_equal(tails[0], c["x"][-3:])


@pytest.mark.parametrize("m", [0, 1, 2, 3])
def test_one_hot_tap_is_a_shift(m):
    """w[:, m] = 1 makes y[p] the extended input E[p + m]: the document's inputs shifted by 3 - m,
    with the start (pool entry, the forked document's last three inputs, or zeros) in front."""
    c = rand_case(2, [9, 2, 6], 3, n_init=1)
    w = np.zeros((3, 4))
    w[:, m] = 1.0
    ii = [0, 1, -1]  # pool entry 0; document 1 forks document 0 (n_init + 0); zeros
    y, _ = oc.conv_fwd(c["x"], w, None, c["cu"], ii, c["conv_init"])
    starts = [c["conv_init"][0], c["x"][6:9], np.zeros((3, 3))]
    for i, (a, b) in enumerate(zip(c["cu"][:-1], c["cu"][1:])):
        E = np.concatenate([starts[i], c["x"][a:b]])
        np.testing.assert_array_equal(y[a:b], E[m:m + (b - a)])


def test_packed_equals_separate_runs_and_probe():
    c = rand_case(3, [20, 1, 0, 13], 4)
    y, tails = oc.conv_fwd(c["x"], c["w"], c["bias"], c["cu"])
    for a, b in zip(c["cu"][:-1], c["cu"][1:]):
        ys, _ = oc.conv_fwd(c["x"][a:b], c["w"], c["bias"], [0, b - a])
        np.testing.assert_array_equal(y[a:b], ys)
    x2 = c["x"].copy()
    x2[:20] += 100.0  # document 0 ends differently: nothing after it may change
    y2, _ = oc.conv_fwd(x2, c["w"], c["bias"], c["cu"])
    np.testing.assert_array_equal(y2[20:], y[20:])
    np.testing.assert_array_equal(tails[2], np.zeros((3, 4)))  # an empty document passes its (zero) start on


def test_fork_equals_two_calls_forward_and_backward():
    c = rand_case(4, [11, 7, 2], 3)
    r = rng(5)
    dy = r.standard_normal(c["x"].shape)
    ii = [-1, 0, 0]  # n_init = 0: both continuations fork document 0
    y, _ = oc.conv_fwd(c["x"], c["w"], c["bias"], c["cu"], ii)
    full = oc.conv_bwd(c["x"], c["w"], c["bias"], c["cu"], dy, None, ii)
    yp, tp = oc.conv_fwd(c["x"][:11], c["w"], c["bias"], [0, 11])
    cont = slice(11, 20)
    yc, _ = oc.conv_fwd(c["x"][cont], c["w"], c["bias"], [0, 7, 9], [0, 0], tp)
    np.testing.assert_allclose(y[:11], yp, rtol=0, atol=1e-14)
    np.testing.assert_allclose(y[cont], yc, rtol=0, atol=1e-14)
    gc = oc.conv_bwd(c["x"][cont], c["w"], c["bias"], [0, 7, 9], dy[cont], None, [0, 0], tp)
    gp = oc.conv_bwd(c["x"][:11], c["w"], c["bias"], [0, 11], dy[:11], gc["dinit"])  # tail gradients sum into P
    np.testing.assert_allclose(full["dx"][:11], gp["dx"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(full["dx"][cont], gc["dx"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(full["dw"], gp["dw"] + gc["dw"], rtol=0, atol=1e-12)


def _loss(c, ii, dy, dtail, x=None, w=None, b=None, ci=None):
    y, t = oc.conv_fwd(c["x"] if x is None else x, c["w"] if w is None else w, c["bias"] if b is None else b,
                       c["cu"], ii, c["conv_init"] if ci is None else ci)
    return float(np.sum(y * dy) + np.sum(t * dtail))


def test_backward_matches_finite_differences():
    c = rand_case(6, [5, 2, 0, 4, 1], 3, n_init=2)
    ii = [1, 0, 2, 3, 4]  # pool entries 1 and 0; documents 2, 3, 4 fork documents 0, 1 and the empty 2
    r = rng(7)
    dy = r.standard_normal(c["x"].shape)
    dtail = r.standard_normal((5, 3, 3))
    g = oc.conv_bwd(c["x"], c["w"], c["bias"], c["cu"], dy, dtail, ii, c["conv_init"])
    eps = 1e-6
    for name, key in (("x", "dx"), ("w", "dw"), ("bias", "dbias"), ("conv_init", "dinit")):
        arr = c[name]
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = _loss(c, ii, dy, dtail)
            arr[idx] = old - eps
            lm = _loss(c, ii, dy, dtail)
            arr[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g[key], num, rtol=0, atol=1e-7, err_msg=key)


# Mutants: plausible slips substituted for the oracle's functions; some pin above must fail.
def _mut_tail_from_front(x, w, bias, cu, init_idx=None, conv_init=None):
    y, t = oc_orig_fwd(x, w, bias, cu, init_idx, conv_init)
    cu = np.asarray(cu)
    for i in range(len(cu) - 1):
        if cu[i + 1] - cu[i] >= 3:
            t[i] = np.asarray(x, dtype=np.float64)[cu[i]:cu[i] + 3]
    return y, t


def _mut_reversed_taps(x, w, bias, cu, init_idx=None, conv_init=None):
    return oc_orig_fwd(x, np.asarray(w)[:, ::-1], bias, cu, init_idx, conv_init)


def _mut_no_fork_gradient(x, w, bias, cu, dy, dtail=None, init_idx=None, conv_init=None):
    ii = None if init_idx is None else [v if v < (0 if conv_init is None else conv_init.shape[0]) else -1
                                        for v in init_idx]
    g = oc_orig_bwd(x, w, bias, cu, dy, dtail, init_idx, conv_init)
    g2 = oc_orig_bwd(x, w, bias, cu, dy, dtail, ii, conv_init)
    g["dx"] = g2["dx"]
    return g


oc_orig_fwd, oc_orig_bwd = oc.conv_fwd, oc.conv_bwd
MUTANTS = [("tail from the front", "conv_fwd", _mut_tail_from_front),
           ("reversed taps", "conv_fwd", _mut_reversed_taps),
           ("fork gradient dropped", "conv_bwd", _mut_no_fork_gradient)]
PINS = [test_matches_numpy_convolve_on_one_document, test_packed_equals_separate_runs_and_probe,
        test_fork_equals_two_calls_forward_and_backward, test_backward_matches_finite_differences]


@pytest.mark.parametrize("name,attr,fn", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, attr, fn, monkeypatch):
    monkeypatch.setattr(oc, attr, fn)
    failed = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed, f"no pin caught '{name}'"
