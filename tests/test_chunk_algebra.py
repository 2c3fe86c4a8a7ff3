"""The chunk algebra the kernels implement, checked in fp64 against the oracle:
chunked forward, exact segment split (affine scan), truncation mode and its
error bound, and the chunked reverse mode."""
import json
import os

import numpy as np
import pytest

import oracle
from tests import chunked_ref as cr

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def one_doc(seed, L, Dk=16, Dv=12, g_mean=2.0, with_s0=True):
    r = np.random.default_rng(seed)
    q = r.standard_normal((L, Dk)) / np.sqrt(Dk)
    k = r.standard_normal((L, Dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = r.standard_normal((L, Dv))
    u = r.standard_normal(L) + g_mean
    g = -np.logaddexp(0.0, -u)
    beta = 1 / (1 + np.exp(-r.standard_normal(L)))
    S0 = 0.3 * r.standard_normal((Dk, Dv)) if with_s0 else np.zeros((Dk, Dv))
    return q, k, v, g, beta, S0


def oracle_doc(q, k, v, g, beta, S0):
    out, fin = oracle.fwd(q[:, None], k[:, None], v[:, None], g[:, None], beta[:, None], [0, q.shape[0]],
                          [0], S0[None, None])
    return out[:, 0], fin[0, 0]


@pytest.mark.parametrize("L", [1, 63, 64, 65, 200, 301])
def test_chunked_forward_matches_recurrence(L):
    q, k, v, g, beta, S0 = one_doc(L, L)
    O, S, _ = cr.doc_fwd(q, k, v, g, beta, S0)
    Or, Sr = oracle_doc(q, k, v, g, beta, S0)
    np.testing.assert_allclose(O, Or, atol=1e-11)
    np.testing.assert_allclose(S, Sr, atol=1e-11)


@pytest.mark.parametrize("L,seg", [(640, 1), (700, 3), (64 * 9 + 5, 4)])
def test_exact_segment_split_matches_recurrence(L, seg):
    q, k, v, g, beta, S0 = one_doc(100 + L, L, g_mean=5.0)  # slow decay: the carry matters
    O, S = cr.doc_fwd_split(q, k, v, g, beta, S0, seg)
    Or, Sr = oracle_doc(q, k, v, g, beta, S0)
    np.testing.assert_allclose(O, Or, atol=1e-10)
    np.testing.assert_allclose(S, Sr, atol=1e-10)


def test_truncation_error_within_printed_bound():
    """Truncation error <= e^{threshold} * ||S at the window start||: each chunk
    map has spectral norm <= e^{sum g} because ||I - beta k k^T||_2 = 1 for unit k."""
    c = json.load(open(os.path.join(GOLD, "printed_constants.json")))
    thr = c["trunc_log_threshold"]
    assert abs(np.exp(thr) - c["trunc_printed_value"]) <= c["trunc_printed_rel_precision"] * c["trunc_printed_value"]
    L = 64 * 24
    q, k, v, g, beta, S0 = one_doc(7, L, g_mean=3.0)  # ~-0.05 per token: windows of several chunks
    Ot, St, nw = cr.doc_fwd_truncated(q, k, v, g, beta, S0, seg_chunks=4, log_threshold=thr)
    Oe, Se, starts = cr.doc_fwd(q, k, v, g, beta, S0)
    assert max(nw) >= 2
    smax = max(np.linalg.norm(s, 2) for s in starts)
    bound = np.exp(thr) * smax
    err_S = np.linalg.norm(St - Se, 2)
    assert err_S <= bound * 1.0001
    err_o = np.max(np.linalg.norm(Ot - Oe, axis=1))
    assert err_o <= bound * np.max(np.linalg.norm(q, axis=1)) * 1.0001
    assert err_S > 0  # it is an approximation


def test_exact_warmup_cut_is_below_fp32_resolution():
    """The exact split starts a segment from zero over a window of whole chunks whose summed
    log-decay is below -30: the neglected term is at most e^-30 (about 2^-43) of the norm of the
    state at the window's start, 19 bits under fp32's unit roundoff. Checked in fp64 with the same
    window rule at that cut, on gates where windows span several chunks."""
    cut = -30.0
    assert np.exp(cut) < 2.0 ** -43 * 1.1 and np.exp(cut) < 2.0 ** -24 / 2.0 ** 19 * 1.1
    L = 64 * 24
    q, k, v, g, beta, S0 = one_doc(11, L, g_mean=2.0)  # about -8 per chunk: windows of about 4 chunks
    Ow, Sw, nw = cr.doc_fwd_truncated(q, k, v, g, beta, S0, seg_chunks=4, log_threshold=cut)
    Oe, Se, starts = cr.doc_fwd(q, k, v, g, beta, S0)
    assert min(nw[1:]) >= 3
    smax = max(np.linalg.norm(s, 2) for s in starts)
    bound = np.exp(cut) * smax
    assert np.linalg.norm(Sw - Se, 2) <= bound * 1.0001 + 1e-14 * smax
    assert np.max(np.linalg.norm(Ow - Oe, axis=1)) <= bound * np.max(np.linalg.norm(q, axis=1)) * 1.0001 + 1e-14 * smax
    # what it neglects is far below what fp32 resolves of the state itself
    assert bound < 2.0 ** -24 * smax / 1000


@pytest.mark.parametrize("L", [1, 50, 64, 130])
def test_chunked_backward_matches_oracle(L):
    q, k, v, g, beta, S0 = one_doc(200 + L, L, Dk=8, Dv=6)
    r = np.random.default_rng(L)
    dO = r.standard_normal(v.shape)
    dS = r.standard_normal(S0.shape)
    dS0, gr = cr.doc_bwd(q, k, v, g, beta, S0, dO, dS)
    ref = oracle.bwd(q[:, None], k[:, None], v[:, None], g[:, None], beta[:, None], [0, L], dO[:, None],
                     dS[None, None], [0], S0[None, None])
    np.testing.assert_allclose(gr["dq"], ref["dq"][:, 0], atol=1e-10)
    np.testing.assert_allclose(gr["dk"], ref["dk"][:, 0], atol=1e-10)
    np.testing.assert_allclose(gr["dv"], ref["dv"][:, 0], atol=1e-10)
    np.testing.assert_allclose(gr["dg"], ref["dg"][:, 0], atol=1e-10)
    np.testing.assert_allclose(gr["dbeta"], ref["dbeta"][:, 0], atol=1e-10)
    np.testing.assert_allclose(dS0, ref["dinit"][0, 0], atol=1e-10)
