"""Edge cases of the call itself on the GPU: a call whose documents are all empty (T = 0). No
chunk kernel runs; the final states are the initial states (a pool entry, zero, or an earlier
document's final state through a fork) and the backward gives d(initial state) from dfinal_state
alone, summed over the documents that share a start, as the fp64 oracle does."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, run_bwd, run_fwd, run_train

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _empty_problem():
    # documents: pool entry 1, zero, pool entry 0, a fork of document 0's final state
    return synth.make_problem("all_empty", 5151, [0, 0, 0, 0], 2, 4, init_idx=[1, -1, 0, 2 + 0], n_init=2,
                              with_dout=True, with_dfinal=True)


def test_all_documents_empty_forward():
    p = _empty_problem()
    out, fin = run_fwd(p)
    ro, rf = oracle.fwd_problem(p)
    assert out.shape == ro.shape == (0, p.Hv, 128)
    np.testing.assert_array_equal(fin, rf)
    h0 = p.initial_state.astype(np.float64)
    np.testing.assert_array_equal(fin[0], h0[1])
    np.testing.assert_array_equal(fin[1], 0.0)
    np.testing.assert_array_equal(fin[2], h0[0])
    np.testing.assert_array_equal(fin[3], h0[1])


@pytest.mark.parametrize("path", ["recompute", "train"])
def test_all_documents_empty_backward(path):
    p = _empty_problem()
    if path == "train":
        _, fin, got = run_train(p)
        np.testing.assert_array_equal(fin, oracle.fwd_problem(p)[1])
    else:
        got = run_bwd(p)
    ref = oracle.bwd_problem(p)
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        assert got[key].shape == ref[key].shape and got[key].size == 0
    # pool entry 1 collects dfinal of document 0 and of its fork (document 3); entry 0 document 2's
    assert_close("all_empty dinit", got["dinit"], ref["dinit"])
    df = p.dfinal.astype(np.float64)
    np.testing.assert_allclose(got["dinit"][1], df[0] + df[3], rtol=1e-6, atol=1e-6)
    np.testing.assert_array_equal(got["dinit"][0], df[2])


def _many_documents_problem(with_dout=False):
    # 600 documents of 0-90 tokens (some empty, most shorter than a chunk): the planner's scans
    # over documents and segments run in several tiles, and most chunks are partial
    rng = np.random.default_rng(5252)
    lens = [int(x) for x in rng.integers(0, 91, size=600)]
    lens[::37] = [0] * len(lens[::37])
    return synth.make_problem("many_docs", 5252, lens, 1, 2, with_dout=with_dout)


def test_many_short_documents_forward():
    p = _many_documents_problem()
    out, fin = run_fwd(p)
    ro, rf = oracle.fwd_problem(p)
    assert_close("many_docs out", out, ro)
    assert_close("many_docs final_state", fin, rf)


def test_many_short_documents_backward():
    p = _many_documents_problem(with_dout=True)
    got = run_bwd(p)
    ref = oracle.bwd_problem(p)
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        assert_close(f"many_docs {key}", got[key], ref[key])
