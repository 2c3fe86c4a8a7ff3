"""Training step on the GPU: a forward that keeps its records for the backward
(save_for_backward), then the backward that reuses them (reuse_forward) on the same workspace.
o, the final states and every gradient against the fp64 oracle on the same seeded inputs
(relative L2 <= 1e-2, max-abs <= 2e-2), and the gradients bit-for-bit equal to those of the
backward that recomputes the forward itself."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, errors, fast_then_slow_problem, mixed_decay_problem, run_bwd, run_train

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import linear_attention_varlen_gb300 as gdn  # noqa: E402

KEYS = ("dq", "dk", "dv", "dg", "dbeta")
STRESS_MAX_REL = 5e-3  # as for the backward's stress inputs: largest error relative to the largest entry


def check_train(p, options=None, stress=False, record=None):
    out, fin, got = run_train(p, options)
    ro, rf = oracle.fwd_problem(p)
    res = {"out": assert_close(f"{p.name} out", out, ro), "final_state": None}
    rel, mx = errors(fin, rf)
    if stress:
        assert rel <= 1e-2 and mx <= STRESS_MAX_REL * max(float(np.abs(rf).max()), 1.0), f"{p.name} final: {rel} {mx}"
        res["final_state"] = (rel, mx)
    else:
        res["final_state"] = assert_close(f"{p.name} final_state", fin, rf)
    ref = oracle.bwd_problem(p)
    keys = KEYS + (("dinit",) if p.initial_state is not None else ())
    for key in keys:
        rel, mx = errors(got[key], ref[key])
        print(f"ERRS {p.name} {key} rel={rel:.3e} maxabs={mx:.3e}")
        if stress:
            mref = float(np.abs(ref[key]).max())
            assert rel <= 1e-2 and mx <= STRESS_MAX_REL * max(mref, 1.0), f"{p.name} {key}: {rel:.3e} {mx:.3e}"
            res[key] = (rel, mx)
        else:
            res[key] = assert_close(f"{p.name} {key}", got[key], ref[key])
    if record is not None:
        for k, (rel, mx) in res.items():
            record(f"{k}_rel_l2", rel)
            record(f"{k}_max_abs", mx)
    return got


@pytest.mark.parametrize("T", [1, 65, 200])
@pytest.mark.parametrize("Hk,Hv", [(1, 1), (2, 8)])
def test_train_single_document_shapes(T, Hk, Hv):
    # the backward tests' problems (seed 300 + T)
    p = synth.make_problem(f"train_T{T}", 300 + T, [T], Hk, Hv, with_dout=True)
    check_train(p)


def test_train_packed_ragged_documents():
    lens = [1, 0, 64, 5, 129, 0, 63, 300, 2]
    p = synth.make_problem("train_ragged", 412, lens, 2, 4, with_dout=True)
    check_train(p)


def test_train_pool_states_shared_and_forks():
    lens = [70, 0, 130, 64, 9, 200]
    init = [1, 0, 3, 0, 5, -1]
    p = synth.make_problem("train_forks", 413, lens, 2, 4, init_idx=init, n_init=2, with_dout=True, with_dfinal=True)
    check_train(p, stress=True)


@pytest.mark.parametrize("seg", [2, 5])
def test_train_with_split(seg):
    p = synth.make_problem(f"train_split{seg}", 420 + seg, [64 * 13 + 9, 64 * 4], 2, 4, with_dout=True, g_mean=5.0)
    check_train(p, gdn.Options(segment_chunks=seg))


def test_train_slow_decay_long():
    p = synth.make_problem("train_slow", 430, [2048], 1, 2, with_dout=True, g_mean=6.0)
    check_train(p, stress=True)


@pytest.mark.parametrize("seg", [0, 3])
def test_train_gradients_equal_recompute(seg):
    """The forward's records are the backward's recompute: identical gradients."""
    p = synth.make_problem(f"train_eq{seg}", 440 + seg, [64 * 10 + 5, 64 * 7, 300], 2, 4, init_idx=[-1, 0, 0],
                           with_dout=True)
    opts = gdn.Options(segment_chunks=seg)
    _, _, a = run_train(p, opts)
    b = run_bwd(p, opts)
    for key in KEYS:
        np.testing.assert_array_equal(a[key], b[key])


def test_train_split_mixed_decay_equals_recompute():
    p = mixed_decay_problem("train_mixed", 460, with_dout=True, beta_boost=3.0)
    opts = gdn.Options(segment_chunks=3)
    check_train(p, opts, stress=True)
    _, _, a = run_train(p, opts)
    b = run_bwd(p, opts)
    for key in KEYS:
        np.testing.assert_array_equal(a[key], b[key])


def test_train_split_warm_segment_publishes():
    """Forward and reverse: segments that warm up next to segments that wait for a publication."""
    p = fast_then_slow_problem("train_warm_pub", 470, with_dout=True)
    check_train(p, gdn.Options(segment_chunks=4), stress=True)


def test_train_rejects_truncation_mode():
    p = synth.make_problem("train_trunc", 450, [200], 1, 2, with_dout=True)
    with pytest.raises(gdn.GdnError):
        run_train(p, gdn.Options(mode="truncate"))


def test_train_workload_train_full(record_property):
    """Full-size training step: 4 documents x 16384 tokens, 8 value heads over 2 key heads."""
    check_train(synth.workload_train(), record=record_property)


def test_train_workload_long_full(record_property):
    """Full-size long prefill shape as a training step: one 32768-token document, 8 value heads."""
    p = synth.make_problem("train_long_T32768_H8", synth.SEEDS[2], [32768], 2, 8, with_dout=True)
    check_train(p, record=record_property)
