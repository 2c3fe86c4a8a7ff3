"""Backward parity on the GPU: dq, dk, dv, dg, dbeta and d(initial_state) from the CUDA
library against the fp64 hand-written reverse mode of the oracle, on the same seeded
inputs (relative L2 <= 1e-2 and max-abs <= 2e-2 per tensor)."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, errors, mixed_decay_problem, run_bwd

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import linear_attention_varlen_gb300 as gdn  # noqa: E402

KEYS = ("dq", "dk", "dv", "dg", "dbeta")


# Stress inputs outside the workloads' distributions (an elementwise N(0, 1) gradient of the
# final state, a decay 30x slower than the workloads') inflate every gradient 10-30x. The
# absolute max-abs bound is stated for the workloads; these tests keep the relative-L2 bound
# and bound the largest error relative to the largest reference entry instead.
STRESS_MAX_REL = 5e-3


def check_bwd(p, options=None, record=None, stress=False):
    got = run_bwd(p, options)
    ref = oracle.bwd_problem(p)
    res = {}
    keys = KEYS + (("dinit",) if p.initial_state is not None else ())
    for key in keys:
        rel, mx = errors(got[key], ref[key])
        print(f"ERRS {p.name} {key} rel={rel:.3e} maxabs={mx:.3e} maxref={np.abs(ref[key]).max():.3e}")
    for key in keys:
        if stress:
            rel, mx = errors(got[key], ref[key])
            mref = float(np.abs(ref[key]).max())
            assert rel <= 1e-2 and mx <= STRESS_MAX_REL * max(mref, 1.0), f"{p.name} {key}: {rel:.3e} {mx:.3e}"
            res[key] = (rel, mx)
        else:
            res[key] = assert_close(f"{p.name} {key}", got[key], ref[key])
    if record is not None:
        for k, (rel, mx) in res.items():
            record(f"{k}_rel_l2", rel)
            record(f"{k}_max_abs", mx)
    return got, ref


@pytest.mark.parametrize("T", [1, 7, 64, 65, 200])
@pytest.mark.parametrize("Hk,Hv", [(1, 1), (2, 8), (1, 4)])
def test_bwd_single_document_shapes(T, Hk, Hv):
    p = synth.make_problem(f"bwd_T{T}", 300 + T, [T], Hk, Hv, with_dout=True)
    check_bwd(p)


def test_bwd_final_state_gradient():
    p = synth.make_problem("bwd_dfinal", 311, [130, 64], 2, 4, with_dout=True, with_dfinal=True)
    check_bwd(p, stress=True)


def test_bwd_packed_ragged_documents():
    lens = [1, 0, 64, 5, 129, 0, 63, 300, 2]
    p = synth.make_problem("bwd_ragged", 312, lens, 2, 4, with_dout=True)
    check_bwd(p)


def test_bwd_pool_states_shared_and_forks():
    """Two documents share pool entry 0 (their d(initial state) add up), one forks another;
    with an elementwise N(0, 1) final-state gradient (stress bound)."""
    lens = [70, 0, 130, 64, 9, 200]
    init = [1, 0, 3, 0, 5, -1]
    p = synth.make_problem("bwd_forks", 313, lens, 2, 4, init_idx=init, n_init=2, with_dout=True, with_dfinal=True)
    check_bwd(p, stress=True)


def test_bwd_fork_gradient_sums_into_prefix():
    p = synth.workload_fork(prefix=512, n_branch=3, lo=100, hi=300, Hk=1, Hv=2)
    p.dout = synth.to_bf16_bits(synth.normal(7, 99, p.T * p.Hv * 128).reshape(p.T, p.Hv, 128))
    check_bwd(p)


@pytest.mark.parametrize("seg", [2, 5])
def test_bwd_with_split_recompute(seg):
    p = synth.make_problem(f"bwd_split{seg}", 320 + seg, [64 * 13 + 9], 2, 4, with_dout=True, g_mean=5.0)
    check_bwd(p, gdn.Options(segment_chunks=seg))


def test_bwd_slow_decay_long():
    p = synth.make_problem("bwd_slow", 330, [2048], 1, 2, with_dout=True, g_mean=6.0)
    check_bwd(p, stress=True)


def test_bwd_deterministic():
    p = synth.make_problem("bwd_det", 340, [700, 300], 2, 8, with_dout=True)
    a = run_bwd(p)
    b = run_bwd(p)
    for key in KEYS:
        np.testing.assert_array_equal(a[key], b[key])


def test_bwd_workload_train_full(record_property):
    """Full-size training step: 4 documents x 16384 tokens, 8 value heads over 2 key heads."""
    check_bwd(synth.workload_train(), record=record_property)


def test_bwd_split_document_with_forks():
    """A document split into segments whose final state two later (also split) documents fork
    from: its last segment's end gradient waits for the forks' start gradients."""
    lens = [64 * 10 + 5, 64 * 7, 300]
    p = synth.make_problem("bwd_split_forks", 350, lens, 2, 4, init_idx=[-1, 0, 0], with_dout=True)
    check_bwd(p, gdn.Options(segment_chunks=3))


def test_bwd_split_zero_transitions():
    """A decay fast enough that segment transitions are exactly zero in fp32: the reverse split
    takes the local start gradient without waiting for the next segment."""
    p = synth.make_problem("bwd_fast_decay", 351, [64 * 12 + 17, 64 * 9], 1, 2, with_dout=True, g_mean=-3.0)
    check_bwd(p, gdn.Options(segment_chunks=2))


@pytest.mark.parametrize("boost", [None, 3.0])
def test_bwd_split_mixed_decay(boost):
    """Reverse split over regimes that warm up and regimes that wait for a publication."""
    p = mixed_decay_problem(f"bwd_mixed_b{boost}", 360, with_dout=True, beta_boost=boost)
    check_bwd(p, gdn.Options(segment_chunks=3), stress=True)


def test_bwd_ignores_truncation_mode():
    """The backward is that of the exact forward whatever the mode option says."""
    p = synth.make_problem("bwd_trunc_opt", 352, [64 * 20 + 3], 1, 2, with_dout=True)
    a = run_bwd(p, gdn.Options(segment_chunks=4))
    b = run_bwd(p, gdn.Options(segment_chunks=4, mode="truncate"))
    for key in KEYS:
        np.testing.assert_array_equal(a[key], b[key])


def test_bwd_workload_long_full(record_property):
    """Full-size long prefill shape: one 32768-token document, 8 value heads over 2 key heads,
    automatic exact split in both directions."""
    p = synth.make_problem("bwd_long_T32768_H8", synth.SEEDS[2], [32768], 2, 8, with_dout=True)
    check_bwd(p, record=record_property)
