"""The q scale of the boundary (gdn_options.scale) on the GPU: q enters unscaled (unit norm per
token and head) and the library applies scale = fp32(1/sqrt(128)) itself, in the forward (the
intra-chunk P and the inter-chunk Q~), the recomputing backward and the training step. The fp64
oracle runs on q multiplied by that same fp32 value; dq is the gradient with respect to the
unscaled input, i.e. scale times the oracle's gradient with respect to the scaled q ("Using it,
and the fine print" on "How to Speed Up GDN Kernels for Qwen Models": the drop-in call takes a
scale argument). Tolerances as everywhere: relative L2 <= 1e-2 and max-abs <= 2e-2."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, run_bwd, run_fwd, run_train

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import linear_attention_varlen_gb300 as gdn  # noqa: E402

SCALE = float(np.float32(1.0 / np.sqrt(128.0)))
KEYS = ("dq", "dk", "dv", "dg", "dbeta")


def unscaled_problem(name, seed, lengths, Hk=2, Hv=8, **kw):
    return synth.make_problem(name, seed, lengths, Hk, Hv, with_dout=True, q_scale=1.0, **kw)


def oracle_scaled(p):
    f = p.as_f64()
    q = f["q"] * SCALE
    out, fin = oracle.fwd(q, f["k"], f["v"], f["g"], f["beta"], p.cu_seqlens, p.init_idx, f.get("initial_state"))
    gr = oracle.bwd(q, f["k"], f["v"], f["g"], f["beta"], p.cu_seqlens, f["dout"], f.get("dfinal"), p.init_idx,
                    f.get("initial_state"))
    gr["dq"] = gr["dq"] * SCALE  # the gradient with respect to the unscaled input
    return out, fin, gr


@pytest.fixture(scope="module")
def problems():
    # ragged documents, a fork and a split document (short segments), GQA 4:2
    a = unscaled_problem("scale_fork", 1301, [300, 0, 129, 200], init_idx=[-1, -1, 0, 2], n_init=0)
    b = unscaled_problem("scale_long", 1302, [64 * 30 + 7], Hk=1, Hv=2)
    return [(a, None), (b, 6)]


def test_q_scale_unit_norm_q(problems):
    # the unscaled q really is unit norm: scale = 1 would give outputs about 11x too large
    p, _ = problems[0]
    qn = np.linalg.norm(p.as_f64()["q"], axis=-1)
    assert np.allclose(qn, 1.0, atol=1e-2)


@pytest.mark.parametrize("which", [0, 1])
def test_forward_with_scale(problems, which):
    p, seg = problems[which]
    opts = gdn.Options(scale=SCALE, segment_chunks=seg or 0)
    out, fin = run_fwd(p, opts)
    ro, rf, _ = oracle_scaled(p)
    assert_close(f"{p.name} out", out, ro)
    assert_close(f"{p.name} final_state", fin, rf)
    # the scale is not applied twice nor left out: scale 1 on the same q is far off
    out1, _ = run_fwd(p, gdn.Options(segment_chunks=seg or 0))
    assert np.abs(out1 - ro).max() > 10 * 2e-2


@pytest.mark.parametrize("which", [0, 1])
def test_recomputing_backward_with_scale(problems, which):
    p, seg = problems[which]
    got = run_bwd(p, gdn.Options(scale=SCALE, segment_chunks=seg or 0))
    _, _, ref = oracle_scaled(p)
    for key in KEYS:
        assert_close(f"{p.name} {key}", got[key], ref[key])


@pytest.mark.parametrize("which", [0, 1])
def test_training_step_with_scale(problems, which):
    p, seg = problems[which]
    out, fin, got = run_train(p, gdn.Options(scale=SCALE, segment_chunks=seg or 0))
    ro, rf, ref = oracle_scaled(p)
    assert_close(f"{p.name} train out", out, ro)
    assert_close(f"{p.name} train final_state", fin, rf)
    for key in KEYS:
        assert_close(f"{p.name} train {key}", got[key], ref[key])
