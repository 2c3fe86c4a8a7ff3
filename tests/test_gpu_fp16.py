"""fp16 inputs on the GPU (GDN_FLAG_FP16_INPUTS, set by the binding from the tensors' dtype): the
workloads' draws rounded to IEEE fp16 instead of bf16 ("How to Speed Up GDN Kernels for Qwen
Models", "Using it, and the fine print": bf16 or fp16 inputs). The fp64 oracle runs on the exact fp16
values; the library rounds each input once to bf16 for its matrix operands.

Tolerances: the stated ones (relative L2 <= 1e-2, max-abs <= 2e-2) are for bf16 inputs, which the
operands carry exactly. With fp16 inputs every q, k, v and dO element moves by up to 2^-9 of itself
before any arithmetic, and the whole computation inherits that perturbation. o and the final states
(magnitudes near 1) keep both bounds. The gradients keep relative L2 <= 1e-2; their max-abs bound is
max(2e-2, 2^-7 max|ref|): four input-rounding units of conditioning on the largest entry (dq reaches
about 20 at the workloads' distributions, so 2^-9 of it alone is 0.04)."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, bf16_to_f64, run_bwd, run_fwd, run_train

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import linear_attention_varlen_gb300 as gdn  # noqa: E402

KEYS = ("dq", "dk", "dv", "dg", "dbeta")
GRAD_REL = 2.0 ** -7  # max-abs of a gradient relative to its largest reference entry


def assert_grad_close(name, got, ref):
    return assert_close(name, got, ref, max_abs=max(2e-2, GRAD_REL * float(np.abs(ref).max())))


def f16_problem(name, seed, lengths, Hk=2, Hv=8, **kw):
    return synth.make_problem(name, seed, lengths, Hk, Hv, with_dout=True, dtype="f16", **kw)


@pytest.fixture(scope="module")
def problems():
    return [(f16_problem("f16_fork", 2101, [300, 0, 129, 200], init_idx=[-1, -1, 0, 2]), 0),
            (f16_problem("f16_long", 2102, [64 * 30 + 7], Hk=1, Hv=2, g_mean=5.0), 6),
            (synth.make_problem("f16_packed", 2103, synth.lognormal_lengths(2103, 12, 4096), 2, 8, with_dout=True,
                                dtype="f16"), 0)]


def test_inputs_are_fp16(problems):
    p, _ = problems[0]
    d = synth.to_device(p)
    assert d["q"].dtype == torch.float16 and d["v"].dtype == torch.float16 and d["dout"].dtype == torch.float16
    # the values are not all representable in bf16: the fp16 draws carry more mantissa bits
    x = p.as_f64()["v"].astype(np.float32)
    assert np.any(synth.bf16_bits_to_f32(synth.to_bf16_bits(x)) != x)


@pytest.mark.parametrize("which", [0, 1, 2])
def test_forward(problems, which):
    p, seg = problems[which]
    out, fin = run_fwd(p, gdn.Options(segment_chunks=seg))
    ro, rf = oracle.fwd_problem(p)
    assert_close(f"{p.name} out", out, ro)
    assert_close(f"{p.name} final_state", fin, rf)


@pytest.mark.parametrize("which", [0, 1])
def test_backward(problems, which):
    p, seg = problems[which]
    got = run_bwd(p, gdn.Options(segment_chunks=seg))
    ref = oracle.bwd_problem(p)
    for key in KEYS:
        assert_grad_close(f"{p.name} {key}", got[key], ref[key])


def test_training_step(problems):
    p, seg = problems[0]
    out, fin, got = run_train(p, gdn.Options(segment_chunks=seg))
    ro, rf = oracle.fwd_problem(p)
    ref = oracle.bwd_problem(p)
    assert_close("train out", out, ro)
    assert_close("train final_state", fin, rf)
    for key in KEYS:
        assert_grad_close(f"train {key}", got[key], ref[key])


def test_fp16_with_normalisation():
    scale = float(np.float32(1.0 / np.sqrt(128.0)))
    p = f16_problem("f16_l2", 2104, [200, 77], q_scale=1.0)
    r = np.random.default_rng(2104)
    for attr in ("q", "k"):
        x = synth.f16_bits_to_f32(getattr(p, attr)).astype(np.float64) * r.uniform(0.25, 4.0, (p.T, p.Hk, 1))
        setattr(p, attr, synth.to_f16_bits(x))
    opts = gdn.Options(scale=scale, l2norm_qk=True)
    out, fin = run_fwd(p, opts)
    got = run_bwd(p, opts)
    f = p.as_f64()
    qn, kn = oracle.l2norm_rows(f["q"]), oracle.l2norm_rows(f["k"])
    ro, rf = oracle.fwd(qn * scale, kn, f["v"], f["g"], f["beta"], p.cu_seqlens)
    ref = oracle.bwd(qn * scale, kn, f["v"], f["g"], f["beta"], p.cu_seqlens, f["dout"])
    ref["dq"] = oracle.l2norm_rows_bwd(f["q"], ref["dq"] * scale)
    ref["dk"] = oracle.l2norm_rows_bwd(f["k"], ref["dk"])
    assert_close("f16+l2 out", out, ro)
    assert_close("f16+l2 final_state", fin, rf)
    for key in KEYS:
        assert_grad_close(f"f16+l2 {key}", got[key], ref[key])


def test_decode_fp16():
    B, n_pool = 21, 40
    idx = np.random.default_rng(2105).choice(n_pool, size=B, replace=False).astype(np.int32)
    p = f16_problem("f16_decode", 2105, [1] * B, init_idx=list(idx), n_init=n_pool)
    d = synth.to_device(p)
    pool = d["initial_state"].clone()
    out = gdn.decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, d["init_idx"])
    ro, rf = oracle.fwd_problem(p)
    assert_close("decode f16 out", bf16_to_f64(out), ro)
    assert_close("decode f16 states", pool.double().cpu().numpy()[idx], rf)


def test_mixed_dtypes_are_refused(problems):
    p, _ = problems[0]
    d = synth.to_device(p)
    with pytest.raises(ValueError):
        gdn.chunk_fwd(d["q"], d["k"], d["v"].to(torch.bfloat16), d["g"], d["beta"], d["cu_seqlens"], d["init_idx"])
