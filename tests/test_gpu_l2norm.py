"""q / k L2 normalisation on the GPU (GDN_FLAG_L2NORM_QK): the library receives unnormalised q and
k, scales each (token, key head) row to unit norm itself, and returns gradients with respect to the
unnormalised inputs ("Musings on long-context fine-tuning", section "Triton autotuning in the first
backward pass"). Reference: the fp64 oracle on oracle.l2norm_rows of the same inputs, and
oracle.l2norm_rows_bwd of its gradients. Tolerances as everywhere: relative L2 <= 1e-2, max-abs
<= 2e-2."""
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

SCALE = float(np.float32(1.0 / np.sqrt(128.0)))
KEYS = ("dq", "dk", "dv", "dg", "dbeta")


def raw_problem(name, seed, lengths, Hk=2, Hv=8, **kw):
    """The workload's q and k with every (token, head) row multiplied by a random factor in
    [0.25, 4] (so the library's normalisation matters), rounded to bf16 again."""
    p = synth.make_problem(name, seed, lengths, Hk, Hv, with_dout=True, q_scale=1.0, **kw)
    r = np.random.default_rng(seed + 7)
    for attr in ("q", "k"):
        x = synth.bf16_bits_to_f32(getattr(p, attr)).astype(np.float64)
        x *= r.uniform(0.25, 4.0, x.shape[:2] + (1,))
        setattr(p, attr, synth.to_bf16_bits(x))
    return p


def oracle_normalised(p):
    f = p.as_f64()
    qn, kn = oracle.l2norm_rows(f["q"]), oracle.l2norm_rows(f["k"])
    out, fin = oracle.fwd(qn * SCALE, kn, f["v"], f["g"], f["beta"], p.cu_seqlens, p.init_idx, f.get("initial_state"))
    gr = oracle.bwd(qn * SCALE, kn, f["v"], f["g"], f["beta"], p.cu_seqlens, f["dout"], f.get("dfinal"), p.init_idx,
                    f.get("initial_state"))
    gr["dq"] = oracle.l2norm_rows_bwd(f["q"], gr["dq"] * SCALE)
    gr["dk"] = oracle.l2norm_rows_bwd(f["k"], gr["dk"])
    return out, fin, gr


@pytest.fixture(scope="module")
def problems():
    a = raw_problem("l2_fork", 1901, [300, 0, 129, 200], init_idx=[-1, -1, 0, 2])
    b = raw_problem("l2_long", 1902, [64 * 30 + 7], Hk=1, Hv=2)
    return [(a, 0), (b, 6)]


def test_inputs_are_not_unit_norm(problems):
    p, _ = problems[0]
    n = np.linalg.norm(p.as_f64()["q"], axis=-1)
    assert n.min() < 0.5 and n.max() > 2.0


@pytest.mark.parametrize("which", [0, 1])
def test_forward_normalises_q_and_k(problems, which):
    p, seg = problems[which]
    out, fin = run_fwd(p, gdn.Options(scale=SCALE, segment_chunks=seg, l2norm_qk=True))
    ro, rf, _ = oracle_normalised(p)
    assert_close(f"{p.name} out", out, ro)
    assert_close(f"{p.name} final_state", fin, rf)


@pytest.mark.parametrize("which", [0, 1])
def test_backward_returns_gradients_of_the_raw_inputs(problems, which):
    p, seg = problems[which]
    got = run_bwd(p, gdn.Options(scale=SCALE, segment_chunks=seg, l2norm_qk=True))
    _, _, ref = oracle_normalised(p)
    for key in KEYS:
        assert_close(f"{p.name} {key}", got[key], ref[key])


def test_training_step_with_normalisation(problems):
    p, seg = problems[0]
    out, fin, got = run_train(p, gdn.Options(scale=SCALE, segment_chunks=seg, l2norm_qk=True))
    ro, rf, ref = oracle_normalised(p)
    assert_close("train out", out, ro)
    assert_close("train final_state", fin, rf)
    for key in KEYS:
        assert_close(f"train {key}", got[key], ref[key])


def test_allocation_free_forward_with_normalisation(problems):
    import ctypes
    p, _ = problems[0]
    d = synth.to_device(p)
    lib = gdn.load()
    out = torch.empty((p.T, p.Hv, 128), dtype=torch.bfloat16, device="cuda")
    fin = torch.empty((p.N, p.Hv, 128, 128), dtype=torch.float32, device="cuda")
    o = gdn.Options(scale=SCALE, l2norm_qk=True).c()
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = lib.gdn_chunk_fwd_noalloc(P(d["q"]), P(d["k"]), P(d["v"]), P(d["g"]), P(d["beta"]), P(d["cu_seqlens"]),
                                   p.N, p.T, p.Hk, p.Hv, 128, P(d["init_idx"]), None, 0, P(out), P(fin),
                                   ctypes.byref(o), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == gdn.GDN_OK
    torch.cuda.synchronize()
    ro, rf, _ = oracle_normalised(p)
    assert_close("noalloc out", bf16_to_f64(out), ro)
    assert_close("noalloc final_state", fin.double().cpu().numpy(), rf)


def test_decode_with_normalisation():
    B, n_pool = 19, 30
    rng = np.random.default_rng(1903)
    idx = rng.choice(n_pool, size=B, replace=False).astype(np.int32)
    p = raw_problem("l2_decode", 1903, [1] * B, init_idx=list(idx), n_init=n_pool)
    d = synth.to_device(p)
    pool = d["initial_state"].clone()
    out = gdn.decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, d["init_idx"],
                          options=gdn.Options(scale=SCALE, l2norm_qk=True))
    ro, rf, _ = oracle_normalised(p)
    assert_close("decode out", bf16_to_f64(out), ro)
    assert_close("decode states", pool.double().cpu().numpy()[idx], rf)
