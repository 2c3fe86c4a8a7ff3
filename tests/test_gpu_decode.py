"""Decode on the GPU (gdn_decode_step): B sequences advance by one token each, in place on a pool
of states. The fp64 oracle sees the same step as B one-token documents whose initial states are
the pool entries; their final states are the updated entries ("How to Speed Up GDN Kernels for
Qwen Models", FAQ "Does this help decode too?"). Tolerances as everywhere: relative L2 <= 1e-2 and
max-abs <= 2e-2; pool entries that no sequence names must not change at all."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, bf16_to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import linear_attention_varlen_gb300 as gdn  # noqa: E402

N_POOL = 50


def decode_problem(seed, B, steps, Hk=2, Hv=8, q_scale=None):
    """B sequences of `steps` tokens each (packed sequence-major), starting from distinct pool entries."""
    rng = np.random.default_rng(seed)
    idx = rng.choice(N_POOL, size=B, replace=False).astype(np.int32)
    p = synth.make_problem(f"decode_{seed}", seed, [steps] * B, Hk, Hv, init_idx=list(idx), n_init=N_POOL,
                           q_scale=q_scale)
    return p, idx


def step_inputs(d, p, j):
    """Token j of every sequence, as contiguous [B, ...] device tensors."""
    rows = torch.from_numpy(p.cu_seqlens[:-1].astype(np.int64) + j).to("cuda")
    return [d[x].index_select(0, rows).contiguous() for x in ("q", "k", "v", "g", "beta")]


@pytest.mark.parametrize("B,Hk,Hv", [(1, 1, 1), (37, 2, 8), (5, 4, 4)])
def test_single_step_matches_oracle(B, Hk, Hv):
    p, idx = decode_problem(1500 + B, B, 1, Hk, Hv)
    d = synth.to_device(p)
    pool = d["initial_state"].clone()
    before = pool.clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gdn.decode_step(*step_inputs(d, p, 0), pool, d["init_idx"], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ro, rf = oracle.fwd_problem(p)
    assert_close("decode out", bf16_to_f64(out), ro)
    got = pool.double().cpu().numpy()
    assert_close("decode states", got[idx], rf)
    untouched = np.setdiff1d(np.arange(N_POOL), idx)
    assert torch.equal(pool[torch.from_numpy(untouched).cuda()], before[torch.from_numpy(untouched).cuda()])


def test_steps_in_a_row_equal_the_recurrence_over_the_tokens():
    """Six decode steps per sequence equal the oracle's run over the six tokens (outputs of every
    step, final states), and the chunked forward over the same documents."""
    B, steps = 23, 6
    p, idx = decode_problem(1601, B, steps)
    d = synth.to_device(p)
    pool = d["initial_state"].clone()
    outs = []
    for j in range(steps):
        outs.append(bf16_to_f64(gdn.decode_step(*step_inputs(d, p, j), pool, d["init_idx"])))
    torch.cuda.synchronize()
    ro, rf = oracle.fwd_problem(p)
    for j in range(steps):
        assert_close(f"decode step {j}", outs[j], ro[p.cu_seqlens[:-1] + j])
    assert_close("decode final states", pool.double().cpu().numpy()[idx], rf)
    co, cf = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_idx"],
                           d["initial_state"])
    assert_close("chunked forward final states", cf.double().cpu().numpy(), rf)
    assert_close("decode vs chunked final states", pool.double().cpu().numpy()[idx], cf.double().cpu().numpy())


def test_scale_option_applies_to_q():
    scale = float(np.float32(1.0 / np.sqrt(128.0)))
    p, idx = decode_problem(1701, 17, 1, q_scale=1.0)
    d = synth.to_device(p)
    pool = d["initial_state"].clone()
    out = gdn.decode_step(*step_inputs(d, p, 0), pool, d["init_idx"], options=gdn.Options(scale=scale))
    f = p.as_f64()
    ro, rf = oracle.fwd(f["q"] * scale, f["k"], f["v"], f["g"], f["beta"], p.cu_seqlens, p.init_idx,
                        f["initial_state"])
    assert_close("decode out with scale", bf16_to_f64(out), ro)
    assert_close("decode states with scale", pool.double().cpu().numpy()[idx], rf)


def test_out_of_range_index_is_skipped_and_reported():
    p, idx = decode_problem(1801, 9, 1)
    d = synth.to_device(p)
    bad = d["init_idx"].clone()
    bad[3] = N_POOL + 7
    pool = d["initial_state"].clone()
    before = pool.clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gdn.decode_step(*step_inputs(d, p, 0), pool, bad, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == gdn.GDN_ERR_INVALID_ARG
    assert float(out[3].float().abs().max()) == 0.0
    ro, rf = oracle.fwd_problem(p)
    keep = [b for b in range(9) if b != 3]
    assert_close("decode out, valid rows", bf16_to_f64(out)[keep], ro[keep])
    assert_close("decode states, valid rows", pool.double().cpu().numpy()[idx[keep]], rf[keep])
    assert torch.equal(pool[int(idx[3])], before[int(idx[3])])


def test_empty_batch_is_a_no_op():
    z = lambda *s, dt=torch.bfloat16: torch.zeros(s, dtype=dt, device="cuda")
    pool = torch.ones((2, 8, 128, 128), dtype=torch.float32, device="cuda")
    out = gdn.decode_step(z(0, 2, 128), z(0, 2, 128), z(0, 8, 128), z(0, 8, dt=torch.float32),
                          z(0, 8, dt=torch.float32), pool, z(0, dt=torch.int32))
    assert out.shape == (0, 8, 128) and bool((pool == 1).all())
