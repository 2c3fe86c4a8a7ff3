"""The width-4 causal convolution on the GPU (gdn_conv_fwd / gdn_conv_bwd) against the fp64 oracle
(oracle/conv.py) on the same seeded inputs: every gradient (fp32) at relative L2 <= 1e-2 and max-abs
<= 2e-2, the final tails bit-exact (they are copies of inputs). y is rounded once to bf16, and its
magnitude follows the weights (unlike the recurrence's outputs, which stay near 1): half an ulp of
|y| >= 8 is already 2^-5, so y keeps relative L2 <= 1e-2 with max-abs <= max(2e-2, 2^-8 max|ref|),
one bf16 ulp of the largest output. Layouts: packed lognormal documents,
a shared prefix forked by several continuations ("Musings on long-context fine-tuning", sections
"Isolating the recurrent layers" and "Backward through P"), pool starts, empty and short documents."""
import numpy as np
import pytest

import oracle.conv as oc
import synth
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import linear_attention_varlen_gb300 as gdn  # noqa: E402


def conv_case(seed, lengths, C, init_idx=None, n_init=0, with_bias=True, with_dtail=False):
    """x, dy ~ N(0, 1) rounded to bf16; w ~ N(0, 1/4), bias ~ N(0, 1/10) in fp32; pool starts are bf16
    inputs; the final-tail gradient N(0, 1) in fp32."""
    T = int(sum(lengths))
    bf = lambda stream, n: synth.bf16_bits_to_f32(synth.to_bf16_bits(synth.normal(seed, stream, n)))
    c = dict(x=bf(11, T * C).reshape(T, C), dy=bf(12, T * C).reshape(T, C),
             w=(0.5 * synth.normal(seed, 13, C * 4)).astype(np.float32).reshape(C, 4),
             bias=(0.1 * synth.normal(seed, 14, C)).astype(np.float32) if with_bias else None,
             cu=np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32),
             init_idx=None if init_idx is None else np.asarray(init_idx, dtype=np.int32),
             conv_init=bf(15, n_init * 3 * C).reshape(n_init, 3, C) if n_init else None,
             dtail=synth.normal(seed, 16, len(lengths) * 3 * C).astype(np.float32).reshape(len(lengths), 3, C)
             if with_dtail else None)
    return c


def on_device(c):
    to_bf = lambda a: torch.from_numpy(synth.to_bf16_bits(a)).view(torch.bfloat16).cuda()
    f32 = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    return dict(x=to_bf(c["x"]), dy=to_bf(c["dy"]), w=f32(c["w"]), bias=f32(c["bias"]),
                cu=torch.from_numpy(c["cu"]).cuda(),
                init_idx=None if c["init_idx"] is None else torch.from_numpy(c["init_idx"]).cuda(),
                conv_init=None if c["conv_init"] is None else to_bf(c["conv_init"]), dtail=f32(c["dtail"]))


def run_and_check(c, backward=True):
    d = on_device(c)
    y, tail = gdn.conv_fwd(d["x"], d["w"], d["cu"], d["bias"], d["init_idx"], d["conv_init"])
    ws = torch.empty(gdn.conv_workspace_size(len(c["cu"]) - 1, c["x"].shape[0], c["x"].shape[1], True),
                     dtype=torch.uint8, device="cuda")
    g = gdn.conv_bwd(d["x"], d["w"], d["cu"], d["dy"], d["bias"], d["init_idx"], d["conv_init"], d["dtail"],
                     workspace=ws) if backward else None
    torch.cuda.synchronize()
    assert gdn.workspace_status(ws) == gdn.GDN_OK if backward else True
    ry, rt = oc.conv_fwd(c["x"], c["w"], c["bias"], c["cu"], c["init_idx"], c["conv_init"])
    assert_close("conv y", y.double().cpu().numpy(), ry, max_abs=max(2e-2, 2.0 ** -8 * float(np.abs(ry).max())))
    np.testing.assert_array_equal(tail.float().cpu().numpy(), rt.astype(np.float32))
    if backward:
        rg = oc.conv_bwd(c["x"], c["w"], c["bias"], c["cu"], c["dy"], c["dtail"], c["init_idx"], c["conv_init"])
        assert_close("conv dx", g["dx"].double().cpu().numpy(), rg["dx"])
        assert_close("conv dw", g["dw"].double().cpu().numpy(), rg["dw"])
        if c["bias"] is not None:
            assert_close("conv dbias", g["dbias"].double().cpu().numpy(), rg["dbias"])
        if c["conv_init"] is not None:
            assert_close("conv dconv_init", g["dconv_init"].double().cpu().numpy(), rg["dinit"])


@pytest.mark.parametrize("T,C", [(1, 8), (3, 16), (130, 264), (1000, 1536)])
def test_one_document(T, C):
    run_and_check(conv_case(2200 + T, [T], C))


def test_packed_lognormal_documents():
    run_and_check(conv_case(2210, synth.lognormal_lengths(2210, 12, 4096), 1536))


def test_shared_prefix_with_continuations():
    """One prefix forked by ten continuations (one of them empty, one shorter than the tail), with
    gradients on the final tails: every continuation's start is the prefix's last three inputs, and
    their gradients sum into those inputs."""
    lens = [700] + [60, 0, 2, 129, 64, 300, 1, 3, 90, 41]
    ii = [-1] + [0] * 10
    run_and_check(conv_case(2211, lens, 264, init_idx=ii, with_dtail=True))


def test_pool_starts_forks_of_forks_and_short_documents():
    lens = [5, 2, 0, 4, 1, 130, 7]
    ii = [1, 0, 2, 3, 4, 6, -1]  # n_init = 2: pool 1, pool 0, forks of 0, 1, the empty 2, the one-token 4, zeros
    run_and_check(conv_case(2212, lens, 136, init_idx=ii, n_init=2, with_dtail=True))


def test_without_bias():
    run_and_check(conv_case(2213, [300, 200], 64, with_bias=False))


def test_two_calls_equal_one_packed_call():
    """The prefix alone, then its continuations with conv_init = the prefix's final tail, gives the
    packed call's outputs; the continuations' d(conv_init) fed back as the prefix's d(final tail)
    gives the packed call's gradient on the prefix."""
    lens = [500, 100, 37, 2]
    c = conv_case(2214, lens, 264, init_idx=[-1, 0, 0, 0])
    d = on_device(c)
    y, _ = gdn.conv_fwd(d["x"], d["w"], d["cu"], d["bias"], d["init_idx"])
    g = gdn.conv_bwd(d["x"], d["w"], d["cu"], d["dy"], d["bias"], d["init_idx"])
    P = 500
    cu_p = torch.tensor([0, P], dtype=torch.int32, device="cuda")
    cu_c = torch.tensor([0, 100, 137, 139], dtype=torch.int32, device="cuda")
    yp, tp = gdn.conv_fwd(d["x"][:P].contiguous(), d["w"], cu_p, d["bias"])
    zero = torch.zeros(3, dtype=torch.int32, device="cuda")
    yc, _ = gdn.conv_fwd(d["x"][P:].contiguous(), d["w"], cu_c, d["bias"], zero, tp)
    gc = gdn.conv_bwd(d["x"][P:].contiguous(), d["w"], cu_c, d["dy"][P:].contiguous(), d["bias"], zero, tp)
    gp = gdn.conv_bwd(d["x"][:P].contiguous(), d["w"], cu_p, d["dy"][:P].contiguous(), d["bias"],
                      dfinal_tail=gc["dconv_init"])
    assert torch.equal(y[:P], yp) and torch.equal(y[P:], yc)
    assert_close("prefix dx", gp["dx"].double().cpu().numpy(), g["dx"][:P].double().cpu().numpy())
    assert_close("continuation dx", gc["dx"].double().cpu().numpy(), g["dx"][P:].double().cpu().numpy())


def test_invalid_layout_is_reported_on_device():
    c = conv_case(2215, [40, 30], 64)
    d = on_device(c)
    d["cu"] = torch.tensor([0, 50, 40], dtype=torch.int32, device="cuda")  # not monotone (and cu[N] != T)
    ws = torch.empty(gdn.conv_workspace_size(2, 70, 64), dtype=torch.uint8, device="cuda")
    gdn.conv_fwd(d["x"], d["w"], d["cu"], d["bias"], workspace=ws)
    assert gdn.workspace_status(ws) == gdn.GDN_ERR_INVALID_ARG
