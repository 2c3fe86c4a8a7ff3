"""A bounded device-side wait that runs out: with the test hook GDN_FLAG_TEST_WITHHOLD_FORK no
document publishes its final state, so the document forked from it waits for a flag that nothing
sets. Its wait gives up after gdn_options.flag_wait_us, the kernel drains its own copies and tensor
work, frees its tensor memory and returns; the host reads GDN_ERR_TIMEOUT from the status word.
The GPU stays usable: the next ordinary call on it matches the oracle. Nothing here faults, traps
or hangs the GPU: every wait involved is bounded."""
import time

import pytest

import oracle
import synth
from tests.gpu_util import assert_close, bf16_to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import linear_attention_varlen_gb300 as gdn  # noqa: E402


@pytest.mark.parametrize("mode", ["exact", "truncate"])
def test_withheld_fork_state_times_out_and_the_gpu_recovers(mode):
    p = synth.make_problem("timeout", 1401, [200, 100, 64], 1, 2, init_idx=[-1, 0, -1])  # document 1 forks 0
    d = synth.to_device(p)
    ws = torch.empty(gdn.fwd_workspace_size(p.N, p.T, p.Hk, p.Hv), dtype=torch.uint8, device="cuda")
    hook = gdn.Options(mode=mode, test_withhold_fork=True, flag_wait_us=20000)  # 20 ms
    t0 = time.perf_counter()
    gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_idx"], options=hook,
                  workspace=ws)
    st = gdn.workspace_status(ws)
    waited = time.perf_counter() - t0
    assert st == gdn.GDN_ERR_TIMEOUT, gdn.status_string(st)
    assert waited < 10.0
    # the same GPU, the same workspace: an ordinary call succeeds and is correct
    out, fin = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_idx"],
                             options=gdn.Options(mode=mode), workspace=ws)
    assert gdn.workspace_status(ws) == gdn.GDN_OK
    ro, rf = oracle.fwd_problem(p)
    assert_close("after timeout out", bf16_to_f64(out), ro)
    assert_close("after timeout final_state", fin.double().cpu().numpy(), rf)


def test_backward_rejects_the_test_hook():
    p = synth.make_problem("timeout_b", 1402, [70], 1, 2, with_dout=True)
    d = synth.to_device(p)
    with pytest.raises(gdn.GdnError) as e:
        gdn.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["dout"],
                      options=gdn.Options(test_withhold_fork=True))
    assert e.value.status == gdn.GDN_ERR_INVALID_ARG
