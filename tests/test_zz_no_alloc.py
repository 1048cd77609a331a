"""The decode step on the library's built-in workspace (for callers that
cannot allocate device memory) gives what mk_decode_step gives with a
caller-allocated workspace, call after call, and refuses schedules that do
not fit its 8 MiB.  Collected last: it shares nothing with the other tests
but the cached device model."""
import numpy as np
import pytest
import torch

import synth
import synth.device
import moe_decode_megakernel_gb300 as mk
import parity

pytestmark = pytest.mark.gpu


def _inputs_on_device(inp):
    dev = "cuda"
    return (torch.as_tensor(inp.tokens, device=dev), torch.as_tensor(inp.seq_lens, device=dev),
            torch.as_tensor(inp.block_tables, device=dev))


@pytest.mark.parametrize("workload", ["small", "full_bs1_8k"])
def test_built_in_workspace_matches_caller_workspace(workload):
    inp = synth.make_inputs(workload)
    w = inp.workload
    sh = w.shape
    model = parity._device_model(sh, w.seed, inp.router_bias)
    sched = mk.Sched(model, w.batch, int(inp.seq_lens.max()))
    assert sched.workspace_bytes() <= 8 << 20
    sess = mk.Session(model, sched)  # uploads the task lists; its workspace gives the reference
    kp, vp = synth.device.device_pools(sh, w.seed, inp.num_pages)
    tok, sl, bt = _inputs_on_device(inp)
    ref = torch.empty(w.batch, sh.vocab, dtype=torch.float32, device="cuda")
    sess.step(tok, sl, bt, kp, vp, ref)
    sess.check()
    ref = ref.cpu().numpy()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):  # the array keeps the previous call's contents
        out = torch.full((w.batch, sh.vocab), float("nan"), dtype=torch.float32, device="cuda")
        mk.decode_step_static_ws(model, sched, tok.data_ptr(), sl.data_ptr(), bt.data_ptr(), w.batch,
                                 bt.shape[1], kp.data_ptr(), vp.data_ptr(), inp.num_pages,
                                 out.data_ptr(), stream)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got))
        err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
        assert err <= parity.LOGIT_TOL, err
        assert np.array_equal(got, ref)  # the same kernel on the same inputs


def test_built_in_workspace_refuses_large_schedules():
    inp = synth.make_inputs("small")
    w = inp.workload
    model = parity._device_model(w.shape, w.seed, inp.router_bias)
    big = mk.Sched(model, 64, 262144)
    assert big.workspace_bytes() > 8 << 20
    dev = "cuda"
    z = torch.zeros(64, dtype=torch.int32, device=dev)
    out = torch.empty(64, w.shape.vocab, dtype=torch.float32, device=dev)
    with pytest.raises(mk.MkError) as e:
        mk.decode_step_static_ws(model, big, z.data_ptr(), z.data_ptr(), z.data_ptr(), 64, 1,
                                 z.data_ptr(), z.data_ptr(), 1, out.data_ptr(), 0)
    assert e.value.code == mk.MK_ERR_ARG and "8388608" in str(e.value)
