"""Failure detection on the GPU without a fault: a task waits on a count that
nothing will reach; the wait gives up after the watchdog limit, the kernel
returns, mk_check_step reports MK_ERR_TIMEOUT with the stalled wait, and the
context stays usable for the next step."""
import numpy as np
import pytest
import torch

import synth
import synth.device
import moe_decode_megakernel_gb300 as mk
import parity

pytestmark = pytest.mark.gpu


def test_unsatisfiable_wait_times_out_and_context_survives():
    inp = synth.make_inputs("tiny")
    w = inp.workload
    sh = w.shape
    model = parity._device_model(sh, w.seed, None)
    sched = mk.Sched(model, 1, 64, mk.default_sched_opts(watchdog_ms=200))
    # one QKV task waits for one arrival more than its RMSNorm will ever give
    victim = None
    for sm in range(sched.num_sms):
        for i in range(sched.num_tasks(sm)):
            d = sched.get_task(sm, i)
            if d[mk.F_OP] == 2 and d[mk.F_LAYER] == 1:
                victim = (sm, i, d.copy())
                break
        if victim:
            break
    sm, i, d = victim
    d[mk.F_TGT0] += 1
    sched.set_task(sm, i, d)
    sess = mk.Session(model, sched)  # uploads the altered lists
    kp, vp = synth.device.device_pools(sh, w.seed, inp.num_pages)
    dev = "cuda"
    tok = torch.as_tensor(inp.tokens, device=dev)
    sl = torch.as_tensor(inp.seq_lens, device=dev)
    bt = torch.as_tensor(inp.block_tables, device=dev)
    logits = torch.empty(1, sh.vocab, device=dev)
    sess.step(tok, sl, bt, kp, vp, logits)
    with pytest.raises(mk.MkError) as e:
        sess.check()
    assert e.value.code == mk.MK_ERR_TIMEOUT
    # the first wait to give up may be the victim's or one stalled behind it;
    # the diagnosis against the schedule names the victim as the root
    msg = str(e.value)
    assert f"root: task {d[mk.F_TASK]} " in msg and f"on barrier {d[mk.F_WAIT0]}," in msg, msg
    # the context is intact: a correct schedule runs and matches the oracle
    good = parity.run_gpu(inp)
    rep = parity.compare(inp, good)
    assert rep.max_rel_err <= parity.LOGIT_TOL


def test_page_id_out_of_range_is_reported():
    """A block table naming a page past the pool is refused on the device (the
    copy is skipped and recorded), not read out of bounds."""
    inp = synth.make_inputs("tiny")
    w = inp.workload
    sh = w.shape
    model = parity._device_model(sh, w.seed, None)
    sched = mk.Sched(model, 1, 64)
    sess = mk.Session(model, sched)
    kp, vp = synth.device.device_pools(sh, w.seed, inp.num_pages)
    bt = inp.block_tables.copy()
    bt[0, 1] = inp.num_pages + 5
    dev = "cuda"
    logits = torch.empty(1, sh.vocab, device=dev)
    sess.step(torch.as_tensor(inp.tokens, device=dev), torch.as_tensor(inp.seq_lens, device=dev),
              torch.as_tensor(bt, device=dev), kp, vp, logits)
    with pytest.raises(mk.MkError) as e:
        sess.check()
    assert e.value.code == mk.MK_ERR_DEVICE and "page id" in str(e.value)
