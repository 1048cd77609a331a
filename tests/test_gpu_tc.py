"""Batches beyond two rows run their projections and expert tiles as tcgen05
GEMM items (128 weight rows per MMA tile, the batch's activation rows as BF16
hi/lo operand rows, fp32 accumulators in TMEM): the step against the CPU
oracle at several batch sizes and raggedness, on the tiny and small shapes
("Cohere: a decode megakernel for North Mini Code", section "Tasks": the GEMM
opcodes share one tensor-core pipeline)."""
import numpy as np
import pytest

import synth
import moe_decode_megakernel_gb300 as mk
import parity

pytestmark = pytest.mark.gpu


def _ragged(model, seq_lens, seed):
    sh = synth.MODELS[model]
    w = synth.Workload(f"{model}_tc_b{len(seq_lens)}", model, len(seq_lens), ("fixed", 0), seed)
    sl = np.asarray(seq_lens, np.int32)
    bt, npages = synth.block_tables_for(sl, sh.page_size, seed, slack_pages=2)
    rng = np.random.default_rng(seed)
    tok = rng.integers(0, sh.vocab, size=len(sl)).astype(np.int32)
    return synth.StepInputs(w, tok, sl, bt, npages, None)


def _check(rep):
    assert not rep.routing_violations, rep.routing_violations
    assert rep.router_err.max() <= parity.ROUTER_TOL, rep.router_err.max()
    assert rep.weight_err <= 1e-4
    assert rep.max_rel_err <= parity.LOGIT_TOL, rep.max_rel_err
    assert rep.greedy_agree == rep.greedy_total
    assert rep.kv_max_err <= 2e-2


def test_schedule_takes_the_tensor_core_build():
    """A schedule for more than two rows carries the tcgen05 operand rows."""
    inp = _ragged("tiny", [5, 17, 40], 3)
    model = parity._device_model(inp.workload.shape, inp.workload.seed, None)
    assert mk.Sched(model, 3, 64).workspace_offset("xb") >= 0
    assert mk.Sched(model, 2, 64).workspace_offset("xb") == -1


@pytest.mark.parametrize("model,seq_lens,seed", [
    ("tiny", [5, 17, 40], 41),
    ("tiny", [1, 16, 17, 64], 42),
    ("tiny", list(range(3, 64, 8)), 43),
    ("tiny", [int(x) for x in np.random.default_rng(5).integers(1, 64, 33)], 44),
    ("small", [1024, 3, 511], 45),
    ("small", [int(x) for x in np.random.default_rng(6).integers(1, 1024, 16)], 46),
])
def test_tensor_core_items_match_oracle(model, seq_lens, seed):
    inp = _ragged(model, seq_lens, seed)
    g = parity.run_gpu(inp, mk.default_sched_opts(trace_queue=1))
    rep = parity.compare(inp, g)
    print(model, len(seq_lens), f"logit rel err {rep.max_rel_err:.2e} router err {rep.router_err.max():.2e} "
          f"routing exact {rep.exact_routing}/{rep.total_routing} ties {rep.tie_routing} kv {rep.kv_max_err:.2e}")
    _check(rep)
    assert parity.compare_queue(inp, g) == inp.workload.shape.n_layers


def test_batch_below_tc_schedule_max():
    """A tensor-core schedule built for 16 rows runs steps of 3 and of 1."""
    import torch
    for rows in ([10, 40, 64], [33]):
        inp = _ragged("tiny", rows, 47)
        w = inp.workload
        model = parity._device_model(w.shape, w.seed, None)
        sched = mk.Sched(model, 16, 64, mk.default_sched_opts())
        sess = mk.Session(model, sched)
        kp, vp = synth.device.device_pools(w.shape, w.seed, inp.num_pages)
        dev = "cuda"
        logits = torch.empty(len(rows), w.shape.vocab, device=dev)
        sess.step(torch.as_tensor(inp.tokens, device=dev), torch.as_tensor(inp.seq_lens, device=dev),
                  torch.as_tensor(inp.block_tables, device=dev), kp, vp, logits)
        sess.check()
        ref = parity.run_gpu(inp)  # a schedule of exactly len(rows) rows
        g = logits.cpu().numpy()
        err = np.max(np.abs(g - ref.logits)) / np.max(np.abs(ref.logits))
        assert err <= 1e-5, err
