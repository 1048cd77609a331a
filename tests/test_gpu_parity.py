"""GPU decode step against the CPU oracle through the C ABI: logits within
2e-2 (max-normalised per row), routing exact away from 1e-3 ties, greedy
tokens, and the new K/V written to the pool."""
import numpy as np
import pytest
import torch

import synth
import moe_decode_megakernel_gb300 as mk
import parity

pytestmark = pytest.mark.gpu


def check(rep, total_rows):
    print(f"logit rel err {rep.max_rel_err:.3e}  router err max {rep.router_err.max():.3e} "
          f"(per layer {np.array2string(rep.router_err, precision=1)})  weights {rep.weight_err:.2e}  "
          f"routing exact {rep.exact_routing}/{rep.total_routing} ties {rep.tie_routing}  "
          f"kv {rep.kv_max_err:.2e}")
    assert not rep.routing_violations, rep.routing_violations
    assert rep.router_err.max() <= parity.ROUTER_TOL, rep.router_err
    assert rep.weight_err <= 1e-4, rep.weight_err
    assert rep.max_rel_err <= parity.LOGIT_TOL, rep
    assert rep.greedy_agree == rep.greedy_total, rep
    assert rep.exact_routing + rep.tie_routing == rep.total_routing
    assert rep.kv_max_err <= 2e-2, rep


@pytest.mark.parametrize("workload", ["tiny", "small", "tiny_gains", "small_gains"])
def test_small_configs(workload):
    """tiny and small, with unit and with seeded non-unit RMSNorm gains (the
    gains pin each layer's gain row and the final gain on the GPU side); the
    MoE queue of every layer bit-exact."""
    inp = synth.make_inputs(workload)
    g = parity.run_gpu(inp, mk.default_sched_opts(trace_queue=1))
    rep = parity.compare(inp, g)
    print(workload, rep)
    check(rep, 1)
    assert parity.compare_queue(inp, g) == inp.workload.shape.n_layers


@pytest.mark.parametrize("workload", ["full_bs1_8k", "full_gains_bs1_8k"])
def test_full_bs1_8k(workload):
    inp = synth.make_inputs(workload)
    g = parity.run_gpu(inp, mk.default_sched_opts(trace_queue=1))
    rep = parity.compare(inp, g)
    print(workload, rep)
    check(rep, 1)
    assert parity.compare_queue(inp, g) == 48


@pytest.mark.parametrize("order", [1, 2, 3, 4, 5, 6])
def test_wave_orders_bit_identical(order):
    """Any schedule without a cyclic wait computes the same step ("all these
    schedules produce correct outputs"); reductions have a fixed order, so
    the logits are bit-identical."""
    inp = synth.make_inputs("small")
    a = parity.run_gpu(inp)
    b = parity.run_gpu(inp, mk.default_sched_opts(wave_order=order, attn_split_pages=1,
                                                  moe_claimers=37))
    assert np.array_equal(a.logits, b.logits)
    assert np.array_equal(a.ids, b.ids)


@pytest.mark.parametrize("opts", [dict(fuse_finalize=0), dict(fuse_moe_combine=0),
                                  dict(explicit_gather=1), dict(moe_queue=1),
                                  dict(moe_claimers=7), dict(moe_static=0),
                                  dict(moe_static=0, moe_claimers=7), dict(fuse_routing=0),
                                  dict(fuse_norm_qkv=0), dict(attn_static=0),
                                  dict(moe_balance=1), dict(placement=1)])
def test_unfused_variants_bit_identical(opts):
    inp = synth.make_inputs("small")
    a = parity.run_gpu(inp)
    b = parity.run_gpu(inp, mk.default_sched_opts(**opts))
    assert np.array_equal(a.logits, b.logits)


def _ragged_tiny(seq_lens, seed=21):
    sh = synth.MODELS["tiny"]
    w = synth.Workload("tiny_ragged", "tiny", len(seq_lens), ("fixed", 0), seed)
    sl = np.asarray(seq_lens, np.int32)
    bt, npages = synth.block_tables_for(sl, sh.page_size, seed, slack_pages=3)
    rng = np.random.default_rng(seed)
    tok = rng.integers(0, sh.vocab, size=len(sl)).astype(np.int32)
    return synth.StepInputs(w, tok, sl, bt, npages, None)


def test_edge_lengths():
    """seq_len 1 (the new token alone), page boundaries on both sides, a
    partial last page, rows of very different length in one batch."""
    P = synth.MODELS["tiny"].page_size
    inp = _ragged_tiny([1, P, P + 1, 2 * P - 1, 5 * P, 3])
    g = parity.run_gpu(inp)
    rep = parity.compare(inp, g)
    print(rep)
    check(rep, 6)


def test_sliding_window_layers():
    """A window shorter than the context on every other layer (tiny shape)."""
    from dataclasses import replace
    base = _ragged_tiny([1, 20, 33, 64, 100])
    sh = replace(synth.MODELS["tiny"], window=24, full_period=2)
    w = synth.Workload("tiny_window", "tiny", 5, ("fixed", 0), 21, shape_override=sh)
    inp = synth.StepInputs(w, base.tokens, base.seq_lens, base.block_tables, base.num_pages, None)
    g = parity.run_gpu(inp)
    rep = parity.compare(inp, g)
    print(rep)
    check(rep, 5)


def test_batch_below_schedule_max():
    """A schedule built for 8 rows runs a step of 3."""
    inp = _ragged_tiny([10, 40, 64])
    w = inp.workload
    model = parity._device_model(w.shape, w.seed, None)
    sched = mk.Sched(model, 8, 64, mk.default_sched_opts())
    sess = mk.Session(model, sched)
    kp, vp = synth.device.device_pools(w.shape, w.seed, inp.num_pages)
    dev = "cuda"
    logits = torch.empty(3, w.shape.vocab, device=dev)
    sess.step(torch.as_tensor(inp.tokens, device=dev), torch.as_tensor(inp.seq_lens, device=dev),
              torch.as_tensor(inp.block_tables, device=dev), kp, vp, logits)
    sess.check()
    ref = parity.run_gpu(inp)
    assert np.array_equal(logits.cpu().numpy(), ref.logits)


def test_empty_batch_is_rejected_before_launch():
    """A step of no rows is an argument error: nothing is launched, the
    logits and the schedule's next step are untouched."""
    inp = _ragged_tiny([10, 40, 64])
    w = inp.workload
    model = parity._device_model(w.shape, w.seed, None)
    sched = mk.Sched(model, 4, 64, mk.default_sched_opts())
    sess = mk.Session(model, sched)
    kp, vp = synth.device.device_pools(w.shape, w.seed, inp.num_pages)
    dev = "cuda"
    logits = torch.full((3, w.shape.vocab), 7.0, device=dev)
    tok = torch.as_tensor(inp.tokens, device=dev)
    sl = torch.as_tensor(inp.seq_lens, device=dev)
    bt = torch.as_tensor(inp.block_tables, device=dev)
    with pytest.raises(mk.MkError) as e:
        sess.step(tok[:0], sl[:0], bt, kp, vp, logits)
    assert e.value.code == mk.MK_ERR_ARG
    torch.cuda.synchronize()
    assert bool((logits == 7.0).all())
    sess.step(tok, sl, bt, kp, vp, logits)  # the session still works
    sess.check()
    assert np.array_equal(logits.cpu().numpy(), parity.run_gpu(inp).logits)


def test_two_rows_window_layers():
    """Two rows, sliding and full layers (tiny shape): the QKV tiles compute
    the RMSNorm themselves and the slices are merged per (row, group),
    over a dynamic slice count on full layers and the static one on sliding
    layers; one merge task per (row, group, head) agrees with the oracle too."""
    from dataclasses import replace
    base = _ragged_tiny([33, 100], seed=23)
    sh = replace(synth.MODELS["tiny"], window=24, full_period=2)
    w = synth.Workload("tiny_window2", "tiny", 2, ("fixed", 0), 23, shape_override=sh)
    inp = synth.StepInputs(w, base.tokens, base.seq_lens, base.block_tables, base.num_pages, None)
    g = parity.run_gpu(inp)
    rep = parity.compare(inp, g)
    print(rep)
    check(rep, 2)
    # the same step with the RMSNorm as a separate task: the same arithmetic
    u = parity.run_gpu(inp, mk.default_sched_opts(fuse_norm_qkv=0))
    assert np.array_equal(g.logits, u.logits)
    check(parity.compare(inp, parity.run_gpu(inp, mk.default_sched_opts(combine_per_head=1))), 2)


def test_one_row_on_two_row_schedule():
    """A schedule built for two rows runs a step of one: the absent row's
    merge tasks wait for no slices and do nothing."""
    inp = _ragged_tiny([57])
    w = inp.workload
    model = parity._device_model(w.shape, w.seed, None)
    sched = mk.Sched(model, 2, 64, mk.default_sched_opts())
    sess = mk.Session(model, sched)
    kp, vp = synth.device.device_pools(w.shape, w.seed, inp.num_pages)
    dev = "cuda"
    logits = torch.empty(1, w.shape.vocab, device=dev)
    sess.step(torch.as_tensor(inp.tokens, device=dev), torch.as_tensor(inp.seq_lens, device=dev),
              torch.as_tensor(inp.block_tables, device=dev), kp, vp, logits)
    sess.check()
    ref = parity.run_gpu(inp)
    assert np.array_equal(logits.cpu().numpy(), ref.logits)
