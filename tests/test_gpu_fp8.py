"""FP8 expert weights (E4M3 codes, one fp32 scale per output row) through
the C ABI against the CPU oracle, which dequantizes the same codes; the
generator's device codes against its host codes.  Above two rows the expert
tiles run on the tensor cores (kind::f8f6f4 MMAs: the E4M3 codes against the
activations as four E4M3 terms, the row scale applied to the accumulator)."""
import numpy as np
import pytest
import torch

import synth
import synth.device
import moe_decode_megakernel_gb300 as mk
import parity

pytestmark = pytest.mark.gpu


def test_device_codes_match_host():
    sh = synth.MODELS["small_fp8"]
    w = synth.device.device_weights(sh, 12)
    for name, kind, rows, cols in (("w_gate", synth.WG, sh.inter, sh.hidden),
                                   ("w_down", synth.WD, sh.hidden, sh.inter)):
        got = w[name][3, 5].cpu().numpy().reshape(-1)
        assert np.array_equal(got, synth.fill_fp8_host(rows * cols, 12, kind, layer=3, expert=5))
    got = w["w_up_scale"][3, 5].cpu().numpy()
    assert np.array_equal(got, synth.fill_scales_host(sh.inter, 12, synth.SU, 3, 5, sh.weight_sigma))


@pytest.mark.parametrize("workload", ["small_fp8", "small_fp8_b2", "full_fp8_bs1_8k", "full_fp8_bs2_8k"])
def test_fp8_against_oracle(workload):
    inp = synth.make_inputs(workload)
    g = parity.run_gpu(inp)
    rep = parity.compare(inp, g)
    print(workload, f"logit rel err {rep.max_rel_err:.3e} router err {rep.router_err.max():.3e} "
          f"routing exact {rep.exact_routing}/{rep.total_routing} ties {rep.tie_routing}")
    assert not rep.routing_violations, rep.routing_violations
    assert rep.weight_err <= 1e-4
    assert rep.max_rel_err <= parity.LOGIT_TOL, rep
    assert rep.greedy_agree == rep.greedy_total
    assert rep.exact_routing + rep.tie_routing == rep.total_routing
    assert rep.kv_max_err <= 2e-2
    parity.release()


@pytest.mark.parametrize("opts", [dict(wave_order=1), dict(moe_static=0), dict(fuse_routing=0)])
def test_fp8_variants_bit_identical(opts):
    inp = synth.make_inputs("small_fp8")
    a = parity.run_gpu(inp)
    b = parity.run_gpu(inp, mk.default_sched_opts(**opts))
    assert np.array_equal(a.logits, b.logits)


@pytest.mark.parametrize("seq_lens,seed", [
    ([1024, 3, 511], 61),
    ([int(x) for x in np.random.default_rng(7).integers(1, 1024, 32)], 62),
])
def test_fp8_tensor_core_batches(seq_lens, seed):
    """Ragged batches of 3 and 32 rows (the largest FP8 schedule) on the small
    FP8 shape: every row against the oracle, the MoE queue bit-exact."""
    sh = synth.MODELS["small_fp8"]
    w = synth.Workload(f"small_fp8_tc_b{len(seq_lens)}", "small_fp8", len(seq_lens), ("fixed", 0), seed)
    sl = np.asarray(seq_lens, np.int32)
    bt, npages = synth.block_tables_for(sl, sh.page_size, seed, slack_pages=2)
    tok = np.random.default_rng(seed).integers(0, sh.vocab, size=len(sl)).astype(np.int32)
    inp = synth.StepInputs(w, tok, sl, bt, npages, None)
    g = parity.run_gpu(inp, mk.default_sched_opts(trace_queue=1))
    rep = parity.compare(inp, g)
    print(len(seq_lens), f"logit rel err {rep.max_rel_err:.3e} router err {rep.router_err.max():.3e} "
          f"routing exact {rep.exact_routing}/{rep.total_routing} ties {rep.tie_routing} kv {rep.kv_max_err:.2e}")
    assert not rep.routing_violations, rep.routing_violations
    assert rep.router_err.max() <= parity.ROUTER_TOL
    assert rep.weight_err <= 1e-4
    assert rep.max_rel_err <= parity.LOGIT_TOL, rep.max_rel_err
    assert rep.greedy_agree == rep.greedy_total
    assert rep.kv_max_err <= 2e-2
    assert parity.compare_queue(inp, g) == sh.n_layers
    parity.release()


def test_fp8_tensor_core_workload_b16():
    inp = synth.make_inputs("small_fp8_b16")
    rep = parity.compare(inp, parity.run_gpu(inp))
    assert not rep.routing_violations
    assert rep.max_rel_err <= parity.LOGIT_TOL, rep.max_rel_err
    assert rep.greedy_agree == rep.greedy_total
    parity.release()


def test_fp8_full_shape_batch32():
    """The full FP8 shape at the ragged batch of 32 (contexts U[512, 32768],
    Zipf(1.1) routing): the shortest, the longest and four random rows against
    the oracle, the routing of every row a valid top-k."""
    inp = synth.make_inputs("batch32_fp8_ragged")
    g = parity.run_gpu(inp, mk.default_sched_opts(trace_queue=1))
    rng = np.random.default_rng(3)
    rows = sorted({int(np.argmin(inp.seq_lens)), int(np.argmax(inp.seq_lens))}
                  | set(rng.choice(32, size=4, replace=False).tolist()))
    rep = parity.compare(inp, g, rows=rows)
    print(f"rows {rows}: logit rel err {rep.max_rel_err:.3e} router err {rep.router_err.max():.3e}")
    assert not rep.routing_violations, rep.routing_violations
    assert rep.router_err.max() <= parity.ROUTER_TOL
    assert rep.max_rel_err <= parity.LOGIT_TOL, rep.max_rel_err
    assert rep.greedy_agree == rep.greedy_total
    assert parity.compare_queue(inp, g) == inp.workload.shape.n_layers
    parity.release()


def test_fp8_tensor_core_range_error():
    """The SwiGLU activations enter the tensor-core down tiles as E4M3 terms,
    finite up to 448: with layer 0's up rows scaled by 10^4 a batch of 32
    (about four rows per expert: tensor-core tiles; experts with one or two
    rows take the GEMV, whose f16 operands hold 65504) fails with
    MK_ERR_DEVICE naming the limit, and the same model with the original
    scales runs clean."""
    sh = synth.MODELS["small_fp8"]
    seed = 63
    rng = np.random.default_rng(seed)
    sl = rng.integers(1, 512, size=32).astype(np.int32)
    bt, npages = synth.block_tables_for(sl, sh.page_size, seed, slack_pages=2)
    tok = rng.integers(0, sh.vocab, size=32).astype(np.int32)
    w = synth.device.device_weights(sh, seed)
    dev = "cuda"
    for boost, ok in ((1.0, True), (1e4, False)):
        ws = dict(w)
        ws["w_up_scale"] = w["w_up_scale"].clone()
        ws["w_up_scale"][0] *= boost
        model = mk.Model(mk.config_from(sh), mk.weights_from(ws), keepalive=ws)
        sess = mk.Session(model, mk.Sched(model, 32, 512))
        kp, vp = synth.device.device_pools(sh, seed, npages)
        logits = torch.empty(32, sh.vocab, device=dev)
        sess.step(torch.as_tensor(tok, device=dev), torch.as_tensor(sl, device=dev),
                  torch.as_tensor(bt, device=dev), kp, vp, logits)
        if ok:
            sess.check()
        else:
            with pytest.raises(mk.MkError) as e:
                sess.check()
            assert e.value.code == mk.MK_ERR_DEVICE and "448" in str(e.value), str(e.value)
