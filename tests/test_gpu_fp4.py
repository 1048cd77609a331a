"""FP4 expert weights (E2M1 codes, E4M3 block scales, fp32 row scales) through
the C ABI against the CPU oracle, which dequantizes the same codes and scales; the
generator's device codes against its host codes."""
import numpy as np
import pytest
import torch

import synth
import synth.device
import moe_decode_megakernel_gb300 as mk
import parity

pytestmark = pytest.mark.gpu


def test_device_codes_match_host():
    sh = synth.MODELS["small_fp4"]
    w = synth.device.device_weights(sh, 14)
    for name, kind, rows, cols in (("w_gate", synth.WG, sh.inter, sh.hidden),
                                   ("w_down", synth.WD, sh.hidden, sh.inter)):
        got = w[name][3, 5].cpu().numpy().reshape(-1)
        assert np.array_equal(got, synth.fill_fp4_host(rows * cols // 2, 14, kind, layer=3, expert=5))
    got = w["w_up_bscale"][3, 5].cpu().numpy().reshape(-1)
    assert np.array_equal(got, synth.fill_bscales_host(sh.inter * sh.hidden // 16, 14, synth.BU, 3, 5))
    got = w["w_down_scale"][3, 5].cpu().numpy()
    assert np.array_equal(got, synth.fill_scales4_host(sh.hidden, 14, synth.SD, 3, 5, sh.weight_sigma))


@pytest.mark.parametrize("workload", ["small_fp4", "small_fp4_b2", "full_fp4_bs1_8k", "full_fp4_bs2_8k"])
def test_fp4_against_oracle(workload):
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
def test_fp4_variants_bit_identical(opts):
    inp = synth.make_inputs("small_fp4")
    a = parity.run_gpu(inp)
    b = parity.run_gpu(inp, mk.default_sched_opts(**opts))
    assert np.array_equal(a.logits, b.logits)
