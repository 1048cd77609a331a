"""The dense model (one expert taken by every token with weight 1, i.e. a
SwiGLU FFN) through the C ABI against the CPU oracle: static FFN_UPGATE_ACT
/ FFN_DOWN tiles instead of the router and the MoE claimers ("Cohere: a
serving engine for North Mini Code built around a decode megakernel",
section "Tasks": the dense FFN opcodes)."""
import numpy as np
import pytest

import synth
import moe_decode_megakernel_gb300 as mk
import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("workload", ["dense_small", "dense_batch5"])
def test_dense_against_oracle(workload):
    inp = synth.make_inputs(workload)
    g = parity.run_gpu(inp)
    rep = parity.compare(inp, g)
    print(workload, f"logit rel err {rep.max_rel_err:.3e} kv {rep.kv_max_err:.2e}")
    assert rep.max_rel_err <= parity.LOGIT_TOL, rep
    assert rep.greedy_agree == rep.greedy_total, rep
    assert rep.kv_max_err <= 2e-2, rep


@pytest.mark.parametrize("opts", [dict(wave_order=1), dict(wave_order=2), dict(fuse_norm_qkv=0),
                                  dict(fuse_moe_combine=0)])
def test_dense_variants_bit_identical(opts):
    inp = synth.make_inputs("dense_small")
    a = parity.run_gpu(inp)
    b = parity.run_gpu(inp, mk.default_sched_opts(**opts))
    assert np.array_equal(a.logits, b.logits)
