"""The three large workloads on the GPU against the CPU oracle, on sampled
rows (each row of a step is independent, so the oracle computes only the
sampled ones): continuous batching with ragged lengths and Zipf-skewed
routing, a 262144-token context, and a batch of 64."""
import numpy as np
import pytest

import synth
import parity

pytestmark = pytest.mark.gpu


def _rows(inp, extra):
    sl = inp.seq_lens
    rows = {int(np.argmin(sl)), int(np.argmax(sl))} | set(extra)
    return sorted(r for r in rows if r < len(sl))


@pytest.mark.parametrize("workload,extra", [("batch32_ragged", [7, 19]), ("long_256k", [0]),
                                            ("batch64_ragged", [33]),
                                            # two rows on the lean build; four rows on the any-batch
                                            # build (every GEMV streamed once per pair of rows)
                                            ("full_bs2_8k", [1]), ("full_bs4_8k", [2])])
def test_large_workloads(workload, extra):
    inp = synth.make_inputs(workload)
    g = parity.run_gpu(inp, parity.mk.default_sched_opts(trace_queue=1))
    # the MoE queue of every layer, bit-exact (Zipf-skewed routing at batch 32)
    assert parity.compare_queue(inp, g) == inp.workload.shape.n_layers
    rows = _rows(inp, extra)
    rep = parity.compare(inp, g, rows=rows)
    print(workload, "rows", rows, f"logit rel err {rep.max_rel_err:.3e} router err {rep.router_err.max():.3e} "
          f"routing exact {rep.exact_routing}/{rep.total_routing} ties {rep.tie_routing} kv {rep.kv_max_err:.2e}")
    assert not rep.routing_violations, rep.routing_violations
    assert rep.router_err.max() <= parity.ROUTER_TOL
    assert rep.weight_err <= 1e-4
    assert rep.max_rel_err <= parity.LOGIT_TOL
    assert rep.greedy_agree == rep.greedy_total
    assert rep.kv_max_err <= 2e-2
    # the routing of every row (not only the sampled ones) is a valid top-k set
    L, K, E = inp.workload.shape.n_layers, inp.workload.shape.top_k, inp.workload.shape.n_experts
    for l in range(L):
        for b in range(inp.workload.batch):
            ids = g.ids[l, b]
            assert len(set(ids.tolist())) == K and ids.min() >= 0 and ids.max() < E
            lg = g.extra["router_logits"][l, b]
            assert np.all(np.diff(lg[ids]) <= 0)  # descending by the GPU's own logits
            assert lg[ids].min() >= np.delete(lg, ids).max()  # and they are its top-k
    parity.release()
