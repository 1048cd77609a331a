"""FP8 expert weights on the CPU: the generator's E4M3 encoder against the
oracle's decoder written from the format definition (OCP 8-bit floating
point, E4M3: 1 sign, 4 exponent bits biased by 7, 3 mantissa bits,
subnormals below 2^-6, 448 the largest finite value, no infinities), the
generated codes and row scales, the oracle's FP8 expert rows, and the
schedules."""
import numpy as np
import pytest

import oracle
import synth
import moe_decode_megakernel_gb300 as mk
from test_abi_sched import fake_model, NUM_SMS


def test_golden_codes():
    # values fixed by the format: (-1)^s 2^(e-7) (1 + m/8), subnormals 2^-6 m/8
    assert oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0xB8) == -1.0
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x08) == 2.0 ** -6
    assert oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_value(0x00) == 0.0
    assert np.isnan(oracle.e4m3_value(0x7F)) and np.isnan(oracle.e4m3_value(0xFF))
    assert synth.e4m3(1.0) == 0x38 and synth.e4m3(448.0) == 0x7E and synth.e4m3(-2.0 ** -9) == 0x81


def test_every_finite_code_round_trips():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert synth.e4m3(oracle.e4m3_value(c)) == c, hex(c)


def test_encoder_rounds_to_nearest_even():
    codes = [c for c in range(256) if c & 0x7F != 0x7F]
    vals = np.array([oracle.e4m3_value(c) for c in codes])
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.uniform(-448, 448, 3000).astype(np.float32),
                         rng.uniform(-0.05, 0.05, 3000).astype(np.float32),
                         # midpoints between neighbours: ties
                         np.float32((np.sort(vals)[1:] + np.sort(vals)[:-1]) / 2)])
    for x in xs:
        got = synth.e4m3(float(x))
        d = np.abs(vals - float(x))
        best = d.min()
        assert abs(oracle.e4m3_value(got) - float(x)) == best, (x, hex(got))
        ties = [codes[i] for i in np.nonzero(d == best)[0]]
        if len(ties) > 1 and not (float(x) == 0.0):
            assert got & 1 == 0, (x, [hex(t) for t in ties], hex(got))  # even mantissa


def test_generated_weights_and_scales():
    seed, I, H = 5, 64, 256
    codes = synth.fill_fp8_host(I * H, seed, synth.WG, layer=1, expert=3).reshape(I, H)
    assert not np.any((codes & 0x7F) == 0x7F)  # no NaN codes
    q = np.vectorize(oracle.e4m3_value)(codes)
    assert 0.9 * 129.3 < q.std() < 1.1 * 129.3  # ih4 std * 3.5 * 2^-10
    sc = synth.fill_scales_host(I, seed, synth.SG, layer=1, expert=3, sigma=0.02)
    base = np.float32(0.02 / (37837.22651061575 * 0.00341796875))
    assert np.all(sc >= base) and np.all(sc < 1.5 * base)
    w = q * sc[:, None].astype(np.float64)
    assert 0.02 < w.std() < 0.03  # sigma to 1.5 sigma per row


def test_oracle_fp8_expert_rows():
    """The oracle's FP8 expert matrix = the oracle's E4M3 decode of the
    generator's codes times the row scales (the generator's own route)."""
    sh = synth.MODELS["small_fp8"]
    seed, layer, expert = 12, 2, 7
    got = oracle.synth_matrix(sh, seed, synth.WD, layer, expert)
    codes = synth.fill_fp8_host(sh.hidden * sh.inter, seed, synth.WD, layer, expert).reshape(sh.hidden, sh.inter)
    sc = synth.fill_scales_host(sh.hidden, seed, synth.SD, layer, expert, sh.weight_sigma)
    want = np.vectorize(oracle.e4m3_value)(codes) * sc[:, None].astype(np.float64)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("workload", ["small_fp8", "small_fp8_b2", "small_fp8_b16"])
def test_fp8_schedules(workload):
    w = synth.WORKLOADS[workload]
    inp = synth.make_inputs(w)
    m = fake_model(w.shape)
    s = mk.Sched(m, w.batch, int(inp.seq_lens.max()), mk.default_sched_opts(num_sms=NUM_SMS))
    s.validate()
    s.simulate(inp.seq_lens, seed=4)


def test_fp8_batch_limit():
    """Above two rows FP8 experts take the tensor-core build (its operand rows
    are E4M3 terms: xg8 / u8 instead of the BF16 xgb / ub), up to 32 rows: four
    term rows per routed row fill the MMA's 128 columns."""
    m = fake_model(synth.MODELS["small_fp8"])
    s = mk.Sched(m, 3, 1024, mk.default_sched_opts(num_sms=NUM_SMS))
    assert s.workspace_offset("xg8") >= 0 and s.workspace_offset("xgb") == -1
    s = mk.Sched(m, 32, 1024, mk.default_sched_opts(num_sms=NUM_SMS))
    assert s.workspace_offset("u8") >= 0
    assert mk.Sched(m, 2, 1024, mk.default_sched_opts(num_sms=NUM_SMS)).workspace_offset("xg8") == -1
    with pytest.raises(mk.MkError) as e:
        mk.Sched(m, 33, 1024, mk.default_sched_opts(num_sms=NUM_SMS))
    assert e.value.code == mk.MK_ERR_UNSUPPORTED
