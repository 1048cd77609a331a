"""FP4 expert weights on the CPU: the generator's E2M1 encoder against the
oracle's decoder written from the format definition (E2M1: 1 sign bit, 2
exponent bits biased by 1, 1 mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4,
6), the packing of two codes per byte, the E4M3 block scales (one per 16
inputs of a row), the row scales, and the oracle's FP4 expert rows."""
import numpy as np
import pytest

import oracle
import synth

MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_golden_codes():
    for c, v in enumerate(MAGS):
        assert oracle.e2m1_value(c) == v
        assert oracle.e2m1_value(c | 8) == -v
    assert synth.e2m1(6.0) == 7 and synth.e2m1(-0.5) == 9 and synth.e2m1(1.5) == 3


def test_every_code_round_trips():
    for c in range(16):
        if c == 8:  # -0 encodes as +0
            continue
        assert synth.e2m1(oracle.e2m1_value(c)) == c, c


def test_encoder_rounds_to_nearest_even():
    # the midpoints go to the code with an even mantissa bit
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for x, c in ties.items():
        assert synth.e2m1(x) == c, x
        assert synth.e2m1(-x) == c | 8, -x  # the sign survives a round to zero (-0)
    rng = np.random.default_rng(1)
    vals = np.array(MAGS)
    for x in rng.uniform(-6, 6, 4000).astype(np.float32):
        got = synth.e2m1(float(x))
        d = np.abs(vals - abs(float(x)))
        assert abs(abs(oracle.e2m1_value(got)) - abs(float(x))) == d.min(), (x, got)
        assert (got & 8 == 8) == (x < 0)


def test_generated_codes_and_scales():
    seed, I, H = 6, 64, 256
    packed = synth.fill_fp4_host(I * H // 2, seed, synth.WU, layer=2, expert=1)
    codes = np.stack([packed & 15, packed >> 4], axis=1).reshape(I, H)
    q = np.vectorize(oracle.e2m1_value)(codes)
    # ih4 * 3 * 2^-16 has std 1.732; rounding to E2M1 keeps it within a few %
    assert 1.6 < q.std() < 1.9 and np.abs(q).max() <= 6.0
    bs = synth.fill_bscales_host(I * H // 16, seed, synth.BU, layer=2, expert=1)
    assert np.all((bs & 0xF8) == 0x30)  # 0.5 * (1 + m/8)
    bv = np.vectorize(oracle.e4m3_value)(bs)
    assert set(np.unique(bv)) <= {0.5 * (1 + m / 8) for m in range(8)} and 0.66 < bv.mean() < 0.78
    rs = synth.fill_scales4_host(I, seed, synth.SU, layer=2, expert=1, sigma=0.02)
    base = np.float32(0.02 / (37837.22651061575 * 3 * 2.0 ** -16 * 0.71875))
    assert synth.fp4_base(0.02) == base
    assert np.all(rs >= base) and np.all(rs < 1.5 * base)
    w = q * np.repeat(bv.reshape(I, H // 16), 16, axis=1) * rs[:, None].astype(np.float64)
    assert 0.015 < w.std() < 0.035


@pytest.mark.parametrize("kind,rows_of", [(synth.WG, "inter"), (synth.WD, "hidden")])
def test_oracle_fp4_expert_rows(kind, rows_of):
    """The oracle's FP4 expert matrix = nibble-unpacked codes (element 2j in
    the low nibble of byte j) decoded, times the block scale of each run of
    16 inputs, times the row scale."""
    sh = synth.MODELS["small_fp4"]
    seed, layer, expert = 14, 3, 5
    rows, cols = (sh.inter, sh.hidden) if rows_of == "inter" else (sh.hidden, sh.inter)
    bkind = {synth.WG: synth.BG, synth.WD: synth.BD}[kind]
    skind = {synth.WG: synth.SG, synth.WD: synth.SD}[kind]
    got = oracle.synth_matrix(sh, seed, kind, layer, expert)
    packed = synth.fill_fp4_host(rows * cols // 2, seed, kind, layer, expert)
    codes = np.empty(rows * cols, np.int64)
    codes[0::2] = packed & 15
    codes[1::2] = packed >> 4
    q = np.vectorize(oracle.e2m1_value)(codes.reshape(rows, cols))
    bs = synth.fill_bscales_host(rows * cols // 16, seed, bkind, layer, expert).reshape(rows, cols // 16)
    bv = np.repeat(np.vectorize(oracle.e4m3_value)(bs), 16, axis=1)
    rs = synth.fill_scales4_host(rows, seed, skind, layer, expert, sh.weight_sigma).astype(np.float64)
    assert np.array_equal(got, q * bv * rs[:, None])


# ---- the boundary: FP4 models and schedules (no GPU)

import moe_decode_megakernel_gb300 as mk  # noqa: E402
from test_abi_sched import fake_model, NUM_SMS  # noqa: E402


@pytest.mark.parametrize("workload", ["small_fp4", "small_fp4_b2", "full_fp4_bs1_8k"])
def test_fp4_schedules(workload):
    w = synth.WORKLOADS[workload]
    inp = synth.make_inputs(w)
    m = fake_model(w.shape)
    s = mk.Sched(m, w.batch, int(inp.seq_lens.max()), mk.default_sched_opts(num_sms=NUM_SMS))
    s.validate()
    s.simulate(inp.seq_lens, seed=4)


def test_fp4_needs_small_batch_and_one_format():
    from dataclasses import replace
    m = fake_model(synth.MODELS["small_fp4"])
    with pytest.raises(mk.MkError) as e:
        mk.Sched(m, 3, 1024, mk.default_sched_opts(num_sms=NUM_SMS))
    assert e.value.code == mk.MK_ERR_UNSUPPORTED
    with pytest.raises(mk.MkError) as e:
        fake_model(replace(synth.MODELS["small_fp4"], expert_fp8=True))
    assert e.value.code == mk.MK_ERR_ARG
    w = mk.MkWeights(*[0x10000 * (i + 1) for i in range(len(mk.MkWeights._fields_))])
    w.w_down_bscale = None
    with pytest.raises(mk.MkError) as e:
        mk.Model(mk.config_from(synth.MODELS["small_fp4"]), w)
    assert e.value.code == mk.MK_ERR_ARG
