"""The seeded input generator: pinned to splitmix64's published output and to
the statistics the recipe promises."""
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "splitmix64_seed1234567.txt")


def test_raw_draw_is_splitmix64():
    want = [int(l) for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    got = [synth.raw(1234567, i) for i in range(len(want))]
    assert got == want


def test_bf16_values_bounded_and_scaled():
    a = synth.bf16_bits_to_f32(synth.fill_host(1, 1 << 20, 3, synth.WQKV, sigma=0.02))
    assert abs(float(a.mean())) < 1e-4
    assert abs(float(a.std()) - 0.02) < 2e-4
    # Irwin-Hall(4) support: |v| <= 131070 * scale (plus the BF16 rounding)
    assert float(np.abs(a).max()) <= 131070 * (0.02 / synth.workloads.math.sqrt((65536.0 ** 2 - 1) / 3)) * 1.004


def test_streams_are_independent_and_addressable():
    a = synth.fill_host(3, 64, 9, synth.WG, layer0=5, expert0=2)
    b = synth.fill_host(1, 64, 9, synth.WG, layer0=5, expert0=3)
    assert np.array_equal(a[1], b[0])
    c = synth.fill_host(2, 64, 9, synth.KPOOL, layer0=4, vary_layer=True, sigma=1.0)
    d = synth.fill_host(1, 64, 9, synth.KPOOL, layer0=5, sigma=1.0)
    assert np.array_equal(c[1], d[0])
    assert not np.array_equal(a[0], a[1])


def test_inputs_recipe():
    inp = synth.make_inputs("batch32_ragged")
    assert inp.seq_lens.min() >= 512 and inp.seq_lens.max() <= 32768
    P = inp.workload.shape.page_size
    used = inp.block_tables[inp.block_tables >= 0]
    assert np.array_equal(np.sort(used), np.arange(inp.num_pages))  # a permutation of the pool
    for b, s in enumerate(inp.seq_lens):
        assert (inp.block_tables[b] >= 0).sum() == (s + P - 1) // P
    p = np.exp(inp.router_bias.astype(np.float64))
    assert abs(p.sum() - 1.0) < 1e-5
    inp64 = synth.make_inputs("batch64_ragged")
    assert inp64.seq_lens.min() >= 1024 and inp64.seq_lens.max() <= 65536
    tiny = synth.make_inputs("tiny")
    assert list(tiny.seq_lens) == [64] and tiny.block_tables.shape == (1, 4)
    assert not np.array_equal(tiny.block_tables[0], np.arange(4))  # shuffled


def test_step_bytes_full_bs1_8k():
    """Per-step algorithmic bytes of the full shape at batch 1, 8K context:
    5.730 GB of weights and 0.503 GB of KV (12 full + 36 sliding layers)."""
    sh = synth.MODELS["full"]
    w = sh.n_layers * (sh.nonexpert_layer_bytes() + sh.top_k * sh.expert_bytes()) + 2 * sh.vocab * sh.hidden
    kv = synth.step_kv_bytes(sh, [8192])
    assert abs(w / 1e9 - 5.730) < 0.002
    assert abs(kv / 1e9 - 0.503) < 0.001
