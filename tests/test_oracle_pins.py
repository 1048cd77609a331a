"""Pins of the CPU oracle to facts that do not come from the oracle itself:
closed forms, invariants, library routines and brute force on tiny inputs.
Each test names the mistake it is there to catch."""
import math
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import synth

RNG = np.random.default_rng(1234)


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_closed_form():
    # x = (3, 4): mean square 12.5 -> out = x / sqrt(12.5 + eps)
    out = oracle.rmsnorm([3.0, 4.0], eps=1e-5)
    want = np.array([3.0, 4.0]) / math.sqrt(12.5 + 1e-5)
    assert np.allclose(out, want, rtol=0, atol=1e-15)


def test_rmsnorm_unit_rms_and_library():
    x = RNG.normal(size=1024) * 3.0
    out = oracle.rmsnorm(x, eps=0.0)
    assert abs(math.sqrt(np.mean(out ** 2)) - 1.0) < 1e-12  # mean over n, not n-1
    g = RNG.normal(size=1024)
    ref = torch.nn.functional.rms_norm(torch.tensor(x), (1024,), torch.tensor(g), eps=1e-5)
    assert np.allclose(oracle.rmsnorm(x, g, eps=1e-5), ref.numpy(), rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------- RoPE

def test_rope_identity_at_zero():
    v = RNG.normal(size=128)
    assert np.array_equal(oracle.rope(v, 0), v)


def test_rope_closed_form_direction():
    # d = 2: theta_0 = 1, so (1, 0) at position 1 turns to (cos 1, sin 1):
    # a wrong sign or a swapped pair fails here.
    assert np.allclose(oracle.rope([1.0, 0.0], 1), [math.cos(1), math.sin(1)], atol=1e-15)
    # d = 4, base 10000: the second pair turns by pos * 10000^(-2/4) = pos / 100
    out = oracle.rope([0.0, 0.0, 1.0, 0.0], 7, base=10000.0)
    assert np.allclose(out, [0.0, 0.0, math.cos(0.07), math.sin(0.07)], atol=1e-15)


def test_rope_relative_position():
    q, k = RNG.normal(size=64), RNG.normal(size=64)
    a = oracle.rope(q, 1000) @ oracle.rope(k, 990)
    b = oracle.rope(q, 10) @ oracle.rope(k, 0)
    assert abs(a - b) < 1e-9
    assert abs(np.linalg.norm(oracle.rope(q, 12345)) - np.linalg.norm(q)) < 1e-12


def test_rope_is_complex_rotation():
    d, pos, base = 64, 4321, 500000.0
    v = RNG.normal(size=d)
    z = (v[0::2] + 1j * v[1::2]) * np.exp(1j * pos * base ** (-np.arange(0, d, 2) / d))
    out = oracle.rope(v, pos, base)
    assert np.allclose(out[0::2], z.real, atol=1e-12) and np.allclose(out[1::2], z.imag, atol=1e-12)


# ---------------------------------------------------------------- softmax

def test_softmax_closed_form():
    p = oracle.softmax([0.0, math.log(2.0), math.log(3.0)])
    assert np.allclose(p, [1 / 6, 2 / 6, 3 / 6], atol=1e-15)
    s = RNG.normal(size=17) * 30
    assert abs(oracle.softmax(s).sum() - 1.0) < 1e-14
    assert np.allclose(oracle.softmax(s + 1000.0), oracle.softmax(s), atol=1e-15)


# -------------------------------------------------------------- attention

def test_attention_matches_library_sdpa():
    d, n = 64, 300
    q, K, V = RNG.normal(size=d), RNG.normal(size=(n, d)), RNG.normal(size=(n, d))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q)[None, None, None], torch.tensor(K)[None, None], torch.tensor(V)[None, None])
    out = oracle.attend(q, K, V, 1 / math.sqrt(d))
    assert np.allclose(out, ref.numpy().reshape(-1), rtol=1e-12, atol=1e-12)


def test_attention_special_cases():
    d = 8
    K, V = RNG.normal(size=(1, d)), RNG.normal(size=(1, d))
    assert np.allclose(oracle.attend(RNG.normal(size=d), K, V, 0.3), V[0], atol=1e-15)
    K, V = RNG.normal(size=(5, d)), RNG.normal(size=(5, d))
    assert np.allclose(oracle.attend(np.zeros(d), K, V, 1.0), V.mean(0), atol=1e-15)


@pytest.mark.parametrize("cuts", [[], [1], [37, 38], [0, 5, 200, 299], list(range(10, 300, 10))])
def test_split_combine_equals_unsplit(cuts):
    d, n = 32, 300
    q, K, V = RNG.normal(size=d) * 2, RNG.normal(size=(n, d)), RNG.normal(size=(n, d))
    bounds = [0] + cuts + [n]
    parts = [oracle.attend_partial(q, K[a:b], V[a:b], 0.2) for a, b in zip(bounds, bounds[1:])]
    m = np.array([p[0] for p in parts])
    l_ = np.array([p[1] for p in parts])
    o = np.stack([p[2] for p in parts])
    out = oracle.attend_combine(m, l_, o)
    assert np.allclose(out, oracle.attend(q, K, V, 0.2), rtol=1e-12, atol=1e-12)


def test_partial_of_empty_slice():
    m, l_, o = oracle.attend_partial(np.ones(4), np.zeros((0, 4)), np.zeros((0, 4)), 1.0)
    assert m == -math.inf and l_ == 0.0 and np.all(o == 0)


# -------------------------------------------------------------------- top-k

def test_topk_brute_force_and_ties():
    for _ in range(50):
        x = RNG.integers(-3, 4, size=32).astype(np.float32)  # many ties
        ids, margin = oracle.topk(x, 8)
        order = sorted(range(32), key=lambda e: (-x[e], e))
        assert list(ids) == order[:8]
        assert margin == x[order[7]] - x[order[8]]
    ids, margin = oracle.topk(np.array([1, 2, 3], np.float32), 3)
    assert list(ids) == [2, 1, 0] and margin == math.inf


# ---------------------------------------------------------- expert and MoE

def test_swiglu_closed_form():
    silu1 = 1.0 / (1.0 + math.exp(-1.0))
    assert abs(oracle.silu(1.0) - silu1) < 1e-16
    # H = I = 1: out = wd * silu(wg x) * (wu x): the SiLU sits on the gate
    out = oracle.swiglu_expert([[1.0]], [[2.0]], [[3.0]], [1.0])
    assert abs(out[0] - 3.0 * silu1 * 2.0) < 1e-15
    out = oracle.swiglu_expert([[2.0]], [[1.0]], [[1.0]], [1.0])
    assert abs(out[0] - 2.0 / (1.0 + math.exp(-2.0))) < 1e-15


def test_swiglu_orientation():
    # H = 2, I = 3 with distinct entries: a transposed operand changes the result
    Wg = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    Wu = np.array([[2.0, 0.0], [0.0, 3.0], [1.0, -1.0]])
    Wd = np.array([[1.0, 0.0, 1.0], [0.0, 1.0, 2.0]])
    x = np.array([0.5, -2.0])
    g = np.array([0.5, -2.0, -1.5])
    u = np.array([1.0, -6.0, 2.5])
    a = g / (1 + np.exp(-g)) * u
    want = np.array([a[0] + a[2], a[1] + 2 * a[2]])
    assert np.allclose(oracle.swiglu_expert(Wg, Wu, Wd, x), want, atol=1e-15)


def test_moe_routed_equals_dense_gated():
    H, I, E, k = 16, 8, 6, 3
    Wg = [RNG.normal(size=(I, H)) for _ in range(E)]
    Wu = [RNG.normal(size=(I, H)) for _ in range(E)]
    Wd = [RNG.normal(size=(H, I)) for _ in range(E)]
    x = RNG.normal(size=H)
    logits = RNG.normal(size=E).astype(np.float32)
    ids, _ = oracle.topk(logits, k)
    w = oracle.softmax(logits[ids].astype(np.float64))
    assert abs(w.sum() - 1.0) < 1e-14
    gate = np.zeros(E)
    gate[ids] = w
    out = oracle.moe_routed(ids, w, Wg, Wu, Wd, x)
    ref = oracle.moe_dense_gated(gate, Wg, Wu, Wd, x)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ paging

def test_kv_slot():
    row = [5, 9, 2]
    assert oracle.kv_slot(37, 16, row) == (2, 5)  # logical page 2, offset 5
    assert oracle.kv_slot(16, 16, row) == (9, 0)
    assert oracle.kv_slot(48, 16, row) is None  # beyond the table
    assert oracle.kv_slot(20, 16, [5, -1]) is None  # unallocated page


def test_pool_vec_is_generator_layout():
    sh = synth.MODELS["tiny"]
    layer, page, head, slot = 1, 3, 1, 7
    flat = synth.fill_host(1, (page + 1) * sh.n_kv * sh.page_size * sh.head_dim, 11, synth.VPOOL,
                           layer0=layer, sigma=1.0)[0]
    base = ((page * sh.n_kv + head) * sh.page_size + slot) * sh.head_dim
    want = synth.bf16_bits_to_f32(flat[base:base + sh.head_dim]).astype(np.float64)
    assert np.array_equal(oracle.pool_vec(sh, 11, 1, layer, page, head, slot), want)


# ---------------------------------------------------------- the whole step

def _bf16(a):
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return synth.bf16_bits_to_f32(u.astype(np.uint16)).astype(np.float64)


def _tiny_inputs():
    return synth.make_inputs("tiny")


def test_step_embedding_and_lm_head():
    inp = _tiny_inputs()
    sh = inp.workload.shape
    r = oracle.decode_step(sh, inp.workload.seed, inp.tokens, inp.seq_lens, inp.block_tables,
                           want_hidden=True)
    emb = synth.bf16_bits_to_f32(synth.fill_host(1, sh.vocab * sh.hidden, inp.workload.seed,
                                                 synth.EMB)[0]).reshape(sh.vocab, sh.hidden)
    assert np.array_equal(r.hidden[0, 0], emb[inp.tokens[0]].astype(np.float64))
    # logits = W_lm RMSNorm(h_L), gamma = 1
    wlm = synth.bf16_bits_to_f32(synth.fill_host(1, sh.vocab * sh.hidden, inp.workload.seed,
                                                 synth.WLM)[0]).reshape(sh.vocab, sh.hidden)
    h = r.hidden[-1, 0]
    xf = h / np.sqrt(np.mean(h ** 2) + sh.eps)
    assert np.allclose(r.logits[0], wlm.astype(np.float64) @ xf, rtol=1e-10, atol=1e-10)


def test_step_routing_invariants():
    inp = synth.make_inputs("small")
    sh = inp.workload.shape
    r = oracle.decode_step(sh, inp.workload.seed, inp.tokens, inp.seq_lens, inp.block_tables)
    assert np.allclose(r.weights.sum(-1), 1.0, atol=1e-12)
    for l in range(sh.n_layers):
        ids, margin = oracle.topk(r.router_logits[l, 0], sh.top_k)
        assert list(ids) == list(r.own_ids[l, 0]) == list(r.ids[l, 0])
        assert len(set(ids)) == sh.top_k
        assert np.all(np.diff(r.router_logits[l, 0][ids]) <= 0)


def test_step_new_token_only():
    """seq_len = 1: each head attends to the new token alone, so its output is
    the BF16 value vector of its own KV group (head i reads group i // G)."""
    sh = synth.MODELS["tiny"]
    r = oracle.decode_step(sh, 5, np.array([3], np.int32), np.array([1], np.int32),
                           np.array([[2]], np.int32), want_kv=True, want_attn=True)
    G = sh.n_q // sh.n_kv
    for l in range(sh.n_layers):
        v = r.kv_new[l, 0, 1]  # [n_kv, d], before the BF16 store
        for i in range(sh.n_q):
            got = r.attn[l, 0, i * sh.head_dim:(i + 1) * sh.head_dim]
            want = v[i // G]
            # the pool holds BF16: within one BF16 rounding of the fp64 value
            assert np.allclose(got, want, rtol=2 ** -8, atol=0)


def test_window_boundaries():
    """Sliding layers attend to the last `window` positions, the new one
    included: window >= seq_len equals full attention, window = 1 sees only
    the new token."""
    base = synth.MODELS["tiny"]
    inp = _tiny_inputs()
    args = (inp.workload.seed, inp.tokens, inp.seq_lens, inp.block_tables)
    full = oracle.decode_step(base, *args, want_attn=True, want_kv=True)
    wide = oracle.decode_step(replace(base, window=64, full_period=2), *args, want_attn=True)
    assert np.array_equal(full.logits, wide.logits)
    one = oracle.decode_step(replace(base, window=1, full_period=2), *args, want_attn=True,
                             want_kv=True)
    G = base.n_q // base.n_kv
    # layer 0 is sliding ((0+1) % 2 != 0), layer 1 full
    for i in range(base.n_q):
        got = one.attn[0, 0, i * base.head_dim:(i + 1) * base.head_dim]
        assert np.allclose(got, one.kv_new[0, 0, 1, i // G], rtol=2 ** -8, atol=0)
    assert not np.allclose(one.attn[1], one.kv_new[1, 0, 1].repeat(G, 0).reshape(-1), rtol=1e-3)


def test_window_two_keys():
    """window = 2: the new token and position seq_len - 2, read through the
    block table from the generated pool."""
    base = replace(synth.MODELS["tiny"], window=2, full_period=2)
    inp = _tiny_inputs()
    s = int(inp.seq_lens[0])
    r = oracle.decode_step(base, inp.workload.seed, inp.tokens, inp.seq_lens, inp.block_tables,
                           want_attn=True, want_kv=True, want_hidden=True)
    l, d, G = 0, base.head_dim, base.n_q // base.n_kv
    x = r.hidden[0, 0] / np.sqrt(np.mean(r.hidden[0, 0] ** 2) + base.eps)
    for i in range(base.n_q):
        g = i // G
        page, off = oracle.kv_slot(s - 2, base.page_size, inp.block_tables[0])
        k_old = oracle.pool_vec(base, inp.workload.seed, 0, l, page, g, off)
        v_old = oracle.pool_vec(base, inp.workload.seed, 1, l, page, g, off)
        kb = _bf16(r.kv_new[l, 0, 0, g])
        vb = _bf16(r.kv_new[l, 0, 1, g])
        # recompute q from the layer input to pin the head/row mapping
        wqkv = synth.bf16_bits_to_f32(synth.fill_host(1, base.qkv_rows() * base.hidden,
                                                      inp.workload.seed, synth.WQKV, layer0=l)[0])
        q = wqkv.reshape(base.qkv_rows(), base.hidden)[i * d:(i + 1) * d].astype(np.float64) @ x
        q = oracle.rope(q, s - 1)
        ref = oracle.attend(q, np.stack([k_old, kb]), np.stack([v_old, vb]), 1 / math.sqrt(d))
        got = r.attn[l, 0, i * d:(i + 1) * d]
        assert np.allclose(got, ref, rtol=1e-9, atol=1e-12)


def test_rows_are_independent():
    """Each batch row is computed alone: a subset of rows gives the same
    values as the full batch."""
    sh = replace(synth.MODELS["tiny"])
    rng = np.random.default_rng(3)
    B = 3
    sl = np.array([5, 40, 17], np.int32)
    bt, _ = synth.block_tables_for(sl, sh.page_size, 9)
    tok = rng.integers(0, sh.vocab, size=B).astype(np.int32)
    a = oracle.decode_step(sh, 2, tok, sl, bt)
    b = oracle.decode_step(sh, 2, tok, sl, bt, rows=[2, 0])
    assert np.array_equal(a.logits[[2, 0]], b.logits)
