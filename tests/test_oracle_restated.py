"""The oracle's whole decode step against an independent fp64 restatement in
torch CPU tensor ops, and the invariants of paging, explicit pools and the
MoE work queue.

The restatement below is written from the same definitions as the oracle
(the parallel layer of "Cohere: a decode megakernel for North Mini Code",
section "1. Reduce wave quantization": x = RMSNorm(h), h <- h + W_o attn(x) +
MoE(x); RoPE and write-then-attend from "tiny-vllm 5. The decode path",
sections "RoPE" and "The decode loop") but shares none of its code: weights
come straight from the input generator, attention is torch's
scaled_dot_product_attention over K/V gathered through the block table,
RoPE is a complex multiplication, top-k is torch.topk and the norms are
torch's rms_norm.  Comparing every layer's residual pins the layer
composition: a dropped residual, W_o applied to the wrong operand, the MoE
reading h instead of x, or a gain at the wrong layer fails here.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(synth.bf16_bits_to_f32(a).astype(np.float64))


class Weights:
    """The synthetic model's weights as fp64 tensors, read from the generator
    (experts on demand)."""

    def __init__(self, shape, seed):
        self.shape, self.seed = shape, seed
        L, H, V, E = shape.n_layers, shape.hidden, shape.vocab, shape.n_experts
        QKV, NQD, sg = shape.qkv_rows(), shape.n_q * shape.head_dim, shape.weight_sigma
        self.emb = _bf16(synth.fill_host(1, V * H, seed, synth.EMB, sigma=sg)).view(V, H)
        self.wqkv = _bf16(synth.fill_host(L, QKV * H, seed, synth.WQKV, vary_layer=True, sigma=sg)).view(L, QKV, H)
        self.wo = _bf16(synth.fill_host(L, H * NQD, seed, synth.WO, vary_layer=True, sigma=sg)).view(L, H, NQD)
        self.wr = _bf16(synth.fill_host(L, E * H, seed, synth.WR, vary_layer=True, sigma=sg)).view(L, E, H)
        self.wlm = _bf16(synth.fill_host(1, V * H, seed, synth.WLM, sigma=sg)).view(V, H)
        self._experts = {}

    def expert(self, l, e):
        if (l, e) not in self._experts:
            H, I, sg = self.shape.hidden, self.shape.inter, self.shape.weight_sigma
            g = _bf16(synth.fill_host(1, I * H, self.seed, synth.WG, layer0=l, expert0=e, sigma=sg)).view(I, H)
            u = _bf16(synth.fill_host(1, I * H, self.seed, synth.WU, layer0=l, expert0=e, sigma=sg)).view(I, H)
            d = _bf16(synth.fill_host(1, H * I, self.seed, synth.WD, layer0=l, expert0=e, sigma=sg)).view(H, I)
            self._experts[(l, e)] = (g, u, d)
        return self._experts[(l, e)]


def host_pools(shape, seed, num_pages):
    """The generator's K and V pools [L][pages][n_kv][P][d] as BF16 bits."""
    per = num_pages * shape.n_kv * shape.page_size * shape.head_dim
    dims = (shape.n_layers, num_pages, shape.n_kv, shape.page_size, shape.head_dim)
    k = synth.fill_host(shape.n_layers, per, seed, synth.KPOOL, vary_layer=True, sigma=shape.kv_sigma)
    v = synth.fill_host(shape.n_layers, per, seed, synth.VPOOL, vary_layer=True, sigma=shape.kv_sigma)
    return k.reshape(dims).copy(), v.reshape(dims).copy()


def rope_complex(v: torch.Tensor, pos: int, base: float) -> torch.Tensor:
    """Pairs (2i, 2i+1) as complex numbers turned by pos * base^(-2i/d)."""
    n, d = v.shape
    theta = base ** (-torch.arange(0, d, 2, dtype=torch.float64) / d)
    rot = torch.polar(torch.ones_like(theta), pos * theta)
    return torch.view_as_real(torch.view_as_complex(v.reshape(n, d // 2, 2).contiguous()) * rot).reshape(n, d)


def restated_step(W: Weights, tok, s, block_row, kpool, vpool, gains=None, bias=None):
    """One decode step of one row; returns (residual entering each layer and the
    last [L+1][H], logits [V], routing ids [L][k])."""
    sh = W.shape
    L, H, nq, nkv, d, k = sh.n_layers, sh.hidden, sh.n_q, sh.n_kv, sh.head_dim, sh.top_k
    G, P = nq // nkv, sh.page_size
    pos = s - 1
    ones = torch.ones(H, dtype=torch.float64)
    h = W.emb[tok].clone()
    hidden, ids_all = [h.clone()], []
    t_all = torch.arange(s)
    pages = torch.as_tensor(block_row, dtype=torch.long)[t_all // P]
    offs = t_all % P
    for l in range(L):
        gam = torch.from_numpy(gains[0][l].astype(np.float64)) if gains is not None else ones
        x = F.rms_norm(h, (H,), gam, eps=sh.eps)
        qkv = W.wqkv[l] @ x
        q = rope_complex(qkv[:nq * d].view(nq, d), pos, sh.rope_base)
        kn = rope_complex(qkv[nq * d:(nq + nkv) * d].view(nkv, d), pos, sh.rope_base)
        vn = qkv[(nq + nkv) * d:].view(nkv, d)
        # the pool is BF16: the new entry is rounded on its way in
        kn = kn.float().bfloat16().double()
        vn = vn.float().bfloat16().double()
        K = _bf16(kpool[l][pages.numpy(), :, offs.numpy(), :])  # [s, nkv, d]
        V = _bf16(vpool[l][pages.numpy(), :, offs.numpy(), :])
        K[pos], V[pos] = kn, vn
        lo = 0 if sh.is_full_layer(l) else max(0, s - sh.window)
        Kh = K[lo:].permute(1, 0, 2).repeat_interleave(G, dim=0)  # [nq, n, d]
        Vh = V[lo:].permute(1, 0, 2).repeat_interleave(G, dim=0)
        a = F.scaled_dot_product_attention(q[:, None, :], Kh, Vh, scale=1.0 / math.sqrt(d))
        o = W.wo[l] @ a.reshape(nq * d)
        r = W.wr[l] @ x
        if bias is not None:
            r = r + torch.from_numpy(np.asarray(bias, np.float64))
        r32 = r.float()
        top = torch.topk(r32, k + 1)
        assert top.values[k - 1] > top.values[k]  # no tie at the boundary for these inputs
        ids = top.indices[:k]
        w = torch.softmax(r[ids], 0)
        moe = torch.zeros(H, dtype=torch.float64)
        for j in range(k):
            g_, u_, d_ = W.expert(l, int(ids[j]))
            moe += w[j] * (d_ @ (F.silu(g_ @ x) * (u_ @ x)))
        h = h + o + moe
        hidden.append(h.clone())
        ids_all.append([int(e) for e in ids])
    gf = torch.from_numpy(gains[1].astype(np.float64)) if gains is not None else ones
    logits = W.wlm @ F.rms_norm(h, (H,), gf, eps=sh.eps)
    return torch.stack(hidden).numpy(), logits.numpy(), np.array(ids_all)


@pytest.mark.parametrize("workload", ["tiny", "tiny_gains", "small", "small_gains"])
def test_whole_step_matches_restatement(workload):
    inp = synth.make_inputs(workload)
    w = inp.workload
    sh = w.shape
    gains = synth.gains_host(sh, w.seed) if w.gains else None
    ref = oracle.decode_step(sh, w.seed, inp.tokens, inp.seq_lens, inp.block_tables, inp.router_bias,
                             want_hidden=True, gains=gains)
    W = Weights(sh, w.seed)
    kp, vp = host_pools(sh, w.seed, inp.num_pages)
    hid, logits, ids = restated_step(W, int(inp.tokens[0]), int(inp.seq_lens[0]), inp.block_tables[0], kp, vp,
                                     gains, inp.router_bias)
    assert np.array_equal(ids, ref.ids[:, 0, :])
    for l in range(sh.n_layers + 1):
        err = np.max(np.abs(hid[l] - ref.hidden[l, 0])) / np.max(np.abs(hid[l]))
        assert err < 1e-12, (l, err)
    lerr = np.max(np.abs(logits - ref.logits[0])) / np.max(np.abs(logits))
    assert lerr < 1e-12, lerr


def test_gains_change_the_step():
    """Non-unit gains reach every layer's norm and the final norm (a gain that
    is read but not applied, or applied at one layer only, changes nothing)."""
    inp = synth.make_inputs("tiny")
    w = inp.workload
    sh = w.shape
    ng, fg = synth.gains_host(sh, 77)
    base = oracle.decode_step(sh, w.seed, inp.tokens, inp.seq_lens, inp.block_tables, want_hidden=True)
    ones_g = oracle.decode_step(sh, w.seed, inp.tokens, inp.seq_lens, inp.block_tables, want_hidden=True,
                                gains=(np.ones_like(ng), np.ones_like(fg)))
    assert np.array_equal(base.logits, ones_g.logits)
    only_final = oracle.decode_step(sh, w.seed, inp.tokens, inp.seq_lens, inp.block_tables, want_hidden=True,
                                    gains=(np.ones_like(ng), fg))
    assert np.array_equal(only_final.hidden, base.hidden)  # the final gain touches only the logits
    assert not np.allclose(only_final.logits, base.logits)
    for l in range(sh.n_layers):
        g = np.ones_like(ng)
        g[l] = ng[l]
        r = oracle.decode_step(sh, w.seed, inp.tokens, inp.seq_lens, inp.block_tables, want_hidden=True,
                               gains=(g, np.ones_like(fg)))
        assert np.array_equal(r.hidden[:l + 1], base.hidden[:l + 1])  # layers before l untouched
        assert not np.allclose(r.hidden[l + 1], base.hidden[l + 1])


def test_gains_generator():
    """Gains lie in [0.5, 2), both binades occur, the final norm's stream is
    not a layer's, and the values are reproducible."""
    sh = synth.MODELS["small"]
    ng, fg = synth.gains_host(sh, 5)
    assert ng.shape == (sh.n_layers, sh.hidden) and fg.shape == (sh.hidden,)
    allg = np.concatenate([ng.ravel(), fg])
    assert allg.min() >= 0.5 and allg.max() < 2.0
    assert 0.4 < np.mean(allg >= 1.0) < 0.6
    assert not any(np.array_equal(fg, ng[l]) for l in range(sh.n_layers))
    ng2, fg2 = synth.gains_host(sh, 5)
    assert np.array_equal(ng, ng2) and np.array_equal(fg, fg2)


def test_explicit_pool_equals_generator_pool():
    """The generator's pool passed explicitly gives bit-identical results (same
    values, same summation order), and the step writes exactly the new
    token's K/V (BF16) at position seq_len - 1 and nothing else."""
    inp = synth.make_inputs("tiny")
    w = inp.workload
    sh = w.shape
    gen = oracle.decode_step(sh, w.seed, inp.tokens, inp.seq_lens, inp.block_tables, want_kv=True)
    kp, vp = host_pools(sh, w.seed, inp.num_pages)
    k0, v0 = kp.copy(), vp.copy()
    exp = oracle.decode_step(sh, w.seed, inp.tokens, inp.seq_lens, inp.block_tables, pools=(kp, vp))
    assert np.array_equal(gen.logits, exp.logits)
    pos = int(inp.seq_lens[0]) - 1
    page, off = int(inp.block_tables[0, pos // sh.page_size]), pos % sh.page_size
    changed = np.argwhere((kp != k0).any(axis=-1))
    assert {(int(c[1]), int(c[3])) for c in changed} <= {(page, off)}
    for l in range(sh.n_layers):
        for g in range(sh.n_kv):
            for pool, which in ((kp, 0), (vp, 1)):
                got = synth.bf16_bits_to_f32(pool[l, page, g, off])
                ref = torch.from_numpy(gen.kv_new[l, 0, which, g]).float().bfloat16().float().numpy()
                assert np.array_equal(got, ref), (l, g, which)


def test_paged_equals_contiguous():
    """Attention through a shuffled block table equals attention over the same
    keys laid out contiguously (identity block table): bit-identical logits."""
    inp = synth.make_inputs("tiny")  # a shuffled block table over 4 pages
    w = inp.workload
    sh = w.shape
    bt = inp.block_tables
    assert not np.array_equal(bt[0], np.arange(bt.shape[1]))
    kp, vp = host_pools(sh, w.seed, inp.num_pages)
    n = bt.shape[1]
    kc, vc = np.ascontiguousarray(kp[:, bt[0]]), np.ascontiguousarray(vp[:, bt[0]])  # logical order
    ident = np.arange(n, dtype=np.int32)[None, :]
    a = oracle.decode_step(sh, w.seed, inp.tokens, inp.seq_lens, bt, pools=(kp, vp), want_hidden=True)
    b = oracle.decode_step(sh, w.seed, inp.tokens, inp.seq_lens, ident, pools=(kc, vc), want_hidden=True)
    assert np.array_equal(a.logits, b.logits)
    assert np.array_equal(a.hidden, b.hidden)
    assert np.array_equal(kp[:, bt[0]], kc) and np.array_equal(vp[:, bt[0]], vc)  # same writes
    # and a wrong layout (pages in another order) does change the step
    perm = np.roll(np.arange(n), 1)
    c = oracle.decode_step(sh, w.seed, inp.tokens, inp.seq_lens, ident,
                           pools=(np.ascontiguousarray(kp[:, bt[0][perm]]), np.ascontiguousarray(vp[:, bt[0][perm]])))
    assert not np.array_equal(a.logits, c.logits)


def test_consecutive_steps_read_what_earlier_steps_wrote():
    """Two steps over explicit pools: the second attends over the K/V the
    first one wrote, as the restatement over the updated pool says."""
    sh = synth.MODELS["tiny"]
    seed, P = 41, sh.page_size
    sl = np.array([30], np.int32)
    bt, npages = synth.block_tables_for(np.array([40]), P, seed)
    kp, vp = host_pools(sh, seed, npages)
    first = oracle.decode_step(sh, seed, np.array([5], np.int32), sl, bt, pools=(kp, vp))
    nxt = int(np.argmax(first.logits[0]))
    k_after, v_after = kp.copy(), vp.copy()
    second = oracle.decode_step(sh, seed, np.array([nxt], np.int32), sl + 1, bt, pools=(kp, vp))
    W = Weights(sh, seed)
    _, logits, _ = restated_step(W, nxt, 31, bt[0], k_after, v_after)
    assert np.max(np.abs(logits - second.logits[0])) / np.max(np.abs(logits)) < 1e-12
    # without the first step's write the second step differs
    k0, v0 = host_pools(sh, seed, npages)
    _, stale, _ = restated_step(W, nxt, 31, bt[0], k0, v0)
    assert np.max(np.abs(stale - second.logits[0])) / np.max(np.abs(stale)) > 1e-6


# -------------------------------------------------------- the MoE work queue

def _queue_by_sort(ids, E):
    """The canonical queue by library routines: a stable sort of the routed
    entries by expert id, bincount and cumsum."""
    flat = np.asarray(ids).ravel()
    rows = np.argsort(flat, kind="stable").astype(np.int32)
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    act = np.array([[e, offsets[e], counts[e]] for e in range(E) if counts[e] > 0], np.int32).reshape(-1, 3)
    return counts, offsets, rows, act


@pytest.mark.parametrize("B,k,E", [(1, 8, 128), (2, 4, 16), (5, 4, 32), (32, 8, 128), (64, 8, 128), (3, 1, 1)])
def test_route_queue_matches_stable_sort(B, k, E):
    rng = np.random.default_rng(B * 1000 + k)
    # rows of distinct experts (a top-k), skewed towards low ids
    ids = np.stack([rng.choice(E, size=k, replace=False, p=(np.arange(E, 0, -1) / (E * (E + 1) / 2)))
                    for _ in range(B)]).astype(np.int32)
    q = oracle.route_queue(ids, E)
    c, o, r, a = _queue_by_sort(ids, E)
    assert np.array_equal(q.counts, c) and np.array_equal(q.offsets, o)
    assert np.array_equal(q.rows, r) and np.array_equal(q.active, a)
    # invariants: a permutation of the entries, each list segment holds its expert
    assert sorted(q.rows.tolist()) == list(range(B * k))
    for e, off, n in q.active:
        seg = q.rows[off:off + n]
        assert all(ids.ravel()[i] == e for i in seg) and list(seg) == sorted(seg)


def test_route_queue_closed_form():
    # rows 0: experts (3, 1), 1: (1, 0): counts 1, 2, 0, 1; list = [b1j1 | b0j1, b1j0 | b0j0]
    q = oracle.route_queue(np.array([[3, 1], [1, 0]], np.int32), 4)
    assert q.counts.tolist() == [1, 2, 0, 1]
    assert q.offsets.tolist() == [0, 1, 3, 3, 4]
    assert q.rows.tolist() == [3, 1, 2, 0]
    assert q.active.tolist() == [[0, 0, 1], [1, 1, 2], [3, 3, 1]]
    with pytest.raises(ValueError):
        oracle.route_queue(np.array([[4]], np.int32), 4)
