"""Runs the decode step on the GPU through the C ABI and compares it with the
CPU oracle (test infrastructure).

Routing: both sides decide the top-k in binary32.  Where the oracle's logits
put two experts within `margin_tol` of the k-th/(k+1)-th boundary, either
choice is correct; the oracle then follows the GPU's choice (force_ids) so
that the rest of the step stays comparable, and the check is that every GPU
choice is a valid top-k of the oracle's logits within that tolerance.
"""
from __future__ import annotations

import gc
from dataclasses import dataclass

import numpy as np
import torch

import oracle
import synth
import synth.device
import moe_decode_megakernel_gb300 as mk

LOGIT_TOL = 2e-2      # max |gpu - oracle| / max |oracle| per row
MARGIN_TOL = 1e-3     # router-logit gap below which a top-k swap is a tie
# Router logits: half the tie margin.  Two logits whose oracle values are
# more than MARGIN_TOL apart cannot swap when each is within MARGIN_TOL / 2 of
# the oracle's, so the routing is exact away from ties.
ROUTER_TOL = MARGIN_TOL / 2

_cache: dict = {}


def _device_model(shape, seed, bias, gains=False):
    key = (shape, seed, None if bias is None else bias.tobytes(), gains)
    if _cache.get("key") != key:
        _cache.clear()
        gc.collect()
        torch.cuda.empty_cache()
        w = synth.device.device_weights(shape, seed, router_bias=bias, gains=gains)
        model = mk.Model(mk.config_from(shape), mk.weights_from(w), keepalive=w)
        _cache.update(key=key, w=w, model=model)
    return _cache["model"]


def release():
    _cache.clear()
    gc.collect()
    torch.cuda.empty_cache()


@dataclass
class GpuStep:
    logits: np.ndarray   # [B, V] fp32
    ids: np.ndarray      # [L, B, k]
    weights: np.ndarray  # [L, B, k]
    kv_k: np.ndarray     # [L, B, n_kv, d] new K as written to the pool (bf16 -> f32)
    kv_v: np.ndarray
    session: object
    extra: dict


def run_gpu(inp: synth.StepInputs, opts=None, steps: int = 1) -> GpuStep:
    w = inp.workload
    shape, B = w.shape, w.batch
    model = _device_model(shape, w.seed, inp.router_bias, w.gains)
    o = opts if opts is not None else mk.default_sched_opts()
    sched = mk.Sched(model, B, int(inp.seq_lens.max()), o)
    sess = mk.Session(model, sched)
    dev = "cuda"
    kp, vp = synth.device.device_pools(shape, w.seed, inp.num_pages)
    tok = torch.as_tensor(inp.tokens, device=dev)
    sl = torch.as_tensor(inp.seq_lens, device=dev)
    bt = torch.as_tensor(inp.block_tables, device=dev)
    logits = torch.empty(B, shape.vocab, dtype=torch.float32, device=dev)
    for _ in range(steps):
        sess.step(tok, sl, bt, kp, vp, logits)
    sess.check()
    torch.cuda.synchronize()
    L, K = shape.n_layers, shape.top_k
    ids = sess.region("topk_ids", torch.int32, L * B * K).view(L, B, K)  # stride MB == B
    rlog = sess.region("router_logits", torch.float32, L * B * shape.n_experts).view(L, B, -1)
    wts = sess.region("topk_w", torch.float32, L * B * K).view(L, B, K)
    # the new K/V of every layer, read back from the pool at position seq_len - 1
    pos = inp.seq_lens - 1
    P = shape.page_size
    pages = inp.block_tables[np.arange(B), pos // P]
    kk = torch.stack([kp[:, int(pages[b]), :, int(pos[b] % P), :] for b in range(B)], 1)
    vv = torch.stack([vp[:, int(pages[b]), :, int(pos[b] % P), :] for b in range(B)], 1)
    to_f = lambda t: synth.bf16_bits_to_f32(t.cpu().numpy())
    extra = {"router_logits": rlog.cpu().numpy().copy()}
    if o.trace_queue:
        E = shape.n_experts
        stride = queue_trace_stride(E, B * K)
        extra["queue_trace"] = sess.region("queue_trace", torch.int32, L * stride).view(L, stride).cpu().numpy()
        extra["expert_count"] = sess.region("expert_count", torch.int32, L * E).view(L, E).cpu().numpy()
    res = GpuStep(logits.cpu().numpy(), ids.cpu().numpy().copy(), wts.cpu().numpy().copy(),
                  to_f(kk), to_f(vv), sess, extra)
    del kp, vp
    return res


def queue_trace_stride(E: int, n_routed_max: int) -> int:
    """Ints per layer of the "queue_trace" region (the layout mk.h states)."""
    return (4 * E + (E + 1) + n_routed_max + 2 + 3) // 4 * 4


def compare_queue(inp: synth.StepInputs, g: GpuStep) -> int:
    """Every layer's MoE work queue as the GPU built it (active-expert list,
    offsets, expert-ordered rows, counts) against the oracle's canonical queue
    of the GPU's own routing: bit-exact.  Returns the layers checked."""
    w = inp.workload
    L, K, E, B = w.shape.n_layers, w.shape.top_k, w.shape.n_experts, w.batch
    qt = g.extra["queue_trace"]
    for l in range(L):
        ref = oracle.route_queue(g.ids[l, :B], E)
        rec = qt[l]
        n_act, n_rows = int(rec[5 * E + 1 + B * K]), int(rec[5 * E + 1 + B * K + 1])
        assert n_act == len(ref.active) and n_rows == B * K, (l, n_act, n_rows)
        act = rec[:4 * E].reshape(E, 4)[:n_act]
        assert np.array_equal(act[:, :3], ref.active), (l, act[:, :3], ref.active)
        assert np.array_equal(rec[4 * E:5 * E + 1], ref.offsets), l
        assert np.array_equal(rec[5 * E + 1:5 * E + 1 + B * K], ref.rows), l
        assert np.array_equal(g.extra["expert_count"][l], ref.counts), l
    return L


def bf16_round(a):
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return synth.bf16_bits_to_f32(u.astype(np.uint16))


@dataclass
class Report:
    max_rel_err: float
    rows_rel_err: np.ndarray
    exact_routing: int
    tie_routing: int
    total_routing: int
    greedy_agree: int     # argmax equal, or within the logit tolerance of a near-tie
    greedy_total: int
    greedy_exact: int     # argmax equal
    kv_max_err: float
    router_err: np.ndarray  # per layer: max |gpu - oracle| router logit
    weight_err: float
    routing_violations: list


def compare(inp: synth.StepInputs, g: GpuStep, rows=None) -> Report:
    w = inp.workload
    shape = w.shape
    B, L, K = w.batch, shape.n_layers, shape.top_k
    rows = np.arange(B) if rows is None else np.asarray(rows)
    # a dense model (one expert, top-1) has no router on the GPU: every row
    # takes expert 0 with weight 1, which is the oracle's routing too
    dense = shape.n_experts == 1 and K == 1
    ids = np.zeros_like(g.ids) if dense else g.ids
    gains = synth.gains_host(shape, w.seed) if w.gains else None
    ref = oracle.decode_step(shape, w.seed, inp.tokens, inp.seq_lens, inp.block_tables,
                             inp.router_bias, rows=rows, force_ids=ids, want_kv=True, gains=gains)
    rerr = np.zeros(L) if dense else np.array(
        [max(float(np.max(np.abs(g.extra["router_logits"][l, b] - ref.router_logits[l, r])))
             for r, b in enumerate(rows)) for l in range(L)])
    # routing: the GPU's experts must be a top-k of the oracle's logits (within a tie)
    exact = ties = 0
    bad = []
    for l in range(L):
        for r, b in enumerate(rows):
            gi = [int(e) for e in ids[l, b]]
            own = [int(e) for e in ref.own_ids[l, r]]
            lg = ref.router_logits[l, r].astype(np.float64)
            assert len(set(gi)) == K and all(0 <= e < shape.n_experts for e in gi), (l, b, gi)
            if gi == own:
                exact += 1
                continue
            kth = np.sort(lg)[::-1][K - 1]
            ok = all(lg[e] >= kth - MARGIN_TOL for e in gi)
            ok &= all(lg[e] <= kth + MARGIN_TOL for e in set(own) - set(gi))
            ok &= all(lg[gi[j]] >= lg[gi[j + 1]] - MARGIN_TOL for j in range(K - 1))
            if ok:
                ties += 1
            else:
                bad.append(f"layer {l} row {b}: GPU experts {gi} vs oracle {own} "
                           f"(logits {lg[gi]} / {lg[own]})")
    # weights: softmax over the chosen logits
    werr = 0.0 if dense else max(float(np.max(np.abs(g.weights[l, b] - ref.weights[l, r])))
                                 for l in range(L) for r, b in enumerate(rows))
    # logits
    errs = []
    agree = exact_greedy = 0
    for r, b in enumerate(rows):
        o = ref.logits[r]
        e = np.max(np.abs(g.logits[b] - o)) / np.max(np.abs(o))
        errs.append(e)
        ga, oa = int(np.argmax(g.logits[b])), int(np.argmax(o))
        exact_greedy += ga == oa
        srt = np.sort(o)[::-1]
        if ga == oa or (o[oa] - o[ga]) <= 2 * LOGIT_TOL * np.max(np.abs(o)) and srt[0] - srt[1] < 1e-2:
            agree += 1
    # new K/V written to the pool: the oracle's values, rounded to BF16
    kvo = ref.kv_new  # [L, R, 2, n_kv, d]
    kerr = 0.0
    for r, b in enumerate(rows):
        for l in range(L):
            for which, gv in ((0, g.kv_k), (1, g.kv_v)):
                want = kvo[l, r, which]
                got = gv[l, b]
                scale = max(1.0, np.max(np.abs(want)))
                kerr = max(kerr, float(np.max(np.abs(got - want)) / scale))
    return Report(float(max(errs)), np.array(errs), exact, ties, L * len(rows), agree, len(rows), exact_greedy,
                  kerr, rerr, werr, bad)
