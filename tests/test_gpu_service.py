"""The decode service with the GPU step (mk_gpu_step: mk_decode_step plus
the library's argmax) on the tiny model: prompts fed token by token, greedy
samples, two sequences batched -- against one-sequence-at-a-time loops of
mk_decode_step and torch.argmax over the same positions and pages.

"Cohere: a serving engine for North Mini Code built around a decode
megakernel", section "The inference engine around the kernel"."""
import numpy as np
import pytest
import torch

import synth
import synth.device
import moe_decode_megakernel_gb300 as mk
from moe_decode_megakernel_gb300 import service as sv

pytestmark = pytest.mark.gpu

SH = synth.MODELS["tiny"]
SEED = 31
NUM_PAGES = 24
MAX_PAGES = 8


def _model():
    w = synth.device.device_weights(SH, SEED)
    return mk.Model(mk.config_from(SH), mk.weights_from(w), keepalive=w)


def _manual(model, prompt, n_new, pages):
    """One sequence through Session.step: feed the prompt, then the samples."""
    kp, vp = synth.device.device_pools(SH, SEED, NUM_PAGES)
    sched = mk.Sched(model, 1, MAX_PAGES * SH.page_size)
    sess = mk.Session(model, sched)
    bt = torch.full((1, MAX_PAGES), -1, dtype=torch.int32, device="cuda")
    logits = torch.empty(1, SH.vocab, device="cuda")
    feed, out, n_ctx = list(prompt), [], 0
    while len(out) < n_new:
        tok = feed.pop(0)
        bt[0, n_ctx // SH.page_size] = pages[n_ctx // SH.page_size]
        sess.step(torch.tensor([tok], dtype=torch.int32, device="cuda"),
                  torch.tensor([n_ctx + 1], dtype=torch.int32, device="cuda"), bt, kp, vp, logits)
        sess.check()
        n_ctx += 1
        if not feed:
            t = int(torch.argmax(logits[0]).item())
            out.append(t)
            feed.append(t)
    return out


def test_argmax_rows_ties_and_nan():
    g = torch.Generator(device="cuda").manual_seed(3)
    x = torch.randn(5, 1000, device="cuda", generator=g)
    x[1, 10] = x[1, 900] = 50.0  # a tie: the lower index wins
    x[2, :] = float("nan")
    x[2, 17] = 1.0  # NaN never wins
    x[3, :] = -3.0  # all equal: index 0
    nxt = torch.empty(5, dtype=torch.int32, device="cuda")
    sv.argmax_rows(x, nxt, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    ref = torch.argmax(torch.nan_to_num(x, nan=-float("inf")), dim=1).to(torch.int32)
    assert nxt.tolist() == ref.tolist()
    assert nxt[1].item() == 10 and nxt[2].item() == 17 and nxt[3].item() == 0


def test_service_matches_single_sequence_loops():
    model = _model()
    kp, vp = synth.device.device_pools(SH, SEED, NUM_PAGES)
    ctx = MAX_PAGES * SH.page_size
    scheds = [mk.Sched(model, 1, ctx), mk.Sched(model, 2, ctx)]
    gstep = sv.GpuStep(model, scheds, kp, vp, MAX_PAGES)
    svc = sv.Service(NUM_PAGES, SH.page_size, MAX_PAGES, 2, gstep)
    rng = np.random.default_rng(8)
    prompts = {1: rng.integers(0, SH.vocab, 5).tolist(), 2: rng.integers(0, SH.vocab, 21).tolist()}
    svc.add(1, prompts[1], max_new=12)
    svc.add(2, prompts[2], max_new=6)
    pages = {}
    out = {}
    while True:
        for sid in (1, 2):  # record the pages while the sequences hold them
            if svc.query(sid).state != sv.FINISHED:
                pages[sid] = svc.pages(sid)
        rows, toks = svc.step()
        for sid, t in toks:
            out.setdefault(sid, []).append(t)
        if rows == 0:
            break
    assert len(out[1]) == 12 and len(out[2]) == 6
    assert svc.free_pages == NUM_PAGES
    for sid, n in ((1, 12), (2, 6)):
        assert out[sid] == _manual(model, prompts[sid], n, pages[sid]), sid


def test_park_resume_on_the_gpu():
    model = _model()
    kp, vp = synth.device.device_pools(SH, SEED, NUM_PAGES)
    ctx = MAX_PAGES * SH.page_size
    gstep = sv.GpuStep(model, [mk.Sched(model, 2, ctx)], kp, vp, MAX_PAGES)
    svc = sv.Service(NUM_PAGES, SH.page_size, MAX_PAGES, 2, gstep)
    prompt = [3, 14, 15, 92]
    svc.add(5, prompt, max_new=8)
    first = []
    while len(first) < 3:
        _, toks = svc.step()
        first += [t for _, t in toks]
    svc.park(5)
    assert svc.step() == (0, [])
    appended = [65, 35, 89]
    svc.resume(5, appended)
    rest = svc.run()[5]
    # one uninterrupted loop with the appended tokens fed after the third
    # sample, over the same pages (the only sequence: pages 0, 1, ... in order)
    ref = _manual_forced(model, prompt, first, appended, 5, list(range(MAX_PAGES)))
    assert first + rest == ref


def _manual_forced(model, prompt, first, appended, n_more, pages):
    kp, vp = synth.device.device_pools(SH, SEED, NUM_PAGES)
    sched = mk.Sched(model, 1, MAX_PAGES * SH.page_size)
    sess = mk.Session(model, sched)
    bt = torch.full((1, MAX_PAGES), -1, dtype=torch.int32, device="cuda")
    logits = torch.empty(1, SH.vocab, device="cuda")
    out = []
    feed = list(prompt)
    n_ctx = 0
    forced_after = {len(first): list(appended)}
    while len(out) < len(first) + n_more:
        tok = feed.pop(0)
        bt[0, n_ctx // SH.page_size] = pages[n_ctx // SH.page_size]
        sess.step(torch.tensor([tok], dtype=torch.int32, device="cuda"),
                  torch.tensor([n_ctx + 1], dtype=torch.int32, device="cuda"), bt, kp, vp, logits)
        sess.check()
        n_ctx += 1
        if not feed:
            t = int(torch.argmax(logits[0]).item())
            out.append(t)
            feed.append(t)
            feed += forced_after.pop(len(out), [])
    return out


def _host_pools(shape, seed, num_pages):
    """The generator's K and V pools as BF16 bits, the same values the device
    pools start from."""
    per = num_pages * shape.n_kv * shape.page_size * shape.head_dim
    dims = (shape.n_layers, num_pages, shape.n_kv, shape.page_size, shape.head_dim)
    k = synth.fill_host(shape.n_layers, per, seed, synth.KPOOL, vary_layer=True, sigma=shape.kv_sigma)
    v = synth.fill_host(shape.n_layers, per, seed, synth.VPOOL, vary_layer=True, sigma=shape.kv_sigma)
    return k.reshape(dims).copy(), v.reshape(dims).copy()


@pytest.mark.parametrize("name,num_pages,max_pages", [("tiny", 24, 8), ("small", 12, 4)])
def test_service_matches_oracle_over_many_steps(name, num_pages, max_pages):
    """The GPU decode service over 40+ steps (two sequences batched, prompts
    fed token by token, greedy samples, one sequence parked for two steps and
    resumed with appended tokens) against the CPU oracle replaying each
    sequence over its own KV pool: every sample equals the oracle's greedy
    token (teacher-forced with the GPU's samples; a near-tie within the logit
    tolerance may go either way), and the K/V the GPU wrote at every position
    of every layer equal the oracle's: each head's vector within the logits'
    tolerance of its largest entry (later positions depend on the history,
    where single BF16 roundings may go the other way), most entries
    bit-equal."""
    import oracle
    import parity
    sh, seed = synth.MODELS[name], 37
    w = synth.device.device_weights(sh, seed)
    model = mk.Model(mk.config_from(sh), mk.weights_from(w), keepalive=w)
    kp, vp = synth.device.device_pools(sh, seed, num_pages)
    ctx = max_pages * sh.page_size
    gstep = sv.GpuStep(model, [mk.Sched(model, 1, ctx), mk.Sched(model, 2, ctx)], kp, vp, max_pages)
    svc = sv.Service(num_pages, sh.page_size, max_pages, 2, gstep)
    rng = np.random.default_rng(11)
    prompts = {1: rng.integers(0, sh.vocab, 9).tolist(), 2: rng.integers(0, sh.vocab, 21).tolist()}
    appended = [7, 8]
    svc.add(1, prompts[1], max_new=30)
    svc.add(2, prompts[2], max_new=20)
    pages, out, steps = {}, {1: [], 2: []}, 0
    parked_at = None
    while True:
        for sid in (1, 2):
            if svc.query(sid).state != sv.FINISHED:
                pages[sid] = svc.pages(sid)
        rows, toks = svc.step()
        if rows:
            steps += 1
        for sid, t in toks:
            out[sid].append(t)
        if parked_at is None and len(out[1]) == 5:
            svc.park(1)
            parked_at = steps
        elif parked_at is not None and parked_at > 0 and (steps >= parked_at + 2 or rows == 0):
            svc.resume(1, appended)
            parked_at = -1
        if rows == 0 and parked_at == -1:
            break
    assert steps >= 32 and len(out[1]) == 30 and len(out[2]) == 20
    torch.cuda.synchronize()
    kg, vg = kp.cpu().numpy(), vp.cpu().numpy()
    P = sh.page_size
    exact = total = 0
    kv_worst = 0.0
    for sid in (1, 2):
        ko, vo = _host_pools(sh, seed, num_pages)
        bt = np.full((1, max_pages), -1, np.int32)
        bt[0, :len(pages[sid])] = pages[sid]
        feed, n_ctx, k = list(prompts[sid]), 0, 0
        forced_after = {5: list(appended)} if sid == 1 else {}
        while k < len(out[sid]):
            tok = feed.pop(0)
            r = oracle.decode_step(sh, seed, np.array([tok], np.int32), np.array([n_ctx + 1], np.int32), bt,
                                   pools=(ko, vo))
            n_ctx += 1
            if not feed:  # this position produced sample k
                g_tok, o = out[sid][k], r.logits[0]
                oa = int(np.argmax(o))
                exact += g_tok == oa
                total += 1
                assert g_tok == oa or o[oa] - o[g_tok] <= 2 * parity.LOGIT_TOL * np.max(np.abs(o)), (sid, k)
                k += 1
                feed.append(g_tok)
                feed += forced_after.pop(k, [])
        # what the GPU wrote at every position of this sequence
        pos = np.arange(n_ctx)
        pg, off = bt[0, pos // P], pos % P
        for gpool, opool in ((kg, ko), (vg, vo)):
            gv = synth.bf16_bits_to_f32(gpool[:, pg, :, off, :])  # [position][layer][head][d]
            ov = synth.bf16_bits_to_f32(opool[:, pg, :, off, :])
            # each head's vector within the logits' tolerance of its largest entry
            err = np.max(np.abs(gv - ov), axis=-1) / np.max(np.abs(ov), axis=-1)
            kv_worst = max(kv_worst, float(err.max()))
            same = np.mean(gv == ov)
            assert err.max() <= parity.LOGIT_TOL, (sid, float(err.max()))
            assert same >= 0.9, same  # most entries round to the same BF16 value
    print(f"{name}: {steps} service steps, greedy agreement {exact}/{total}, worst K/V error {kv_worst:.2e}")
    assert exact >= 0.99 * total


def test_service_four_sequences_tensor_core_steps():
    """Four sequences decoded together on the small shape (a schedule of 4
    rows: the tensor-core build, its QKV epilogue appending every K/V; the
    2-row schedule once two have finished) over 30+ steps.  Every step is
    replayed by the oracle over the K/V history the GPU wrote (each position
    is written once), so each comparison is of one step: the oracle's new K/V
    against what the GPU wrote at that position (each head vector within the
    logits' tolerance of its largest entry), and its greedy token against the
    GPU's sample (teacher-forced; near-ties within the tolerance either way)."""
    import oracle
    import parity
    sh, seed, num_pages, max_pages = synth.MODELS["small"], 41, 16, 3
    w = synth.device.device_weights(sh, seed)
    model = mk.Model(mk.config_from(sh), mk.weights_from(w), keepalive=w)
    kp, vp = synth.device.device_pools(sh, seed, num_pages)
    ctx = max_pages * sh.page_size
    gstep = sv.GpuStep(model, [mk.Sched(model, 2, ctx), mk.Sched(model, 4, ctx)], kp, vp, max_pages)
    svc = sv.Service(num_pages, sh.page_size, max_pages, 4, gstep)
    rng = np.random.default_rng(13)
    lens, new = {1: 3, 2: 11, 3: 6, 4: 17}, {1: 24, 2: 18, 3: 30, 4: 12}
    prompts = {sid: rng.integers(0, sh.vocab, n).tolist() for sid, n in lens.items()}
    for sid in prompts:
        svc.add(sid, prompts[sid], max_new=new[sid])
    pages, out, steps = {}, {sid: [] for sid in prompts}, 0
    while True:
        for sid in prompts:
            if svc.query(sid).state != sv.FINISHED:
                pages[sid] = svc.pages(sid)
        rows, toks = svc.step()
        if rows == 0:
            break
        steps += 1
        for sid, t in toks:
            out[sid].append(t)
    assert steps >= 30 and all(len(out[sid]) == new[sid] for sid in prompts)
    torch.cuda.synchronize()
    kg, vg = kp.cpu().numpy(), vp.cpu().numpy()
    P = sh.page_size
    exact = total = 0
    kv_worst = 0.0
    for sid in prompts:
        ko, vo = kg.copy(), vg.copy()  # the GPU's history; each position is compared, then restored
        bt = np.full((1, max_pages), -1, np.int32)
        bt[0, :len(pages[sid])] = pages[sid]
        feed, n_ctx, k = list(prompts[sid]), 0, 0
        while k < len(out[sid]):
            tok = feed.pop(0)
            r = oracle.decode_step(sh, seed, np.array([tok], np.int32), np.array([n_ctx + 1], np.int32), bt,
                                   pools=(ko, vo))
            pg, off = bt[0, n_ctx // P], n_ctx % P
            for gpool, opool in ((kg, ko), (vg, vo)):
                gv = synth.bf16_bits_to_f32(gpool[:, pg, :, off, :])  # [layer][head][d]
                ov = synth.bf16_bits_to_f32(opool[:, pg, :, off, :])
                err = np.max(np.abs(gv - ov), axis=-1) / np.max(np.abs(ov), axis=-1)
                kv_worst = max(kv_worst, float(err.max()))
                assert err.max() <= parity.LOGIT_TOL, (sid, n_ctx, float(err.max()))
                opool[:, pg, :, off, :] = gpool[:, pg, :, off, :]
            n_ctx += 1
            if not feed:
                g_tok, o = out[sid][k], r.logits[0]
                oa = int(np.argmax(o))
                exact += g_tok == oa
                total += 1
                assert g_tok == oa or o[oa] - o[g_tok] <= 2 * parity.LOGIT_TOL * np.max(np.abs(o)), (sid, k)
                k += 1
                feed.append(g_tok)
    print(f"small, 4 sequences: {steps} service steps, greedy agreement {exact}/{total}, "
          f"worst one-step K/V error {kv_worst:.2e}")
    assert exact >= 0.99 * total
