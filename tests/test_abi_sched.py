"""The C ABI library on the host: it loads, exports what include/mk.h declares,
and its scheduler builds task lists that the validator and the simulator
accept -- and rejects lists with a wrong arrive count or a cyclic wait."""
import os
import re

import numpy as np
import pytest

import synth
import moe_decode_megakernel_gb300 as mk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NUM_SMS = 152


@pytest.fixture(scope="module", autouse=True)
def built():
    if not os.path.exists(mk.LIB_PATH):
        from moe_decode_megakernel_gb300.build import build
        build()


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for h in sorted(os.listdir(inc)):
        if h.endswith(".h"):
            src = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, h)).read(), flags=re.S)
            names |= set(re.findall(r"\b(mk_\w+)\s*\(", src))
    return sorted(names)


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 19 + 19 and "mk_service_step" in names and "mk_gpu_step_run" in names
    L = mk.lib()
    for n in names:
        assert hasattr(L, n), n


def fake_model(shape):
    w = mk.MkWeights(*[0x10000 * (i + 1) for i in range(len(mk.MkWeights._fields_))])
    return mk.Model(mk.config_from(shape), w)


def test_load_model_rejects_unknown_shape():
    from dataclasses import replace
    with pytest.raises(mk.MkError) as e:
        fake_model(replace(synth.MODELS["tiny"], hidden=512))
    assert e.value.code == mk.MK_ERR_UNSUPPORTED
    with pytest.raises(mk.MkError) as e:
        mk.Model(mk.config_from(synth.MODELS["tiny"]), mk.MkWeights())
    assert e.value.code == mk.MK_ERR_ARG


def test_load_model_rejects_misaligned_weights():
    n = len(mk.MkWeights._fields_)
    for i in range(n):  # every pointer is streamed in 16-byte units
        ptrs = [0x10000 * (k + 1) for k in range(n)]
        ptrs[i] += 8
        with pytest.raises(mk.MkError) as e:
            mk.Model(mk.config_from(synth.MODELS["tiny"]), mk.MkWeights(*ptrs))
        assert e.value.code == mk.MK_ERR_ARG, mk.MkWeights._fields_[i]


def sched_for(workload, **opts):
    w = synth.WORKLOADS[workload]
    inp = synth.make_inputs(w)
    m = fake_model(w.shape)
    o = mk.default_sched_opts(num_sms=NUM_SMS, **opts)
    s = mk.Sched(m, w.batch, int(inp.seq_lens.max()), o)
    return m, s, inp


@pytest.mark.parametrize("workload", ["tiny", "small", "full_bs1_8k", "batch32_ragged"])
@pytest.mark.parametrize("order", [0, 1, 2, 3, 4, 5, 6])
def test_schedules_validate_and_simulate(workload, order):
    m, s, inp = sched_for(workload, wave_order=order)
    s.validate()
    s.simulate(inp.seq_lens, seed=order)
    # a shorter batch than the schedule's maximum also completes
    if inp.seq_lens.size > 1:
        s.simulate(inp.seq_lens[:3], seed=7)


@pytest.mark.parametrize("opts", [dict(fuse_finalize=0), dict(fuse_moe_combine=0),
                                  dict(explicit_gather=1), dict(attn_split_pages=1, moe_claimers=5,
                                                               attn_claimers=3),
                                  dict(moe_queue=1), dict(moe_queue=1, moe_claimers=3),
                                  dict(moe_static=0), dict(moe_static=0, moe_claimers=5),
                                  dict(moe_queue=1, moe_static=0), dict(fuse_routing=0),
                                  dict(fuse_routing=0, fuse_finalize=0), dict(fuse_norm_qkv=0),
                                  dict(fuse_norm_qkv=0, fuse_routing=0), dict(combine_per_head=1),
                                  dict(attn_static=0), dict(attn_static=0, attn_claimers=3),
                                  dict(moe_balance=1), dict(placement=1), dict(placement=1, wave_order=1),
                                  dict(placement=1, moe_static=0), dict(placement=1, moe_claimers=5),
                                  dict(placement=2), dict(placement=2, attn_sms=20),
                                  dict(placement=2, wave_order=2), dict(placement=2, moe_static=0),
                                  dict(placement=3), dict(placement=3, wave_order=1),
                                  dict(placement=3, moe_static=0), dict(placement=3, fuse_norm_qkv=0),
                                  dict(placement=4)])
def test_schedule_variants(opts):
    m, s, inp = sched_for("small", **opts)
    s.validate()
    s.simulate(inp.seq_lens, seed=1)


def test_long_context_bucket():
    m, s, inp = sched_for("long_256k")
    s.validate()
    s.simulate(inp.seq_lens, seed=3)


def test_full_list_shape():
    """Every SM gets tasks; one list covers every layer; counts per opcode."""
    m, s, inp = sched_for("full_bs1_8k")
    counts = {}
    for sm in range(s.num_sms):
        n = s.num_tasks(sm)
        assert n > 0
        for i in range(n):
            d = s.get_task(sm, i)
            counts[mk.OPS[int(d[mk.F_OP])]] = counts.get(mk.OPS[int(d[mk.F_OP])], 0) + 1
    sh = synth.MODELS["full"]
    assert counts["RESID_NORM"] == sh.n_layers + 1
    # one QKV tile per SM that holds no routing task (32 to 48 rows, within one
    # KV group); the pages quote 80 tiles of 64
    assert counts["QKV_PROJ"] == sh.n_layers * 140  # 35 per KV group, none on the routing SMs
    # the last router task of a layer runs the top-k: no top-k tasks
    assert counts.get("ROUTER_TOPK", 0) == 0 and counts["ROUTER_GEMM"] == sh.n_layers * 8
    # one up/gate and one down claimer per SM per layer
    assert counts["MOE_UPGATE_ACT_DRAIN"] == counts["MOE_DOWN_DRAIN"] == sh.n_layers * NUM_SMS
    m2, s2, _ = sched_for("full_bs1_8k", moe_queue=1)  # one combined queue
    n_dn = sum(int(s2.get_task(k, i)[mk.F_OP] == 15) for k in range(s2.num_sms) for i in range(s2.num_tasks(k)))
    assert n_dn == 0
    assert counts["ATTN_DRAIN"] > 0 and counts["ATTN_DECODE"] > 0 and counts["LM_HEAD"] > 0


def find_task(s, op, layer=None):
    for sm in range(s.num_sms):
        for i in range(s.num_tasks(sm)):
            d = s.get_task(sm, i)
            if d[mk.F_OP] == op and (layer is None or d[mk.F_LAYER] == layer):
                return sm, i, d
    raise LookupError(op)


def test_dropped_arrive_is_caught():
    m, s, inp = sched_for("tiny")
    sm, i, d = find_task(s, 3, layer=0)  # an O_PROJ task
    d = d.copy()
    d[mk.F_SIG0] = -1
    s.set_task(sm, i, d)
    with pytest.raises(mk.MkError, match="arrivals"):
        s.validate()
    with pytest.raises(mk.MkError, match="deadlock"):
        s.simulate(inp.seq_lens)


def test_doubled_arrive_is_caught():
    m, s, inp = sched_for("tiny")
    sm, i, d = find_task(s, 3, layer=0)
    d = d.copy()
    d[mk.F_SIG1] = d[mk.F_SIG0]  # arrives twice
    s.set_task(sm, i, d)
    with pytest.raises(mk.MkError, match="arrivals"):
        s.validate()
    with pytest.raises(mk.MkError, match="ended at"):
        s.simulate(inp.seq_lens)


def test_wrong_wait_count_is_caught():
    m, s, inp = sched_for("small")
    sm, i, d = find_task(s, 2, layer=3)  # a QKV task waits on the norm
    d = d.copy()
    d[mk.F_TGT0] += 1
    s.set_task(sm, i, d)
    with pytest.raises(mk.MkError):
        s.validate()
    with pytest.raises(mk.MkError, match="deadlock"):
        s.simulate(inp.seq_lens)


def test_cycle_is_caught():
    m, s, inp = sched_for("tiny")
    # layer 0's first RMSNorm waits for the LM head: no order can satisfy it
    sm, i, d = find_task(s, 1, layer=0)
    _, _, lm = find_task(s, 6)
    n_lm = sum(int(s.get_task(k, i)[mk.F_OP] == 6) for k in range(s.num_sms) for i in range(s.num_tasks(k)))
    d = d.copy()
    d[mk.F_WAIT0], d[mk.F_TGT0] = lm[mk.F_SIG0], n_lm
    s.set_task(sm, i, d)
    with pytest.raises(mk.MkError, match="cyclic"):
        s.validate()
    with pytest.raises(mk.MkError, match="deadlock"):
        s.simulate(inp.seq_lens)


def test_rejects_bad_bucket():
    m = fake_model(synth.MODELS["tiny"])
    with pytest.raises(mk.MkError):
        mk.Sched(m, 65, 64, mk.default_sched_opts(num_sms=NUM_SMS))
    with pytest.raises(mk.MkError):
        mk.Sched(m, 1, 0, mk.default_sched_opts(num_sms=NUM_SMS))
    s = mk.Sched(m, 2, 64, mk.default_sched_opts(num_sms=NUM_SMS))
    with pytest.raises(mk.MkError):
        s.simulate([65])  # longer than the bucket


@pytest.mark.parametrize("seq", [[8192, 3000], [8192], [1, 40000]])
def test_two_row_schedule(seq):
    """A schedule for at most two rows: the QKV tiles compute the RMSNorm
    (they wait for what the RMSNorm waits for); one merge task per (row, KV
    group), or per (row, KV group, head); a one-row step on it waits for no
    slices of the absent row."""
    w = synth.WORKLOADS["full_bs1_8k"]
    sh = w.shape
    G = sh.n_q // sh.n_kv
    m = fake_model(sh)
    for per_head in (0, 1):
        s = mk.Sched(m, 2, 40000, mk.default_sched_opts(num_sms=NUM_SMS, combine_per_head=per_head))
        s.validate()
        tasks = [s.get_task(sm, i) for sm in range(s.num_sms) for i in range(s.num_tasks(sm))]
        comb = [d for d in tasks if mk.OPS[int(d[mk.F_OP])] == "ATTN_COMBINE"]
        assert len(comb) == sh.n_layers * 2 * sh.n_kv * (G if per_head else 1)
        heads = sorted({int(d[mk.F_A0 + 3]) for d in comb})
        assert heads == (list(range(G)) if per_head else [-1])
        qkv = [d for d in tasks if mk.OPS[int(d[mk.F_OP])] == "QKV_PROJ"]
        assert all(int(d[mk.F_A0 + 7]) == 1 for d in qkv)
        s.simulate(np.asarray(seq, np.int32), seed=5)


@pytest.mark.parametrize("workload", ["dense_small", "dense_batch5"])
def test_dense_schedules(workload):
    """A dense model: no router, top-k or MoE claimers; one static FFN
    up/gate tile per 64-row slice of the intermediate and one down tile per
    32 outputs, every down tile after all the up/gate tiles of its layer."""
    m, s, inp = sched_for(workload)
    s.validate()
    s.simulate(inp.seq_lens, seed=2)
    sh = synth.WORKLOADS[workload].shape
    counts = {}
    for sm in range(s.num_sms):
        for i in range(s.num_tasks(sm)):
            op = mk.OPS[int(s.get_task(sm, i)[mk.F_OP])]
            counts[op] = counts.get(op, 0) + 1
    assert not any(k in counts for k in ("ROUTER_GEMM", "ROUTER_TOPK", "ROUTE_FINALIZE",
                                          "MOE_UPGATE_ACT_DRAIN", "MOE_DOWN_DRAIN"))
    assert counts["FFN_UPGATE_ACT"] == sh.n_layers * (sh.inter // 64)
    assert counts["FFN_DOWN"] == sh.n_layers * (sh.hidden // 32)


def test_host_input_check_refuses_before_launch():
    """mk_check_inputs: a seq_len beyond the schedule's max_ctx, a page id
    outside the pool, a block table too narrow for the length, a token outside
    the vocabulary or a batch beyond max_batch is MK_ERR_ARG with the row named;
    valid inputs pass.  Host only (no device)."""
    sh = synth.MODELS["tiny"]
    model = fake_model(sh)
    opts = mk.default_sched_opts(num_sms=NUM_SMS)
    s = mk.Sched(model, 4, 64, opts)
    P = sh.page_size
    sl = np.array([64, 17, 1], np.int32)
    bt = np.array([[0, 1, 2, 3], [4, 5, -1, -1], [6, -1, -1, -1]], np.int32)
    tok = np.array([0, 5, sh.vocab - 1], np.int32)
    s.check_inputs(tok, sl, bt, 7)
    s.check_inputs(None, sl, bt, 7)
    cases = [
        (tok, np.array([65, 17, 1], np.int32), bt, 7, "seq_len 65"),      # > max_ctx
        (tok, np.array([64, 0, 1], np.int32), bt, 7, "seq_len 0"),
        (tok, sl, bt, 6, "page 6"),                                        # outside the pool
        (tok, np.array([64, 33, 1], np.int32), bt, 7, "page -1"),          # a page that is not there
        (np.array([0, 5, sh.vocab], np.int32), sl, bt, 7, "token"),
        (tok, sl, bt[:, :2], 7, "needs 4 pages"),
    ]
    for t, l, b, n, what in cases:
        with pytest.raises(mk.MkError) as e:
            s.check_inputs(t, l, b, n)
        assert e.value.code == mk.MK_ERR_ARG and what in str(e.value), (what, str(e.value))
    with pytest.raises(mk.MkError) as e:
        s.check_inputs(np.zeros(5, np.int32), np.full(5, 8, np.int32), np.zeros((5, 1), np.int32), 7)
    assert e.value.code == mk.MK_ERR_ARG and "batch 5" in str(e.value)
    assert P == 16


def test_queue_trace_region_size():
    """The "queue_trace" region holds L records of the stride mk.h states."""
    sh = synth.MODELS["full"]
    model = fake_model(sh)
    for B in (1, 32):
        s = mk.Sched(model, B, 8192, mk.default_sched_opts(num_sms=NUM_SMS, trace_queue=1))
        off = s.workspace_offset("queue_trace")
        stride = (4 * sh.n_experts + sh.n_experts + 1 + B * sh.top_k + 2 + 3) // 4 * 4
        assert off >= 0 and off % 16 == 0
        assert s.workspace_bytes() - off >= sh.n_layers * stride * 4
        assert s.workspace_bytes() - off < sh.n_layers * stride * 4 + 256
        assert mk.Sched(model, B, 8192, mk.default_sched_opts(num_sms=NUM_SMS)).workspace_offset("queue_trace") == -1


@pytest.mark.parametrize("workload", ["full_bs1_8k", "batch32_ragged", "long_256k"])
def test_split_placement_keeps_branches_apart(workload):
    """placement 2: every attention-branch task on SMs [0, attn_sms), every
    MoE-branch task on the others, the LM head over all SMs; the lists
    validate and simulate."""
    w = synth.WORKLOADS[workload]
    for attn_sms in (0, 48):
        m, s, inp = sched_for(workload, placement=2, attn_sms=attn_sms)
        s.validate()
        s.simulate(inp.seq_lens, seed=2)
        attn_ops = {2, 3, 7, 8, 9}
        moe_ops = {1, 10, 11, 12, 13, 14, 15, 16}
        na = None
        lm_sms = set()
        for sm in range(s.num_sms):
            for i in range(s.num_tasks(sm)):
                op, l = int(s.get_task(sm, i)[0]), int(s.get_task(sm, i)[1])
                if op == 6:
                    lm_sms.add(sm)
                elif op in attn_ops:
                    na = sm if na is None else max(na, sm)
        assert len(lm_sms) == s.num_sms
        na += 1
        if attn_sms:
            assert na == attn_sms
        for sm in range(s.num_sms):
            for i in range(s.num_tasks(sm)):
                op, l = int(s.get_task(sm, i)[0]), int(s.get_task(sm, i)[1])
                if l < w.shape.n_layers:
                    assert (op in attn_ops) == (sm < na), (sm, op, l)
                    assert op in attn_ops or op in moe_ops


def test_affinity_placement_follows_producers():
    """placement 3: an attention slice of a sliding layer runs on an SM that
    ran one of its KV group's QKV tiles whenever that SM has room, no SM holds
    more than the per-layer cap, and the lists validate and simulate on the
    full shape."""
    m, s, inp = sched_for("full_bs1_8k", placement=3)
    s.validate()
    s.simulate(inp.seq_lens, seed=3)
    by_layer = {}
    for sm in range(s.num_sms):
        for i in range(s.num_tasks(sm)):
            d = s.get_task(sm, i)
            by_layer.setdefault(int(d[1]), []).append((sm, d))
    colocated = total = 0
    for l, items in by_layer.items():
        cap = -(-len(items) // s.num_sms)
        counts = np.bincount([sm for sm, _ in items], minlength=s.num_sms)
        assert counts.max() <= cap, (l, counts.max(), cap)
        if l >= 48 or synth.MODELS["full"].is_full_layer(l):
            continue
        qkv_sms = {}
        for sm, d in items:
            if int(d[0]) == 2:  # QKV tile: signals the group's QKV barrier
                qkv_sms.setdefault(int(d[6]), set()).add(sm)
        for sm, d in items:
            if int(d[0]) == 7:  # a static slice waits on its group's QKV barrier
                total += 1
                colocated += sm in qkv_sms.get(int(d[2]), set())
    assert total > 0 and colocated >= 0.9 * total, (colocated, total)


def _lists(s):
    return [[tuple(s.get_task(sm, i)) for i in range(s.num_tasks(sm))] for sm in range(s.num_sms)]


@pytest.mark.parametrize("workload,batch,order", [("small", 1, 0), ("full_bs2_8k", 2, 0),
                                                  ("full_bs4_8k", 4, 5), ("batch32_ragged", 32, 1)])
def test_default_wave_order_per_build(workload, batch, order):
    """wave_order -1 (the default) takes the pages' order for batch <= 2
    schedules and, for the tensor-core schedules, O-proj before the down
    tiles up to 8 rows and the interleaved order beyond: the task lists equal
    those of the explicit order."""
    w = synth.WORKLOADS[workload]
    inp = synth.make_inputs(w)
    m = fake_model(w.shape)
    ctx = int(inp.seq_lens.max())
    auto = mk.Sched(m, batch, ctx, mk.default_sched_opts(num_sms=NUM_SMS))
    explicit = mk.Sched(m, batch, ctx, mk.default_sched_opts(num_sms=NUM_SMS, wave_order=order))
    other = mk.Sched(m, batch, ctx, mk.default_sched_opts(num_sms=NUM_SMS, wave_order=2))
    assert _lists(auto) == _lists(explicit)
    assert _lists(auto) != _lists(other)
