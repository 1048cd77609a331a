#!/usr/bin/env python
"""Decode throughput of the GB300 decode megakernel.

One step = one decode step of the full-shape parallel-attention/MoE model
(48 layers, hidden 2048, 32 q / 4 kv heads of 128, 128 experts top-8,
intermediate 768, vocab 65536) at batch 1 with an 8192-token context, from
the token ids to the logits, through the C ABI (mk_decode_step).  Weights
(random BF16 ~ N(0, 0.02)) and the KV cache (random BF16 ~ N(0, 1)) are
synthetic and resident in HBM; every step streams 6.2 GB, far more than the
129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference]

--impl reference times the CPU oracle (oracle/, plain fp64 C) on the host's
cores for the same workload and metric.  N > 1 runs N independent replicas
(the step has no exchange between GPUs), one per rank under torchrun.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tok/s at bs1 8K ctx (1 GB300); achieved HBM TB/s as % of speed-of-light"
UNIT = "tok/s"
SOL_TBPS = 8.0  # the speed-of-light bandwidth the metric is quoted against


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--workload", default="full_bs1_8k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--trace", default="", help="write a Chrome trace of one step here")
    ap.add_argument("--opts", nargs="*", default=[], metavar="KEY=VALUE",
                    help="schedule options (mk_sched_opts fields, e.g. wave_order=1 placement=3) for "
                         "the timed schedule; the line's config names them")
    ap.add_argument("--service", type=int, default=0,
                    help="time G tokens of the host decode service (GPU step, greedy) after an "
                         "8191-token prompt, instead of the contract line")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's x: N replicas take as long as the slowest."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput of `world` replicas that each processed
    `units_per_rank` units within `ms` milliseconds."""
    return world * units_per_rank / (ms / 1e3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel sources as they are now (else None)."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    from moe_decode_megakernel_gb300.build import source_hash
    if kv.get("kernel_sources_sha256") != source_hash():
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        pass

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            text, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            text, _ = self.proc.communicate()
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in text.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "power_w_max": max(power), "reasons": sorted(reasons)}


def cpu_oracle_rate(inp, budget_s: float = 20.0):
    """The CPU oracle (as it stands) on this host's cores: whole decode steps of
    the same workload until about budget_s seconds have passed."""
    import oracle
    w = inp.workload
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.decode_step(w.shape, w.seed, inp.tokens, inp.seq_lens, inp.block_tables,
                           inp.router_bias)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (el / n) * (n + 1) > 2.5 * budget_s:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    threads = int(os.environ.get("OMP_NUM_THREADS", cores))
    return {"value": w.batch * n / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n} whole decode step(s) of the {w.name} workload ({el:.1f} s)"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import synth
    inp = synth.make_inputs(args.workload)
    w = inp.workload
    # a step of the reference arm is one whole decode step on the CPU; the run is
    # bounded to about a minute however many steps were asked for
    import oracle
    oracle.decode_step(w.shape, w.seed, inp.tokens, inp.seq_lens, inp.block_tables,
                       inp.router_bias)  # warm-up (page-in, thread pool)
    times = []
    t_all = time.perf_counter()
    for _ in range(max(1, args.steps)):
        t0 = time.perf_counter()
        oracle.decode_step(w.shape, w.seed, inp.tokens, inp.seq_lens, inp.block_tables,
                           inp.router_bias)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all > 60.0:
            break
    total = sum(times)
    value = w.batch * len(times) / total
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": len(times), "warmup": 1, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, inp),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": int(os.environ.get("OMP_NUM_THREADS", cores)),
                         "kind": "oracle",
                         "sample": f"{len(times)} whole decode step(s) of {w.name} (bounded to ~60 s)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def dtype_text(sh):
    if sh.expert_fp8:
        return "f32 (fp8 E4M3 experts, bf16 other weights and KV)"
    if sh.expert_fp4:
        return "f32 (fp4 E2M1 experts with E4M3 block scales, bf16 other weights and KV)"
    return "f32 (bf16 weights and KV)"


def weights_text(sh):
    if sh.expert_fp8:
        return ("experts: E4M3 codes with one fp32 scale per output row (std 0.02 to 0.03 after "
                "scaling); the rest bf16 random N(0,0.02)")
    if sh.expert_fp4:
        return ("experts: E2M1 codes, an E4M3 scale per 16 inputs and an fp32 scale per output row "
                "(std about 0.02 after scaling); the rest bf16 random N(0,0.02)")
    return "bf16 random N(0,0.02)"


def workload_config(w, inp):
    sh = w.shape
    attn = (f"sliding window {sh.window} except every {sh.full_period}th layer" if sh.window
            else "full attention on every layer")
    return {"workload": w.name, "model": (f"{sh.n_layers} parallel attention/MoE layers, hidden {sh.hidden}, "
                                          f"{sh.n_q}q/{sh.n_kv}kv heads x {sh.head_dim}, {sh.n_experts} experts "
                                          f"top-{sh.top_k}, intermediate {sh.inter}, vocab {sh.vocab}, {attn}"),
            "global_batch": int(w.batch), "seq_len": int(inp.seq_lens.max()), "page_size": sh.page_size,
            "weights": weights_text(sh), "kv": "bf16 random N(0,1)",
            "l2": "inputs larger than L2 (whole model and KV streamed every step), no flush",
            "parallelism": "replicas (no cross-GPU exchange)"}


def run_mine(args):
    import numpy as np
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import synth
    import synth.device
    import moe_decode_megakernel_gb300 as mk

    inp = synth.make_inputs(args.workload)
    w = inp.workload
    sh = w.shape
    weights = synth.device.device_weights(sh, w.seed, device=dev, router_bias=inp.router_bias)
    kp, vp = synth.device.device_pools(sh, w.seed, inp.num_pages, device=dev)
    model = mk.Model(mk.config_from(sh), mk.weights_from(weights), keepalive=weights)
    sched_opts = {k: int(v) for k, v in (o.split("=", 1) for o in args.opts)}
    sched = mk.Sched(model, w.batch, int(inp.seq_lens.max()), mk.default_sched_opts(**sched_opts))
    sess = mk.Session(model, sched, device=dev)
    stream = torch.cuda.current_stream(dev)
    tok = torch.as_tensor(inp.tokens, device=dev)
    sl = torch.as_tensor(inp.seq_lens, device=dev)
    bt = torch.as_tensor(inp.block_tables, device=dev)
    logits = torch.empty(w.batch, sh.vocab, dtype=torch.float32, device=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(max(3, args.warmup)):
        sess.step(tok, sl, bt, kp, vp, logits)
    sess.check()
    torch.cuda.synchronize()

    # ---- device-timed: inputs resident in HBM
    K = args.steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").replace(",", "").isdigit() else local
    sampler = ClockSampler(gpu_index).__enter__()
    barrier()
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(K):
        sess.step(tok, sl, bt, kp, vp, logits)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    sess.check()
    step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(K)]
    total_ms = max_over_ranks(ev[0].elapsed_time(ev[K]), world, dev)
    value = job_rate(w.batch * K, world, total_ms)

    # ---- end to end through the C ABI: host inputs in, host logits out
    h_tok = torch.as_tensor(inp.tokens).pin_memory()
    h_sl = torch.as_tensor(inp.seq_lens).pin_memory()
    h_bt = torch.as_tensor(inp.block_tables).pin_memory()
    h_logits = torch.empty(w.batch, sh.vocab, dtype=torch.float32).pin_memory()
    d_tok, d_sl, d_bt = torch.empty_like(tok), torch.empty_like(sl), torch.empty_like(bt)
    Ke = max(10, K // 3)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    for _ in range(Ke):
        d_tok.copy_(h_tok, non_blocking=True)
        d_sl.copy_(h_sl, non_blocking=True)
        d_bt.copy_(h_bt, non_blocking=True)
        sess.step(d_tok, d_sl, d_bt, kp, vp, logits)
        h_logits.copy_(logits, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier()
    e2e_ms = max_over_ranks(max(e0.elapsed_time(e1), wall * 1e3), world, dev)
    e2e_value = job_rate(w.batch * Ke, world, e2e_ms)
    h2d = (h_tok.numel() + h_sl.numel() + h_bt.numel()) * 4
    d2h = h_logits.numel() * 4

    # ---- roofline: algorithmic bytes of a step / its device time
    L = sh.n_layers
    ids = sess.region("topk_ids", torch.int32, L * w.batch * sh.top_k).view(L, w.batch, sh.top_k).cpu().numpy()
    distinct = sum(len(np.unique(ids[l])) for l in range(L))
    weight_bytes = L * sh.nonexpert_layer_bytes() + distinct * sh.expert_bytes() + 2 * sh.vocab * sh.hidden
    kv_bytes = synth.step_kv_bytes(sh, inp.seq_lens)
    alg = weight_bytes + kv_bytes
    mean_ms = total_ms / K
    peak, peak_kind = measured_peaks()
    achieved = alg / (mean_ms / 1e3) / 1e9
    # (the recorded traffic is the default schedule's)
    traffic = recorded_traffic(args.workload) if not sched_opts else None

    if args.trace:
        from moe_decode_megakernel_gb300 import trace as mktrace
        tsched = mk.Sched(model, w.batch, int(inp.seq_lens.max()), mk.default_sched_opts(trace=1, **sched_opts))
        tsess = mk.Session(model, tsched, device=dev)
        for _ in range(3):
            tsess.step(tok, sl, bt, kp, vp, logits)
        tsess.check()
        t = mktrace.read(tsess)
        mktrace.chrome_trace(t, args.trace)
        if rank == 0:
            print(mktrace.summary(t), file=sys.stderr)
            print(mktrace.phases(t), file=sys.stderr)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_rate(inp)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": mean_ms,
            "ms_per_step_median": statistics.median(step_ms),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": dtype_text(sh), "data": "synthetic",
            "config": dict(workload_config(w, inp), **({"sched_opts": sched_opts} if sched_opts else {})),
            "hbm_bytes_per_step": alg, "achieved_TBps": achieved / 1e3,
            "frac_of_sol_8TBps": achieved / 1e3 / SOL_TBPS,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                         "traffic": traffic},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": K,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "pages_reference": {"value": 292, "unit": UNIT, "hardware": "1x H100 (132 SMs)",
                                "note": "the pages' own megakernel on its own model: context, not the target"},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_service(args):
    """The host decode service (include/mk_service.h) on the full model at batch
    1: one sequence whose 8191-token prompt is fed one token per step, then G
    greedy tokens timed through mk_service_run (each step: inputs copied in,
    the megakernel, the device argmax, the token copied back, the host's
    bookkeeping) against the megakernel alone at the same contexts."""
    import numpy as np
    import torch
    import synth
    import synth.device
    import moe_decode_megakernel_gb300 as mk
    from moe_decode_megakernel_gb300 import service as sv
    G = args.service
    sh = synth.MODELS["full"]
    seed, P = 3, 8191
    ctx = P + G
    page = sh.page_size
    max_pages = (ctx + page - 1) // page
    weights = synth.device.device_weights(sh, seed)
    model = mk.Model(mk.config_from(sh), mk.weights_from(weights), keepalive=weights)
    kp, vp = synth.device.device_pools(sh, seed, max_pages)
    sched = mk.Sched(model, 1, ctx)
    gstep = sv.GpuStep(model, [sched], kp, vp, max_pages)
    svc = sv.Service(max_pages, page, max_pages, 1, gstep)
    prompt = np.random.default_rng(seed).integers(0, sh.vocab, P)
    svc.add(1, prompt, max_new=G)
    svc.run(max_steps=P - 1)  # the prompt but its last token
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    out = svc.run()  # the last prompt token, then G - 1 fed samples: G steps, G tokens
    wall = time.perf_counter() - t0
    assert len(out[1]) == G and svc.last_run_steps == G
    # the megakernel alone over the same contexts (the pool holds the service's pages)
    sess = mk.Session(model, sched)
    # the only sequence of a fresh service holds pages 0, 1, ... in order
    bt = torch.arange(max_pages, dtype=torch.int32, device="cuda")[None, :]
    logits = torch.empty(1, sh.vocab, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    lens = [torch.tensor([P + i + 1], dtype=torch.int32, device="cuda") for i in range(G)]
    for i in range(3):
        sess.step(tok, lens[0], bt, kp, vp, logits)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(G):
        sess.step(tok, lens[i], bt, kp, vp, logits)
    e1.record()
    torch.cuda.synchronize()
    sess.check()
    kernel_ms = e0.elapsed_time(e1) / G
    print(json.dumps({
        "mode": "service", "metric": "host decode service tok/s (GPU step, greedy), batch 1",
        "value": G / wall, "unit": "tok/s", "tokens": G, "context": [P + 1, P + G],
        "ms_per_token": 1e3 * wall / G, "kernel_ms_per_step": kernel_ms,
        "host_and_copies_ms_per_step": 1e3 * wall / G - kernel_ms,
        "config": {"workload": "full shape, one sequence, 8191-token prompt fed token by token",
                   "weights": "bf16 random N(0,0.02)", "data": "synthetic"}}), flush=True)


def main():
    args = parse()
    if args.service:
        run_service(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_mine(args)


if __name__ == "__main__":
    main()
