"""Model shapes and seeded input recipes of the decode-step workloads.

The decode step belongs to a parallel-attention/MoE transformer (the model of
"Cohere: a decode megakernel for North Mini Code", sections "1. Reduce wave
quantization" and "Tasks").  The pages fix the full-size shape only in part
(128 experts, top-8, BF16, 8K context, ~0.5 GB of KV); the rest of each shape
below is the workload definition these inputs are generated for.

Nothing here computes any part of the decode step: this module only states
shapes and draws seeded integers (tokens, sequence lengths, block tables) and
the router bias that skews routing for the continuous-batching workload.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, asdict

import numpy as np


@dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    hidden: int
    n_q: int
    n_kv: int
    head_dim: int
    n_experts: int
    top_k: int
    inter: int
    vocab: int
    page_size: int
    window: int  # 0: every layer attends to the whole context
    full_period: int  # layer l is full-attention iff window == 0 or (l + 1) % full_period == 0
    rope_base: float = 500000.0
    eps: float = 1e-5
    weight_sigma: float = 0.02
    kv_sigma: float = 1.0
    expert_fp8: bool = False  # expert matrices as E4M3 codes with one scale per output row
    expert_fp4: bool = False  # E2M1 codes, an E4M3 scale per 16 inputs, one fp32 scale per output row

    def is_full_layer(self, layer: int) -> bool:
        return self.window == 0 or (layer + 1) % self.full_period == 0

    def as_dict(self) -> dict:
        return asdict(self)

    # algorithmic byte counts (BF16 weights and KV)
    def qkv_rows(self) -> int:
        return (self.n_q + 2 * self.n_kv) * self.head_dim

    def nonexpert_layer_bytes(self) -> int:
        h = self.hidden
        return 2 * (self.qkv_rows() * h + h * self.n_q * self.head_dim + self.n_experts * h)

    def expert_bytes(self) -> int:
        if self.expert_fp8:  # E4M3 codes plus one fp32 scale per output row
            return 3 * self.hidden * self.inter + 4 * (2 * self.inter + self.hidden)
        if self.expert_fp4:  # half-byte codes, a byte per 16 codes, fp32 per output row
            return 3 * self.hidden * self.inter // 2 + 3 * self.hidden * self.inter // 16 + \
                4 * (2 * self.inter + self.hidden)
        return 2 * 3 * self.hidden * self.inter

    def kv_bytes_per_token_layer(self) -> int:
        return 2 * 2 * self.n_kv * self.head_dim


MODELS = {
    "tiny": ModelShape("tiny", n_layers=2, hidden=256, n_q=4, n_kv=2, head_dim=64, n_experts=16,
                       top_k=4, inter=128, vocab=1024, page_size=16, window=0, full_period=1),
    "small": ModelShape("small", n_layers=8, hidden=1024, n_q=16, n_kv=2, head_dim=64,
                        n_experts=32, top_k=4, inter=512, vocab=32768, page_size=64, window=0,
                        full_period=1),
    "full": ModelShape("full", n_layers=48, hidden=2048, n_q=32, n_kv=4, head_dim=128,
                       n_experts=128, top_k=8, inter=768, vocab=65536, page_size=64,
                       window=4096, full_period=4),
    # the full shape's dimensions in two layers, the second one full-attention:
    # a case small enough for multi-pass profiler captures (about 2.8 GB)
    "full_l2": ModelShape("full_l2", n_layers=2, hidden=2048, n_q=32, n_kv=4, head_dim=128,
                          n_experts=128, top_k=8, inter=768, vocab=65536, page_size=64,
                          window=4096, full_period=2),
    # a dense model: one expert that every token takes with weight 1 is a
    # SwiGLU FFN (intermediate 2048); half the layers sliding-window
    # FP8 expert weights (E4M3 codes, one fp32 scale per output row)
    "small_fp8": ModelShape("small_fp8", n_layers=8, hidden=1024, n_q=16, n_kv=2, head_dim=64,
                            n_experts=32, top_k=4, inter=512, vocab=32768, page_size=64, window=0,
                            full_period=1, expert_fp8=True),
    "full_fp8": ModelShape("full_fp8", n_layers=48, hidden=2048, n_q=32, n_kv=4, head_dim=128,
                           n_experts=128, top_k=8, inter=768, vocab=65536, page_size=64,
                           window=4096, full_period=4, expert_fp8=True),
    # the same two full-shape layers with FP8 experts (profiling case of the FP8 tensor-core build)
    "full_fp8_l2": ModelShape("full_fp8_l2", n_layers=2, hidden=2048, n_q=32, n_kv=4, head_dim=128,
                              n_experts=128, top_k=8, inter=768, vocab=65536, page_size=64,
                              window=4096, full_period=2, expert_fp8=True),
    # FP4 expert weights (E2M1 codes, E4M3 block scales, fp32 row scales)
    "small_fp4": ModelShape("small_fp4", n_layers=8, hidden=1024, n_q=16, n_kv=2, head_dim=64,
                            n_experts=32, top_k=4, inter=512, vocab=32768, page_size=64, window=0,
                            full_period=1, expert_fp4=True),
    "full_fp4": ModelShape("full_fp4", n_layers=48, hidden=2048, n_q=32, n_kv=4, head_dim=128,
                           n_experts=128, top_k=8, inter=768, vocab=65536, page_size=64,
                           window=4096, full_period=4, expert_fp4=True),
    "dense": ModelShape("dense", n_layers=8, hidden=1024, n_q=16, n_kv=2, head_dim=64, n_experts=1,
                        top_k=1, inter=2048, vocab=32768, page_size=64, window=512, full_period=2),
}


@dataclass(frozen=True)
class Workload:
    name: str
    model: str
    batch: int
    seq: tuple  # ("fixed", C) | ("uniform", lo, hi) | ("loguniform", lo, hi)
    seed: int
    zipf: float | None = None
    desc: str = ""
    shape_override: ModelShape | None = None
    gains: bool = False  # seeded RMSNorm gains in [0.5, 2) instead of ones

    @property
    def shape(self) -> ModelShape:
        return self.shape_override if self.shape_override is not None else MODELS[self.model]


WORKLOADS = {
    "tiny": Workload("tiny", "tiny", 1, ("fixed", 64), 1,
                     desc="tiny: 2 layers, B=1, context 64 in 16-token pages, shuffled block table"),
    "small": Workload("small", "small", 1, ("fixed", 1024), 2,
                      desc="small: 8 layers, B=1, context 1024 in 64-token pages"),
    "full_bs1_8k": Workload("full_bs1_8k", "full", 1, ("fixed", 8192), 3,
                            desc="full shape, B=1, context 8192"),
    # the wave-order ablation's other batch sizes (8K context, uniform routing)
    "full_bs2_8k": Workload("full_bs2_8k", "full", 2, ("fixed", 8192), 16,
                            desc="full shape, B=2, context 8192"),
    "full_bs4_8k": Workload("full_bs4_8k", "full", 4, ("fixed", 8192), 17,
                            desc="full shape, B=4, context 8192"),
    "batch32_ragged": Workload("batch32_ragged", "full", 32, ("uniform", 512, 32768), 4, zipf=1.1,
                               desc="full shape, B=32, seq_lens U[512,32768], Zipf(1.1) router bias"),
    "long_256k": Workload("long_256k", "full", 1, ("fixed", 262144), 5,
                          desc="full shape, B=1, context 262144"),
    "batch64_ragged": Workload("batch64_ragged", "full", 64, ("loguniform", 1024, 65536), 6,
                               desc="full shape, B=64, seq_lens log-uniform [1024,65536]"),
    "dense_small": Workload("dense_small", "dense", 1, ("fixed", 1024), 9,
                            desc="dense SwiGLU model: 8 layers, B=1, context 1024"),
    "dense_batch5": Workload("dense_batch5", "dense", 5, ("uniform", 1, 1500), 10,
                             desc="dense SwiGLU model: 8 layers, B=5, seq_lens U[1,1500]"),
    "small_fp8": Workload("small_fp8", "small_fp8", 1, ("fixed", 1024), 12,
                          desc="small shape with FP8 experts: 8 layers, B=1, context 1024"),
    "small_fp8_b2": Workload("small_fp8_b2", "small_fp8", 2, ("uniform", 1, 1024), 13,
                             desc="small shape with FP8 experts: 8 layers, B=2, seq_lens U[1,1024]"),
    "full_fp8_bs1_8k": Workload("full_fp8_bs1_8k", "full_fp8", 1, ("fixed", 8192), 3,
                                desc="full shape with FP8 experts, B=1, context 8192"),
    "full_fp8_bs2_8k": Workload("full_fp8_bs2_8k", "full_fp8", 2, ("fixed", 8192), 16,
                                desc="full shape with FP8 experts, B=2, context 8192"),
    # FP8 experts above batch 2: the tensor-core build's FP8 expert tiles
    "small_fp8_b16": Workload("small_fp8_b16", "small_fp8", 16, ("uniform", 1, 1024), 18,
                              desc="small shape with FP8 experts: 8 layers, B=16, seq_lens U[1,1024]"),
    "batch32_fp8_ragged": Workload("batch32_fp8_ragged", "full_fp8", 32, ("uniform", 512, 32768), 4, zipf=1.1,
                                   desc="full shape with FP8 experts, B=32, seq_lens U[512,32768], "
                                        "Zipf(1.1) router bias"),
    "small_fp4": Workload("small_fp4", "small_fp4", 1, ("fixed", 1024), 14,
                          desc="small shape with FP4 experts: 8 layers, B=1, context 1024"),
    "small_fp4_b2": Workload("small_fp4_b2", "small_fp4", 2, ("uniform", 1, 1024), 15,
                             desc="small shape with FP4 experts: 8 layers, B=2, seq_lens U[1,1024]"),
    "full_fp4_bs1_8k": Workload("full_fp4_bs1_8k", "full_fp4", 1, ("fixed", 8192), 3,
                                desc="full shape with FP4 experts, B=1, context 8192"),
    "full_fp4_bs2_8k": Workload("full_fp4_bs2_8k", "full_fp4", 2, ("fixed", 8192), 16,
                                desc="full shape with FP4 experts, B=2, context 8192"),
    # seeded, non-unit RMSNorm gains (every layer's and the final norm's)
    "tiny_gains": Workload("tiny_gains", "tiny", 1, ("fixed", 64), 31, gains=True,
                           desc="tiny with seeded RMSNorm gains in [0.5, 2)"),
    "small_gains": Workload("small_gains", "small", 1, ("fixed", 1024), 32, gains=True,
                            desc="small with seeded RMSNorm gains in [0.5, 2)"),
    "full_gains_bs1_8k": Workload("full_gains_bs1_8k", "full", 1, ("fixed", 8192), 33, gains=True,
                                  desc="full shape, B=1, context 8192, seeded RMSNorm gains"),
    "prof_l2_b32": Workload("prof_l2_b32", "full_l2", 32, ("uniform", 512, 8192), 8, zipf=1.1,
                            desc="full-shape layers, 2 of them, B=32 ragged U[512,8192], Zipf(1.1) routing "
                                 "(profiling case of the tensor-core build)"),
    "prof_l2_fp8_b32": Workload("prof_l2_fp8_b32", "full_fp8_l2", 32, ("uniform", 512, 8192), 8, zipf=1.1,
                                desc="full-shape layers with FP8 experts, 2 of them, B=32 ragged U[512,8192], "
                                     "Zipf(1.1) routing (profiling case of the FP8 tensor-core build)"),
    "prof_l2_8k": Workload("prof_l2_8k", "full_l2", 1, ("fixed", 8192), 7,
                           desc="full-shape layers, 2 of them, B=1, context 8192 (profiling case)"),
}


def seq_lens_for(w: Workload) -> np.ndarray:
    """Sequence lengths of the step; each includes the token being decoded."""
    rng = np.random.default_rng([w.seed, 11])
    kind = w.seq[0]
    if kind == "fixed":
        s = np.full(w.batch, w.seq[1], dtype=np.int64)
    elif kind == "uniform":
        s = rng.integers(w.seq[1], w.seq[2] + 1, size=w.batch)
    elif kind == "loguniform":
        lo, hi = math.log(w.seq[1]), math.log(w.seq[2])
        s = np.floor(np.exp(rng.uniform(lo, hi, size=w.batch))).astype(np.int64)
        s = np.clip(s, w.seq[1], w.seq[2])
    else:
        raise ValueError(kind)
    return s.astype(np.int32)


def block_tables_for(seq_lens: np.ndarray, page_size: int, seed: int, slack_pages: int = 0):
    """Random page placement: a seeded permutation of the pool's pages is dealt
    out to the sequences in order.  Returns (block_tables [B][max_pages] int32,
    padded with -1, num_pages)."""
    rng = np.random.default_rng([seed, 12])
    pages = [(int(s) + page_size - 1) // page_size for s in seq_lens]
    num_pages = sum(pages) + slack_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    max_pages = max(pages)
    bt = np.full((len(seq_lens), max_pages), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt, num_pages


def tokens_for(w: Workload) -> np.ndarray:
    rng = np.random.default_rng([w.seed, 13])
    return rng.integers(0, w.shape.vocab, size=w.batch).astype(np.int32)


def zipf_router_bias(n_experts: int, s: float, seed: int) -> np.ndarray:
    """bias_e = ln(p_e), p_e proportional to rank_e^-s, ranks a seeded
    permutation of the experts: adding it to the router logits skews the
    routing towards low-rank experts the way a Zipf(s) popularity would."""
    rng = np.random.default_rng([seed, 14])
    ranks = rng.permutation(n_experts) + 1
    p = ranks.astype(np.float64) ** (-s)
    p /= p.sum()
    return np.log(p).astype(np.float32)


@dataclass
class StepInputs:
    workload: Workload
    tokens: np.ndarray
    seq_lens: np.ndarray
    block_tables: np.ndarray
    num_pages: int
    router_bias: np.ndarray | None
    extra: dict = field(default_factory=dict)

    @property
    def max_pages(self) -> int:
        return int(self.block_tables.shape[1])


def make_inputs(w: Workload | str) -> StepInputs:
    if isinstance(w, str):
        w = WORKLOADS[w]
    sl = seq_lens_for(w)
    bt, npages = block_tables_for(sl, w.shape.page_size, w.seed)
    bias = zipf_router_bias(w.shape.n_experts, w.zipf, w.seed) if w.zipf else None
    return StepInputs(w, tokens_for(w), sl, bt, npages, bias)


def step_kv_bytes(shape: ModelShape, seq_lens) -> int:
    """KV bytes the step reads: every layer reads the keys and values of the
    positions it attends to (all of them for a full layer, the last `window`
    ones for a sliding layer)."""
    tot = 0
    for l in range(shape.n_layers):
        for s in seq_lens:
            n = int(s) if shape.is_full_layer(l) else min(int(s), shape.window)
            tot += n * shape.kv_bytes_per_token_layer()
    return tot
