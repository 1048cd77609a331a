/*
 * mk.h -- C ABI of the GB300 (sm_103a) decode megakernel.
 *
 * One decode step of a parallel-attention / MoE transformer runs as a single
 * persistent kernel: one CTA per SM walks a host-built list of fixed-size
 * task descriptors, synchronises with other SMs only through counters in
 * global memory, and pulls runtime-sized work (full-attention KV slices, MoE
 * expert tiles) from shared work queues.  This follows "Cohere: a decode
 * megakernel for North Mini Code" (sections "What is a Megakernel?", "The
 * task descriptor", "Barriers", "Task scheduler"), re-designed for GB300.
 *
 * Conventions for every entry point:
 *  - All device memory is allocated by the caller and passed as plain
 *    pointers; the library never allocates device memory.  Host handles
 *    (mk_model, mk_sched) are allocated by the library and freed with
 *    mk_free_model / mk_free_sched.
 *  - Functions return MK_OK (0) or a negative MK_ERR_* code; mk_last_error()
 *    then returns a message (thread-local, valid until the next call).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - BF16 tensors are raw uint16 bit patterns of bfloat16.
 *  - There is no CPU fallback: without a GB300 the compute entry points return
 *    MK_ERR_CUDA.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MK_OK 0
#define MK_ERR_ARG (-1)         /* a bad argument; nothing was launched */
#define MK_ERR_CUDA (-2)        /* a CUDA runtime call failed */
#define MK_ERR_TIMEOUT (-3)     /* a device-side wait gave up (watchdog) */
#define MK_ERR_UNSUPPORTED (-4) /* no compiled kernel for this model shape */
#define MK_ERR_DEVICE (-5)      /* a device-side check failed (e.g. page id out of range) */

/* Model shape.  Layer l attends to its whole context iff window == 0 or
 * (l + 1) % full_period == 0; otherwise to the last `window` positions.
 * The compiled kernels cover four shapes (hidden, n_q, n_kv, head_dim,
 * n_experts, top_k, inter, page_size): (256,4,2,64,16,4,128,16),
 * (1024,16,2,64,32,4,512,64), (2048,32,4,128,128,8,768,64) and the dense
 * (1024,16,2,64,1,1,2048,64); n_layers, vocab, window and full_period are
 * free.  n_experts = top_k = 1 is a dense model: every token takes the one
 * expert with weight 1, i.e. a SwiGLU FFN (w_gate, w_up, w_down of "expert
 * 0"), run as static FFN_UPGATE_ACT / FFN_DOWN tiles with no router (the
 * pages' "Tasks": the dense FFN opcodes); w_router may then be NULL. */
typedef struct {
  int32_t n_layers, hidden, n_q, n_kv, head_dim, n_experts, top_k, inter, vocab;
  int32_t page_size, window, full_period;
  float rope_base, eps;
  int32_t expert_fp8;  /* 1: w_gate, w_up, w_down hold OCP FP8 E4M3 codes (1 byte each,
                          same [L][E][rows][cols] layout) and each output row has one
                          fp32 scale (w_*_scale): weight = e4m3 value * row scale.
                          Schedules for it need max_batch <= 32; above 2 the expert
                          tiles run on FP8 tensor-core MMAs (E4M3 weights against the
                          activations as four E4M3 terms each: the gathered rows scaled
                          by a power of two per row, the SwiGLU activations as they
                          are), which needs hidden and inter multiples of 128; a SwiGLU
                          activation beyond 448 in magnitude fails the step
                          (MK_ERR_DEVICE from mk_check_step) */
  int32_t expert_fp4;  /* 1 (not with expert_fp8): w_gate, w_up, w_down hold FP4 E2M1 codes,
                          two per byte (element 2j in the low nibble of byte j), the same
                          [L][E][rows][cols] layout at half a byte per weight; each run of 16
                          inputs of a row has an E4M3 block scale (w_*_bscale) and each output
                          row an fp32 scale (w_*_scale): weight = e2m1 * block scale * row
                          scale.  hidden and inter multiples of 128; max_batch <= 2 */
} mk_config;

/* Device pointers to the weights, row-major with the output dimension first
 * ([out][in], the layout of a linear layer's weight).  Stacked over layers
 * (and experts) with no padding.  Every pointer is 16-byte aligned (the rows
 * are streamed by bulk copies); mk_load_model fails with MK_ERR_ARG
 * otherwise.  The library keeps the pointers; the caller keeps the memory
 * alive and unchanged while the model is in use. */
typedef struct {
  const void* embedding;   /* bf16 [vocab][hidden] */
  const void* w_qkv;       /* bf16 [L][(n_q + 2 n_kv) head_dim][hidden]: q heads, k heads, v heads */
  const void* w_o;         /* bf16 [L][hidden][n_q head_dim] */
  const void* w_router;    /* bf16 [L][n_experts][hidden] */
  const float* router_bias;/* fp32 [n_experts] added to every layer's router logits, or NULL */
  const void* w_gate;      /* bf16 [L][n_experts][inter][hidden] */
  const void* w_up;        /* bf16 [L][n_experts][inter][hidden] */
  const void* w_down;      /* bf16 [L][n_experts][hidden][inter] */
  const float* norm_gamma; /* fp32 [L][hidden] input RMSNorm gain of each layer */
  const float* final_gamma;/* fp32 [hidden] final RMSNorm gain */
  const void* w_lm;        /* bf16 [vocab][hidden] */
  const float* w_gate_scale; /* fp32 [L][n_experts][inter] (expert_fp8 only, else NULL) */
  const float* w_up_scale;   /* fp32 [L][n_experts][inter] */
  const float* w_down_scale; /* fp32 [L][n_experts][hidden] */
  const void* w_gate_bscale; /* E4M3 bytes [L][n_experts][inter][hidden/16] (expert_fp4 only) */
  const void* w_up_bscale;   /* E4M3 bytes [L][n_experts][inter][hidden/16] */
  const void* w_down_bscale; /* E4M3 bytes [L][n_experts][hidden][inter/16] */
} mk_weights;

typedef struct mk_model mk_model;
typedef struct mk_sched mk_sched;

/* Loads a model: validates the shape against the compiled kernels and
 * records the weight pointers ("Cohere: a decode megakernel for North Mini
 * Code", section "One ABI for every operation": every operation reads its
 * weights through pointers fixed before the step, so the kernel takes the
 * model as plain device addresses).  The [out][in] layout is already
 * tile-contiguous for the row tiles the kernel streams, so nothing is
 * repacked.  Host only: no device call, no copy.  MK_ERR_UNSUPPORTED for a
 * shape no kernel was compiled for; MK_ERR_ARG for a null or misaligned
 * pointer or an invalid field.  *out is freed with mk_free_model. */
int mk_load_model(const mk_config* cfg, const mk_weights* w, mk_model** out);
void mk_free_model(mk_model* m);

/* Wave orders of one layer ("Task scheduler: mapping tasks to SMs"):
 * DEFAULT     router, top-k, route setup, gather, qkv, attention (+combine),
 *             MoE up/down, O-proj, RMSNorm (the pages' order with the
 *             router ahead of QKV);
 * INTERLEAVED attention, MoE up/down, attention combine, MoE combine,
 *             O-proj, RMSNorm;
 * ATTN_FIRST  attention, attention combine, O-proj, MoE up/down, MoE
 *             combine, RMSNorm. */
#define MK_WAVES_DEFAULT 0
#define MK_WAVES_INTERLEAVED 1
#define MK_WAVES_ATTN_FIRST 2
#define MK_WAVES_MOE_FIRST 3   /* up/gate tiles ahead of attention on each SM */
#define MK_WAVES_MOE_FIRST_O 4 /* the same, with O-proj ahead of the down tiles */
#define MK_WAVES_O_BEFORE_DOWN 5 /* attention, merge, up/gate, O-proj, then the down tiles */
#define MK_WAVES_INTERLEAVED_O 6 /* attention, up/gate, merge, O-proj, then the down tiles */

typedef struct {
  int32_t num_sms;          /* SMs to schedule for; 0 = the current device's count */
  int32_t wave_order;       /* MK_WAVES_*; -1 (default): MK_WAVES_DEFAULT for max_batch <= 2,
                               above it (the tensor-core build) MK_WAVES_O_BEFORE_DOWN up to 8
                               rows and MK_WAVES_INTERLEAVED beyond: the fastest measured */
  int32_t attn_split_pages; /* KV pages per attention task; 0 = choose from the context */
  int32_t attn_claimers;    /* ATTN_DRAIN claimers per full-attention layer; 0 = auto */
  int32_t moe_claimers;     /* claimers per MoE drain per layer; 0 = auto */
  int32_t qkv_tile_rows;    /* output rows per QKV task; 0 = auto */
  int32_t o_tile_rows;      /* output rows per O-proj task (per KV group); 0 = auto */
  int32_t lm_tile_rows;     /* vocab rows per LM-head task; 0 = auto */
  int32_t fuse_finalize;    /* 1: the (single) top-k task also builds the MoE queue */
  int32_t fuse_moe_combine; /* 1: the residual RMSNorm also does the MoE combine */
  int32_t explicit_gather;  /* 1: MOE_GATHER materialises expert-ordered rows */
  int32_t trace_hidden;     /* 1: keep the residual entering every layer in the workspace */
  int32_t watchdog_ms;      /* device-side wait limit; 0 = 2000 ms */
  int32_t trace;            /* 1: record every work item's timestamps ("trace", "stats") */
  int32_t moe_queue;        /* 0: separate up/gate and down drains; 1: one MoE queue with each
                               expert's down tiles one expert behind its up/gate tiles */
  int32_t moe_static;       /* 1: claimer c takes MoE units c, c + n, c + 2n, ... of the queue
                               (n claimers), no atomics; 0: the first unit so and the rest from
                               a claim counter; -1 (default): 1 for max_batch <= 2, 0 for the
                               tensor-core schedules (max_batch > 2, BF16 experts) */
  int32_t fuse_routing;     /* 1 (default): the last router task to finish runs the top-k and
                               builds the MoE queue (no separate top-k task), and at batch <= 2
                               each router task computes the layer's RMSNorm itself instead of
                               waiting for it; needs fuse_finalize */
  int32_t fuse_norm_qkv;    /* 1 (default) at batch <= 2: each QKV tile computes the layer's
                               RMSNorm itself instead of waiting for a separate RMSNorm task */
  int32_t attn_static;      /* 1 (default): full-attention claimer i of n takes queue entries
                               i, i + n, ... (no atomics; the claimers start together, after
                               the QKV tiles); 0: each claims the next entry from a counter,
                               at most one slice ahead of its running one */
  int32_t moe_balance;      /* 1 (with moe_static and separate up/down drains): the claimers'
                               static ranks go to the SMs estimated to reach their claimer
                               first, so the extra MoE tiles land there; 0 (default): rank =
                               claimer index, down units shifted past the up units */
  int32_t combine_per_head; /* 1: when max_batch * n_kv * (n_q / n_kv) <= num_sms, one
                               attention-combine task per (row, KV group, query head), each
                               spread over the whole block; 0 (default): one per (row, KV
                               group), a warp per head (fewer SMs held by merges) */
  int32_t placement;        /* 0 (default): task k of the flattened waves runs on SM k mod
                               num_sms; 1: greedy, each layer's tasks in order go to the SM
                               where a cost model (typical ready and busy time per op, a
                               claimer's static unit count) says they finish first;
                               2: split, the attention branch (QKV, attention slices and
                               claimers, merges, O-proj) round robin over SMs [0, attn_sms)
                               and the MoE branch (RMSNorm, router, routing, MoE drains) over
                               the others, so neither branch queues behind the other; the LM
                               head over all SMs; 3: dependency affinity ("Task scheduler"),
                               each task to the least loaded SM that ran a task it waits on,
                               within a per-layer cap of the layer's tasks per SM (rounded
                               up), else to the least loaded SM; 4: round robin, but each
                               layer's static attention slices go first (at most 3 each) to the
                               SMs whose static up/gate claimer gets no tile */
  int32_t attn_sms;         /* placement 2: SMs of the attention branch; 0 = in proportion
                               to the branch's bytes per layer (QKV, O-proj and KV against
                               router and experts) */
  int32_t trace_queue;      /* 1: keep every layer's MoE work queue in the workspace
                               ("queue_trace", see mk_workspace_offset) */
} mk_sched_opts;

/* Fills opts with the defaults (all zero except fuse_* = 1, attn_static = 1 and
 * moe_static = -1). */
void mk_default_sched_opts(mk_sched_opts* opts);

/* Builds and validates the per-SM task lists for steps with batch <=
 * max_batch and every seq_len <= max_ctx ("Task scheduler": the list is
 * built on the host once and reused by every step).  Host only; no device
 * call unless opts->num_sms == 0.  max_batch <= 64. */
int mk_build_tasks(const mk_model* m, int32_t max_batch, int32_t max_ctx,
                   const mk_sched_opts* opts, mk_sched** out);
void mk_free_sched(mk_sched* s);

/* Bytes of the device copy of the task lists, and the upload into a
 * caller-allocated buffer of that size (16-byte aligned). */
size_t mk_sched_bytes(const mk_sched* s);
int mk_sched_upload(mk_sched* s, void* sched_dev, size_t bytes, void* stream);

/* Bytes of device scratch one step needs (barriers, activations, queues). */
size_t mk_workspace_bytes(const mk_sched* s);

/* One decode step ("What is a Megakernel?": one launch per step).
 *  last_tokens   device int32 [batch]: the token decoded at this step
 *  seq_lens      device int32 [batch]: sequence length including that token,
 *                1 <= seq_len <= max_ctx; the new K/V go to position seq_len-1
 *  block_tables  device int32 [batch][max_pages]: physical page of logical
 *                page j of row b; pages for positions < seq_len must exist
 *  k_pool,v_pool device bf16 [n_layers][num_pages][n_kv][page_size][head_dim];
 *                the step writes the new token's K and V into them
 *  workspace     device, mk_workspace_bytes(s) bytes, 256-byte aligned
 *  logits        device fp32 [batch][vocab]
 * Asynchronous on `stream` (one memset and one cooperative launch; the host
 * never waits).  MK_ERR_ARG for a bad shape or pointer (nothing launched).
 * Values are checked on the device: a seq_len, token or page id out of
 * range, or a watchdog timeout, is reported by mk_check_step. */
int mk_decode_step(mk_model* m, mk_sched* s, const int32_t* last_tokens,
                   const int32_t* seq_lens, const int32_t* block_tables, int32_t batch,
                   int32_t max_pages, void* k_pool, void* v_pool, int64_t num_pages,
                   void* workspace, size_t workspace_bytes, float* logits, void* stream);

/* Host-side check of a step's inputs before it is launched, for a caller
 * that holds host copies of them (the decode service does).  mk_decode_step
 * takes its inputs as device arrays and checks their values on the device
 * (reported by mk_check_step), so that a step never waits for the host; this
 * call refuses the same inputs before launch instead.  Checks: batch in [1,
 * max_batch]; every seq_len in [1, max_ctx]; every page id the step reads
 * (logical pages 0 .. (seq_len - 1) / page_size of each row) in [0,
 * num_pages) and within max_pages columns; with last_tokens (may be NULL)
 * every token in [0, vocab).  Host pointers: seq_lens [batch], block_tables
 * [batch][max_pages], last_tokens [batch].  Returns MK_OK or MK_ERR_ARG
 * naming the first offending row (mk_last_error()). */
int mk_check_inputs(const mk_sched* s, const int32_t* last_tokens, const int32_t* seq_lens,
                    const int32_t* block_tables, int32_t batch, int32_t max_pages, int64_t num_pages);

/* mk_decode_step with a built-in workspace, for callers that cannot allocate
 * device memory: their device memory belongs to another allocator (a host
 * framework's caching allocator, a runtime whose budget is fixed at start-up)
 * and they may not call cudaMalloc while running -- cudaMalloc can
 * synchronise the device and can fail under a fixed budget.  The pages
 * describe no such entry point; it has no counterpart there.
 * Same arguments and behaviour as mk_decode_step, without the workspace
 * pair.  The workspace is one 8 MiB device array inside the library: every
 * GPU that loads the library holds it until the process exits.  Returns
 * MK_ERR_ARG if the schedule needs more (mk_workspace_bytes(s) > 8 MiB).  It
 * allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress), with that device current; make that first call
 * before any stream capture.  A lookup that fails is not remembered: the
 * next call tries again.  All calls share the array and it keeps the
 * last call's contents (each step zeroes its own counters first): calls
 * whose executions overlap on the GPU, on any streams, race on it.
 * Device-side failures (watchdog, page id out of range) are recorded in that
 * array and cannot be read back through this entry point; where they matter,
 * use mk_decode_step and mk_check_step. */
int mk_decode_step_static_ws(mk_model* m, mk_sched* s, const int32_t* last_tokens,
                             const int32_t* seq_lens, const int32_t* block_tables, int32_t batch,
                             int32_t max_pages, void* k_pool, void* v_pool, int64_t num_pages,
                             float* logits, void* stream);

/* Waits for `stream`, then reads the step's device error record: MK_OK,
 * MK_ERR_TIMEOUT or MK_ERR_DEVICE (details in mk_last_error()).  A timeout
 * names the first wait that gave up (SM, task, opcode, layer, barrier index,
 * count seen, target): the stalled task itself, or a task downstream of it
 * whose wait began earlier.  The message then adds a diagnosis from the
 * barrier counts against the schedule: the task whose wait target exceeds
 * the number of tasks that signal its barrier (the root of the stall), or
 * else the barriers still short of their signallers. */
int mk_check_step(const mk_sched* s, const void* workspace, void* stream);

const char* mk_last_error(void);

/* ---- inspection (tests, tracing) ---- */

/* Byte offsets of named regions inside the workspace (-1 if absent):
 * "topk_ids" int32 [L][B][k], "topk_w" fp32 [L][B][k], "router_logits"
 * fp32 [L][B][E], "expert_count" int32 [L][E], "moe_queue" int32 [E][4] (last
 * layer's active experts, ascending: {expert, first expert-ordered row,
 * rows, 0}; the MoE queues are (active expert, tile) in that order),
 * "moe_queue_len" int32 [2] (active experts, routed rows),
 * "perm" int32 [B*k] (last layer), "hidden_trace" fp32 [L+1][B][H],
 * with opts.trace_queue "queue_trace" int32 [L][R], R = (5E + 1 + B*k + 2)
 * rounded up to a multiple of 4, each layer's record being the active-expert
 * list [E][4] ({expert, first expert-ordered row, rows, 0}; entries past the
 * active count are stale), the row offsets [E+1], the expert-ordered rows
 * [B*k] (entry i = b*k + j) and {active experts, routed rows},
 * "error" uint32 [8], "barriers" uint32, with opts.trace "trace" uint64
 * [num_sms][cap][4] (popped, waits done, end in ns of %globaltimer; op |
 * layer << 8 | task << 16 | first argument << 40; unused records zero) and
 * "stats" uint64 [num_sms][8] (consumer: ns waiting on counters, ns waiting on
 * stages, ns busy, items; producer: ns waiting on free stages, on routing, on
 * the work ring, claims), and the activations "h", "x", "q",
 * "kvnew", "attn_out", "opart", "u", "y", "moe_out" of the last layer. */
int64_t mk_workspace_offset(const mk_sched* s, const char* name);

/* Task list access for tests: counts, a copy of one descriptor (32 int32),
 * and replacement of one descriptor (host copy only; re-upload after). */
int32_t mk_sched_num_sms(const mk_sched* s);
int32_t mk_sched_num_tasks(const mk_sched* s, int32_t sm);
int mk_sched_get_task(const mk_sched* s, int32_t sm, int32_t idx, int32_t desc[32]);
int mk_sched_set_task(mk_sched* s, int32_t sm, int32_t idx, const int32_t desc[32]);
int32_t mk_sched_num_barriers(const mk_sched* s);

/* Static validation of the lists: every waited-on barrier is signalled by
 * enough tasks that come earlier in the global order, static barriers
 * receive exactly their target, claimers precede what waits on them.
 * Returns MK_OK or MK_ERR_ARG with the first violation in mk_last_error(). */
int mk_sched_validate(const mk_sched* s);

/* Host simulation of the lists as the device runs them (in order per SM,
 * waits on counters, claimers draining queues) for a given batch, host
 * seq_lens and routing (int32 [L][batch][k], or NULL for a seeded uniform
 * routing).  Returns MK_OK if every task finishes and every barrier ends at
 * exactly its target, MK_ERR_ARG (deadlock or miscount, described in
 * mk_last_error()) otherwise. */
int mk_sched_simulate(const mk_sched* s, int32_t batch, const int32_t* seq_lens,
                      const int32_t* routing, uint64_t seed);

#ifdef __cplusplus
}
#endif
#endif /* MK_H */
