// mk_internal.h -- definitions shared by the host scheduler and the device
// kernel: opcodes, the 32 x int32 task descriptor, stage geometry, and the
// kernel's parameter block.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace mk {

// ---------------------------------------------------------------- opcodes
// The sixteen operations of one decode step ("Cohere: a decode megakernel
// for North Mini Code", section "Tasks"), plus the no-op.
enum Op : int32_t {
  OP_NOP = 0,
  OP_RESID_NORM = 1,        // residual add (+ MoE combine) + RMSNorm; embedding at layer 0
  OP_QKV_PROJ = 2,          // one row tile of x W_qkv, RoPE + KV append in the epilogue
  OP_O_PROJ = 3,            // one row tile of attn W_o over one KV group's columns (split-K)
  OP_FFN_UPGATE_ACT = 4,    // dense SwiGLU up/gate tile (a one-expert, top-1 model)
  OP_FFN_DOWN = 5,          // dense down projection tile
  OP_LM_HEAD = 6,           // one vocab tile of the LM head
  OP_ATTN_DECODE = 7,       // one static KV slice of one (row, KV group)
  OP_ATTN_COMBINE = 8,      // merge of the slice partials of one (row, KV group)
  OP_ATTN_DRAIN = 9,        // claimer over the full-attention queue
  OP_ROUTER_GEMM = 10,      // router logits for a tile of experts
  OP_ROUTER_TOPK = 11,      // top-k experts and weights of a range of rows
  OP_ROUTE_FINALIZE = 12,   // per-expert counts, offsets, row order and the MoE queues
  OP_MOE_GATHER = 13,       // expert-ordered copy of the routed rows
  OP_MOE_UPGATE_ACT_DRAIN = 14,  // claimer over the up/gate tile queue
  OP_MOE_DOWN_DRAIN = 15,   // claimer over the down tile queue
  OP_MOE_COMBINE = 16,      // weighted sum of each row's expert outputs
  OP_COUNT = 17,
  // work items made by the producer warp from claimer tasks (never in a list)
  W_ATTN = 32,      // one KV slice (from ATTN_DECODE or ATTN_DRAIN)
  W_UP_TILE = 33,   // one claimed up/gate tile
  W_DOWN_TILE = 34, // one claimed down tile
  W_CLAIM_END = 35, // a claimer found its queue empty: signal completion
  W_EXIT = 36,      // end of this SM's list
};

// ------------------------------------------------------ task descriptor
// "The task descriptor": 32 int32, field 0 the opcode, then the layer, the
// barriers to wait on with their counts, the barriers to signal, and the
// op-specific fields.
enum Field : int {
  F_OP = 0,
  F_LAYER = 1,
  F_WAIT0 = 2,  // barrier index or -1
  F_TGT0 = 3,   // count to wait for (TGT_DYN_SPLITS: the row's number of KV slices)
  F_WAIT1 = 4,
  F_TGT1 = 5,
  F_SIG0 = 6,   // barrier incremented when the task (or tile) is done, or -1
  F_SIG1 = 7,
  F_A0 = 8,     // op-specific arguments F_A0 .. F_A0 + 15
  F_TASK = 24,  // global index of the task (error reports, tracing)
  F_NSTAGE = 25,  // work items: shared-memory stages that belong to the item
  F_POS = 26,   // descriptors as uploaded: position in the SM's list (ring check)
  F_SEQ = 27,   // work items: sequence number on the SM's work ring (ring check)
  F_DESC_INTS = 32,
};
constexpr int32_t TGT_DYN_SPLITS = -2;

// op-specific argument slots
// RESID_NORM:   A0 b0, A1 b1 (row range), A2 final (1 = final norm before the LM head)
//               A3 fused MoE combine of the previous layer
// dense GEMV:   A0 row0, A1 n_rows, A2 KV group (O_PROJ split-K slice), A3 O_PROJ merges the
//               group's slices itself, A7 QKV_PROJ computes the RMSNorm itself
// ATTN_DECODE:  A0 b, A1 g, A2 slice index within the window, A3 counter base
// ATTN_DRAIN:   A0 claim counter, A1 counter base, A2 QKV barrier base, A3 QKV target,
//               A4 static claimer index (-1: claims from the counter), A5 claimers
// ATTN_COMBINE: A0 b, A1 g, A2 counter base
// ROUTER_TOPK:  A0 b0, A1 b1, A2 1 = also finalize (single top-k task)
// MOE_GATHER:   A0 row0, A1 n_rows
// MOE_*_DRAIN:  A0 claim counter, A1 up barrier base (per expert), A2 explicit-gather barrier
//               (or -1), A3 its target, A4 this claimer's index (or rank), A5 claimers, A6 queue
//               mode (0 up and down tiles interleaved, 1 up tiles only), A7 static claims (0 no,
//               1 by index with the down units shifted past the up units, 2 by host-set rank)
// MOE_COMBINE:  A0 b0, A1 b1
// W_ATTN:       A0 b, A1 g, A2 t0, A3 t1, A4 first page, A5 partial slot
// FFN_UPGATE_ACT / FFN_DOWN: A0 tile index
// W_UP_TILE / W_DOWN_TILE: A0 expert, A1 tile index, A2 row0, A3 n_rows, A8..A9 the
//               rows' output slots and A10..A11 their weights (down tiles of <= kTB rows),
//               A12 dense (rows are the batch rows: slot = row, weight 1)

// ------------------------------------------------------- stage geometry
constexpr int kStageBytes = 32768;   // one shared-memory stage
constexpr int kStages = 6;           // stage ring depth (192 KB)
constexpr int kDescRing = 4;         // descriptor ring (controller -> producer)
constexpr int kWorkRing = 8;         // work-item ring (producer -> consumers)
constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (3 + kConsumerWarps);  // controller, producer, storer, consumers
constexpr int kTB = 2;               // activation rows per GEMV pass
constexpr int kMaxStageRows = 64;
constexpr int kMaxBatch = 64;
// per-SM counters: consumer ns waiting on counters, on stages, busy ns, items;
// producer ns waiting on free stages, on routing, on the work ring, claims
constexpr int kStats = 8;

// Rows of a [rows][k] bf16 matrix that fit one stage, a multiple of 8, at most 64.
constexpr int stage_rows(int k) {
  int r = kStageBytes / (2 * k);
  r = r > kMaxStageRows ? kMaxStageRows : r;
  return r >= 8 ? (r / 8) * 8 : r;
}

// Kernel builds: the persistent kernel is instantiated per shape and per
// mode, each instantiation holding only the GEMV paths its steps take (the
// kernel's code size matters: instruction fetch is among its top stalls).
enum KernelMode : int {
  kModeSmallBatch = 0,  // BF16 experts, max_batch <= kTB, lean schedules: fused routing and MoE
                        // combine, a warp per head in the merges, static separate claims
  kModeAnyBatch = 1,    // BF16 experts, any batch (two-row passes above kTB), any schedule
  kModeFp8 = 2,         // FP8 experts (max_batch <= kTB), any schedule
  kModeFp4 = 3,         // FP4 experts (max_batch <= kTB), any schedule
  kModeFp8Lean = 4,     // FP8 experts, lean schedules
  kModeFp4Lean = 5,     // FP4 experts, lean schedules
  kModeTc = 6,          // BF16 experts, max_batch > kTB: GEMM items on the tcgen05 tensor cores
  kModeTcFp8 = 7,       // FP8 experts, max_batch > kTB: kModeTc with the expert tiles on FP8 MMAs
  kModeCount = 8
};
#if defined(__CUDACC__)
#define MK_HOST_DEVICE __host__ __device__
#else
#define MK_HOST_DEVICE
#endif
MK_HOST_DEVICE constexpr bool mode_fp8(int m) { return m == kModeFp8 || m == kModeFp8Lean; }
MK_HOST_DEVICE constexpr bool mode_fp4(int m) { return m == kModeFp4 || m == kModeFp4Lean; }
MK_HOST_DEVICE constexpr bool mode_tc(int m) { return m == kModeTc || m == kModeTcFp8; }
MK_HOST_DEVICE constexpr bool mode_lean(int m) {
  return m == kModeSmallBatch || m == kModeFp8Lean || m == kModeFp4Lean;
}

struct ShapeDims {
  int H, NQ, NKV, D, E, K, I, P;
};

// Stage plan of the MoE tiles: an up/gate stage holds `up_half` gate rows
// and as many up rows; a tile is `up_stages` stages.  A down stage holds
// `dn_rows` rows of W_down[e] ([H][I]); a tile is `dn_stages` stages.
struct MoePlan {
  int up_half, up_stages, up_tile, up_tiles;  // up_tile outputs per tile, tiles per expert
  int dn_rows, dn_stages, dn_tile, dn_tiles;
};

// Tiles are as large as keeps at least 16 up/gate and 32 down tiles per
// expert: each tile is a work item with a fixed cost (its barrier, its
// activation load, its epilogue), and at batch 1 the eight routed experts'
// 128 up/gate tiles and 256 down tiles still cover the SMs (full shape: up/gate
// tiles of 12 stages, 48 intermediate rows; down tiles of 4 stages, 64 rows).
constexpr int moe_stages(int rows, int rows_per_stage, int min_tiles) {
  const int cand[6] = {12, 8, 6, 4, 2, 1};
  for (int i = 0; i < 6; ++i)
    if (rows % (cand[i] * rows_per_stage) == 0 && rows / (cand[i] * rows_per_stage) >= min_tiles) return cand[i];
  return 1;
}
// Rows of a [rows][k] matrix of 1-byte (FP8) elements per stage: a power of
// two (so the stages divide the power-of-two matrix sides), at most 64.
constexpr int stage_rows8(int k) {
  int r = kStageBytes / k;
  r = r > kMaxStageRows ? kMaxStageRows : r;
  int p = 8;
  while (p * 2 <= r) p *= 2;
  return r >= 8 ? p : r;
}

// FP4 stages are 16-row groups of the tensor-core GEMV (up/gate: one group
// of 8 gate and 8 up rows), the rows' E2M1 codes followed by their block
// scales.  A down stage takes kFp4DownGroups groups where they fit (its rows
// are short: at inter 768 one group is 6.75 KB of a 32 KB stage), one group
// per consumer team; otherwise one.
constexpr int kFp4StageRows = 16;
constexpr int kFp4DownGroups = 4;
constexpr int fp4_stage_bytes(int k) { return kFp4StageRows * (k / 2 + k / 16); }
constexpr int fp4_groups_per_stage(int k) {
  return kFp4DownGroups * fp4_stage_bytes(k) <= kStageBytes ? kFp4DownGroups : 1;
}
static_assert(kFp4DownGroups * kFp4StageRows <= kMaxStageRows, "row scales of a down stage fit the slot's area");

constexpr MoePlan moe_plan(ShapeDims s) {
  MoePlan p{};
  p.up_half = stage_rows(s.H) / 2;
  p.up_stages = moe_stages(s.I, p.up_half, 16);
  p.up_tile = p.up_half * p.up_stages;
  p.up_tiles = s.I / p.up_tile;
  p.dn_rows = stage_rows(s.I);
  p.dn_stages = moe_stages(s.H, p.dn_rows, 32);
  p.dn_tile = p.dn_rows * p.dn_stages;
  p.dn_tiles = s.H / p.dn_tile;
  return p;
}
// the same plan for FP8 expert rows (twice the rows per stage)
constexpr MoePlan moe_plan8(ShapeDims s) {
  MoePlan p{};
  p.up_half = stage_rows8(s.H) / 2;
  p.up_stages = moe_stages(s.I, p.up_half, 16);
  p.up_tile = p.up_half * p.up_stages;
  p.up_tiles = s.I / p.up_tile;
  p.dn_rows = stage_rows8(s.I);
  p.dn_stages = moe_stages(s.H, p.dn_rows, 32);
  p.dn_tile = p.dn_rows * p.dn_stages;
  p.dn_tiles = s.H / p.dn_tile;
  return p;
}
// the plan for FP4 expert rows: 16-row stages
constexpr MoePlan moe_plan4(ShapeDims s) {
  MoePlan p{};
  p.up_half = kFp4StageRows / 2;
  p.up_stages = moe_stages(s.I, p.up_half, 16);
  p.up_tile = p.up_half * p.up_stages;
  p.up_tiles = s.I / p.up_tile;
  p.dn_rows = kFp4StageRows * fp4_groups_per_stage(s.I);
  p.dn_stages = moe_stages(s.H, p.dn_rows, 32);
  p.dn_tile = p.dn_rows * p.dn_stages;
  p.dn_tiles = s.H / p.dn_tile;
  return p;
}

// One layer's record of the MoE queue trace (int32): the active-expert list
// [E][4], the row offsets [E + 1], the expert-ordered rows [n_routed_max],
// {active experts, routed rows}; padded to a multiple of 4 (16 bytes).
MK_HOST_DEVICE constexpr int queue_trace_stride(int E, int n_routed_max) {
  return (4 * E + (E + 1) + n_routed_max + 2 + 3) / 4 * 4;
}

// tcgen05 GEMM items (kModeTc): an item is one tile of kTcRows weight rows
// (the M side of the MMA) over the whole K, streamed as k-blocks of kTcK
// elements; a stage holds one k-block of the weight tile (kTcRows x kTcK
// BF16, 16 KB) and of the activation operand (up to kTcMaxN rows: every
// activation row as a BF16 hi row and lo row).
constexpr int kTcRows = 128;
constexpr int kTcK = 64;
constexpr int kTcABytes = kTcRows * kTcK * 2;
constexpr int kTcMaxN = (kStageBytes - kTcABytes) / (kTcK * 2);
constexpr int kTcRouterRows = 16;  // rows of a router task (its weight box; the MMA's other rows unused)
constexpr int kTcDenseRows = 64;   // rows of a QKV, O-proj or LM-head tile (the MMA's other rows unused)
constexpr int kTcMoeRows = 128;    // weight rows of an expert tile: 64 gate + 64 up rows, or 128 down rows
// k-blocks per stage of a tcgen05 item whose weight box holds a_bytes per
// k-block and whose activation box holds tc_nb rows: as many pairs of boxes
// as fill the stage (the weight boxes first, then the activation boxes; both
// sizes are multiples of 1024 bytes, so every box starts on a swizzle atom),
// at most 8: one for full expert tiles, up to 3 for the 64-row dense tiles
// at small batches, up to 8 for a router task's 16-row boxes.
MK_HOST_DEVICE constexpr int tc_kblocks_per_stage(uint32_t a_bytes, int tc_nb) {
  int k = a_bytes >= (uint32_t)kTcABytes ? 1 : (int)((uint32_t)kTcABytes / a_bytes);
  const int kb_fit = (kStageBytes - kTcABytes) / (tc_nb * kTcK * 2);
  k = k < kb_fit ? k : kb_fit;
  return k < 1 ? 1 : (k > 8 ? 8 : k);
}
static_assert(kTcMaxN >= 2 * kMaxBatch, "hi/lo rows of the largest batch fit a stage");

// FP8 expert tiles of kModeTcFp8: a k-block is 128 E4M3 weights (128 bytes,
// the same 16 KB box of kTcRows rows).  The activation operand holds every
// routed row as kTcF8Terms E4M3 rows whose values, scaled by 16^-j for row j,
// sum to the activation within 2^-16 of it (E4M3 keeps 4 significant bits:
// each term leaves at most 1/16 of the rest); the gathered rows are first
// scaled by a power of two into range, the SwiGLU activations must stay
// within +-448.  The MMA's N is kTcF8Terms per routed row, at most kTcMaxN:
// batches of at most kTcF8MaxBatch rows.
constexpr int kTcK8 = 128;
constexpr int kTcF8Terms = 4;
constexpr int kTcF8MaxBatch = kTcMaxN / kTcF8Terms;
static_assert(kTcF8MaxBatch >= 32, "FP8 expert tiles up to batch 32");

// The MoE plan of tcgen05 items: up/gate tiles of kTcMoeRows / 2 gate rows
// and the same up rows, down tiles of kTcMoeRows rows (the MMA's M = 128 has
// the rest unused); "stages" count k-blocks.
constexpr MoePlan moe_plan_tc(ShapeDims s) {
  MoePlan p{};
  p.up_half = kTcMoeRows / 2;
  p.up_stages = s.H / kTcK;
  p.up_tile = kTcMoeRows / 2;
  p.up_tiles = s.I / p.up_tile;
  p.dn_rows = kTcMoeRows;
  p.dn_stages = s.I / kTcK;
  p.dn_tile = kTcMoeRows;
  p.dn_tiles = s.H / p.dn_tile;
  return p;
}
// the same tiles over FP8 expert rows: k-blocks of kTcK8
constexpr MoePlan moe_plan_tc8(ShapeDims s) {
  MoePlan p = moe_plan_tc(s);
  p.up_stages = s.H / kTcK8;
  p.dn_stages = s.I / kTcK8;
  return p;
}

// In the tensor-core builds an expert with at most kTB routed rows takes the
// batch <= kTB GEMV instead (its tiles would fill one 16-row MMA column block
// with one or two rows): the same tiles, streamed in GEMV stages of whole
// rows (BF16, or FP8 with their row scales), so that a stage carries 32 KB
// of weights where a tcgen05 item's carries 16 KB next to its activations.
constexpr MoePlan moe_plan_tc_gemv(ShapeDims s) {
  MoePlan p = moe_plan_tc(s);
  p.up_half = stage_rows(s.H) / 2;
  p.up_stages = p.up_tile / p.up_half;
  p.dn_rows = stage_rows(s.I);
  p.dn_stages = p.dn_tile / p.dn_rows;
  return p;
}
constexpr MoePlan moe_plan_tc8_gemv(ShapeDims s) {
  MoePlan p = moe_plan_tc8(s);
  p.up_half = stage_rows8(s.H) / 2;
  p.up_stages = p.up_tile / p.up_half;
  p.dn_rows = stage_rows8(s.I);
  p.dn_stages = p.dn_tile / p.dn_rows;
  return p;
}
constexpr bool gemv_plan_fits(MoePlan p) {
  return p.up_half > 0 && p.up_tile % p.up_half == 0 && p.dn_rows > 0 && p.dn_tile % p.dn_rows == 0;
}

// ------------------------------------------------------ kernel parameters
struct Params {
  // the KV pools as 2-D tensors [L*pages*n_kv*P][d] for TMA tiles of
  // (P rows, 64 dims) with the 128-byte swizzle
  CUtensorMap tm_k, tm_v;
  // weights ([out][in] row-major BF16 unless noted)
  const uint16_t* emb;
  const uint16_t* wqkv;
  const uint16_t* wo;
  const uint16_t* wr;
  const float* rbias;
  const uint16_t* wg;   // bf16, or FP8 (E4M3 bytes) when expert_fp8
  const uint16_t* wu;
  const uint16_t* wd;
  int expert_fp8;       // expert rows are E4M3 bytes with one fp32 scale per row
  const float* sg;      // [L][E][I] row scales of w_gate (FP8 only)
  const float* su;      // [L][E][I]
  const float* sd;      // [L][E][H]
  int expert_fp4;       // expert rows are E2M1 nibbles, an E4M3 scale per 16, fp32 per row
  const uint8_t* bg;    // [L][E][I][H/16] block scales of w_gate (FP4 only)
  const uint8_t* bu;    // [L][E][I][H/16]
  const uint8_t* bd;    // [L][E][H][I/16]
  const float* gamma;
  const float* gamma_f;
  const uint16_t* wlm;
  int L, V, window, full_period;
  float rope_base, eps;

  // step inputs and outputs
  int B, MB;  // batch, schedule's max batch (buffer stride)
  const int32_t* tokens;
  const int32_t* block_tables;
  int max_pages;
  uint16_t* kpool;
  uint16_t* vpool;
  int64_t num_pages;
  float* logits;

  // task lists: [num_sms][2] (offset in int32, count) then descriptors
  const int32_t* sched;

  // workspace regions
  uint32_t* bars;
  uint32_t* err;        // [8]: code, sm, task, barrier, observed, target, op, layer
  uint32_t* prog;       // [num_sms][8]: where each role of each SM is (read after a failed step)
  const int32_t* seq_lens;  // [B] device, length including the decoded token
  int max_ctx;
  float* h;             // [MB][H] residual stream
  float* x;             // [MB][H] normalised layer input
  float* q;             // [MB][NQ][D] RoPE'd queries
  uint16_t* kvnew;      // [MB][2][NKV][D] the new token's K and V (bf16, as stored)
  float* part_o;        // [MB][NKV][max_slots][G][D] unnormalised slice outputs
  float* part_ml;       // [MB][NKV][max_slots][G][2] slice max (log2 domain) and sum
  float* attn_out;      // [MB][NQ D]
  float* opart;         // [2][NKV][MB][H] O-proj split-K partials, by layer parity
  float* rlog;          // [L][MB][E] router logits
  int32_t* topk_ids;    // [L][MB][K]
  float* topk_w;        // [L][MB][K]
  int32_t* ecount;      // [L][E]
  int32_t* eoff;        // [E + 1] row offset of each expert (current layer)
  int32_t* perm;        // [MB K] expert-ordered row -> b * K + j
  int32_t* inv;         // [MB K] b * K + j -> expert-ordered row
  int32_t* act;         // [E][4] active experts ascending: {expert, first row, rows, 0}
  int32_t* qlen;        // [2] active experts, routed rows
  float* xg;            // [MB K][H] gathered rows (explicit gather)
  float* u;             // [MB K][I] SwiGLU activations
  float* y;             // [MB K][H] expert outputs
  float* moe_out;       // [MB][H]
  float* htrace;        // [L + 1][MB][H] or null
  int32_t* qtrace;      // [L][queue_trace_stride(E, MB K)] or null

  uint64_t* trace;      // [num_sms][trace_cap][2] per work item, or null
  int trace_cap;
  uint64_t* stats;      // [num_sms][kStats] stall counters, or null

  // tcgen05 items (kModeTc): 2-D tensor maps of the weights (boxes of kTcK
  // columns by kTcRows rows, or kTcRows / 2 rows for the gate and up
  // matrices, 128-byte swizzle) and of the activation operands (boxes of kTcK
  // columns by tc_nb rows), and the operands themselves: every activation row
  // r as BF16 rows 2r (hi = bf16(x)) and 2r + 1 (lo = bf16(x - hi))
  CUtensorMap tm_wqkv, tm_wo, tm_wr, tm_wlm, tm_wg, tm_wu, tm_wd;
  CUtensorMap tm_xb, tm_attnb, tm_xgb, tm_ub;
  uint16_t* xb;         // [MB][2][H]      the layer input x (written by the RMSNorm)
  uint16_t* attnb;      // [MB][2][NQ D]   the attention output (written by the merges)
  uint16_t* xgb;        // [MB K][2][H]    the routed rows in expert order (written by MOE_GATHER)
  uint16_t* ub;         // [MB K][2][I]    the SwiGLU activations (written by the up/gate tiles)
  int tc_nb;            // rows of an activation box: 2 MB rounded up to 16 (the MMA's N)
  // kModeTcFp8: the expert tiles' activation operands as E4M3 term rows
  // (row kTcF8Terms r + j holds term j of routed row r), boxes of kTcK8
  // columns by tc_nb8 rows; the weight maps tm_wg, tm_wu, tm_wd hold E4M3 bytes
  CUtensorMap tm_xg8, tm_u8;
  uint8_t* xg8;         // [MB K][kTcF8Terms][H] the routed rows in expert order (MOE_GATHER)
  uint8_t* u8;          // [MB K][kTcF8Terms][I] the SwiGLU activations (the up/gate tiles)
  float* xg8s;          // [MB K] the inverse of each gathered row's power-of-two scale
  int tc_nb8;           // kTcF8Terms MB rounded up to 16 (the expert tiles' N)

  int split_len;        // tokens per KV slice
  int n_static;         // static slices per (row, group) of a sliding layer
  int max_slots;
  int explicit_gather;
  int64_t watchdog_ns;
};

}  // namespace mk
