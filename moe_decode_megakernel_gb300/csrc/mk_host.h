// mk_host.h -- host-side objects behind the C ABI handles.
#pragma once

#include <array>
#include <string>
#include <vector>

#include "../../include/mk.h"
#include "mk_internal.h"

struct mk_model {
  mk_config cfg;
  mk_weights w;
  int shape_id;  // index into the compiled shapes
  mk::ShapeDims dims;
  mk::MoePlan plan;
  // tensor maps of the weights for tcgen05 items (made at the first step that needs them)
  bool tm_ready = false;
  CUtensorMap tm_w[7];  // w_qkv, w_o, w_router, w_lm, w_gate, w_up, w_down
};

namespace mk {

using Desc = std::array<int32_t, 32>;

// What a barrier counts, for validation and simulation.
enum BarKind : int8_t {
  BK_STATIC = 0,   // +1 per signalling task; waited on with a fixed count
  BK_UP_EXPERT,    // +1 per up/gate tile of one expert (count fixed per expert)
  BK_ATTN_COUNT,   // +1 per KV slice of one (row, group)
  BK_CLAIM,        // a claim counter (atomicAdd), never waited on
};

struct WsLayout {
  size_t total = 0;
  std::vector<std::pair<std::string, size_t>> regions;  // name -> byte offset
  size_t off(const char* name) const;
  size_t add(const char* name, size_t bytes);
};

// Barrier indices of one layer (or -1 where absent).
struct LayerBars {
  int norm = -1, router = -1, topk = -1, fin = -1, gather = -1, o = -1, mcomb = -1;
  int upd = -1, dnd = -1, attn_done = -1;
  int claim_attn = -1, claim_up = -1, claim_dn = -1;
  int rarrive = -1;  // router tasks that finished (the last one runs the top-k)
  int qkv = -1;    // base, n_kv entries
  int acomb = -1;  // base, n_kv entries
  int cnt = -1;    // base, MB * n_kv entries
  int up = -1;     // base, n_experts entries
  // task counts behind the static targets
  int n_norm = 0, n_router = 0, n_topk = 0, n_gather = 0, n_o = 0, n_mcomb = 0;
  int n_up_claim = 0, n_dn_claim = 0, n_attn_claim = 0;
  std::vector<int> n_qkv_g, n_acomb_g;
};

}  // namespace mk

struct mk_sched {
  mk_config cfg;
  mk::ShapeDims dims;
  mk::MoePlan plan;
  mk_sched_opts opts;
  int num_sms = 0, max_batch = 0, max_ctx = 0;
  // the lean kernel build runs it: fused routing and MoE combine, merges a
  // warp per head, static separate claims (no task the lean build leaves out)
  bool lean = false;
  // tcgen05 GEMM items (kModeTc): BF16 experts of an MoE model at max_batch >
  // kTB; 128-row weight tiles, explicit gather, the BF16 hi/lo operand rows
  bool tc = false;
  int tc_nb = 0;  // rows of an activation operand box (2 max_batch, rounded up to 16)
  // FP8 experts (kModeTcFp8): the expert tiles on FP8 MMAs, their activation
  // operands as E4M3 term rows (boxes of kTcF8Terms max_batch, rounded up to 16)
  bool tc_fp8 = false;
  int tc_nb8 = 0;
  // tensor maps of the activation operands, for the workspace they were made for
  const void* tm_ws = nullptr;
  CUtensorMap tm_act[4];
  int split_len = 0, n_static = 0, max_slots = 0, max_attn_entries = 0;
  int lm_bar = -1;
  int trace_cap = 0;
  std::vector<mk::Desc> tasks;              // global order
  std::vector<std::vector<int>> per_sm;     // task indices in execution order
  std::vector<int8_t> bar_kind;
  std::vector<mk::LayerBars> lb;            // [L + 1]
  mk::WsLayout ws;
  std::vector<int32_t> upload;              // host image of the device task lists
  // tensor maps of the last KV pools seen (re-encoded when the pools change)
  const void* tm_kpool = nullptr;
  const void* tm_vpool = nullptr;
  int64_t tm_pages = 0;
  CUtensorMap tm_k, tm_v;
  const void* sched_dev = nullptr;          // uploaded lists
  int64_t watchdog_ns = 0;
};

namespace mk {
void set_error(const std::string& msg);
int fail(int code, const std::string& msg);
int attn_slices(const mk_sched* s, int seq_len);  // KV slices of a full-attention row
int query_num_sms();                              // SMs of the current device, -1 without one
int attn_group_sms(const mk_sched* s);            // SMs of the attention branch (split placement)
bool is_full_layer(const mk_config& c, int l);
// mk_check_step on a host copy of the step's error record (8 words at the
// workspace's "error" offset); the workspace and stream serve the stall
// diagnosis of a timeout
int check_record(const mk_sched* s, const uint32_t* rec, const void* workspace, void* stream);
}  // namespace mk
