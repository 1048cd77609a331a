// mk_api.cpp -- the C ABI: model and schedule handles, upload, the decode
// step launch and its error check.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <string>
#include <vector>

#include "mk_host.h"

namespace mk {

namespace {
thread_local std::string g_error;
}

void set_error(const std::string& msg) { g_error = msg; }

int fail(int code, const std::string& msg) {
  g_error = msg;
  return code;
}

int query_num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return n;
}

// launch_<shape>_<mode>: mk_shape.cu compiled per shape and KernelMode
#define MK_DECLARE_SHAPE(name)                                     \
  int launch_##name##_0(const Params& p, int grid, cudaStream_t s); \
  int launch_##name##_1(const Params& p, int grid, cudaStream_t s); \
  int launch_##name##_2(const Params& p, int grid, cudaStream_t s); \
  int launch_##name##_3(const Params& p, int grid, cudaStream_t s); \
  int launch_##name##_4(const Params& p, int grid, cudaStream_t s); \
  int launch_##name##_5(const Params& p, int grid, cudaStream_t s); \
  int launch_##name##_6(const Params& p, int grid, cudaStream_t s); \
  int launch_##name##_7(const Params& p, int grid, cudaStream_t s);
MK_DECLARE_SHAPE(tiny)
MK_DECLARE_SHAPE(small)
MK_DECLARE_SHAPE(dense)
MK_DECLARE_SHAPE(full)
#undef MK_DECLARE_SHAPE

namespace {

struct CompiledShape {
  ShapeDims dims;
  int (*launch[kModeCount])(const Params&, int, cudaStream_t);  // by KernelMode
};

const CompiledShape kShapes[] = {
    {{256, 4, 2, 64, 16, 4, 128, 16}, {launch_tiny_0, launch_tiny_1, launch_tiny_2, launch_tiny_3, launch_tiny_4, launch_tiny_5, launch_tiny_6, launch_tiny_7}},
    {{1024, 16, 2, 64, 32, 4, 512, 64}, {launch_small_0, launch_small_1, launch_small_2, launch_small_3, launch_small_4, launch_small_5, launch_small_6, launch_small_7}},
    // dense SwiGLU FFN (one expert, top-1)
    {{1024, 16, 2, 64, 1, 1, 2048, 64}, {launch_dense_0, launch_dense_1, launch_dense_2, launch_dense_3, launch_dense_4, launch_dense_5, launch_dense_6, launch_dense_7}},
    {{2048, 32, 4, 128, 128, 8, 768, 64}, {launch_full_0, launch_full_1, launch_full_2, launch_full_3, launch_full_4, launch_full_5, launch_full_6, launch_full_7}},
};

int cuda_fail(cudaError_t e, const char* what) {
  return fail(MK_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// A KV pool [L][pages][n_kv][P][d] as the 2-D tensor [L*pages*n_kv*P][d]; one
// TMA box is (P rows, 64 dims) = P x 128 bytes, swizzled in 128-byte rows so
// the attention's ldmatrix reads hit distinct banks.
int encode_pool(CUtensorMap* tm, void* pool, const mk_sched* s, int64_t num_pages) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const ShapeDims& D = s->dims;
  const uint64_t rows = (uint64_t)s->cfg.n_layers * (uint64_t)num_pages * D.NKV * D.P;
  if (rows >= (1ull << 31)) return fail(MK_ERR_ARG, "KV pool too large for 32-bit TMA row coordinates");
  cuuint64_t dims[2] = {(cuuint64_t)D.D, rows};
  cuuint64_t strides[1] = {(cuuint64_t)D.D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)D.P};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pool, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
  return MK_OK;
}

// A row-major matrix [rows][cols] of BF16 (elem_bytes 2) or 8-bit codes
// (elem_bytes 1) as a 2-D tensor for the tcgen05 items: boxes of 128 bytes
// of a row (kTcK BF16 or kTcK8 codes) by box_rows rows, swizzled in 128-byte
// rows (the K-major operand layout the MMA descriptors name).
int encode_operand(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                   const char* what, int elem_bytes = 2) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const uint32_t box_cols = 128u / (uint32_t)elem_bytes;
  if (!base || rows >= (1ull << 31) || cols % box_cols != 0)
    return fail(MK_ERR_ARG, std::string("no tcgen05 operand layout for ") + what);
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * elem_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(tm, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MK_ERR_CUDA, std::string("cuTensorMapEncodeTiled failed for ") + what + " (" + std::to_string((int)r) + ")");
  return MK_OK;
}

// The weights as tcgen05 A operands: boxes of the rows one item copies --
// kTcDenseRows for QKV, O-proj and LM-head tiles, kTcRouterRows for router
// tasks, kTcMoeRows for down tiles, blocks of 16 rows of the gate and up
// matrices (an up/gate tile interleaves them).  FP8 experts: the expert
// matrices as E4M3 bytes.
int encode_weight_maps(mk_model* m) {
  if (m->tm_ready) return MK_OK;
  const mk_config& c = m->cfg;
  const ShapeDims& D = m->dims;
  const uint64_t L = (uint64_t)c.n_layers, QKV = (uint64_t)(D.NQ + 2 * D.NKV) * D.D;
  const mk_weights& w = m->w;
  int rc = encode_operand(&m->tm_w[0], w.w_qkv, L * QKV, D.H, kTcDenseRows, "w_qkv");
  if (rc == MK_OK) rc = encode_operand(&m->tm_w[1], w.w_o, L * D.H, (uint64_t)D.NQ * D.D, kTcDenseRows, "w_o");
  if (rc == MK_OK) rc = encode_operand(&m->tm_w[2], w.w_router, L * D.E, D.H, kTcRouterRows, "w_router");
  if (rc == MK_OK) rc = encode_operand(&m->tm_w[3], w.w_lm, (uint64_t)c.vocab, D.H, kTcDenseRows, "w_lm");
  const int eb = c.expert_fp8 ? 1 : 2;
  if (rc == MK_OK) rc = encode_operand(&m->tm_w[4], w.w_gate, L * D.E * D.I, D.H, 16, "w_gate", eb);
  if (rc == MK_OK) rc = encode_operand(&m->tm_w[5], w.w_up, L * D.E * D.I, D.H, 16, "w_up", eb);
  if (rc == MK_OK) rc = encode_operand(&m->tm_w[6], w.w_down, L * D.E * D.H, D.I, kTcMoeRows, "w_down", eb);
  if (rc == MK_OK) m->tm_ready = true;
  return rc;
}

// The activation operands of the tcgen05 items in the workspace: boxes of
// tc_nb rows (every activation row as a hi row and a lo row); with FP8
// experts the expert tiles' operands are E4M3 term rows in boxes of tc_nb8.
int encode_act_maps(mk_sched* s, uint8_t* ws) {
  if (s->tm_ws == ws) return MK_OK;
  const ShapeDims& D = s->dims;
  const uint64_t nb = (uint64_t)s->tc_nb;
  int rc = encode_operand(&s->tm_act[0], ws + s->ws.off("xb"), nb, D.H, s->tc_nb, "xb");
  if (rc == MK_OK) rc = encode_operand(&s->tm_act[1], ws + s->ws.off("attnb"), nb, (uint64_t)D.NQ * D.D, s->tc_nb, "attnb");
  if (s->tc_fp8) {
    const uint64_t routed = std::max<uint64_t>((uint64_t)kTcF8Terms * s->max_batch * D.K, (uint64_t)s->tc_nb8);
    if (rc == MK_OK) rc = encode_operand(&s->tm_act[2], ws + s->ws.off("xg8"), routed, D.H, s->tc_nb8, "xg8", 1);
    if (rc == MK_OK) rc = encode_operand(&s->tm_act[3], ws + s->ws.off("u8"), routed, D.I, s->tc_nb8, "u8", 1);
  } else {
    const uint64_t routed = std::max<uint64_t>(2ull * s->max_batch * D.K, nb);
    if (rc == MK_OK) rc = encode_operand(&s->tm_act[2], ws + s->ws.off("xgb"), routed, D.H, s->tc_nb, "xgb");
    if (rc == MK_OK) rc = encode_operand(&s->tm_act[3], ws + s->ws.off("ub"), routed, D.I, s->tc_nb, "ub");
  }
  s->tm_ws = rc == MK_OK ? ws : nullptr;
  return rc;
}

// After a timeout: the counters as the step left them, against the schedule.
// A wait whose target exceeds the number of tasks that signal its barrier can
// never be met; that task is the root of the stall, and every other timed-out
// wait depends on it.  Otherwise the barriers still short of their signallers
// are listed.
std::string stall_diagnosis(const mk_sched* s, const void* workspace, cudaStream_t st) {
  const size_t nb = s->bar_kind.size();
  std::vector<uint32_t> cnt(nb);
  if (cudaMemcpyAsync(cnt.data(), static_cast<const uint8_t*>(workspace) + s->ws.off("barriers"),
                      sizeof(uint32_t) * nb, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return "";
  std::vector<int64_t> sig(nb, 0);
  for (const Desc& d : s->tasks) {
    for (int f : {F_SIG0, F_SIG1})
      if (d[f] >= 0 && (size_t)d[f] < nb) ++sig[d[f]];
    // fused routing: the last router task of a layer signals the routing barrier
    if (d[F_OP] == OP_ROUTER_GEMM && d[F_A0 + 5] && d[F_A0 + 6] == 0 && d[F_A0 + 4] >= 0 &&
        (size_t)d[F_A0 + 4] < nb)
      ++sig[d[F_A0 + 4]];
  }
  for (int sm = 0; sm < s->num_sms; ++sm)
    for (int ti : s->per_sm[sm]) {
      const Desc& d = s->tasks[ti];
      for (int k = 0; k < 2; ++k) {
        const int b = d[k == 0 ? F_WAIT0 : F_WAIT1], tgt = d[k == 0 ? F_TGT0 : F_TGT1];
        if (b < 0 || (size_t)b >= nb || s->bar_kind[b] != BK_STATIC || tgt <= sig[b]) continue;
        return "; root: task " + std::to_string(d[F_TASK]) + " (sm " + std::to_string(sm) + ", op " +
               std::to_string(d[F_OP]) + ", layer " + std::to_string(d[F_LAYER]) + ") waits for " +
               std::to_string(tgt) + " signals on barrier " + std::to_string(b) + ", which " +
               std::to_string(sig[b]) + " tasks signal (count " + std::to_string(cnt[b]) + ")";
      }
    }
  // the SMs whose consumers stopped in the earliest layer: where the stall is
  std::string lag;
  std::vector<uint32_t> pr(8 * (size_t)s->num_sms);
  if (cudaMemcpyAsync(pr.data(), static_cast<const uint8_t*>(workspace) + s->ws.off("progress"),
                      sizeof(uint32_t) * pr.size(), cudaMemcpyDeviceToHost, st) == cudaSuccess &&
      cudaStreamSynchronize(st) == cudaSuccess) {
    std::vector<std::pair<uint32_t, int>> order;
    for (int sm = 0; sm < s->num_sms; ++sm)
      if (pr[8 * sm + 3] < s->per_sm[sm].size()) order.push_back({(pr[8 * sm + 1] >> 8) & 0xff, sm});
    std::sort(order.begin(), order.end());
    for (size_t k = 0; k < order.size() && k < 3; ++k) {
      const uint32_t* r = &pr[8 * order[k].second];
      lag += "; sm " + std::to_string(order[k].second) + ": consumer item " + std::to_string(r[0]) + " (op " +
             std::to_string(r[1] & 0xff) + ", layer " + std::to_string((r[1] >> 8) & 0xff) + ", task " +
             std::to_string(r[1] >> 16) + ", stages " + std::to_string(r[2]) + "), producer task " +
             std::to_string(r[3]) + " of " + std::to_string(s->per_sm[order[k].second].size()) + " (stages " +
             std::to_string(r[4]) + ", items " + std::to_string(r[5]) + "), storer " + std::to_string(r[6]);
    }
  }
  std::string short_bars;
  int n = 0;
  for (size_t b = 0; b < nb; ++b)
    if (s->bar_kind[b] == BK_STATIC && cnt[b] < sig[b] && n++ < 4)
      short_bars += " " + std::to_string(b) + " (" + std::to_string(cnt[b]) + " of " + std::to_string(sig[b]) + ")";
  return (n ? "; barriers short of their signallers:" + short_bars + (n > 4 ? " ..." : "") : std::string()) + lag;
}

}  // namespace
}  // namespace mk

using namespace mk;

extern "C" {

const char* mk_last_error(void) { return g_error.c_str(); }

int mk_load_model(const mk_config* cfg, const mk_weights* w, mk_model** out) {
  if (!cfg || !w || !out) return fail(MK_ERR_ARG, "null argument");
  *out = nullptr;
  const mk_config& c = *cfg;
  if (c.n_layers < 1 || c.vocab < 1 || c.window < 0 || c.full_period < 1 || !(c.rope_base > 0.f) ||
      !(c.eps >= 0.f))
    return fail(MK_ERR_ARG, "invalid config (layers, vocab, window, full_period, rope_base or eps)");
  int id = -1;
  for (int i = 0; i < (int)(sizeof(kShapes) / sizeof(kShapes[0])); ++i) {
    const ShapeDims& d = kShapes[i].dims;
    if (d.H == c.hidden && d.NQ == c.n_q && d.NKV == c.n_kv && d.D == c.head_dim && d.E == c.n_experts &&
        d.K == c.top_k && d.I == c.inter && d.P == c.page_size)
      id = i;
  }
  if (id < 0) return fail(MK_ERR_UNSUPPORTED, "no compiled kernel for this model shape");
  const bool dense = c.n_experts == 1 && c.top_k == 1;  // no router: w_router may be null
  if (!w->embedding || !w->w_qkv || !w->w_o || (!w->w_router && !dense) || !w->w_gate || !w->w_up ||
      !w->w_down || !w->norm_gamma || !w->final_gamma || !w->w_lm)
    return fail(MK_ERR_ARG, "a weight pointer is null");
  if (c.expert_fp8 != 0 && c.expert_fp8 != 1) return fail(MK_ERR_ARG, "expert_fp8 must be 0 or 1");
  if (c.expert_fp8 && (!w->w_gate_scale || !w->w_up_scale || !w->w_down_scale))
    return fail(MK_ERR_ARG, "FP8 experts need the three row-scale arrays");
  if (c.expert_fp4 != 0 && c.expert_fp4 != 1) return fail(MK_ERR_ARG, "expert_fp4 must be 0 or 1");
  if (c.expert_fp4 && c.expert_fp8) return fail(MK_ERR_ARG, "expert_fp8 and expert_fp4 exclude each other");
  if (c.expert_fp4 && (!w->w_gate_scale || !w->w_up_scale || !w->w_down_scale || !w->w_gate_bscale ||
                       !w->w_up_bscale || !w->w_down_bscale))
    return fail(MK_ERR_ARG, "FP4 experts need the three row-scale and three block-scale arrays");
  const void* ptrs[] = {w->embedding, w->w_qkv, w->w_o, w->w_router, w->router_bias, w->w_gate, w->w_up,
                        w->w_down, w->norm_gamma, w->final_gamma, w->w_lm, w->w_gate_scale, w->w_up_scale,
                        w->w_down_scale, w->w_gate_bscale, w->w_up_bscale, w->w_down_bscale};
  for (const void* q : ptrs)
    if (reinterpret_cast<uintptr_t>(q) & 15u) return fail(MK_ERR_ARG, "weight pointers must be 16-byte aligned");
  if (c.expert_fp8) {
    // the row scales travel with each stage in 16-byte units
    const MoePlan p8 = moe_plan8(kShapes[id].dims);
    // and the rows go to the tensor cores in groups of 16 (gate/up: 8 + 8)
    if (p8.up_half % 8 || p8.dn_rows % 16 || 2 * p8.up_half > kMaxStageRows || p8.dn_rows > kMaxStageRows)
      return fail(MK_ERR_UNSUPPORTED, "no FP8 stage plan for this model shape");
  }
  if (c.expert_fp4) {
    // 128-input chunks per MMA step; a 16-row stage (codes and block scales) in one slot
    const ShapeDims& d = kShapes[id].dims;
    const MoePlan p4 = moe_plan4(d);
    if (d.H % 128 || d.I % 128 || fp4_stage_bytes(d.H) > kStageBytes || fp4_stage_bytes(d.I) > kStageBytes ||
        p4.up_tile * p4.up_tiles != d.I || p4.dn_tile * p4.dn_tiles != d.H)
      return fail(MK_ERR_UNSUPPORTED, "no FP4 stage plan for this model shape");
  }
  mk_model* m = new mk_model();
  m->cfg = c;
  m->w = *w;
  m->shape_id = id;
  m->dims = kShapes[id].dims;
  m->plan = c.expert_fp8 ? moe_plan8(m->dims) : c.expert_fp4 ? moe_plan4(m->dims) : moe_plan(m->dims);
  *out = m;
  return MK_OK;
}

void mk_free_model(mk_model* m) { delete m; }

int mk_sched_upload(mk_sched* s, void* dev, size_t bytes, void* stream) {
  if (!s || !dev) return fail(MK_ERR_ARG, "null argument");
  if (bytes < mk_sched_bytes(s)) return fail(MK_ERR_ARG, "sched buffer too small");
  if (reinterpret_cast<uintptr_t>(dev) & 127u) return fail(MK_ERR_ARG, "sched buffer must be 128-byte aligned");
  // [num_sms][2] (offset, count) header, then each SM's descriptors
  const int nsm = s->num_sms;
  size_t off = ((size_t)2 * nsm + 31) / 32 * 32;
  s->upload.assign(off + 32 * s->tasks.size(), 0);
  for (int sm = 0; sm < nsm; ++sm) {
    s->upload[2 * sm] = (int32_t)off;
    s->upload[2 * sm + 1] = (int32_t)s->per_sm[sm].size();
    int pos = 0;
    for (int t : s->per_sm[sm]) {
      std::memcpy(&s->upload[off], s->tasks[t].data(), sizeof(int32_t) * 32);
      s->upload[off + F_POS] = pos++;
      off += 32;
    }
  }
  cudaError_t e = cudaMemcpyAsync(dev, s->upload.data(), sizeof(int32_t) * s->upload.size(),
                                  cudaMemcpyHostToDevice, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "upload of the task lists");
  s->sched_dev = dev;
  return MK_OK;
}

int mk_check_inputs(const mk_sched* s, const int32_t* last_tokens, const int32_t* seq_lens,
                    const int32_t* block_tables, int32_t batch, int32_t max_pages, int64_t num_pages) {
  if (!s || !seq_lens || !block_tables) return fail(MK_ERR_ARG, "null argument");
  if (batch < 1 || batch > s->max_batch)
    return fail(MK_ERR_ARG, "batch " + std::to_string(batch) + " outside [1, " + std::to_string(s->max_batch) + "]");
  if (max_pages < 1 || num_pages < 1) return fail(MK_ERR_ARG, "max_pages and num_pages must be positive");
  const int P = s->dims.P;
  for (int32_t b = 0; b < batch; ++b) {
    const int32_t len = seq_lens[b];
    if (len < 1 || len > s->max_ctx)
      return fail(MK_ERR_ARG, "row " + std::to_string(b) + ": seq_len " + std::to_string(len) + " outside [1, " +
                                  std::to_string(s->max_ctx) + "] (the schedule's max_ctx)");
    const int32_t pages = (len + P - 1) / P;
    if (pages > max_pages)
      return fail(MK_ERR_ARG, "row " + std::to_string(b) + ": seq_len " + std::to_string(len) + " needs " +
                                  std::to_string(pages) + " pages, the block table has " + std::to_string(max_pages));
    for (int32_t j = 0; j < pages; ++j) {
      const int32_t pg = block_tables[(size_t)b * max_pages + j];
      if (pg < 0 || pg >= num_pages)
        return fail(MK_ERR_ARG, "row " + std::to_string(b) + ": page " + std::to_string(pg) + " at logical page " +
                                    std::to_string(j) + " outside [0, " + std::to_string(num_pages) + ")");
    }
    if (last_tokens && (last_tokens[b] < 0 || last_tokens[b] >= s->cfg.vocab))
      return fail(MK_ERR_ARG, "row " + std::to_string(b) + ": token " + std::to_string(last_tokens[b]) +
                                  " outside [0, " + std::to_string(s->cfg.vocab) + ")");
  }
  return MK_OK;
}

int mk_decode_step(mk_model* m, mk_sched* s, const int32_t* last_tokens, const int32_t* seq_lens,
                   const int32_t* block_tables, int32_t batch, int32_t max_pages, void* k_pool,
                   void* v_pool, int64_t num_pages, void* workspace, size_t workspace_bytes,
                   float* logits, void* stream) {
  if (!m || !s) return fail(MK_ERR_ARG, "null model or schedule");
  if (!s->sched_dev) return fail(MK_ERR_ARG, "schedule not uploaded");
  if (std::memcmp(&m->cfg, &s->cfg, sizeof(mk_config)) != 0)
    return fail(MK_ERR_ARG, "schedule was built for another model");
  if (batch < 1 || batch > s->max_batch) return fail(MK_ERR_ARG, "batch outside [1, max_batch]");
  if (!last_tokens || !seq_lens || !block_tables || !k_pool || !v_pool || !workspace || !logits)
    return fail(MK_ERR_ARG, "null device pointer");
  if (max_pages < 1 || num_pages < 1) return fail(MK_ERR_ARG, "max_pages and num_pages must be positive");
  if (workspace_bytes < s->ws.total) return fail(MK_ERR_ARG, "workspace too small");
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(MK_ERR_ARG, "workspace must be 256-byte aligned");
  if ((reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool)) & 15u)
    return fail(MK_ERR_ARG, "KV pools must be 16-byte aligned");

  const ShapeDims& D = s->dims;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto at = [&](const char* name) -> uint8_t* {
    const size_t o = s->ws.off(name);
    return o == (size_t)-1 ? nullptr : ws + o;
  };
  Params p{};
  const mk_weights& w = m->w;
  p.emb = static_cast<const uint16_t*>(w.embedding);
  p.wqkv = static_cast<const uint16_t*>(w.w_qkv);
  p.wo = static_cast<const uint16_t*>(w.w_o);
  p.wr = static_cast<const uint16_t*>(w.w_router);
  p.rbias = w.router_bias;
  p.wg = static_cast<const uint16_t*>(w.w_gate);
  p.wu = static_cast<const uint16_t*>(w.w_up);
  p.wd = static_cast<const uint16_t*>(w.w_down);
  p.expert_fp8 = m->cfg.expert_fp8;
  p.sg = w.w_gate_scale;
  p.su = w.w_up_scale;
  p.sd = w.w_down_scale;
  p.expert_fp4 = m->cfg.expert_fp4;
  p.bg = static_cast<const uint8_t*>(w.w_gate_bscale);
  p.bu = static_cast<const uint8_t*>(w.w_up_bscale);
  p.bd = static_cast<const uint8_t*>(w.w_down_bscale);
  p.gamma = w.norm_gamma;
  p.gamma_f = w.final_gamma;
  p.wlm = static_cast<const uint16_t*>(w.w_lm);
  p.L = m->cfg.n_layers;
  p.V = m->cfg.vocab;
  p.window = m->cfg.window;
  p.full_period = m->cfg.full_period;
  p.rope_base = m->cfg.rope_base;
  p.eps = m->cfg.eps;
  p.B = batch;
  p.MB = s->max_batch;
  p.tokens = last_tokens;
  p.block_tables = block_tables;
  p.max_pages = max_pages;
  p.kpool = static_cast<uint16_t*>(k_pool);
  p.vpool = static_cast<uint16_t*>(v_pool);
  p.num_pages = num_pages;
  p.logits = logits;
  p.sched = static_cast<const int32_t*>(s->sched_dev);
  p.bars = reinterpret_cast<uint32_t*>(at("barriers"));
  p.err = reinterpret_cast<uint32_t*>(at("error"));
  p.prog = reinterpret_cast<uint32_t*>(at("progress"));
  p.seq_lens = seq_lens;
  p.max_ctx = s->max_ctx;
  p.h = reinterpret_cast<float*>(at("h"));
  p.x = reinterpret_cast<float*>(at("x"));
  p.q = reinterpret_cast<float*>(at("q"));
  p.kvnew = reinterpret_cast<uint16_t*>(at("kvnew"));
  p.part_o = reinterpret_cast<float*>(at("part_o"));
  p.part_ml = reinterpret_cast<float*>(at("part_ml"));
  p.attn_out = reinterpret_cast<float*>(at("attn_out"));
  p.opart = reinterpret_cast<float*>(at("opart"));
  p.rlog = reinterpret_cast<float*>(at("router_logits"));
  p.topk_ids = reinterpret_cast<int32_t*>(at("topk_ids"));
  p.topk_w = reinterpret_cast<float*>(at("topk_w"));
  p.ecount = reinterpret_cast<int32_t*>(at("expert_count"));
  p.eoff = reinterpret_cast<int32_t*>(at("expert_offset"));
  p.perm = reinterpret_cast<int32_t*>(at("perm"));
  p.inv = reinterpret_cast<int32_t*>(at("inv"));
  p.act = reinterpret_cast<int32_t*>(at("moe_queue"));
  p.qlen = reinterpret_cast<int32_t*>(at("moe_queue_len"));
  p.xg = reinterpret_cast<float*>(at("xg"));
  p.u = reinterpret_cast<float*>(at("u"));
  p.y = reinterpret_cast<float*>(at("y"));
  p.moe_out = reinterpret_cast<float*>(at("moe_out"));
  p.htrace = reinterpret_cast<float*>(at("hidden_trace"));
  p.qtrace = reinterpret_cast<int32_t*>(at("queue_trace"));
  p.trace = reinterpret_cast<uint64_t*>(at("trace"));
  p.trace_cap = s->trace_cap;
  p.stats = reinterpret_cast<uint64_t*>(at("stats"));
  p.split_len = s->split_len;
  p.n_static = s->n_static;
  p.max_slots = s->max_slots;
  p.explicit_gather = s->opts.explicit_gather;
  p.watchdog_ns = s->watchdog_ns;
  (void)D;

  if (s->tm_kpool != k_pool || s->tm_vpool != v_pool || s->tm_pages != num_pages) {
    int rc = encode_pool(&s->tm_k, k_pool, s, num_pages);
    if (rc == MK_OK) rc = encode_pool(&s->tm_v, v_pool, s, num_pages);
    if (rc != MK_OK) {
      s->tm_kpool = s->tm_vpool = nullptr;
      return rc;
    }
    s->tm_kpool = k_pool;
    s->tm_vpool = v_pool;
    s->tm_pages = num_pages;
  }
  p.tm_k = s->tm_k;
  p.tm_v = s->tm_v;
  if (s->tc) {
    int rc = encode_weight_maps(m);
    if (rc == MK_OK) rc = encode_act_maps(s, ws);
    if (rc != MK_OK) return rc;
    p.tm_wqkv = m->tm_w[0]; p.tm_wo = m->tm_w[1]; p.tm_wr = m->tm_w[2]; p.tm_wlm = m->tm_w[3];
    p.tm_wg = m->tm_w[4]; p.tm_wu = m->tm_w[5]; p.tm_wd = m->tm_w[6];
    p.tm_xb = s->tm_act[0]; p.tm_attnb = s->tm_act[1];
    p.xb = reinterpret_cast<uint16_t*>(at("xb"));
    p.attnb = reinterpret_cast<uint16_t*>(at("attnb"));
    p.tc_nb = s->tc_nb;
    if (s->tc_fp8) {
      p.tm_xg8 = s->tm_act[2]; p.tm_u8 = s->tm_act[3];
      p.xg8 = at("xg8");
      p.u8 = at("u8");
      p.xg8s = reinterpret_cast<float*>(at("xg8s"));
      p.tc_nb8 = s->tc_nb8;
    } else {
      p.tm_xgb = s->tm_act[2]; p.tm_ub = s->tm_act[3];
      p.xgb = reinterpret_cast<uint16_t*>(at("xgb"));
      p.ub = reinterpret_cast<uint16_t*>(at("ub"));
    }
  }

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // "Barriers": the counters are zeroed before each step (with the error record)
  const size_t zero_bytes = s->ws.off("progress") + sizeof(uint32_t) * 8 * (size_t)s->num_sms;
  cudaError_t e = cudaMemsetAsync(workspace, 0, zero_bytes, st);
  if (e != cudaSuccess) return cuda_fail(e, "barrier reset");
  // the kernel build for the model's expert format and the schedule's batch
  const int mode = s->tc               ? (s->tc_fp8 ? kModeTcFp8 : kModeTc)
                   : m->cfg.expert_fp4 ? (s->lean ? kModeFp4Lean : kModeFp4)
                   : m->cfg.expert_fp8 ? (s->lean ? kModeFp8Lean : kModeFp8)
                   : s->max_batch <= kTB && s->lean ? kModeSmallBatch : kModeAnyBatch;
  const int rc = kShapes[m->shape_id].launch[mode](p, s->num_sms, st);
  if (rc != 0) return cuda_fail((cudaError_t)rc, "megakernel launch");
  return MK_OK;
}

}  // extern "C"

namespace mk {
int check_record(const mk_sched* s, const uint32_t* rec, const void* workspace, void* stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (rec[0] == 0) return MK_OK;
  const std::string where = " (sm " + std::to_string(rec[1]) + ", task " + std::to_string((int32_t)rec[2]) +
                            ", op " + std::to_string((int32_t)rec[6]) + ", layer " +
                            std::to_string((int32_t)rec[7]) + ", index " + std::to_string((int32_t)rec[3]) +
                            ", value " + std::to_string((int32_t)rec[4]) + ", limit " +
                            std::to_string((int32_t)rec[5]) + ")";
  if (rec[0] == 1) return fail(MK_ERR_TIMEOUT, "device wait timed out" + where + stall_diagnosis(s, workspace, st));
  if (rec[0] == 2) return fail(MK_ERR_DEVICE, "page id out of range" + where);
  if (rec[0] == 4) return fail(MK_ERR_DEVICE, "shared memory base not 1024-byte aligned" + where);
  if (rec[0] == 5)
    return fail(MK_ERR_DEVICE, "descriptor or work ring out of step (a stale entry was read)" + where);
  if (rec[0] == 6)
    return fail(MK_ERR_DEVICE, "an FP8 or FP4 expert tile's activation is beyond the range of its operand format (|x| > " +
                                   std::to_string(rec[5]) + ")" + where);
  return fail(MK_ERR_DEVICE, "index out of range" + where);
}
}  // namespace mk

extern "C" {

int mk_check_step(const mk_sched* s, const void* workspace, void* stream) {
  if (!s || !workspace) return fail(MK_ERR_ARG, "null argument");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t rec[8];
  cudaError_t e = cudaMemcpyAsync(rec, static_cast<const uint8_t*>(workspace) + s->ws.off("error"), sizeof rec,
                                  cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "step");
  return mk::check_record(s, rec, workspace, stream);
}

}  // extern "C"
