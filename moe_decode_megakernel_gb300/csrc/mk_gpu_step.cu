// mk_gpu_step.cu -- the decode service's step on the GPU: the host arrays
// to the device, mk_decode_step with the smallest schedule that covers the
// batch, a greedy argmax per row on the device, the tokens back.
#include <cuda_runtime.h>

#include <algorithm>
#include <cfloat>
#include <string>
#include <vector>

#include "../../include/mk_service.h"
#include "mk_host.h"

using mk::fail;

namespace {

constexpr int kArgmaxThreads = 512;

// One block per row: each thread scans a strided part of the row; the
// (value, index) pairs meet by warp shuffles, then across warps in shared
// memory.  Ties go to the lower index; NaN compares false, so it never wins.
__global__ void __launch_bounds__(kArgmaxThreads) argmax_rows(const float* __restrict__ logits, int vocab,
                                                                int32_t* __restrict__ next,
                                                                const uint32_t* __restrict__ rec_src,
                                                                uint32_t* __restrict__ rec_dst) {
  // the GPU step's copy of the step's error record, beside the tokens
  if (rec_src && blockIdx.x == 0 && threadIdx.x < 8) rec_dst[threadIdx.x] = rec_src[threadIdx.x];
  const float* row = logits + (size_t)blockIdx.x * vocab;
  float best = -FLT_MAX;
  int idx = vocab;  // "none yet": any real index is lower
  for (int i = threadIdx.x; i < vocab; i += blockDim.x) {
    const float v = row[i];
    if (v > best || (v == best && i < idx)) {
      best = v;
      idx = i;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    if (b2 > best || (b2 == best && i2 < idx)) {
      best = b2;
      idx = i2;
    }
  }
  __shared__ float wb[kArgmaxThreads / 32];
  __shared__ int wi[kArgmaxThreads / 32];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    wb[w] = best;
    wi[w] = idx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < (int)(blockDim.x >> 5); ++k)
      if (wb[k] > best || (wb[k] == best && wi[k] < idx)) {
        best = wb[k];
        idx = wi[k];
      }
    next[blockIdx.x] = idx < vocab ? idx : 0;  // every value NaN: token 0
  }
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

}  // namespace

struct mk_gpu_step {
  ~mk_gpu_step() {
    for (auto& gr : graphs) cudaGraphExecDestroy(gr.exec);
    if (h_in) cudaFreeHost(h_in);
    if (h_out) cudaFreeHost(h_out);
  }
  // one captured step per (schedule, batch): the input copy, mk_decode_step,
  // the argmax and the output copy replayed by one launch; off for good if a
  // capture fails (the steps are then issued one by one)
  struct Graph {
    mk_sched* s;
    int32_t batch;
    cudaGraphExec_t exec;
  };
  std::vector<Graph> graphs;
  bool graphs_off = false;
  mk_model* model = nullptr;
  std::vector<mk_sched*> scheds;
  void* k_pool = nullptr;
  void* v_pool = nullptr;
  int64_t num_pages = 0;
  int32_t max_pages = 0, max_batch = 0;
  void* workspace = nullptr;
  size_t ws_bytes = 0;
  cudaStream_t stream = nullptr;
  // device parts of dev_buf: the inputs as one block (tokens, lengths, block
  // tables of the step's batch), the outputs (tokens, then the error record)
  int32_t* d_in = nullptr;
  int32_t* d_out = nullptr;
  float* d_logits = nullptr;
  // pinned host copies of both: one copy each way per step
  int32_t* h_in = nullptr;
  int32_t* h_out = nullptr;
};

namespace {
// One step on the stream: the packed inputs in (one copy), mk_decode_step,
// the greedy tokens and the step's error record side by side, one copy out.
int enqueue_step(mk_gpu_step* g, mk_sched* s, int32_t batch, int32_t max_pages) {
  cudaStream_t st = g->stream;
  const size_t B = (size_t)batch;
  cudaError_t e = cudaMemcpyAsync(g->d_in, g->h_in, sizeof(int32_t) * B * (2 + (size_t)max_pages),
                                  cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return fail(MK_ERR_CUDA, std::string("step inputs: ") + cudaGetErrorString(e));
  const int rc = mk_decode_step(g->model, s, g->d_in, g->d_in + B, g->d_in + 2 * B, batch, max_pages, g->k_pool,
                                g->v_pool, g->num_pages, g->workspace, g->ws_bytes, g->d_logits, st);
  if (rc != MK_OK) return rc;
  const uint32_t* rec = reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(g->workspace) +
                                                          s->ws.off("error"));
  argmax_rows<<<batch, kArgmaxThreads, 0, st>>>(g->d_logits, g->model->cfg.vocab, g->d_out, rec,
                                                reinterpret_cast<uint32_t*>(g->d_out + B));
  e = cudaGetLastError();
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(g->h_out, g->d_out, sizeof(int32_t) * (B + 8), cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return fail(MK_ERR_CUDA, std::string("step outputs: ") + cudaGetErrorString(e));
  return MK_OK;
}
}  // namespace

extern "C" {

int mk_argmax_rows(const float* logits, int32_t rows, int32_t vocab, int32_t* next, void* stream) {
  if (!logits || !next || rows < 0 || vocab < 1) return fail(MK_ERR_ARG, "bad argmax arguments");
  if (rows == 0) return MK_OK;
  argmax_rows<<<rows, kArgmaxThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(logits, vocab, next, nullptr,
                                                                                   nullptr);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MK_ERR_CUDA, std::string("argmax launch: ") + cudaGetErrorString(e));
  return MK_OK;
}

size_t mk_gpu_step_dev_bytes(const mk_model* m, int32_t max_batch, int32_t max_pages) {
  if (!m || max_batch < 1 || max_pages < 1) return 0;
  const size_t B = (size_t)max_batch;
  return align256(sizeof(int32_t) * B * (2 + (size_t)max_pages)) + align256(sizeof(int32_t) * (B + 8)) +
         align256(sizeof(float) * B * m->cfg.vocab);
}

int mk_gpu_step_create(mk_model* m, mk_sched* const* scheds, int32_t n_scheds, void* k_pool, void* v_pool,
                       int64_t num_pages, int32_t max_pages, void* workspace, size_t workspace_bytes,
                       void* dev_buf, size_t dev_bytes, void* stream, mk_gpu_step** out) {
  if (!m || !scheds || n_scheds < 1 || !k_pool || !v_pool || !workspace || !dev_buf || !out)
    return fail(MK_ERR_ARG, "null argument");
  *out = nullptr;
  if (num_pages < 1 || max_pages < 1) return fail(MK_ERR_ARG, "num_pages and max_pages must be positive");
  int32_t mb = 0;
  for (int32_t i = 0; i < n_scheds; ++i) {
    if (!scheds[i] || !scheds[i]->sched_dev) return fail(MK_ERR_ARG, "schedule " + std::to_string(i) + " not uploaded");
    if (mk_workspace_bytes(scheds[i]) > workspace_bytes)
      return fail(MK_ERR_ARG, "workspace smaller than schedule " + std::to_string(i) + " needs");
    mb = std::max(mb, (int32_t)scheds[i]->max_batch);
  }
  const size_t need = mk_gpu_step_dev_bytes(m, mb, max_pages);
  if (dev_bytes < need) return fail(MK_ERR_ARG, "dev_buf holds " + std::to_string(dev_bytes) + " bytes, " +
                                                    std::to_string(need) + " needed");
  mk_gpu_step* g = new mk_gpu_step;
  g->model = m;
  g->scheds.assign(scheds, scheds + n_scheds);
  g->k_pool = k_pool;
  g->v_pool = v_pool;
  g->num_pages = num_pages;
  g->max_pages = max_pages;
  g->max_batch = mb;
  g->workspace = workspace;
  g->ws_bytes = workspace_bytes;
  g->stream = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* b = static_cast<uint8_t*>(dev_buf);
  const size_t B = (size_t)mb;
  const size_t in_words = B * (2 + (size_t)max_pages), out_words = B + 8;
  g->d_in = reinterpret_cast<int32_t*>(b);
  b += align256(sizeof(int32_t) * in_words);
  g->d_out = reinterpret_cast<int32_t*>(b);
  b += align256(sizeof(int32_t) * out_words);
  g->d_logits = reinterpret_cast<float*>(b);
  cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&g->h_in), sizeof(int32_t) * in_words, cudaHostAllocDefault);
  if (e == cudaSuccess)
    e = cudaHostAlloc(reinterpret_cast<void**>(&g->h_out), sizeof(int32_t) * out_words, cudaHostAllocDefault);
  if (e != cudaSuccess) {
    delete g;
    return fail(MK_ERR_CUDA, std::string("pinned staging buffers: ") + cudaGetErrorString(e));
  }
  *out = g;
  return MK_OK;
}

void mk_gpu_step_free(mk_gpu_step* g) { delete g; }

int mk_gpu_step_run(void* ctx, const int32_t* last_tokens, const int32_t* seq_lens, const int32_t* block_tables,
                    int32_t batch, int32_t max_pages, int32_t* next_tokens) {
  mk_gpu_step* g = static_cast<mk_gpu_step*>(ctx);
  if (!g || !last_tokens || !seq_lens || !block_tables || !next_tokens) return fail(MK_ERR_ARG, "null argument");
  if (batch < 1 || batch > g->max_batch || max_pages != g->max_pages)
    return fail(MK_ERR_ARG, "batch or block-table width outside what the GPU step was made for");
  int32_t longest = 0;
  for (int32_t r = 0; r < batch; ++r) longest = std::max(longest, seq_lens[r]);
  mk_sched* s = nullptr;
  for (mk_sched* c : g->scheds)
    if (c->max_batch >= batch && c->max_ctx >= longest) {
      s = c;
      break;
    }
  if (!s) return fail(MK_ERR_ARG, "no schedule covers batch " + std::to_string(batch) + " at context " +
                                      std::to_string(longest));
  // the host holds the inputs: refuse bad ones before anything is launched
  const int chk = mk_check_inputs(s, last_tokens, seq_lens, block_tables, batch, max_pages, g->num_pages);
  if (chk != MK_OK) return chk;
  cudaStream_t st = g->stream;
  const size_t B = (size_t)batch;
  // the inputs, packed in pinned memory (read when the copy runs)
  std::copy(last_tokens, last_tokens + B, g->h_in);
  std::copy(seq_lens, seq_lens + B, g->h_in + B);
  std::copy(block_tables, block_tables + B * max_pages, g->h_in + 2 * B);
  cudaGraphExec_t exec = nullptr;
  for (const auto& gr : g->graphs)
    if (gr.s == s && gr.batch == batch) exec = gr.exec;
  if (!exec && !g->graphs_off) {
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal);
    int rc = e == cudaSuccess ? enqueue_step(g, s, batch, max_pages) : MK_ERR_CUDA;
    if (e == cudaSuccess) e = cudaStreamEndCapture(st, &graph);
    if (rc == MK_OK && e == cudaSuccess) e = cudaGraphInstantiate(&exec, graph, 0);
    if (graph) cudaGraphDestroy(graph);
    if (rc != MK_OK || e != cudaSuccess) {
      g->graphs_off = true;
      exec = nullptr;
      cudaGetLastError();  // the failed capture is not the step's error
    } else {
      g->graphs.push_back({s, batch, exec});
    }
  }
  cudaError_t e = cudaSuccess;
  if (exec) {
    e = cudaGraphLaunch(exec, st);
  } else {
    const int rc = enqueue_step(g, s, batch, max_pages);
    if (rc != MK_OK) return rc;
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail(MK_ERR_CUDA, std::string("step outputs: ") + cudaGetErrorString(e));
  const int rc = mk::check_record(s, reinterpret_cast<const uint32_t*>(g->h_out + B), g->workspace, st);
  if (rc != MK_OK) return rc;
  std::copy(g->h_out, g->h_out + B, next_tokens);
  return MK_OK;
}

}  // extern "C"
