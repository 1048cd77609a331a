// mk_static_ws.cu -- the decode step with a built-in workspace, for callers
// that cannot allocate device memory.
//
// mk_decode_step takes a caller-allocated workspace.  Some callers cannot
// provide one: their device memory is owned by another allocator (a host
// framework's caching allocator, or a runtime whose memory budget is fixed at
// start-up) and they may not call cudaMalloc once running -- cudaMalloc can
// synchronise the device and can fail under a fixed budget.  For them this
// file keeps one workspace in a file-scope device array, loaded with the
// library on every device that uses it, and runs the unchanged decode step
// on it.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "mk_host.h"

namespace {

// 8 MiB: enough for the schedules of the bundled shapes at batch 1 up to long
// contexts (the full shape at 8K context needs about 1.3 MiB); larger
// schedules are rejected.
constexpr size_t kStaticWorkspaceBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_ws_mutex[kMaxDevices];
void* g_ws_ptr[kMaxDevices];  // the array's device address on each device, once found

// The array's device address on `dev` (current): the host-side name of the
// array is only a stand-in, the kernel needs its device address.  Only a
// successful lookup is kept, so a lookup that failed (for example during a
// stream capture) is tried again on the next call.
cudaError_t resolve_workspace(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_ws_mutex[dev]);
  if (!g_ws_ptr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_workspace);
    if (e != cudaSuccess) {
      cudaGetLastError();  // do not leave the error for the caller's next CUDA call
      return e;
    }
    g_ws_ptr[dev] = ptr;
  }
  *out = g_ws_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int mk_decode_step_static_ws(mk_model* m, mk_sched* s, const int32_t* last_tokens,
                                        const int32_t* seq_lens, const int32_t* block_tables,
                                        int32_t batch, int32_t max_pages, void* k_pool, void* v_pool,
                                        int64_t num_pages, float* logits, void* stream) {
  if (!m || !s) return mk::fail(MK_ERR_ARG, "null model or schedule");
  const size_t need = mk_workspace_bytes(s);
  if (need > kStaticWorkspaceBytes)
    return mk::fail(MK_ERR_ARG, "this schedule needs " + std::to_string(need) +
                                    " bytes of workspace; the built-in workspace holds " +
                                    std::to_string(kStaticWorkspaceBytes) +
                                    " bytes: use mk_decode_step with a caller-allocated workspace");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return mk::fail(MK_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return mk::fail(MK_ERR_ARG, "device ordinal beyond the supported range");
  void* ws = nullptr;
  e = resolve_workspace(dev, &ws);
  if (e != cudaSuccess)
    return mk::fail(MK_ERR_CUDA, std::string("cudaGetSymbolAddress of the built-in workspace: ") +
                                     cudaGetErrorString(e));
  return mk_decode_step(m, s, last_tokens, seq_lens, block_tables, batch, max_pages, k_pool, v_pool, num_pages,
                        ws, kStaticWorkspaceBytes, logits, stream);
}
