// synth_fill.cu -- fills host or device buffers with the synthetic BF16
// inputs defined in synth.h (weights and KV pools of the decode step).
//
// Exported C ABI (libsynth.so):
//   synth_fill_device(dst, n_streams, per_stream, seed, kind, layer0, expert0,
//                     vary_layer, sigma, stream) -> 0 or a cudaError_t value
//   synth_fill_host(...)  same, on the host, into a host buffer
//
// Element i of sub-stream j (0 <= j < n_streams) goes to dst[j*per_stream+i]
// and equals synth_bf16(key(seed, stream(kind, L, X)), i, scale(sigma)) with
// (L, X) = (layer0 + j, expert0) if vary_layer else (layer0, expert0 + j).
#include <cuda_runtime.h>
#include <stdint.h>
#include "synth.h"

namespace {

__device__ __forceinline__ uint64_t stream_of(uint32_t kind, uint32_t layer0, uint32_t expert0,
                                              int vary_layer, uint64_t j) {
  return vary_layer ? synth_stream(kind, layer0 + (uint32_t)j, expert0)
                    : synth_stream(kind, layer0, expert0 + (uint32_t)j);
}

// 8 consecutive elements per thread, one 16-byte store (per_stream % 8 == 0).
__global__ void fill_vec8(uint16_t* __restrict__ dst, uint64_t n_streams, uint64_t per_stream,
                          uint64_t seed, uint32_t kind, uint32_t layer0, uint32_t expert0,
                          int vary_layer, float scale) {
  const uint64_t groups_per_stream = per_stream / 8;
  const uint64_t total = n_streams * groups_per_stream;
  for (uint64_t g = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t j = g / groups_per_stream;
    const uint64_t i0 = (g - j * groups_per_stream) * 8;
    const uint64_t key = synth_key(seed, stream_of(kind, layer0, expert0, vary_layer, j));
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t lo = synth_bf16(key, i0 + 2 * q, scale);
      uint32_t hi = synth_bf16(key, i0 + 2 * q + 1, scale);
      w[q] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(dst + j * per_stream + i0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__global__ void fill_scalar(uint16_t* __restrict__ dst, uint64_t n_streams, uint64_t per_stream,
                            uint64_t seed, uint32_t kind, uint32_t layer0, uint32_t expert0,
                            int vary_layer, float scale) {
  const uint64_t total = n_streams * per_stream;
  for (uint64_t g = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t j = g / per_stream;
    const uint64_t i = g - j * per_stream;
    const uint64_t key = synth_key(seed, stream_of(kind, layer0, expert0, vary_layer, j));
    dst[g] = synth_bf16(key, i, scale);
  }
}

}  // namespace

extern "C" int synth_fill_device(void* dst, uint64_t n_streams, uint64_t per_stream, uint64_t seed,
                                 uint32_t kind, uint32_t layer0, uint32_t expert0, int vary_layer,
                                 double sigma, void* stream) {
  if (dst == nullptr || n_streams == 0 || per_stream == 0) return (int)cudaErrorInvalidValue;
  const float scale = synth_scale(sigma);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int threads = 256;
  const int blocks = (sms > 0 ? sms : 1) * 8;
  if (per_stream % 8 == 0 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
    fill_vec8<<<blocks, threads, 0, s>>>(static_cast<uint16_t*>(dst), n_streams, per_stream, seed,
                                         kind, layer0, expert0, vary_layer, scale);
  } else {
    fill_scalar<<<blocks, threads, 0, s>>>(static_cast<uint16_t*>(dst), n_streams, per_stream,
                                           seed, kind, layer0, expert0, vary_layer, scale);
  }
  return (int)cudaGetLastError();
}

// The raw 64-bit draw (for checking the generator against splitmix64's
// published output sequence).
extern "C" uint64_t synth_raw(uint64_t key, uint64_t idx) { return synth_draw(key, idx); }

extern "C" void synth_fill_host(uint16_t* dst, uint64_t n_streams, uint64_t per_stream,
                                uint64_t seed, uint32_t kind, uint32_t layer0, uint32_t expert0,
                                int vary_layer, double sigma) {
  const float scale = synth_scale(sigma);
  for (uint64_t j = 0; j < n_streams; ++j) {
    const uint64_t sid = vary_layer ? synth_stream(kind, layer0 + (uint32_t)j, expert0)
                                    : synth_stream(kind, layer0, expert0 + (uint32_t)j);
    const uint64_t key = synth_key(seed, sid);
    for (uint64_t i = 0; i < per_stream; ++i) dst[j * per_stream + i] = synth_bf16(key, i, scale);
  }
}
