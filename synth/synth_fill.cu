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

// FP8 expert weights: 16 consecutive E4M3 codes per thread, one 16-byte store
// (per_stream % 16 == 0, dst 16-byte aligned).
__global__ void fill_fp8_vec16(uint8_t* __restrict__ dst, uint64_t n_streams, uint64_t per_stream,
                               uint64_t seed, uint32_t kind, uint32_t layer0, uint32_t expert0,
                               int vary_layer) {
  const uint64_t groups_per_stream = per_stream / 16;
  const uint64_t total = n_streams * groups_per_stream;
  for (uint64_t g = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t j = g / groups_per_stream;
    const uint64_t i0 = (g - j * groups_per_stream) * 16;
    const uint64_t key = synth_key(seed, stream_of(kind, layer0, expert0, vary_layer, j));
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      w[q] = 0u;
#pragma unroll
      for (int b = 0; b < 4; ++b) w[q] |= (uint32_t)synth_fp8(key, i0 + 4 * q + b) << (8 * b);
    }
    *reinterpret_cast<uint4*>(dst + j * per_stream + i0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Row scales of FP8 expert matrices: element r of sub-stream j.
__global__ void fill_row_scales(float* __restrict__ dst, uint64_t n_streams, uint64_t rows, uint64_t seed,
                                uint32_t kind, uint32_t layer0, uint32_t expert0, int vary_layer, float base) {
  const uint64_t total = n_streams * rows;
  for (uint64_t g = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t j = g / rows, r = g - j * rows;
    const uint64_t key = synth_key(seed, stream_of(kind, layer0, expert0, vary_layer, j));
    dst[g] = synth_row_scale(key, r, base);
  }
}

// FP4 expert weights: 16 bytes (32 E2M1 codes) per thread, one 16-byte store
// (per_stream bytes % 16 == 0, dst 16-byte aligned).
__global__ void fill_fp4_vec16(uint8_t* __restrict__ dst, uint64_t n_streams, uint64_t per_stream,
                               uint64_t seed, uint32_t kind, uint32_t layer0, uint32_t expert0,
                               int vary_layer) {
  const uint64_t groups_per_stream = per_stream / 16;
  const uint64_t total = n_streams * groups_per_stream;
  for (uint64_t g = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t j = g / groups_per_stream;
    const uint64_t i0 = (g - j * groups_per_stream) * 16;
    const uint64_t key = synth_key(seed, stream_of(kind, layer0, expert0, vary_layer, j));
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      w[q] = 0u;
#pragma unroll
      for (int b = 0; b < 4; ++b) w[q] |= (uint32_t)synth_fp4_byte(key, i0 + 4 * q + b) << (8 * b);
    }
    *reinterpret_cast<uint4*>(dst + j * per_stream + i0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Block scales (E4M3 bytes) of FP4 expert matrices: block b of sub-stream j.
__global__ void fill_block_scales(uint8_t* __restrict__ dst, uint64_t n_streams, uint64_t per_stream, uint64_t seed,
                                  uint32_t kind, uint32_t layer0, uint32_t expert0, int vary_layer) {
  const uint64_t total = n_streams * per_stream;
  for (uint64_t g = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t j = g / per_stream, b = g - j * per_stream;
    const uint64_t key = synth_key(seed, stream_of(kind, layer0, expert0, vary_layer, j));
    dst[g] = synth_fp4_bscale(key, b);
  }
}

// RMSNorm gains: element i of sub-stream j (layer layer0 + j).
__global__ void fill_gains(float* __restrict__ dst, uint64_t n_streams, uint64_t per_stream, uint64_t seed,
                           uint32_t layer0) {
  const uint64_t total = n_streams * per_stream;
  for (uint64_t g = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t j = g / per_stream, i = g - j * per_stream;
    const uint64_t key = synth_key(seed, synth_stream(SYNTH_GAMMA, layer0 + (uint32_t)j, 0));
    dst[g] = synth_gain(key, i);
  }
}

int launch_blocks() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return (sms > 0 ? sms : 1) * 8;
}

}  // namespace

// FP8 expert weights (E4M3 codes) on the device: element i of sub-stream j
// goes to dst[j*per_stream+i]; per_stream % 16 == 0 and dst 16-byte aligned.
extern "C" int synth_fill_fp8_device(void* dst, uint64_t n_streams, uint64_t per_stream, uint64_t seed,
                                     uint32_t kind, uint32_t layer0, uint32_t expert0, int vary_layer,
                                     void* stream) {
  if (dst == nullptr || n_streams == 0 || per_stream == 0 || per_stream % 16 != 0 ||
      (reinterpret_cast<uintptr_t>(dst) & 15u) != 0)
    return (int)cudaErrorInvalidValue;
  fill_fp8_vec16<<<launch_blocks(), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t*>(dst), n_streams, per_stream, seed, kind, layer0, expert0, vary_layer);
  return (int)cudaGetLastError();
}

// Row scales (binary32) on the device: `rows` per sub-stream.
extern "C" int synth_fill_scales_device(float* dst, uint64_t n_streams, uint64_t rows, uint64_t seed,
                                        uint32_t kind, uint32_t layer0, uint32_t expert0, int vary_layer,
                                        double sigma, void* stream) {
  if (dst == nullptr || n_streams == 0 || rows == 0) return (int)cudaErrorInvalidValue;
  fill_row_scales<<<launch_blocks(), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      dst, n_streams, rows, seed, kind, layer0, expert0, vary_layer, synth_fp8_base(sigma));
  return (int)cudaGetLastError();
}

// FP4 expert weights on the device: byte i of sub-stream j goes to
// dst[j*per_stream+i]; per_stream % 16 == 0 and dst 16-byte aligned.
extern "C" int synth_fill_fp4_device(void* dst, uint64_t n_streams, uint64_t per_stream, uint64_t seed,
                                     uint32_t kind, uint32_t layer0, uint32_t expert0, int vary_layer,
                                     void* stream) {
  if (dst == nullptr || n_streams == 0 || per_stream == 0 || per_stream % 16 != 0 ||
      (reinterpret_cast<uintptr_t>(dst) & 15u) != 0)
    return (int)cudaErrorInvalidValue;
  fill_fp4_vec16<<<launch_blocks(), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t*>(dst), n_streams, per_stream, seed, kind, layer0, expert0, vary_layer);
  return (int)cudaGetLastError();
}

// FP4 block scales on the device: `per_stream` blocks per sub-stream.
extern "C" int synth_fill_bscales_device(void* dst, uint64_t n_streams, uint64_t per_stream, uint64_t seed,
                                         uint32_t kind, uint32_t layer0, uint32_t expert0, int vary_layer,
                                         void* stream) {
  if (dst == nullptr || n_streams == 0 || per_stream == 0) return (int)cudaErrorInvalidValue;
  fill_block_scales<<<launch_blocks(), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t*>(dst), n_streams, per_stream, seed, kind, layer0, expert0, vary_layer);
  return (int)cudaGetLastError();
}

// Row scales with an explicit base (FP4 matrices use synth_fp4_base).
extern "C" int synth_fill_scales_base_device(float* dst, uint64_t n_streams, uint64_t rows, uint64_t seed,
                                             uint32_t kind, uint32_t layer0, uint32_t expert0, int vary_layer,
                                             float base, void* stream) {
  if (dst == nullptr || n_streams == 0 || rows == 0) return (int)cudaErrorInvalidValue;
  fill_row_scales<<<launch_blocks(), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      dst, n_streams, rows, seed, kind, layer0, expert0, vary_layer, base);
  return (int)cudaGetLastError();
}

extern "C" void synth_fill_fp4_host(uint8_t* dst, uint64_t n_bytes, uint64_t seed, uint32_t kind, uint32_t layer,
                                    uint32_t expert) {
  const uint64_t key = synth_key(seed, synth_stream(kind, layer, expert));
  for (uint64_t j = 0; j < n_bytes; ++j) dst[j] = synth_fp4_byte(key, j);
}

extern "C" void synth_fill_bscales_host(uint8_t* dst, uint64_t n, uint64_t seed, uint32_t kind, uint32_t layer,
                                        uint32_t expert) {
  const uint64_t key = synth_key(seed, synth_stream(kind, layer, expert));
  for (uint64_t b = 0; b < n; ++b) dst[b] = synth_fp4_bscale(key, b);
}

extern "C" void synth_fill_scales_base_host(float* dst, uint64_t rows, uint64_t seed, uint32_t kind, uint32_t layer,
                                            uint32_t expert, float base) {
  const uint64_t key = synth_key(seed, synth_stream(kind, layer, expert));
  for (uint64_t r = 0; r < rows; ++r) dst[r] = synth_row_scale(key, r, base);
}

extern "C" float synth_fp4_base_of(double sigma) { return synth_fp4_base(sigma); }

// RMSNorm gains on the device: `per_stream` gains of layers layer0 .. layer0 + n_streams - 1.
extern "C" int synth_fill_gains_device(float* dst, uint64_t n_streams, uint64_t per_stream, uint64_t seed,
                                       uint32_t layer0, void* stream) {
  if (dst == nullptr || n_streams == 0 || per_stream == 0) return (int)cudaErrorInvalidValue;
  fill_gains<<<launch_blocks(), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(dst, n_streams, per_stream,
                                                                                  seed, layer0);
  return (int)cudaGetLastError();
}

extern "C" void synth_fill_gains_host(float* dst, uint64_t n_streams, uint64_t per_stream, uint64_t seed,
                                      uint32_t layer0) {
  for (uint64_t j = 0; j < n_streams; ++j) {
    const uint64_t key = synth_key(seed, synth_stream(SYNTH_GAMMA, layer0 + (uint32_t)j, 0));
    for (uint64_t i = 0; i < per_stream; ++i) dst[j * per_stream + i] = synth_gain(key, i);
  }
}
extern "C" uint8_t synth_e2m1(float f) { return synth_f32_to_e2m1_rne(f); }

extern "C" void synth_fill_fp8_host(uint8_t* dst, uint64_t n, uint64_t seed, uint32_t kind, uint32_t layer,
                                    uint32_t expert) {
  const uint64_t key = synth_key(seed, synth_stream(kind, layer, expert));
  for (uint64_t i = 0; i < n; ++i) dst[i] = synth_fp8(key, i);
}

extern "C" void synth_fill_scales_host(float* dst, uint64_t rows, uint64_t seed, uint32_t kind, uint32_t layer,
                                       uint32_t expert, double sigma) {
  const uint64_t key = synth_key(seed, synth_stream(kind, layer, expert));
  const float base = synth_fp8_base(sigma);
  for (uint64_t r = 0; r < rows; ++r) dst[r] = synth_row_scale(key, r, base);
}

extern "C" uint8_t synth_e4m3(float f) { return synth_f32_to_e4m3_rne(f); }

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
