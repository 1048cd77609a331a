// mk_launch.cuh -- launch of the persistent kernel for one compiled shape.
#pragma once

#include "mk_kernel.cuh"

namespace mk {

// One CTA per SM; a cooperative launch so that every CTA is resident at once
// (CTAs wait on each other's counters, so a CTA left unscheduled would stall
// the step until the watchdog).
template <class S, int M>
int launch_shape(const Params& p, int grid, cudaStream_t stream) {
  const void* fn = reinterpret_cast<const void*>(&dev::mk_persistent<S, M>);
  constexpr size_t smem = dev::smem_bytes<S>();
  static_assert(smem <= dev::kMaxSmemPerCta, "shared memory of one CTA");
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  void* args[] = {const_cast<Params*>(&p)};
  e = cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kThreads), args, smem, stream);
  return (int)e;
}

}  // namespace mk
