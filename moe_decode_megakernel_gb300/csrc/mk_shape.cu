// One instantiation of the persistent kernel: the build compiles this file
// once per compiled shape and kernel mode, defining
//   MK_DIM0 .. MK_DIM7  hidden, n_q, n_kv, head_dim, n_experts, top_k, inter, page_size
//   MK_MODE        a KernelMode
//   MK_LAUNCH_FN   the name of the launch function (declared in mk_api.cpp).
#include "mk_launch.cuh"

#if !defined(MK_DIM7) || !defined(MK_MODE) || !defined(MK_LAUNCH_FN)
#error "mk_shape.cu is compiled with MK_DIM0..MK_DIM7, MK_MODE and MK_LAUNCH_FN defined"
#endif

namespace mk {
int MK_LAUNCH_FN(const Params& p, int grid, cudaStream_t s) {
  return launch_shape<dev::Shape<MK_DIM0, MK_DIM1, MK_DIM2, MK_DIM3, MK_DIM4, MK_DIM5, MK_DIM6, MK_DIM7>, MK_MODE>(
      p, grid, s);
}
}  // namespace mk
