// Kernel instantiation: a dense SwiGLU model -- hidden 1024, 16 q / 2 kv
// heads of 64, one expert taken by every token (the FFN), intermediate 2048,
// 64-token pages.
#include "mk_launch.cuh"
namespace mk {
int launch_dense(const Params& p, int grid, cudaStream_t s) {
  return launch_shape<dev::Shape<1024, 16, 2, 64, 1, 1, 2048, 64>>(p, grid, s);
}
}  // namespace mk
