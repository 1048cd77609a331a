// Kernel instantiation: hidden 2048, 32 q / 4 kv heads of 128, 128 experts
// top-8, expert intermediate 768, 64-token pages.
#include "mk_launch.cuh"
namespace mk {
int launch_full(const Params& p, int grid, cudaStream_t s) {
  return launch_shape<dev::Shape<2048, 32, 4, 128, 128, 8, 768, 64>>(p, grid, s);
}
}  // namespace mk
