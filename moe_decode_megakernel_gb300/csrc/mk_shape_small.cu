// Kernel instantiation: hidden 1024, 16 q / 2 kv heads of 64, 32 experts
// top-4, expert intermediate 512, 64-token pages.
#include "mk_launch.cuh"
namespace mk {
int launch_small(const Params& p, int grid, cudaStream_t s) {
  return launch_shape<dev::Shape<1024, 16, 2, 64, 32, 4, 512, 64>>(p, grid, s);
}
}  // namespace mk
