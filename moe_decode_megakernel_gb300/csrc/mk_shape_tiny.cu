// Kernel instantiation: hidden 256, 4 q / 2 kv heads of 64, 16 experts top-4,
// expert intermediate 128, 16-token pages.
#include "mk_launch.cuh"
namespace mk {
int launch_tiny(const Params& p, int grid, cudaStream_t s) {
  return launch_shape<dev::Shape<256, 4, 2, 64, 16, 4, 128, 16>>(p, grid, s);
}
}  // namespace mk
