// Kernel instantiations for 256-channel output tiles (all three loaders).
#include "conv2d_kernel.cuh"

namespace sgb {
SGB_INSTANTIATE_CONV2D(256)
}  // namespace sgb
