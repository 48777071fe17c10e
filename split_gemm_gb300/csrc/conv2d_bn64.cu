// Kernel instantiations for 64-channel output tiles (all three loaders).
#include "conv2d_kernel.cuh"

namespace sgb {
SGB_INSTANTIATE_CONV2D(64)
SGB_INSTANTIATE_CONV2D_BOX256(64)
}  // namespace sgb
