// Kernel instantiations for 128-channel output tiles (all three loaders).
#include "conv2d_kernel.cuh"

namespace sgb {
SGB_INSTANTIATE_CONV2D(128)
SGB_INSTANTIATE_CONV2D_BOX256(128)
}  // namespace sgb
