// Kernel instantiations of the one-CTA kernel for 64-channel output tiles (every loader kind, plain and fused epilogue).
#include "conv2d_kernel.cuh"

namespace sgb {
SGB_INSTANTIATE_CONV2D(64)
SGB_INSTANTIATE_CONV2D_BOX256(64)
}  // namespace sgb
