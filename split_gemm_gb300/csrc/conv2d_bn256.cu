// Kernel instantiations of the one-CTA kernel for 256-channel output tiles (every loader kind, plain and fused epilogue).
#include "conv2d_kernel.cuh"

namespace sgb {
SGB_INSTANTIATE_CONV2D(256)
}  // namespace sgb
