// Instantiations of the row-window kernel (few input channels) for every tile width.
#include "conv2d_rowwin.cuh"

namespace sgb {
template SGB_ROWWIN_SIG(64);
template SGB_ROWWIN_SIG(128);
template SGB_ROWWIN_SIG(256);
}  // namespace sgb
