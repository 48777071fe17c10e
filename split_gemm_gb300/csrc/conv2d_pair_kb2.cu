// CTA-pair kernel instantiations with 2 k-blocks per pipeline stage.
#define SGB_PAIR_KBS 2
#include "conv2d_pair_inst.cuh"
