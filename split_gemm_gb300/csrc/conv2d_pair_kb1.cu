// CTA-pair kernel instantiations with 1 k-block per pipeline stage.
#define SGB_PAIR_KBS 1
#include "conv2d_pair_inst.cuh"
