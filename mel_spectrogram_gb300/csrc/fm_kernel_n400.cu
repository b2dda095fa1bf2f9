// n_fft = 400: M = 200 = 10 x 20 (pass 1: 20-point DFTs; pass 2: 10-point DFTs),
// two frames per thread with packed f32x2 arithmetic
#include "fm_kernel_x2.cuh"
FM_DEFINE_VARIANT_X2(kVariant400, 400, 10, 20)
