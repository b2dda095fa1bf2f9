// n_fft = 400: M = 200 = 10 x 20 (pass 1: 20-point DFTs; pass 2: 10-point DFTs)
#include "fm_kernel.cuh"
FM_DEFINE_VARIANT(kVariant400, 400, 10, 20, 16, 2)
