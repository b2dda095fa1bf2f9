// n_fft = 512: M = 256 = 16 x 16
#include "fm_kernel.cuh"
FM_DEFINE_VARIANT(kVariant512, 512, 16, 16, 16, 2)
