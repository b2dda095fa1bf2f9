// n_fft = 1024: M = 512 = 16 x 32
#include "fm_kernel.cuh"
FM_DEFINE_VARIANT(kVariant1024, 1024, 16, 32, 16, 2)
