// Odd hops (one frame per thread, contiguous staging): n_fft = 2048 (M = 32 x 32)
#include "fm_kernel.cuh"
FM_DEFINE_VARIANT_ODD(kVariant2048odd, 2048, 32, 32, 16, 1)
