// Odd hops (one frame per thread, contiguous staging): n_fft = 512 (M = 16 x 16)
// and 1024 (16 x 32), tiles and buffers as for even hops
#include "fm_kernel.cuh"
FM_DEFINE_VARIANT_ODD(kVariant512odd, 512, 16, 16, 16, 2)
FM_DEFINE_VARIANT_ODD(kVariant1024odd, 1024, 16, 32, 16, 1)
