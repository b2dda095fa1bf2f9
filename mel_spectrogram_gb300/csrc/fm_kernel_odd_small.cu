// Odd hops (one frame per thread, contiguous staging): n_fft = 64 (M = 4 x 8),
// 128 (8 x 8), 256 (8 x 16) and 400 (10 x 20)
#include "fm_kernel.cuh"
FM_DEFINE_VARIANT_ODD(kVariant64odd, 64, 4, 8, 32, 2)
FM_DEFINE_VARIANT_ODD(kVariant128odd, 128, 8, 8, 32, 2)
FM_DEFINE_VARIANT_ODD(kVariant256odd, 256, 8, 16, 32, 2)
FM_DEFINE_VARIANT_ODD(kVariant400odd, 400, 10, 20, 32, 2)
