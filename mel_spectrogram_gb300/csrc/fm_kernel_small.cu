// n_fft = 64, 128, 256: M = 32 = 4 x 8, 64 = 8 x 8, 128 = 8 x 16
#include "fm_kernel.cuh"
FM_DEFINE_VARIANT(kVariant64, 64, 4, 8, 32, 2)
FM_DEFINE_VARIANT(kVariant128, 128, 8, 8, 32, 2)
FM_DEFINE_VARIANT(kVariant256, 256, 8, 16, 32, 2)
