// n_fft = 64 (M = 4 x 8), 128 (M = 8 x 8) and 256 (M = 8 x 16): two frames
// per thread, packed, three tile groups per CTA
#include "fm_kernel_x2.cuh"
FM_DEFINE_VARIANT_X2(kVariant64, 64, 4, 8, 3, 0)
FM_DEFINE_VARIANT_X2(kVariant128, 128, 8, 8, 3, 0)
FM_DEFINE_VARIANT_X2(kVariant256, 256, 8, 16, 3, 0)
