// Hop-specialised builds of the packed two-frame kernel at hop n_fft / 4 for
// n_fft 128, 256 and 512 (the group counts of their any-hop builds). On the
// size sweep (B = 32 x 160000, 128 mels, GB300): 35.3, 27.3 and 35.0 us per
// launch against 37.7, 27.9 and 36.2 us for the any-hop builds. (At n_fft 64
// the hop-16 build measured slower, 59.8 against 53.5 us, and is not kept.)
#include "fm_kernel_x2.cuh"
FM_DEFINE_VARIANT_X2(kVariant128h32, 128, 8, 8, 1, 32)
FM_DEFINE_VARIANT_X2(kVariant256h64, 256, 8, 16, 3, 64)
FM_DEFINE_VARIANT_X2(kVariant512h128, 512, 16, 16, 2, 128)
