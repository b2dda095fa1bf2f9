// n_fft = 512: M = 256 = 16 x 16. Two frames per thread, packed, with two tile
// groups per CTA (three groups of 256 threads would leave 80 registers a
// thread); one frame per thread for hops whose staged tiles leave the packed
// kernel no room. Measured on the size sweep (B = 32 x 160000, hop 128): 36.1
// us per launch against 40.4 us for the one-frame kernel and 42.4 us for one
// packed group per CTA (136 registers, one CTA per SM)
#include "fm_kernel_x2.cuh"
FM_DEFINE_VARIANT_X2(kVariant512x2, 512, 16, 16, 2, 0)
FM_DEFINE_VARIANT(kVariant512, 512, 16, 16, 16, 2)
