// n_fft = 256 and 512 for long even hops: the packed two-frame kernel with
// fewer tile groups per CTA (256: two, then one; 512: one), which leaves room
// for longer staged tiles; past that, 512 takes the one-frame kernel.
#include "fm_kernel_x2.cuh"
FM_DEFINE_VARIANT_X2(kVariant256g2, 256, 8, 16, 2, 0)
FM_DEFINE_VARIANT_X2(kVariant256g1, 256, 8, 16, 1, 0)
FM_DEFINE_VARIANT_X2(kVariant512g1, 512, 16, 16, 1, 0)
