// n_fft = 1024 (M = 512 = 8 x 8 x 8) and 2048 (M = 1024 = 16 x 16 x 4) for
// hops whose staged tiles leave the one-frame kernel no shared memory (f32:
// 1024 from hop ~2250 on, 2048 from ~810, half-overlap hop 1024 among them):
// the large-transform kernel, which reads each tile's frames straight from
// the signal when its span does not fit a staging buffer. Two tile groups of
// 16 and 8 frames.
#include "fm_kernel_big.cuh"
FM_DEFINE_VARIANT_BIG(kVariant1024big, 1024, 2)
FM_DEFINE_VARIANT_BIG(kVariant2048big, 2048, 2)
