// n_fft = 4096 (M = 2048 = 16 x 16 x 8), 8192 (16 x 16 x 16) and 16384
// (16 x 16 x 32): three autosorting shared-memory passes per tile. At 4096
// and 8192 the CTA runs two tile groups of 256 threads (four and two frames
// a tile), whose barriers and phases do not wait on each other: on the size
// sweep (B = 32 x 160000, hop n_fft/4, 128 mels) 66.9 and 71.6 us per launch
// against 75.7 and 82.8 us for one group of 512; at 16384 one group (two
// groups of one-frame tiles measured 88.6 against 86.8 us, and 290.6 against
// 287.6 us on 16 x 30 s at 44.1 kHz with 256 mels).
#include "fm_kernel_big.cuh"
FM_DEFINE_VARIANT_BIG(kVariant4096, 4096, 2)
FM_DEFINE_VARIANT_BIG(kVariant8192, 8192, 2)
FM_DEFINE_VARIANT_BIG(kVariant16384, 16384, 1)
