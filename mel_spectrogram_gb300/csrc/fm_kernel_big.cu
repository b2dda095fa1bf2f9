// n_fft = 4096 (M = 2048 = 16 x 16 x 8), 8192 (16 x 16 x 16) and 16384
// (16 x 16 x 32): three autosorting shared-memory passes per tile
#include "fm_kernel_big.cuh"
FM_DEFINE_VARIANT_BIG(kVariant4096, 4096)
FM_DEFINE_VARIANT_BIG(kVariant8192, 8192)
FM_DEFINE_VARIANT_BIG(kVariant16384, 16384)
