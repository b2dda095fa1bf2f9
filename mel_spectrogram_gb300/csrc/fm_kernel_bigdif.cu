// n_fft = 4096, 8192 and 16384 as 16 x (128, 256, 512) by decimation in
// frequency: the first 16-point DFTs fused with the load, then one warp per
// sub-frame group (16 x 8, 16 x 16, 16 x 32 in shared memory).
#include "fm_kernel_bigdif.cuh"
FM_DEFINE_VARIANT_BIGDIF(kVariant4096dif, 4096)
FM_DEFINE_VARIANT_BIGDIF(kVariant8192dif, 8192)
FM_DEFINE_VARIANT_BIGDIF(kVariant16384dif, 16384)
