// n_fft = 400: M = 200 = 10 x 20 (pass 1: 20-point DFTs; pass 2: 10-point DFTs),
// two frames per thread with packed f32x2 arithmetic; a build for hop 160
// (whisper-style framing) with compile-time tile offsets, and one for any hop
#include "fm_kernel_x2.cuh"
FM_DEFINE_VARIANT_X2(kVariant400h160, 400, 10, 20, 3, 160)
FM_DEFINE_VARIANT_X2(kVariant400, 400, 10, 20, 3, 0)
