// n_fft = 400, hop 160: the lane-pair variant of the two-frame packed kernel
// (each DFT shared by two lanes, ten warps per tile group)
#include "fm_kernel_x2h.cuh"
FM_DEFINE_VARIANT_X2H(kVariant400h160x2h, 400, 10, 20, 3, 160)
