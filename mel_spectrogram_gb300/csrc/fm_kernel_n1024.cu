// n_fft = 1024: M = 512 = 16 x 32; one input buffer, so that two CTAs share an SM
// (107 KB of shared memory each instead of 127 KB)
#include "fm_kernel.cuh"
FM_DEFINE_VARIANT(kVariant1024, 1024, 16, 32, 16, 1)
