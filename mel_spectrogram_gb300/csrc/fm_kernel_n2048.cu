// n_fft = 2048: M = 1024 = 32 x 32, 16 frames per tile (the exchange buffer must fit shared memory)
#include "fm_kernel.cuh"
FM_DEFINE_VARIANT(kVariant2048, 2048, 32, 32, 16, 1)
