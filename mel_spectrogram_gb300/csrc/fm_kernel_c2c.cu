// n_fft = 400 as one 400-point complex transform per frame pair (N = 20 x 20),
// the diagnostic alternative to the two-frame packed kernel
#include "fm_kernel_c2c.cuh"
namespace fm {
template __global__ void mel_kernel_c2c<kC2cN>(const KernelParams);
extern const Variant kVariant400c2c = {kC2cN, kC2cP, kC2cQ, 2 * kC2cPairs, kC2cThreads, 2, 3,
                                       (const void*)&mel_kernel_c2c<kC2cN>, kEvenHops};
}  // namespace fm
