// n_fft = 64 (M = 4 x 8), 128 (M = 8 x 8) and 256 (M = 8 x 16): two frames
// per thread, packed. At 64 and 128 one tile group per CTA, several CTAs per
// SM (five and three), so that each group has a producer warp of its own:
// their tiles are small beside the staging work per tile, and on the size
// sweep (B = 32 x 160000, hop n_fft/4) that measured 52.5 and 37.7 us per
// launch against 63.6 and 41.0 us with three groups sharing one producer in a
// CTA. At 256 three groups per CTA (28.0 us against 31.1 us with one group).
#include "fm_kernel_x2.cuh"
FM_DEFINE_VARIANT_X2(kVariant64, 64, 4, 8, 1, 0)
FM_DEFINE_VARIANT_X2(kVariant128, 128, 8, 8, 1, 0)
FM_DEFINE_VARIANT_X2(kVariant256, 256, 8, 16, 3, 0)
