// Hop-specialised builds of the packed two-frame kernel at n_fft 400 (the
// hop a compile-time constant: tiles staged in lines of two hops, tile
// offsets folded into the pass-1 loads): hop 100 (n_fft / 4, three groups)
// and torchaudio's default hop 200 (two groups, as the any-hop build at that
// hop). On GB300: 400 / 100 on the size sweep (B = 32 x 160000, 128 mels)
// 25.4 against 27.2 us per launch for the any-hop build; 400 / 200 on the
// speech batch (B = 8 x 480000) 13.7 against 14.0 us.
#include "fm_kernel_x2.cuh"
FM_DEFINE_VARIANT_X2(kVariant400h100, 400, 10, 20, 3, 100)
FM_DEFINE_VARIANT_X2(kVariant400h200, 400, 10, 20, 2, 200)
