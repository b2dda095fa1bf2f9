// n_fft = 400 for long even hops: the packed two-frame kernel with two tile
// groups per CTA (hops up to ~400 with f32 input), then one (up to ~1200).
// Each group keeps its own exchange buffer and staged tile, so fewer groups
// leave room for longer tiles; on the speech batch at torchaudio's default hop
// of 200 two groups took 13.9 us per launch against 17.4 us for the one-frame
// kernel, and 9.5 against 15.8 us at hop 400.
#include "fm_kernel_x2.cuh"
FM_DEFINE_VARIANT_X2(kVariant400g2, 400, 10, 20, 2, 0)
FM_DEFINE_VARIANT_X2(kVariant400g1, 400, 10, 20, 1, 0)
