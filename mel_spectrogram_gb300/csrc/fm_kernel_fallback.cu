// One frame per thread, even hops, for n_fft = 64, 128, 256 and 400: the
// packed two-frame kernel keeps one exchange buffer and one staged tile per
// tile group, three groups per CTA, so long hops (n_fft 400 from hop 190 on,
// torchaudio's default hop 200 among them) leave it no shared memory; these
// stage 32 frames in two buffers and take hops up to about 600-850.
#include "fm_kernel.cuh"
FM_DEFINE_VARIANT(kVariant64one, 64, 4, 8, 32, 2)
FM_DEFINE_VARIANT(kVariant128one, 128, 8, 8, 32, 2)
FM_DEFINE_VARIANT(kVariant256one, 256, 8, 16, 32, 2)
FM_DEFINE_VARIANT(kVariant400one, 400, 10, 20, 32, 2)
