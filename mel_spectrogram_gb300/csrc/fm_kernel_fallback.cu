// One frame per thread, even hops, for n_fft = 256 and 400: the packed
// two-frame kernel at these sizes keeps three tile groups per CTA, each with
// an exchange buffer and a staged tile, so long hops (n_fft 400 from hop 190
// on, torchaudio's default hop 200 among them) leave it no shared memory;
// these stage 32 frames in two buffers and take hops up to about 650-750.
// (At 64 and 128 the packed kernel runs one group per CTA and takes longer
// hops than this kernel would.)
#include "fm_kernel.cuh"
FM_DEFINE_VARIANT(kVariant256one, 256, 8, 16, 32, 2)
FM_DEFINE_VARIANT(kVariant400one, 400, 10, 20, 32, 2)
