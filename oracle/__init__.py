"""Float64 CPU oracle for the mel spectrogram (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package. The product path never does.
"""
from .mel_oracle import (  # noqa: F401
    bin_frequencies,
    dft_onesided,
    filter_vertices,
    frame,
    hann_periodic,
    hz_to_mel,
    mel_filterbank,
    mel_spectrogram,
    mel_to_hz,
    n_frames,
    power_spectrogram,
    reflect_pad,
    spectral_power,
    to_float64,
)
