"""Batched mel spectrogram for GB300 (sm_103a): C ABI + thin Python binding.

The compute path is one hand-written CUDA kernel in ``libfm_mel.so``
(``mel_spectrogram_gb300/csrc``); this package only marshals arguments. Build
the library with ``python -m mel_spectrogram_gb300.build``.
"""
from ._binding import (  # noqa: F401
    EXPORTS,
    FM_ERR_CUDA,
    FM_ERR_INVALID_ARG,
    FM_ERR_KERNEL_TIMEOUT,
    FM_ERR_OOM,
    FM_ERR_UNSUPPORTED,
    FM_OK,
    FmError,
    fm_mel_filterbank_csr,
    fm_mel_forward,
    fm_mel_forward_host,
    fm_mel_forward_host_noalloc,
    fm_n_frames,
    fm_plan_create,
    fm_plan_create_ex,
    fm_plan_destroy,
    fm_plan_get_info,
    fm_plan_poll_error,
    fm_selftest_wait_timeout,
    lib,
    status_string,
)
from .transform import MelSpectrogram  # noqa: F401
