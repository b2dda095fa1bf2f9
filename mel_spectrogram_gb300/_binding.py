"""ctypes binding of libfm_mel.so (include/fm_mel.h), same names as the C ABI.

Argument marshalling only: every step of the mel path runs in the library's
CUDA kernel. torch is used for device memory and the current stream. If the
library has not been built this module raises; there is no fallback.
"""
from __future__ import annotations

import contextlib
import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfm_mel.so")
# the debug build: the same kernels with an index check on every guarded
# access (-DFM_BOUNDS_CHECK), built beside the release library
CHECK_LIB_PATH = os.path.join(_HERE, "libfm_mel_check.so")

FM_OK, FM_ERR_INVALID_ARG, FM_ERR_UNSUPPORTED, FM_ERR_CUDA, FM_ERR_OOM, FM_ERR_KERNEL_TIMEOUT, FM_ERR_BOUNDS = range(7)
FM_MEL_HTK, FM_MEL_SLANEY = 0, 1
FM_NORM_NONE, FM_NORM_SLANEY = 0, 1
FM_F32, FM_I16, FM_F16 = 0, 1, 2
FM_PAD_REFLECT, FM_PAD_CONSTANT, FM_PAD_REPLICATE, FM_PAD_CIRCULAR = 0, 1, 2, 3
FM_NORMALIZED_NONE, FM_NORMALIZED_WINDOW, FM_NORMALIZED_FRAME_LENGTH = 0, 1, 2

# every symbol include/fm_mel.h declares
EXPORTS = [
    "fm_plan_create",
    "fm_plan_create_ex",
    "fm_plan_destroy",
    "fm_n_frames",
    "fm_mel_forward",
    "fm_mel_forward_host",
    "fm_mel_forward_host_noalloc",
    "fm_mel_filterbank_csr",
    "fm_plan_get_info",
    "fm_plan_poll_error",
    "fm_status_string",
    "fm_selftest_wait_timeout",
]


class FmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class fm_plan_info(C.Structure):
    _fields_ = [
        ("n_fft", C.c_int), ("hop", C.c_int), ("win_length", C.c_int), ("n_mels", C.c_int), ("n_freqs", C.c_int),
        ("in_dtype", C.c_int), ("out_dtype", C.c_int), ("nnz", C.c_int64), ("frames_per_tile", C.c_int),
        ("threads_per_block", C.c_int), ("blocks_per_sm", C.c_int), ("grid_limit", C.c_int),
        ("smem_bytes", C.c_int), ("device", C.c_int),
        ("center", C.c_int), ("pad_mode", C.c_int), ("pad", C.c_int), ("normalized", C.c_int),
    ]


class fm_plan_params(C.Structure):
    _fields_ = [
        ("sr", C.c_int), ("n_fft", C.c_int), ("hop", C.c_int), ("win_length", C.c_int), ("n_mels", C.c_int),
        ("f_min", C.c_double), ("f_max", C.c_double), ("power", C.c_double),
        ("mel_scale", C.c_int), ("norm", C.c_int), ("in_dtype", C.c_int), ("out_dtype", C.c_int),
        ("center", C.c_int), ("pad_mode", C.c_int), ("pad", C.c_int), ("normalized", C.c_int),
    ]


_lib = None
_loaded: dict[str, C.CDLL] = {}


def lib() -> C.CDLL:
    """Load libfm_mel.so (built by mel_spectrogram_gb300.build); raise if absent."""
    global _lib
    if _lib is None:
        _lib = load(LIB_PATH)
    return _lib


@contextlib.contextmanager
def library(path: str):
    """Route every call of this module through the library at `path` (e.g.
    CHECK_LIB_PATH, the debug build) inside the block. Plans are bound to
    the library that created them: create and destroy them inside one block."""
    global _lib
    prev = _lib
    _lib = load(path)
    try:
        yield _lib
    finally:
        _lib = prev


def load(path: str) -> C.CDLL:
    """Load one build of the library with its prototypes declared (cached)."""
    if path in _loaded:
        return _loaded[path]
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -m mel_spectrogram_gb300.build` "
            "(the mel path has no CPU fallback)"
        )
    L = C.CDLL(path)
    vp, i64, ci, cd = C.c_void_p, C.c_int64, C.c_int, C.c_double
    L.fm_plan_create.argtypes = [C.POINTER(vp), ci, ci, ci, ci, ci, cd, cd, cd, ci, ci, ci, ci]
    L.fm_plan_create.restype = ci
    L.fm_plan_create_ex.argtypes = [C.POINTER(vp), C.POINTER(fm_plan_params)]
    L.fm_plan_create_ex.restype = ci
    L.fm_plan_destroy.argtypes = [vp]
    L.fm_plan_destroy.restype = ci
    L.fm_n_frames.argtypes = [vp, i64]
    L.fm_n_frames.restype = i64
    L.fm_mel_forward.argtypes = [vp, vp, i64, i64, vp, vp]
    L.fm_mel_forward.restype = ci
    L.fm_mel_forward_host.argtypes = [vp, vp, i64, i64, vp, vp, vp, vp]
    L.fm_mel_forward_host.restype = ci
    L.fm_mel_forward_host_noalloc.argtypes = [vp, vp, i64, i64, vp, vp]
    L.fm_mel_forward_host_noalloc.restype = ci
    L.fm_mel_filterbank_csr.argtypes = [ci, ci, ci, cd, cd, ci, ci, vp, vp, vp, vp, C.POINTER(i64)]
    L.fm_mel_filterbank_csr.restype = ci
    L.fm_plan_get_info.argtypes = [vp, C.POINTER(fm_plan_info)]
    L.fm_plan_get_info.restype = ci
    L.fm_plan_poll_error.argtypes = [vp]
    L.fm_plan_poll_error.restype = ci
    L.fm_status_string.argtypes = [ci]
    L.fm_status_string.restype = C.c_char_p
    L.fm_selftest_wait_timeout.argtypes = [vp, ci, ci, vp, C.POINTER(ci), C.POINTER(cd)]
    L.fm_selftest_wait_timeout.restype = ci
    _loaded[path] = L
    return L


def status_string(status: int) -> str:
    return lib().fm_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != FM_OK:
        raise FmError(status, what)


_SCALES = {"htk": FM_MEL_HTK, "slaney": FM_MEL_SLANEY}
_NORMS = {None: FM_NORM_NONE, "none": FM_NORM_NONE, "slaney": FM_NORM_SLANEY}
_DTYPES = {"f32": FM_F32, "i16": FM_I16, "f16": FM_F16}
_PAD_MODES = {"reflect": FM_PAD_REFLECT, "constant": FM_PAD_CONSTANT, "replicate": FM_PAD_REPLICATE,
              "circular": FM_PAD_CIRCULAR}
_NORMALIZED = {False: FM_NORMALIZED_NONE, None: FM_NORMALIZED_NONE, "none": FM_NORMALIZED_NONE,
               True: FM_NORMALIZED_WINDOW, "window": FM_NORMALIZED_WINDOW,
               "frame_length": FM_NORMALIZED_FRAME_LENGTH}


def fm_plan_create(sr, n_fft, hop, win_length, n_mels, f_min, f_max, power, mel_scale="htk", norm=None,
                   in_dtype="f32", out_dtype="f32") -> int:
    """Create a plan on the current CUDA device; returns the opaque handle."""
    h = C.c_void_p()
    st = lib().fm_plan_create(
        C.byref(h), int(sr), int(n_fft), int(hop), int(win_length or 0), int(n_mels), float(f_min),
        float(f_max if f_max is not None else 0.0), float(power), _SCALES.get(mel_scale, mel_scale),
        _NORMS.get(norm, norm), _DTYPES.get(in_dtype, in_dtype), _DTYPES.get(out_dtype, out_dtype),
    )
    _check(st, "fm_plan_create")
    return h.value


def fm_plan_create_ex(sr, n_fft, hop, win_length, n_mels, f_min, f_max, power, mel_scale="htk", norm=None,
                      in_dtype="f32", out_dtype="f32", center=True, pad_mode="reflect", pad=0,
                      normalized=False) -> int:
    """fm_plan_create with torchaudio's framing options (center, pad_mode,
    pad, normalized as False / True / "window" / "frame_length")."""
    p = fm_plan_params(
        int(sr), int(n_fft), int(hop), int(win_length or 0), int(n_mels), float(f_min),
        float(f_max if f_max is not None else 0.0), float(power), _SCALES.get(mel_scale, mel_scale),
        _NORMS.get(norm, norm), _DTYPES.get(in_dtype, in_dtype), _DTYPES.get(out_dtype, out_dtype),
        1 if center else 0, _PAD_MODES.get(pad_mode, pad_mode), int(pad),
        _NORMALIZED[normalized] if isinstance(normalized, (bool, str, type(None))) else int(normalized),
    )
    h = C.c_void_p()
    _check(lib().fm_plan_create_ex(C.byref(h), C.byref(p)), "fm_plan_create_ex")
    return h.value


def fm_plan_destroy(plan) -> None:
    _check(lib().fm_plan_destroy(plan), "fm_plan_destroy")


def fm_n_frames(plan, T: int) -> int:
    return int(lib().fm_n_frames(plan, int(T)))


def fm_mel_forward(plan, d_in: int, B: int, T: int, d_out: int, stream: int = 0) -> None:
    """Raw-pointer launch (device pointers as ints, stream as a cudaStream_t int)."""
    _check(lib().fm_mel_forward(plan, d_in, int(B), int(T), d_out, stream or None), "fm_mel_forward")


def fm_mel_forward_host(plan, h_in: int, B: int, T: int, h_out: int, d_in: int, d_out: int, stream: int = 0):
    _check(lib().fm_mel_forward_host(plan, h_in, int(B), int(T), h_out, d_in, d_out, stream or None),
           "fm_mel_forward_host")


# size of the device staging array of fm_mel_forward_host_noalloc (FM_NOALLOC_MAX_BYTES)
FM_NOALLOC_MAX_BYTES = 32 << 20


def fm_selftest_wait_timeout(plan, kind: int, log2_polls: int, stream: int = 0) -> tuple[int, float]:
    """Run out one of the kernels' bounded waits on purpose (diagnostic).

    kind 0: a tile group's wait for its staged tile; kind 1: the producer
    warp's wait for a free staging area. Returns (groups that passed their
    wait, kernel microseconds); the timeout itself is then reported by
    fm_plan_poll_error.
    """
    done, us = C.c_int(0), C.c_double(0.0)
    _check(lib().fm_selftest_wait_timeout(plan, int(kind), int(log2_polls), stream or None, C.byref(done),
                                          C.byref(us)), "fm_selftest_wait_timeout")
    return done.value, us.value


def fm_mel_forward_host_noalloc(plan, h_in: int, B: int, T: int, h_out: int, stream: int = 0) -> None:
    """Host buffers in and out, device staging in the library's static array.

    For callers that cannot allocate device memory at call time (a real-time
    audio callback, or a process whose device memory belongs to another
    allocator). The input bytes (rounded up to 256) plus the output bytes must
    fit in FM_NOALLOC_MAX_BYTES; calls that overlap on the GPU share the array
    and race, so queue them on one stream.
    """
    st = lib().fm_mel_forward_host_noalloc(plan, h_in, int(B), int(T), h_out, stream or None)
    if st == FM_ERR_INVALID_ARG:
        raise FmError(st, "fm_mel_forward_host_noalloc (a NULL buffer, T <= n_fft/2, or input + output beyond "
                          f"the {FM_NOALLOC_MAX_BYTES}-byte staging array)")
    _check(st, "fm_mel_forward_host_noalloc")


def fm_plan_get_info(plan) -> dict:
    info = fm_plan_info()
    _check(lib().fm_plan_get_info(plan, C.byref(info)), "fm_plan_get_info")
    return {name: getattr(info, name) for name, _ in info._fields_}


def fm_plan_poll_error(plan) -> int:
    return int(lib().fm_plan_poll_error(plan))


def fm_mel_filterbank_csr(sr, n_fft, n_mels, f_min, f_max, mel_scale="htk", norm=None):
    """Host-only filterbank CSR -> (start, len, off, weights) numpy arrays."""
    import numpy as np

    L = lib()
    nnz = C.c_int64(0)
    args = (int(sr), int(n_fft), int(n_mels), float(f_min), float(f_max if f_max is not None else 0.0),
            _SCALES.get(mel_scale, mel_scale), _NORMS.get(norm, norm))
    _check(L.fm_mel_filterbank_csr(*args, None, None, None, None, C.byref(nnz)), "fm_mel_filterbank_csr")
    start = np.zeros(n_mels, np.int32)
    ln = np.zeros(n_mels, np.int32)
    off = np.zeros(n_mels + 1, np.int32)
    w = np.zeros(max(1, nnz.value), np.float32)
    _check(L.fm_mel_filterbank_csr(*args, start.ctypes.data, ln.ctypes.data, off.ctypes.data, w.ctypes.data,
                                   C.byref(nnz)), "fm_mel_filterbank_csr")
    return start, ln, off, w[: nnz.value]
