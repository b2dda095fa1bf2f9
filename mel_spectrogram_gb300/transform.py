"""torchaudio-style MelSpectrogram on top of the C ABI.

flashmel README, "Usage": MelSpectrogram(torchaudio arguments, dtype=...)(x)
with x of shape (..., time) on the GPU, float32 or int16 PCM (here also
float16), returning (..., n_mels, n_frames) in float32 or float16, with the
torchaudio arguments pad, center, pad_mode and normalized. The window is
always the periodic Hann (no window_fn), the spectrum one-sided.
"""
from __future__ import annotations

from . import _binding as fb


class MelSpectrogram:
    """Callable mel transform; owns one plan per (device, input dtype)."""

    def __init__(self, sample_rate=16000, n_fft=400, win_length=None, hop_length=None, f_min=0.0, f_max=None,
                 pad=0, n_mels=128, power=2.0, normalized=False, center=True, pad_mode="reflect", onesided=True,
                 norm=None, mel_scale="htk", dtype=None):
        import torch

        if not onesided:
            raise ValueError("onesided=False is not supported (the mel scale takes one-sided spectra)")
        self.pad = int(pad)
        self.normalized = normalized
        self.center = bool(center)
        self.pad_mode = pad_mode

        self.sample_rate = int(sample_rate)
        self.n_fft = int(n_fft)
        self.win_length = int(win_length) if win_length is not None else self.n_fft
        self.hop_length = int(hop_length) if hop_length is not None else self.win_length // 2
        self.f_min = float(f_min)
        self.f_max = float(f_max) if f_max is not None else self.sample_rate / 2.0
        self.n_mels = int(n_mels)
        self.power = float(power)
        self.mel_scale = mel_scale
        self.norm = norm
        self.dtype = dtype or torch.float32
        if self.dtype not in (torch.float32, torch.float16):
            raise ValueError("output dtype must be torch.float32 or torch.float16")
        self._plans: dict = {}

    def _plan(self, device_index: int, in_dtype: str):
        import torch

        key = (device_index, in_dtype)
        if key not in self._plans:
            with torch.cuda.device(device_index):
                self._plans[key] = fb.fm_plan_create_ex(
                    self.sample_rate, self.n_fft, self.hop_length, self.win_length, self.n_mels, self.f_min,
                    self.f_max, self.power, self.mel_scale, self.norm, in_dtype,
                    "f16" if self.dtype == torch.float16 else "f32", self.center, self.pad_mode, self.pad,
                    self.normalized,
                )
        return self._plans[key]

    def n_frames(self, T: int) -> int:
        Tp = int(T) + 2 * self.pad
        if self.center:
            return 1 + Tp // self.hop_length
        return 1 + (Tp - self.n_fft) // self.hop_length if Tp >= self.n_fft else -1

    def __call__(self, x, out=None):
        import torch

        if not x.is_cuda:
            raise ValueError("input must be a CUDA tensor (the mel path runs only on the GPU)")
        if x.requires_grad and torch.is_grad_enabled():
            raise RuntimeError("inference only: no backward is implemented")
        tags = {torch.float32: "f32", torch.int16: "i16", torch.float16: "f16"}
        if x.dtype not in tags:
            raise TypeError(f"input dtype {x.dtype} not supported (float32, int16, float16)")
        lead, T = tuple(x.shape[:-1]), int(x.shape[-1])
        xc = x.contiguous()
        B = xc.numel() // T if T else 0
        if self.n_frames(T) < 1:
            raise ValueError(f"{T} samples are too short for this framing")
        shape = (*lead, self.n_mels, self.n_frames(T))
        if out is None:
            out = torch.empty(shape, dtype=self.dtype, device=x.device)
        elif tuple(out.shape) != shape or out.dtype != self.dtype or not out.is_contiguous():
            raise ValueError("out has the wrong shape, dtype or layout")
        with torch.cuda.device(x.device):
            plan = self._plan(x.device.index, tags[x.dtype])
            stream = torch.cuda.current_stream(x.device).cuda_stream
            fb.fm_mel_forward(plan, xc.data_ptr(), B, T, out.data_ptr(), stream)
        return out

    def close(self) -> None:
        for p in self._plans.values():
            fb.fm_plan_destroy(p)
        self._plans.clear()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
