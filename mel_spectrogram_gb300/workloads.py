"""Seeded synthetic workloads: shapes, parameters and input recipes.

This module holds no step of the mel computation. It only describes the five
workloads (signal shapes, storage dtypes and transform parameters) and draws
their seeded inputs with numpy's PCG64 generator, so that the CUDA path and
the float64 oracle are fed the same samples.

The workloads stand in for "30 s of 16 kHz speech" (the Whisper-style case the
flashmel README benchmarks under "Performance") and "30 s of 22.05 kHz music";
no public dataset is involved.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    in_dtype: str  # "f32" | "i16" | "f16"
    out_dtype: str  # "f32" | "f16"
    sr: int
    n_fft: int
    hop: int
    win_length: int
    n_mels: int
    f_min: float
    f_max: float
    power: float
    mel_scale: str  # "htk" | "slaney"
    norm: str | None  # None | "slaney"
    recipe: str  # "normal" | "pcm16" | "sines" | "music16"
    seed: int
    extra: dict = field(default_factory=dict)

    @property
    def n_frames(self) -> int:
        return 1 + self.T // self.hop

    @property
    def out_shape(self) -> tuple[int, int, int]:
        return (self.B, self.n_mels, self.n_frames)

    def resized(self, B: int | None = None, T: int | None = None) -> "Workload":
        return replace(self, B=self.B if B is None else B, T=self.T if T is None else T)

    def in_bytes(self) -> int:
        return self.B * self.T * {"f32": 4, "i16": 2, "f16": 2}[self.in_dtype]

    def out_bytes(self) -> int:
        return self.B * self.n_mels * self.n_frames * {"f32": 4, "f16": 2}[self.out_dtype]


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny", 1, 16000, "f32", "f32", 16000, 400, 160, 400, 80, 0.0, 8000.0, 2.0, "htk", None, "normal", 0),
        Workload("speech", 8, 480000, "f32", "f32", 16000, 400, 160, 400, 128, 0.0, 8000.0, 2.0, "htk", None, "normal", 1),
        Workload("int16", 32, 480000, "i16", "f32", 16000, 400, 160, 400, 128, 0.0, 8000.0, 2.0, "htk", None, "pcm16", 2),
        Workload("pow2", 64, 32768, "f32", "f32", 16000, 1024, 256, 1024, 80, 0.0, 8000.0, 2.0, "htk", None, "sines", 3),
        Workload("music", 64, 661500, "f16", "f16", 22050, 2048, 512, 2048, 128, 0.0, 11025.0, 1.0, "slaney", "slaney", "music16", 4),
        # the flashmel README's "huge" case (n_fft 16384, hop 4096, 256 mels at
        # 44.1 kHz, batch 16; its signal length is not stated: 30 s here)
        Workload("huge", 16, 1323000, "f32", "f32", 44100, 16384, 4096, 16384, 256, 0.0, 22050.0, 2.0, "htk", None, "normal", 5),
    ]
}

# the order the workloads are listed in (index == seed)
ORDER = ["tiny", "speech", "int16", "pow2", "music"]
# further workloads the bench also times (the largest transform size)
EXTRA = ["huge"]


def make_input(w: Workload, seed: int | None = None) -> np.ndarray:
    """Draw the [B, T] input of workload ``w`` in its storage dtype.

    normal  : float32 N(0, 1)
    pcm16   : int16 uniform over [-32768, 32767]
    sines   : float32, per signal the sum of three cosines with frequencies
              U(50, 7000) Hz, amplitudes U(0.1, 1), phases U(0, 2 pi), plus
              0.01 N(0, 1) noise
    music16 : float16 of 0.3 N(0, 1) clipped to [-1, 1]
    """
    rng = np.random.default_rng(w.seed if seed is None else seed)
    B, T = w.B, w.T
    if w.recipe == "normal":
        return rng.standard_normal((B, T), dtype=np.float32)
    if w.recipe == "pcm16":
        return rng.integers(-32768, 32767, size=(B, T), endpoint=True, dtype=np.int16)
    if w.recipe == "sines":
        f = rng.uniform(50.0, 7000.0, size=(B, 3, 1))
        a = rng.uniform(0.1, 1.0, size=(B, 3, 1))
        ph = rng.uniform(0.0, 2.0 * np.pi, size=(B, 3, 1))
        n = np.arange(T, dtype=np.float64)[None, None, :]
        x = (a * np.cos(2.0 * np.pi * f * n / w.sr + ph)).sum(axis=1)
        x += 0.01 * rng.standard_normal((B, T))
        return x.astype(np.float32)
    if w.recipe == "music16":
        x = 0.3 * rng.standard_normal((B, T), dtype=np.float32)
        return np.clip(x, -1.0, 1.0).astype(np.float16)
    raise ValueError(w.recipe)


def make_input_device(w: Workload, device, seed: int | None = None):
    """Draw a [B, T] input of workload ``w`` directly in device memory with
    torch's seeded generator on that device (for batches too large to draw on
    the host): normal -> float32 N(0, 1), pcm16 -> int16 uniform over
    [-32768, 32767]. Same recipes as make_input, not the same values."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    if w.recipe == "normal":
        return torch.randn((w.B, w.T), generator=g, device=device, dtype=torch.float32)
    if w.recipe == "pcm16":
        return torch.randint(-32768, 32768, (w.B, w.T), generator=g, device=device, dtype=torch.int16)
    raise ValueError(w.recipe)


def shard_rows(B: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous batch rows [lo, hi) owned by ``rank`` of ``world`` replicas."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, rem = divmod(B, world)
    lo = rank * base + min(rank, rem)
    return lo, lo + base + (1 if rank < rem else 0)
