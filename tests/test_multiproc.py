"""Replica sharding across ranks, on CPU with the gloo backend (2 ranks).

The mel path shards by signal with no exchange: each rank runs its own rows.
These tests cover the host-side logic: contiguous shards that tile the batch
exactly, per-rank results that concatenate to the single-process result, and
the max-over-ranks step time the bench reports.
"""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from mel_spectrogram_gb300.workloads import WORKLOADS, make_input, shard_rows


@pytest.mark.parametrize("B,world", [(8, 2), (7, 2), (1, 3), (64, 8), (3, 5)])
def test_shards_tile_the_batch(B, world):
    seen = []
    for r in range(world):
        lo, hi = shard_rows(B, r, world)
        assert 0 <= lo <= hi <= B
        seen.extend(range(lo, hi))
    assert seen == list(range(B))
    sizes = [shard_rows(B, r, world)[1] - shard_rows(B, r, world)[0] for r in range(world)]
    assert max(sizes) - min(sizes) <= 1


def test_shard_rows_rejects_bad_rank():
    with pytest.raises(ValueError):
        shard_rows(4, 2, 2)
    with pytest.raises(ValueError):
        shard_rows(4, 0, 0)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    import torch

    import oracle.mel_oracle as o

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = WORKLOADS["speech"].resized(B=5, T=4000)
        x = make_input(w)
        lo, hi = shard_rows(w.B, rank, world)
        mine = o.mel_spectrogram(x[lo:hi], w.sr, w.n_fft, w.hop, w.n_mels, w.f_min, w.f_max, w.power, w.mel_scale,
                                 w.norm)
        # every rank contributes its rows; rank 0 assembles them
        parts = [None] * world
        dist.all_gather_object(parts, (lo, hi, mine))
        # the bench's step time is the max over ranks
        t = torch.tensor([float(rank + 1)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        if rank == 0:
            full = np.concatenate([p[2] for p in sorted(parts, key=lambda p: p[0])], axis=0)
            np.save(os.path.join(out_dir, "full.npy"), full)
            np.save(os.path.join(out_dir, "tmax.npy"), t.numpy())
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_match_single_process(tmp_path):
    import oracle.mel_oracle as o

    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    full = np.load(tmp_path / "full.npy")
    w = WORKLOADS["speech"].resized(B=5, T=4000)
    x = make_input(w)
    ref = o.mel_spectrogram(x, w.sr, w.n_fft, w.hop, w.n_mels, w.f_min, w.f_max, w.power, w.mel_scale, w.norm)
    assert full.shape == ref.shape
    assert np.array_equal(full, ref)
    assert float(np.load(tmp_path / "tmax.npy")[0]) == float(world)


def test_reference_arm_runs_on_rank_zero_only(tmp_path):
    """Under torchrun the oracle arm of bench.py runs and prints on rank 0
    alone; any other rank exits 0 without work or output."""
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3", "--workload", "tiny"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
