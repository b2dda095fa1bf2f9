"""Benchmark of the fused mel-spectrogram kernel on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference] [--sweep]

A step is one pass of the whole path (pad, frame, window, real DFT, |X|^p,
mel projection) over one batch of the workload: one fm_mel_forward launch.
Steps rotate over 16 input/output buffer sets (more bytes than the 129 MB
L2), are captured in a CUDA graph and replayed; the timed region is exactly K
steps between barriers and device synchronisations, timed with CUDA events on
the launching stream. Under torchrun every rank runs its own replica (weak
scaling, no collective on the data path); the reported time is the max over
ranks. `--impl reference` times the float64 CPU oracle on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mel_spectrogram_gb300.workloads import EXTRA, ORDER, WORKLOADS, make_input  # noqa: E402

BUFFER_SETS = 16
HOST_SLACK_CYCLES = 200_000  # ~0.1 ms of device-side wait ahead of a timed region
SINGLE_GRAPH_MAX = 512  # up to this many timed steps go into one captured graph
L2_BYTES = 129 * 1024 * 1024
def kernel_sha() -> str:
    """Fingerprint of the device code (every kernel source and header)."""
    import glob

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mel_spectrogram_gb300", "csrc")
    for f in sorted(glob.glob(os.path.join(csrc, "fm_kernel*")) + glob.glob(os.path.join(csrc, "fm_fft*.cuh")) +
                    [os.path.join(csrc, "fm_internal.h")]):
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "sm_max_mhz": float(d.get("sm_max_mhz", 2070.0)),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0, "source": "fallback"}


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if still current."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_sha") != kernel_sha():
        return None  # the kernel changed since the counters were taken
    v = d.get("bytes_per_launch", {}).get(workload)
    return float(v) if v is not None else None


def recorded_l2_write_bytes(workload: str):
    """L2 write sectors x 32 B per launch (the output side, which DRAM shows
    only later as write-back), from the same record, if still current."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_sha") != kernel_sha():
        return None
    v = d.get("l2_write_sectors", {}).get(workload)
    return 32.0 * v if v is not None else None


def recorded_fma_pipe(workload: str):
    """ncu FMA-pipe utilisation (% of peak, active cycles) of the kernel, if current."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_sha") != kernel_sha():
        return None
    v = d.get("fma_pipe_pct", {}).get(workload)
    return float(v) if v is not None else None


def describe(w) -> str:
    norm = "Slaney norm" if w.norm else "no norm"
    return (f"{w.name}: B={w.B} x T={w.T} {w.in_dtype}, sr {w.sr}, n_fft {w.n_fft}, hop {w.hop}, "
            f"{w.n_mels} mels {w.mel_scale.upper()} {norm}, power {w.power:g}, {w.out_dtype} out "
            f"-> [{w.B},{w.n_mels},{w.n_frames}]")


def conventional_flops(w) -> float:
    """Per frame: real FFT 2.5 N log2 N + window N + power 3 n_freqs + mel 2 nnz."""
    from mel_spectrogram_gb300 import fm_mel_filterbank_csr

    _, _, _, wts = fm_mel_filterbank_csr(w.sr, w.n_fft, w.n_mels, w.f_min, w.f_max, w.mel_scale, w.norm)
    N = w.n_fft
    per_frame = 2.5 * N * np.log2(N) + N + 3 * (N // 2 + 1) + 2 * len(wts)
    return per_frame * w.B * w.n_frames


class ClockSampler:
    """nvidia-smi clocks and throttle reasons while the timed region runs."""

    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self, t_start: float, t_end: float) -> dict:
        import datetime

        rows = [r.split(",") for r in (self.out or "").strip().splitlines() if r.count(",") >= 7]
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                ts = datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
                if ts < t_start - 0.05 or ts > t_end + 0.05:
                    continue  # outside the timed region
                mhz.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for name, flag in zip(names, r[4:8]):
                if flag.strip().lower() in ("active", "1"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


# ----------------------------------------------------------------- GPU arm
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return world, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def metric_for(w) -> str:
    """The metric string for workload ``w`` (the headline names the speech batch)."""
    return (f"mel frames/sec and achieved HBM GB/s (fraction of roofline) at B={w.B}×{w.T} "
            f"{ {'f32': 'fp32', 'i16': 'int16', 'f16': 'f16'}[w.in_dtype] }")


class WorkloadRun:
    """One workload's plan, rotating device buffers and timing helpers."""

    def __init__(self, fb, w, stream):
        import torch

        self.fb, self.w, self.s = fb, w, stream
        self.x = make_input(w)
        tdt = {"f32": torch.float32, "i16": torch.int16, "f16": torch.float16}
        self.out_dtype = tdt[w.out_dtype]
        self.plan = fb.fm_plan_create(w.sr, w.n_fft, w.hop, w.win_length, w.n_mels, w.f_min, w.f_max, w.power,
                                      w.mel_scale, w.norm, w.in_dtype, w.out_dtype)
        self.info = fb.fm_plan_get_info(self.plan)
        self.nf = fb.fm_n_frames(self.plan, w.T)
        xin = torch.from_numpy(self.x).cuda()
        self.d_in = [xin.clone() for _ in range(BUFFER_SETS)]
        self.d_out = [torch.empty((w.B, w.n_mels, self.nf), dtype=self.out_dtype, device="cuda")
                      for _ in range(BUFFER_SETS)]
        self.graphs = {}

    def launch(self, i):
        w = self.w
        self.fb.fm_mel_forward(self.plan, self.d_in[i].data_ptr(), w.B, w.T, self.d_out[i].data_ptr(),
                               self.s.cuda_stream)

    def graph(self, n, same_set=False):
        """A CUDA graph of n launches rotating over the buffer sets (i mod 16),
        or of n launches on set 0."""
        import torch

        key = (n, same_set)
        if key not in self.graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.s):
                for i in range(n):
                    self.launch(0 if same_set else i % BUFFER_SETS)
            with torch.cuda.stream(self.s):
                g.replay()  # upload
            self.s.synchronize()
            self.graphs[key] = g
        return self.graphs[key]

    def warm(self, W):
        import torch

        with torch.cuda.stream(self.s):
            for i in range(W):
                self.launch(i % BUFFER_SETS)
        self.s.synchronize()

    def steps_graphs(self, K):
        """The graphs that replay exactly K launches: one graph of K launches
        when K is at most SINGLE_GRAPH_MAX (no gap between graph launches in
        the timed region), else graphs of 16 launches and one of the rest."""
        if K <= SINGLE_GRAPH_MAX:
            return [self.graph(K)]
        full, rest = divmod(K, BUFFER_SETS)
        return [self.graph(BUFFER_SETS)] * full + ([self.graph(rest)] if rest else [])

    def timed_steps_ms(self, K):
        """Device time of exactly K launches replayed from graphs over the
        rotating sets. A device-side wait queued ahead of the start event keeps
        the host's graph submission out of the timed region."""
        import torch

        gs = self.steps_graphs(K)
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.s):
            torch.cuda._sleep(HOST_SLACK_CYCLES)
            a.record(self.s)
            for g in gs:
                g.replay()
            z.record(self.s)
        self.s.synchronize()
        return a.elapsed_time(z)

    def replay_us(self, g, n, reps):
        import torch

        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.s):
            torch.cuda._sleep(HOST_SLACK_CYCLES)
            a.record(self.s)
            for _ in range(reps):
                g.replay()
            z.record(self.s)
        self.s.synchronize()
        return a.elapsed_time(z) * 1e3 / (n * reps)

    def single_launch_us(self, n=32):
        """Median device time of one launch on its own (nothing queued before or
        after it, so no dependent-launch overlap: every launch pays its full
        start-up and first-tile fetch)."""
        import torch

        ts = []
        for i in range(n):
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(self.s):
                torch.cuda._sleep(HOST_SLACK_CYCLES)
                a.record(self.s)
                self.launch(i % BUFFER_SETS)
                z.record(self.s)
            self.s.synchronize()
            ts.append(a.elapsed_time(z) * 1e3)
        return statistics.median(ts)

    def figures(self, step_s, clk_mhz, props):
        """Throughput, roofline and FP32 fractions for a step time."""
        w = self.w
        pk = peaks()
        in_b, out_b = w.in_bytes(), w.out_bytes()
        achieved = (in_b + out_b) / step_s / 1e9
        flops = conventional_flops(w)
        fp32_peak = props.multi_processor_count * 128 * 2 * clk_mhz * 1e6 / 1e12
        return {
            "frames_per_s": w.B * self.nf / step_s,
            "audio_seconds_per_s": w.B * w.T / w.sr / step_s,
            "hbm_gbs": achieved,
            "roofline": {
                "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"],
                "peak_source": f"{pk['source']} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                "algorithmic_bytes_per_launch": in_b + out_b,
                "traffic": recorded_traffic(w.name),
                "l2_write_bytes": recorded_l2_write_bytes(w.name),
            },
            "fp32": {"achieved_tflops": flops / step_s / 1e12, "peak_tflops": fp32_peak,
                     "frac": flops / step_s / 1e12 / fp32_peak,
                     "peak_basis": f"{props.multi_processor_count} SMs x 128 lanes x 2 x {clk_mhz:.0f} MHz",
                     "ncu_fma_pipe_pct": recorded_fma_pipe(w.name)},
        }

    def close(self):
        self.fb.fm_plan_destroy(self.plan)


def sweep_workloads():
    """The flashmel README's size sweep ("Performance": hop = n_fft/4, 128 mels,
    B=32, T=160000), one workload per supported n_fft, f32 in and out."""
    from mel_spectrogram_gb300.workloads import Workload

    sizes = [64, 128, 256, 400, 512, 1024, 2048, 4096, 8192, 16384]
    return [Workload(f"sweep{n}", 32, 160000, "f32", "f32", 16000, n, n // 4, n, 128, 0.0, 8000.0, 2.0, "htk",
                     None, "normal", 100 + i) for i, n in enumerate(sizes)]


def run_sweep(args) -> dict:
    """Time the size sweep on one GPU; one JSON line with a row per size."""
    import torch

    torch.cuda.set_device(0)
    from mel_spectrogram_gb300.build import build

    build()
    from mel_spectrogram_gb300 import _binding as fb

    s = torch.cuda.Stream()
    props = torch.cuda.get_device_properties(0)
    rows = {}
    for w in sweep_workloads():
        r = WorkloadRun(fb, w, s)
        K = min(args.steps, args.other_steps)
        r.warm(args.warmup)
        r.steps_graphs(K)
        with ClockSampler(0) as ck:
            torch.cuda.synchronize()
            ta = time.time()
            ms = r.timed_steps_ms(K)
            torch.cuda.synchronize()
            tb = time.time()
        clk = ck.summary(ta, tb)
        assert fb.fm_plan_poll_error(r.plan) == fb.FM_OK
        fig = r.figures(ms / 1e3 / K, clk["sm_mhz"] or peaks()["sm_max_mhz"], props)
        rows[w.name] = {"n_fft": w.n_fft, "hop": w.hop, "us_per_step": ms * 1e3 / K,
                        "hbm_frac": fig["roofline"]["frac"], "hbm_gbs": fig["hbm_gbs"],
                        "fp32_frac": fig["fp32"]["frac"], "frames_per_s": fig["frames_per_s"],
                        "threads_per_block": r.info["threads_per_block"], "frames_per_tile": r.info["frames_per_tile"],
                        "blocks_per_sm": r.info["blocks_per_sm"], "clocks": clk}
        r.close()
    return {"sweep": "flashmel README size sweep: hop = n_fft/4, 128 mels, B=32 x T=160000 f32, sr 16000, "
                     "HTK, power 2, f32 out; kernel only, 16 rotating input/output sets",
            "steps": min(args.steps, args.other_steps), "rows": rows}


def run_gpu_arm(args) -> dict | None:
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from mel_spectrogram_gb300.build import build

    if local == 0:
        build()
    if world > 1:
        dist.barrier()
    from mel_spectrogram_gb300 import _binding as fb

    w = WORKLOADS[args.workload]
    s = torch.cuda.Stream()
    run = WorkloadRun(fb, w, s)
    K, W = args.steps, args.warmup
    run.warm(W)
    run.steps_graphs(K)  # captured and uploaded before the timed region

    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_start = time.time()
        ms = run.timed_steps_ms(K)
        torch.cuda.synchronize()
        t_end = time.time()
        if world > 1:
            dist.barrier()
    if world > 1:
        t = torch.tensor([ms], device="cuda", dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    clocks = clk.summary(t_start, t_end)
    assert fb.fm_plan_poll_error(run.plan) == fb.FM_OK

    # after the timed region: five repeats of the cold-L2 replay (median), a
    # warm-L2 replay that reuses one input/output set, and single launches
    # (all labelled, none of them the reported value)
    reps = max(1, min(K, 2000) // BUFFER_SETS)
    repeat_us = [run.replay_us(run.graph(BUFFER_SETS), BUFFER_SETS, reps) for _ in range(5)]
    warm_us = run.replay_us(run.graph(BUFFER_SETS, same_set=True), BUFFER_SETS, reps)
    single_us = run.single_launch_us()

    # end to end through the public C ABI with host buffers (copies in the region)
    Ke = max(3, min(K, args.e2e_steps))
    h_in = torch.from_numpy(run.x).pin_memory()
    h_out = torch.empty((w.B, w.n_mels, run.nf), dtype=run.out_dtype).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def e2e_step(i):
        fb.fm_mel_forward_host(run.plan, h_in.data_ptr(), w.B, w.T, h_out.data_ptr(), run.d_in[i].data_ptr(),
                               run.d_out[i].data_ptr(), s.cuda_stream)

    for i in range(3):
        e2e_step(i)
    s.synchronize()
    if world > 1:
        dist.barrier()
    e0.record(s)
    h0 = time.perf_counter()
    for i in range(Ke):
        e2e_step(i % BUFFER_SETS)
    enqueue_us = (time.perf_counter() - h0) * 1e6 / Ke  # host time to queue one step
    e1.record(s)
    s.synchronize()
    e_ms = e0.elapsed_time(e1)
    # the same host-buffer call captured once into a CUDA graph and replayed
    # (uploads, kernels and downloads as the call queued them): the device-side
    # pipeline without the host's per-call queueing cost; reported beside e2e
    ge_us = None
    try:
        ge = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ge, stream=s):
            e2e_step(0)
        with torch.cuda.stream(s):
            ge.replay()
        s.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            torch.cuda._sleep(HOST_SLACK_CYCLES)
            g0.record(s)
            for _ in range(Ke):
                ge.replay()
            g1.record(s)
        s.synchronize()
        ge_us = g0.elapsed_time(g1) * 1e3 / Ke
    except RuntimeError:
        ge_us = None
    if world > 1:
        t = torch.tensor([e_ms], device="cuda", dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e_ms = float(t.item())
    info, nf = run.info, run.nf
    run.close()

    # the other workloads, timed the same way on this rank (rank 0 reports them)
    others = {}
    if not args.only:
        for name in ORDER + EXTRA:
            if name == w.name:
                continue
            ow = WORKLOADS[name]
            r2 = WorkloadRun(fb, ow, s)
            K2 = min(K, args.other_steps)
            r2.warm(W)
            r2.steps_graphs(K2)
            with ClockSampler(local) as c2:
                torch.cuda.synchronize()
                ta = time.time()
                ms2 = r2.timed_steps_ms(K2)
                torch.cuda.synchronize()
                tb = time.time()
            ck = c2.summary(ta, tb)
            assert fb.fm_plan_poll_error(r2.plan) == fb.FM_OK
            reps2 = max(1, min(K2, 2000) // BUFFER_SETS)
            rep2 = statistics.median(r2.replay_us(r2.graph(BUFFER_SETS), BUFFER_SETS, reps2) for _ in range(3))
            props = torch.cuda.get_device_properties(0)
            fig = r2.figures(ms2 / 1e3 / K2, ck["sm_mhz"] or peaks()["sm_max_mhz"], props)
            others[name] = {"metric": metric_for(ow), "workload": describe(ow), "steps": K2,
                            "us_per_step": ms2 * 1e3 / K2, "repeats_median_us": rep2,
                            "single_launch_us": r2.single_launch_us(16), **fig,
                            "grid": min(r2.info["grid_limit"], ow.B * -(-r2.nf // r2.info["frames_per_tile"])),
                            "block": r2.info["threads_per_block"], "clocks": ck}
            r2.close()
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return None

    frames_step = w.B * nf
    step_s = ms / 1e3 / K
    pk = peaks()
    in_b, out_b = w.in_bytes(), w.out_bytes()
    props = torch.cuda.get_device_properties(0)
    clk_mhz = clocks["sm_mhz"] or pk["sm_max_mhz"]
    fig = run.figures(step_s, clk_mhz, props)
    line = {
        "metric": metric_for(w),
        "value": world * frames_step / step_s,
        "unit": "frames/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": f"synthetic, seeded ({w.recipe}, seed {w.seed})",
        "config": {
            "workload": describe(w),
            "B": w.B, "T": w.T, "n_fft": w.n_fft, "hop": w.hop, "n_mels": w.n_mels,
            "in_dtype": w.in_dtype, "out_dtype": w.out_dtype,
            "l2": f"{BUFFER_SETS} rotating input/output sets, "
                  f"{BUFFER_SETS * (in_b + out_b) / 1e6:.0f} MB > {L2_BYTES / 1e6:.0f} MB L2",
            "launch": (f"one CUDA graph of the {K} fm_mel_forward launches" if K <= SINGLE_GRAPH_MAX else
                       f"CUDA graphs of {BUFFER_SETS} fm_mel_forward launches, replayed") +
                      " over the rotating sets; a device-side wait queued ahead of the start event keeps host "
                      "submission out of the timed region",
            "grid": min(info["grid_limit"], w.B * -(-nf // info["frames_per_tile"])),
            "block": info["threads_per_block"], "smem_bytes": info["smem_bytes"],
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "audio_seconds_per_s": world * fig["audio_seconds_per_s"],
        "hbm_gbs": fig["hbm_gbs"],
        "roofline": fig["roofline"],
        "fp32": fig["fp32"],
        "e2e": {"value": world * frames_step * Ke / (e_ms / 1e3), "unit": "frames/s",
                "h2d_bytes_per_step": in_b, "d2h_bytes_per_step": out_b, "steps": Ke,
                "api": "fm_mel_forward_host (pinned host buffers; per step the upload, kernel and download "
                       "of up to four signal chunks, overlapped on plan-owned streams)",
                "us_per_step": e_ms * 1e3 / Ke, "host_enqueue_us_per_step": enqueue_us,
                "graph_replay_us_per_step": ge_us,
                "graph_note": "the same call captured once into a CUDA graph and replayed (copies in the region); "
                              "not the reported value"},
        "repeats": {"us_per_step": [round(v, 3) for v in repeat_us], "median_us": statistics.median(repeat_us),
                    "launches_each": reps * BUFFER_SETS,
                    "note": "cold L2 (16 rotating sets), timed after the main region"},
        "warm_l2": {"us_per_step": warm_us, "launches": reps * BUFFER_SETS,
                    "note": "one input/output set replayed: inputs and outputs stay in L2; not the reported value"},
        "single_launch": {"us": single_us, "note": "one launch with nothing queued around it (no dependent-launch "
                                                  "overlap with a previous call): the latency one isolated call "
                                                  "sees; median of 32, not the reported value"},
        "gpu_launches": K,
        "clocks": clocks,
    }
    if others:
        line["workloads"] = others
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(w, run.x, args.cpu_seconds)
    return line


# ------------------------------------------------------- oracle on the host
def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_segment(w, x, frames: int):
    """Signal 0 cut so that centre framing yields about `frames` frames."""
    Ts = max(w.n_fft // 2 + 1, (frames - 1) * w.hop)
    Ts = min(Ts, w.T)
    return x[0:1, :Ts], 1 + Ts // w.hop


def oracle_run(w, seg):
    import oracle.mel_oracle as o

    return o.mel_spectrogram(seg, w.sr, w.n_fft, w.hop, w.n_mels, w.f_min, w.f_max, w.power, w.mel_scale, w.norm,
                             w.win_length)


def oracle_baseline(w, x, seconds: float) -> dict:
    """The oracle as it stands, timed on a bounded sample (repeated for ~seconds)."""
    seg, fr = oracle_segment(w, x, min(w.n_frames, 512))
    oracle_run(w, seg)
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_run(w, seg)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": n * fr / el, "unit": "frames/s", "cores": host_cores(), "kind": "oracle",
            "sample": f"{fr} frames of signal 0 (first {seg.shape[1]} samples), {n} repeats in {el:.1f} s; "
                      f"float64 numpy, naive DFT as a matmul; BLAS threads = host cores"}


def run_reference_arm(args) -> dict | None:
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    w = WORKLOADS[args.workload]
    x = make_input(w)
    probe, fr_probe = oracle_segment(w, x, 64)
    oracle_run(w, probe)
    t0 = time.perf_counter()
    oracle_run(w, probe)
    per_frame = (time.perf_counter() - t0) / fr_probe
    K, W = args.steps, args.warmup
    budget = args.ref_seconds
    frames = int(max(1, min(w.n_frames, budget / max(1, K + W) / per_frame)))
    seg, fr = oracle_segment(w, x, frames)
    for _ in range(W):
        oracle_run(w, seg)
    t0 = time.perf_counter()
    for _ in range(K):
        oracle_run(w, seg)
    el = time.perf_counter() - t0
    v = fr * K / el
    sample = f"{fr} frames of signal 0 per step (first {seg.shape[1]} samples), {K} steps in {el:.1f} s"
    return {
        "impl": "reference", "metric": metric_for(w), "value": v, "unit": "frames/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": el * 1e3 / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": f"synthetic, seeded ({w.recipe}, seed {w.seed})",
        "config": {"workload": describe(w), "B": w.B, "T": w.T, "n_fft": w.n_fft, "hop": w.hop,
                   "n_mels": w.n_mels, "in_dtype": w.in_dtype, "out_dtype": w.out_dtype,
                   "parallelism": "host cores (rank 0 only)"},
        "cpu_baseline": {"value": v, "unit": "frames/s", "cores": host_cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "frames/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main() -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default="speech", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", action="store_true", help="time the chosen workload only")
    ap.add_argument("--sweep", action="store_true",
                    help="time every n_fft on the pages' sweep configuration instead (one JSON line)")
    ap.add_argument("--other-steps", type=int, default=2000,
                    help="timed steps of each of the other workloads (at most --steps)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.sweep:
        print(json.dumps(run_sweep(args)), flush=True)
        return 0
    line = run_reference_arm(args) if args.impl == "reference" else run_gpu_arm(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
