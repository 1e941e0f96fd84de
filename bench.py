"""Benchmark of the vocoder decode on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload music_window]

One step = one full decode (every layer of the decoder) of one batch of the
workload's synthetic latents, already resident in HBM.  Each timed step is
bracketed by CUDA events on the decode stream; a 256 MiB buffer (larger than the
129 MB L2) is written between timed steps, outside the events.  The per-kernel
rooflines ("stages", "roofline") come from as many further steps run with an
event pair around every launch (VOC_FLAG_PROFILE); those events serialise the
launches, so the headline uses the steps without them.  Several ranks
(torchrun, one GPU each) decode independent copies of the workload: weak
scaling with no collective on the data path (a scalar max-reduction of the step
time only).  Rank 0 prints one JSON line.

--workload encode_music_window times the mirror encoder instead: one step encodes a
stereo 689-frame window of audio into latents (metric: audio samples encoded per second).

--impl reference times the CPU oracle on this host's cores on a bounded sample
of the same workload (a slice of latent frames per step)."""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from dac_vocoder_decode_gb300 import workloads as W  # noqa: E402

METRIC = "vocoder audio samples/sec"
ENC_METRIC = "encoder audio samples/sec"  # audio samples encoded into latents per second
UNIT = "samples/s"
SAMPLE_RATE = {"encode_music_window": 44100, "music_window": 44100, "music_batch8": 44100, "music_long": 44100, "speech": 24000,
               "speech_snakebeta": 24000, "tiny": 44100, "tiny_cal": 44100}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def source_hash() -> str:
    """Hash of the CUDA sources and the C header: identifies the kernels a profile was taken on."""
    import glob
    import hashlib
    h = hashlib.sha1()
    files = sorted(glob.glob(os.path.join(ROOT, "dac_vocoder_decode_gb300", "csrc", "*.cu*")) +
                   glob.glob(os.path.join(ROOT, "include", "*.h")))
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# Workloads whose per-launch DRAM traffic is taken from another workload's ncu capture,
# scaled by the ratio of latent frames per item (same architecture and batch): a capture of
# the full-length decode would hold tens of GB on the device, and each layer's traffic grows
# in proportion to its rows (the weights stay in L2).
TRAFFIC_SCALED_FROM = {"music_long": "music_window"}


def measured_traffic(workload: str, layer: str):
    """DRAM bytes (read + write) of one launch of `layer` and where they come from, from the
    ncu summary committed under profiles/; (None, None) when there is none or it was taken on
    other kernel sources."""
    src = TRAFFIC_SCALED_FROM.get(workload, workload)
    path = os.path.join(ROOT, "profiles", f"traffic_{src}.md")
    if not os.path.exists(path):
        return None, None
    with open(path) as f:
        text = f.read()
    if f"source hash: {source_hash()}" not in text:
        return None, None
    for ln in text.splitlines():
        cells = [c.strip() for c in ln.strip().strip("|").split("|")]
        if len(cells) >= 4 and cells[0] == layer:
            try:
                value = int(cells[3])
            except ValueError:
                return None, None
            if src == workload:
                return value, f"ncu capture of {workload} (profiles/traffic_{src}.md)"
            T_src, T_dst = W.WORKLOADS[src][2][2], W.WORKLOADS[workload][2][2]
            return (int(round(value * T_dst / T_src)),
                    f"ncu capture of {src} (profiles/traffic_{src}.md) scaled by "
                    f"{T_dst}/{T_src} latent frames per item")
    return None, None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def tensor_peak(peaks: dict, mmas_per_mac: float, timed_s: float, reasons) -> tuple:
    """Useful tensor rate the kernels are held to (TFLOP/s) and which measured figure it is: the
    burst bf16 rate (a GEMM timed alone), or the sustained one (a seconds-long loop under the
    power cap) when the timed steps -- inside which every kernel is timed -- ran for at least
    half a second with the power cap active.  Divided by the MMAs per useful multiply-add."""
    sustained = timed_s >= 0.5 and "sw_power_cap" in reasons
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    return peaks.get(key, FALLBACK_PEAKS[key]) / mmas_per_mac, ("sustained" if sustained else "burst")


def tracks_per_batch(name: str, B: int) -> float:
    """Tracks delivered per decode: a stereo pair counts once (music), speech items are mono."""
    return B / 2.0 if name.startswith("music") else float(B)


def config_of(wl, name):
    desc = W.WORKLOADS[name][4]
    return {"workload": f"{name}: {desc}", "latent": list(wl.latent.shape),
            "audio": [wl.B, 1, wl.T * wl.arch.hop], "hop": wl.arch.hop,
            "sample_rate": SAMPLE_RATE[name],
            "l2": "flushed between timed steps (256 MiB write, outside the timed events)"}


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        return self.summarize(self.lines)

    @staticmethod
    def summarize(lines):
        """Median SM clock, the largest reported maximum and every throttle reason seen Active
        in `nvidia-smi --format=csv,noheader,nounits` lines of FIELDS; malformed lines (a header,
        a partial last line, "[N/A]") are skipped."""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- ranks
def max_over_ranks(value: float, device="cpu") -> float:
    """Largest value over all ranks of the default process group (the step time that
    the slowest replica needed); the value itself when there is no group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- workloads
def is_encode(name: str) -> bool:
    return name in W.ENC_WORKLOADS


def metric_of(name: str) -> str:
    return ENC_METRIC if is_encode(name) else METRIC


def load_workload(name: str, frames=None):
    return W.make_named_encode_workload(name, frames) if is_encode(name) else W.make_workload(name)


def workload_config(wl, name):
    if not is_encode(name):
        return config_of(wl, name)
    arch = wl.arch
    B, C, L = wl.latent.shape
    return {"workload": f"{name}: {W.ENC_WORKLOADS[name][4]}", "audio": [B, C, L],
            "latent": [B, arch.latent_channels, L // arch.hop], "hop": arch.hop,
            "sample_rate": SAMPLE_RATE[name],
            "l2": "flushed between timed steps (256 MiB write, outside the timed events)"}


def realtime_seconds(wl, name) -> float:
    """Seconds of music / speech one step delivers (a stereo pair counts once; the windowed
    workload delivers its stitched track, not the overlapping windows)."""
    if is_encode(name):
        B, _, L = wl.latent.shape
        return B / 2.0 * L / SAMPLE_RATE[name]
    if getattr(wl, "stitch", None):
        st = wl.stitch
        frames = (st["win_frames"] - st["crop_left"] - st["crop_right"]) * (st["n_win"] - 1) \
            + st["win_frames"]
        return frames * st["hop"] / SAMPLE_RATE[name]
    return tracks_per_batch(name, wl.B) * wl.T * wl.arch.hop / SAMPLE_RATE[name]


# ----------------------------------------------------------------------------- CPU legs
def oracle_sample(wl, frames: int, folded=None, encode=False):
    """Time the oracle on one item's first `frames` latent frames (bounded CPU work); returns
    (audio samples decoded or encoded, seconds, folded parameters)."""
    from oracle import oracle as O
    if folded is None:
        folded = O.fold_params(wl.params)
    if encode:
        hop = wl.arch.hop
        audio = np.ascontiguousarray(wl.latent[:1, :, :min(frames * hop, wl.latent.shape[2])])
        t0 = time.perf_counter()
        O.encode(wl.arch, None, audio, 0, folded)
        return audio.size, time.perf_counter() - t0, folded
    lat = W.slice_latent(wl.latent[:1], 0, min(frames, wl.T))
    t0 = time.perf_counter()
    y = O.decode(wl.arch, None, lat, 0, folded)
    dt = time.perf_counter() - t0
    return y.size, dt, folded


def cpu_threads():
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n and n.isdigit() else (os.cpu_count() or 1)


def cpu_baseline(wl, name, frames):
    enc = is_encode(name)
    samples, dt, _ = oracle_sample(wl, frames, encode=enc)
    what = (f"1 item x {samples} audio samples ({samples // wl.arch.hop} latent frames) of {name} "
            f"encoded" if enc else
            f"1 item x {min(frames, wl.T)} latent frames of {name} ({samples} samples) decoded")
    return {"value": samples / dt, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
            "sample": f"{what} in {dt:.2f} s (fp64 direct loops, OpenMP)"}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    enc = is_encode(args.workload)
    wl = load_workload(args.workload)
    frames = args.ref_frames
    folded = None
    for _ in range(args.warmup):
        _, _, folded = oracle_sample(wl, frames, folded, encode=enc)
    times = []
    samples = 0
    for _ in range(args.steps):
        samples, dt, folded = oracle_sample(wl, frames, folded, encode=enc)
        times.append(dt)
    ms = 1e3 * statistics.mean(times)
    value = samples / (ms / 1e3)
    rate = SAMPLE_RATE[args.workload]
    line = {"impl": "reference", "metric": metric_of(args.workload), "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "x_realtime": value / rate / (2.0 if "music" in args.workload else 1.0),
            "config": workload_config(wl, args.workload),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(),
                             "kind": "oracle",
                             "sample": f"each step: 1 item x {samples} audio samples "
                                       f"({samples // wl.arch.hop} latent frames) of "
                                       f"{args.workload}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU leg
class DecodeJob:
    """One decode of the workload per step, through vocoder_decode (device buffers) or
    vocoder_decode_host (host buffers, copies inside the call).  A windowed workload (`stitch`
    set) also runs the overlap-crop stitch of its decoded windows in every step."""

    def __init__(self, V, wl, precision, dev):
        import torch
        self.V, self.wl = V, wl
        self.ctx = V.Vocoder(wl.arch, V.fold_params(wl.params), precision=precision)
        B, T, hop = wl.B, wl.T, wl.arch.hop
        self.x = torch.from_numpy(wl.latent).to(dev)
        self.y = torch.empty((B, 1, T * hop), dtype=torch.float32, device=dev)
        self.ws = self.ctx.alloc_workspace(B, T)
        self.samples = B * T * hop
        self.st = wl.stitch
        self.z = None
        if self.st:
            st = self.st
            self.stitched = V.vocoder_stitched_length(st["n_win"], st["win_frames"],
                                                      st["crop_left"], st["crop_right"], st["hop"])
            self.z = torch.empty((st["n_sides"], self.stitched), dtype=torch.float32, device=dev)
        self.h2d = int(wl.latent.nbytes)
        self.d2h = int((self.z if self.st else self.y).numel() * 4)
        self.stitch_ms = []

    def _stitch(self, stream, y, z):
        st = self.st
        self.V.vocoder_stitch(y, st["n_win"], st["n_sides"], st["win_frames"], st["crop_left"],
                              st["crop_right"], st["hop"], z, stream)

    def step(self, stream, flags=0):
        self.V.vocoder_decode(self.ctx.handle, self.x, self.y, self.ws, stream, flags)
        if self.st:
            if flags & self.V.VOC_FLAG_PROFILE:  # the stitch's own launch time
                import torch
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                self._stitch(stream, self.y, self.z)
                e1.record(stream)
                e1.synchronize()
                self.stitch_ms.append(e0.elapsed_time(e1))
            else:
                self._stitch(stream, self.y, self.z)

    def setup_host(self):
        import torch
        wl = self.wl
        self.x_h = torch.from_numpy(wl.latent).pin_memory()
        out = self.z if self.st else self.y
        self.y_h = torch.empty(tuple(out.shape), dtype=torch.float32).pin_memory()
        self.ws_h = self.ctx.alloc_workspace(wl.B, wl.T, host_io=True)

    def host_step(self, stream):
        if not self.st:
            self.V.vocoder_decode_host(self.ctx.handle, self.x_h, self.y_h, self.ws_h, stream)
            return
        # windows: latent in, decode, stitch, the stitched track out (host copies on the stream)
        import torch
        with torch.cuda.stream(stream):
            self.x.copy_(self.x_h, non_blocking=True)
            self.V.vocoder_decode(self.ctx.handle, self.x, self.y, self.ws, stream)
            self._stitch(stream, self.y, self.z)
            self.y_h.copy_(self.z, non_blocking=True)
        stream.synchronize()

    def profile(self):
        prof = self.V.vocoder_profile(self.ctx.handle)
        if self.st and self.stitch_ms:
            n = self.z.numel()
            prof.append(dict(name="stitch", ms=self.stitch_ms[-1], flops=0.0, bytes=8.0 * n))
        return prof

    def launches(self):
        return (self.V.vocoder_launches_per_decode(self.ctx.handle, self.wl.B, self.wl.T)
                + (1 if self.st else 0))

    def close(self):
        self.ctx.close()


class StreamJob(DecodeJob):
    """A causal decoder's latent decoded chunk by chunk (vocoder_stream_decode, `frames`
    latent frames per call, contexts carried between calls); one step decodes the whole
    workload this way, from reset contexts.  The profiled steps run whole-sequence decodes
    (the same kernels) for the per-kernel rooflines."""

    def __init__(self, V, wl, precision, dev, frames):
        import torch
        super().__init__(V, wl, precision, dev)
        self.F = frames
        B, T, hop = wl.B, wl.T, wl.arch.hop
        self.n_calls = (T + frames - 1) // frames
        self.chunks = [self.x[:, :, i * frames:min(T, (i + 1) * frames)].contiguous()
                       for i in range(self.n_calls)]
        # one contiguous audio buffer per call ([B, 1, frames of this call * hop])
        self.ys = [torch.empty((B, 1, c.shape[2] * hop), dtype=torch.float32, device=dev)
                   for c in self.chunks]
        self.sh = V.VocoderStream(self.ctx, B, frames)
        self.call_ms = []

    def _chunks(self, stream, chunks):
        self.sh.reset(stream)
        for i, c in enumerate(chunks):
            self.sh.decode(c, audio=self.ys[i], stream=stream)

    def step(self, stream, flags=0):
        if flags & self.V.VOC_FLAG_PROFILE:
            super().step(stream, flags)
            return
        self._chunks(stream, self.chunks)

    def time_calls(self, stream, n=50):
        """Latency of single calls (events around each), after a reset."""
        import torch
        self.sh.reset(stream)
        with torch.cuda.stream(stream):
            for i in range(min(n, self.n_calls)):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                self.sh.decode(self.chunks[i], audio=self.ys[i], stream=stream)
                e1.record(stream)
                e1.synchronize()
                self.call_ms.append(e0.elapsed_time(e1))

    def setup_host(self):
        import torch
        self.x_h = [c.cpu().pin_memory() for c in self.chunks]
        self.y_h = [torch.empty(tuple(y.shape), dtype=torch.float32).pin_memory() for y in self.ys]

    def host_step(self, stream):
        # each call as a streaming client makes it: its latent chunk in, the call, its audio out
        import torch
        with torch.cuda.stream(stream):
            self.sh.reset(stream)
            for i in range(self.n_calls):
                self.chunks[i].copy_(self.x_h[i], non_blocking=True)
                self.sh.decode(self.chunks[i], audio=self.ys[i], stream=stream)
                self.y_h[i].copy_(self.ys[i], non_blocking=True)
        stream.synchronize()

    def launches(self):
        # per call: the decode's launches plus the two context copies
        per = self.V.vocoder_launches_per_decode(self.ctx.handle, self.wl.B, self.F) + 2
        return per * self.n_calls

    def close(self):
        self.sh.close()
        super().close()


class EncodeJob(DecodeJob):
    """One encode of the workload's audio per step (vocoder_encode / vocoder_encode_host)."""

    def __init__(self, V, wl, precision, dev):
        import torch
        self.V, self.wl = V, wl
        self.ctx = V.Encoder(wl.arch, V.fold_params(wl.params), precision=precision)
        B, C, L = wl.latent.shape
        self.x = torch.from_numpy(wl.latent).to(dev)
        self.y = torch.empty((B, wl.arch.latent_channels, L // wl.arch.hop), dtype=torch.float32,
                             device=dev)
        self.ws = self.ctx.alloc_workspace(B, L)
        self.samples = B * L
        self.h2d, self.d2h = int(wl.latent.nbytes), int(self.y.numel() * 4)

    def step(self, stream, flags=0):
        self.V.vocoder_encode(self.ctx.handle, self.x, self.y, self.ws, stream, flags)

    def setup_host(self):
        import torch
        B, _, L = self.wl.latent.shape
        self.x_h = torch.from_numpy(self.wl.latent).pin_memory()
        self.y_h = torch.empty(tuple(self.y.shape), dtype=torch.float32).pin_memory()
        self.ws_h = self.ctx.alloc_workspace(B, L, host_io=True)

    def host_step(self, stream):
        self.V.vocoder_encode_host(self.ctx.handle, self.x_h, self.y_h, self.ws_h, stream)

    def profile(self):
        return self.V.vocoder_encoder_profile(self.ctx.handle)

    def launches(self):
        B, _, L = self.wl.latent.shape
        return self.V.vocoder_encoder_launches(self.ctx.handle, B, L)


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from dac_vocoder_decode_gb300 import binding as V

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks, peaks_kind = load_peaks()
    wl = load_workload(args.workload)
    f16w = args.precision == "f16w"
    one_plane = args.precision in ("f16w", "bf16w")  # one weight plane, two MMAs per MAC
    prec = {"bf16x3": V.VOC_PREC_BF16X3, "f16w": V.VOC_PREC_F16W,
            "bf16w": V.VOC_PREC_BF16W}[args.precision]
    if args.stream_frames > 0:
        if is_encode(args.workload) or wl.arch.padding != W.PAD_CAUSAL:
            raise SystemExit("--stream-frames needs a causal decoder workload (speech)")
        job = StreamJob(V, wl, prec, dev, args.stream_frames)
    else:
        job = (EncodeJob if is_encode(args.workload) else DecodeJob)(V, wl, prec, dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            job.step(stream)
    torch.cuda.synchronize()

    launches = job.launches()
    per_kernel = {}
    step_ms, prof_ms = [], []

    def timed_steps(flags, out):
        """args.steps steps, each bracketed by CUDA events on the job's stream, L2 flushed
        before each (outside the events)."""
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                flush.fill_(1.0)  # evict the previous step's data from L2 (not timed)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                job.step(stream, flags)
                e1.record(stream)
                e1.synchronize()
                out.append(e0.elapsed_time(e1))
                if flags & V.VOC_FLAG_PROFILE:
                    for i, p in enumerate(job.profile()):
                        rec = per_kernel.setdefault(i, dict(name=p["name"], ms=[],
                                                            flops=p["flops"], bytes=p["bytes"],
                                                            impl_bytes=p.get("impl_bytes")))
                        rec["ms"].append(p["ms"])

    clocks = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    # the headline steps: the kernels chain with programmatic dependent launch
    timed_steps(0, step_ms)
    # the per-kernel breakdown: the same steps with an event pair around every launch (the
    # events keep each launch from overlapping the previous one, so these steps run longer)
    timed_steps(V.VOC_FLAG_PROFILE, prof_ms)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, dev)
    med_max = max_over_ranks(statistics.median(step_ms), dev)  # every rank takes part
    total_samples = job.samples * world
    value = total_samples / (ms_max / 1e3)

    if isinstance(job, StreamJob):
        job.time_calls(stream)

    # end to end through the host-buffer entry point: H2D of the input, the whole path, D2H
    # of the output, inside the timed region
    job.setup_host()
    for _ in range(max(1, args.warmup)):
        job.host_step(stream)
    e2e_s = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        job.host_step(stream)
        e2e_s.append(time.perf_counter() - t0)
    e2e_t = max_over_ranks(statistics.mean(e2e_s), dev)

    # per-kernel roofline: bf16x3 issues three bf16 MMAs per useful multiply-add, f16w two
    # f16 MMAs (f16 and bf16 share the dense tensor rate)
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    mmas_per_mac = 2.0 if one_plane else 3.0
    timed_s = (sum(step_ms) + sum(prof_ms)) / 1e3
    tc_peak, peak_kind = tensor_peak(peaks, mmas_per_mac, timed_s, clk.get("reasons") or [])
    sustained = peak_kind == "sustained"
    tc_burst = tensor_peak(peaks, mmas_per_mac, 0.0, [])[0]
    ridge = tc_peak * 1e12 / (hbm * 1e9)
    stages = []
    for i in sorted(per_kernel):
        r = per_kernel[i]
        avg = statistics.mean(r["ms"])
        tfl = r["flops"] / (avg / 1e3) / 1e12 if avg > 0 else 0.0
        gbs = r["bytes"] / (avg / 1e3) / 1e9 if avg > 0 else 0.0
        ai = r["flops"] / r["bytes"] if r["bytes"] else 0.0
        bound = "tensor" if (r["flops"] > 0 and ai > ridge) else "hbm"
        frac = tfl / tc_peak if bound == "tensor" else gbs / hbm
        impl = r.get("impl_bytes") or 0.0
        stages.append(dict(name=r["name"], ms=round(avg, 4), tflops=round(tfl, 2),
                           gbs=round(gbs, 1), ai=round(ai, 1), bound=bound, frac=round(frac, 3),
                           bytes=r["bytes"], impl_bytes=impl,
                           impl_gbs=round(impl / (avg / 1e3) / 1e9, 1) if avg > 0 else 0.0))
    dom = max(stages, key=lambda s: s["ms"])
    dom_rec = next(per_kernel[i] for i in per_kernel if per_kernel[i]["name"] == dom["name"])
    traffic, traffic_src = measured_traffic(args.workload, dom["name"])
    per_launch = {"flops": dom_rec["flops"], "bytes": dom_rec["bytes"],
                  "impl_bytes": dom_rec.get("impl_bytes"), "avg_ms": dom["ms"]}
    if dom["bound"] == "tensor":
        roof = {"bound": "tensor", "kernel": dom["name"], "achieved": dom["tflops"],
                "peak": round(tc_peak, 1), "unit": "TFLOP/s", "frac": dom["frac"],
                "peak_kind": peak_kind,
                "frac_of_burst": round(dom["tflops"] / tc_burst, 3),
                "traffic": traffic, "traffic_source": traffic_src, "per_launch": per_launch,
                "peak_note": (f"bf16 dense {peaks_kind} {peak_kind} / 2 (two {'f16' if f16w else 'bf16'} "
                              f"MMAs per useful MAC)" if one_plane else
                              f"bf16 dense {peaks_kind} {peak_kind} / 3 (three bf16 MMAs per useful MAC)")
                + ("; sustained: the timed steps ran >= 0.5 s under the power cap" if sustained else "")}
    else:
        roof = {"bound": "hbm", "kernel": dom["name"], "achieved": dom["gbs"], "peak": hbm,
                "unit": "GB/s", "frac": dom["frac"], "traffic": traffic,
                "traffic_source": traffic_src, "per_launch": per_launch,
                "peak_note": f"HBM copy bandwidth ({peaks_kind})"}

    line = None
    if rank == 0:
        line = {"metric": metric_of(args.workload), "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
                "ms_per_step_median": med_max,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": {"f16w": "f16w (f16 weights, f16 hi/lo activations, fp32 accumulate)",
                          "bf16w": "bf16w (bf16 weights, bf16 hi/lo activations, fp32 accumulate)",
                          "bf16x3": "bf16x3 (hi/lo split, fp32 accumulate)"}[args.precision],
                "data": "synthetic",
                "x_realtime": realtime_seconds(wl, args.workload) * world / (ms_max / 1e3),
                "config": dict(workload_config(wl, args.workload), precision=args.precision,
                               **({"stream_frames": args.stream_frames}
                                  if args.stream_frames > 0 else {})),
                "e2e": {"value": total_samples / e2e_t, "unit": UNIT,
                        "h2d_bytes_per_step": job.h2d, "d2h_bytes_per_step": job.d2h,
                        "ms_per_step": e2e_t * 1e3},
                "gpu_launches": launches * args.steps,
                "profiled_ms_per_step": statistics.mean(prof_ms),
                **({"stream": {"frames_per_call": job.F, "calls_per_step": job.n_calls,
                               "ms_per_call": statistics.median(job.call_ms),
                               "audio_ms_per_call": job.F * wl.arch.hop * 1e3 / SAMPLE_RATE[args.workload],
                               "stages_from": "whole-sequence decodes (same kernels)"}}
                   if isinstance(job, StreamJob) else {}),
                **({"stitched_samples_per_s": job.z.numel() * world / (ms_max / 1e3),
                    "stitched_track_s": realtime_seconds(wl, args.workload)}
                   if getattr(job, "z", None) is not None else {}),
                "roofline": roof,
                "clocks": clk,
                "stages": stages}
        if world == 1 and not args.no_cpu_baseline:
            frames = args.cpu_frames if args.cpu_frames is not None else (
                256 if is_encode(args.workload) else 689)
            line["cpu_baseline"] = cpu_baseline(wl, args.workload, frames)
        print(json.dumps(line), flush=True)
    job.close()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="music_long",
                    choices=sorted(W.WORKLOADS) + sorted(W.ENC_WORKLOADS))
    ap.add_argument("--cpu-frames", type=int, default=None,
                    help="latent frames of one item the CPU baseline decodes or encodes (about "
                         "10 s on 16 cores; default 689 to decode, 256 to encode)")
    ap.add_argument("--ref-frames", type=int, default=48,
                    help="latent frames of one item per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stream-frames", type=int, default=0,
                    help="decode a causal workload chunk by chunk, this many latent frames per "
                         "call (vocoder_stream_decode); 0: whole-sequence decode")
    ap.add_argument("--precision", choices=["bf16x3", "f16w", "bf16w"], default="bf16x3",
                    help="bf16x3 (default): full fp32-equivalent inputs; f16w: the pages' F16 "
                         "conv weights; bf16w: bfloat16 conv weights")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        return run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
