"""Benchmark of the vocoder decode on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload music_window]

One step = one full decode (every layer of the decoder) of one batch of the
workload's synthetic latents, already resident in HBM.  Each timed step is
bracketed by CUDA events on the decode stream; a 256 MiB buffer (larger than the
129 MB L2) is written between timed steps, outside the events.  Several ranks
(torchrun, one GPU each) decode independent copies of the workload: weak
scaling with no collective on the data path (a scalar max-reduction of the step
time only).  Rank 0 prints one JSON line.

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
UNIT = "samples/s"
SAMPLE_RATE = {"music_window": 44100, "music_batch8": 44100, "music_long": 44100, "speech": 24000,
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


def measured_traffic(workload: str, layer: str):
    """DRAM bytes (read + write) of one launch of `layer`, from the ncu summary committed
    under profiles/, or None when there is none or it was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.md")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        text = f.read()
    if f"source hash: {source_hash()}" not in text:
        return None
    for ln in text.splitlines():
        cells = [c.strip() for c in ln.strip().strip("|").split("|")]
        if len(cells) >= 4 and cells[0] == layer:
            try:
                return int(cells[3])
            except ValueError:
                return None
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


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
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
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


# ----------------------------------------------------------------------------- CPU legs
def oracle_sample(wl, frames: int, folded=None):
    """Time the oracle on one item's first `frames` latent frames (bounded CPU work)."""
    from oracle import oracle as O
    if folded is None:
        folded = O.fold_params(wl.params)
    lat = W.slice_latent(wl.latent[:1], 0, min(frames, wl.T))
    t0 = time.perf_counter()
    y = O.decode(wl.arch, None, lat, 0, folded)
    dt = time.perf_counter() - t0
    return y.size, dt, folded


def cpu_threads():
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n and n.isdigit() else (os.cpu_count() or 1)


def cpu_baseline(wl, name, frames):
    samples, dt, _ = oracle_sample(wl, frames)
    return {"value": samples / dt, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
            "sample": f"1 item x {min(frames, wl.T)} latent frames of {name} "
                      f"({samples} samples) decoded in {dt:.2f} s (fp64 direct loops, OpenMP)"}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    wl = W.make_workload(args.workload)
    frames = args.ref_frames
    folded = None
    for _ in range(args.warmup):
        _, _, folded = oracle_sample(wl, frames, folded)
    times = []
    samples = 0
    for _ in range(args.steps):
        samples, dt, folded = oracle_sample(wl, frames, folded)
        times.append(dt)
    ms = 1e3 * statistics.mean(times)
    value = samples / (ms / 1e3)
    rate = SAMPLE_RATE[args.workload]
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "x_realtime": value / rate / (2.0 if args.workload.startswith("music") else 1.0),
            "config": config_of(wl, args.workload),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(),
                             "kind": "oracle",
                             "sample": f"each step: 1 item x {min(frames, wl.T)} latent frames "
                                       f"of {args.workload} ({samples} samples)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU leg
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from dac_vocoder_decode_gb300 import binding as V

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks, peaks_kind = load_peaks()
    wl = W.make_workload(args.workload)
    f16w = args.precision == "f16w"
    voc = V.Vocoder(wl.arch, V.fold_params(wl.params),
                    precision=V.VOC_PREC_F16W if f16w else V.VOC_PREC_BF16X3)
    B, T, hop = wl.B, wl.T, wl.arch.hop
    stream = torch.cuda.Stream(device=dev)
    lat = torch.from_numpy(wl.latent).to(dev)
    audio = torch.empty((B, 1, T * hop), dtype=torch.float32, device=dev)
    ws = voc.alloc_workspace(B, T)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            V.vocoder_decode(voc.handle, lat, audio, ws, stream)
    torch.cuda.synchronize()

    launches = V.vocoder_launches_per_decode(voc.handle, B, T)
    per_kernel = {}
    step_ms = []
    clocks = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            flush.fill_(1.0)  # evict the previous step's data from L2 (not timed)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            V.vocoder_decode(voc.handle, lat, audio, ws, stream, V.VOC_FLAG_PROFILE)
            e1.record(stream)
            e1.synchronize()
            step_ms.append(e0.elapsed_time(e1))
            for i, p in enumerate(V.vocoder_profile(voc.handle)):
                rec = per_kernel.setdefault(i, dict(name=p["name"], ms=[], flops=p["flops"],
                                                    bytes=p["bytes"]))
                rec["ms"].append(p["ms"])
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, dev)
    total_samples = B * T * hop * world
    value = total_samples / (ms_max / 1e3)

    # end to end through the host-buffer entry point: H2D of the latent, decode, D2H of the audio
    lat_h = torch.from_numpy(wl.latent).pin_memory()
    aud_h = torch.empty((B, 1, T * hop), dtype=torch.float32).pin_memory()
    ws_h = voc.alloc_workspace(B, T, host_io=True)
    for _ in range(max(1, args.warmup)):
        V.vocoder_decode_host(voc.handle, lat_h, aud_h, ws_h, stream)
    e2e_s = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        V.vocoder_decode_host(voc.handle, lat_h, aud_h, ws_h, stream)
        e2e_s.append(time.perf_counter() - t0)
    e2e_t = max_over_ranks(statistics.mean(e2e_s), dev)

    # per-kernel roofline: bf16x3 issues three bf16 MMAs per useful multiply-add
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    # bf16x3 issues three bf16 MMAs per useful multiply-add, f16w two f16 MMAs (f16 and bf16
    # share the dense tensor rate)
    mmas_per_mac = 2.0 if f16w else 3.0
    tc_peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]) / mmas_per_mac
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
        stages.append(dict(name=r["name"], ms=round(avg, 4), tflops=round(tfl, 2),
                           gbs=round(gbs, 1), ai=round(ai, 1), bound=bound, frac=round(frac, 3)))
    dom = max(stages, key=lambda s: s["ms"])
    dom_rec = next(per_kernel[i] for i in per_kernel if per_kernel[i]["name"] == dom["name"])
    traffic = measured_traffic(args.workload, dom["name"])
    if dom["bound"] == "tensor":
        roof = {"bound": "tensor", "kernel": dom["name"], "achieved": dom["tflops"],
                "peak": round(tc_peak, 1), "unit": "TFLOP/s", "frac": dom["frac"],
                "traffic": traffic,
                "per_launch": {"flops": dom_rec["flops"], "bytes": dom_rec["bytes"],
                               "avg_ms": dom["ms"]},
                "peak_note": (f"bf16 dense {peaks_kind} burst / 2 (two f16 MMAs per useful MAC)"
                              if f16w else
                              f"bf16 dense {peaks_kind} burst / 3 (three bf16 MMAs per useful MAC)")}
    else:
        roof = {"bound": "hbm", "kernel": dom["name"], "achieved": dom["gbs"], "peak": hbm,
                "unit": "GB/s", "frac": dom["frac"], "traffic": traffic,
                "per_launch": {"flops": dom_rec["flops"], "bytes": dom_rec["bytes"],
                               "avg_ms": dom["ms"]},
                "peak_note": f"HBM copy bandwidth ({peaks_kind})"}

    line = None
    if rank == 0:
        rate = SAMPLE_RATE[args.workload]
        tracks = tracks_per_batch(args.workload, B) * world
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": ("f16w (f16 weights, f16 hi/lo activations, fp32 accumulate)" if f16w
                          else "bf16x3 (hi/lo split, fp32 accumulate)"), "data": "synthetic",
                "x_realtime": tracks * T * hop / rate / (ms_max / 1e3),
                "config": dict(config_of(wl, args.workload), precision=args.precision),
                "e2e": {"value": total_samples / e2e_t, "unit": UNIT,
                        "h2d_bytes_per_step": int(wl.latent.nbytes),
                        "d2h_bytes_per_step": int(B * T * hop * 4),
                        "ms_per_step": e2e_t * 1e3},
                "gpu_launches": launches * args.steps,
                "roofline": roof,
                "clocks": clk,
                "stages": stages}
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl, args.workload, args.cpu_frames)
        print(json.dumps(line), flush=True)
    voc.close()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="music_window", choices=sorted(W.WORKLOADS))
    ap.add_argument("--cpu-frames", type=int, default=689,
                    help="latent frames of one item the CPU baseline decodes (about 10 s on 16 cores)")
    ap.add_argument("--ref-frames", type=int, default=48,
                    help="latent frames of one item per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--precision", choices=["bf16x3", "f16w"], default="bf16x3",
                    help="bf16x3 (default): full fp32-equivalent inputs; f16w: the pages' F16 "
                         "conv weights")
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
