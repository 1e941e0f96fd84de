"""Shared helpers of the GPU parity tests: run the CUDA library and the oracle on
the same seeded inputs and compare."""
from __future__ import annotations

import functools

import numpy as np

from dac_vocoder_decode_gb300 import binding as V
from dac_vocoder_decode_gb300 import workloads as W
from oracle import oracle as O
from tests.util import frame_margins, snr_db

# Tolerance on decoded audio in [-1, 1]: max |gpu - oracle| <= 2e-3 and SNR >= 60 dB.
AUDIO_MAX_ABS = 2e-3
AUDIO_MIN_SNR_DB = 60.0


@functools.lru_cache(maxsize=8)
def workload(name: str, T=None, B=None):
    return W.make_workload(name, T=T, B=B)


@functools.lru_cache(maxsize=8)
def oracle_folded(name: str):
    return O.fold_params(workload(name).params)


def gpu_decoder(wl):
    return V.Vocoder(wl.arch, V.fold_params(wl.params))


def gpu_decode(voc, latent_np, flags=0):
    import torch
    lat = torch.from_numpy(np.ascontiguousarray(latent_np)).cuda()
    audio = voc.decode(lat, flags=flags | V.VOC_FLAG_SYNC)
    torch.cuda.synchronize()
    return audio[:, 0].cpu().numpy().astype(np.float64)


def compare_audio(ref, got, label=""):
    err = float(np.max(np.abs(ref - got)))
    snr = snr_db(ref, got)
    assert got.shape == ref.shape, (label, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), label
    assert err <= AUDIO_MAX_ABS, f"{label}: max abs err {err:.3g} > {AUDIO_MAX_ABS}"
    assert snr >= AUDIO_MIN_SNR_DB, f"{label}: SNR {snr:.1f} dB < {AUDIO_MIN_SNR_DB}"
    return err, snr


def sampled_windows(arch, T: int, n: int = 3, width: int = 8):
    """Frame windows [a, b) at the start, spread through the middle and at the end."""
    if T <= 3 * width:
        return [(0, T)]
    starts = [0] + [int(round(x)) for x in np.linspace(width, T - 2 * width, n - 2)] + [T - width]
    return [(a, min(T, a + width)) for a in starts]


def oracle_window(wl, folded, item: int, a: int, b: int):
    """Oracle output samples [a*hop, b*hop) of item `item`, computed from a latent
    slice that extends past [a, b) by the receptive field (exact: every sample
    inside only depends on frames inside the slice)."""
    left, right = frame_margins(wl.arch)
    lo = max(0, a - left - 1)
    hi = min(wl.T, b + right + 1)
    lat = W.slice_latent(wl.latent[item:item + 1], lo, hi)
    y = O.decode(wl.arch, None, lat, 0, folded)[0]
    hop = wl.arch.hop
    return y[(a - lo) * hop:(b - lo) * hop]
