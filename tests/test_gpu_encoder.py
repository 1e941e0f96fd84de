"""GPU parity of the mirror encoder (minimaxmusic.cpp Architecture, "Flow VAE": conv_in,
blocks of residual units followed by Snake and a strided conv k = 2s, Snake, conv_out k3,
posterior mean projection k1), called through the C ABI, against the CPU oracle.

Small architectures run in full: several 128-row tiles at the audio rate, ragged tails,
odd strides (3, 5), a stride-1 block, two audio channels, SnakeBeta, and the F16-weight
precision (against the oracle with the same f16-rounded weights).  The published music
encoder runs in full on a short clip and, on a stereo 689-frame window, on sampled latent
frames that the oracle computes exactly from audio slices covering their receptive field.

Tolerance: the latents are O(1) (max |z| about 1.5 with the calibrated parameters), and the
encoder runs the decoder's arithmetic, so it is held to the decoder's audio bound scaled by
the latent's magnitude: max |gpu - oracle| <= 2e-3 * max(1, max |oracle|) and SNR >= 60 dB."""
from __future__ import annotations

import dataclasses
import functools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("no CUDA device", allow_module_level=True)

from dac_vocoder_decode_gb300 import binding as V  # noqa: E402
from dac_vocoder_decode_gb300 import workloads as W  # noqa: E402
from oracle import oracle as O  # noqa: E402
from tests.util import encoder_frame_margins, snr_db  # noqa: E402

MAX_ABS = 2e-3
MIN_SNR_DB = 60.0

SMALL = W.EncArch(1, 16, (2, 4), (32, 48), 8)
ODD = W.EncArch(2, 24, (3, 5, 1), (40, 56, 56), 12, dilations=(1, 3))
WIDE = W.EncArch(1, 48, (4, 2), (96, 200), 20)  # 200 channels: two column tiles, padded
# more audio channels than the direct fp32 conv_in takes (4): conv_in as a tensor-core GEMM
MULTI = W.EncArch(6, 16, (2, 4), (32, 48), 8)

CASES = {
    # name: (arch, B, frames, seed)
    "small": (SMALL, 2, 40, 11),
    "small_ragged": (SMALL, 3, 13, 12),
    "odd_strides": (ODD, 2, 30, 13),
    "wide": (WIDE, 1, 50, 14),
    "snake_beta": (dataclasses.replace(SMALL, snake_beta=True), 2, 21, 15),
    "music_short": (W.ENC_MUSIC, 1, 24, 16),
    "six_channels": (MULTI, 2, 20, 17),
}


def compare(ref, got, label):
    assert got.shape == ref.shape, (label, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), label
    err = float(np.max(np.abs(ref - got)))
    bound = MAX_ABS * max(1.0, float(np.max(np.abs(ref))))
    snr = snr_db(ref, got)
    assert err <= bound, f"{label}: max abs err {err:.3g} > {bound:.3g}"
    assert snr >= MIN_SNR_DB, f"{label}: SNR {snr:.1f} dB < {MIN_SNR_DB}"
    return err, snr


def gpu_encode(enc, audio_np, flags=0):
    audio = torch.from_numpy(np.ascontiguousarray(audio_np)).cuda()
    z = enc.encode(audio, flags=flags | V.VOC_FLAG_SYNC)
    torch.cuda.synchronize()
    return z.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name", list(CASES))
def test_encode_matches_oracle(name):
    arch, B, frames, seed = CASES[name]
    wl = W.make_encode_workload(arch, B, frames, seed)
    ref = O.encode(arch, wl.params, wl.latent)
    enc = V.Encoder(arch, V.fold_params(wl.params))
    got = gpu_encode(enc, wl.latent)
    compare(ref, got, name)
    enc.close()


def test_encode_f16_weights():
    """VOC_PREC_F16W against the oracle with every conv weight rounded to half precision."""
    arch, B, frames, seed = CASES["small"]
    wl = W.make_encode_workload(arch, B, frames, seed)
    ref = O.encode(arch, wl.params, wl.latent, folded=O.fold_params(wl.params, f16_weights=True))
    enc = V.Encoder(arch, V.fold_params(wl.params), precision=V.VOC_PREC_F16W)
    compare(ref, gpu_encode(enc, wl.latent), "f16w")
    enc.close()


def test_encode_is_deterministic_and_reuses_workspace():
    arch, B, frames, seed = CASES["small"]
    wl = W.make_encode_workload(arch, B, frames, seed)
    enc = V.Encoder(arch, V.fold_params(wl.params))
    audio = torch.from_numpy(wl.latent).cuda()
    ws = enc.alloc_workspace(B, audio.shape[2])
    z1 = enc.encode(audio, ws=ws, flags=V.VOC_FLAG_SYNC).clone()
    # another length through the same context rebuilds its descriptors, then back again
    short = audio[:, :, : 5 * enc.hop].contiguous()
    enc.encode(short, flags=V.VOC_FLAG_SYNC)
    z2 = enc.encode(audio, ws=ws, flags=V.VOC_FLAG_SYNC)
    torch.cuda.synchronize()
    assert torch.equal(z1, z2)
    enc.close()


def test_encode_rejects_bad_lengths_and_workspace():
    arch, B, frames, seed = CASES["small"]
    wl = W.make_encode_workload(arch, B, frames, seed)
    enc = V.Encoder(arch, V.fold_params(wl.params))
    assert enc.workspace_bytes(B, enc.hop * frames + 1) == 0
    assert enc.workspace_bytes(B, 0) == 0 and enc.workspace_bytes(0, enc.hop) == 0
    audio = torch.zeros((B, 1, enc.hop * 4 + 3), device="cuda")
    z = torch.empty((B, arch.latent_channels, 4), device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(V.VocoderError) as e:
        V.vocoder_encode(enc.handle, audio, z, ws)
    assert e.value.status == V.VOC_INVALID_ARG
    for empty in (audio[:, :, :0], audio[:0]):  # no samples, no items
        with pytest.raises(V.VocoderError) as e:
            V.vocoder_encode(enc.handle, empty, z, ws)
        assert e.value.status == V.VOC_INVALID_ARG
    audio = torch.zeros((B, 1, enc.hop * 4), device="cuda")
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(V.VocoderError) as e:
        V.vocoder_encode(enc.handle, audio, z, small)
    assert e.value.status == V.VOC_WORKSPACE_TOO_SMALL
    enc.close()


def test_encode_profile_records_every_launch():
    arch, B, frames, seed = CASES["small"]
    wl = W.make_encode_workload(arch, B, frames, seed)
    enc = V.Encoder(arch, V.fold_params(wl.params))
    gpu_encode(enc, wl.latent, flags=V.VOC_FLAG_PROFILE)
    prof = V.vocoder_encoder_profile(enc.handle)
    assert len(prof) == V.vocoder_encoder_launches(enc.handle, B, wl.latent.shape[2])
    names = [p["name"] for p in prof]
    # one audio channel: conv_in runs directly on the audio (no hi/lo preparation launch)
    assert names[0] == "conv_in" and names[-1] == "latent_out"
    assert "b0.down" in names and "b1.down" in names
    assert all(p["ms"] >= 0 for p in prof)
    enc.close()
    # six audio channels: the audio is prepared as hi/lo planes for the conv_in GEMM
    arch, B, frames, seed = CASES["six_channels"]
    wl = W.make_encode_workload(arch, B, frames, seed)
    enc = V.Encoder(arch, V.fold_params(wl.params))
    gpu_encode(enc, wl.latent, flags=V.VOC_FLAG_PROFILE)
    names = [p["name"] for p in V.vocoder_encoder_profile(enc.handle)]
    assert names[0] == "prep_audio" and names[1] == "conv_in"
    assert len(names) == V.vocoder_encoder_launches(enc.handle, B, wl.latent.shape[2])
    enc.close()


# ----------------------------------------------------------------------------- full size
MUSIC_WINDOW_FRAMES = 689  # one decode window of the music pipeline: [2, 1, 689 * 512] audio


@functools.lru_cache(maxsize=1)
def music_window():
    wl = W.make_named_encode_workload("encode_music_window")  # the bench's encoder workload
    assert wl.latent.shape == (2, 1, MUSIC_WINDOW_FRAMES * W.ENC_MUSIC.hop)
    return wl


def test_music_window_sampled_frames():
    """A stereo 689-frame window (2 x 352768 samples), encoded in one call as the bench times
    it; latent frames at the start, the middle and the end against the oracle run on audio
    slices that hold each window's receptive field."""
    wl = music_window()
    arch = W.ENC_MUSIC
    hop = arch.hop
    enc = V.Encoder(arch, V.fold_params(wl.params))
    got = gpu_encode(enc, wl.latent)
    enc.close()
    T = MUSIC_WINDOW_FRAMES
    assert got.shape == (2, arch.latent_channels, T)
    ml, mr = encoder_frame_margins(arch)
    folded = O.fold_params(wl.params)
    for item, (a, b) in [(0, (0, 6)), (1, (340, 346)), (0, (T - 6, T)), (1, (T - 6, T))]:
        f0, f1 = max(0, a - ml), min(T, b + mr)
        piece = np.ascontiguousarray(wl.latent[item:item + 1, :, f0 * hop:f1 * hop])
        ref = O.encode(arch, None, piece, folded=folded)[0, :, a - f0:b - f0]
        compare(ref, got[item, :, a:b], f"item {item} frames [{a}, {b})")


def test_encode_host_matches_device_encode():
    """vocoder_encode_host (pinned host buffers, copies inside the call) gives the device
    entry point's latents bit for bit."""
    arch, B, frames, seed = CASES["odd_strides"]
    wl = W.make_encode_workload(arch, B, frames, seed)
    enc = V.Encoder(arch, V.fold_params(wl.params))
    z_dev = gpu_encode(enc, wl.latent)
    audio_h = torch.from_numpy(wl.latent).pin_memory()
    z_h = torch.empty((B, arch.latent_channels, frames), dtype=torch.float32).pin_memory()
    ws = enc.alloc_workspace(B, audio_h.shape[2], host_io=True)
    V.vocoder_encode_host(enc.handle, audio_h, z_h, ws)
    assert np.array_equal(z_h.numpy().astype(np.float64), z_dev)
    enc.close()
