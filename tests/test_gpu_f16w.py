"""GPU: the F16-weight precision (VOC_PREC_F16W; minimaxmusic.cpp Architecture, "Flow VAE":
conv weights stored F16 on the device with F32 activations) against the oracle run with the
same half-precision weights, and its distance from the full-precision decoder."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("no CUDA device", allow_module_level=True)

from dac_vocoder_decode_gb300 import binding as V  # noqa: E402
from dac_vocoder_decode_gb300 import workloads as W  # noqa: E402
from oracle import oracle as O  # noqa: E402
from tests import gpu_common as G  # noqa: E402
from tests.util import snr_db  # noqa: E402

MID_MUSIC = W.Arch(latent_channels=64, channels0=384, strides=(8, 8, 4, 2), widths=(192, 96, 96, 48))
MID_SPEECH = W.Arch(latent_channels=64, channels0=256, strides=(8, 5, 4, 4, 3),
                    widths=(192, 96, 48, 48, 32), padding=W.PAD_CAUSAL)


def _f16_decoder(arch, params):
    return V.Vocoder(arch, V.fold_params(params), precision=V.VOC_PREC_F16W)


@pytest.mark.parametrize("arch", [W.TINY, MID_MUSIC, MID_SPEECH,
                                  dataclasses.replace(MID_SPEECH, snake_beta=True)],
                         ids=["tiny", "music", "speech_causal", "speech_snakebeta"])
def test_f16w_matches_f16_weight_oracle(arch):
    wl = W.make_custom(arch, B=2, T=23, seed=404)
    got = G.gpu_decode(_f16_decoder(arch, wl.params), wl.latent)
    ref = O.decode(arch, None, wl.latent, 0, O.fold_params(wl.params, f16_weights=True))
    G.compare_audio(ref, got, "f16w vs f16-weight oracle")
    # the activations carry about 22 bits: well inside the bf16x3 tolerance
    assert snr_db(ref, got) >= 80.0
    # against the full-precision decoder the weights' rounding shows
    full = O.decode(arch, wl.params, wl.latent)
    assert snr_db(full, got) >= 40.0


@pytest.mark.parametrize("arch", [MID_MUSIC, MID_SPEECH], ids=["music", "speech_causal"])
def test_f16w_every_unit_fused_matches_the_oracle(arch):
    """fuse_max_channels=192: the units of at most 128 channels, which this precision runs as
    two kernels by default, in the fused kernel's one-plane form."""
    wl = W.make_custom(arch, B=2, T=23, seed=405)
    voc = V.Vocoder(arch, V.fold_params(wl.params), fuse_max_channels=192,
                    precision=V.VOC_PREC_F16W)
    got = G.gpu_decode(voc, wl.latent)
    ref = O.decode(arch, None, wl.latent, 0, O.fold_params(wl.params, f16_weights=True))
    G.compare_audio(ref, got, "f16w, every unit fused, vs f16-weight oracle")
    assert snr_db(ref, got) >= 80.0


def test_f16w_music_window_sampled():
    """The full-size one-window music decode, on sampled windows."""
    wl = G.workload("music_window")
    folded = O.fold_params(wl.params, f16_weights=True)
    got = G.gpu_decode(_f16_decoder(wl.arch, wl.params), wl.latent)
    hop = wl.arch.hop
    for item in range(wl.B):
        for (a, b) in G.sampled_windows(wl.arch, wl.T, n=3, width=8):
            ref = G.oracle_window(wl, folded, item, a, b)
            G.compare_audio(ref, got[item, a * hop:b * hop], f"f16w music[{item}][{a}:{b}]")


def test_f16w_stream_equals_whole_decode():
    arch = W.Arch(latent_channels=64, channels0=256, strides=(8, 5, 4, 4, 3),
                  widths=(192, 96, 48, 48, 32), padding=W.PAD_CAUSAL)
    wl = W.make_custom(arch, B=2, T=19, seed=81)
    voc = _f16_decoder(arch, wl.params)
    whole = G.gpu_decode(voc, wl.latent)
    s = V.VocoderStream(voc, 2, 8)
    lat = torch.from_numpy(np.ascontiguousarray(wl.latent)).cuda()
    outs, t = [], 0
    for n in [1, 2, 8, 3, 5]:
        outs.append(s.decode(lat[:, :, t:t + n].contiguous(), flags=V.VOC_FLAG_SYNC))
        t += n
    got = torch.cat(outs, dim=2)[:, 0].cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(got, whole)
