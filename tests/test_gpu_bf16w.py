"""GPU: the BF16-weight precision (VOC_PREC_BF16W: every conv weight rounded to bfloat16, bf16
hi/lo activations, two bf16 MMAs per K step) against the oracle run with the same
bfloat16-rounded weights, and its distance from the full-precision decoder and encoder."""
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


def _bf16_decoder(arch, params):
    return V.Vocoder(arch, V.fold_params(params), precision=V.VOC_PREC_BF16W)


@pytest.mark.parametrize("arch", [W.TINY, MID_MUSIC, MID_SPEECH,
                                  dataclasses.replace(MID_SPEECH, snake_beta=True)],
                         ids=["tiny", "music", "speech_causal", "speech_snakebeta"])
def test_bf16w_matches_bf16_weight_oracle(arch):
    wl = W.make_custom(arch, B=2, T=23, seed=404)
    got = G.gpu_decode(_bf16_decoder(arch, wl.params), wl.latent)
    ref = O.decode(arch, None, wl.latent, 0, O.fold_params(wl.params, bf16_weights=True))
    G.compare_audio(ref, got, "bf16w vs bf16-weight oracle")
    # against the full-precision decoder the 8-bit weights show (the oracle gives 35-41 dB on
    # these architectures)
    full = O.decode(arch, wl.params, wl.latent)
    assert snr_db(full, got) >= 30.0


@pytest.mark.parametrize("arch", [MID_MUSIC, MID_SPEECH], ids=["music", "speech_causal"])
def test_bf16w_every_unit_fused_matches_the_oracle(arch):
    """fuse_max_channels=192: the units of at most 128 channels, which this precision runs as
    two kernels by default, in the fused kernel's one-plane form."""
    wl = W.make_custom(arch, B=2, T=23, seed=405)
    voc = V.Vocoder(arch, V.fold_params(wl.params), fuse_max_channels=192,
                    precision=V.VOC_PREC_BF16W)
    got = G.gpu_decode(voc, wl.latent)
    ref = O.decode(arch, None, wl.latent, 0, O.fold_params(wl.params, bf16_weights=True))
    G.compare_audio(ref, got, "bf16w, every unit fused, vs bf16-weight oracle")


def test_bf16w_music_window_sampled():
    """The full-size one-window music decode, on sampled windows."""
    wl = G.workload("music_window")
    folded = O.fold_params(wl.params, bf16_weights=True)
    got = G.gpu_decode(_bf16_decoder(wl.arch, wl.params), wl.latent)
    hop = wl.arch.hop
    for item in range(wl.B):
        for (a, b) in G.sampled_windows(wl.arch, wl.T, n=3, width=8):
            ref = G.oracle_window(wl, folded, item, a, b)
            G.compare_audio(ref, got[item, a * hop:b * hop], f"bf16w music[{item}][{a}:{b}]")


def test_bf16w_stream_equals_whole_decode():
    wl = W.make_custom(MID_SPEECH, B=2, T=19, seed=81)
    voc = _bf16_decoder(MID_SPEECH, wl.params)
    whole = G.gpu_decode(voc, wl.latent)
    s = V.VocoderStream(voc, 2, 8)
    lat = torch.from_numpy(np.ascontiguousarray(wl.latent)).cuda()
    outs, t = [], 0
    for n in [1, 2, 8, 3, 5]:
        outs.append(s.decode(lat[:, :, t:t + n].contiguous(), flags=V.VOC_FLAG_SYNC))
        t += n
    got = torch.cat(outs, dim=2)[:, 0].cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(got, whole)


def test_bf16w_encoder():
    """The mirror encoder in the BF16-weight precision against the oracle encoder with the same
    rounded weights (odd strides and a stride-1 block included)."""
    from tests.test_gpu_encoder import CASES, compare, gpu_encode
    for name in ("small", "odd_strides"):
        arch, B, frames, seed = CASES[name]
        wl = W.make_encode_workload(arch, B, frames, seed)
        ref = O.encode(arch, wl.params, wl.latent,
                       folded=O.fold_params(wl.params, bf16_weights=True))
        enc = V.Encoder(arch, V.fold_params(wl.params), precision=V.VOC_PREC_BF16W)
        got = gpu_encode(enc, wl.latent)
        compare(ref, got, f"bf16w {name}")
        assert snr_db(O.encode(arch, wl.params, wl.latent), got) >= 30.0
        enc.close()
