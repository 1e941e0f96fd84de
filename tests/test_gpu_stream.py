"""GPU: stateful streaming decode of causal decoders (qwentts.cpp Architecture, "Streaming
decode (stateful path)"): a sequence decoded chunk by chunk, down to one latent frame at a
time, must equal the decode of the whole sequence bit for bit, and so match the oracle
within the decode tolerance."""
from __future__ import annotations

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

# causal; strides 8, 5, 4, 4, 3 as in the speech codec; every residual unit (at most 192
# channels) runs as one fused kernel by default, as two kernels with fuse_max_channels=-1
MID_CAUSAL = W.Arch(latent_channels=64, channels0=256, strides=(8, 5, 4, 4, 3),
                    widths=(192, 96, 48, 48, 32), padding=W.PAD_CAUSAL)
MID_CAUSAL_PROJ = W.Arch(latent_channels=64, channels0=256, strides=(8, 5, 4, 4, 3),
                         widths=(192, 96, 48, 48, 32), padding=W.PAD_CAUSAL, in_proj_channels=128)


def _stream(voc, latent, chunks, max_frames, stream_obj=None):
    B, _, T = latent.shape
    assert sum(chunks) == T
    s = stream_obj or V.VocoderStream(voc, B, max_frames)
    lat = torch.from_numpy(np.ascontiguousarray(latent)).cuda()
    outs, t = [], 0
    for n in chunks:
        outs.append(s.decode(lat[:, :, t:t + n].contiguous(), flags=V.VOC_FLAG_SYNC))
        t += n
    torch.cuda.synchronize()
    return torch.cat(outs, dim=2)[:, 0].cpu().numpy().astype(np.float64), s


@pytest.mark.parametrize("arch,cta_pair,fuse", [(MID_CAUSAL, 0, 0), (MID_CAUSAL, 1, 0),
                                                (MID_CAUSAL_PROJ, 0, 0), (MID_CAUSAL, 0, -1)],
                         ids=["mid", "mid_cta_pair", "mid_in_proj", "mid_two_kernel_units"])
def test_stream_equals_whole_decode(arch, cta_pair, fuse):
    wl = W.make_custom(arch, B=2, T=37, seed=81)
    voc = V.Vocoder(arch, V.fold_params(wl.params), cta_pair=cta_pair, fuse_max_channels=fuse)
    whole = G.gpu_decode(voc, wl.latent)
    got, _ = _stream(voc, wl.latent, [1, 1, 2, 5, 8, 3, 8, 8, 1], max_frames=8)
    assert got.shape == whole.shape
    np.testing.assert_array_equal(got, whole)
    G.compare_audio(O.decode(arch, wl.params, wl.latent), got, "stream vs oracle")


def test_stream_speech_one_frame_at_a_time():
    """The 24 kHz speech decoder (1024 latent channels, hop 1920), one frame per call."""
    wl = G.workload("speech", T=24, B=2)
    voc = G.gpu_decoder(wl)
    whole = G.gpu_decode(voc, wl.latent)
    got, _ = _stream(voc, wl.latent, [1] * 24, max_frames=1)
    np.testing.assert_array_equal(got, whole)


def test_stream_reset_starts_a_new_sequence():
    wl = W.make_custom(MID_CAUSAL, B=1, T=12, seed=82)
    voc = V.Vocoder(MID_CAUSAL, V.fold_params(wl.params))
    first, s = _stream(voc, wl.latent, [4, 4, 4], max_frames=4)
    s.reset()
    again, _ = _stream(voc, wl.latent, [3, 3, 3, 3], max_frames=4, stream_obj=s)
    np.testing.assert_array_equal(first, again)
    # without the reset the contexts carry over and the start differs
    other, _ = _stream(voc, wl.latent, [4, 4, 4], max_frames=4, stream_obj=s)
    assert np.max(np.abs(other - first)) > 0


def test_stream_rejections():
    wl = W.make_custom(MID_CAUSAL, B=1, T=4, seed=83)
    voc = V.Vocoder(MID_CAUSAL, V.fold_params(wl.params))
    s = V.VocoderStream(voc, 1, 2)
    lat = torch.from_numpy(wl.latent).cuda()
    for frames in (3, 0):  # more than max_frames, none
        with pytest.raises(V.VocoderError) as e:
            V.vocoder_stream_decode(voc.handle, s.handle, lat[:, :, :frames],
                                    torch.empty((1, 1, 3 * voc.hop), device="cuda"))
        assert e.value.status == V.VOC_INVALID_ARG
    music = G.workload("tiny")
    vm = G.gpu_decoder(music)
    with pytest.raises(V.VocoderError) as e:
        V.VocoderStream(vm, 1, 4)
    assert e.value.status == V.VOC_UNSUPPORTED
