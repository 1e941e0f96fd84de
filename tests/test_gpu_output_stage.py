"""GPU: the output stage after the stitch (minimaxmusic.cpp Architecture, "Post-processing"):
percentile peak normalisation and WAV encoding on the device, compared byte for byte with
the oracle's encoder on the same planar input.  The normalisation level (an exact order
statistic of |x|) is also read back from the encoder's scratch and compared with the oracle's
percentile."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("no CUDA device", allow_module_level=True)

from dac_vocoder_decode_gb300 import binding as V  # noqa: E402
from oracle import oracle as O  # noqa: E402
from tests import gpu_common as G  # noqa: E402

SR = 44100


def _gpu_wav(planar: np.ndarray, bits: int, peak_clip: int, sr: int = SR):
    """Encode on the device; returns (file bytes, level read from the select state)."""
    x = torch.from_numpy(np.ascontiguousarray(planar, dtype=np.float32)).cuda()
    n_ch, n = x.shape
    size = V.vocoder_wav_bytes(n_ch, n, bits)
    scratch = torch.zeros(V.vocoder_wav_scratch_bytes(), dtype=torch.uint8, device="cuda")
    out = torch.full((size,), 0xA5, dtype=torch.uint8, device="cuda")
    V.vocoder_encode_wav(x, sr, bits, peak_clip, out, scratch)
    torch.cuda.synchronize()
    # select state: k (u64), prefix (u32), mask (u32), level (f32), gain (f32)
    level = float(scratch[16:20].cpu().numpy().view(np.float32)[0])
    return out.cpu().numpy().tobytes(), level


def _signal(n_ch: int, n: int, seed: int, kind: str) -> np.ndarray:
    rng = np.random.default_rng(seed)
    if kind == "tanh":  # the decoder's output range
        return np.tanh(rng.standard_normal((n_ch, n)) * 0.7).astype(np.float32)
    if kind == "loud":  # beyond [-1, 1]: clamped after normalisation only if clipped
        return (rng.standard_normal((n_ch, n)) * 3.0).astype(np.float32)
    if kind == "ties":  # few distinct magnitudes: the rank falls inside runs of equal values
        return (rng.integers(-6, 7, (n_ch, n)) / 8.0).astype(np.float32)
    if kind == "tiny":  # subnormal magnitudes (the gain's reciprocal overflows), signed zeros
        v = rng.integers(-40, 41, (n_ch, n)).astype(np.float32) * np.float32(1e-44)
        v[:, ::7] = -0.0
        return v
    raise ValueError(kind)


@pytest.mark.parametrize("bits", [16, 24, 32])
@pytest.mark.parametrize("peak_clip", [0, 10, 1000, 250000])
@pytest.mark.parametrize("n_ch,n,kind", [(1, 100003, "tanh"), (2, 65537, "loud"),
                                         (2, 40001, "ties"), (3, 999, "tiny")])
def test_encode_wav_matches_oracle(bits, peak_clip, n_ch, n, kind):
    x = _signal(n_ch, n, seed=1000 + n + bits + peak_clip, kind=kind)
    got, level = _gpu_wav(x, bits, peak_clip)
    ref = O.encode_wav(x, SR, bits, peak_clip)
    assert len(got) == len(ref) == 44 + n_ch * n * bits // 8
    assert got == ref
    if bits != 32:
        assert level == O.abs_percentile(x, peak_clip)


@pytest.mark.parametrize("n", [0, 1, 2, 255, 256, 257])
def test_encode_wav_short_inputs(n):
    x = _signal(2, n, seed=77 + n, kind="tanh")
    for bits in (16, 24, 32):
        got, _ = _gpu_wav(x, bits, 0)
        assert got == O.encode_wav(x, SR, bits, 0)


def test_encode_wav_all_zero_and_constant():
    z = np.zeros((2, 5000), dtype=np.float32)
    got, level = _gpu_wav(z, 16, 0)
    assert level == 0.0 and got == O.encode_wav(z, SR, 16, 0)
    c = np.full((1, 5000), -0.3, dtype=np.float32)
    got, level = _gpu_wav(c, 24, 1000)
    assert level == np.float32(0.3) and got == O.encode_wav(c, SR, 24, 1000)


def test_stitched_music_to_wav():
    """The windowed music workload end to end: decode, stitch, encode (16-bit, with the
    pages' clipping percentile form), against the oracle's encoder of the stitched audio."""
    wl = G.workload("music_batch8")
    st = wl.stitch
    voc = G.gpu_decoder(wl)
    audio = voc.decode(torch.from_numpy(wl.latent).cuda(), flags=V.VOC_FLAG_SYNC)
    n = V.vocoder_stitched_length(st["n_win"], st["win_frames"], st["crop_left"],
                                  st["crop_right"], st["hop"])
    out = torch.empty((st["n_sides"], n), dtype=torch.float32, device="cuda")
    V.vocoder_stitch(audio, st["n_win"], st["n_sides"], st["win_frames"], st["crop_left"],
                     st["crop_right"], st["hop"], out)
    for bits, clip in ((16, 10), (24, 0)):  # 10: the pages' default peak_clip
        wav = V.encode_wav(out, SR, bits, clip)
        torch.cuda.synchronize()
        ref = O.encode_wav(out.cpu().numpy(), SR, bits, clip)
        assert wav.cpu().numpy().tobytes() == ref


def test_encode_wav_rejections():
    x = torch.zeros((1, 64), dtype=torch.float32, device="cuda")
    out = torch.empty(V.vocoder_wav_bytes(1, 64, 16), dtype=torch.uint8, device="cuda")
    scratch = torch.empty(V.vocoder_wav_scratch_bytes(), dtype=torch.uint8, device="cuda")
    with pytest.raises(V.VocoderError, match="VOC_INVALID_ARG"):
        V.vocoder_encode_wav(x, SR, 20, 0, out, scratch)
    with pytest.raises(V.VocoderError, match="VOC_INVALID_ARG"):
        V.vocoder_encode_wav(x, SR, 16, 1000001, out, scratch)
    with pytest.raises(V.VocoderError, match="VOC_INVALID_ARG"):
        V.vocoder_encode_wav(x, 0, 16, 0, out, scratch)
    with pytest.raises(V.VocoderError, match="VOC_WORKSPACE_TOO_SMALL"):
        V.vocoder_encode_wav(x, SR, 16, 0, out[:-1], scratch)
    with pytest.raises(V.VocoderError, match="VOC_WORKSPACE_TOO_SMALL"):
        V.vocoder_encode_wav(x, SR, 16, 0, out, scratch[:100])
    with pytest.raises(V.VocoderError, match="VOC_INVALID_ARG"):
        V.vocoder_encode_wav(x, SR, 16, 0, out[1:], scratch)  # misaligned file
