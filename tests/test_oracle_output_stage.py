"""Pins of the oracle's output stage (minimaxmusic.cpp Architecture, "Post-processing"):
percentile peak normalisation targeting the 1 - peak_clip/1e6 percentile (peak_clip = 0 is
plain peak normalisation), WAV 16/24-bit PCM, and WAV 32-bit float written raw."""
from __future__ import annotations

import io
import struct
import wave

import numpy as np
import pytest

from oracle import oracle as O


@pytest.mark.parametrize("peak_clip", [0, 1, 10, 1000, 250000, 999999, 1000000])
def test_percentile_is_nearest_rank(peak_clip):
    """Against numpy's inverted-CDF percentile, which is the nearest-rank definition: the
    smallest |x| whose share of values at or below it reaches q."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal(5003).astype(np.float32)
    x[:40] = 0.75  # ties
    q = 1.0 - peak_clip / 1e6
    got = O.abs_percentile(x, peak_clip)
    ref = np.percentile(np.abs(x).astype(np.float64), 100.0 * q, method="inverted_cdf")
    assert got == ref


def test_peak_clip_zero_is_plain_peak():
    x = np.array([[0.2, -0.9, 0.4], [0.1, 0.3, -0.05]], np.float32)
    assert O.abs_percentile(x, 0) == np.float32(0.9)


def _pcm_reference(planar, bits, peak_clip):
    """Samples written with numpy float32 arithmetic and packed by the standard library."""
    x = np.asarray(planar, np.float32)
    level = np.float32(O.abs_percentile(x, peak_clip))
    with np.errstate(over="ignore"):
        gain = np.float32(1.0) / level if level > 0 else np.float32(1.0)
    gain = min(gain, np.finfo(np.float32).max)  # reciprocal of a subnormal level overflows
    full = np.float32((1 << (bits - 1)) - 1)
    y = np.clip(x * gain, np.float32(-1), np.float32(1))
    q = np.rint(y * full).astype(np.int64)  # numpy rounds half to even
    inter = q.T.ravel()  # interleave channels
    if bits == 16:
        data = inter.astype("<i2").tobytes()
    else:
        data = b"".join(int(v).to_bytes(3, "little", signed=True) for v in inter)
    buf = io.BytesIO()
    with wave.open(buf, "wb") as w:
        w.setnchannels(x.shape[0])
        w.setsampwidth(bits // 8)
        w.setframerate(44100)
        w.writeframes(data)
    return buf.getvalue()


@pytest.mark.parametrize("bits", [16, 24])
@pytest.mark.parametrize("peak_clip", [0, 50000])
def test_pcm_wav_matches_standard_library(bits, peak_clip):
    rng = np.random.default_rng(6)
    planar = (rng.standard_normal((2, 2001)) * 0.3).astype(np.float32)
    got = O.encode_wav(planar, 44100, bits, peak_clip)
    assert got == _pcm_reference(planar, bits, peak_clip)


def test_pcm_edge_values():
    """Level 1: full scale maps to 2^15 - 1, halves round to even, values beyond are clipped."""
    x = np.array([[1.0, -1.0, 0.5, -0.5, 2.0, -2.0, 0.0, 1.0 / 65534.0]], np.float32)
    wav = O.encode_wav(x, 8000, 16, peak_clip=250000)  # rank ceil(0.75 * 8) = 6: |x| = 1.0
    assert O.abs_percentile(x, 250000) == 1.0
    vals = np.frombuffer(wav[44:], dtype="<i2")
    assert vals.tolist() == [32767, -32767, 16384, -16384, 32767, -32767, 0, 0]


def test_subnormal_level_keeps_zeros_and_order():
    """All-subnormal input: 1/level overflows single precision; the largest finite gain is
    used, zeros stay zero and the loudest sample maps to round(level * FLT_MAX * 32767)."""
    k = np.array([[3, -7, 0, 12, -12, 0, 5]], np.float32)
    x = k * np.float32(1e-44)  # multiples of 2^-149 * 7 (subnormal)
    assert 0 < abs(float(x[0, 3])) < float(np.finfo(np.float32).tiny)
    wav = O.encode_wav(x, 44100, 16, 0)
    assert wav == _pcm_reference(x, 16, 0)
    # x = k * 7 * 2^-149 exactly; times FLT_MAX (about 2^128) and 32767 that is k * 0.1093:
    # 0.33, 0.77, 1.31 and 0.55 for |k| = 3, 7, 12 and 5
    vals = np.frombuffer(wav[44:], dtype="<i2")
    assert vals.tolist() == [0, -1, 0, 1, -1, 0, 1]


def test_float_wav_is_raw():
    rng = np.random.default_rng(7)
    planar = (rng.standard_normal((2, 300)) * 3.0).astype(np.float32)  # not normalised
    wav = O.encode_wav(planar, 48000, 32, peak_clip=10)
    riff, size, wavefmt, fmt_len, fmt_tag, n_ch, rate, byte_rate, align, bits = struct.unpack(
        "<4sI8sIHHIIHH", wav[:36])
    assert (riff, wavefmt, fmt_len, fmt_tag, n_ch, rate, bits) == (b"RIFF", b"WAVEfmt ", 16, 3, 2,
                                                                   48000, 32)
    assert byte_rate == 48000 * 8 and align == 8 and size == len(wav) - 8
    assert wav[36:40] == b"data" and struct.unpack("<I", wav[40:44])[0] == 2 * 300 * 4
    np.testing.assert_array_equal(np.frombuffer(wav[44:], "<f4"), planar.T.ravel())
