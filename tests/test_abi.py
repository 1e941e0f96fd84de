"""C-ABI checks that need no GPU: the library loads, exports exactly the symbols
the header declares, a plain C99 program consumes the header and every entry
point's validation path, and the host-side helpers agree with the layer shapes
and with the oracle's weight-norm fold."""
from __future__ import annotations

import ctypes
import dataclasses
import os
import re
import subprocess

import numpy as np
import pytest

from dac_vocoder_decode_gb300 import binding as V
from dac_vocoder_decode_gb300 import build as B
from dac_vocoder_decode_gb300 import workloads as W
from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vocoder.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return V.load_library()


def declared_symbols():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(vocoder_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(V.EXPORTED) == names


def test_exports_nothing_else(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True,
                         check=True).stdout
    syms = [ln.split()[-1] for ln in out.splitlines() if " T " in ln]
    extra = [s for s in syms if not s.startswith("vocoder_")]
    assert not extra, extra[:10]


def test_c99_consumer(lib, tmp_path):
    exe = str(tmp_path / "abi_c")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "abi_c.c"),
           "-L", os.path.dirname(B.LIB), "-lvocoder", "-Wl,-rpath," + os.path.dirname(B.LIB),
           "-o", exe]
    subprocess.run(cmd, check=True)
    res = subprocess.run([exe], capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    assert "abi_c ok" in res.stdout


@pytest.mark.parametrize("arch", [W.TINY, W.MUSIC, W.SPEECH, W.MUSIC_FULL,
                                  dataclasses.replace(W.SPEECH, snake_beta=True)],
                         ids=["tiny", "music", "speech", "music_full", "speech_snake_beta"])
def test_param_shapes_match_layer_list(lib, arch):
    shapes = arch.param_shapes()
    assert V.vocoder_param_count(arch) == len(shapes)
    for i, (_name, shape) in enumerate(shapes):
        assert V.vocoder_param_shape(arch, i) == shape


def test_fold_matches_oracle(lib):
    rng = np.random.default_rng(3)
    for shape in [(8, 4, 7), (4, 8, 16), (1, 96, 7)]:
        v = rng.standard_normal(shape).astype(np.float32)
        g = rng.uniform(0.5, 2, shape[0]).astype(np.float32)
        w = V.vocoder_fold_weight_norm(g, v)
        ref = O.fold_weight_norm(g, v)
        np.testing.assert_allclose(w, ref, rtol=2 ** -23, atol=0)


def test_fold_rejects_zero_row(lib):
    v = np.zeros((2, 3), np.float32)
    v[1] = 1
    with pytest.raises(V.VocoderError) as e:
        V.vocoder_fold_weight_norm(np.ones(2, np.float32), v)
    assert e.value.status == V.VOC_INVALID_ARG


def test_stitched_length(lib):
    assert V.vocoder_stitched_length(8, 689, 86, 258, 512) == 1589248
    for args in [(3, 10, 2, 3, 4), (1, 689, 86, 258, 512), (5, 100, 0, 0, 7)]:
        assert V.vocoder_stitched_length(*args) == O.stitched_length(*args)
    assert V.vocoder_stitched_length(3, 10, 6, 5, 4) == -1  # the middle piece would end before it starts
    assert O.stitched_length(3, 10, 6, 5, 4) == -1


def test_wav_sizes(lib):
    """Host-only size queries of the output stage agree with the oracle's file layout."""
    for n_ch, n, bits in [(1, 0, 16), (2, 7, 24), (3, 999, 32), (2, 1000, 16)]:
        wav = O.encode_wav(np.zeros((n_ch, n), np.float32), 44100, bits)
        assert V.vocoder_wav_bytes(n_ch, n, bits) == len(wav)
    assert V.vocoder_wav_bytes(2, 1589248, 24) == 44 + 2 * 1589248 * 3
    assert V.vocoder_wav_bytes(1, 10, 8) == 0
    assert V.vocoder_wav_bytes(0, 10, 16) == 0
    assert V.vocoder_wav_bytes(1, -1, 16) == 0
    assert V.vocoder_wav_bytes(1, 1 << 31, 16) == 0  # beyond the 32-bit RIFF size field
    assert V.vocoder_wav_scratch_bytes() >= 256 + 4 * 2048


def test_create_validates_before_device_work(lib):
    bad = W.Arch(latent_channels=4, channels0=8, strides=(3, 2), widths=(4, 4))  # odd, symmetric
    with pytest.raises(V.VocoderError) as e:
        V.vocoder_create(bad, [None] * V.vocoder_param_count(W.TINY))
    assert e.value.status == V.VOC_INVALID_ARG
    n = V.vocoder_param_count(W.TINY)
    with pytest.raises(V.VocoderError) as e:
        V.vocoder_create(W.TINY, [None] * (n - 1))
    assert e.value.status == V.VOC_INVALID_ARG
    assert "n_params" in V.vocoder_last_error()


def test_precision_field_validation(lib):
    """VOC_PREC_F16W and VOC_PREC_BF16W are valid precisions (same parameter list); unknown
    precisions and the one-plane precisions with CTA pairs are rejected before any device
    work."""
    n = V.vocoder_param_count(W.TINY)
    d = V.make_desc(W.TINY, precision=V.VOC_PREC_F16W)
    assert lib.vocoder_param_count(ctypes.byref(d)) == n
    d = V.make_desc(W.TINY, precision=V.VOC_PREC_BF16W)
    assert lib.vocoder_param_count(ctypes.byref(d)) == n
    d = V.make_desc(W.TINY, precision=3)
    assert lib.vocoder_param_count(ctypes.byref(d)) == -1
    with pytest.raises(V.VocoderError) as e:
        V.vocoder_create(W.TINY, [None] * n, cta_pair=1, precision=V.VOC_PREC_BF16W)
    assert e.value.status == V.VOC_INVALID_ARG
    with pytest.raises(V.VocoderError) as e:
        V.vocoder_create(W.TINY, [None] * n, cta_pair=1, precision=V.VOC_PREC_F16W)
    assert e.value.status == V.VOC_INVALID_ARG
    assert "cta_pair" in V.vocoder_last_error()


ENC_ARCHS = [W.ENC_MUSIC, W.EncArch(1, 16, (2, 4), (32, 48), 8),
             W.EncArch(2, 24, (3, 5, 1), (40, 56, 56), 12, dilations=(1, 3)),
             dataclasses.replace(W.ENC_MUSIC, snake_beta=True)]


@pytest.mark.parametrize("arch", ENC_ARCHS, ids=["music", "small", "odd_strides", "snake_beta"])
def test_encoder_param_shapes_match_layer_list(lib, arch):
    shapes = arch.param_shapes()
    assert V.vocoder_encoder_param_count(arch) == len(shapes)
    for i, (_name, shape) in enumerate(shapes):
        assert V.vocoder_encoder_param_shape(arch, i) == shape


def test_encoder_create_validates_before_device_work(lib):
    n = V.vocoder_encoder_param_count(W.ENC_MUSIC)
    with pytest.raises(V.VocoderError) as e:
        V.vocoder_encoder_create(W.ENC_MUSIC, [None] * (n - 1))
    assert e.value.status == V.VOC_INVALID_ARG
    assert "n_params" in V.vocoder_encoder_last_error()
    bad = dataclasses.replace(W.ENC_MUSIC, strides=(2, 17, 8, 8))
    assert V.vocoder_encoder_param_count(bad) == -1
    with pytest.raises(V.VocoderError) as e:
        V.vocoder_encoder_create(bad, [None] * n)
    assert e.value.status == V.VOC_INVALID_ARG
    d = V.make_enc_desc(W.ENC_MUSIC, precision=3)
    assert lib.vocoder_encoder_param_count(ctypes.byref(d)) == -1
    # a weight is required (only biases may be NULL): rejected before any device call
    with pytest.raises(V.VocoderError) as e:
        V.vocoder_encoder_create(W.ENC_MUSIC, [None] * n)
    assert "params[0]" in V.vocoder_encoder_last_error()
    assert V.vocoder_encoder_hop(None) == -1
    assert V.vocoder_encoder_workspace_bytes(None, 1, 512) == 0
    assert V.vocoder_encoder_launches(None, 1, 512) == -1
