"""Pins of the oracle's mirror encoder (minimaxmusic.cpp Architecture, "Flow VAE": conv_in,
blocks of residual units followed by Snake and a strided conv k = 2s, pad s/2, Snake, conv_out
k3, posterior mean projection k1) against definitions that do not go through it."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from dac_vocoder_decode_gb300 import workloads as W
from oracle import oracle as O


@pytest.mark.parametrize("s", [2, 4, 8])
def test_strided_conv_matches_torch(s):
    rng = np.random.default_rng(s)
    Cin, Cout, T = 5, 3, 8 * s
    x = rng.standard_normal((Cin, T))
    w = rng.standard_normal((Cout, Cin, 2 * s))
    b = rng.standard_normal(Cout)
    got = O.conv1d_strided(x, w, b, s, s // 2, T // s)
    ref = torch.nn.functional.conv1d(torch.from_numpy(x)[None], torch.from_numpy(w),
                                     torch.from_numpy(b), stride=s, padding=s // 2)[0].numpy()
    assert ref.shape == (Cout, T // s)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("s", [2, 3, 4, 8])
def test_strided_conv_is_adjoint_of_transposed_conv(s):
    """<ConvT(u), x> = <u, Strided(x)> for the same [C_a][C_b][2s] weights and crop s // 2:
    the strided conv reads exactly the samples the transposed conv writes."""
    rng = np.random.default_rng(10 + s)
    Ca, Cb, T = 4, 6, 9
    w = rng.standard_normal((Ca, Cb, 2 * s))
    u = rng.standard_normal((Ca, T))
    x = rng.standard_normal((Cb, T * s))
    lhs = np.sum(O.conv_transpose1d(u, w, None, s, s // 2, T * s) * x)
    rhs = np.sum(u * O.conv1d_strided(x, w, None, s, s // 2, T))
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(lhs))


def _corr(x, w, pad_left, dil, stride, T_out):
    """y[t] = sum_k w[k] x[t*stride + k*dil - pad_left], zero outside: one channel, loops."""
    y = np.zeros(T_out)
    for t in range(T_out):
        for k in range(len(w)):
            j = t * stride + k * dil - pad_left
            if 0 <= j < len(x):
                y[t] += w[k] * x[j]
    return y


def test_width_one_encoder_is_its_convolution_cascade():
    """One channel everywhere and Snake replaced by the identity: the encoder is conv_in
    (pad 3), residual units x + conv2(conv1(x)) (dilations 1, 3, 9, 'same' padding),
    strided convs (k = 2s, pad s/2), conv_out (k3, pad 1) and the projection, with biases."""
    arch = W.EncArch(in_channels=1, channels0=1, strides=(2, 4), widths=(1, 1), latent_channels=1)
    wl = W.make_encode_workload(arch, B=1, frames=6, seed=21)
    f = O.fold_params(wl.params)
    got = O.encode(arch, None, wl.latent, O.FLAG_SNAKE_IDENTITY, f)[0, 0]
    x = wl.latent[0, 0].astype(np.float64)
    p = 0
    y = _corr(x, f[p][0, 0], 3, 1, 1, len(x)) + f[p + 1][0]
    p += 2
    for s in arch.strides:
        for d in arch.dilations:
            h = _corr(y, f[p + 1][0, 0], 3 * d, d, 1, len(y)) + f[p + 2][0]
            h = _corr(h, f[p + 4][0, 0], 0, 1, 1, len(h)) + f[p + 5][0]
            y = y + h
            p += 6
        y = _corr(y, f[p + 1][0, 0], s // 2, 1, s, len(y) // s) + f[p + 2][0]
        p += 3
    y = _corr(y, f[p + 1][0, 0], 1, 1, 1, len(y)) + f[p + 2][0]
    y = _corr(y, f[p + 3][0, 0], 0, 1, 1, len(y)) + f[p + 4][0]
    assert got.shape == (6,)
    np.testing.assert_allclose(got, y, rtol=1e-12, atol=1e-12)


def test_encoder_length_and_affinity():
    """The music encoder maps 512 samples to one latent frame; with Snake removed it is an
    affine map of the audio."""
    wl = W.make_encode_workload(W.ENC_MUSIC, B=1, frames=3, seed=5)
    arch = W.ENC_MUSIC
    f = O.fold_params(wl.params)
    z = O.encode(arch, None, wl.latent, 0, f)
    assert z.shape == (1, 64, 3)
    rng = np.random.default_rng(2)
    a1 = rng.uniform(-0.5, 0.5, wl.latent.shape).astype(np.float32)
    a2 = rng.uniform(-0.5, 0.5, wl.latent.shape).astype(np.float32)
    E = lambda a: O.encode(arch, None, a, O.FLAG_SNAKE_IDENTITY, f)  # noqa: E731
    e0 = E(np.zeros_like(a1))
    lhs = E((0.25 * a1 + 0.5 * a2).astype(np.float32)) - e0
    rhs = 0.25 * (E(a1) - e0) + 0.5 * (E(a2) - e0)
    np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-6 * np.max(np.abs(rhs)))


def test_encoder_receptive_field_helper_is_tight():
    """The sampled full-size GPU checks rely on tests.util.encoder_sample_span: changing one
    audio sample just outside the span of latent frame u leaves z[u] unchanged, and just
    inside it changes z[u] (the span is neither too small nor loose at its ends)."""
    from tests.util import encoder_sample_span
    arch = W.EncArch(1, 8, (2, 4), (8, 8), 4, dilations=(1, 3))
    frames, u = 24, 12
    wl = W.make_encode_workload(arch, 1, frames, 5)
    f = O.fold_params(wl.params)
    base = O.encode(arch, None, wl.latent, 0, f)[0, :, u]
    lo, hi = encoder_sample_span(arch, u)
    assert 0 < lo and hi < frames * arch.hop - 1
    for pos, inside in [(lo - 1, False), (hi + 1, False), (lo, True), (hi, True)]:
        a = wl.latent.copy()
        a[0, 0, pos] += 0.5
        z = O.encode(arch, None, a, 0, f)[0, :, u]
        assert (np.max(np.abs(z - base)) > 1e-9) == inside, (pos, inside)
