"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a closed form,
a library routine (numpy / torch CPU in fp64) on small cases, an adjoint
identity, a dense brute force, linearity, an impulse response built with
np.convolve, shift equivariance, locality from the layer list, causality, or a
value the pages print.  A plausible slip in the oracle (a dropped term, a wrong
sign, index, padding or operand order) fails at least one of them."""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

from dac_vocoder_decode_gb300 import workloads as W
from oracle import oracle as O
from tests.util import frame_margins, latent_span

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

SMALL_MUSIC = W.Arch(latent_channels=4, channels0=8, strides=(8, 8, 4, 2), widths=(8, 4, 4, 4))
SMALL_SPEECH = W.Arch(latent_channels=4, channels0=8, strides=(8, 5, 4, 4, 3),
                      widths=(8, 4, 4, 4, 4), padding=W.PAD_CAUSAL)


# --------------------------------------------------------------------------- Snake
@pytest.mark.parametrize("alpha", [0.5, 1.0, 2.0, 1.37])
def test_snake_closed_form_points(alpha):
    """x = 0 -> 0; x = k*pi/alpha -> x (sin^2 vanishes); x = pi/(2 alpha) -> x + 1/(alpha + 1e-9)."""
    x = np.array([[0.0, math.pi / alpha, -3 * math.pi / alpha, 7 * math.pi / alpha,
                   math.pi / (2 * alpha), -math.pi / (2 * alpha)]])
    y = O.snake(x, np.array([alpha]))[0]
    inv_b = 1.0 / (alpha + 1e-9)
    assert y[0] == 0.0
    np.testing.assert_allclose(y[1:4], x[0, 1:4], rtol=0, atol=1e-13)
    np.testing.assert_allclose(y[4], x[0, 4] + inv_b, rtol=0, atol=1e-13)
    np.testing.assert_allclose(y[5], x[0, 5] + inv_b, rtol=0, atol=1e-13)


def test_snake_reads_alpha_verbatim():
    """MiniMax-Music-3 -> CMF README ("What the conversion had to get right"):
    alpha is used as stored, not exponentiated.  With alpha = 2 the peak of
    sin^2 sits at pi/4 and adds 1/2; an exp(alpha) reading would not."""
    y = O.snake(np.array([[math.pi / 4]]), np.array([2.0]))[0, 0]
    assert abs(y - (math.pi / 4 + 0.5)) < 1e-9
    a = math.exp(2.0)
    y_exp = math.pi / 4 + math.sin(a * math.pi / 4) ** 2 / a
    assert abs(y - y_exp) > 0.1


def test_snake_period_and_identity():
    """sin^2 has period pi/alpha, so Snake(x + pi/alpha) = Snake(x) + pi/alpha."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 50)) * 4
    alpha = np.array([0.6, 1.1, 1.45])
    y = O.snake(x, alpha)
    y2 = O.snake(x + (math.pi / alpha)[:, None], alpha)
    np.testing.assert_allclose(y2 - y, np.broadcast_to((math.pi / alpha)[:, None], y.shape),
                               atol=1e-12)
    assert np.all(y - x >= 0)  # the added term is a square over a positive alpha
    np.testing.assert_array_equal(O.snake(x, alpha, identity=True), x)


# --------------------------------------------------------------------------- weight norm
def test_fold_row_norm_is_abs_g():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((6, 5, 7)).astype(np.float32)
    g = rng.standard_normal(6).astype(np.float32)
    w = O.fold_weight_norm(g, v)
    norms = np.sqrt((w.reshape(6, -1) ** 2).sum(1))
    np.testing.assert_allclose(norms, np.abs(g.astype(np.float64)), rtol=1e-14)
    # direction of each row is that of v (times the sign of g)
    vd = v.reshape(6, -1).astype(np.float64)
    cos = (w.reshape(6, -1) * vd).sum(1) / (norms * np.sqrt((vd ** 2).sum(1)))
    np.testing.assert_allclose(cos, np.sign(g), atol=1e-13)


def test_fold_scale_invariant_and_axis0():
    """w does not change under v -> c v (c > 0); the norm runs over axis 0 of the
    stored tensor, so for a ConvTranspose1d [Cin, Cout, K] it is per input channel."""
    rng = np.random.default_rng(2)
    v = rng.standard_normal((4, 3, 6)).astype(np.float32)  # ConvT layout [Cin, Cout, K]
    g = np.array([0.5, 1.0, 2.0, 3.0], dtype=np.float32)
    w1 = O.fold_weight_norm(g, v)
    w2 = O.fold_weight_norm(g, (v * np.float32(4.0)))
    np.testing.assert_allclose(w1, w2, rtol=1e-6)
    per_cin = np.sqrt((w1 ** 2).sum(axis=(1, 2)))
    np.testing.assert_allclose(per_cin, g, rtol=1e-14)
    # cross-check with torch's weight-norm parametrisation (dim 0), fp64
    wt = torch._weight_norm(torch.from_numpy(v.astype(np.float64)),
                            torch.from_numpy(g.astype(np.float64)).view(4, 1, 1), 0)
    np.testing.assert_allclose(w1, wt.numpy(), rtol=1e-13, atol=1e-15)


def test_fold_zero_row_rejected():
    v = np.zeros((2, 3), dtype=np.float32)
    v[0] = 1
    with pytest.raises(ValueError):
        O.fold_weight_norm(np.ones(2, np.float32), v)


# --------------------------------------------------------------------------- conv1d
@pytest.mark.parametrize("K,d,pl,pr", [(7, 1, 3, 3), (7, 3, 9, 9), (7, 9, 27, 27), (1, 1, 0, 0),
                                       (7, 9, 54, 0), (3, 2, 0, 0)])
def test_conv1d_matches_library_and_correlate(K, d, pl, pr):
    rng = np.random.default_rng(K * 100 + d)
    Cin, Cout, T = 3, 4, 70
    x = rng.standard_normal((Cin, T))
    w = rng.standard_normal((Cout, Cin, K))
    b = rng.standard_normal(Cout)
    y = O.conv1d(x, w, b, d, pl, pr)
    # torch (fp64, CPU) with explicit zero padding
    xt = torch.nn.functional.pad(torch.from_numpy(x)[None], (pl, pr))
    yt = torch.nn.functional.conv1d(xt, torch.from_numpy(w), torch.from_numpy(b), dilation=d)[0]
    np.testing.assert_allclose(y, yt.numpy(), rtol=0, atol=1e-12)
    # numpy: correlate each channel pair with the dilated kernel
    xp = np.pad(x, ((0, 0), (pl, pr)))
    ref = np.zeros_like(y) + b[:, None]
    for co in range(Cout):
        for ci in range(Cin):
            kd = np.zeros(d * (K - 1) + 1)
            kd[::d] = w[co, ci]
            ref[co] += np.correlate(xp[ci], kd, mode="valid")
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)


def test_conv1d_impulse_picks_kernel_taps():
    """A unit impulse at position t0 returns the kernel taps reversed in time:
    y[co][t0 + pl - k d] = w[co][0][k]."""
    K, d, pl = 7, 3, 9
    x = np.zeros((1, 80))
    x[0, 40] = 1.0
    w = np.arange(1, 8, dtype=np.float64).reshape(1, 1, 7)
    y = O.conv1d(x, w, None, d, pl, pl)[0]
    for k in range(K):
        assert y[40 + pl - k * d] == w[0, 0, k]
    assert np.count_nonzero(y) == K


# --------------------------------------------------------------------------- transposed conv
@pytest.mark.parametrize("s,causal", [(2, False), (4, False), (8, False), (5, True), (3, True),
                                      (8, True)])
def test_conv_transpose_scatter_matches_library_and_zero_stuffing(s, causal):
    rng = np.random.default_rng(s * 10 + causal)
    Cin, Cout, T = 3, 2, 23
    K = 2 * s
    p = 0 if causal else s // 2
    x = rng.standard_normal((Cin, T))
    w = rng.standard_normal((Cin, Cout, K))
    b = rng.standard_normal(Cout)
    T_out = T * s
    y = O.conv_transpose1d(x, w, b, s, p, T_out)
    # (a) torch fp64: full transposed conv, then crop p on the left and keep T*s
    full = torch.nn.functional.conv_transpose1d(torch.from_numpy(x)[None], torch.from_numpy(w),
                                                torch.from_numpy(b), stride=s)[0].numpy()
    assert full.shape[1] == (T - 1) * s + K
    np.testing.assert_allclose(y, full[:, p:p + T_out], rtol=0, atol=1e-12)
    # (b) textbook identity: zero-stuff x by s, convolve with the kernel, crop
    ref = np.zeros((Cout, T_out)) + b[:, None]
    for co in range(Cout):
        for ci in range(Cin):
            up = np.zeros(T * s)
            up[::s] = x[ci]
            c = np.convolve(up, w[ci, co])  # c[j] = sum_k w[k] up[j-k]
            ref[co] += c[p:p + T_out]
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("s", [2, 4, 8])
def test_conv_transpose_is_adjoint_of_strided_conv(s):
    """<ConvT_w(x), y> = <x, Conv_w,stride s(y)> with the same weights and no bias;
    the strided conv is built here by dense brute force from its definition."""
    rng = np.random.default_rng(77 + s)
    Cin, Cout, T = 3, 2, 11
    K, p = 2 * s, s // 2
    x = rng.standard_normal((Cin, T))
    w = rng.standard_normal((Cin, Cout, K))
    yv = rng.standard_normal((Cout, T * s))
    lhs = np.sum(O.conv_transpose1d(x, w, None, s, p, T * s) * yv)
    z = np.zeros((Cin, T))  # z[ci][t] = sum_co sum_k w[ci][co][k] y[co][t s + k - p]
    for ci in range(Cin):
        for t in range(T):
            for co in range(Cout):
                for k in range(K):
                    j = t * s + k - p
                    if 0 <= j < T * s:
                        z[ci, t] += w[ci, co, k] * yv[co, j]
    rhs = np.sum(x * z)
    assert abs(lhs - rhs) < 1e-10 * max(1.0, abs(lhs))


def test_col2im_length_formula():
    """qwentts.cpp Architecture, "Custom GGML ops": T_out = (T_in - 1) s + K - 2p;
    with K = 2s and p = s/2 that is T_in * s."""
    for s in (2, 4, 8):
        for T in (1, 5, 689):
            assert (T - 1) * s + 2 * s - 2 * (s // 2) == T * s


# --------------------------------------------------------------------------- decoder
def _small_workload(arch, B=2, T=40, seed=11, recipe="calibrated"):
    return W.make_custom(arch, B, T, seed, recipe)


def test_pages_lengths_golden():
    """The pages' own numbers: 12 latent frames -> 6144 samples per side at hop 512
    (MiniMax-Music-3 -> CMF README, "What is verified, and how"); the speech codec
    turns each 12.5 Hz frame into 1920 samples at 24 kHz (qwentts.cpp Architecture,
    "Audio tokenizer decoder")."""
    with open(os.path.join(GOLDEN, "pages_values.json")) as f:
        g = json.load(f)
    wl = _small_workload(SMALL_MUSIC, B=2, T=g["music_frames"], seed=3)
    y = O.decode(wl.arch, wl.params, wl.latent)
    assert y.shape == (2, g["music_samples_per_side"])
    assert wl.arch.hop == g["music_hop"] == W.MUSIC.hop
    assert W.SPEECH.hop == g["speech_hop"]
    assert np.all(np.abs(y) <= 1.0)
    assert np.std(y) > 1e-3  # above silence
    assert np.max(np.abs(y[0] - y[1])) > 0  # left differs from right


def test_tiny_workload_length():
    wl = W.make_workload("tiny")
    y = O.decode(wl.arch, wl.params, wl.latent)
    assert y.shape == (1, 16384)
    assert np.all(np.isfinite(y)) and np.all(np.abs(y) <= 1)


def test_decoder_linearity_without_nonlinearities():
    """Snake -> identity, tanh removed, biases 0: D(a x + b y) = a D(x) + b D(y)."""
    wl = _small_workload(SMALL_MUSIC, B=1, T=24, seed=5)
    params = [W.RawConv(p.g, p.v, None) if isinstance(p, W.RawConv) else p for p in wl.params]
    fl = O.FLAG_SNAKE_IDENTITY | O.FLAG_NO_TANH
    rng = np.random.default_rng(9)
    # multiples of 1/64: a x + b y below is then exact in fp32 (no input rounding)
    x = (np.round(rng.standard_normal(wl.latent.shape) * 64) / 64).astype(np.float32)
    y = (np.round(rng.standard_normal(wl.latent.shape) * 64) / 64).astype(np.float32)
    a, b = 0.75, -1.25
    comb = (np.float64(a) * x + np.float64(b) * y)
    assert np.all(comb.astype(np.float32) == comb)
    folded = O.fold_params(params)
    dx = O.decode(wl.arch, params, x, fl, folded)
    dy = O.decode(wl.arch, params, y, fl, folded)
    dc = O.decode(wl.arch, params, comb.astype(np.float32), fl, folded)
    np.testing.assert_allclose(dc, a * dx + b * dy, rtol=0, atol=1e-11 * np.max(np.abs(dc)))


def _impulse_response_closed_form(arch, folded, T, t0):
    """The decoder with every width 1, Snake = identity, no tanh and no bias is a
    multirate LTI chain.  Build its response to a unit impulse at frame t0 with
    np.convolve: a k-tap conv with left pad pl is y[t] = sum_k w[k] x[t + k d - pl];
    a transposed conv is (zero-stuffed x) convolved with w, cropped by p; a
    residual unit is x + w2 * conv1(x)."""
    def corr(x, w, d, pl):
        K = len(w)
        kd = np.zeros(d * (K - 1) + 1)
        kd[::d] = w
        # y[t] = sum_m kd[m] x[t + m - pl]  ->  full convolution with the reversed kernel
        full = np.convolve(x, kd[::-1])  # full[n] = sum_m kd[m] x[n - (len-1) + m]
        off = len(kd) - 1 - pl
        out = np.zeros(len(x))
        for t in range(len(x)):
            n = t + off
            if 0 <= n < len(full):
                out[t] = full[n]
        return out

    causal = arch.padding == W.PAD_CAUSAL
    def pad_l(K, d):
        return d * (K - 1) if causal else d * (K - 1) // 2

    x = np.zeros(T)
    x[t0] = 1.0
    it = iter(folded)
    w_in = next(it); next(it)
    x = corr(x, w_in[0, 0], 1, pad_l(arch.in_kernel, 1))
    for s in arch.strides:
        next(it)  # alpha
        wt = next(it); next(it)
        up = np.zeros(len(x) * s)
        up[::s] = x
        c = np.convolve(up, wt[0, 0])
        p = 0 if causal else s // 2
        x = c[p:p + len(up)]
        for d in arch.dilations:
            next(it); w1 = next(it); next(it); next(it); w2 = next(it); next(it)
            x = x + w2[0, 0, 0] * corr(x, w1[0, 0], d, pad_l(arch.res_kernel, d))
    next(it)
    w_out = next(it)
    return corr(x, w_out[0, 0], 1, pad_l(arch.out_kernel, 1))


@pytest.mark.parametrize("arch", [
    W.Arch(latent_channels=1, channels0=1, strides=(8, 8, 4, 2), widths=(1, 1, 1, 1)),
    W.Arch(latent_channels=1, channels0=1, strides=(8, 5, 4, 4, 3), widths=(1, 1, 1, 1, 1),
           padding=W.PAD_CAUSAL)], ids=["music", "speech_causal"])
def test_impulse_response_width_one(arch):
    wl = _small_workload(arch, B=1, T=30, seed=21)
    params = [W.RawConv(p.g, p.v, None) if isinstance(p, W.RawConv) else p for p in wl.params]
    folded = O.fold_params(params)
    lat = np.zeros((1, 1, 30), dtype=np.float32)
    lat[0, 0, 13] = 1.0
    y = O.decode(arch, params, lat, O.FLAG_SNAKE_IDENTITY | O.FLAG_NO_TANH, folded)[0]
    ref = _impulse_response_closed_form(arch, folded, 30, 13)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12 * max(1.0, np.max(np.abs(ref))))
    assert np.max(np.abs(ref)) > 0


def test_shift_equivariance():
    """Shifting the latent by one frame shifts the audio by hop samples, away from
    the ends (holds for the full nonlinear decoder)."""
    arch = SMALL_MUSIC
    wl = _small_workload(arch, B=1, T=48, seed=31)
    folded = O.fold_params(wl.params)
    lat = wl.latent
    lat2 = np.concatenate([np.zeros_like(lat[:, :, :1]), lat[:, :, :-1]], axis=2)
    y = O.decode(arch, wl.params, lat, 0, folded)[0]
    y2 = O.decode(arch, wl.params, lat2, 0, folded)[0]
    left, right = frame_margins(arch)
    hop = arch.hop
    lo, hi = (left + 2) * hop, (48 - right - 2) * hop
    np.testing.assert_allclose(y2[lo + hop:hi + hop], y[lo:hi], rtol=0, atol=1e-13)


@pytest.mark.parametrize("arch", [SMALL_MUSIC, SMALL_SPEECH], ids=["music", "speech_causal"])
def test_locality_from_layer_list(arch):
    """Changing latent frame t0 changes exactly the samples whose receptive field
    (derived from taps, dilations, strides and paddings) contains t0; every other
    sample is bit-identical."""
    T, t0 = 60, 30
    wl = _small_workload(arch, B=1, T=T, seed=41)
    folded = O.fold_params(wl.params)
    y = O.decode(arch, wl.params, wl.latent, 0, folded)[0]
    lat2 = wl.latent.copy()
    lat2[0, :, t0] += 1.0
    y2 = O.decode(arch, wl.params, lat2, 0, folded)[0]
    changed = y != y2
    hop = arch.hop
    may = np.zeros(T * hop, dtype=bool)
    for j in range(T * hop):
        lo, hi = latent_span(arch, j)
        may[j] = lo <= t0 <= hi
    assert not np.any(changed & ~may)
    assert np.any(changed)
    if arch.padding == W.PAD_CAUSAL:
        assert not np.any(changed[:t0 * hop])  # causality: nothing before the frame moves
        assert changed[t0 * hop:(t0 + 1) * hop].any()


def test_receptive_field_bound():
    """The music decoder's receptive field is under 13 latent frames per side, so
    crops of 86 / 258 frames leave every kept sample seam-exact."""
    left, right = frame_margins(W.MUSIC)
    assert left <= 13 and right <= 13
    assert W.STITCH_CROP_LEFT > left and W.STITCH_CROP_RIGHT > right


def test_batch_items_independent_and_stereo_fold():
    """The decode of a batch equals the decodes of its items; a 128-channel latent
    is two 64-channel tracks (channels 0..63 = left) decoded independently, and
    the two sides differ (MiniMax-Music-3 -> CMF README, "What the conversion had
    to get right"; minimaxmusic.cpp Architecture, "Flow VAE")."""
    arch = SMALL_MUSIC
    wl = _small_workload(arch, B=1, T=20, seed=51)
    folded = O.fold_params(wl.params)
    rng = np.random.default_rng(3)
    stereo = rng.standard_normal((1, 2 * arch.latent_channels, 20)).astype(np.float32)
    folded_lat = stereo.reshape(2, arch.latent_channels, 20)  # [b,2C,t] -> [2b,C,t]
    yb = O.decode(arch, wl.params, folded_lat, 0, folded)
    yl = O.decode(arch, wl.params, stereo[:, :arch.latent_channels], 0, folded)
    yr = O.decode(arch, wl.params, stereo[:, arch.latent_channels:], 0, folded)
    np.testing.assert_array_equal(yb[0], yl[0])
    np.testing.assert_array_equal(yb[1], yr[0])
    assert np.max(np.abs(yb[0] - yb[1])) > 1e-3


def test_calibrated_tiny_is_nonlinear_and_unsaturated():
    """The calibrated synthetic weights give a pre-tanh signal with RMS in
    [0.05, 1], so the tests exercise the nonlinear regime without saturating."""
    wl = W.make_workload("tiny_cal")
    y, pre = O.decode(wl.arch, wl.params, wl.latent, return_pre_tanh=True)
    rms = float(np.sqrt(np.mean(pre ** 2)))
    assert 0.05 <= rms <= 1.0, rms
    yl = O.decode(wl.arch, wl.params, wl.latent, O.FLAG_SNAKE_IDENTITY)
    assert np.max(np.abs(yl - y)) > 1e-2  # Snake matters


# --------------------------------------------------------------------------- stitch
def test_stitch_length_and_clamp():
    assert O.stitched_length(8, 689, 86, 258, 512) == 3104 * 512 == 1589248
    assert O.stitched_length(1, 689, 86, 258, 512) == 689 * 512
    dec = np.full((2, 5 * 4), 2.0)
    dec[1] = -3.0
    out = O.stitch(dec, 1, 2, 5, 1, 1, 4)
    np.testing.assert_array_equal(out, np.stack([np.ones(20), -np.ones(20)]))


def test_stitch_piece_positions():
    """Window w contributes frames [w == 0 ? 0 : cl, w == last ? W : W - cr)."""
    n_win, n_sides, Wf, cl, cr, hop = 3, 2, 10, 2, 3, 4
    dec = np.zeros((n_win * n_sides, Wf * hop))
    for w in range(n_win):
        for side in range(n_sides):
            dec[w * n_sides + side] = (w * 10 + side + np.arange(Wf * hop) / 1000.0) / 100.0
    out = O.stitch(dec, n_win, n_sides, Wf, cl, cr, hop)
    assert out.shape == (2, (7 + 5 + 8) * hop)
    np.testing.assert_array_equal(out[1, :7 * hop], dec[1, :7 * hop])
    np.testing.assert_array_equal(out[0, 7 * hop:12 * hop], dec[2, cl * hop:(Wf - cr) * hop])
    np.testing.assert_array_equal(out[1, 12 * hop:], dec[5, cl * hop:])


@pytest.mark.slow
def test_windowed_stitch_equals_single_pass():
    """Windows cut at hop 345 from one continuous latent, decoded and stitched
    with crops 86 / 258, equal a single pass over the whole latent: every kept
    sample lies more than the receptive field away from its window's edges."""
    arch = W.Arch(latent_channels=4, channels0=4, strides=(8, 8, 4, 2), widths=(4, 2, 2, 2))
    wl = _small_workload(arch, B=1, T=8, seed=61)
    folded = O.fold_params(wl.params)
    rng = np.random.default_rng(62)
    total = W.STITCH_HOP_FRAMES * (W.STITCH_WINDOWS - 1) + W.STITCH_WIN_FRAMES
    cont = rng.standard_normal((2, 4, total)).astype(np.float32)
    wins = np.stack([cont[side, :, w * 345:w * 345 + 689] for w in range(8) for side in range(2)])
    dec = O.decode(arch, wl.params, wins, 0, folded)
    st = O.stitch(dec, 8, 2, 689, 86, 258, arch.hop)
    full = O.decode(arch, wl.params, cont, 0, folded)
    assert st.shape == full.shape == (2, 1589248)
    np.testing.assert_allclose(st, full, rtol=0, atol=1e-13)


def test_full_music_model_parameter_count():
    """The published music decoder with its input projection (dec_in_proj 64 -> 1024, not
    weight normalised, then conv_in 1024 -> 1536) has 54 M parameters per the pages; the
    folded tensors of the architecture add up to that (weight-norm gains are not stored
    once folded)."""
    with open(os.path.join(GOLDEN, "pages_values.json")) as f:
        gold = json.load(f)
    n = sum(int(np.prod(s)) for _, s in W.MUSIC_FULL.param_shapes())
    assert round(n / 1e6) == gold["music_vocoder_params_millions"]
    assert n == 54157665
    # the oracle sees the same tensor list
    assert len(W.MUSIC_FULL.param_shapes()) == len(W.MUSIC.param_shapes()) + 2


def test_identity_projection_reproduces_plain_decoder():
    """An input projection that copies the C_lat latent channels into the first C_lat of
    its P outputs (zero bias), followed by a conv_in whose weights on the extra P - C_lat
    channels are zero, decodes exactly like the decoder without the projection."""
    base = W.Arch(latent_channels=6, channels0=24, strides=(4, 2), widths=(12, 8))
    full = W.Arch(latent_channels=6, channels0=24, strides=(4, 2), widths=(12, 8),
                  in_proj_channels=16)
    wl = W.make_custom(base, B=2, T=18, seed=77)
    folded = O.fold_params(wl.params)
    w_in = folded[0]  # conv_in [C0][C_lat][K]
    proj = np.zeros((16, 6, 1))
    proj[:6, :, 0] = np.eye(6)
    w_in_full = np.zeros((24, 16, w_in.shape[2]))
    w_in_full[:, :6, :] = w_in
    folded_full = [proj, np.zeros(16), w_in_full] + folded[1:]
    y0 = O.decode(base, None, wl.latent, 0, folded)
    y1 = O.decode(full, None, wl.latent, 0, folded_full)
    np.testing.assert_array_equal(y0, y1)
    # and a non-trivial projection changes the result
    proj2 = proj.copy()
    proj2[7, 0, 0] = 1.0
    w_in_full2 = w_in_full.copy()
    w_in_full2[:, 7, :] = w_in[:, 0, :]
    y2 = O.decode(full, None, wl.latent, 0, [proj2, np.zeros(16), w_in_full2] + folded[1:])
    assert np.max(np.abs(y2 - y0)) > 1e-3


# ----------------------------------------------------------------------------- SnakeBeta
@pytest.mark.parametrize("la,lb", [(0.0, 0.0), (math.log(1.37), math.log(0.61)), (-0.4, 0.9)])
def test_snake_beta_closed_form_points(la, lb):
    """y = x + sin^2(e^la x) / (e^lb + 1e-9): zero at the zeros of sin, 1/(e^lb + 1e-9) added
    at its peaks, and sin^2 = 1/2 at an eighth of the period."""
    a, b = math.exp(la), math.exp(lb)
    k = np.arange(-5, 6, dtype=np.float64)
    zeros = k * math.pi / a
    peaks = (k + 0.5) * math.pi / a
    eighth = (k + 0.25) * math.pi / a
    y0 = O.snake_beta(zeros[None], [la], [lb])[0]
    y1 = O.snake_beta(peaks[None], [la], [lb])[0]
    y2 = O.snake_beta(eighth[None], [la], [lb])[0]
    np.testing.assert_allclose(y0, zeros, rtol=0, atol=1e-13)
    np.testing.assert_allclose(y1, peaks + 1.0 / (b + 1e-9), rtol=0, atol=1e-12)
    np.testing.assert_allclose(y2, eighth + 0.5 / (b + 1e-9), rtol=0, atol=1e-12)


def test_snake_beta_period_and_equal_parameters():
    rng = np.random.default_rng(31)
    x = rng.uniform(-20, 20, size=(1, 500))
    la, lb = 0.3, -0.2
    per = math.pi / math.exp(la)
    d0 = O.snake_beta(x, [la], [lb]) - x
    d1 = O.snake_beta(x + per, [la], [lb]) - (x + per)
    np.testing.assert_allclose(d0, d1, rtol=0, atol=1e-11)
    # alpha = beta: plain Snake with alpha = e^la
    np.testing.assert_allclose(O.snake_beta(x, [la], [la]), O.snake(x, [math.exp(la)]),
                               rtol=0, atol=1e-13)


def test_snake_beta_decoder_uses_both_rows():
    """The decoder reads every SnakeBeta parameter as [log alpha; log beta]:
    (a) beta = alpha decodes like the plain-Snake decoder with alpha' = e^alpha;
    (b) beta = 80 (divisor e^80) decodes like the decoder with Snake replaced by identity,
    and swapping the rows (alpha = 80) does not."""
    plain = W.Arch(latent_channels=6, channels0=24, strides=(4, 2), widths=(12, 8))
    beta = W.Arch(latent_channels=6, channels0=24, strides=(4, 2), widths=(12, 8),
                  snake_beta=True)
    wl = W.make_custom(plain, B=2, T=14, seed=91)
    folded = O.fold_params(wl.params)
    kinds = [n for n, _ in plain.param_shapes()]
    rng = np.random.default_rng(5)

    def with_snakes(fn):
        return [fn(f) if k.endswith(".alpha") else f for k, f in zip(kinds, folded)]

    logs = {}

    def equal_rows(f):
        la = np.log(rng.uniform(0.5, 1.5, size=f.shape))
        logs[id(f)] = la
        return np.stack([la, la])

    fb = with_snakes(equal_rows)
    fp = [np.exp(logs[id(f)]) if k.endswith(".alpha") else f for k, f in zip(kinds, folded)]
    np.testing.assert_allclose(O.decode(beta, None, wl.latent, 0, fb),
                               O.decode(plain, None, wl.latent, 0, fp), rtol=0, atol=1e-12)

    fb80 = with_snakes(lambda f: np.stack([np.full(f.shape, 0.3), np.full(f.shape, 80.0)]))
    ident = O.decode(plain, None, wl.latent, O.FLAG_SNAKE_IDENTITY, folded)
    np.testing.assert_allclose(O.decode(beta, None, wl.latent, 0, fb80), ident, rtol=0, atol=1e-12)
    swapped = with_snakes(lambda f: np.stack([np.full(f.shape, 80.0), np.full(f.shape, 0.3)]))
    assert np.max(np.abs(O.decode(beta, None, wl.latent, 0, swapped) - ident)) > 1e-3


# ----------------------------------------------------------------------------- F16 weights
def test_round_half_matches_numpy():
    """Single then half precision, ties to even, against numpy's float32 -> float16 casts."""
    rng = np.random.default_rng(17)
    mags = 10.0 ** rng.uniform(-9, 5, size=4000)
    x = mags * rng.choice([-1.0, 1.0], size=mags.size)
    ties = []
    for e in range(-24, 16):  # exact halfway points between neighbouring halves
        q = 2.0 ** max(e - 10, -24)
        for k in (1, 2, 3, 1023, 1024, 2047):
            ties.append((k + 0.5) * q)
    edges = [0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 6.1e-5, 2.0 ** -24, 2.0 ** -25,
             1.5 * 2.0 ** -25]
    x = np.concatenate([x, np.array(ties), -np.array(ties), np.array(edges)])
    with np.errstate(over="ignore"):
        ref = np.float16(np.float32(x)).astype(np.float64)
    got = O.round_half(x)
    assert np.array_equal(np.signbit(got), np.signbit(ref))
    np.testing.assert_array_equal(got, ref)


def test_f16_weights_round_only_convolution_weights():
    """fold_params(f16_weights=True) rounds every convolution weight (weight-normalised or
    not) and leaves biases and Snake parameters as they are."""
    arch = W.Arch(latent_channels=6, channels0=24, strides=(4, 2), widths=(12, 8),
                  in_proj_channels=10)
    wl = W.make_custom(arch, B=1, T=9, seed=5)
    full = O.fold_params(wl.params)
    half = O.fold_params(wl.params, f16_weights=True)
    names = [n for n, _ in arch.param_shapes()]
    changed = 0
    for n, a, b in zip(names, full, half):
        if n.endswith(".w"):
            np.testing.assert_array_equal(b, O.round_half(a))
            changed += int(np.any(a != b))
        elif a is None:
            assert b is None
        else:
            np.testing.assert_array_equal(a, b)
    assert changed == sum(n.endswith(".w") for n in names)
    # half-precision weights move the decode by about the weights' relative rounding (2^-11)
    y0 = O.decode(arch, None, wl.latent, 0, full)
    y1 = O.decode(arch, None, wl.latent, 0, half)
    d = np.max(np.abs(y1 - y0))
    assert 1e-7 < d < 1e-2


# ----------------------------------------------------------------------------- BF16 weights
def test_round_bf16_matches_torch():
    """Single then bfloat16 precision, ties to even, against torch's float32 -> bfloat16
    conversion (a library routine), on random magnitudes over the whole exponent range,
    exact halfway points and the overflow / subnormal edges."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(19)
    mags = 10.0 ** rng.uniform(-40, 38, size=4000)
    x = mags * rng.choice([-1.0, 1.0], size=mags.size)
    ties = []
    for e in (-133, -130, -126, -20, -1, 0, 1, 30, 127):  # halfway between neighbouring bf16s
        q = 2.0 ** max(e - 7, -133)
        for k in (1, 2, 3, 127, 128, 255):
            ties.append((k + 0.5) * q)
    fmax = float(np.finfo(np.float32).max)
    edges = [0.0, -0.0, fmax, -fmax, 3.3895e38, 3.3896e38, 2.0 ** -126, 2.0 ** -133,
             2.0 ** -134, 1.5 * 2.0 ** -134, 1e-45]
    x = np.concatenate([x, np.array(ties), -np.array(ties), np.array(edges)])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_bf16(x)
    assert np.array_equal(np.signbit(got), np.signbit(ref))
    np.testing.assert_array_equal(got, ref)


def test_round_bf16_hand_values():
    """Values fixed by the format alone: spacing 2^-7 above 1, ties to the even neighbour."""
    cases = [(1.0 + 2.0 ** -8, 1.0),                       # halfway, 1.0 is even
             (1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -6),       # halfway, 1 + 2^-6 is even
             (1.0 + 2.0 ** -8 + 2.0 ** -20, 1.0 + 2.0 ** -7),
             (-(1.0 + 5 * 2.0 ** -8), -(1.0 + 2 * 2.0 ** -7)),  # halfway, mantissa 2 is even
             (255.5, 256.0), (254.5, 254.0), (0.1, 0.10009765625)]
    for x, want in cases:
        assert O.round_bf16(np.array([x]))[0] == want, (x, want)


def test_bf16_weights_round_only_convolution_weights():
    """fold_params(bf16_weights=True) rounds every convolution weight and leaves biases and
    Snake parameters as they are; bf16 rounding moves more weights further than f16's."""
    arch = W.Arch(latent_channels=6, channels0=24, strides=(4, 2), widths=(12, 8),
                  in_proj_channels=10)
    wl = W.make_custom(arch, B=1, T=9, seed=5)
    full = O.fold_params(wl.params)
    bf = O.fold_params(wl.params, bf16_weights=True)
    half = O.fold_params(wl.params, f16_weights=True)
    names = [n for n, _ in arch.param_shapes()]
    for n, a, b, h in zip(names, full, bf, half):
        if n.endswith(".w"):
            np.testing.assert_array_equal(b, O.round_bf16(a))
            assert np.max(np.abs(b - a)) >= np.max(np.abs(h - a))
            rel = np.abs(b - a) / np.maximum(np.abs(a), 1e-30)
            assert np.max(rel) <= 2.0 ** -8 * (1 + 1e-12)  # half a unit in the 8th bit
        elif a is None:
            assert b is None
        else:
            np.testing.assert_array_equal(a, b)
