"""GPU parity: the CUDA library, called through its C ABI, against the CPU oracle.

Per-layer checks run each tensor-core layer kind (k7 dilated conv, k1 conv,
conv_in, polyphase transposed conv, symmetric and causal) on shapes that span
several 128-row tiles, a ragged tail and several column tiles.  End-to-end
checks decode every workload: the small ones in full, the full-size ones
element by element on sampled windows that the oracle computes exactly from
latent slices covering the receptive field.

Tolerances: decoded audio (in [-1, 1]) must satisfy max |gpu - oracle| <= 2e-3
and SNR >= 60 dB.  Single layers are held to a bound derived from the bf16x3
arithmetic: each product carries a relative error of about 2^-16 (the dropped
lo*lo term and the two splits), so |err| <= 2^-14 * sum |w x| leaves a 4x margin
over the fp32-accumulated worst case of these sizes."""
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

LAYER_REL = 2.0 ** -14


# ----------------------------------------------------------------------------- single layers
CONV_CASES = [
    # B, Cin, Cout, T, K, dil, padding
    (2, 96, 96, 300, 7, 1, W.PAD_SYMMETRIC),
    (1, 96, 96, 257, 7, 3, W.PAD_SYMMETRIC),
    (2, 192, 192, 200, 7, 9, W.PAD_SYMMETRIC),
    (1, 384, 384, 130, 7, 9, W.PAD_CAUSAL),
    (2, 768, 768, 129, 1, 1, W.PAD_SYMMETRIC),
    (1, 64, 1536, 150, 7, 1, W.PAD_SYMMETRIC),   # conv_in shape
    (1, 1024, 256, 70, 7, 1, W.PAD_CAUSAL),      # speech conv_in (cut to 256 outputs)
    (1, 4, 4, 140, 7, 3, W.PAD_SYMMETRIC),       # padded channels (tiny decoder)
    (1, 48, 48, 400, 7, 9, W.PAD_CAUSAL),
    (3, 16, 40, 33, 7, 1, W.PAD_SYMMETRIC),      # ragged T shorter than one tile
]


@pytest.mark.parametrize("case", CONV_CASES, ids=[str(c) for c in CONV_CASES])
@pytest.mark.parametrize("with_snake", [True, False])
def test_op_conv1d(case, with_snake):
    B, Cin, Cout, T, K, dil, padding = case
    rng = np.random.default_rng(hash(case) % 2**32)
    x = rng.standard_normal((B, Cin, T)).astype(np.float32)
    w = (rng.standard_normal((Cout, Cin, K)) / np.sqrt(Cin * K)).astype(np.float32)
    b = (rng.standard_normal(Cout) * 0.1).astype(np.float32)
    alpha = rng.uniform(0.5, 1.5, Cin).astype(np.float32) if with_snake else None
    y = torch.empty((B, Cout, T), dtype=torch.float32, device="cuda")
    V.vocoder_op_conv1d(torch.from_numpy(x).cuda(), w, b, dil, padding, alpha, y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    span = dil * (K - 1)
    pl = span if padding == W.PAD_CAUSAL else span // 2
    wd = w.astype(np.float64)
    for bi in range(B):
        xs = O.snake(x[bi], alpha) if with_snake else x[bi].astype(np.float64)
        ref = O.conv1d(xs, wd, b, dil, pl, span - pl)
        mag = O.conv1d(np.abs(xs), np.abs(wd), None, dil, pl, span - pl)
        err = np.abs(got[bi] - ref)
        assert np.all(err <= LAYER_REL * mag + 1e-6), (bi, float(err.max()), float(mag.max()))


def test_snake_accuracy_wide_range():
    """The GPU Snake (sin^2 reduced by multiples of pi, then __sinf; sinf beyond
    |a x| > 8192) through a 1x1 identity conv, so y = Snake(x) carried as a bf16
    hi/lo pair.  Bound: 2^-16 |y| for the hi/lo split plus 4e-6 absolute for the
    reduction (k * ulp(pi_lo) <= 2^-22) and __sinf (about 2^-21 on [-pi, pi])."""
    rng = np.random.default_rng(7)
    C, T = 32, 3000
    parts = [rng.uniform(-4, 4, (C, 1000)), rng.uniform(-300, 300, (C, 1000)),
             rng.uniform(-2e4, 2e4, (C, 1000))]
    x = np.concatenate(parts, axis=1).astype(np.float32)[None]
    x[0, :, :8] = 0.0
    alpha = rng.uniform(0.5, 1.5, C).astype(np.float32)
    w = np.eye(C, dtype=np.float32)[:, :, None]
    y = torch.empty((1, C, T), dtype=torch.float32, device="cuda")
    V.vocoder_op_conv1d(torch.from_numpy(x).cuda(), w, None, 1, W.PAD_SYMMETRIC, alpha, y)
    torch.cuda.synchronize()
    got = y.cpu().numpy()[0].astype(np.float64)
    ref = O.snake(x[0], alpha)
    err = np.abs(got - ref)
    assert np.all(err <= 2.0 ** -16 * np.abs(ref) + 4e-6), float(np.max(err - 2.0 ** -16 * np.abs(ref)))
    assert np.all(got[:, :8] == 0.0)


CONVT_CASES = [
    # B, Cin, Cout, T, stride, padding
    (2, 192, 96, 300, 2, W.PAD_SYMMETRIC),
    (1, 320, 160, 77, 2, W.PAD_SYMMETRIC),        # two column tiles, each with phase halves of 80
    (1, 384, 192, 140, 4, W.PAD_SYMMETRIC),
    (2, 768, 384, 129, 8, W.PAD_SYMMETRIC),
    (1, 1536, 768, 40, 8, W.PAD_SYMMETRIC),
    (1, 96, 48, 200, 3, W.PAD_CAUSAL),
    (2, 768, 384, 65, 5, W.PAD_CAUSAL),
    (1, 192, 96, 131, 4, W.PAD_CAUSAL),
    (1, 8, 4, 50, 2, W.PAD_SYMMETRIC),           # padded channels
    (1, 24, 12, 33, 3, W.PAD_CAUSAL),            # odd phase count, padded channels, odd length
]


@pytest.mark.parametrize("case", CONVT_CASES, ids=[str(c) for c in CONVT_CASES])
def test_op_conv_transpose1d(case):
    B, Cin, Cout, T, s, padding = case
    rng = np.random.default_rng(hash(case) % 2**32)
    x = rng.standard_normal((B, Cin, T)).astype(np.float32)
    w = (rng.standard_normal((Cin, Cout, 2 * s)) / np.sqrt(Cin)).astype(np.float32)
    b = (rng.standard_normal(Cout) * 0.1).astype(np.float32)
    alpha = rng.uniform(0.5, 1.5, Cin).astype(np.float32)
    y = torch.empty((B, Cout, T * s), dtype=torch.float32, device="cuda")
    V.vocoder_op_conv_transpose1d(torch.from_numpy(x).cuda(), w, b, s, padding, alpha, y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    p = 0 if padding == W.PAD_CAUSAL else s // 2
    wd = w.astype(np.float64)
    for bi in range(B):
        xs = O.snake(x[bi], alpha)
        ref = O.conv_transpose1d(xs, wd, b, s, p, T * s)
        mag = O.conv_transpose1d(np.abs(xs), np.abs(wd), None, s, p, T * s)
        err = np.abs(got[bi] - ref)
        assert np.all(err <= LAYER_REL * mag + 1e-6), (bi, float(err.max()), float(mag.max()))


RU_CASES = [
    # B, C, T, dil, padding   (C <= 192: fused kernel; above: conv1 + conv2 kernels)
    (2, 96, 300, 9, W.PAD_SYMMETRIC),
    (1, 96, 257, 1, W.PAD_CAUSAL),
    (2, 96, 777, 9, W.PAD_SYMMETRIC),   # six 128-row tiles and a ragged one per item
    (1, 128, 300, 3, W.PAD_CAUSAL),     # the widest B2 form (N = 2 x 128 accumulator columns)
    (1, 80, 513, 9, W.PAD_SYMMETRIC),   # 5 column chunks over 3 epilogue groups, one row past 4 tiles
    (2, 112, 40, 1, W.PAD_SYMMETRIC),   # shorter than one tile
    (2, 192, 200, 3, W.PAD_SYMMETRIC),  # H as four parts in a ring of two slots
    (1, 192, 300, 9, W.PAD_SYMMETRIC),  # six parts (the tap span leaves room for 32-channel k-blocks)
    (1, 160, 260, 1, W.PAD_CAUSAL),     # five parts of 32 channels
    (1, 48, 400, 9, W.PAD_CAUSAL),
    (3, 16, 70, 3, W.PAD_SYMMETRIC),
    (1, 4, 129, 9, W.PAD_SYMMETRIC),
    (1, 32, 1000, 1, W.PAD_SYMMETRIC),
    (2, 384, 130, 9, W.PAD_SYMMETRIC),
    (1, 768, 140, 3, W.PAD_CAUSAL),
]


@pytest.mark.parametrize("case", RU_CASES, ids=[str(c) for c in RU_CASES])
def test_op_residual_unit(case):
    """y = x + conv2(Snake2(conv1(Snake1(x)) + b1)) + b2.  Bound: the conv2 error
    2^-14 sum|w2 s2| plus the conv1 error carried through Snake2 (slope <= 2) and
    conv2, plus the hi/lo split of Snake2's output."""
    B, C, T, d, padding = case
    rng = np.random.default_rng(hash(case) % 2**32)
    x = rng.standard_normal((B, C, T)).astype(np.float32)
    w1 = (rng.standard_normal((C, C, 7)) * 0.5 / np.sqrt(7 * C)).astype(np.float32)
    w2 = (rng.standard_normal((C, C, 1)) * 0.5 / np.sqrt(C)).astype(np.float32)
    b1 = (rng.standard_normal(C) * 0.02).astype(np.float32)
    b2 = (rng.standard_normal(C) * 0.02).astype(np.float32)
    a1 = rng.uniform(0.5, 1.5, C).astype(np.float32)
    a2 = rng.uniform(0.5, 1.5, C).astype(np.float32)
    y = torch.empty((B, C, T), dtype=torch.float32, device="cuda")
    V.vocoder_op_residual_unit(torch.from_numpy(x).cuda(), a1, w1, b1, d, a2, w2, b2, padding, y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    span = 6 * d
    pl = span if padding == W.PAD_CAUSAL else span // 2
    w1d, w2d = w1.astype(np.float64), w2.astype(np.float64)
    for bi in range(B):
        s1 = O.snake(x[bi], a1)
        h = O.conv1d(s1, w1d, b1, d, pl, span - pl)
        s2 = O.snake(h, a2)
        ref = x[bi].astype(np.float64) + O.conv1d(s2, w2d, b2, 1, 0, 0)
        m1 = O.conv1d(np.abs(s1), np.abs(w1d), None, d, pl, span - pl)
        m2 = O.conv1d(np.abs(s2), np.abs(w2d), None, 1, 0, 0)
        carried = O.conv1d(2 * LAYER_REL * m1 + 2.0 ** -16 * np.abs(s2), np.abs(w2d), None, 1, 0, 0)
        bound = LAYER_REL * m2 + carried + 2e-6
        err = np.abs(got[bi] - ref)
        assert np.all(err <= bound), (bi, float(np.max(err - bound)))


# ----------------------------------------------------------------------------- full decodes
@pytest.mark.parametrize("name", ["tiny", "tiny_cal"])
def test_decode_tiny_full(name):
    wl = G.workload(name)
    voc = G.gpu_decoder(wl)
    got = G.gpu_decode(voc, wl.latent)
    ref = O.decode(wl.arch, None, wl.latent, 0, G.oracle_folded(name))
    G.compare_audio(ref, got, name)


@pytest.mark.parametrize("T", [1, 2, 7, 31, 129])
def test_decode_edge_lengths(T):
    """Single frame, lengths inside one tile, one past a tile (in latent frames;
    every stage multiplies the rows, so the later layers see ragged tails too)."""
    wl = G.workload("tiny_cal")
    lat = np.random.default_rng(T).standard_normal((2, 16, T)).astype(np.float32)
    voc = G.gpu_decoder(wl)
    got = G.gpu_decode(voc, lat)
    ref = O.decode(wl.arch, None, lat, 0, G.oracle_folded("tiny_cal"))
    assert got.shape == (2, T * 512)
    G.compare_audio(ref, got, f"T={T}")


def test_empty_inputs_are_rejected_and_leave_the_context_usable():
    """B = 0 or T = 0 (zero-length views of a real latent, so the pointers are valid) is an
    invalid argument, rejected before any launch; the next decode through the same context
    gives the same audio bit for bit."""
    wl = G.workload("tiny_cal")
    voc = G.gpu_decoder(wl)
    before = G.gpu_decode(voc, wl.latent)
    lat = torch.from_numpy(wl.latent).cuda()
    audio = torch.empty((wl.B, 1, wl.T * voc.hop), device="cuda")
    ws = voc.alloc_workspace(wl.B, wl.T)
    for bad in (lat[:, :, :0], lat[:0]):
        with pytest.raises(V.VocoderError) as e:
            V.vocoder_decode(voc.handle, bad, audio, ws)
        assert e.value.status == V.VOC_INVALID_ARG
    assert voc.workspace_bytes(0, wl.T) == 0 and voc.workspace_bytes(wl.B, 0) == 0
    after = G.gpu_decode(voc, wl.latent)
    assert np.array_equal(before, after)
    voc.close()


def test_batch_equals_items():
    """Items of a batch decode independently: identical to one-item decodes, bit for bit."""
    wl = G.workload("tiny_cal")
    lat = np.random.default_rng(4).standard_normal((3, 16, 40)).astype(np.float32)
    voc = G.gpu_decoder(wl)
    yb = G.gpu_decode(voc, lat)
    for i in range(3):
        yi = G.gpu_decode(voc, lat[i:i + 1])
        np.testing.assert_array_equal(yb[i], yi[0])


MID_MUSIC = W.Arch(latent_channels=64, channels0=384, strides=(8, 8, 4, 2), widths=(192, 96, 96, 48))
MID_SPEECH = W.Arch(latent_channels=64, channels0=256, strides=(8, 5, 4, 4, 3),
                    widths=(192, 96, 48, 48, 32), padding=W.PAD_CAUSAL)


@pytest.mark.parametrize("arch", [MID_MUSIC, MID_SPEECH], ids=["music", "speech_causal"])
@pytest.mark.parametrize("fuse", [-1, 192], ids=["unfused", "fused"])
def test_decode_fusion_variants(arch, fuse):
    """Residual units as one fused kernel or as conv1 + conv2 kernels, over many tiles per
    CTA (several waves), checked sample by sample against the oracle."""
    wl = W.make_custom(arch, B=2, T=60, seed=71)
    voc = V.Vocoder(arch, V.fold_params(wl.params), fuse_max_channels=fuse)
    got = G.gpu_decode(voc, wl.latent)
    ref = O.decode(arch, wl.params, wl.latent)
    G.compare_audio(ref, got, f"fuse={fuse}")


def test_fused_units_match_two_kernel_units_on_the_music_window():
    """The bench's decoder with its residual units fused (the default) and as conv1 + conv2
    kernels: the same arithmetic in another summation order, so the two decodes agree within
    the audio tolerance everywhere, not only where the oracle samples them."""
    wl = G.workload("music_window")
    lat = wl.latent[:, :, :160]
    fused = G.gpu_decode(V.Vocoder(wl.arch, V.fold_params(wl.params)), lat)
    two = G.gpu_decode(V.Vocoder(wl.arch, V.fold_params(wl.params), fuse_max_channels=-1), lat)
    G.compare_audio(two, fused, "fused vs two-kernel residual units")


PROJ_MUSIC = W.Arch(latent_channels=64, channels0=384, strides=(8, 8, 4, 2), widths=(192, 96, 96, 48),
                    in_proj_channels=256)


def test_decode_input_projection():
    """The 1x1 input projection (no weight norm) in front of conv_in, over several waves,
    against the oracle sample by sample."""
    wl = W.make_custom(PROJ_MUSIC, B=2, T=60, seed=74)
    voc = V.Vocoder(PROJ_MUSIC, V.fold_params(wl.params))
    got = G.gpu_decode(voc, wl.latent)
    ref = O.decode(PROJ_MUSIC, wl.params, wl.latent)
    G.compare_audio(ref, got, "in_proj")


def test_decode_full_music_model_sampled():
    """The published 54 M music decoder (dec_in_proj 64 -> 1024, conv_in 1024 -> 1536) on the
    one-window music latent, checked on sampled windows against the oracle."""
    wl = W.make_custom(W.MUSIC_FULL, B=2, T=689, seed=2000)
    folded = O.fold_params(wl.params)
    voc = V.Vocoder(W.MUSIC_FULL, V.fold_params(wl.params))
    got = G.gpu_decode(voc, wl.latent)
    hop = wl.arch.hop
    assert got.shape == (2, 689 * hop)
    for item in range(2):
        for (a, b) in G.sampled_windows(wl.arch, wl.T, n=3, width=8):
            ref = G.oracle_window(wl, folded, item, a, b)
            G.compare_audio(ref, got[item, a * hop:b * hop], f"full[{item}][{a}:{b}]")


ODD_HEAD = W.Arch(latent_channels=16, channels0=64, strides=(4, 2), widths=(32, 16),
                  in_kernel=5, res_kernel=5, out_kernel=9)


def test_decode_other_kernel_sizes():
    """conv_in, residual and output kernels of 5, 5 and 9 taps (the 7-tap output head has its
    own register-blocked kernel; other tap counts take the general one)."""
    wl = W.make_custom(ODD_HEAD, B=2, T=50, seed=73)
    voc = V.Vocoder(ODD_HEAD, V.fold_params(wl.params))
    got = G.gpu_decode(voc, wl.latent)
    ref = O.decode(ODD_HEAD, wl.params, wl.latent)
    G.compare_audio(ref, got, "kernel sizes 5/5/9")


@pytest.mark.parametrize("arch", [MID_MUSIC, MID_SPEECH], ids=["music", "speech_causal"])
def test_decode_cta_pair(arch):
    """Every tensor-core layer on 2-CTA clusters (one 256-row MMA per pair, each CTA staging
    half of the weights) over several waves, checked sample by sample against the oracle,
    and against the single-CTA decode of the same input."""
    wl = W.make_custom(arch, B=2, T=60, seed=72)
    pair = V.Vocoder(arch, V.fold_params(wl.params), cta_pair=1)
    single = V.Vocoder(arch, V.fold_params(wl.params), cta_pair=-1)
    got = G.gpu_decode(pair, wl.latent)
    ref = O.decode(arch, wl.params, wl.latent)
    G.compare_audio(ref, got, "cta_pair=1")
    G.compare_audio(G.gpu_decode(single, wl.latent), got, "pair vs single")


def _sampled_full_size(name, n_items=None, width=8, n=3, cta_pair=0):
    wl = G.workload(name)
    folded = G.oracle_folded(name)
    voc = V.Vocoder(wl.arch, V.fold_params(wl.params), cta_pair=cta_pair)
    got = G.gpu_decode(voc, wl.latent)
    hop = wl.arch.hop
    assert got.shape == (wl.B, wl.T * hop)
    assert np.all(np.abs(got) <= 1.0)
    items = range(wl.B) if n_items is None else range(min(n_items, wl.B))
    worst_err, worst_snr = 0.0, np.inf
    for item in items:
        for (a, b) in G.sampled_windows(wl.arch, wl.T, n=n, width=width):
            ref = G.oracle_window(wl, folded, item, a, b)
            err, snr = G.compare_audio(ref, got[item, a * hop:b * hop], f"{name}[{item}][{a}:{b}]")
            worst_err, worst_snr = max(worst_err, err), min(worst_snr, snr)
    return got, worst_err, worst_snr


def test_decode_music_window_sampled():
    _sampled_full_size("music_window")


def test_decode_music_window_sampled_cta_pair():
    _sampled_full_size("music_window", cta_pair=1)


def test_decode_speech_sampled():
    _sampled_full_size("speech", n_items=3)


def test_decode_speech_snakebeta_sampled():
    """The speech codec with SnakeBeta activations (log-scale alpha and beta, exponentiated
    on the host), at the full workload size, on sampled windows."""
    _sampled_full_size("speech_snakebeta", n_items=2)


@pytest.mark.parametrize("arch", [MID_MUSIC, MID_SPEECH], ids=["music", "speech_causal"])
def test_decode_snake_beta(arch):
    """Every Snake as SnakeBeta, whole outputs against the oracle (fused and unfused
    residual units both run: the mid-size stages span both sides of the fusion limit)."""
    beta_arch = dataclasses.replace(arch, snake_beta=True)
    wl = W.make_custom(beta_arch, B=2, T=21, seed=303)
    voc = V.Vocoder(beta_arch, V.fold_params(wl.params))
    got = G.gpu_decode(voc, wl.latent)
    G.compare_audio(O.decode(beta_arch, wl.params, wl.latent), got, "snake_beta")


@pytest.mark.slow
def test_decode_music_long_sampled():
    _sampled_full_size("music_long", n=4)


def test_music_batch8_stitch():
    """Windowed workload: GPU decode of the 16 window items, GPU stitch, checked
    (a) bit-exactly against the oracle's stitch of the same decoded windows and
    (b) against the oracle's single pass over the continuous latent at sampled
    positions (the windows' crops exceed the receptive field)."""
    wl = G.workload("music_batch8")
    st = wl.stitch
    voc = G.gpu_decoder(wl)
    lat = torch.from_numpy(wl.latent).cuda()
    audio = voc.decode(lat, flags=V.VOC_FLAG_SYNC)
    n = V.vocoder_stitched_length(st["n_win"], st["win_frames"], st["crop_left"],
                                  st["crop_right"], st["hop"])
    assert n == 1589248
    out = torch.empty((st["n_sides"], n), dtype=torch.float32, device="cuda")
    V.vocoder_stitch(audio, st["n_win"], st["n_sides"], st["win_frames"], st["crop_left"],
                     st["crop_right"], st["hop"], out)
    torch.cuda.synchronize()
    dec = audio[:, 0].cpu().numpy().astype(np.float64)
    ref_st = O.stitch(dec, st["n_win"], st["n_sides"], st["win_frames"], st["crop_left"],
                      st["crop_right"], st["hop"])
    np.testing.assert_array_equal(out.cpu().numpy().astype(np.float64), ref_st)
    # against a single pass of the continuous latent
    cont = W.Workload(name="cont", arch=wl.arch, latent=wl.continuous_latent, params=wl.params)
    folded = G.oracle_folded("music_batch8")
    got = out.cpu().numpy().astype(np.float64)
    hop = wl.arch.hop
    total = wl.continuous_latent.shape[2]
    for side in range(2):
        for (a, b) in [(0, 6), (428, 434), (773, 779), (1500, 1506), (total - 6, total)]:
            ref = G.oracle_window(cont, folded, side, a, b)
            G.compare_audio(ref, got[side, a * hop:b * hop], f"stitch side {side} [{a}:{b}]")


# ----------------------------------------------------------------------------- API paths
def test_decode_host_matches_device():
    wl = G.workload("tiny_cal")
    voc = G.gpu_decoder(wl)
    lat = torch.from_numpy(wl.latent).pin_memory()
    out = torch.empty((wl.B, 1, wl.T * 512), dtype=torch.float32).pin_memory()
    ws = voc.alloc_workspace(wl.B, wl.T, host_io=True)
    V.vocoder_decode_host(voc.handle, lat, out, ws)
    dev = G.gpu_decode(voc, wl.latent)
    np.testing.assert_array_equal(out[:, 0].numpy().astype(np.float64), dev)


def test_workspace_too_small_and_nonfinite():
    wl = G.workload("tiny_cal")
    voc = G.gpu_decoder(wl)
    lat = torch.from_numpy(wl.latent).cuda()
    audio = torch.empty((1, 1, wl.T * 512), device="cuda")
    need = voc.workspace_bytes(1, wl.T)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(V.VocoderError) as e:
        V.vocoder_decode(voc.handle, lat, audio, small)
    assert e.value.status == V.VOC_WORKSPACE_TOO_SMALL
    bad = lat.clone()
    bad[0, 3, 5] = float("nan")
    ws = voc.alloc_workspace(1, wl.T)
    with pytest.raises(V.VocoderError) as e:
        V.vocoder_decode(voc.handle, bad, audio, ws, flags=V.VOC_FLAG_CHECK_FINITE)
    assert e.value.status == V.VOC_NONFINITE
    # the context stays usable after the error
    V.vocoder_decode(voc.handle, lat, audio, ws, flags=V.VOC_FLAG_CHECK_FINITE | V.VOC_FLAG_SYNC)


def test_profile_records_every_launch():
    wl = G.workload("tiny_cal")
    voc = G.gpu_decoder(wl)
    lat = torch.from_numpy(wl.latent).cuda()
    voc.decode(lat, flags=V.VOC_FLAG_PROFILE | V.VOC_FLAG_SYNC)
    prof = V.vocoder_profile(voc.handle)
    assert len(prof) == V.vocoder_launches_per_decode(voc.handle, 1, wl.T)
    assert all(p["ms"] >= 0 for p in prof)
    assert sum(p["flops"] for p in prof) > 0


@pytest.mark.parametrize("T", [1, 3, 4, 8, 9])
def test_folded_head_and_its_fallback(T):
    """The output head folded into the last conv2 (non-causal decoders) and its fallback to the
    separate head when the fold's partial sums would not fit the buffer it borrows (a one-stage
    decoder whose last stage is its widest: T <= 4 falls back, T >= 8 folds), both against the
    oracle; and a causal decoder of the same shape (always the separate head)."""
    sym = W.Arch(latent_channels=8, channels0=16, strides=(2,), widths=(64,))
    for arch in (sym, dataclasses.replace(sym, strides=(3,), padding=W.PAD_CAUSAL)):
        wl = W.make_custom(arch, B=2, T=T, seed=31 + T)
        voc = V.Vocoder(arch, V.fold_params(wl.params))
        got = G.gpu_decode(voc, wl.latent)
        ref = O.decode(arch, wl.params, wl.latent)
        G.compare_audio(ref, got, f"T={T} padding={arch.padding}")
        voc.close()
