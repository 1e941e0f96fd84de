"""Seeded synthetic inputs for the vocoder decoder: architectures, latents, raw weights.

This module is shared by the tests, the benchmark and the smoke check, and it
feeds both the CUDA library and the CPU oracle.  It holds NONE of the method's
arithmetic: it draws random numbers and describes layer shapes, nothing else.
Weight-norm folding, Snake, the convolutions and the stitch live on each side
separately.

Distributions (no trained weights exist for this decoder here, so every input
is synthetic):

* latent ~ N(0, 1) fp32, shape [B, C_lat, T].
* alpha  ~ U(0.5, 1.5) per channel for every Snake; for SnakeBeta decoders (log-scale
  alpha and beta) log U(0.5, 1.5) for each of the two, so that exp(alpha) and exp(beta)
  have the plain Snake's alpha distribution.
* convolution weights in weight-norm form (g, v):
  - "literal" (tiny decoder): g, v, bias ~ N(0, 0.02).
  - "calibrated" (all other workloads): v ~ N(0, 1), g = gain * U(0.9, 1.1),
    bias ~ N(0, 0.02), with gain 1 for conv_in, sqrt(s/2) for the transposed
    conv of stride s (variance preserving: its norm runs over C_out * 2s taps
    and each output sample sees 2 taps of 2*C_out inputs), 0.5 for the two
    convolutions of a residual unit and 0.3 for conv_out (set once so that
    the pre-tanh RMS of every calibrated workload lies in [0.05, 1]).
* seeds: 1000 * workload index + {0: latent, 1: weights, 2: alpha}, numpy PCG64.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

PAD_SYMMETRIC = 0
PAD_CAUSAL = 1


@dataclasses.dataclass(frozen=True)
class Arch:
    """Layer shapes of one decoder (minimaxmusic.cpp Architecture, "Flow VAE")."""

    latent_channels: int
    channels0: int
    strides: Tuple[int, ...]
    widths: Tuple[int, ...]
    dilations: Tuple[int, ...] = (1, 3, 9)
    in_kernel: int = 7
    res_kernel: int = 7
    out_kernel: int = 7
    padding: int = PAD_SYMMETRIC
    # 0, or P: a 1x1 projection C_lat -> P (bias, no weight norm) before conv_in (the
    # published music model's dec_in_proj 64 -> 1024; conv_in then maps P -> channels0)
    in_proj_channels: int = 0
    # SnakeBeta activations (the speech codec's, qwentts.cpp Architecture): every Snake
    # parameter is [2, C], log-scale alpha then log-scale beta
    snake_beta: bool = False

    @property
    def hop(self) -> int:
        return int(np.prod(self.strides))

    def stage_channels(self) -> List[Tuple[int, int]]:
        """(C_in, C_out) of every upsampling stage."""
        cins = [self.channels0] + list(self.widths[:-1])
        return list(zip(cins, self.widths))

    def param_shapes(self) -> List[Tuple[str, Tuple[int, ...]]]:
        """Canonical order and PyTorch layouts of the folded parameter tensors.

        conv weights [C_out, C_in, K]; transposed-conv weights [C_in, C_out, K];
        biases [C_out]; Snake alphas [C] (SnakeBeta: [2, C], log alpha and log beta)."""
        out: List[Tuple[str, Tuple[int, ...]]] = []

        def sn(c):
            return (2, c) if self.snake_beta else (c,)

        c_in = self.latent_channels
        if self.in_proj_channels:
            out.append(("in_proj.w", (self.in_proj_channels, self.latent_channels, 1)))
            out.append(("in_proj.b", (self.in_proj_channels,)))
            c_in = self.in_proj_channels
        out.append(("conv_in.w", (self.channels0, c_in, self.in_kernel)))
        out.append(("conv_in.b", (self.channels0,)))
        for i, ((cin, cout), s) in enumerate(zip(self.stage_channels(), self.strides)):
            out.append((f"block{i}.snake.alpha", sn(cin)))
            out.append((f"block{i}.convT.w", (cin, cout, 2 * s)))
            out.append((f"block{i}.convT.b", (cout,)))
            for j, _d in enumerate(self.dilations):
                out.append((f"block{i}.res{j}.snake1.alpha", sn(cout)))
                out.append((f"block{i}.res{j}.conv1.w", (cout, cout, self.res_kernel)))
                out.append((f"block{i}.res{j}.conv1.b", (cout,)))
                out.append((f"block{i}.res{j}.snake2.alpha", sn(cout)))
                out.append((f"block{i}.res{j}.conv2.w", (cout, cout, 1)))
                out.append((f"block{i}.res{j}.conv2.b", (cout,)))
        c_last = self.widths[-1]
        out.append(("snake_out.alpha", sn(c_last)))
        out.append(("conv_out.w", (1, c_last, self.out_kernel)))
        out.append(("conv_out.b", (1,)))
        return out


@dataclasses.dataclass(frozen=True)
class EncArch:
    """Layer shapes of the mirror encoder (minimaxmusic.cpp Architecture, "Flow VAE": per
    side, conv_in, blocks of residual units followed by Snake and a strided conv k = 2s,
    Snake, conv_out k3 and the posterior mean projection k1)."""

    in_channels: int
    channels0: int
    strides: Tuple[int, ...]
    widths: Tuple[int, ...]  # output channels of each block's strided conv
    latent_channels: int
    dilations: Tuple[int, ...] = (1, 3, 9)
    in_kernel: int = 7
    res_kernel: int = 7
    out_kernel: int = 3
    snake_beta: bool = False

    @property
    def hop(self) -> int:
        return int(np.prod(self.strides))

    def block_channels(self) -> List[Tuple[int, int]]:
        """(C_in, C_out) of every downsampling block."""
        cins = [self.channels0] + list(self.widths[:-1])
        return list(zip(cins, self.widths))

    def param_shapes(self) -> List[Tuple[str, Tuple[int, ...]]]:
        """Canonical order and PyTorch layouts (conv weights [C_out, C_in, K])."""
        def sn(c):
            return (2, c) if self.snake_beta else (c,)

        out: List[Tuple[str, Tuple[int, ...]]] = []
        out.append(("conv_in.w", (self.channels0, self.in_channels, self.in_kernel)))
        out.append(("conv_in.b", (self.channels0,)))
        for i, ((cin, cout), s) in enumerate(zip(self.block_channels(), self.strides)):
            for j, _d in enumerate(self.dilations):
                out.append((f"block{i}.res{j}.snake1.alpha", sn(cin)))
                out.append((f"block{i}.res{j}.conv1.w", (cin, cin, self.res_kernel)))
                out.append((f"block{i}.res{j}.conv1.b", (cin,)))
                out.append((f"block{i}.res{j}.snake2.alpha", sn(cin)))
                out.append((f"block{i}.res{j}.conv2.w", (cin, cin, 1)))
                out.append((f"block{i}.res{j}.conv2.b", (cin,)))
            out.append((f"block{i}.snake.alpha", sn(cin)))
            out.append((f"block{i}.down.w", (cout, cin, 2 * s)))
            out.append((f"block{i}.down.b", (cout,)))
        c_last = self.widths[-1]
        out.append(("snake_out.alpha", sn(c_last)))
        out.append(("conv_out.w", (c_last, c_last, self.out_kernel)))
        out.append(("conv_out.b", (c_last,)))
        out.append(("proj.w", (self.latent_channels, c_last, 1)))
        out.append(("proj.b", (self.latent_channels,)))
        return out


@dataclasses.dataclass
class RawConv:
    """A convolution in weight-norm form: w = g * v / ||v|| along axis 0 of v."""

    g: np.ndarray  # [v.shape[0]]
    v: np.ndarray  # PyTorch layout
    b: Optional[np.ndarray]


@dataclasses.dataclass
class PlainConv:
    """A convolution stored without weight norm (the input projection)."""

    w: np.ndarray  # PyTorch layout
    b: Optional[np.ndarray]


@dataclasses.dataclass
class Workload:
    name: str
    arch: Arch
    latent: np.ndarray  # [B, C_lat, T] fp32
    params: list  # canonical order; RawConv for (w, b) pairs, np.ndarray for alphas
    # windowed stitch (the batch of overlapping windows), else None
    stitch: Optional[dict] = None
    continuous_latent: Optional[np.ndarray] = None

    @property
    def B(self) -> int:
        return int(self.latent.shape[0])

    @property
    def T(self) -> int:
        return int(self.latent.shape[2])

    @property
    def out_samples(self) -> int:
        return self.B * self.T * self.arch.hop


MUSIC = Arch(latent_channels=64, channels0=1536, strides=(8, 8, 4, 2), widths=(768, 384, 192, 96))
SPEECH = Arch(latent_channels=1024, channels0=1536, strides=(8, 5, 4, 4, 3),
              widths=(768, 384, 192, 96, 48), padding=PAD_CAUSAL)
TINY = Arch(latent_channels=16, channels0=64, strides=(8, 8, 4, 2), widths=(32, 16, 8, 4))
# the published music model's front end: dec_in_proj 64 -> 1024, conv_in 1024 -> 1536
MUSIC_FULL = dataclasses.replace(MUSIC, in_proj_channels=1024)
# the speech codec's own activation (qwentts.cpp Architecture, "Audio tokenizer decoder")
SPEECH_BETA = dataclasses.replace(SPEECH, snake_beta=True)

# name -> (index used for seeds, arch, latent shape, weight recipe, description)
WORKLOADS = {
    "tiny": (1, TINY, (1, 16, 32), "literal",
             "tiny DAC decoder fp32, latent [1,16,32], literal g,v ~ N(0,.02)"),
    "tiny_cal": (1, TINY, (1, 16, 32), "calibrated",
                 "tiny DAC decoder fp32, latent [1,16,32], calibrated gains"),
    "music_window": (2, MUSIC, (2, 64, 689), "calibrated",
                     "music vocoder, one 689-frame window, stereo pair [2,64,689] -> [2,1,352768]"),
    "music_batch8": (3, MUSIC, (16, 64, 689), "calibrated",
                     "music vocoder, 8 overlapping windows x stereo [16,64,689] + overlap-crop stitch"),
    "music_long": (4, MUSIC, (2, 64, 15504), "calibrated",
                   "music vocoder, 180 s single pass [2,64,15504] -> [2,1,7938048]"),
    "speech": (5, SPEECH, (8, 1024, 250), "calibrated",
               "speech codec DAC decoder, causal, hop 1920, [8,1024,250] -> [8,1,480000]"),
    "speech_snakebeta": (6, SPEECH_BETA, (8, 1024, 250), "calibrated",
                         "speech codec DAC decoder with SnakeBeta activations, causal, hop 1920, "
                         "[8,1024,250] -> [8,1,480000]"),
}

# overlap-crop stitch of the windowed music workload (minimaxmusic.cpp
# Architecture, "Denoising stage" and "Decode and stitch")
STITCH_WINDOWS = 8
STITCH_WIN_FRAMES = 689
STITCH_CROP_LEFT = 86
STITCH_CROP_RIGHT = 258
STITCH_HOP_FRAMES = STITCH_WIN_FRAMES - STITCH_CROP_LEFT - STITCH_CROP_RIGHT  # 345


def gen_params(arch: Arch, recipe: str, seed_w: int, seed_a: int) -> list:
    """Raw parameters in canonical order (see Arch.param_shapes)."""
    rw = np.random.Generator(np.random.PCG64(seed_w))
    ra = np.random.Generator(np.random.PCG64(seed_a))

    def conv(shape, gain):
        if recipe == "literal":
            v = (rw.standard_normal(shape, dtype=np.float32) * np.float32(0.02))
            g = (rw.standard_normal((shape[0],), dtype=np.float32) * np.float32(0.02))
        else:
            v = rw.standard_normal(shape, dtype=np.float32)
            g = (gain * rw.uniform(0.9, 1.1, size=(shape[0],))).astype(np.float32)
        return v, g

    def bias(n):
        return (rw.standard_normal((n,), dtype=np.float32) * np.float32(0.02))

    def alpha(shape):
        if len(shape) == 2:  # SnakeBeta: log alpha, log beta
            return np.log(ra.uniform(0.5, 1.5, size=shape)).astype(np.float32)
        return ra.uniform(0.5, 1.5, size=shape).astype(np.float32)

    shapes = arch.param_shapes()
    out = []
    i = 0
    while i < len(shapes):
        name, shape = shapes[i]
        if name.endswith(".alpha"):
            out.append(alpha(shape))
            i += 1
            continue
        assert name.endswith(".w")
        if name.startswith("in_proj"):
            # no weight norm: w ~ N(0, 1/C_lat) (calibrated, variance preserving) or N(0, .02)
            std = 0.02 if recipe == "literal" else 1.0 / math.sqrt(shape[1])
            w = (rw.standard_normal(shape, dtype=np.float32) * np.float32(std))
            out.append(PlainConv(w=w, b=bias(shapes[i + 1][1][0])))
            i += 2
            continue
        if name.startswith("conv_in"):
            gain = 1.0
        elif ".convT." in name:
            stride = shape[2] // 2
            gain = math.sqrt(stride / 2.0)
        elif ".down." in name or name.startswith("proj"):
            gain = 1.0  # the norm runs over every input a strided or 1x1 output sees
        elif name.startswith("conv_out"):
            gain = 0.3
        else:
            gain = 0.5
        v, g = conv(shape, gain)
        b = bias(shapes[i + 1][1][0])
        out.append(RawConv(g=g, v=v, b=b))
        i += 2
    return out


def make_workload(name: str, T: Optional[int] = None, B: Optional[int] = None) -> Workload:
    """Build a named workload.  T / B override the latent length / batch (used
    for reduced-size parity cases; the seeds stay those of the named workload)."""
    idx, arch, shape, recipe, _desc = WORKLOADS[name]
    b, c, t = shape
    if T is not None:
        t = T
    if B is not None:
        b = B
    params = gen_params(arch, recipe, 1000 * idx + 1, 1000 * idx + 2)
    rl = np.random.Generator(np.random.PCG64(1000 * idx + 0))
    stitch = None
    cont = None
    if name == "music_batch8" and T is None and B is None:
        n_sides = 2
        total = STITCH_HOP_FRAMES * (STITCH_WINDOWS - 1) + STITCH_WIN_FRAMES  # 3104
        cont = rl.standard_normal((n_sides, c, total), dtype=np.float32)
        lat = np.empty((STITCH_WINDOWS * n_sides, c, STITCH_WIN_FRAMES), dtype=np.float32)
        for w in range(STITCH_WINDOWS):
            off = w * STITCH_HOP_FRAMES
            for side in range(n_sides):
                lat[w * n_sides + side] = cont[side, :, off:off + STITCH_WIN_FRAMES]
        stitch = dict(n_win=STITCH_WINDOWS, n_sides=n_sides, win_frames=STITCH_WIN_FRAMES,
                      crop_left=STITCH_CROP_LEFT, crop_right=STITCH_CROP_RIGHT, hop=arch.hop)
    else:
        lat = rl.standard_normal((b, c, t), dtype=np.float32)
    return Workload(name=name, arch=arch, latent=lat, params=params, stitch=stitch,
                    continuous_latent=cont)


def make_custom(arch: Arch, B: int, T: int, seed: int, recipe: str = "calibrated") -> Workload:
    """A workload for an arbitrary architecture (small parity and pin cases)."""
    params = gen_params(arch, recipe, seed + 1, seed + 2)
    rl = np.random.Generator(np.random.PCG64(seed))
    lat = rl.standard_normal((B, arch.latent_channels, T), dtype=np.float32)
    return Workload(name=f"custom{seed}", arch=arch, latent=lat, params=params)


# the music model's encoder: 64 -> 128 -> 256 -> 512 -> 1024 over strides 2, 4, 8, 8 (x512)
ENC_MUSIC = EncArch(in_channels=1, channels0=64, strides=(2, 4, 8, 8), widths=(128, 256, 512, 1024),
                    latent_channels=64)


def make_encode_workload(arch: EncArch, B: int, frames: int, seed: int,
                         recipe: str = "calibrated") -> Workload:
    """Audio [B, in_channels, frames * hop] in (-1, 1) (tanh of N(0, 0.5^2) samples) and the
    encoder's raw parameters; the audio is stored in the workload's `latent` field."""
    params = gen_params(arch, recipe, seed + 1, seed + 2)
    rl = np.random.Generator(np.random.PCG64(seed))
    audio = np.tanh(rl.standard_normal((B, arch.in_channels, frames * arch.hop),
                                       dtype=np.float32) * np.float32(0.5)).astype(np.float32)
    return Workload(name=f"encode{seed}", arch=arch, latent=audio, params=params)


# Encoder workloads: (arch, B, frames, seed, description); audio of frames * hop samples.
ENC_WORKLOADS = {
    "encode_music_window": (ENC_MUSIC, 2, 689, 21,
                            "music encoder, one stereo 689-frame window: audio [2,1,352768] -> "
                            "latent [2,64,689]"),
}


def make_named_encode_workload(name: str, frames: Optional[int] = None) -> Workload:
    arch, B, fr, seed, _desc = ENC_WORKLOADS[name]
    return make_encode_workload(arch, B, frames or fr, seed)


def slice_latent(latent: np.ndarray, t0: int, t1: int) -> np.ndarray:
    """Frames [t0, t1) of a latent (a copy), for receptive-field sampled checks."""
    return np.ascontiguousarray(latent[:, :, t0:t1])
