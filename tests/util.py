"""Test helpers: receptive fields from the layer list, error metrics.

Nothing here repeats the oracle's arithmetic; the receptive field is derived
from the layer shapes alone (taps, dilations, strides, paddings)."""
from __future__ import annotations

import math

import numpy as np

from dac_vocoder_decode_gb300.workloads import PAD_CAUSAL


def _conv_pads(arch, K, d):
    span = d * (K - 1)
    if arch.padding == PAD_CAUSAL:
        return span, 0
    return span // 2, span - span // 2


def latent_span(arch, j: int):
    """Inclusive interval [lo, hi] of latent frames that output sample j can depend on.

    Walks the stack from the output back to the latent.  A k-tap conv with left
    pad pl and dilation d maps [a, b] to [a - pl, b - pl + d(k-1)]; a transposed
    conv of stride s, K = 2s, left crop p maps [a, b] to
    [ceil((a + p - K + 1)/s), floor((b + p)/s)]; a residual unit adds its conv1
    span (conv2 is 1x1 and the skip is the identity)."""
    a = b = j
    pl, _ = _conv_pads(arch, arch.out_kernel, 1)
    a, b = a - pl, b - pl + (arch.out_kernel - 1)
    for st in reversed(range(len(arch.strides))):
        for d in reversed(arch.dilations):
            pl, _ = _conv_pads(arch, arch.res_kernel, d)
            a, b = a - pl, b - pl + d * (arch.res_kernel - 1)
        s = arch.strides[st]
        K = 2 * s
        p = 0 if arch.padding == PAD_CAUSAL else s // 2
        a, b = -((-(a + p - K + 1)) // s), (b + p) // s
    pl, _ = _conv_pads(arch, arch.in_kernel, 1)
    a, b = a - pl, b - pl + (arch.in_kernel - 1)
    return a, b


def frame_margins(arch):
    """(left, right): how many latent frames before / after its own frame an
    output sample can depend on, maximised over the hop phases."""
    hop = arch.hop
    t0 = 64
    left = right = 0
    for r in range(hop):
        lo, hi = latent_span(arch, t0 * hop + r)
        left = max(left, t0 - lo)
        right = max(right, hi - t0)
    return left, right


def snr_db(ref: np.ndarray, got: np.ndarray) -> float:
    ref = np.asarray(ref, dtype=np.float64)
    err = np.asarray(got, dtype=np.float64) - ref
    num = float(np.sum(ref * ref))
    den = float(np.sum(err * err))
    if den == 0.0:
        return math.inf
    return 10.0 * math.log10(num / den)


def encoder_sample_span(arch, u: int):
    """Inclusive interval [lo, hi] of audio samples that latent frame u of the (non-causal)
    mirror encoder can depend on.  Walks from the latent back to the audio: a k-tap conv
    with dilation d maps [a, b] to [a - d(k-1)/2, b + d(k-1)/2]; a strided conv of stride s,
    k = 2s, pad s/2 maps [a, b] to [a s - s/2, b s - s/2 + 2s - 1]; a residual unit adds its
    conv1 span."""
    a = b = u
    h = (arch.out_kernel - 1) // 2
    a, b = a - h, b + h
    for st in reversed(range(len(arch.strides))):
        s = arch.strides[st]
        a, b = a * s - s // 2, b * s - s // 2 + 2 * s - 1
        for d in reversed(arch.dilations):
            h = d * (arch.res_kernel - 1) // 2
            a, b = a - h, b + h
    h = (arch.in_kernel - 1) // 2
    return a - h, b + h


def encoder_frame_margins(arch):
    """(left, right) latent frames of audio context that one latent frame reads around its
    own hop of samples."""
    hop = arch.hop
    u = 64
    lo, hi = encoder_sample_span(arch, u)
    left = -((lo - u * hop) // hop)
    right = -(-(hi - (u * hop + hop - 1)) // hop)
    return max(left, 0), max(right, 0)
