"""The no-allocation decode (vocoder_decode_static) against the regular decode.

vocoder_decode_static serves callers that may not call cudaMalloc while they
run -- a real-time audio thread, where an allocation can synchronise the device
and stall long enough to drop a buffer, or a host whose own allocator owns the
device memory.  It keeps its workspace in a fixed-size device array inside the
library.  These tests call it through the C ABI twice in a row (the array keeps
the first call's contents when the second starts) and require each result to
equal vocoder_decode's bit for bit: both run the same kernels on the same
inputs, so any difference would mean that the decode read a workspace byte it
had not written in that call (a stale value left by an earlier call).  The same
property is checked directly on the regular path, on a workspace filled with
0xFF bytes (NaN in every float and bf16 plane) beforehand.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("no CUDA device", allow_module_level=True)

from dac_vocoder_decode_gb300 import binding as V  # noqa: E402
from dac_vocoder_decode_gb300 import workloads as W  # noqa: E402


def _latent(rng, B, C, T):
    return torch.from_numpy(rng.standard_normal((B, C, T)).astype(np.float32)).cuda()


def _same(ref, got):
    torch.cuda.synchronize()
    assert bool(torch.all(torch.isfinite(got)))
    np.testing.assert_array_equal(got.cpu().numpy(), ref.cpu().numpy())


@pytest.mark.parametrize("name,B,T", [("tiny_cal", 2, 48), ("music_window", 1, 60)])
def test_static_workspace_decode_matches_regular_decode(name, B, T):
    wl = W.make_workload(name, T=T, B=B)
    voc = V.Vocoder(wl.arch, V.fold_params(wl.params))
    assert voc.workspace_bytes(B, T) <= V.VOC_STATIC_WORKSPACE_BYTES
    rng = np.random.default_rng(123)
    ws = voc.alloc_workspace(B, T)
    for call in range(2):  # two calls in a row: the second starts on the first's leftovers
        lat = _latent(rng, B, wl.arch.latent_channels, T)
        ref = torch.empty((B, 1, T * voc.hop), device="cuda")
        got = torch.full((B, 1, T * voc.hop), float("nan"), device="cuda")
        V.vocoder_decode(voc.handle, lat, ref, ws, flags=V.VOC_FLAG_SYNC)
        V.vocoder_decode_static(voc.handle, lat, got, flags=V.VOC_FLAG_SYNC)
        _same(ref, got)
    voc.close()


def test_static_workspace_after_a_larger_decode():
    """A larger decode leaves valid data all over the array; a shorter one whose planes end
    on other rows (37 frames: not a multiple of 8 at the latent rate) must not read it."""
    wl = W.make_workload("tiny_cal", T=48, B=2)
    voc = V.Vocoder(wl.arch, V.fold_params(wl.params))
    rng = np.random.default_rng(7)
    C = wl.arch.latent_channels
    for B, T in [(3, 64), (1, 37), (2, 21)]:
        lat = _latent(rng, B, C, T)
        ref = torch.empty((B, 1, T * voc.hop), device="cuda")
        got = torch.full((B, 1, T * voc.hop), float("nan"), device="cuda")
        V.vocoder_decode(voc.handle, lat, ref, voc.alloc_workspace(B, T), flags=V.VOC_FLAG_SYNC)
        V.vocoder_decode_static(voc.handle, lat, got, flags=V.VOC_FLAG_SYNC)
        _same(ref, got)
    voc.close()


def test_regular_decode_ignores_a_poisoned_workspace():
    wl = W.make_workload("tiny_cal", T=37, B=2)
    voc = V.Vocoder(wl.arch, V.fold_params(wl.params))
    B, T = 2, 37
    lat = torch.from_numpy(wl.latent).cuda()
    clean = voc.alloc_workspace(B, T).zero_()
    poisoned = voc.alloc_workspace(B, T).fill_(0xFF)
    ref = torch.empty((B, 1, T * voc.hop), device="cuda")
    got = torch.empty((B, 1, T * voc.hop), device="cuda")
    V.vocoder_decode(voc.handle, lat, ref, clean, flags=V.VOC_FLAG_SYNC)
    V.vocoder_decode(voc.handle, lat, got, poisoned, flags=V.VOC_FLAG_SYNC)
    _same(ref, got)
    voc.close()


def test_static_workspace_rejects_sizes_beyond_its_array():
    wl = W.make_workload("tiny_cal")
    voc = V.Vocoder(wl.arch, V.fold_params(wl.params))
    T = 4096  # the tiny decoder needs 16 * 16 * 512 bytes of workspace per latent frame
    assert voc.workspace_bytes(1, T) > V.VOC_STATIC_WORKSPACE_BYTES
    lat = torch.zeros((1, wl.arch.latent_channels, T), device="cuda")
    out = torch.empty((1, 1, T * voc.hop), device="cuda")
    with pytest.raises(V.VocoderError) as e:
        V.vocoder_decode_static(voc.handle, lat, out)
    assert e.value.status == V.VOC_WORKSPACE_TOO_SMALL
    assert "workspace" in V.vocoder_last_error(voc.handle)
    voc.close()
