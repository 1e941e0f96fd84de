"""GPU: the library's failure and control paths, each made to happen on purpose without
faulting the GPU.

* Bounded waits: a context whose wait bound is a few hundred cycles gives up inside its
  kernels (which drain their own copies and tensor-core work before returning) and the
  decode reports VOC_DEVICE_TIMEOUT; the same context with the default bound then decodes
  exactly as a fresh one does.
* Allocation failure: an out-of-memory cudaMalloc injected at every position of
  vocoder_create (and of vocoder_stream_create) returns VOC_OOM and leaves no device
  allocation behind.
* Cancellation (the pattern of minimaxmusic.cpp Architecture, "mm-server reference",
  "Concurrency": a cancel flag polled between VAE windows): with the flag set, every decode
  entry point returns VOC_CANCELLED without touching its outputs; cleared, decoding goes on.
"""
from __future__ import annotations

import ctypes

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

SMALL_CAUSAL = W.Arch(latent_channels=16, channels0=64, strides=(4, 2), widths=(48, 32),
                      padding=W.PAD_CAUSAL)


def test_short_wait_bound_reports_timeout_then_recovers():
    """The music decoder (a 32-frame window: every kernel's first waits last tens of
    microseconds, far longer than one suspended mbarrier wait) under a 300-cycle bound."""
    wl = G.workload("music_window", T=32, B=1)
    voc = G.gpu_decoder(wl)
    lat = torch.from_numpy(wl.latent).cuda()
    V.vocoder_set_wait_budget(voc.handle, 300)  # cycles: every kernel gives up at once
    for _ in range(2):  # twice: the first give-up leaves the context usable
        with pytest.raises(V.VocoderError) as e:
            voc.decode(lat, flags=V.VOC_FLAG_SYNC)
        assert e.value.status == V.VOC_DEVICE_TIMEOUT
        assert "bounded wait" in V.vocoder_last_error(voc.handle)
    V.vocoder_set_wait_budget(voc.handle, 0)  # the default bound again
    got = G.gpu_decode(voc, wl.latent)
    fresh = G.gpu_decoder(wl)
    np.testing.assert_array_equal(got, G.gpu_decode(fresh, wl.latent))
    assert np.all(np.isfinite(got)) and float(np.max(np.abs(got))) > 0.0
    with pytest.raises(V.VocoderError) as e:
        V.vocoder_set_wait_budget(voc.handle, -1)
    assert e.value.status == V.VOC_INVALID_ARG
    fresh.close()
    voc.close()


def _create_fails_cleanly(make, what, min_failures):
    """Inject an allocation failure at positions 0, 1, 2, ... of `make()` until it succeeds;
    every failing call must return VOC_OOM and leave the live allocation count unchanged."""
    live0 = V.vocoder_debug_live_allocations()
    n, failures = 0, 0
    try:
        while True:
            V.vocoder_debug_fail_allocation(n)
            try:
                obj = make()
            except V.VocoderError as e:
                assert e.status == V.VOC_OOM, (what, n, e)
                assert V.vocoder_debug_live_allocations() == live0, (what, n)
                failures += 1
                n = n + 1 if n < 8 else n * 2  # every early position, then doubling
                continue
            break
    finally:
        V.vocoder_debug_fail_allocation(-1)
    assert failures >= min_failures, (what, failures)
    return obj, live0


def test_injected_allocation_failure_in_create_frees_everything():
    wl = G.workload("tiny_cal")
    folded = V.fold_params(wl.params)
    voc, live0 = _create_fails_cleanly(lambda: V.Vocoder(wl.arch, folded), "vocoder_create",
                                      min_failures=10)
    assert V.vocoder_debug_live_allocations() > live0
    # the decoder that finally came up decodes correctly; destroying it frees everything
    G.compare_audio(O.decode(wl.arch, wl.params, wl.latent), G.gpu_decode(voc, wl.latent),
                    "decoder created after injected failures")
    voc.close()
    assert V.vocoder_debug_live_allocations() == live0


def test_injected_allocation_failure_in_stream_create():
    wl = W.make_custom(SMALL_CAUSAL, B=1, T=6, seed=91)
    voc = V.Vocoder(SMALL_CAUSAL, V.fold_params(wl.params))
    s, live0 = _create_fails_cleanly(lambda: V.VocoderStream(voc, 1, 3), "vocoder_stream_create",
                                    min_failures=1)
    s.close()
    assert V.vocoder_debug_live_allocations() == live0
    voc.close()


def test_cancel_flag_stops_every_decode_entry_point():
    wl = G.workload("tiny_cal")
    voc = G.gpu_decoder(wl)
    B, _, T = wl.latent.shape
    lat = torch.from_numpy(wl.latent).cuda()
    flag = ctypes.c_int(0)
    V.vocoder_set_cancel_flag(voc.handle, flag)
    before = G.gpu_decode(voc, wl.latent)  # flag clear: decodes
    flag.value = 1
    out = torch.full((B, 1, T * voc.hop), 7.0, device="cuda")
    ws = voc.alloc_workspace(B, T)
    calls = [
        lambda: V.vocoder_decode(voc.handle, lat, out, ws, flags=V.VOC_FLAG_SYNC),
        lambda: V.vocoder_decode_static(voc.handle, lat, out, flags=V.VOC_FLAG_SYNC),
        lambda: V.vocoder_decode_host(voc.handle, torch.from_numpy(wl.latent.copy()),
                                      torch.full((B, 1, T * voc.hop), 7.0),
                                      voc.alloc_workspace(B, T, host_io=True)),
    ]
    for call in calls:
        with pytest.raises(V.VocoderError) as e:
            call()
        assert e.value.status == V.VOC_CANCELLED
    torch.cuda.synchronize()
    assert bool(torch.all(out == 7.0))  # nothing was enqueued
    flag.value = 0
    np.testing.assert_array_equal(G.gpu_decode(voc, wl.latent), before)
    V.vocoder_set_cancel_flag(voc.handle, None)
    voc.close()


def test_cancel_flag_between_stream_chunks():
    wl = W.make_custom(SMALL_CAUSAL, B=1, T=6, seed=92)
    voc = V.Vocoder(SMALL_CAUSAL, V.fold_params(wl.params))
    whole = G.gpu_decode(voc, wl.latent)
    flag = ctypes.c_int(0)
    V.vocoder_set_cancel_flag(voc.handle, flag)
    s = V.VocoderStream(voc, 1, 3)
    lat = torch.from_numpy(wl.latent).cuda()
    first = s.decode(lat[:, :, :3].contiguous(), flags=V.VOC_FLAG_SYNC)
    flag.value = 1  # cancelled between two chunks: the second is refused, the state kept
    with pytest.raises(V.VocoderError) as e:
        s.decode(lat[:, :, 3:].contiguous(), flags=V.VOC_FLAG_SYNC)
    assert e.value.status == V.VOC_CANCELLED
    flag.value = 0  # resumed: the stream continues where it stopped
    second = s.decode(lat[:, :, 3:].contiguous(), flags=V.VOC_FLAG_SYNC)
    got = torch.cat([first, second], dim=2)[:, 0].cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(got, whole)
    V.vocoder_set_cancel_flag(voc.handle, None)
    s.close()
    voc.close()
