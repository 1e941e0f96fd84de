"""The no-allocation decode (vocoder_decode_static) against the regular decode.

vocoder_decode_static serves callers that may not call cudaMalloc while they
run -- a real-time audio thread, where an allocation can synchronise the device
and stall long enough to drop a buffer, or a host whose own allocator owns the
device memory.  It keeps its workspace in a fixed-size device array inside the
library.  These tests call it through the C ABI twice in a row (the array keeps
the first call's contents when the second starts) and check each result against
vocoder_decode, which takes a caller-provided workspace, within the audio
tolerance used by every decode test (max |err| <= 2e-3, SNR >= 60 dB).

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
from tests.util import snr_db  # noqa: E402

MAX_ABS = 2e-3
MIN_SNR_DB = 60.0


def _check_close(ref, got):
    ref = ref.double().cpu().numpy()
    got = got.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert float(np.max(np.abs(ref - got))) <= MAX_ABS
    assert snr_db(ref, got) >= MIN_SNR_DB


@pytest.mark.parametrize("name,B,T", [("tiny_cal", 2, 48), ("music_window", 1, 60)])
def test_static_workspace_decode_matches_regular_decode(name, B, T):
    wl = W.make_workload(name, T=T, B=B)
    voc = V.Vocoder(wl.arch, V.fold_params(wl.params))
    assert voc.workspace_bytes(B, T) <= V.VOC_STATIC_WORKSPACE_BYTES
    rng = np.random.default_rng(123)
    ws = voc.alloc_workspace(B, T)
    for call in range(2):  # two calls in a row: the second starts on the first's leftovers
        lat = torch.from_numpy(
            rng.standard_normal((B, wl.arch.latent_channels, T)).astype(np.float32)).cuda()
        ref = torch.empty((B, 1, T * voc.hop), device="cuda")
        got = torch.full((B, 1, T * voc.hop), float("nan"), device="cuda")
        V.vocoder_decode(voc.handle, lat, ref, ws, flags=V.VOC_FLAG_SYNC)
        V.vocoder_decode_static(voc.handle, lat, got, flags=V.VOC_FLAG_SYNC)
        torch.cuda.synchronize()
        _check_close(ref, got)
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
