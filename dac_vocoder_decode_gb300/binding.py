"""ctypes binding of libvocoder.so (include/vocoder.h), with the same entry-point names.

Argument marshalling only: every step of the decode runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  If the compiled library
is missing this module raises instead of falling back to anything else; build
it with ``python -m dac_vocoder_decode_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import numpy as np

from . import build as _build

VOC_ABI_VERSION = 5
VOC_OK = 0
VOC_INVALID_ARG = -1
VOC_UNSUPPORTED = -2
VOC_CUDA_ERROR = -3
VOC_OOM = -4
VOC_WORKSPACE_TOO_SMALL = -5
VOC_NONFINITE = -6
VOC_CANCELLED = -7
VOC_DEVICE_TIMEOUT = -8
VOC_PAD_SYMMETRIC = 0
VOC_PAD_CAUSAL = 1
VOC_PREC_BF16X3 = 0
VOC_PREC_F16W = 1
VOC_PREC_BF16W = 2
VOC_SNAKE = 0
VOC_SNAKE_BETA = 1
VOC_FLAG_CHECK_FINITE = 1
VOC_FLAG_SYNC = 2
VOC_FLAG_PROFILE = 4

STATUS_NAMES = {0: "VOC_OK", -1: "VOC_INVALID_ARG", -2: "VOC_UNSUPPORTED", -3: "VOC_CUDA_ERROR",
                -4: "VOC_OOM", -5: "VOC_WORKSPACE_TOO_SMALL", -6: "VOC_NONFINITE",
                -7: "VOC_CANCELLED", -8: "VOC_DEVICE_TIMEOUT"}

EXPORTED = [
    "vocoder_abi_version", "vocoder_param_count", "vocoder_param_shape",
    "vocoder_fold_weight_norm", "vocoder_create", "vocoder_hop", "vocoder_workspace_bytes",
    "vocoder_workspace_bytes_host", "vocoder_decode", "vocoder_decode_host",
    "vocoder_decode_static",
    "vocoder_stitched_length", "vocoder_stitch", "vocoder_op_conv1d",
    "vocoder_op_conv_transpose1d", "vocoder_op_residual_unit", "vocoder_launches_per_decode",
    "vocoder_profile_count",
    "vocoder_profile_entry", "vocoder_profile_impl_bytes", "vocoder_last_error",
    "vocoder_destroy", "vocoder_set_cancel_flag", "vocoder_set_wait_budget",
    "vocoder_debug_fail_allocation", "vocoder_debug_live_allocations",
    "vocoder_stream_create", "vocoder_stream_decode", "vocoder_stream_reset",
    "vocoder_stream_destroy", "vocoder_wav_bytes", "vocoder_wav_scratch_bytes",
    "vocoder_encode_wav",
    "vocoder_encoder_param_count", "vocoder_encoder_param_shape", "vocoder_encoder_create",
    "vocoder_encoder_hop", "vocoder_encoder_workspace_bytes", "vocoder_encode",
    "vocoder_encoder_workspace_bytes_host", "vocoder_encode_host",
    "vocoder_encoder_launches", "vocoder_encoder_profile_count", "vocoder_encoder_profile_entry",
    "vocoder_encoder_profile_impl_bytes",
    "vocoder_encoder_last_error", "vocoder_encoder_destroy",
]


class VocoderError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class VocDesc(ctypes.Structure):
    _fields_ = [("abi_version", ctypes.c_int), ("latent_channels", ctypes.c_int),
                ("in_kernel", ctypes.c_int), ("channels0", ctypes.c_int),
                ("n_stages", ctypes.c_int), ("strides", ctypes.POINTER(ctypes.c_int)),
                ("widths", ctypes.POINTER(ctypes.c_int)), ("n_dilations", ctypes.c_int),
                ("dilations", ctypes.POINTER(ctypes.c_int)), ("res_kernel", ctypes.c_int),
                ("out_kernel", ctypes.c_int), ("out_channels", ctypes.c_int),
                ("padding", ctypes.c_int), ("precision", ctypes.c_int),
                ("fuse_max_channels", ctypes.c_int), ("cta_pair", ctypes.c_int),
                ("in_proj_channels", ctypes.c_int), ("snake", ctypes.c_int)]


class VocEncDesc(ctypes.Structure):
    _fields_ = [("abi_version", ctypes.c_int), ("in_channels", ctypes.c_int),
                ("channels0", ctypes.c_int), ("in_kernel", ctypes.c_int),
                ("n_stages", ctypes.c_int), ("strides", ctypes.POINTER(ctypes.c_int)),
                ("widths", ctypes.POINTER(ctypes.c_int)), ("n_dilations", ctypes.c_int),
                ("dilations", ctypes.POINTER(ctypes.c_int)), ("res_kernel", ctypes.c_int),
                ("out_kernel", ctypes.c_int), ("latent_channels", ctypes.c_int),
                ("precision", ctypes.c_int), ("snake", ctypes.c_int)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load_library():
    """Load libvocoder.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -m dac_vocoder_decode_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    F = ctypes.POINTER(ctypes.c_float)
    lib.vocoder_abi_version.restype = I
    lib.vocoder_abi_version.argtypes = []
    lib.vocoder_param_count.restype = I
    lib.vocoder_param_count.argtypes = [ctypes.POINTER(VocDesc)]
    lib.vocoder_param_shape.restype = I
    lib.vocoder_param_shape.argtypes = [ctypes.POINTER(VocDesc), I, ctypes.POINTER(I),
                                        ctypes.POINTER(I)]
    lib.vocoder_fold_weight_norm.restype = I
    lib.vocoder_fold_weight_norm.argtypes = [F, F, I, ctypes.c_longlong, F]
    lib.vocoder_create.restype = I
    lib.vocoder_create.argtypes = [ctypes.POINTER(VocDesc), ctypes.POINTER(F), I,
                                   ctypes.POINTER(P)]
    lib.vocoder_hop.restype = ctypes.c_longlong
    lib.vocoder_hop.argtypes = [P]
    lib.vocoder_workspace_bytes.restype = ctypes.c_size_t
    lib.vocoder_workspace_bytes.argtypes = [P, I, I]
    lib.vocoder_workspace_bytes_host.restype = ctypes.c_size_t
    lib.vocoder_workspace_bytes_host.argtypes = [P, I, I]
    lib.vocoder_decode.restype = I
    lib.vocoder_decode.argtypes = [P, P, I, I, P, P, ctypes.c_size_t, P, ctypes.c_uint]
    lib.vocoder_decode_host.restype = I
    lib.vocoder_decode_host.argtypes = [P, P, I, I, P, P, ctypes.c_size_t, P, ctypes.c_uint]
    lib.vocoder_decode_static.restype = I
    lib.vocoder_decode_static.argtypes = [P, P, I, I, P, P, ctypes.c_uint]
    lib.vocoder_stitched_length.restype = ctypes.c_longlong
    lib.vocoder_stitched_length.argtypes = [I, I, I, I, I]
    lib.vocoder_stitch.restype = I
    lib.vocoder_stitch.argtypes = [P, I, I, I, I, I, I, P, P]
    lib.vocoder_op_conv1d.restype = I
    lib.vocoder_op_conv1d.argtypes = [P, I, I, I, F, F, I, I, I, I, F, P, P]
    lib.vocoder_op_conv_transpose1d.restype = I
    lib.vocoder_op_conv_transpose1d.argtypes = [P, I, I, I, F, F, I, I, I, F, P, P]
    lib.vocoder_op_residual_unit.restype = I
    lib.vocoder_op_residual_unit.argtypes = [P, I, I, I, F, F, F, I, I, F, F, F, I, P, P]
    lib.vocoder_launches_per_decode.restype = I
    lib.vocoder_launches_per_decode.argtypes = [P, I, I]
    lib.vocoder_profile_count.restype = I
    lib.vocoder_profile_count.argtypes = [P]
    lib.vocoder_profile_entry.restype = I
    lib.vocoder_profile_entry.argtypes = [P, I, ctypes.POINTER(ctypes.c_char_p),
                                          ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(ctypes.c_double)]
    lib.vocoder_profile_impl_bytes.restype = I
    lib.vocoder_profile_impl_bytes.argtypes = [P, I, ctypes.POINTER(ctypes.c_double)]
    lib.vocoder_last_error.restype = ctypes.c_char_p
    lib.vocoder_last_error.argtypes = [P]
    lib.vocoder_destroy.restype = None
    lib.vocoder_destroy.argtypes = [P]
    lib.vocoder_set_cancel_flag.restype = I
    lib.vocoder_set_cancel_flag.argtypes = [P, P]
    lib.vocoder_set_wait_budget.restype = I
    lib.vocoder_set_wait_budget.argtypes = [P, ctypes.c_longlong]
    lib.vocoder_debug_fail_allocation.restype = None
    lib.vocoder_debug_fail_allocation.argtypes = [I]
    lib.vocoder_debug_live_allocations.restype = ctypes.c_longlong
    lib.vocoder_debug_live_allocations.argtypes = []
    lib.vocoder_wav_bytes.restype = ctypes.c_size_t
    lib.vocoder_wav_bytes.argtypes = [I, ctypes.c_longlong, I]
    lib.vocoder_wav_scratch_bytes.restype = ctypes.c_size_t
    lib.vocoder_wav_scratch_bytes.argtypes = []
    lib.vocoder_encode_wav.restype = I
    lib.vocoder_encode_wav.argtypes = [P, I, ctypes.c_longlong, I, I, I, P, ctypes.c_size_t, P,
                                       ctypes.c_size_t, P]
    lib.vocoder_stream_create.restype = I
    lib.vocoder_stream_create.argtypes = [P, I, I, ctypes.POINTER(P)]
    lib.vocoder_stream_decode.restype = I
    lib.vocoder_stream_decode.argtypes = [P, P, I, P, P, ctypes.c_uint]
    lib.vocoder_stream_reset.restype = I
    lib.vocoder_stream_reset.argtypes = [P, P]
    lib.vocoder_stream_destroy.restype = None
    lib.vocoder_stream_destroy.argtypes = [P]
    ED = ctypes.POINTER(VocEncDesc)
    lib.vocoder_encoder_param_count.restype = I
    lib.vocoder_encoder_param_count.argtypes = [ED]
    lib.vocoder_encoder_param_shape.restype = I
    lib.vocoder_encoder_param_shape.argtypes = [ED, I, ctypes.POINTER(I), ctypes.POINTER(I)]
    lib.vocoder_encoder_create.restype = I
    lib.vocoder_encoder_create.argtypes = [ED, ctypes.POINTER(F), I, ctypes.POINTER(P)]
    lib.vocoder_encoder_hop.restype = ctypes.c_longlong
    lib.vocoder_encoder_hop.argtypes = [P]
    lib.vocoder_encoder_workspace_bytes.restype = ctypes.c_size_t
    lib.vocoder_encoder_workspace_bytes.argtypes = [P, I, ctypes.c_longlong]
    lib.vocoder_encode.restype = I
    lib.vocoder_encode.argtypes = [P, P, I, ctypes.c_longlong, P, P, ctypes.c_size_t, P,
                                   ctypes.c_uint]
    lib.vocoder_encoder_workspace_bytes_host.restype = ctypes.c_size_t
    lib.vocoder_encoder_workspace_bytes_host.argtypes = [P, I, ctypes.c_longlong]
    lib.vocoder_encode_host.restype = I
    lib.vocoder_encode_host.argtypes = [P, P, I, ctypes.c_longlong, P, P, ctypes.c_size_t, P,
                                        ctypes.c_uint]
    lib.vocoder_encoder_launches.restype = I
    lib.vocoder_encoder_launches.argtypes = [P, I, ctypes.c_longlong]
    lib.vocoder_encoder_profile_count.restype = I
    lib.vocoder_encoder_profile_count.argtypes = [P]
    lib.vocoder_encoder_profile_entry.restype = I
    lib.vocoder_encoder_profile_entry.argtypes = [P, I, ctypes.POINTER(ctypes.c_char_p),
                                                  ctypes.POINTER(ctypes.c_double),
                                                  ctypes.POINTER(ctypes.c_double),
                                                  ctypes.POINTER(ctypes.c_double)]
    lib.vocoder_encoder_profile_impl_bytes.restype = I
    lib.vocoder_encoder_profile_impl_bytes.argtypes = [P, I, ctypes.POINTER(ctypes.c_double)]
    lib.vocoder_encoder_last_error.restype = ctypes.c_char_p
    lib.vocoder_encoder_last_error.argtypes = [P]
    lib.vocoder_encoder_destroy.restype = None
    lib.vocoder_encoder_destroy.argtypes = [P]
    _lib = lib
    return lib


def _check(status: int, handle=None):
    if status != VOC_OK:
        msg = load_library().vocoder_last_error(handle)
        raise VocoderError(status, msg.decode() if msg else "")


def _fptr(a: Optional[np.ndarray]):
    if a is None:
        return ctypes.cast(None, ctypes.POINTER(ctypes.c_float))
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    if hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


def make_desc(arch, fuse_max_channels: int = 0, cta_pair: int = 0,
              precision: int = VOC_PREC_BF16X3) -> VocDesc:
    """voc_desc for an Arch (layer shapes from workloads.Arch or any object with the same fields)."""
    strides = (ctypes.c_int * len(arch.strides))(*arch.strides)
    widths = (ctypes.c_int * len(arch.widths))(*arch.widths)
    dils = (ctypes.c_int * len(arch.dilations))(*arch.dilations)
    d = VocDesc(VOC_ABI_VERSION, arch.latent_channels, arch.in_kernel, arch.channels0,
                len(arch.strides), strides, widths, len(arch.dilations), dils, arch.res_kernel,
                arch.out_kernel, 1, arch.padding, precision, fuse_max_channels, cta_pair,
                getattr(arch, "in_proj_channels", 0),
                VOC_SNAKE_BETA if getattr(arch, "snake_beta", False) else VOC_SNAKE)
    d._keep = (strides, widths, dils)
    return d


# ------------------------------------------------------------------ entry points
def vocoder_abi_version() -> int:
    return load_library().vocoder_abi_version()


def vocoder_param_count(arch) -> int:
    return load_library().vocoder_param_count(ctypes.byref(make_desc(arch)))


def vocoder_param_shape(arch, index: int):
    dims = (ctypes.c_int * 3)()
    nd = ctypes.c_int()
    _check(load_library().vocoder_param_shape(ctypes.byref(make_desc(arch)), index, dims,
                                               ctypes.byref(nd)))
    return tuple(dims[i] for i in range(nd.value))


def vocoder_fold_weight_norm(g: np.ndarray, v: np.ndarray) -> np.ndarray:
    g = np.ascontiguousarray(g, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    w = np.empty_like(v)
    rest = int(np.prod(v.shape[1:])) if v.ndim > 1 else 1
    _check(load_library().vocoder_fold_weight_norm(_fptr(g), _fptr(v), int(v.shape[0]), rest,
                                                    _fptr(w)))
    return w


def vocoder_create(arch, params: Sequence[Optional[np.ndarray]],
                   fuse_max_channels: int = 0, cta_pair: int = 0,
                   precision: int = VOC_PREC_BF16X3) -> ctypes.c_void_p:
    """params: folded fp32 arrays in the canonical order (None for a zero bias)."""
    lib = load_library()
    keep = [None if p is None else np.ascontiguousarray(p, dtype=np.float32) for p in params]
    arr = (ctypes.POINTER(ctypes.c_float) * len(keep))(*[_fptr(p) for p in keep])
    h = ctypes.c_void_p()
    _check(lib.vocoder_create(ctypes.byref(make_desc(arch, fuse_max_channels, cta_pair, precision)), arr,
                              len(keep),
                              ctypes.byref(h)))
    return h


def vocoder_destroy(h) -> None:
    load_library().vocoder_destroy(h)


def vocoder_hop(h) -> int:
    return int(load_library().vocoder_hop(h))


def vocoder_workspace_bytes(h, B: int, T: int) -> int:
    return int(load_library().vocoder_workspace_bytes(h, B, T))


def vocoder_workspace_bytes_host(h, B: int, T: int) -> int:
    return int(load_library().vocoder_workspace_bytes_host(h, B, T))


def vocoder_launches_per_decode(h, B: int, T: int) -> int:
    return int(load_library().vocoder_launches_per_decode(h, B, T))


def vocoder_decode(h, latent, audio, ws, stream=None, flags: int = 0) -> None:
    """latent [B,C,T] fp32 CUDA tensor -> audio [B,1,T*hop] fp32 CUDA tensor; ws uint8 CUDA tensor."""
    B, _, T = latent.shape
    _check(load_library().vocoder_decode(h, ctypes.c_void_p(latent.data_ptr()), B, T,
                                          ctypes.c_void_p(audio.data_ptr()),
                                          ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                          _stream_ptr(stream), flags), h)


def vocoder_decode_host(h, latent_host, audio_host, ws, stream=None, flags: int = 0) -> None:
    """Host (ideally pinned) CPU tensors in and out; copies happen inside the library."""
    B, _, T = latent_host.shape
    _check(load_library().vocoder_decode_host(h, ctypes.c_void_p(latent_host.data_ptr()), B, T,
                                               ctypes.c_void_p(audio_host.data_ptr()),
                                               ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                               _stream_ptr(stream), flags), h)


VOC_STATIC_WORKSPACE_BYTES = 64 << 20


def vocoder_decode_static(h, latent, audio, stream=None, flags: int = 0) -> None:
    """Decode with the library's built-in workspace array: no device allocation
    happens in this call (for callers that may not allocate while they run, such
    as real-time audio threads).  Calls that overlap on the GPU race on the array."""
    B, _, T = latent.shape
    _check(load_library().vocoder_decode_static(h, ctypes.c_void_p(latent.data_ptr()), B, T,
                                                 ctypes.c_void_p(audio.data_ptr()),
                                                 _stream_ptr(stream), flags), h)


def vocoder_stitched_length(n_win, win_frames, crop_left, crop_right, hop) -> int:
    return int(load_library().vocoder_stitched_length(n_win, win_frames, crop_left, crop_right,
                                                      hop))


def vocoder_stitch(decoded, n_win, n_sides, win_frames, crop_left, crop_right, hop, out,
                   stream=None) -> None:
    _check(load_library().vocoder_stitch(ctypes.c_void_p(decoded.data_ptr()), n_win, n_sides,
                                          win_frames, crop_left, crop_right, hop,
                                          ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream)))


def vocoder_op_conv1d(x, w: np.ndarray, b: Optional[np.ndarray], dil: int, padding: int,
                      alpha: Optional[np.ndarray], y, stream=None) -> None:
    B, Cin, T = x.shape
    Cout, _, K = w.shape
    w = np.ascontiguousarray(w, dtype=np.float32)
    b = None if b is None else np.ascontiguousarray(b, dtype=np.float32)
    alpha = None if alpha is None else np.ascontiguousarray(alpha, dtype=np.float32)
    _check(load_library().vocoder_op_conv1d(ctypes.c_void_p(x.data_ptr()), B, Cin, T, _fptr(w),
                                             _fptr(b), Cout, K, dil, padding, _fptr(alpha),
                                             ctypes.c_void_p(y.data_ptr()), _stream_ptr(stream)))


def vocoder_op_conv_transpose1d(x, w: np.ndarray, b: Optional[np.ndarray], stride: int,
                                padding: int, alpha: Optional[np.ndarray], y,
                                stream=None) -> None:
    B, Cin, T = x.shape
    _, Cout, K = w.shape
    assert K == 2 * stride
    w = np.ascontiguousarray(w, dtype=np.float32)
    b = None if b is None else np.ascontiguousarray(b, dtype=np.float32)
    alpha = None if alpha is None else np.ascontiguousarray(alpha, dtype=np.float32)
    _check(load_library().vocoder_op_conv_transpose1d(
        ctypes.c_void_p(x.data_ptr()), B, Cin, T, _fptr(w), _fptr(b), Cout, stride, padding,
        _fptr(alpha), ctypes.c_void_p(y.data_ptr()), _stream_ptr(stream)))


def vocoder_op_residual_unit(x, alpha1: np.ndarray, w1: np.ndarray, b1: Optional[np.ndarray],
                             dil: int, alpha2: np.ndarray, w2: np.ndarray,
                             b2: Optional[np.ndarray], padding: int, y, stream=None) -> None:
    """y = x + conv2(Snake2(conv1(Snake1(x)) + b1)) + b2 on the decoder's kernels."""
    B, C, T = x.shape
    K = w1.shape[2]
    arrs = [np.ascontiguousarray(a, dtype=np.float32) if a is not None else None
            for a in (alpha1, w1, b1, alpha2, w2, b2)]
    _check(load_library().vocoder_op_residual_unit(
        ctypes.c_void_p(x.data_ptr()), B, C, T, _fptr(arrs[0]), _fptr(arrs[1]), _fptr(arrs[2]),
        K, dil, _fptr(arrs[3]), _fptr(arrs[4]), _fptr(arrs[5]), padding,
        ctypes.c_void_p(y.data_ptr()), _stream_ptr(stream)))


def vocoder_profile(h) -> List[dict]:
    """Per-kernel records of the last decode run with VOC_FLAG_PROFILE."""
    lib = load_library()
    out = []
    for i in range(lib.vocoder_profile_count(h)):
        name = ctypes.c_char_p()
        ms, fl, by = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
        _check(lib.vocoder_profile_entry(h, i, ctypes.byref(name), ctypes.byref(ms),
                                          ctypes.byref(fl), ctypes.byref(by)), h)
        ib = ctypes.c_double()
        _check(lib.vocoder_profile_impl_bytes(h, i, ctypes.byref(ib)), h)
        out.append(dict(name=name.value.decode(), ms=ms.value, flops=fl.value, bytes=by.value,
                        impl_bytes=ib.value))
    return out


def vocoder_set_cancel_flag(h, flag: Optional[ctypes.c_int]) -> None:
    """Register a host int (a ctypes.c_int the caller keeps alive) as the context's cancel
    flag; None removes it."""
    ptr = ctypes.cast(ctypes.pointer(flag), ctypes.c_void_p) if flag is not None else None
    _check(load_library().vocoder_set_cancel_flag(h, ptr), h)


def vocoder_set_wait_budget(h, cycles: int) -> None:
    _check(load_library().vocoder_set_wait_budget(h, int(cycles)), h)


def vocoder_debug_fail_allocation(n: int) -> None:
    load_library().vocoder_debug_fail_allocation(int(n))


def vocoder_debug_live_allocations() -> int:
    return int(load_library().vocoder_debug_live_allocations())


def vocoder_last_error(h=None) -> str:
    m = load_library().vocoder_last_error(h)
    return m.decode() if m else ""


# ------------------------------------------------------------------ convenience
def fold_params(params) -> list:
    """Raw canonical parameters (weight-norm g/v pairs and alphas) -> folded fp32
    arrays through the library's host fold (vocoder_fold_weight_norm)."""
    out = []
    for p in params:
        if hasattr(p, "g"):
            out.append(vocoder_fold_weight_norm(p.g, p.v))
            out.append(None if p.b is None else np.ascontiguousarray(p.b, dtype=np.float32))
        elif hasattr(p, "w"):  # a convolution stored without weight norm
            out.append(np.ascontiguousarray(p.w, dtype=np.float32))
            out.append(None if p.b is None else np.ascontiguousarray(p.b, dtype=np.float32))
        else:
            out.append(np.ascontiguousarray(p, dtype=np.float32))
    return out


def vocoder_stream_create(h, B: int, max_frames: int) -> ctypes.c_void_p:
    s = ctypes.c_void_p()
    _check(load_library().vocoder_stream_create(h, B, max_frames, ctypes.byref(s)), h)
    return s


def vocoder_stream_decode(h, s, latent, audio, stream=None, flags: int = 0) -> None:
    """latent [B, C_lat, frames] and audio [B, 1, frames*hop]: contiguous fp32 CUDA tensors."""
    frames = int(latent.shape[2])
    _check(load_library().vocoder_stream_decode(s, ctypes.c_void_p(latent.data_ptr()), frames,
                                                 ctypes.c_void_p(audio.data_ptr()),
                                                 _stream_ptr(stream), flags), h)


def vocoder_stream_reset(h, s, stream=None) -> None:
    _check(load_library().vocoder_stream_reset(s, _stream_ptr(stream)), h)


def vocoder_stream_destroy(s) -> None:
    load_library().vocoder_stream_destroy(s)


def vocoder_wav_bytes(n_ch: int, length: int, bits: int) -> int:
    return int(load_library().vocoder_wav_bytes(n_ch, length, bits))


def vocoder_wav_scratch_bytes() -> int:
    return int(load_library().vocoder_wav_scratch_bytes())


def vocoder_encode_wav(planar, sample_rate: int, bits: int, peak_clip: int, out, scratch=None,
                       stream=None) -> None:
    """planar: contiguous fp32 CUDA tensor [n_ch, len]; out: uint8 CUDA tensor of at least
    vocoder_wav_bytes bytes; scratch: uint8 CUDA tensor of vocoder_wav_scratch_bytes (16/24
    bits)."""
    n_ch, length = (1, int(planar.shape[0])) if planar.dim() == 1 else map(int, planar.shape)
    sp = ctypes.c_void_p(scratch.data_ptr()) if scratch is not None else None
    sb = scratch.numel() if scratch is not None else 0
    _check(load_library().vocoder_encode_wav(ctypes.c_void_p(planar.data_ptr()), n_ch, length,
                                              sample_rate, bits, peak_clip,
                                              ctypes.c_void_p(out.data_ptr()), out.numel(), sp,
                                              sb, _stream_ptr(stream)), None)


def encode_wav(planar, sample_rate: int, bits: int = 16, peak_clip: int = 0, stream=None):
    """Peak-normalise and encode planar [n_ch, len] device audio as a WAV file in a new uint8
    CUDA tensor (see vocoder_encode_wav in include/vocoder.h)."""
    import torch
    planar = planar.contiguous()
    n_ch, length = (1, planar.shape[0]) if planar.dim() == 1 else planar.shape
    size = vocoder_wav_bytes(int(n_ch), int(length), bits)
    if size == 0:
        raise VocoderError(-1, "bad WAV geometry")
    # 256 bytes of head room keep the scratch that follows the file 256-byte aligned
    off = (size + 255) // 256 * 256
    buf = torch.empty(off + vocoder_wav_scratch_bytes(), dtype=torch.uint8, device=planar.device)
    vocoder_encode_wav(planar, sample_rate, bits, peak_clip, buf[:size], buf[off:], stream)
    return buf[:size]


class VocoderStream:
    """Stateful chunk-by-chunk decoding of B sequences on a causal decoder (see
    vocoder_stream_create in include/vocoder.h)."""

    def __init__(self, voc: "Vocoder", B: int, max_frames: int):
        self.voc = voc
        self.B = B
        self.max_frames = max_frames
        self.handle = vocoder_stream_create(voc.handle, B, max_frames)

    def decode(self, latent, audio=None, stream=None, flags: int = 0):
        import torch
        if audio is None:
            audio = torch.empty((self.B, 1, latent.shape[2] * self.voc.hop), dtype=torch.float32,
                                device=latent.device)
        vocoder_stream_decode(self.voc.handle, self.handle, latent.contiguous(), audio, stream,
                              flags)
        return audio

    def reset(self, stream=None):
        vocoder_stream_reset(self.voc.handle, self.handle, stream)

    def close(self):
        if self.handle:
            vocoder_stream_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Vocoder:
    """A decoder on the current CUDA device (owns its library context)."""

    def __init__(self, arch, folded_params, fuse_max_channels: int = 0, cta_pair: int = 0,
                 precision: int = VOC_PREC_BF16X3):
        self.arch = arch
        self.handle = vocoder_create(arch, folded_params, fuse_max_channels, cta_pair, precision)
        self.hop = vocoder_hop(self.handle)

    def close(self):
        if self.handle:
            vocoder_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace_bytes(self, B: int, T: int) -> int:
        return vocoder_workspace_bytes(self.handle, B, T)

    def alloc_workspace(self, B: int, T: int, host_io: bool = False):
        import torch
        n = (vocoder_workspace_bytes_host if host_io else vocoder_workspace_bytes)(self.handle, B, T)
        return torch.empty(n, dtype=torch.uint8, device="cuda")

    def decode(self, latent, ws=None, audio=None, stream=None, flags: int = 0):
        import torch
        B, _, T = latent.shape
        if ws is None:
            ws = self.alloc_workspace(B, T)
        if audio is None:
            audio = torch.empty((B, 1, T * self.hop), dtype=torch.float32, device=latent.device)
        vocoder_decode(self.handle, latent, audio, ws, stream, flags)
        return audio


# ------------------------------------------------------------------ mirror encoder
def _check_enc(status: int, handle=None):
    if status != VOC_OK:
        msg = load_library().vocoder_encoder_last_error(handle)
        raise VocoderError(status, msg.decode() if msg else "")


def make_enc_desc(arch, precision: int = VOC_PREC_BF16X3) -> VocEncDesc:
    """voc_enc_desc for an encoder architecture (workloads.EncArch or the same fields)."""
    strides = (ctypes.c_int * len(arch.strides))(*arch.strides)
    widths = (ctypes.c_int * len(arch.widths))(*arch.widths)
    dils = (ctypes.c_int * len(arch.dilations))(*arch.dilations)
    d = VocEncDesc(VOC_ABI_VERSION, arch.in_channels, arch.channels0, arch.in_kernel,
                   len(arch.strides), strides, widths, len(arch.dilations), dils,
                   arch.res_kernel, arch.out_kernel, arch.latent_channels, precision,
                   VOC_SNAKE_BETA if getattr(arch, "snake_beta", False) else VOC_SNAKE)
    d._keep = (strides, widths, dils)
    return d


def vocoder_encoder_param_count(arch) -> int:
    return load_library().vocoder_encoder_param_count(ctypes.byref(make_enc_desc(arch)))


def vocoder_encoder_param_shape(arch, index: int):
    dims = (ctypes.c_int * 3)()
    nd = ctypes.c_int()
    _check_enc(load_library().vocoder_encoder_param_shape(ctypes.byref(make_enc_desc(arch)), index,
                                                          dims, ctypes.byref(nd)))
    return tuple(dims[i] for i in range(nd.value))


def vocoder_encoder_create(arch, params: Sequence[Optional[np.ndarray]],
                           precision: int = VOC_PREC_BF16X3) -> ctypes.c_void_p:
    """params: folded fp32 arrays in the encoder's canonical order (None for a zero bias)."""
    keep = [None if p is None else np.ascontiguousarray(p, dtype=np.float32) for p in params]
    arr = (ctypes.POINTER(ctypes.c_float) * len(keep))(*[_fptr(p) for p in keep])
    h = ctypes.c_void_p()
    _check_enc(load_library().vocoder_encoder_create(ctypes.byref(make_enc_desc(arch, precision)),
                                                     arr, len(keep), ctypes.byref(h)))
    return h


def vocoder_encoder_destroy(h) -> None:
    load_library().vocoder_encoder_destroy(h)


def vocoder_encoder_hop(h) -> int:
    return int(load_library().vocoder_encoder_hop(h))


def vocoder_encoder_workspace_bytes(h, B: int, L: int) -> int:
    return int(load_library().vocoder_encoder_workspace_bytes(h, B, L))


def vocoder_encoder_workspace_bytes_host(h, B: int, L: int) -> int:
    return int(load_library().vocoder_encoder_workspace_bytes_host(h, B, L))


def vocoder_encode_host(h, audio_host, latent_host, ws, stream=None, flags: int = 0) -> None:
    """Host (ideally pinned) CPU tensors in and out; copies happen inside the library."""
    B, _, L = audio_host.shape
    _check_enc(load_library().vocoder_encode_host(h, ctypes.c_void_p(audio_host.data_ptr()), B, L,
                                                  ctypes.c_void_p(latent_host.data_ptr()),
                                                  ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                                  _stream_ptr(stream), flags), h)


def vocoder_encoder_launches(h, B: int, L: int) -> int:
    return int(load_library().vocoder_encoder_launches(h, B, L))


def vocoder_encode(h, audio, latent, ws, stream=None, flags: int = 0) -> None:
    """audio [B, C_in, L] fp32 CUDA tensor -> latent [B, C_lat, L / hop] fp32 CUDA tensor."""
    B, _, L = audio.shape
    _check_enc(load_library().vocoder_encode(h, ctypes.c_void_p(audio.data_ptr()), B, L,
                                             ctypes.c_void_p(latent.data_ptr()),
                                             ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                             _stream_ptr(stream), flags), h)


def vocoder_encoder_profile(h) -> List[dict]:
    """Per-kernel records of the last encode run with VOC_FLAG_PROFILE."""
    lib = load_library()
    out = []
    for i in range(lib.vocoder_encoder_profile_count(h)):
        name = ctypes.c_char_p()
        ms, fl, by = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
        _check_enc(lib.vocoder_encoder_profile_entry(h, i, ctypes.byref(name), ctypes.byref(ms),
                                                     ctypes.byref(fl), ctypes.byref(by)), h)
        ib = ctypes.c_double()
        _check_enc(lib.vocoder_encoder_profile_impl_bytes(h, i, ctypes.byref(ib)), h)
        out.append(dict(name=name.value.decode(), ms=ms.value, flops=fl.value, bytes=by.value,
                        impl_bytes=ib.value))
    return out


def vocoder_encoder_last_error(h=None) -> str:
    m = load_library().vocoder_encoder_last_error(h)
    return m.decode() if m else ""


class Encoder:
    """The mirror encoder on the current CUDA device (owns its library context)."""

    def __init__(self, arch, folded_params, precision: int = VOC_PREC_BF16X3):
        self.arch = arch
        self.handle = vocoder_encoder_create(arch, folded_params, precision)
        self.hop = vocoder_encoder_hop(self.handle)

    def close(self):
        if self.handle:
            vocoder_encoder_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace_bytes(self, B: int, L: int) -> int:
        return vocoder_encoder_workspace_bytes(self.handle, B, L)

    def alloc_workspace(self, B: int, L: int, host_io: bool = False):
        import torch
        n = (vocoder_encoder_workspace_bytes_host if host_io else vocoder_encoder_workspace_bytes)(
            self.handle, B, L)
        return torch.empty(n, dtype=torch.uint8, device="cuda")

    def encode(self, audio, ws=None, latent=None, stream=None, flags: int = 0):
        import torch
        B, _, L = audio.shape
        if ws is None:
            ws = self.alloc_workspace(B, L)
        if latent is None:
            latent = torch.empty((B, self.arch.latent_channels, L // self.hop), dtype=torch.float32,
                                 device=audio.device)
        vocoder_encode(self.handle, audio.contiguous(), latent, ws, stream, flags)
        return latent
