"""ctypes wrapper around the CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
benchmark's CPU-baseline / reference leg.  The product path never imports it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FLAG_SNAKE_IDENTITY = 1
FLAG_NO_TANH = 2


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (plain C99 + OpenMP, IEEE arithmetic)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC),
                                              os.path.getmtime(os.path.join(_HERE, "oracle.h")))):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC,
           "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            D = ctypes.POINTER(ctypes.c_double)
            F = ctypes.POINTER(ctypes.c_float)
            lib.oracle_fold_weight_norm.argtypes = [F, F, ctypes.c_int, ctypes.c_long, D]
            lib.oracle_fold_weight_norm.restype = ctypes.c_int
            lib.oracle_round_half.argtypes = [D, ctypes.c_long, D]
            lib.oracle_round_half.restype = None
            lib.oracle_round_bf16.argtypes = [D, ctypes.c_long, D]
            lib.oracle_round_bf16.restype = None
            lib.oracle_snake_row.argtypes = [D, ctypes.c_long, ctypes.c_double, ctypes.c_int, D]
            lib.oracle_snake_row.restype = None
            lib.oracle_snake_beta_row.argtypes = [D, ctypes.c_long, ctypes.c_double,
                                                  ctypes.c_double, D]
            lib.oracle_snake_beta_row.restype = None
            lib.oracle_conv1d.argtypes = [D, ctypes.c_int, ctypes.c_int, D, D, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, D]
            lib.oracle_conv1d.restype = ctypes.c_int
            lib.oracle_conv_transpose1d.argtypes = [D, ctypes.c_int, ctypes.c_int, D, D,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int, ctypes.c_int, D]
            lib.oracle_conv_transpose1d.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [ctypes.c_void_p, ctypes.POINTER(D), F, ctypes.c_int,
                                          ctypes.c_int, D, D]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_stitched_length.argtypes = [ctypes.c_int] * 5
            lib.oracle_stitched_length.restype = ctypes.c_long
            lib.oracle_stitch.argtypes = [D, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, D]
            lib.oracle_stitch.restype = ctypes.c_int
            lib.oracle_enc_param_count.argtypes = [ctypes.c_void_p]
            lib.oracle_enc_param_count.restype = ctypes.c_int
            lib.oracle_conv1d_strided.argtypes = [D, ctypes.c_int, ctypes.c_int, D, D, ctypes.c_int,
                                                  ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, D]
            lib.oracle_conv1d_strided.restype = ctypes.c_int
            lib.oracle_encode.argtypes = [ctypes.c_void_p, ctypes.POINTER(D), F, ctypes.c_int,
                                          ctypes.c_long, D]
            lib.oracle_encode.restype = ctypes.c_int
            lib.oracle_param_count.argtypes = [ctypes.c_void_p]
            lib.oracle_param_count.restype = ctypes.c_int
            lib.oracle_abs_percentile.argtypes = [F, ctypes.c_long, ctypes.c_int]
            lib.oracle_abs_percentile.restype = ctypes.c_double
            lib.oracle_wav_bytes.argtypes = [ctypes.c_int, ctypes.c_long, ctypes.c_int]
            lib.oracle_wav_bytes.restype = ctypes.c_long
            lib.oracle_encode_wav.argtypes = [F, ctypes.c_int, ctypes.c_long, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int,
                                              ctypes.POINTER(ctypes.c_ubyte)]
            lib.oracle_encode_wav.restype = ctypes.c_int
            _lib = lib
    return _lib


def _d(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


class _ArchC(ctypes.Structure):
    _fields_ = [("latent_channels", ctypes.c_int), ("channels0", ctypes.c_int),
                ("in_kernel", ctypes.c_int), ("n_stages", ctypes.c_int),
                ("strides", ctypes.POINTER(ctypes.c_int)), ("widths", ctypes.POINTER(ctypes.c_int)),
                ("n_dilations", ctypes.c_int), ("dilations", ctypes.POINTER(ctypes.c_int)),
                ("res_kernel", ctypes.c_int), ("out_kernel", ctypes.c_int),
                ("padding", ctypes.c_int), ("flags", ctypes.c_int),
                ("in_proj_channels", ctypes.c_int), ("snake_beta", ctypes.c_int)]


class _EncArchC(ctypes.Structure):
    _fields_ = [("in_channels", ctypes.c_int), ("channels0", ctypes.c_int),
                ("in_kernel", ctypes.c_int), ("n_stages", ctypes.c_int),
                ("strides", ctypes.POINTER(ctypes.c_int)), ("widths", ctypes.POINTER(ctypes.c_int)),
                ("n_dilations", ctypes.c_int), ("dilations", ctypes.POINTER(ctypes.c_int)),
                ("res_kernel", ctypes.c_int), ("out_kernel", ctypes.c_int),
                ("latent_channels", ctypes.c_int), ("flags", ctypes.c_int),
                ("snake_beta", ctypes.c_int)]


def fold_weight_norm(g: np.ndarray, v: np.ndarray) -> np.ndarray:
    """w = g * v / ||v|| along axis 0 (double result)."""
    lib = _load()
    g = np.ascontiguousarray(g, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    w = np.empty(v.shape, dtype=np.float64)
    rest = int(np.prod(v.shape[1:])) if v.ndim > 1 else 1
    rc = lib.oracle_fold_weight_norm(_f(g), _f(v), int(v.shape[0]), rest, _d(w))
    if rc != 0:
        raise ValueError("weight norm: a row of v has zero norm")
    return w


def snake(x: np.ndarray, alpha: np.ndarray, identity: bool = False) -> np.ndarray:
    """Per-channel Snake of a [C, L] array."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    C, L = x.shape
    for c in range(C):
        lib.oracle_snake_row(_d(x[c]), L, float(alpha[c]), int(identity), _d(y[c]))
    return y


def snake_beta(x: np.ndarray, log_alpha: np.ndarray, log_beta: np.ndarray) -> np.ndarray:
    """Per-channel SnakeBeta (log-scale alpha and beta) of a [C, L] array."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    C, L = x.shape
    for c in range(C):
        lib.oracle_snake_beta_row(_d(x[c]), L, float(log_alpha[c]), float(log_beta[c]), _d(y[c]))
    return y


def conv1d(x: np.ndarray, w: np.ndarray, b: Optional[np.ndarray], dil: int, pad_left: int,
           pad_right: int) -> np.ndarray:
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    Cin, T = x.shape
    Cout, Cin2, K = w.shape
    assert Cin2 == Cin
    T_out = T + pad_left + pad_right - dil * (K - 1)
    y = np.empty((Cout, T_out), dtype=np.float64)
    bb = None if b is None else np.ascontiguousarray(b, dtype=np.float64)
    rc = lib.oracle_conv1d(_d(x), Cin, T, _d(w), None if bb is None else _d(bb), Cout, K, dil,
                           pad_left, pad_right, _d(y))
    assert rc == 0
    return y


def conv_transpose1d(x: np.ndarray, w: np.ndarray, b: Optional[np.ndarray], stride: int,
                     pad_left: int, T_out: int) -> np.ndarray:
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    Cin, T = x.shape
    Cin2, Cout, K = w.shape
    assert Cin2 == Cin
    y = np.empty((Cout, T_out), dtype=np.float64)
    bb = None if b is None else np.ascontiguousarray(b, dtype=np.float64)
    rc = lib.oracle_conv_transpose1d(_d(x), Cin, T, _d(w), None if bb is None else _d(bb), Cout, K,
                                     stride, pad_left, T_out, _d(y))
    assert rc == 0
    return y


def round_half(x: np.ndarray) -> np.ndarray:
    """Round to single, then to IEEE half precision (both to nearest, ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().oracle_round_half(_d(x), x.size, _d(y))
    return y


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to single, then to bfloat16 (both to nearest, ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().oracle_round_bf16(_d(x), x.size, _d(y))
    return y


def fold_params(params: Sequence, f16_weights: bool = False, bf16_weights: bool = False) -> list:
    """Raw canonical parameters (RawConv / alpha arrays) -> list of double arrays
    (folded weight, bias, alpha, ...) in the canonical order.  f16_weights / bf16_weights:
    every convolution weight rounded to half precision / bfloat16 (the F16- and BF16-weight
    precision variants); biases and Snake parameters are kept."""
    assert not (f16_weights and bf16_weights)
    out = []
    wf = round_half if f16_weights else round_bf16 if bf16_weights else (lambda w: w)
    for p in params:
        if hasattr(p, "g"):
            out.append(wf(fold_weight_norm(p.g, p.v)))
            out.append(None if p.b is None else np.ascontiguousarray(p.b, dtype=np.float64))
        elif hasattr(p, "w"):  # a convolution stored without weight norm
            out.append(wf(np.ascontiguousarray(p.w, dtype=np.float64)))
            out.append(None if p.b is None else np.ascontiguousarray(p.b, dtype=np.float64))
        else:
            out.append(np.ascontiguousarray(p, dtype=np.float64))
    return out


def decode(arch, params: Sequence, latent: np.ndarray, flags: int = 0, folded: Optional[list] = None,
           return_pre_tanh: bool = False):
    """Full decode of latent [B, C_lat, T] -> audio [B, T*hop] (double)."""
    lib = _load()
    if folded is None:
        folded = fold_params(params)
    latent = np.ascontiguousarray(latent, dtype=np.float32)
    B, Cl, T = latent.shape
    assert Cl == arch.latent_channels
    strides = (ctypes.c_int * len(arch.strides))(*arch.strides)
    widths = (ctypes.c_int * len(arch.widths))(*arch.widths)
    dils = (ctypes.c_int * len(arch.dilations))(*arch.dilations)
    a = _ArchC(arch.latent_channels, arch.channels0, arch.in_kernel, len(arch.strides), strides,
               widths, len(arch.dilations), dils, arch.res_kernel, arch.out_kernel, arch.padding,
               flags, getattr(arch, "in_proj_channels", 0), int(getattr(arch, "snake_beta", False)))
    n = lib.oracle_param_count(ctypes.byref(a))
    assert n == len(folded), (n, len(folded))
    ptrs = (ctypes.POINTER(ctypes.c_double) * n)()
    for i, t in enumerate(folded):
        ptrs[i] = ctypes.cast(None, ctypes.POINTER(ctypes.c_double)) if t is None else _d(t)
    hop = int(np.prod(arch.strides))
    audio = np.empty((B, T * hop), dtype=np.float64)
    pre = np.empty((B, T * hop), dtype=np.float64) if return_pre_tanh else None
    rc = lib.oracle_decode(ctypes.byref(a), ptrs, _f(latent), B, T, _d(audio),
                           None if pre is None else _d(pre))
    if rc != 0:
        raise RuntimeError(f"oracle_decode failed ({rc})")
    return (audio, pre) if return_pre_tanh else audio


def conv1d_strided(x: np.ndarray, w: np.ndarray, b: Optional[np.ndarray], stride: int,
                   pad_left: int, T_out: int) -> np.ndarray:
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    Cin, T = x.shape
    Cout, Cin2, K = w.shape
    assert Cin2 == Cin
    y = np.empty((Cout, T_out), dtype=np.float64)
    bb = None if b is None else np.ascontiguousarray(b, dtype=np.float64)
    rc = lib.oracle_conv1d_strided(_d(x), Cin, T, _d(w), None if bb is None else _d(bb), Cout, K,
                                   stride, pad_left, T_out, _d(y))
    assert rc == 0
    return y


def encode(arch, params: Sequence, audio: np.ndarray, flags: int = 0,
           folded: Optional[list] = None) -> np.ndarray:
    """Mirror encoder: audio [B, Cin, L] -> latent [B, Cl, L / hop] (double)."""
    lib = _load()
    if folded is None:
        folded = fold_params(params)
    audio = np.ascontiguousarray(audio, dtype=np.float32)
    B, Ci, L = audio.shape
    assert Ci == arch.in_channels
    strides = (ctypes.c_int * len(arch.strides))(*arch.strides)
    widths = (ctypes.c_int * len(arch.widths))(*arch.widths)
    dils = (ctypes.c_int * len(arch.dilations))(*arch.dilations)
    a = _EncArchC(arch.in_channels, arch.channels0, arch.in_kernel, len(arch.strides), strides,
                  widths, len(arch.dilations), dils, arch.res_kernel, arch.out_kernel,
                  arch.latent_channels, flags, int(arch.snake_beta))
    n = lib.oracle_enc_param_count(ctypes.byref(a))
    assert n == len(folded), (n, len(folded))
    ptrs = (ctypes.POINTER(ctypes.c_double) * n)()
    for i, t in enumerate(folded):
        ptrs[i] = ctypes.cast(None, ctypes.POINTER(ctypes.c_double)) if t is None else _d(t)
    hop = int(np.prod(arch.strides))
    out = np.empty((B, arch.latent_channels, L // hop), dtype=np.float64)
    rc = lib.oracle_encode(ctypes.byref(a), ptrs, _f(audio), B, L, _d(out))
    if rc != 0:
        raise RuntimeError(f"oracle_encode failed ({rc})")
    return out


def stitched_length(n_win, win_frames, crop_left, crop_right, hop) -> int:
    return int(_load().oracle_stitched_length(n_win, win_frames, crop_left, crop_right, hop))


def stitch(decoded: np.ndarray, n_win: int, n_sides: int, win_frames: int, crop_left: int,
           crop_right: int, hop: int) -> np.ndarray:
    lib = _load()
    decoded = np.ascontiguousarray(decoded, dtype=np.float64)
    n = stitched_length(n_win, win_frames, crop_left, crop_right, hop)
    if n < 0:
        raise ValueError("bad stitch geometry")
    out = np.empty((n_sides, n), dtype=np.float64)
    rc = lib.oracle_stitch(_d(decoded), n_win, n_sides, win_frames, crop_left, crop_right, hop,
                           _d(out))
    assert rc == 0
    return out


def abs_percentile(x: np.ndarray, peak_clip: int) -> float:
    """Nearest-rank 1 - peak_clip/1e6 percentile of |x| (output stage normalisation level)."""
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    return float(_load().oracle_abs_percentile(_f(x), x.size, peak_clip))


def encode_wav(planar: np.ndarray, sample_rate: int, bits: int, peak_clip: int = 0) -> bytes:
    """Planar [n_ch, len] float -> WAV file bytes (16/24-bit normalised PCM, or 32-bit float)."""
    planar = np.ascontiguousarray(planar, dtype=np.float32)
    if planar.ndim == 1:
        planar = planar[None]
    n_ch, n = planar.shape
    lib = _load()
    size = lib.oracle_wav_bytes(n_ch, n, bits)
    if size < 0:
        raise ValueError("bad WAV geometry")
    out = (ctypes.c_ubyte * size)()
    rc = lib.oracle_encode_wav(_f(planar), n_ch, n, sample_rate, bits, peak_clip, out)
    if rc != 0:
        raise ValueError("oracle_encode_wav failed")
    return bytes(out)
