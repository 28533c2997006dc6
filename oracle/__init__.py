"""fp64 CPU oracle for the forward convolution (conv2d / conv3d + bias + ReLU).

TEST INFRASTRUCTURE ONLY. Only `tests/`, `__graft_entry__.smoke()` and
`bench.py`'s CPU-baseline leg may import this package. It shares no code with
the CUDA library and never imports it.

The arithmetic lives in `conv_ref.c` (the plain loop-nest definition from
lpnh.cn/news/2745477, section 2.2, extended to 3D as in
git.erdda.com/Tencent/ncnn/discussions/7001, section 3.2). This module only
widens the stored inputs to float64 exactly and marshals arrays into the C
entry points.

Storage dtypes accepted: numpy float32, float16, float64, and bfloat16 given as
its raw 16-bit patterns in a uint16 array (`widen(..., "bf16")`).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        ci = ctypes.c_int
        lib.oracle_conv2d.argtypes = [ci] * 9 + [dp, dp, dp, dp]
        lib.oracle_conv3d.argtypes = [ci] * 12 + [dp, dp, dp, dp]
        lib.oracle_conv2d_at.argtypes = ([ci] * 9 + [dp, dp, dp, i64p,
                                                     ctypes.c_int64, dp])
        lib.oracle_conv3d_at.argtypes = ([ci] * 12 + [dp, dp, dp, i64p,
                                                      ctypes.c_int64, dp])
        for f in (lib.oracle_conv2d, lib.oracle_conv3d, lib.oracle_conv2d_at,
                  lib.oracle_conv3d_at, lib.oracle_threads):
            f.restype = ci
        _LIB = lib
    return _LIB


def threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_lib().oracle_threads())


def widen(a, dtype: str = None) -> np.ndarray:
    """Exactly widen a stored array to float64.

    dtype "bf16" means `a` holds bfloat16 bit patterns (uint16): the value is
    those 16 bits as the high half of an IEEE float32, which is exact.
    """
    a = np.asarray(a)
    if dtype == "bf16":
        if a.dtype != np.uint16:
            raise TypeError("bf16 data must be passed as uint16 bit patterns")
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if a.dtype not in (np.float16, np.float32, np.float64):
        raise TypeError(f"unsupported storage dtype {a.dtype}")
    return a.astype(np.float64)


def _ptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def out_extent(n: int, k: int, pad: int, stride: int) -> int:
    """floor((n + 2*pad - k) / stride) + 1, the output length of one axis."""
    return (n + 2 * pad - k) // stride + 1


def _prep(x, w, b, dtype, nsp):
    xd = np.ascontiguousarray(widen(x, dtype))
    wd = np.ascontiguousarray(widen(w, dtype))
    bd = None if b is None else np.ascontiguousarray(np.asarray(b, np.float64))
    if xd.ndim != 2 + nsp or wd.ndim != 2 + nsp:
        raise ValueError("x and w must have %d dims" % (2 + nsp))
    k = wd.shape[2]
    if any(s != k for s in wd.shape[2:]):
        raise ValueError("kernel must be cubic/square")
    if wd.shape[1] != xd.shape[1]:
        raise ValueError("w in-channels differ from x channels")
    if bd is not None and bd.shape != (wd.shape[0],):
        raise ValueError("bias must have OC entries")
    return xd, wd, bd, k


def conv2d(x, w, b=None, stride=1, pad=0, relu=False, dtype=None):
    """y[n,oc,oy,ox] in float64 for x [N,C,H,W], w [OC,C,k,k], b [OC]."""
    xd, wd, bd, k = _prep(x, w, b, dtype, 2)
    N, C, H, W = xd.shape
    OC = wd.shape[0]
    OH, OW = out_extent(H, k, pad, stride), out_extent(W, k, pad, stride)
    if OH <= 0 or OW <= 0:
        raise ValueError("empty output")
    y = np.empty((N, OC, OH, OW), np.float64)
    rc = _lib().oracle_conv2d(N, C, H, W, OC, k, pad, stride, int(bool(relu)),
                              _ptr(xd), _ptr(wd),
                              None if bd is None else _ptr(bd), _ptr(y))
    if rc != 0:
        raise ValueError(f"oracle_conv2d rejected the shape ({rc})")
    return y


TPAD_SYMMETRIC, TPAD_CAUSAL, TPAD_NONE = 0, 1, 2


def frame_pads(k: int, pad: int, tpad: int):
    """(zero frames before, after) the input for a frame-padding mode:
    symmetric (pad, pad); causal (k-1, 0), the video VAE's causal
    Convolution3D (git.erdda.com/Tencent/ncnn/discussions/7001, section 3.3);
    none (0, 0) for a chunk that already carries its predecessor's frames."""
    if tpad == TPAD_SYMMETRIC:
        return pad, pad
    if tpad == TPAD_CAUSAL:
        return k - 1, 0
    if tpad == TPAD_NONE:
        return 0, 0
    raise ValueError(f"unknown frame-padding mode {tpad}")


def conv3d(x, w, b=None, stride=1, pad=0, relu=False, dtype=None, tpad=0):
    """y[n,oc,od,oy,ox] in float64 for x [N,C,D,H,W], w [OC,C,k,k,k]."""
    xd, wd, bd, k = _prep(x, w, b, dtype, 3)
    N, C, D, H, W = xd.shape
    OC = wd.shape[0]
    pd0, pd1 = frame_pads(k, pad, tpad)
    OD = (D + pd0 + pd1 - k) // stride + 1
    OH, OW = (out_extent(s, k, pad, stride) for s in (H, W))
    if OD <= 0 or OH <= 0 or OW <= 0:
        raise ValueError("empty output")
    y = np.empty((N, OC, OD, OH, OW), np.float64)
    rc = _lib().oracle_conv3d(N, C, D, H, W, OC, k, pad, pd0, pd1, stride,
                              int(bool(relu)), _ptr(xd), _ptr(wd),
                              None if bd is None else _ptr(bd), _ptr(y))
    if rc != 0:
        raise ValueError(f"oracle_conv3d rejected the shape ({rc})")
    return y


def conv_at(x, w, b, flat_idx, stride=1, pad=0, relu=False, dtype=None, tpad=0):
    """The outputs y.flat[flat_idx] of conv2d (4D x) or conv3d (5D x) only.

    Computes each requested output on its own, so full-size layers can be
    checked on a sample.
    """
    nsp = np.asarray(x).ndim - 2
    xd, wd, bd, k = _prep(x, w, b, dtype, nsp)
    idx = np.ascontiguousarray(np.asarray(flat_idx, np.int64).ravel())
    out = np.empty(idx.shape[0], np.float64)
    bp = None if bd is None else _ptr(bd)
    ip = idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    OC = wd.shape[0]
    if nsp == 2:
        N, C, H, W = xd.shape
        rc = _lib().oracle_conv2d_at(N, C, H, W, OC, k, pad, stride,
                                     int(bool(relu)), _ptr(xd), _ptr(wd), bp,
                                     ip, idx.shape[0], _ptr(out))
    elif nsp == 3:
        N, C, D, H, W = xd.shape
        pd0, pd1 = frame_pads(k, pad, tpad)
        rc = _lib().oracle_conv3d_at(N, C, D, H, W, OC, k, pad, pd0, pd1, stride,
                                     int(bool(relu)), _ptr(xd), _ptr(wd), bp,
                                     ip, idx.shape[0], _ptr(out))
    else:
        raise ValueError("x must be 4D or 5D")
    if rc != 0:
        raise ValueError(f"oracle rejected the request ({rc})")
    return out


def maxpool2(y):
    """2x2, stride-2 max pool over the last two axes, floor mode (a last odd
    row or column is dropped): out[..., i, j] = max of y[..., 2i+a, 2j+b] over
    a, b in {0, 1}. The pooling that lpnh.cn/news/2745477 section 4.4 fuses
    with conv and ReLU into one shader."""
    y = np.asarray(y, np.float64)
    H, W = y.shape[-2] // 2, y.shape[-1] // 2
    out = np.empty(y.shape[:-2] + (H, W), np.float64)
    for i in range(H):
        for j in range(W):
            out[..., i, j] = np.maximum(
                np.maximum(y[..., 2 * i, 2 * j], y[..., 2 * i, 2 * j + 1]),
                np.maximum(y[..., 2 * i + 1, 2 * j], y[..., 2 * i + 1, 2 * j + 1]))
    return out


def batchnorm(y, gamma, beta, mean, var, eps):
    """Inference BatchNorm over the channel axis (axis 1) of y, in float64:
    gamma * (y - mean) / sqrt(var + eps) + beta."""
    sh = (1, -1) + (1,) * (np.asarray(y).ndim - 2)
    g, bt, m, v = (np.asarray(a, np.float64).reshape(sh) for a in (gamma, beta, mean, var))
    return g * (np.asarray(y, np.float64) - m) / np.sqrt(v + float(eps)) + bt


def fold_batchnorm(w, b, gamma, beta, mean, var, eps):
    """The BatchNorm after a conv folded into its weights and bias, in
    float64 (lpnh.cn/news/2745477 section 3.1): s = gamma / sqrt(var + eps),
    w' = w * s per output channel, b' = (b - mean) * s + beta (b = 0 if None)."""
    w = np.asarray(w, np.float64)
    s = np.asarray(gamma, np.float64) / np.sqrt(np.asarray(var, np.float64) + float(eps))
    b0 = np.zeros(w.shape[0]) if b is None else np.asarray(b, np.float64)
    wf = w * s.reshape((-1,) + (1,) * (w.ndim - 1))
    bf = (b0 - np.asarray(mean, np.float64)) * s + np.asarray(beta, np.float64)
    return wf, bf


def conv(x, w, b=None, stride=1, pad=0, relu=False, dtype=None, tpad=0):
    """conv2d for 4D x, conv3d for 5D x (tpad: frame-padding mode)."""
    if np.asarray(x).ndim == 4:
        if tpad != TPAD_SYMMETRIC:
            raise ValueError("conv2d has no frame axis")
        return conv2d(x, w, b, stride, pad, relu, dtype)
    return conv3d(x, w, b, stride, pad, relu, dtype, tpad)
