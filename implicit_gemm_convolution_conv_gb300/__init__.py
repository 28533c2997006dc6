"""Python binding of libgbconv (include/gbconv.h): argument marshalling only.

Every function here has the name of the C entry point without the `gbconv_`
prefix and passes its arguments straight through ctypes. Tensors are passed
by `data_ptr()`; streams default to torch's current CUDA stream. PyTorch is
used for device memory and streams only: all arithmetic runs in the CUDA
kernels of libgbconv.so. There is no CPU fallback; if the library is missing
the import fails.
"""
import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgbconv.so")

# enums (mirror include/gbconv.h)
OK = 0
ERR_NULL, ERR_SHAPE, ERR_DTYPE, ERR_ACT, ERR_ALIGN, ERR_WORKSPACE = 1, 2, 3, 4, 5, 6
ERR_UNSUPPORTED_DEVICE, ERR_LAUNCH, ERR_TIMEOUT, ERR_ALGO = 7, 8, 9, 10
ERR_LAYOUT, ERR_OVERLAP, ERR_CUDA, ERR_RESERVED = 11, 12, 13, 14
TPAD_SYMMETRIC, TPAD_CAUSAL, TPAD_NONE = 0, 1, 2
FLAG_MAXPOOL2 = 4
FLAG_CHANNELS_LAST = 8
ERR_TOO_LARGE = 15
NOALLOC_SCRATCH_BYTES = 8 << 20
F32, F16, BF16 = 0, 1, 2
ACT_NONE, ACT_RELU = 0, 1
W_OIHW, W_PACKED = 0, 1
ALGO_AUTO, ALGO_DIRECT, ALGO_IGEMM_FFMA, ALGO_IGEMM_TC, ALGO_DIRECT_TC = 0, 1, 2, 3, 4
DTYPES = {"f32": F32, "f16": F16, "bf16": BF16}
SYMBOLS = ["gbconv_conv2d_fwd", "gbconv_conv3d_fwd", "gbconv_output_shape",
           "gbconv_workspace_size", "gbconv_weight_packed_size",
           "gbconv_weight_pack", "gbconv_select_algo",
           "gbconv_device_supported", "gbconv_status_string",
           "gbconv_algo_name", "gbconv_check_device_error",
           "gbconv_set_wait_limit_ns", "gbconv_conv_fwd_noalloc",
           "gbconv_fold_batchnorm"]


class Desc(ctypes.Structure):
    """struct gbconv_desc."""
    _fields_ = [("N", ctypes.c_int), ("C", ctypes.c_int), ("D", ctypes.c_int),
                ("H", ctypes.c_int), ("W", ctypes.c_int), ("OC", ctypes.c_int),
                ("k", ctypes.c_int), ("pad", ctypes.c_int),
                ("stride", ctypes.c_int), ("dtype", ctypes.c_int),
                ("act", ctypes.c_int), ("w_layout", ctypes.c_int),
                ("algo", ctypes.c_int), ("flags", ctypes.c_int),
                ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t)]


class GbconvError(RuntimeError):
    def __init__(self, status):
        self.status = status
        super().__init__(f"gbconv status {status}: {status_string(status)}")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -c 'import "
            f"__graft_entry__ as g; g.build()'` (there is no fallback path)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    DP = ctypes.POINTER(Desc)
    sig = {
        "gbconv_conv2d_fwd": ([DP, P, P, P, P, P], I),
        "gbconv_conv3d_fwd": ([DP, P, P, P, P, P], I),
        "gbconv_output_shape": ([DP, I, ctypes.POINTER(I), ctypes.POINTER(I),
                                 ctypes.POINTER(I)], I),
        "gbconv_workspace_size": ([DP, I, ctypes.POINTER(Z)], I),
        "gbconv_weight_packed_size": ([DP, I, ctypes.POINTER(Z)], I),
        "gbconv_weight_pack": ([DP, I, P, P, P], I),
        "gbconv_select_algo": ([DP, I, ctypes.POINTER(I)], I),
        "gbconv_device_supported": ([I], I),
        "gbconv_status_string": ([I], ctypes.c_char_p),
        "gbconv_algo_name": ([I], ctypes.c_char_p),
        "gbconv_check_device_error": ([P], I),
        "gbconv_set_wait_limit_ns": ([ctypes.c_uint64], I),
        "gbconv_conv_fwd_noalloc": ([DP, I, P, P, P, P, P], I),
        "gbconv_fold_batchnorm": ([DP, I, P, P, P, P, P, P, ctypes.c_float, P, P, P], I),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes, f.restype = args, res
    return lib


LIB = _load()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def make_desc(N, C, H, W, OC, k, pad=0, stride=1, D=1, dtype=F32,
              act=ACT_NONE, w_layout=W_OIHW, algo=ALGO_AUTO, workspace=None,
              workspace_bytes=0, flags=0, tpad=0, pool=False,
              channels_last=False):
    if isinstance(dtype, str):
        dtype = DTYPES[dtype]
    ints = dict(N=N, C=C, H=H, W=W, OC=OC, k=k, pad=pad, stride=stride, D=D, dtype=dtype, act=act,
                w_layout=w_layout, algo=algo, flags=flags, tpad=tpad)
    for name, v in ints.items():
        # the fields are C ints: a wider value would wrap silently in ctypes
        if not isinstance(v, (int, np.integer)) or not -2**31 <= int(v) < 2**31:
            raise ValueError(f"{name}={v!r} is not a 32-bit integer")
    d = Desc()
    d.N, d.C, d.D, d.H, d.W = N, C, D, H, W
    d.OC, d.k, d.pad, d.stride = OC, k, pad, stride
    d.dtype, d.act, d.w_layout, d.algo = dtype, act, w_layout, algo
    d.flags = (flags | tpad | (FLAG_MAXPOOL2 if pool else 0) |
               (FLAG_CHANNELS_LAST if channels_last else 0))
    d.workspace = _ptr(workspace)
    d.workspace_bytes = workspace_bytes
    return d


def conv2d_fwd(desc, x, w, b, y, stream=None):
    """gbconv_conv2d_fwd; returns the status code."""
    return LIB.gbconv_conv2d_fwd(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(b),
                                 _ptr(y), _stream(stream))


def conv3d_fwd(desc, x, w, b, y, stream=None):
    """gbconv_conv3d_fwd; returns the status code."""
    return LIB.gbconv_conv3d_fwd(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(b),
                                 _ptr(y), _stream(stream))


def output_shape(desc, ndim):
    od, oh, ow = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    st = LIB.gbconv_output_shape(ctypes.byref(desc), ndim, ctypes.byref(od),
                                 ctypes.byref(oh), ctypes.byref(ow))
    return st, (od.value, oh.value, ow.value)


def workspace_size(desc, ndim):
    n = ctypes.c_size_t()
    st = LIB.gbconv_workspace_size(ctypes.byref(desc), ndim, ctypes.byref(n))
    return st, n.value


def weight_packed_size(desc, ndim):
    n = ctypes.c_size_t()
    st = LIB.gbconv_weight_packed_size(ctypes.byref(desc), ndim,
                                       ctypes.byref(n))
    return st, n.value


def weight_pack(desc, ndim, w_oihw, w_packed, stream=None):
    return LIB.gbconv_weight_pack(ctypes.byref(desc), ndim, _ptr(w_oihw),
                                  _ptr(w_packed), _stream(stream))


def select_algo(desc, ndim):
    a = ctypes.c_int()
    st = LIB.gbconv_select_algo(ctypes.byref(desc), ndim, ctypes.byref(a))
    return st, a.value


def device_supported(device=0):
    return LIB.gbconv_device_supported(device)


def status_string(status):
    return LIB.gbconv_status_string(status).decode()


def algo_name(algo):
    return LIB.gbconv_algo_name(algo).decode()


def check_device_error(stream=None):
    return LIB.gbconv_check_device_error(_stream(stream))


def set_wait_limit_ns(ns):
    return LIB.gbconv_set_wait_limit_ns(ns)


def conv_fwd_noalloc(desc, ndim, x, w, b, y, stream=None):
    """gbconv_conv_fwd_noalloc: no workspace, no allocation (scratch is a
    fixed array inside the library); returns the status code."""
    return LIB.gbconv_conv_fwd_noalloc(ctypes.byref(desc), ndim, _ptr(x),
                                       _ptr(w), _ptr(b), _ptr(y),
                                       _stream(stream))


def fold_batchnorm(desc, ndim, w, b, gamma, beta, mean, var, eps, w_out, b_out,
                   stream=None):
    """gbconv_fold_batchnorm: BatchNorm folded into the conv's weights and
    bias (w_out, b_out may be w, b); returns the status code."""
    return LIB.gbconv_fold_batchnorm(ctypes.byref(desc), ndim, _ptr(w), _ptr(b),
                                     _ptr(gamma), _ptr(beta), _ptr(mean),
                                     _ptr(var), float(eps), _ptr(w_out),
                                     _ptr(b_out), _stream(stream))


def check(status):
    if status != OK:
        raise GbconvError(status)
