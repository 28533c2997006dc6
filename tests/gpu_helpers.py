"""Shared helpers of the GPU tests: run a layer through the C ABI and compare
with the fp64 oracle at the tolerances the method's arithmetic allows.

Tolerances (stated per storage dtype):
  f32  : relative L2 error <= 1e-5 and max abs error <= 1e-4.
  f16  : NRMSE = ||y - ref||_2 / ||ref||_2 <= 1e-3, and every element within
         2^-10 |ref| + 3e-4 (one f16 ulp of the result plus fp32 accumulation).
  bf16 : NRMSE <= 1e-3 against the exact result rounded to bf16 (bf16
         rounding alone gives NRMSE ~1.5e-3 against the unrounded result),
         NRMSE <= 2.5e-3 against the unrounded result, and every element
         within 2^-7 |ref| + 3e-4.
"""
import numpy as np
import torch

import oracle
import synthetic
from implicit_gemm_convolution_conv_gb300 import ALGO_AUTO
from implicit_gemm_convolution_conv_gb300.torch_ops import (Conv, to_device,
                                                            to_numpy)


def device_inputs(inp: synthetic.Inputs):
    L = inp.layer
    x = to_device(inp.x, L.dtype)
    w = to_device(inp.w, L.dtype)
    b = None if inp.b is None else torch.from_numpy(inp.b).cuda()
    return x, w, b


def run(inp: synthetic.Inputs, algo=ALGO_AUTO, prepack=False):
    """Run the layer on the GPU; returns (y as float64 numpy, Conv)."""
    L = inp.layer
    x, w, b = device_inputs(inp)
    conv = Conv(x, w, b, stride=L.stride, pad=L.pad, relu=L.relu, algo=algo,
                prepack=prepack, tpad=L.tpad, pool=L.pool)
    y = conv()
    torch.cuda.synchronize()
    return oracle.widen(to_numpy(y), L.dtype), conv


# Whole-layer oracle results of the large layers, kept for the session: the
# NCHW and channels-last runs of one layer read the same seeded inputs.
_REF_CACHE = {}
_REF_CACHE_MIN = 1 << 22        # outputs: cache only layers at least this large
_REF_CACHE_MAX = 4              # entries


def _ref_key(inp):
    L = inp.layer
    return (L.N, L.C, L.D, L.H, L.W, L.OC, L.k, L.pad, L.stride, L.dtype, L.relu, L.ndim,
            L.tpad, L.pool, L.seed, L.x_dist, L.w_dist, L.b_dist,
            inp.x.tobytes()[:4096], inp.w.tobytes()[:4096])


def reference(inp: synthetic.Inputs, idx=None):
    L = inp.layer
    if idx is None:
        key = _ref_key(inp)
        if key in _REF_CACHE:
            return _REF_CACHE[key]
        ref = _reference(inp)
        if ref.size >= _REF_CACHE_MIN:
            while len(_REF_CACHE) >= _REF_CACHE_MAX:
                _REF_CACHE.pop(next(iter(_REF_CACHE)))
            _REF_CACHE[key] = ref
        return ref
    return _reference(inp, idx)


def _reference(inp: synthetic.Inputs, idx=None):
    L = inp.layer
    if L.pool:
        full = oracle.maxpool2(oracle.conv(inp.x, inp.w, inp.b, L.stride, L.pad,
                                           L.relu, L.dtype))
        return full if idx is None else full.ravel()[idx]
    if idx is None:
        return oracle.conv(inp.x, inp.w, inp.b, L.stride, L.pad, L.relu,
                           L.dtype, tpad=L.tpad)
    return oracle.conv_at(inp.x, inp.w, inp.b, idx, L.stride, L.pad, L.relu,
                          L.dtype, tpad=L.tpad)


def errors(y, ref):
    err = y - ref
    nref = np.linalg.norm(ref)
    return {"rel_l2": float(np.linalg.norm(err) / max(nref, 1e-300)),
            "max_abs": float(np.max(np.abs(err))) if err.size else 0.0}


def assert_close(dtype, y, ref, what="", tf32x3_k=0):
    """tf32x3_k: for an fp32 call forced onto the tensor cores' three TF32
    products, its reduction length C * k^d. Beyond 1,000 products (where
    AUTO takes the exact CUDA-core GEMM instead) that path's error grows
    with the reduction, and it is held to the fp32 bars scaled by K / 1000,
    its documented bound (include/gbconv.h)."""
    y = np.asarray(y, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    assert y.shape == ref.shape
    assert np.isfinite(y).all(), f"{what}: non-finite output"
    e = errors(y, ref)
    if dtype == "f32":
        scale = max(1.0, tf32x3_k / 1000.0)
        assert e["rel_l2"] <= 1e-5 * scale, (what, e)
        assert e["max_abs"] <= 1e-4 * scale, (what, e)
    elif dtype == "f16":
        assert e["rel_l2"] <= 1e-3, (what, e)
        bad = np.abs(y - ref) > 2.0 ** -10 * np.abs(ref) + 3e-4
        assert not bad.any(), (what, e, int(bad.sum()), np.flatnonzero(bad)[:8])
    elif dtype == "bf16":
        ref_q = oracle.widen(synthetic.to_bf16_bits(ref), "bf16")
        eq = errors(y, ref_q)
        assert eq["rel_l2"] <= 1e-3, (what, eq)
        assert e["rel_l2"] <= 2.5e-3, (what, e)
        bad = np.abs(y - ref) > 2.0 ** -7 * np.abs(ref) + 3e-4
        assert not bad.any(), (what, e, int(bad.sum()), np.flatnonzero(bad)[:8])
    else:
        raise ValueError(dtype)
    return e
