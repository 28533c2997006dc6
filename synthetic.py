"""Seeded synthetic inputs for the convolution layers, shared by tests and bench.

This module draws random tensors and rounds them to their storage dtype. It
holds none of the convolution's arithmetic: it imports neither the oracle nor
the CUDA library, and both sides receive the same arrays from here.

Layer shapes are the five synthetic stand-ins for the conv layers of the
workloads the pages time (a PP-OCR detection stem and text-line batch,
lpnh.cn/news/2745477 section 3; a wide dense 3x3 layer; and a SeedVR2
video-VAE Convolution3D, git.erdda.com/Tencent/ncnn/discussions/7001 sections
3.2-3.3: batch 1, spatial sizes multiples of 16, 4n+1 frames). No dataset or
trained weight is involved.

Recipe: numpy Generator(PCG64(seed)), draws in the order x, w, b, each drawn
in float64 and then rounded to the storage dtype (float32 / float16 by numpy's
round-to-nearest-even; bfloat16 through float32, then round-to-nearest-even on
the top 16 bits). Bias is always float32.
"""
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np


@dataclass(frozen=True)
class Layer:
    """One convolution layer: shapes, storage dtype and input distributions."""
    name: str
    N: int
    C: int
    H: int
    W: int
    OC: int
    k: int
    pad: int
    stride: int
    dtype: str = "f32"          # storage dtype of x, w, y: f32 | f16 | bf16
    relu: bool = False
    D: int = 1                  # frames / depth; used when ndim == 3
    ndim: int = 2               # spatial dims: 2 (conv2d) or 3 (conv3d)
    x_dist: str = "u11"         # u11: U[-1,1]; u01: U[0,1]; relun: ReLU(N(0,1)); n01: N(0,1)
    w_dist: str = "u11"         # u11 or he: N(0, 2/fan_in)
    b_dist: str = "u11"         # u11, u01_1: U[-0.1,0.1], u005: U[-0.05,0.05], none
    seed: int = 20260
    tpad: int = 0               # conv3d frame padding: 0 symmetric, 1 causal (k-1 front), 2 none
    pool: bool = False          # 2x2 stride-2 max pool fused after the activation (2D)
    cl: bool = False            # channels-last x and y on the device (layout only; the
                                # arrays drawn here stay NC(D)HW)

    @property
    def kvol(self) -> int:
        return self.k ** self.ndim

    @property
    def fan_in(self) -> int:
        return self.C * self.kvol

    def out_dims(self):
        def ext(n, p0, p1):
            return (n + p0 + p1 - self.k) // self.stride + 1
        p = self.pad
        if self.ndim == 3:
            f0, f1 = {0: (p, p), 1: (self.k - 1, 0), 2: (0, 0)}[self.tpad]
            return (ext(self.D, f0, f1), ext(self.H, p, p), ext(self.W, p, p))
        return (1, ext(self.H, p, p), ext(self.W, p, p))

    def x_shape(self):
        if self.ndim == 3:
            return (self.N, self.C, self.D, self.H, self.W)
        return (self.N, self.C, self.H, self.W)

    def w_shape(self):
        return (self.OC, self.C) + (self.k,) * self.ndim

    def y_shape(self):
        od, oh, ow = self.out_dims()
        if self.pool:
            oh, ow = oh // 2, ow // 2
        if self.ndim == 3:
            return (self.N, self.OC, od, oh, ow)
        return (self.N, self.OC, oh, ow)

    def flops(self) -> int:
        """2 * N * OC * outVol * IC * kVol (padded taps counted)."""
        od, oh, ow = self.out_dims()
        return 2 * self.N * self.OC * od * oh * ow * self.C * self.kvol

    def elt_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def compulsory_bytes(self) -> int:
        """x read once, w once, b once (fp32), y written once."""
        e = self.elt_bytes()
        nx = int(np.prod(self.x_shape()))
        nw = int(np.prod(self.w_shape()))
        ny = int(np.prod(self.y_shape()))
        nb = self.OC * 4 if self.b_dist != "none" else 0
        return e * (nx + nw + ny) + nb


# The five layer shapes (seed = 20260 + index).
LAYERS = {
    1: Layer("conv2d_f32_1x3x32x32_oc8_k3p1s1", N=1, C=3, H=32, W=32, OC=8,
             k=3, pad=1, stride=1, x_dist="u11", w_dist="u11", b_dist="u11",
             seed=20261),
    2: Layer("conv2d_f32_1x3x640x640_oc32_k3p1s2_relu", N=1, C=3, H=640,
             W=640, OC=32, k=3, pad=1, stride=2, relu=True, x_dist="u01",
             w_dist="he", b_dist="u01_1", seed=20262),
    3: Layer("conv2d_f32_16x64x12x80_oc128_k3p1s1_relu", N=16, C=64, H=12,
             W=80, OC=128, k=3, pad=1, stride=1, relu=True, x_dist="relun",
             w_dist="he", b_dist="u01_1", seed=20263),
    4: Layer("conv2d_f16_1x256x128x128_oc256_k3p1s1", N=1, C=256, H=128,
             W=128, OC=256, k=3, pad=1, stride=1, dtype="f16", x_dist="n01",
             w_dist="he", b_dist="u005", seed=20264),
    5: Layer("conv3d_f16_1x128x5x128x240_oc128_k3p1s1", N=1, C=128, D=5,
             H=128, W=240, OC=128, k=3, pad=1, stride=1, dtype="f16",
             ndim=3, x_dist="n01", w_dist="he", b_dist="u005", seed=20265),
}


def layer(idx: int, **overrides) -> Layer:
    return replace(LAYERS[idx], **overrides)


def _draw(rng, dist, shape, fan_in):
    if dist == "u11":
        return rng.uniform(-1.0, 1.0, shape)
    if dist == "u01":
        return rng.uniform(0.0, 1.0, shape)
    if dist == "u01_1":
        return rng.uniform(-0.1, 0.1, shape)
    if dist == "u005":
        return rng.uniform(-0.05, 0.05, shape)
    if dist == "n01":
        return rng.standard_normal(shape)
    if dist == "relun":
        return np.maximum(rng.standard_normal(shape), 0.0)
    if dist == "he":
        return rng.standard_normal(shape) * np.sqrt(2.0 / fan_in)
    if dist == "ones":
        return np.ones(shape)
    raise ValueError(f"unknown distribution {dist}")


def to_bf16_bits(a64: np.ndarray) -> np.ndarray:
    """float64 -> float32 (RNE) -> bfloat16 bit patterns (RNE on 16 bits)."""
    f = np.ascontiguousarray(a64, np.float32).view(np.uint32).astype(np.uint64)
    rounded = (f + 0x7FFF + ((f >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def to_storage(a64: np.ndarray, dtype: str) -> np.ndarray:
    """Round a float64 array to the storage dtype (bf16 as uint16 bits)."""
    if dtype == "f32":
        return np.ascontiguousarray(a64, np.float32)
    if dtype == "f16":
        return np.ascontiguousarray(a64, np.float16)
    if dtype == "bf16":
        return to_bf16_bits(a64)
    raise ValueError(dtype)


@dataclass
class Inputs:
    layer: Layer
    x: np.ndarray           # storage dtype (bf16: uint16 bits)
    w: np.ndarray           # storage dtype, OIHW / OIDHW
    b: Optional[np.ndarray]  # float32 or None


def make_inputs(L: Layer, seed: Optional[int] = None) -> Inputs:
    rng = np.random.Generator(np.random.PCG64(L.seed if seed is None else seed))
    x = _draw(rng, L.x_dist, L.x_shape(), L.fan_in)
    w = _draw(rng, L.w_dist, L.w_shape(), L.fan_in)
    b = None if L.b_dist == "none" else _draw(rng, L.b_dist, (L.OC,), L.fan_in)
    return Inputs(L, to_storage(x, L.dtype), to_storage(w, L.dtype),
                  None if b is None else np.ascontiguousarray(b, np.float32))


def sample_indices(L: Layer, count: int, seed: int = 7) -> np.ndarray:
    """Flat output indices to check at full size: every corner/edge class plus
    a uniform random sample, sorted and unique."""
    shape = L.y_shape()
    total = int(np.prod(shape))
    rng = np.random.Generator(np.random.PCG64(seed))
    rand = rng.integers(0, total, size=max(0, count))
    # borders: first/last row and column of every (n, oc[, od]) plane sampled
    picks = []
    OW, OH = shape[-1], shape[-2]
    planes = total // (OW * OH)
    for p in rng.integers(0, planes, size=min(planes, 64)):
        base = int(p) * OW * OH
        for oy in (0, OH - 1):
            for ox in (0, 1, OW // 2, OW - 2, OW - 1):
                if 0 <= ox < OW:
                    picks.append(base + oy * OW + ox)
    idx = np.unique(np.concatenate([rand, np.asarray(picks, np.int64)]))
    return idx.astype(np.int64)
