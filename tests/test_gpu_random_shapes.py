"""GPU parity on seeded random problems: whatever kernel AUTO picks, and every
other algorithm that accepts the descriptor, against the fp64 oracle.

Two generators, each with fixed seeds:
- 3 x 48 problems: conv2d or conv3d, f32 / f16 / bf16 storage, NCHW or
  channels-last activations, 1-3 images, 1-80 input and 1-150 output
  channels, 1-40 pixels per side, k 1/3/5, pad 0..k/2+1, stride 1-3, causal
  or symmetric frames, bias or none, ReLU or none (at most 2e8 products);
- 64 wider problems: 1-4 images, 1-300 input and output channels, 1-96
  pixels per side, up to 6 frames, k 1/3/5/7 (at most 1e9 products).
Problems whose output would be empty, or that exceed the oracle's product
budget, are redrawn. Each one runs through AUTO and through
each algorithm forced (DIRECT, IGEMM_FFMA, IGEMM_TC, DIRECT_TC) that the
library accepts for it, so the kernel families meet shapes no hand-written
case chose; the tolerances are the dtype's (gpu_helpers), with fp32 forced
onto the three TF32 products held to that path's reduction-length bound,
and AUTO never giving an fp32 reduction of more than 1,000 products to it.
"""
import numpy as np
import pytest
import torch

import synthetic
import implicit_gemm_convolution_conv_gb300 as gb
from gpu_helpers import assert_close, reference, run
from test_gpu_channels_last import run_cl

pytestmark = pytest.mark.gpu

ALGOS = [gb.ALGO_AUTO, gb.ALGO_DIRECT, gb.ALGO_IGEMM_FFMA, gb.ALGO_IGEMM_TC, gb.ALGO_DIRECT_TC]


def _draw(count=48, seed=2026):
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    while len(out) < count:
        ndim = int(rng.choice([2, 2, 3]))
        k = int(rng.choice([1, 3, 3, 5]))
        pad = int(rng.integers(0, k // 2 + 2))
        stride = int(rng.integers(1, 4))
        dtype = str(rng.choice(["f32", "f16", "bf16"]))
        C = int(rng.choice([int(rng.integers(1, 9)), int(rng.integers(8, 81))]))
        L = synthetic.Layer(
            f"random{len(out)}", N=int(rng.integers(1, 4)), C=C,
            D=int(rng.integers(1, 5)) if ndim == 3 else 1,
            H=int(rng.integers(1, 41)), W=int(rng.integers(1, 41)),
            OC=int(rng.integers(1, 151)), k=k, pad=pad, stride=stride, dtype=dtype,
            relu=bool(rng.integers(0, 2)), ndim=ndim, x_dist="n01", w_dist="he",
            b_dist=str(rng.choice(["u005", "none"])), seed=int(rng.integers(0, 1 << 30)),
            tpad=int(rng.choice([0, 1])) if ndim == 3 else 0, cl=bool(rng.integers(0, 2)))
        # a non-empty output, and few enough products for the oracle
        if min(L.out_dims()) >= 1 and L.flops() <= 4e8:
            out.append(L)
    return out


def _draw_wide(count=64, seed=101):
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    while len(out) < count:
        ndim = int(rng.choice([2, 2, 3]))
        k = int(rng.choice([1, 3, 3, 5, 7]))
        pad = int(rng.integers(0, k // 2 + 2))
        stride = int(rng.integers(1, 4))
        dtype = str(rng.choice(["f32", "f16", "bf16"]))
        C = int(rng.choice([int(rng.integers(1, 9)), int(rng.integers(8, 97)), int(rng.integers(96, 301))]))
        OC = int(rng.choice([int(rng.integers(1, 65)), int(rng.integers(64, 301))]))
        L = synthetic.Layer(
            f"wide{len(out)}", N=int(rng.integers(1, 5)), C=C,
            D=int(rng.integers(1, 7)) if ndim == 3 else 1,
            H=int(rng.integers(1, 97)), W=int(rng.integers(1, 97)),
            OC=OC, k=k, pad=pad, stride=stride, dtype=dtype,
            relu=bool(rng.integers(0, 2)), ndim=ndim, x_dist="n01", w_dist="he",
            b_dist=str(rng.choice(["u005", "none"])), seed=int(rng.integers(0, 1 << 30)),
            tpad=int(rng.choice([0, 1])) if ndim == 3 else 0, cl=bool(rng.integers(0, 2)))
        if min(L.out_dims()) >= 1 and L.flops() <= 1e9:
            out.append(L)
    return out


PROBLEMS = _draw() + _draw(48, 7) + _draw(48, 11) + _draw_wide()


def _accepts(L, algo):
    d = gb.make_desc(L.N, L.C, L.H, L.W, L.OC, L.k, L.pad, L.stride, D=L.D, dtype=L.dtype,
                     algo=algo, tpad=L.tpad, channels_last=L.cl)
    return gb.select_algo(d, L.ndim)[0] == gb.OK


@pytest.mark.parametrize("L", PROBLEMS, ids=[
    f"{i}-{L.ndim}d-{L.dtype}-{'cl' if L.cl else 'nchw'}-N{L.N}C{L.C}D{L.D}H{L.H}W{L.W}OC{L.OC}"
    f"k{L.k}p{L.pad}s{L.stride}t{L.tpad}" for i, L in enumerate(PROBLEMS)])
def test_random_problem(L):
    inp = synthetic.make_inputs(L)
    ref = reference(inp)
    ran = 0
    for algo in ALGOS:
        if not _accepts(L, algo):
            continue
        y, conv = run_cl(inp, algo=algo) if L.cl else run(inp, algo=algo)
        assert y.shape == ref.shape
        if algo == gb.ALGO_AUTO and L.dtype == "f32" and conv.algo == gb.ALGO_IGEMM_TC:
            assert L.C * L.k ** L.ndim <= 1000, "AUTO keeps long fp32 reductions off the TF32 products"
        tf32x3 = L.C * L.k ** L.ndim if (L.dtype == "f32" and conv.algo == gb.ALGO_IGEMM_TC) else 0
        assert_close(L.dtype, y, ref, f"{L} algo {gb.algo_name(conv.algo)}", tf32x3_k=tf32x3)
        ran += 1
    assert ran >= 2          # AUTO and at least the algorithm it resolves to
    torch.cuda.synchronize()
