"""GPU parity of channels-last activations (GBCONV_FLAG_CHANNELS_LAST).

x is [N, (D,) H, W, C] and y is [N, (OD,) OH, OW, OC]. The oracle computes
the plain NCHW definition on the same seeded values; the tests move the
channel axis (pure data movement) on the way in and out. Covered: the
tensor-core GEMM reading x in place (f16/bf16, C a multiple of 8; paired and
odd-OC scalar stores, several output-channel tiles, row and column pixel
tiles, 3D with causal frames) and the CUDA-core GEMM (any dtype and C); the
channels-last result against the NCHW result of the same kernel, bit for
bit; the two tensor-core layer shapes at full size, every output; and
convolutions chained channels-last to channels-last against the oracle
chain, whose intermediate is rounded to the storage dtype as the device
stores it.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import implicit_gemm_convolution_conv_gb300 as gb
from implicit_gemm_convolution_conv_gb300.torch_ops import Conv, to_device, to_numpy
from gpu_helpers import assert_close, reference, run

pytestmark = pytest.mark.gpu

A_FFMA, A_TC = gb.ALGO_IGEMM_FFMA, gb.ALGO_IGEMM_TC


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    assert gb.check_device_error() == gb.OK


def to_cl(a):
    """NC(D)HW numpy array -> N(D)HWC (channel axis last), contiguous."""
    return np.ascontiguousarray(np.moveaxis(a, 1, -1))


def from_cl(a):
    return np.ascontiguousarray(np.moveaxis(a, -1, 1))


def run_cl(inp, algo=gb.ALGO_AUTO, prepack=False, x_dev=None):
    """Run a layer channels-last; returns (y as float64 NC(D)HW, Conv)."""
    L = inp.layer
    x = to_device(to_cl(inp.x), L.dtype) if x_dev is None else x_dev
    w = to_device(inp.w, L.dtype)
    b = None if inp.b is None else torch.from_numpy(inp.b).cuda()
    conv = Conv(x, w, b, stride=L.stride, pad=L.pad, relu=L.relu, algo=algo,
                prepack=prepack, tpad=L.tpad, channels_last=True)
    y = conv()
    torch.cuda.synchronize()
    return from_cl(oracle.widen(to_numpy(y), L.dtype)), conv


def _L(dtype="f16", N=1, C=16, D=1, H=9, W=11, OC=16, k=3, pad=1, stride=1,
       relu=False, bias=True, ndim=2, seed=11, tpad=0):
    return synthetic.Layer("cl_sweep", N=N, C=C, D=D, H=H, W=W, OC=OC, k=k,
                           pad=pad, stride=stride, dtype=dtype, relu=relu,
                           ndim=ndim, x_dist="n01", w_dist="he",
                           b_dist="u005" if bias else "none", seed=seed,
                           tpad=tpad)


SWEEP = [
    # tensor cores, x read in place
    (A_TC, _L(C=64, H=9, W=13, OC=40, relu=True)),
    (A_TC, _L(dtype="bf16", C=16, H=20, W=70, OC=64, stride=2)),
    (A_TC, _L(C=8, H=7, W=12, OC=7, bias=False)),                  # odd OC: scalar stores
    (A_TC, _L(C=32, H=6, W=20, OC=136)),                           # two output-channel tiles
    (A_TC, _L(N=3, C=64, H=30, W=40, OC=320)),                     # three channel tiles, more tiles than SMs
    (A_TC, _L(dtype="bf16", C=24, H=7, W=9, OC=264, relu=True)),   # three channel tiles, an OC tail
    (A_TC, _L(N=2, C=24, H=16, W=10, OC=32, k=1, pad=0)),          # several rows per tile
    (A_TC, _L(C=16, H=3, W=300, OC=16, k=5, pad=2)),               # column tiles
    (A_TC, _L(C=72, H=5, W=9, OC=24, k=3, pad=0, stride=3)),       # ragged channel block
    (A_TC, _L(C=32, D=3, H=8, W=24, OC=32, ndim=3)),
    (A_TC, _L(dtype="bf16", C=24, D=5, H=7, W=9, OC=16, ndim=3,
              tpad=gb.TPAD_CAUSAL, relu=True)),
    (A_TC, _L(N=2, C=16, H=100, W=160, OC=32)),                    # a partial last wave
    # traversal ranges that end below zero (small extents, large padding):
    # the GEMM's L2 prefetch of x must keep to the loads' own coordinates
    (A_TC, _L(N=3, C=8, D=1, H=35, W=25, OC=18, k=5, pad=2, stride=2, ndim=3)),
    (A_TC, _L(dtype="bf16", C=40, D=2, H=16, W=10, OC=149, k=3, pad=2, stride=3, ndim=3,
              tpad=gb.TPAD_CAUSAL)),
    (A_TC, _L(N=2, C=16, H=2, W=1, OC=24, k=5, pad=2)),
    # fp32 on the tensor cores: x split into TF32 halves from channels-last input
    (A_TC, _L(dtype="f32", C=20, H=11, W=13, OC=40, relu=True)),
    (A_TC, _L(dtype="f32", C=64, D=3, H=6, W=20, OC=32, ndim=3)),
    # CUDA-core GEMM: any dtype and channel count
    (A_FFMA, _L(dtype="f32", C=3, H=40, W=42, OC=32, stride=2, relu=True)),
    (A_FFMA, _L(dtype="f32", C=64, H=6, W=20, OC=70)),
    (A_FFMA, _L(dtype="f32", C=5, D=4, H=6, W=7, OC=9, ndim=3)),
    (A_FFMA, _L(C=12, H=11, W=13, OC=20)),
    (A_FFMA, _L(dtype="bf16", C=6, H=13, W=17, OC=10, k=5, pad=2, stride=3)),
]


@pytest.mark.parametrize("algo,L", SWEEP,
                         ids=[f"{gb.algo_name(a)}-{L.dtype}-{L.ndim}d-C{L.C}-OC{L.OC}"
                              f"-{L.H}x{L.W}-k{L.k}s{L.stride}" for a, L in SWEEP])
def test_channels_last_sweep(algo, L):
    inp = synthetic.make_inputs(L)
    y, conv = run_cl(inp, algo=algo)
    assert conv.algo == algo
    tf32x3 = L.C * L.k ** L.ndim if (L.dtype == "f32" and algo == A_TC) else 0
    assert_close(L.dtype, y, reference(inp), f"channels-last {gb.algo_name(algo)}", tf32x3_k=tf32x3)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_channels_last_equals_nchw_bit_for_bit(dtype):
    """The tensor-core kernel accumulates the same products in the same order
    either way, so the channels-last output is the NCHW output transposed,
    exactly; likewise with pre-packed weights."""
    L = _L(dtype=dtype, C=64, H=32, W=32, OC=64, relu=True)
    inp = synthetic.make_inputs(L)
    y_cl, c1 = run_cl(inp)
    y_nchw, c2 = run(inp)
    y_pk, c3 = run_cl(inp, prepack=True)
    assert c1.algo == c2.algo == c3.algo == A_TC
    assert np.array_equal(y_cl, y_nchw)
    assert np.array_equal(y_pk, y_nchw)


@pytest.mark.parametrize("idx", [4, 5])
def test_tensor_core_layers_channels_last_full_output(idx):
    """The wide dense layer and the video-VAE Convolution3D at full size,
    channels-last (no layout pass, no x copy in the workspace): every output
    against the whole oracle result."""
    L = synthetic.LAYERS[idx]
    inp = synthetic.make_inputs(L)
    y, conv = run_cl(inp)
    assert conv.algo == A_TC and y.shape == L.y_shape()
    w_pk = L.kvol * L.OC * L.C * 2             # packed weights only: x is read in place
    assert gb.workspace_size(conv.desc, conv.nsp) == (gb.OK, (w_pk + 255) // 256 * 256)
    assert_close(L.dtype, y, reference(inp), L.name + " channels-last")


def _oracle_chain(layers, inps):
    """Oracle of a chain: each layer's fp64 result rounded to the storage
    dtype (as the device stores it) is the next layer's input."""
    x = inps[0].x
    for L, inp in zip(layers, inps):
        ref = oracle.conv(x, inp.w, inp.b, L.stride, L.pad, L.relu, L.dtype, tpad=L.tpad)
        x = synthetic.to_storage(ref, L.dtype)
    return ref


@pytest.mark.parametrize("dtype,ndim", [("f16", 2), ("bf16", 3)])
def test_chained_layers_channels_last(dtype, ndim):
    """Three convolutions chained on the device with channels-last output
    feeding channels-last input (no re-layout between layers), against the
    oracle chain."""
    if ndim == 2:
        shapes = [dict(C=16, OC=64, H=24, W=40, relu=True),
                  dict(C=64, OC=48, H=24, W=40, relu=True, stride=2),
                  dict(C=48, OC=32, H=12, W=20)]
    else:
        shapes = [dict(C=16, OC=32, D=5, H=8, W=24, relu=True, tpad=gb.TPAD_CAUSAL),
                  dict(C=32, OC=32, D=5, H=8, W=24, relu=True, tpad=gb.TPAD_CAUSAL),
                  dict(C=32, OC=16, D=5, H=8, W=24, tpad=gb.TPAD_CAUSAL)]
    layers, inps = [], []
    for i, sh in enumerate(shapes):
        L = _L(dtype=dtype, ndim=ndim, seed=40 + i, **sh)
        layers.append(L)
        inps.append(synthetic.make_inputs(L))
    x = to_device(to_cl(inps[0].x), dtype)
    for L, inp in zip(layers, inps):
        y, conv = run_cl(inp, x_dev=x)
        assert conv.algo == A_TC
        x = conv.y                      # channels-last output -> next input
    ref = _oracle_chain(layers, inps)
    # Each stored intermediate may sit one storage ulp away from the oracle's
    # rounding of the exact value, and the next layer carries that on, so the
    # single-layer element bound does not apply to a chain. The bars: the
    # single-layer NRMSE bars, and every element within (number of layers) x
    # one relative storage ulp of the largest output.
    y, ref = y.ravel(), ref.ravel()
    assert np.isfinite(y).all()
    nrmse = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    ulp = {"f16": 2.0 ** -10, "bf16": 2.0 ** -7}[dtype]
    assert nrmse <= {"f16": 1e-3, "bf16": 2.5e-3}[dtype], nrmse
    max_abs = np.max(np.abs(y - ref))
    assert max_abs <= len(layers) * ulp * np.max(np.abs(ref)), (max_abs, np.max(np.abs(ref)))
