"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Every case runs on seeded synthetic inputs. The five layer shapes run at full
size through the same call the bench times (AUTO kernel choice, OIHW weights
packed in the call) and are compared element by element with the whole
oracle output. A sweep of small shapes spanning several tiles and ragged tails
covers each kernel family, each storage dtype, 2D and 3D, odd sizes, k = 1/3/5,
pad 0/1/2, stride 1/2/3, no bias, ReLU.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import implicit_gemm_convolution_conv_gb300 as gb
from implicit_gemm_convolution_conv_gb300.torch_ops import Conv, to_numpy
from gpu_helpers import assert_close, device_inputs, reference, run

pytestmark = pytest.mark.gpu

A_DIRECT, A_FFMA, A_TC = gb.ALGO_DIRECT, gb.ALGO_IGEMM_FFMA, gb.ALGO_IGEMM_TC
A_DTC = gb.ALGO_DIRECT_TC
CAUSAL, NOPAD = gb.TPAD_CAUSAL, gb.TPAD_NONE


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    assert gb.device_supported(torch.cuda.current_device()) == 1
    yield
    assert gb.check_device_error() == gb.OK


# ------------------------------------------------------- the five layers
@pytest.mark.parametrize("idx", [1, 2, 3])
def test_layer_full_output(idx):
    L = synthetic.LAYERS[idx]
    inp = synthetic.make_inputs(L)
    y, conv = run(inp)
    ref = reference(inp)
    assert_close(L.dtype, y, ref, L.name)


def test_layer3_on_cuda_cores_full_output():
    """The text-line batch through the exact-fp32 CUDA-core implicit GEMM
    (AUTO runs it on the tensor cores as three TF32 products): every output
    against the fp64 oracle."""
    L = synthetic.LAYERS[3]
    inp = synthetic.make_inputs(L)
    y, conv = run(inp, algo=A_FFMA)
    assert conv.algo == A_FFMA
    assert_close(L.dtype, y, reference(inp), L.name + " on CUDA cores")


def test_layer5_causal_frames_full_output():
    """The video-VAE Convolution3D shape with causal frame padding (the
    SeedVR2 decoder's conv; git.erdda.com/Tencent/ncnn/discussions/7001
    section 3.3): all 19.7 M outputs against the whole oracle result."""
    import dataclasses
    L = dataclasses.replace(synthetic.LAYERS[5], tpad=CAUSAL)
    inp = synthetic.make_inputs(L)
    y, conv = run(inp)
    assert conv.algo == A_TC and y.shape == L.y_shape()
    assert_close(L.dtype, y, reference(inp), L.name + " causal")


def test_layer2_with_fused_maxpool_full_output():
    """The 640x640 stem with its 2x2 max pool fused into the epilogue:
    every pooled output against max-pool(conv) of the oracle."""
    import dataclasses
    L = dataclasses.replace(synthetic.LAYERS[2], pool=True)
    inp = synthetic.make_inputs(L)
    y, conv = run(inp)
    assert conv.algo == A_DIRECT and y.shape == L.y_shape() == (1, 32, 160, 160)
    assert_close(L.dtype, y, reference(inp), L.name + " + maxpool")


def test_layer2_on_tensor_cores_full_output():
    """The 640x640 stem through the three-TF32-product tensor-core kernel,
    every output against the fp64 oracle at the fp32 tolerance."""
    L = synthetic.LAYERS[2]
    inp = synthetic.make_inputs(L)
    y, conv = run(inp, algo=A_DTC)
    assert conv.algo == A_DTC
    assert_close(L.dtype, y, reference(inp), L.name)


@pytest.mark.parametrize("OC,W", [(32, 640), (128, 640), (32, 638)])
def test_stem_tensor_cores_many_tiles_per_group(OC, W):
    """Four 640-row images through the tensor-core stem: 3,200 tiles, so
    every group runs five or more tiles and its two halo buffers are reused
    (barrier phases past the first flip). OC 32 keeps the pixel operand in
    TMEM with four groups, OC 128 in shared memory with two; W = 638 (OW not
    a multiple of 4) takes the plain-load path. Every output is checked."""
    L = synthetic.Layer(f"stem_many_tiles_oc{OC}_w{W}", N=4, C=3, H=640, W=W, OC=OC, k=3, pad=1,
                        stride=2, dtype="f32", relu=True, x_dist="u01", w_dist="he", b_dist="u01_1",
                        seed=77 + OC + W)
    inp = synthetic.make_inputs(L)
    y, conv = run(inp, algo=A_DTC)
    assert conv.algo == A_DTC
    assert_close(L.dtype, y, reference(inp), L.name)


# Stems of 720 and 800 tiles of 2 rows x 64 pixels (five or six tiles per SM
# on 152 SMs, so one or two of a CTA's four groups run a second tile).
STEMS_5_6 = [
    # 720 tiles; OC 24 (padded to 32), no bias
    synthetic.Layer("stem_720_tiles_oc24", N=1, C=2, H=288, W=320, OC=24, k=3, pad=1, stride=1, dtype="f32",
                    x_dist="u01", w_dist="he", b_dist="none", seed=301),
    # 800 tiles, stride 3 (the widest halo box), OC 16, ReLU
    synthetic.Layer("stem_800_tiles_s3", N=1, C=3, H=960, W=960, OC=16, k=3, pad=1, stride=3, dtype="f32",
                    relu=True, x_dist="u01", w_dist="he", b_dist="u01_1", seed=302),
    # 800 tiles over four images, one input channel, a 16-pixel last column tile
    synthetic.Layer("stem_800_tiles_c1_ragged", N=4, C=1, H=200, W=416, OC=8, k=3, pad=1, stride=2, dtype="f32",
                    relu=True, x_dist="u01", w_dist="he", b_dist="u01_1", seed=303),
    # 720 tiles, an odd number of output rows (the last row pair is half empty)
    synthetic.Layer("stem_720_tiles_odd_rows", N=1, C=3, H=574, W=640, OC=32, k=3, pad=1, stride=2, dtype="f32",
                    relu=True, x_dist="u01", w_dist="he", b_dist="u01_1", seed=304),
]


@pytest.mark.parametrize("L", STEMS_5_6, ids=lambda L: L.name)
def test_stem_tensor_cores_five_or_six_tiles_per_sm(L):
    """The tensor-core stem at tile counts near the 640 x 640 stem's: ragged
    channel counts, no bias, stride 3 (the widest halo box), one input
    channel, a part-width last tile and a half-empty last row pair. Every
    output is checked."""
    inp = synthetic.make_inputs(L)
    y, conv = run(inp, algo=A_DTC)
    assert conv.algo == A_DTC
    assert_close(L.dtype, y, reference(inp), L.name)


@pytest.mark.parametrize("idx,dtype", [(4, "f16"), (5, "f16"), (4, "bf16")])
def test_tensor_core_layer_full_output(idx, dtype):
    """The wide dense layer (f16, bf16) and the video-VAE Convolution3D at
    full size through the call the bench times: every output against the
    whole oracle result (a one-index slip in a store can leave most of a
    tensor looking right, so no sampling)."""
    L = synthetic.layer(idx, dtype=dtype)
    inp = synthetic.make_inputs(L)
    y, conv = run(inp)
    assert conv.algo == A_TC
    assert_close(L.dtype, y, reference(inp), L.name)


# --------------------------------------------------------- shape sweep
def _L(dtype="f32", N=1, C=3, D=1, H=9, W=11, OC=4, k=3, pad=1, stride=1,
       relu=False, bias=True, ndim=2, seed=1, tpad=0, pool=False):
    return synthetic.Layer("sweep", N=N, C=C, D=D, H=H, W=W, OC=OC, k=k,
                           pad=pad, stride=stride, dtype=dtype, relu=relu,
                           ndim=ndim, x_dist="n01", w_dist="he",
                           b_dist="u11" if bias else "none", seed=seed,
                           tpad=tpad, pool=pool)


SWEEP = [
    # direct kernel: templated k3/s1, k3/s2 and generic k/s, narrow and wide
    (A_DIRECT, _L(C=3, H=32, W=32, OC=8)),
    (A_DIRECT, _L(C=3, H=33, W=65, OC=40, stride=2, relu=True)),
    (A_DIRECT, _L(C=2, H=1, W=70, OC=5, k=3, pad=1)),
    (A_DIRECT, _L(C=3, H=13, W=17, OC=16, k=5, pad=2, stride=3)),
    (A_DIRECT, _L(C=4, H=6, W=9, OC=33, k=1, pad=0, bias=False)),
    (A_DIRECT, _L(N=3, C=3, H=20, W=70, OC=24, k=3, pad=0, stride=1)),
    (A_DIRECT, _L(C=2, D=4, H=7, W=9, OC=6, ndim=3)),
    (A_DIRECT, _L(C=1, D=5, H=9, W=8, OC=20, ndim=3, stride=2, relu=True)),
    (A_DIRECT, _L(dtype="f16", C=3, H=40, W=67, OC=32, stride=2)),
    (A_DIRECT, _L(dtype="bf16", C=3, H=21, W=30, OC=8)),
    (A_DIRECT, _L(C=4, H=18, W=36, OC=64, stride=2, pad=0, relu=True)),
    (A_DIRECT, _L(C=1, N=2, H=7, W=44, OC=36, stride=1)),
    (A_DIRECT, _L(dtype="f16", C=3, H=24, W=64, OC=16, stride=2)),
    # more than 65,536 outputs: the stem kernel's halo ring (smaller layers
    # take one thread per output): stride 2, two channel blocks, bf16
    (A_DIRECT, _L(dtype="f16", C=3, H=130, W=200, OC=32, stride=2)),
    (A_DIRECT, _L(C=1, N=2, H=70, W=130, OC=36)),
    (A_DIRECT, _L(dtype="bf16", C=3, H=90, W=100, OC=8, relu=True)),
    # CUDA-core implicit GEMM: ragged M, N and K, strides, 3D
    (A_FFMA, _L(N=2, C=20, H=9, W=13, OC=130, relu=True)),
    (A_FFMA, _L(C=64, H=12, W=80, OC=128)),
    (A_FFMA, _L(C=7, H=15, W=16, OC=9, k=5, pad=2, stride=2)),
    (A_FFMA, _L(C=5, H=10, W=10, OC=70, k=1, pad=0, stride=3, bias=False)),
    (A_FFMA, _L(C=6, D=5, H=6, W=7, OC=12, ndim=3)),
    (A_FFMA, _L(C=3, D=6, H=7, W=5, OC=65, ndim=3, stride=2, pad=2)),
    (A_FFMA, _L(dtype="f16", N=2, C=16, H=11, W=12, OC=40)),
    # fp32 with C % 16 == 0 (cp.async stages): a ragged last pixel tile and
    # an OC tail, 3D with stride 2, k = 5, and enough pixels for 128-channel
    # tiles (more tiles than SMs)
    (A_FFMA, _L(N=3, C=32, H=7, W=13, OC=70, relu=True)),
    (A_FFMA, _L(C=16, D=4, H=6, W=10, OC=24, ndim=3, stride=2)),
    (A_FFMA, _L(N=2, C=48, H=20, W=36, OC=200, k=5, pad=2, bias=False)),
    (A_FFMA, _L(N=8, C=32, H=40, W=64, OC=130)),
    (A_FFMA, _L(dtype="bf16", C=12, H=9, W=9, OC=17, relu=True)),
    # tensor-core implicit GEMM: several tiles, ragged tails, partial
    # channel blocks, OC tails, strides, k 1/3/5, 3D incl. a single frame
    (A_TC, _L(dtype="f16", C=64, H=8, W=128, OC=64)),
    (A_TC, _L(dtype="f16", N=2, C=72, H=5, W=150, OC=40, relu=True)),
    (A_TC, _L(dtype="f16", C=3, H=20, W=20, OC=16)),
    (A_TC, _L(dtype="f16", C=136, H=7, W=33, OC=300, bias=False)),
    (A_TC, _L(dtype="f16", C=32, H=17, W=61, OC=48, k=5, pad=2)),
    (A_TC, _L(dtype="f16", C=16, H=12, W=14, OC=24, k=1, pad=0)),
    (A_TC, _L(dtype="f16", C=24, H=19, W=41, OC=32, stride=2)),
    (A_TC, _L(dtype="f16", C=8, H=16, W=300, OC=16, stride=3, pad=2)),
    (A_TC, _L(dtype="bf16", C=64, H=9, W=70, OC=128, relu=True)),
    (A_TC, _L(dtype="f16", C=16, D=5, H=8, W=40, OC=32, ndim=3)),
    (A_TC, _L(dtype="f16", C=32, D=1, H=10, W=12, OC=16, ndim=3)),
    (A_TC, _L(dtype="bf16", C=8, D=6, H=9, W=10, OC=24, ndim=3, stride=2)),
    # tensor-core implicit GEMM read from NCHW in place (stride 1, W % 8 == 0):
    # several rows per tile, one row per tile, column tiles with a ragged
    # tail, partial channel blocks, OC tails, k 1/3/5/7, pad 0..3, 3D
    (A_TC, _L(dtype="f16", N=2, C=72, H=5, W=152, OC=40, relu=True)),
    (A_TC, _L(dtype="f16", C=136, H=7, W=32, OC=300, bias=False)),
    (A_TC, _L(dtype="f16", C=32, H=17, W=64, OC=48, k=5, pad=2)),
    (A_TC, _L(dtype="f16", C=16, H=12, W=16, OC=24, k=1, pad=0)),
    (A_TC, _L(dtype="f16", C=8, H=3, W=520, OC=16)),
    (A_TC, _L(dtype="f16", C=64, H=4, W=256, OC=130, pad=0)),
    (A_TC, _L(dtype="f16", C=3, H=10, W=8, OC=16, pad=2)),
    (A_TC, _L(dtype="f16", C=40, H=9, W=48, OC=20, k=7, pad=3, relu=True)),
    (A_TC, _L(dtype="bf16", C=64, H=9, W=72, OC=128, relu=True)),
    (A_TC, _L(dtype="bf16", C=24, D=3, H=6, W=24, OC=40, ndim=3)),
    (A_TC, _L(dtype="f16", N=3, C=200, D=2, H=5, W=240, OC=64, ndim=3)),
    # fp32 on the tensor-core implicit GEMM (three TF32 products, x and the
    # weights split into hi and lo halves of C rounded up to 32): several
    # tiles, channel counts that are not multiples of 32, OC tails and two
    # output-channel tiles, strides, k 1/3/5, 3D with causal frames, ReLU
    (A_TC, _L(C=64, H=12, W=80, OC=128, relu=True)),
    (A_TC, _L(N=2, C=20, H=9, W=13, OC=40)),
    (A_TC, _L(C=48, H=17, W=61, OC=136, k=5, pad=2, bias=False)),
    (A_TC, _L(C=16, H=12, W=14, OC=24, k=1, pad=0)),
    (A_TC, _L(C=40, H=19, W=41, OC=32, stride=2, relu=True)),
    (A_TC, _L(C=8, H=4, W=300, OC=16, stride=3, pad=2)),
    (A_TC, _L(C=32, D=5, H=8, W=40, OC=32, ndim=3)),
    (A_TC, _L(C=24, D=6, H=7, W=9, OC=20, ndim=3, stride=2, tpad=CAUSAL)),
    # more tiles than SMs (persistent CTAs, staging apart from the ring):
    # fp32 and f16
    (A_TC, _L(N=16, C=32, H=40, W=64, OC=32, relu=True)),
    (A_TC, _L(dtype="f16", N=16, C=64, H=40, W=64, OC=64)),
    (A_TC, _L(N=4, C=32, H=64, W=100, OC=32, bias=False)),
    # 16-bit, more than 128 output channels (several output-channel tiles):
    # more tiles than SMs (persistent loop, two accumulators), three full
    # channel tiles over small images (tiles cross images), 3D with an OC
    # tail, bf16 with stride 2
    (A_TC, _L(dtype="f16", N=4, C=64, H=40, W=64, OC=256)),
    (A_TC, _L(dtype="bf16", N=3, C=40, H=9, W=11, OC=384, relu=True)),
    (A_TC, _L(dtype="f16", C=32, D=3, H=8, W=30, OC=260, ndim=3)),
    (A_TC, _L(dtype="bf16", N=2, C=72, H=33, W=47, OC=200, stride=2, bias=False)),
    # more row tiles than CTAs with a partial last wave, 2D and 3D
    (A_TC, _L(dtype="f16", N=2, C=16, H=100, W=160, OC=32, relu=True)),
    (A_TC, _L(dtype="bf16", C=16, D=3, H=70, W=240, OC=16, ndim=3, tpad=CAUSAL)),
    # fp32 stems on tensor cores (three TF32 products): C 1..3, strides 1..3,
    # ragged 32-pixel groups, OC tails within a 16-channel MMA N, N > 32
    (A_DTC, _L(C=3, H=32, W=32, OC=8)),
    (A_DTC, _L(C=3, H=33, W=65, OC=40, stride=2, relu=True)),
    (A_DTC, _L(C=1, H=7, W=44, OC=36)),
    (A_DTC, _L(N=3, C=2, H=20, W=70, OC=24, pad=0)),
    (A_DTC, _L(C=3, H=40, W=67, OC=64, stride=2, bias=False)),
    (A_DTC, _L(C=3, H=9, W=9, OC=100, stride=3)),
    (A_DTC, _L(C=3, H=12, W=30, OC=128, relu=True)),
    (A_DTC, _L(C=2, H=1, W=5, OC=3)),
    (A_DTC, _L(C=4, H=21, W=37, OC=32, stride=2, relu=True)),
    (A_DTC, _L(N=5, C=3, H=13, W=11, OC=17)),
    (A_DTC, _L(C=4, H=8, W=8, OC=1, pad=0)),
    (A_DTC, _L(N=2, C=3, H=100, W=130, OC=32, stride=2, relu=True)),
    # rows 16-byte aligned: TMA halo loads and tensor stores
    (A_DTC, _L(C=3, H=64, W=64, OC=32, stride=2, relu=True)),
    (A_DTC, _L(N=2, C=3, H=50, W=200, OC=24, stride=2)),
    (A_DTC, _L(C=1, H=30, W=36, OC=128, relu=True)),
    (A_DTC, _L(C=4, H=20, W=68, OC=48)),
    (A_DTC, _L(C=2, H=27, W=96, OC=64, stride=3, bias=False)),
    (A_DTC, _L(N=3, C=3, H=16, W=16, OC=16, stride=2, relu=True)),
    # conv3d frame padding: causal (k-1 zero frames in front) and none, on
    # every kernel family that takes 3D, strides 1 and 2, k 3 and 5
    (A_DIRECT, _L(C=2, D=5, H=7, W=9, OC=6, ndim=3, tpad=CAUSAL)),
    (A_DIRECT, _L(C=1, D=6, H=9, W=8, OC=20, ndim=3, stride=2, tpad=NOPAD)),
    (A_FFMA, _L(C=6, D=5, H=6, W=7, OC=12, ndim=3, tpad=CAUSAL, relu=True)),
    (A_FFMA, _L(C=3, D=7, H=7, W=5, OC=65, ndim=3, k=5, pad=2, tpad=NOPAD)),
    (A_TC, _L(dtype="f16", C=16, D=5, H=8, W=40, OC=32, ndim=3, tpad=CAUSAL)),
    (A_TC, _L(dtype="bf16", C=24, D=9, H=6, W=24, OC=40, ndim=3, stride=2, tpad=CAUSAL)),
    (A_TC, _L(dtype="f16", C=32, D=4, H=10, W=12, OC=16, ndim=3, tpad=NOPAD)),
    # conv + bias + ReLU + 2x2 max pool in one kernel (few-channel 3x3):
    # strides 1/2, pad 0/1, C 1..4, odd rows / columns (floor mode), OC tails,
    # a pooled width not divisible by 4, no ReLU, f16 / bf16
    (A_DIRECT, _L(C=3, H=32, W=32, OC=32, relu=True, pool=True)),
    (A_DIRECT, _L(C=3, H=45, W=70, OC=40, stride=2, relu=True, pool=True)),
    (A_DIRECT, _L(C=1, H=9, W=11, OC=5, pool=True)),
    (A_DIRECT, _L(N=2, C=4, H=17, W=26, OC=64, pad=0, pool=True, relu=True)),
    (A_DIRECT, _L(C=2, H=6, W=38, OC=33, stride=2, pool=True, bias=False)),
    (A_DIRECT, _L(dtype="f16", C=3, H=40, W=64, OC=32, stride=2, relu=True, pool=True)),
    (A_DIRECT, _L(dtype="bf16", C=3, H=21, W=30, OC=8, pool=True)),
]


@pytest.mark.parametrize("algo,L", SWEEP,
                         ids=[f"{gb.algo_name(a)}-{i}" for i, (a, _) in enumerate(SWEEP)])
def test_sweep(algo, L):
    inp = synthetic.make_inputs(L)
    y, conv = run(inp, algo=algo)
    assert conv.algo == algo
    tf32x3 = L.C * L.k ** L.ndim if (L.dtype == "f32" and algo == A_TC) else 0
    assert_close(L.dtype, y, reference(inp), str(L), tf32x3_k=tf32x3)


# -------------------------------------------------- packing, determinism
@pytest.mark.parametrize("idx,algo", [(2, A_DIRECT), (3, A_FFMA), (3, A_TC), (4, A_TC)])
def test_prepacked_weights_give_identical_output(idx, algo):
    inp = synthetic.make_inputs(synthetic.LAYERS[idx])
    y0, _ = run(inp, algo=algo)
    y1, _ = run(inp, algo=algo, prepack=True)
    y2, _ = run(inp, algo=algo)
    np.testing.assert_array_equal(y0, y1)
    np.testing.assert_array_equal(y0, y2)


def test_weight_pack_is_a_permutation():
    """Packed tensor-core weights: wp[tap][oc][c] = w[oc][c][tap], zero pad."""
    L = _L(dtype="f16", C=12, OC=5, k=3)
    inp = synthetic.make_inputs(L)
    _, w, _ = device_inputs(inp)
    d = gb.make_desc(1, 12, 9, 11, 5, 3, 1, 1, dtype=gb.F16, algo=A_TC)
    st, nb = gb.weight_packed_size(d, 2)
    assert st == gb.OK and nb == 9 * 5 * 16 * 2
    wp = torch.zeros(nb // 2 + 128, dtype=torch.float16, device="cuda")
    off = (-wp.data_ptr()) % 256 // 2
    wp = wp[off:off + nb // 2]
    assert gb.weight_pack(d, 2, w, wp) == gb.OK
    got = to_numpy(wp).reshape(9, 5, 16)
    ref = np.zeros((9, 5, 16), np.float16)
    ref[:, :, :12] = inp.w.reshape(5, 12, 9).transpose(2, 0, 1)
    np.testing.assert_array_equal(got, ref)


# --------------------------------------------------------- API behaviour
def test_guard_bands_untouched():
    """Stores stay inside y: canary bands around it keep their bytes."""
    for idx in (1, 3, 4):
        L = synthetic.LAYERS[idx]
        inp = synthetic.make_inputs(L)
        x, w, b = device_inputs(inp)
        ny = int(np.prod(L.y_shape()))
        band = 4096
        buf = torch.full((ny + 2 * band,), -7.0, dtype=x.dtype, device="cuda")
        y = buf[band:band + ny].view(L.y_shape())
        Conv(x, w, b, L.stride, L.pad, L.relu, out=y)()
        torch.cuda.synchronize()
        assert bool((buf[:band] == -7.0).all()) and bool((buf[-band:] == -7.0).all())


def test_graph_capture_and_side_stream():
    L = synthetic.LAYERS[4]
    inp = synthetic.make_inputs(L)
    x, w, b = device_inputs(inp)
    conv = Conv(x, w, b, L.stride, L.pad, L.relu)
    eager = conv().clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        conv.y.zero_()
        conv(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(conv.y, eager)
    g = torch.cuda.CUDAGraph()
    conv.y.zero_()
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        conv()
    conv.y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(conv.y, eager)


def test_repeat_calls_do_not_grow_memory():
    """Many back-to-back calls: no device memory growth (cf. the driver leak
    found by million-iteration loops in githubissues.com/ysh329/OpenCL-101/52)."""
    L = synthetic.LAYERS[2]
    inp = synthetic.make_inputs(L)
    x, w, b = device_inputs(inp)
    conv = Conv(x, w, b, L.stride, L.pad, L.relu)
    conv()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(10000):
        conv()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert abs(free1 - free0) < (8 << 20)
    assert gb.check_device_error() == gb.OK


def test_runtime_errors_on_gpu():
    L = synthetic.LAYERS[4]
    inp = synthetic.make_inputs(L)
    x, w, b = device_inputs(inp)
    y = torch.empty(L.y_shape(), dtype=x.dtype, device="cuda")
    d = gb.make_desc(L.N, L.C, L.H, L.W, L.OC, L.k, L.pad, L.stride, dtype=gb.F16)
    assert gb.conv2d_fwd(d, x, w, b, y) == gb.ERR_WORKSPACE
    d32 = gb.make_desc(1, 5, 8, 8, 4, 3, 1, 1, algo=A_DTC)       # the stem kernel takes C <= 4
    assert gb.conv2d_fwd(d32, x, w, b, y) == gb.ERR_ALGO
    assert gb.conv3d_fwd(d, x, w, b, y) in (gb.ERR_WORKSPACE, gb.ERR_SHAPE)
