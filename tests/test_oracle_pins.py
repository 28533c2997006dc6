"""Pins for the fp64 CPU oracle, independent of the oracle's own code.

Each test checks the oracle against something other than itself: values worked
by hand (tests/golden), closed forms, special cases that reduce to a library
routine (matmul, torch float64 conv), invariants of the definition, and an
independent im2col formulation on tiny inputs. A plausible mistake in the
oracle (a flipped kernel, a wrong pad sign, a dropped bias, a transposed
index, a skipped channel) fails at least one of them; test_oracle_mutants
plants such mistakes in a copy of the oracle and checks that they are caught.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


# ---------------------------------------------------------------- hand-worked
def test_handworked_3x3_golden():
    g = json.load(open(os.path.join(GOLDEN, "handworked_3x3.json")))
    x = np.array(g["x"], np.float64)[None, None]
    w = np.array(g["w"], np.float64)[None, None]
    for case in g["cases"]:
        y = oracle.conv2d(x, w, None, stride=case["stride"], pad=g["pad"])
        np.testing.assert_array_equal(y[0, 0], np.array(case["y"], np.float64))


def test_handworked_3d_golden():
    g = json.load(open(os.path.join(GOLDEN, "handworked_3d.json")))
    x = np.array(g["x"], np.float64)[None, None]
    w = np.array(g["w"], np.float64)[None, None]
    b = np.array([g["b"]], np.float64)
    y = oracle.conv3d(x, w, b, stride=g["stride"], pad=g["pad"])
    np.testing.assert_array_equal(y[0, 0], np.array(g["y"], np.float64))


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("IC,H,W", [(1, 3, 3), (3, 5, 6), (5, 4, 7)])
def test_all_ones_3x3_closed_form(IC, H, W):
    """All-ones x and w, 3x3, pad 1, stride 1, bias beta: a corner output sees
    4 taps per channel, an edge 6, an interior one 9."""
    beta = 0.25
    x = np.ones((1, IC, H, W))
    w = np.ones((2, IC, 3, 3))
    b = np.full(2, beta)
    y = oracle.conv2d(x, w, b, stride=1, pad=1)
    exp = np.full((H, W), 9.0 * IC)
    exp[0, :] = exp[-1, :] = 6.0 * IC
    exp[:, 0] = exp[:, -1] = 6.0 * IC
    for cy, cx in itertools.product((0, H - 1), (0, W - 1)):
        exp[cy, cx] = 4.0 * IC
    for oc in range(2):
        np.testing.assert_array_equal(y[0, oc], exp + beta)


def test_all_ones_3x3x3_closed_form():
    """3D all-ones: a tap count is the product of per-axis counts (2 at a
    border, 3 inside), so corners 8, edges 12, faces 18, interior 27."""
    IC, D, H, W = 2, 4, 3, 5
    y = oracle.conv3d(np.ones((1, IC, D, H, W)), np.ones((1, IC, 3, 3, 3)),
                      np.array([-1.0]), stride=1, pad=1)

    def cnt(i, n):
        return 2.0 if i in (0, n - 1) else 3.0
    for d, h, w in itertools.product(range(D), range(H), range(W)):
        exp = IC * cnt(d, D) * cnt(h, H) * cnt(w, W) - 1.0
        assert y[0, 0, d, h, w] == exp


@pytest.mark.parametrize("stride", [1, 2])
def test_1x1_is_matmul(stride):
    """k=1, pad 0: y[n] = W[OC x IC] @ X[IC x pixels] (numpy matmul), on the
    stride-subsampled pixels."""
    r = _rng(1)
    x = r.standard_normal((2, 5, 6, 7))
    w = r.standard_normal((4, 5, 1, 1))
    b = r.standard_normal(4)
    y = oracle.conv2d(x, w, b, stride=stride, pad=0)
    xs = x[:, :, ::stride, ::stride]
    for n in range(2):
        ref = (w[:, :, 0, 0] @ xs[n].reshape(5, -1)).reshape(
            4, *xs.shape[2:]) + b[:, None, None]
        np.testing.assert_allclose(y[n], ref, rtol=1e-13, atol=1e-13)


def _shifted(x, dy, dx):
    """out[.., i, j] = x[.., i+dy, j+dx], zero where that is outside x."""
    out = np.zeros_like(x)
    H, W = x.shape[-2:]
    for i in range(H):
        for j in range(W):
            if 0 <= i + dy < H and 0 <= j + dx < W:
                out[..., i, j] = x[..., i + dy, j + dx]
    return out


@pytest.mark.parametrize("k,pad", [(3, 1), (5, 2), (3, 0), (2, 1)])
def test_delta_kernel_is_shift(k, pad):
    """w[oc,ic,ty,tx] = [oc==ic][ty==t0y][tx==t0x]: output channel c is input
    channel c shifted by (t0 - pad) and zero-filled; the centre tap with
    pad=(k-1)/2 is the identity."""
    r = _rng(2)
    C = 3
    x = r.standard_normal((1, C, 6, 7))
    H, W = 6, 7
    for ty, tx in itertools.product(range(k), range(k)):
        w = np.zeros((C, C, k, k))
        for c in range(C):
            w[c, c, ty, tx] = 1.0
        y = oracle.conv2d(x, w, None, stride=1, pad=pad)
        OH, OW = H + 2 * pad - k + 1, W + 2 * pad - k + 1
        full = _shifted(np.pad(x, ((0, 0), (0, 0), (0, 8), (0, 8))),
                        ty - pad, tx - pad)
        np.testing.assert_array_equal(y, full[:, :, :OH, :OW])
        if k % 2 == 1 and pad == (k - 1) // 2 and (ty, tx) == (pad, pad):
            np.testing.assert_array_equal(y, x)


def test_delta_kernel_3d_is_shift():
    r = _rng(3)
    x = r.standard_normal((1, 2, 4, 5, 3))
    for td, ty, tx in [(0, 0, 0), (1, 1, 1), (2, 0, 1), (0, 2, 2)]:
        w = np.zeros((2, 2, 3, 3, 3))
        w[0, 0, td, ty, tx] = w[1, 1, td, ty, tx] = 1.0
        y = oracle.conv3d(x, w, None, stride=1, pad=1)
        exp = np.zeros_like(x)
        D, H, W = x.shape[2:]
        for d, h, ww in itertools.product(range(D), range(H), range(W)):
            s = (d + td - 1, h + ty - 1, ww + tx - 1)
            if 0 <= s[0] < D and 0 <= s[1] < H and 0 <= s[2] < W:
                exp[:, :, d, h, ww] = x[:, :, s[0], s[1], s[2]]
        np.testing.assert_array_equal(y, exp)


# ---------------------------------------------------------- border invariants
@pytest.mark.parametrize("k,pad,stride", [(3, 1, 1), (3, 1, 2), (5, 2, 3),
                                          (3, 2, 2), (4, 1, 2)])
def test_single_pixel_footprint(k, pad, stride):
    """x zero but one pixel: the output support is exactly the outputs whose
    window covers that pixel, and there y = v*w[tap] + b; elsewhere y = b."""
    r = _rng(4)
    H, W, C, OC = 9, 8, 2, 3
    w = r.standard_normal((OC, C, k, k))
    b = r.standard_normal(OC)
    OH = (H + 2 * pad - k) // stride + 1
    OW = (W + 2 * pad - k) // stride + 1
    for (c, iy, ix) in [(0, 0, 0), (1, 4, 3), (0, H - 1, W - 1), (1, 0, W - 1)]:
        x = np.zeros((1, C, H, W))
        v = 1.5
        x[0, c, iy, ix] = v
        y = oracle.conv2d(x, w, b, stride=stride, pad=pad)
        for oc, oy, ox in itertools.product(range(OC), range(OH), range(OW)):
            ty, tx = iy - (oy * stride - pad), ix - (ox * stride - pad)
            if 0 <= ty < k and 0 <= tx < k:
                exp = v * w[oc, c, ty, tx] + b[oc]
            else:
                exp = b[oc]
            assert y[0, oc, oy, ox] == exp


def test_padding_only_outputs_equal_bias():
    """With pad >= k, corner outputs see only padding: y = b, or ReLU(b)."""
    r = _rng(5)
    x = r.standard_normal((1, 2, 5, 5))
    w = r.standard_normal((4, 2, 3, 3))
    b = np.array([0.5, -0.5, 0.0, 2.0])
    for relu in (False, True):
        y = oracle.conv2d(x, w, b, stride=1, pad=3, relu=relu)
        for oy, ox in [(0, 0), (0, y.shape[3] - 1), (y.shape[2] - 1, 0),
                       (y.shape[2] - 1, y.shape[3] - 1)]:
            exp = np.maximum(b, 0) if relu else b
            np.testing.assert_array_equal(y[0, :, oy, ox], exp)


# ----------------------------------------------------------------- invariants
def test_linearity():
    r = _rng(6)
    x = r.standard_normal((2, 3, 7, 6))
    w1, w2 = r.standard_normal((2, 4, 3, 3, 3))
    y1 = oracle.conv2d(x, w1, None, stride=2, pad=1)
    y2 = oracle.conv2d(x, w2, None, stride=2, pad=1)
    y12 = oracle.conv2d(x, w1 + w2, None, stride=2, pad=1)
    np.testing.assert_allclose(y12, y1 + y2, rtol=1e-12, atol=1e-12)
    ya = oracle.conv2d(2.5 * x, w1, None, stride=2, pad=1)
    np.testing.assert_allclose(ya, 2.5 * y1, rtol=1e-12, atol=1e-12)


def test_translation_equivariance():
    """Stride 1: shifting x by one pixel shifts outputs away from borders."""
    r = _rng(7)
    x = r.standard_normal((1, 2, 10, 10))
    w = r.standard_normal((3, 2, 3, 3))
    y = oracle.conv2d(x, w, None, stride=1, pad=1)
    xs = np.roll(x, shift=(1, 2), axis=(2, 3))
    ys = oracle.conv2d(xs, w, None, stride=1, pad=1)
    np.testing.assert_allclose(ys[:, :, 3:-1, 4:-1], y[:, :, 2:-2, 2:-3],
                               rtol=1e-12, atol=1e-12)


def test_relu_is_max_of_linear():
    r = _rng(8)
    x = r.standard_normal((1, 3, 6, 6))
    w = r.standard_normal((5, 3, 3, 3))
    b = r.standard_normal(5)
    y0 = oracle.conv2d(x, w, b, stride=1, pad=1, relu=False)
    y1 = oracle.conv2d(x, w, b, stride=1, pad=1, relu=True)
    np.testing.assert_array_equal(y1, np.maximum(y0, 0.0))
    assert (y0 < 0).any() and (y0 > 0).any()


def test_conv3d_centre_temporal_tap_is_per_frame_conv2d():
    r = _rng(9)
    x = r.standard_normal((1, 3, 4, 6, 5))
    w = np.zeros((2, 3, 3, 3, 3))
    w[:, :, 1] = r.standard_normal((2, 3, 3, 3))
    b = r.standard_normal(2)
    y = oracle.conv3d(x, w, b, stride=1, pad=1)
    for t in range(4):
        y2 = oracle.conv2d(x[:, :, t], w[:, :, 1], b, stride=1, pad=1)
        np.testing.assert_allclose(y[:, :, t], y2, rtol=1e-13, atol=1e-13)


def test_conv3d_single_frame_uses_middle_slice():
    """T=1 with pad 1: only the middle temporal slice touches real frames."""
    r = _rng(10)
    x = r.standard_normal((2, 3, 1, 5, 7))
    w = r.standard_normal((4, 3, 3, 3, 3))
    y = oracle.conv3d(x, w, None, stride=1, pad=1)
    y2 = oracle.conv2d(x[:, :, 0], w[:, :, 1], None, stride=1, pad=1)
    np.testing.assert_allclose(y[:, :, 0], y2, rtol=1e-13, atol=1e-13)


# --------------------------------------------------- independent formulations
def _im2col_conv(x, w, b, stride, pad, relu):
    """Second formulation: explicit zero-padded patch matrix, then matmul."""
    nsp = x.ndim - 2
    k = w.shape[-1]
    xp = np.pad(x, [(0, 0), (0, 0)] + [(pad, pad)] * nsp)
    outs = [(n + 2 * pad - k) // stride + 1 for n in x.shape[2:]]
    N, C = x.shape[:2]
    cols = []
    for pos in itertools.product(*[range(o) for o in outs]):
        sl = tuple(slice(p * stride, p * stride + k) for p in pos)
        cols.append(xp[(slice(None), slice(None)) + sl].reshape(N, -1))
    A = np.stack(cols, axis=1)                       # N x P x (C*k^nsp)
    B = w.reshape(w.shape[0], -1).T                  # (C*k^nsp) x OC
    y = A @ B                                        # N x P x OC
    if b is not None:
        y = y + b
    if relu:
        y = np.maximum(y, 0.0)
    return np.moveaxis(y, 2, 1).reshape((N, w.shape[0]) + tuple(outs))


def test_brute_force_im2col_2d():
    r = _rng(11)
    cases = list(itertools.product([1, 3, 5], [0, 1, 2], [1, 2, 3]))
    for i, (k, pad, stride) in enumerate(cases):
        N, C, OC = 1 + i % 2, 1 + i % 4, 1 + (i * 3) % 4
        H, W = 3 + i % 5, 7 - i % 4
        if H + 2 * pad < k or W + 2 * pad < k:
            continue
        x = r.standard_normal((N, C, H, W))
        w = r.standard_normal((OC, C, k, k))
        b = r.standard_normal(OC) if i % 3 else None
        relu = bool(i % 2)
        y = oracle.conv2d(x, w, b, stride=stride, pad=pad, relu=relu)
        ref = _im2col_conv(x, w, b, stride, pad, relu)
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12,
                                   err_msg=str((k, pad, stride)))


def test_brute_force_im2col_3d():
    r = _rng(12)
    for i, (k, pad, stride) in enumerate(itertools.product([1, 3], [0, 1, 2],
                                                           [1, 2])):
        x = r.standard_normal((1 + i % 2, 2, 3 + i % 3, 4, 5))
        w = r.standard_normal((3, 2, k, k, k))
        b = r.standard_normal(3)
        y = oracle.conv3d(x, w, b, stride=stride, pad=pad, relu=bool(i % 2))
        ref = _im2col_conv(x, w, b, stride, pad, bool(i % 2))
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_torch_float64_third_opinion():
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    r = _rng(13)
    x = r.standard_normal((2, 5, 9, 11))
    w = r.standard_normal((6, 5, 3, 3))
    b = r.standard_normal(6)
    for stride, pad in [(1, 1), (2, 1), (3, 0), (1, 2)]:
        y = oracle.conv2d(x, w, b, stride=stride, pad=pad, relu=True)
        ref = F.relu(F.conv2d(torch.from_numpy(x), torch.from_numpy(w),
                              torch.from_numpy(b), stride=stride,
                              padding=pad)).numpy()
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    x3 = r.standard_normal((1, 3, 5, 6, 7))
    w3 = r.standard_normal((4, 3, 3, 3, 3))
    y3 = oracle.conv3d(x3, w3, None, stride=1, pad=1)
    ref3 = F.conv3d(torch.from_numpy(x3), torch.from_numpy(w3), None,
                    stride=1, padding=1).numpy()
    np.testing.assert_allclose(y3, ref3, rtol=1e-12, atol=1e-12)


def test_points_match_full():
    """conv_at (one output at a time) equals the full computation."""
    r = _rng(14)
    x = r.standard_normal((2, 3, 9, 10))
    w = r.standard_normal((4, 3, 3, 3))
    b = r.standard_normal(4)
    y = oracle.conv2d(x, w, b, stride=2, pad=1, relu=True)
    idx = r.integers(0, y.size, 300)
    np.testing.assert_array_equal(
        oracle.conv_at(x, w, b, idx, stride=2, pad=1, relu=True),
        y.ravel()[idx])
    x3 = r.standard_normal((1, 2, 4, 5, 6))
    w3 = r.standard_normal((3, 2, 3, 3, 3))
    y3 = oracle.conv3d(x3, w3, b[:3], stride=1, pad=1)
    idx3 = r.integers(0, y3.size, 200)
    np.testing.assert_array_equal(
        oracle.conv_at(x3, w3, b[:3], idx3, stride=1, pad=1), y3.ravel()[idx3])
    with pytest.raises(ValueError):
        oracle.conv_at(x, w, b, [y.size], stride=2, pad=1)


# ------------------------------------------------ storage widening / inputs
def test_widen_is_exact():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0001, 0x7F7F], np.uint16)
    got = oracle.widen(bits, "bf16")
    exp = np.array([1.0, -1.0, 3.140625, 2.0 ** -133, 3.3895313892515355e38])
    np.testing.assert_array_equal(got, exp)
    h = np.array([1.0, 2.0 ** -24, 65504.0, -0.5], np.float16)
    np.testing.assert_array_equal(oracle.widen(h), [1.0, 2.0 ** -24, 65504.0,
                                                    -0.5])


def test_bf16_rounding_of_inputs():
    """Ties go to even; a value just above a tie rounds up."""
    v = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 +
                  2.0 ** -20, -2.0])
    bits = synthetic.to_bf16_bits(v)
    np.testing.assert_array_equal(oracle.widen(bits, "bf16"),
                                  [1.0, 1.0 + 2 * 2.0 ** -7, 1.0 + 2.0 ** -7,
                                   -2.0])


def test_layer_table_matches_stated_work():
    """FLOP and compulsory-byte counts of the five layers, by hand."""
    L = synthetic.LAYERS
    assert L[1].flops() == 2 * 8 * 32 * 32 * 3 * 9
    assert L[2].flops() == 2 * 32 * 320 * 320 * 3 * 9
    assert L[4].flops() == 2 * 256 * 128 * 128 * 256 * 9
    assert L[5].flops() == 2 * 128 * 5 * 128 * 240 * 128 * 27
    assert L[2].compulsory_bytes() == 4 * (3 * 640 * 640 + 32 * 27 +
                                           32 * 320 * 320) + 4 * 32
    assert L[5].compulsory_bytes() == 2 * (2 * 128 * 5 * 128 * 240 +
                                           128 * 128 * 27) + 4 * 128


# ------------------------------------------------ conv3d frame padding modes
def _ext_count(o, n, k=3, pad=1):
    return sum(1 for t in range(k) if 0 <= o - pad + t < n)


def test_causal_frames_all_ones_closed_form():
    """All-ones input and weights, causal frame padding (k-1 zero frames
    before, none after): output frame t sums min(t+1, k) input frames, so
    y[t, oy, ox] = min(t+1, 3) * (in-bounds rows) * (in-bounds columns)."""
    D, H, W = 5, 4, 5
    y = oracle.conv3d(np.ones((1, 1, D, H, W)), np.ones((1, 1, 3, 3, 3)), None,
                      stride=1, pad=1, tpad=oracle.TPAD_CAUSAL)
    assert y.shape == (1, 1, D, H, W)
    for t in range(D):
        for oy in range(H):
            for ox in range(W):
                exp = min(t + 1, 3) * _ext_count(oy, H) * _ext_count(ox, W)
                assert y[0, 0, t, oy, ox] == exp, (t, oy, ox)


def test_causal_output_never_reads_later_frames():
    """Changing input frames after t leaves output frames 0..t bit-identical;
    changing frame t changes output frame t."""
    r = _rng(31)
    x = r.standard_normal((1, 2, 6, 5, 6))
    w = r.standard_normal((3, 2, 3, 3, 3))
    b = r.standard_normal(3)
    y0 = oracle.conv3d(x, w, b, stride=1, pad=1, tpad=oracle.TPAD_CAUSAL)
    for t in range(5):
        x2 = x.copy()
        x2[:, :, t + 1:] = r.standard_normal(x2[:, :, t + 1:].shape)
        y2 = oracle.conv3d(x2, w, b, stride=1, pad=1, tpad=oracle.TPAD_CAUSAL)
        np.testing.assert_array_equal(y2[:, :, :t + 1], y0[:, :, :t + 1])
        x3 = x.copy()
        x3[:, :, t] += 1.0
        y3 = oracle.conv3d(x3, w, b, stride=1, pad=1, tpad=oracle.TPAD_CAUSAL)
        assert not np.array_equal(y3[:, :, t], y0[:, :, t])


@pytest.mark.parametrize("stride", [1, 2])
def test_frame_padding_modes_match_torch_float64(stride):
    """Causal = PyTorch conv3d on the input with k-1 zero frames prepended and
    no frame padding; none = PyTorch with no frame padding; symmetric = the
    usual padding on all three axes."""
    F = pytest.importorskip("torch.nn.functional")
    import torch
    r = _rng(32 + stride)
    x = r.standard_normal((2, 3, 7, 5, 6))
    w = r.standard_normal((4, 3, 3, 3, 3))
    b = r.standard_normal(4)
    tx, tw, tb = torch.from_numpy(x), torch.from_numpy(w), torch.from_numpy(b)
    causal = F.conv3d(F.pad(tx, (0, 0, 0, 0, 2, 0)), tw, tb, stride=stride,
                      padding=(0, 1, 1)).numpy()
    none = F.conv3d(tx, tw, tb, stride=stride, padding=(0, 1, 1)).numpy()
    sym = F.conv3d(tx, tw, tb, stride=stride, padding=1).numpy()
    for mode, ref in [(oracle.TPAD_CAUSAL, causal), (oracle.TPAD_NONE, none),
                      (oracle.TPAD_SYMMETRIC, sym)]:
        y = oracle.conv3d(x, w, b, stride=stride, pad=1, tpad=mode)
        assert y.shape == ref.shape, mode
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
        idx = r.integers(0, y.size, 200)
        np.testing.assert_array_equal(
            oracle.conv_at(x, w, b, idx, stride=stride, pad=1, tpad=mode),
            y.ravel()[idx])


def test_frame_padding_output_lengths():
    """OD = floor((D-1)/s)+1 causal, floor((D-k)/s)+1 none."""
    for D, s in [(5, 1), (5, 2), (9, 2), (4, 3)]:
        x = np.ones((1, 1, D, 4, 4))
        w = np.ones((1, 1, 3, 3, 3))
        assert oracle.conv3d(x, w, None, s, 1, tpad=oracle.TPAD_CAUSAL).shape[2] == (D - 1) // s + 1
        assert oracle.conv3d(x, w, None, s, 1, tpad=oracle.TPAD_NONE).shape[2] == (D - 3) // s + 1
    with pytest.raises(ValueError):
        oracle.conv(np.ones((1, 1, 4, 4)), np.ones((1, 1, 3, 3)), tpad=oracle.TPAD_CAUSAL)


# ------------------------------------------------------------- max pool 2x2
def test_maxpool2_handworked_and_floor_mode():
    y = np.array([[1., 5., 2., 0., 9.],
                  [3., 4., 8., 7., 9.],
                  [6., 0., 1., 2., 9.]])[None, None]
    np.testing.assert_array_equal(oracle.maxpool2(y)[0, 0], [[5., 8.]])


def test_maxpool2_matches_torch():
    F = pytest.importorskip("torch.nn.functional")
    import torch
    r = _rng(51)
    for shape in [(2, 3, 8, 10), (1, 4, 7, 9), (1, 1, 2, 2)]:
        y = r.standard_normal(shape)
        ref = F.max_pool2d(torch.from_numpy(y), 2, 2).numpy()
        np.testing.assert_array_equal(oracle.maxpool2(y), ref)
