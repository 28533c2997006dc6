"""Plant plausible mistakes in a copy of the oracle and check the pins catch them.

Each mutant is the oracle's C source with one expression changed, compiled
into a temporary library on the CPU. The pins used here (hand-worked goldens,
all-ones closed form, torch float64 conv) must reject every mutant, which
shows they constrain the parts of the definition a slip would touch: kernel
orientation, pad sign, bias, channel range, tap offsets and index order.
"""
import ctypes
import json
import os
import subprocess

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "conv_ref.c")

MUTANTS = {
    "flipped_kernel": (
        "double wv = w[((oc * C + ic) * k + ky) * k + kx];",
        "double wv = w[((oc * C + ic) * k + (k - 1 - ky)) * k + (k - 1 - kx)];"),
    "pad_sign": ("int64_t iy = oy * stride - pad + ky;\n            if (iy < 0 || iy >= H)",
                 "int64_t iy = oy * stride + pad + ky;\n            if (iy < 0 || iy >= H)"),
    "dropped_bias": ("    if (b)\n        acc += b[oc];\n    if (relu && acc < 0.0)\n        acc = 0.0;\n    return acc;\n}\n\n/* One output element of the 3D",
                     "    if (b)\n        acc += 0.0 * b[oc];\n    if (relu && acc < 0.0)\n        acc = 0.0;\n    return acc;\n}\n\n/* One output element of the 3D"),
    "last_channel_skipped": ("for (int64_t ic = 0; ic < C; ic++) {\n        for (int64_t ky",
                             "for (int64_t ic = 0; ic + 1 < C; ic++) {\n        for (int64_t ky"),
    "transposed_input_index": (
        "double xv = x[((n * C + ic) * H + iy) * W + ix];",
        "double xv = x[((n * C + ic) * H + ix) * W + iy];"),
    "stride_on_tap": ("int64_t ix = ox * stride - pad + kx;\n                if (ix < 0 || ix >= W)",
                      "int64_t ix = ox * stride - pad + kx * stride;\n                if (ix < 0 || ix >= W)"),
    "relu_before_bias": (
        "    if (b)\n        acc += b[oc];\n    if (relu && acc < 0.0)\n        acc = 0.0;\n    return acc;\n}\n\n/* One output element of the 3D",
        "    if (relu && acc < 0.0)\n        acc = 0.0;\n    if (b)\n        acc += b[oc];\n    return acc;\n}\n\n/* One output element of the 3D"),
}


def _build_mutant(name, tmp_path):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-std=c99", "-O1", "-fPIC", "-shared", str(path),
                    "-o", str(lib)], check=True, capture_output=True)
    so = ctypes.CDLL(str(lib))
    dp = ctypes.POINTER(ctypes.c_double)
    so.oracle_conv2d.argtypes = [ctypes.c_int] * 9 + [dp] * 4
    so.oracle_conv2d.restype = ctypes.c_int
    return so


def _run2d(so, x, w, b, stride, pad, relu):
    x = np.ascontiguousarray(x, np.float64)
    w = np.ascontiguousarray(w, np.float64)
    N, C, H, W = x.shape
    OC, k = w.shape[0], w.shape[2]
    OH = (H + 2 * pad - k) // stride + 1
    OW = (W + 2 * pad - k) // stride + 1
    y = np.zeros((N, OC, OH, OW))
    dp = ctypes.POINTER(ctypes.c_double)
    bb = None if b is None else np.ascontiguousarray(b, np.float64)
    so.oracle_conv2d(N, C, H, W, OC, k, pad, stride, int(relu),
                     x.ctypes.data_as(dp), w.ctypes.data_as(dp),
                     None if bb is None else bb.ctypes.data_as(dp),
                     y.ctypes.data_as(dp))
    return y


def _pins_pass(conv):
    """The subset of pins applied to a mutant; True only if all hold."""
    g = json.load(open(os.path.join(HERE, "golden", "handworked_3x3.json")))
    x = np.array(g["x"], np.float64)[None, None]
    w = np.array(g["w"], np.float64)[None, None]
    for case in g["cases"]:
        y = conv(x, w, None, case["stride"], g["pad"], False)
        if not np.array_equal(y[0, 0], np.array(case["y"], np.float64)):
            return False
    # all-ones closed form with a bias (square input keeps indexes in range)
    IC, H = 3, 5
    y = conv(np.ones((1, IC, H, H)), np.ones((1, IC, 3, 3)), np.array([0.25]),
             1, 1, False)
    exp = np.full((H, H), 9.0 * IC)
    exp[0, :] = exp[-1, :] = exp[:, 0] = exp[:, -1] = 6.0 * IC
    exp[0, 0] = exp[0, -1] = exp[-1, 0] = exp[-1, -1] = 4.0 * IC
    if not np.array_equal(y[0, 0], exp + 0.25):
        return False
    # torch float64 on a square random case with a negative bias and ReLU
    torch = pytest.importorskip("torch")
    r = np.random.Generator(np.random.PCG64(99))
    xr = r.standard_normal((1, 2, 6, 6))
    wr = r.standard_normal((2, 2, 3, 3))
    br = np.array([-0.7, 0.4])
    y = conv(xr, wr, br, 1, 1, True)
    ref = torch.nn.functional.relu(torch.nn.functional.conv2d(
        torch.from_numpy(xr), torch.from_numpy(wr), torch.from_numpy(br),
        padding=1)).numpy()
    return bool(np.allclose(y, ref, rtol=1e-12, atol=1e-12))


def test_unmutated_oracle_passes_the_subset():
    assert _pins_pass(lambda x, w, b, s, p, r: oracle.conv2d(x, w, b, s, p, r))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    so = _build_mutant(name, tmp_path)
    assert not _pins_pass(lambda x, w, b, s, p, r: _run2d(so, x, w, b, s, p,
                                                          r)), name


# ------------------------------------------------------- conv3d frame padding
MUTANTS_3D = {
    "frame_front_pad_is_spatial_pad": ("int64_t id = od * stride - pd0 + kd;",
                                       "int64_t id = od * stride - pad + kd;"),
    "frame_front_pad_sign": ("int64_t id = od * stride - pd0 + kd;",
                             "int64_t id = od * stride + pd0 + kd;"),
    "frame_extent_ignores_back_pad": ("int64_t span = in + (int64_t)p0 + p1 - k;",
                                      "int64_t span = in + (int64_t)p0 + p0 - k;"),
}


def _run3d(so, x, w, pad, pd0, pd1):
    x = np.ascontiguousarray(x, np.float64)
    w = np.ascontiguousarray(w, np.float64)
    N, C, D, H, W = x.shape
    OC, k = w.shape[0], w.shape[2]
    OD = (D + pd0 + pd1 - k) + 1
    OH, OW = H + 2 * pad - k + 1, W + 2 * pad - k + 1
    # room for any frame count a mutant may compute; read back the true shape
    room = N * OC * (D + 2 * max(pd0, pd1, 1) + 1) * OH * OW
    buf = np.full(room, np.nan)
    dp = ctypes.POINTER(ctypes.c_double)
    rc = so.oracle_conv3d(N, C, D, H, W, OC, k, pad, pd0, pd1, 1, 0,
                          x.ctypes.data_as(dp), w.ctypes.data_as(dp), None,
                          buf.ctypes.data_as(dp))
    return buf[:N * OC * OD * OH * OW].reshape(N, OC, OD, OH, OW) if rc == 0 else None


def _pins3d_pass(run):
    """Frame-padding pins applied to a mutant: PyTorch float64 for the causal
    and no-padding modes."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    r = np.random.Generator(np.random.PCG64(77))
    x = r.standard_normal((1, 2, 5, 4, 4))
    w = r.standard_normal((2, 2, 3, 3, 3))
    tx, tw = torch.from_numpy(x), torch.from_numpy(w)
    for pd0, pd1, ref in [(2, 0, F.conv3d(F.pad(tx, (0, 0, 0, 0, 2, 0)), tw, padding=(0, 1, 1))),
                          (0, 0, F.conv3d(tx, tw, padding=(0, 1, 1)))]:
        y = run(x, w, 1, pd0, pd1)
        if y is None or y.shape != tuple(ref.shape) or not np.allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12):
            return False
    return True


def _build_mutant3d(name, tmp_path):
    src = open(SRC).read()
    old, new = MUTANTS_3D[name]
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-std=c99", "-O1", "-fPIC", "-shared", str(path),
                    "-o", str(lib)], check=True, capture_output=True)
    so = ctypes.CDLL(str(lib))
    dp = ctypes.POINTER(ctypes.c_double)
    so.oracle_conv3d.argtypes = [ctypes.c_int] * 12 + [dp] * 4
    so.oracle_conv3d.restype = ctypes.c_int
    return so


def test_unmutated_oracle_passes_the_frame_subset():
    assert _pins3d_pass(lambda x, w, p, a, b: oracle.conv3d(
        x, w, None, 1, p, tpad=oracle.TPAD_CAUSAL if a else oracle.TPAD_NONE))


@pytest.mark.parametrize("name", sorted(MUTANTS_3D))
def test_frame_mutant_is_caught(name, tmp_path):
    so = _build_mutant3d(name, tmp_path)
    # the mutant's own output length, so a wrong extent shows as a mismatch
    assert not _pins3d_pass(lambda x, w, p, a, b: _run3d(so, x, w, p, a, b)), name
