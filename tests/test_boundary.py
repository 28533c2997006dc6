"""C-ABI boundary tests that need no GPU.

The library loads on a machine without a GPU, exports every entry point the
header declares, lays out gbconv_desc as the C compiler does, and rejects
every malformed descriptor with its status code before any CUDA call (a
rejected call never touches the pointers it was given).
"""
import ctypes
import os
import re
import subprocess

import pytest

import implicit_gemm_convolution_conv_gb300 as gb
import synthetic

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbconv.h")
FAKE = 1 << 20          # a non-NULL, well-aligned address never dereferenced

try:
    import torch
    HAVE_GPU = torch.cuda.is_available()
except Exception:       # pragma: no cover
    HAVE_GPU = False


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gbconv_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    syms = declared_symbols()
    assert len(syms) >= 12
    assert sorted(gb.SYMBOLS) == syms
    out = subprocess.run(["nm", "-D", "--defined-only", gb.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (gbconv_\w+)", out))
    for s in syms:
        assert s in exported, s
        assert hasattr(gb.LIB, s)


def test_desc_layout_matches_c(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "gbconv.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu\\n\", sizeof(gbconv_desc),"
        " offsetof(gbconv_desc, flags), offsetof(gbconv_desc, workspace),"
        " offsetof(gbconv_desc, workspace_bytes));return 0;}\n")
    exe = tmp_path / "layout"
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"),
                            "include")
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
                    str(src), "-o", str(exe)], check=True)
    size, off_res, off_ws, off_wsb = map(int, subprocess.run(
        [str(exe)], capture_output=True, text=True, check=True).stdout.split())
    assert ctypes.sizeof(gb.Desc) == size
    assert gb.Desc.flags.offset == off_res
    assert gb.Desc.workspace.offset == off_ws
    assert gb.Desc.workspace_bytes.offset == off_wsb


def _desc(**kw):
    base = dict(N=1, C=3, H=32, W=32, OC=8, k=3, pad=1, stride=1)
    base.update(kw)
    return gb.make_desc(**base)


BAD = [
    (dict(N=0), gb.ERR_SHAPE), (dict(C=-1), gb.ERR_SHAPE),
    (dict(H=0), gb.ERR_SHAPE), (dict(OC=0), gb.ERR_SHAPE),
    (dict(k=0), gb.ERR_SHAPE), (dict(k=17), gb.ERR_SHAPE),
    (dict(stride=0), gb.ERR_SHAPE), (dict(stride=9), gb.ERR_SHAPE),
    (dict(pad=-1), gb.ERR_SHAPE), (dict(H=2, W=2, k=5, pad=0), gb.ERR_SHAPE),
    (dict(D=2), gb.ERR_SHAPE),                       # conv2d needs D == 1
    (dict(N=70000), gb.ERR_SHAPE),
    (dict(N=4096, C=4096, H=4096, W=4096), gb.ERR_SHAPE),
    (dict(dtype=3), gb.ERR_DTYPE), (dict(dtype=-1), gb.ERR_DTYPE),
    (dict(act=2), gb.ERR_ACT), (dict(act=-7), gb.ERR_ACT),
    (dict(w_layout=2), gb.ERR_LAYOUT), (dict(algo=5), gb.ERR_ALGO), (dict(algo=gb.ALGO_DIRECT_TC, C=5), gb.ERR_ALGO), (dict(algo=gb.ALGO_DIRECT_TC, OC=129), gb.ERR_ALGO),
    (dict(flags=16), gb.ERR_RESERVED), (dict(flags=3), gb.ERR_RESERVED),
    (dict(tpad=gb.TPAD_CAUSAL), gb.ERR_SHAPE),      # conv2d: symmetric frames only
    (dict(C=64, algo=gb.ALGO_DIRECT, k=15, pad=7, H=64, W=64, OC=32),
     gb.ERR_ALGO),                                  # halo does not fit smem
]


@pytest.mark.parametrize("dims,ndim", [
    ((65535,) * 6, 3),                                 # N C D H W OC: 65535^5 wraps int64
    ((65535, 65535, 1, 65535, 65535, 65535), 2),       # x: 65535^4 > 2^63
    ((65535, 1, 65535, 65535, 65535, 1), 3),
    ((1, 65535, 65535, 65535, 65535, 1), 3),
])
def test_element_counts_that_overflow_int64_are_rejected(dims, ndim):
    # Element counts are formed with a capped product, so a shape whose
    # count exceeds int64 cannot wrap below the element limit and pass.
    N, C, D, H, W, OC = dims
    d = gb.make_desc(N, C, H, W, OC, 3, 1, 1, D=D)
    assert gb.workspace_size(d, ndim)[0] == gb.ERR_SHAPE
    assert gb.select_algo(d, ndim)[0] == gb.ERR_SHAPE
    assert gb.output_shape(d, ndim)[0] == gb.ERR_SHAPE
    fwd = gb.conv3d_fwd if ndim == 3 else gb.conv2d_fwd
    assert fwd(d, FAKE, FAKE, FAKE, FAKE * 2, 0) == gb.ERR_SHAPE


def test_direct_tile_kernel_grid_limit():
    # The tile kernel's grid z is images x frames x output-channel blocks,
    # at most 65535: beyond it DIRECT is refused and AUTO picks a GEMM.
    big = gb.make_desc(40000, 1, 8, 8, 64, 5, 2, 1, algo=gb.ALGO_DIRECT)   # 40000 x 2 blocks
    assert gb.select_algo(big, 2)[0] == gb.ERR_ALGO
    st, algo = gb.select_algo(gb.make_desc(40000, 1, 8, 8, 64, 5, 2, 1), 2)
    assert st == gb.OK and algo != gb.ALGO_DIRECT
    ok = gb.make_desc(1000, 1, 8, 8, 64, 5, 2, 1, algo=gb.ALGO_DIRECT)
    assert gb.select_algo(ok, 2) == (gb.OK, gb.ALGO_DIRECT)


def test_element_limit_is_inclusive():
    # 4096^3 = 2^36 elements of x (the limit itself) is a valid shape
    d = gb.make_desc(4096, 4096, 64, 64, 1, 3, 1, 1)
    assert gb.select_algo(d, 2)[0] == gb.OK


@pytest.mark.parametrize("kw,status", BAD)
def test_invalid_desc_rejected_before_cuda(kw, status):
    d = _desc(**kw)
    assert gb.conv2d_fwd(d, FAKE, FAKE, FAKE, FAKE * 2, 0) == status
    assert gb.workspace_size(d, 2)[0] == status
    assert gb.select_algo(d, 2)[0] == status


def test_pointer_checks():
    d = _desc()
    assert gb.conv2d_fwd(d, None, FAKE, None, FAKE * 2, 0) == gb.ERR_NULL
    assert gb.conv2d_fwd(d, FAKE, None, None, FAKE * 2, 0) == gb.ERR_NULL
    assert gb.conv2d_fwd(d, FAKE, FAKE, None, None, 0) == gb.ERR_NULL
    assert gb.conv2d_fwd(d, FAKE + 2, FAKE, None, FAKE * 2, 0) == gb.ERR_ALIGN
    assert gb.conv2d_fwd(d, FAKE, FAKE, FAKE + 2, FAKE * 2, 0) == gb.ERR_ALIGN
    # y overlapping x
    assert gb.conv2d_fwd(d, FAKE, FAKE * 4, None, FAKE + 64, 0) == gb.ERR_OVERLAP
    # 16-bit: 2-byte alignment suffices for x, w, y
    dh = _desc(dtype=gb.F16)
    assert gb.conv2d_fwd(dh, FAKE + 1, FAKE, None, FAKE * 2, 0) == gb.ERR_ALIGN
    # NULL descriptor
    assert gb.LIB.gbconv_conv2d_fwd(None, FAKE, FAKE, None, FAKE * 2, 0) == gb.ERR_NULL


def test_workspace_checks():
    L = synthetic.LAYERS[4]
    d = gb.make_desc(L.N, L.C, L.H, L.W, L.OC, L.k, L.pad, L.stride,
                     dtype=gb.F16)
    st, need = gb.workspace_size(d, 2)
    assert st == gb.OK
    Cp = (L.C + 7) // 8 * 8
    x_cl = L.N * L.H * L.W * Cp * 2
    w_pk = 9 * L.OC * Cp * 2
    assert need == (x_cl + 255) // 256 * 256 + (w_pk + 255) // 256 * 256
    assert gb.conv2d_fwd(d, FAKE, FAKE * 64, None, FAKE * 128, 0) == gb.ERR_WORKSPACE
    d.workspace, d.workspace_bytes = FAKE * 256, need - 1
    assert gb.conv2d_fwd(d, FAKE, FAKE * 64, None, FAKE * 128, 0) == gb.ERR_WORKSPACE
    d.workspace, d.workspace_bytes = FAKE * 256 + 16, need
    assert gb.conv2d_fwd(d, FAKE, FAKE * 64, None, FAKE * 128, 0) == gb.ERR_WORKSPACE
    # pre-packed weights need no weight scratch
    d.w_layout = gb.W_PACKED
    assert gb.workspace_size(d, 2) == (gb.OK, (x_cl + 255) // 256 * 256)
    assert gb.weight_packed_size(d, 2) == (gb.OK, w_pk)


def test_workspace_holds_the_split_k_partial_sums_of_small_fp32_layers():
    """fp32 on the CUDA-core GEMM with C % 16 == 0 and NCHW x: a layer of
    fewer than 160 tiles of 128 x 128 splits K, and its workspace holds S
    slices of [OC][N*OH*OW] fp32 partial sums
    (S = min(8, K steps / 2), fewer if the slices would pass 64 MB); a
    larger layer, a channel count not divisible by 16, channels-last x or
    16-bit storage get none."""
    def ws(N, C, H, W, OC, **kw):
        d = gb.make_desc(N, C, H, W, OC, 3, 1, 1, algo=gb.ALGO_IGEMM_FFMA, w_layout=gb.W_PACKED, **kw)
        st, n = gb.workspace_size(d, 2)
        assert st == gb.OK
        return n
    # layer 3: 120 tiles, K = 9 * 64 = 576 -> 36 steps of 16 -> 8 slices of 128 x 15360 fp32
    slices = 128 * 16 * 12 * 80 * 4
    assert ws(16, 64, 12, 80, 128) == 8 * slices
    # 16 channels: 9 steps -> 4 slices
    assert ws(2, 16, 20, 30, 40) == (4 * 40 * 2 * 20 * 30 * 4 + 255) // 256 * 256
    assert ws(64, 64, 40, 80, 128) == 0                  # 1600 tiles: no split
    assert ws(16, 60, 12, 80, 128) == 0                  # C % 16 != 0
    assert ws(16, 64, 12, 80, 128, channels_last=True) == 0
    assert ws(16, 64, 12, 80, 128, dtype=gb.F16) == 0
    # OIHW weights add the packed copy in front of the partial sums
    d = gb.make_desc(16, 64, 12, 80, 128, 3, 1, 1, algo=gb.ALGO_IGEMM_FFMA)
    w_pk = 9 * 64 * 128 * 4
    assert gb.workspace_size(d, 2) == (gb.OK, (w_pk + 255) // 256 * 256 + 8 * slices)


def test_workspace_overlapping_an_input_is_rejected():
    # The layout pass and the weight pack write the workspace while x, w and
    # b are read: a workspace over any of them is refused before any CUDA call.
    L = synthetic.LAYERS[4]
    d = gb.make_desc(L.N, L.C, L.H, L.W, L.OC, L.k, L.pad, L.stride, dtype=gb.F16)
    need = gb.workspace_size(d, 2)[1]
    x, w, b, y = FAKE, FAKE * 64, FAKE * 96, FAKE * 128      # x spans 8.4 MB from 1 MiB
    d.workspace_bytes = need
    for ws in (x + 4096 * 256, w, b - 256):                   # inside x, at w, over b
        d.workspace = ws
        assert gb.conv2d_fwd(d, x, w, b, y, 0) == gb.ERR_OVERLAP, ws


@pytest.mark.skipif(HAVE_GPU, reason="this check needs a machine without a GPU")
def test_valid_desc_reaches_device_check_without_gpu():
    """A fully valid call on a machine without a GPU returns
    UNSUPPORTED_DEVICE and never crashes."""
    d = _desc()
    assert gb.conv2d_fwd(d, FAKE, FAKE * 4, FAKE * 8, FAKE * 16, 0) == \
        gb.ERR_UNSUPPORTED_DEVICE
    assert gb.device_supported(0) == 0
    assert gb.device_supported(-1) == 0
    assert gb.check_device_error(0) == gb.ERR_CUDA


@pytest.mark.parametrize("idx", sorted(synthetic.LAYERS))
def test_shapes_and_algorithm_of_the_five_layers(idx):
    L = synthetic.LAYERS[idx]
    d = gb.make_desc(L.N, L.C, L.H, L.W, L.OC, L.k, L.pad, L.stride, D=L.D,
                     dtype=L.dtype)
    st, (od, oh, ow) = gb.output_shape(d, L.ndim)
    assert st == gb.OK
    assert (od, oh, ow) == L.out_dims()
    st, algo = gb.select_algo(d, L.ndim)
    assert st == gb.OK
    expect = {1: gb.ALGO_DIRECT, 2: gb.ALGO_DIRECT_TC, 3: gb.ALGO_IGEMM_TC,
              4: gb.ALGO_IGEMM_TC, 5: gb.ALGO_IGEMM_TC}[idx]
    assert algo == expect, gb.algo_name(algo)


def test_auto_keeps_long_fp32_reductions_on_the_cuda_cores():
    """fp32 layers go to the tensor cores' three TF32 products only while
    the reduction C * k^d is at most 1,000 products (the three-product
    error grows with it); longer ones, NCHW or channels-last, go to the
    exact-fp32 CUDA-core GEMM. 16-bit storage stays on the tensor cores."""
    pick = lambda **kw: gb.select_algo(_desc(**kw), 2)[1]
    assert pick(C=64, OC=128, H=12, W=80, k=3, pad=1) == gb.ALGO_IGEMM_TC          # 576
    assert pick(C=111, OC=128, H=12, W=80, k=3, pad=1) == gb.ALGO_IGEMM_TC         # 999
    assert pick(C=112, OC=128, H=12, W=80, k=3, pad=1) == gb.ALGO_IGEMM_FFMA       # 1008
    assert pick(C=48, OC=128, H=12, W=80, k=5, pad=2) == gb.ALGO_IGEMM_FFMA        # 1200
    assert pick(C=256, OC=256, H=32, W=32, k=3, pad=1, dtype=gb.F16) == gb.ALGO_IGEMM_TC
    d = gb.make_desc(1, 128, 32, 32, 64, 3, 1, 1, channels_last=True)
    assert gb.select_algo(d, 2) == (gb.OK, gb.ALGO_IGEMM_FFMA)
    d = gb.make_desc(1, 128, 32, 32, 64, 3, 1, 1, D=4)                             # 3456 in 3D
    assert gb.select_algo(d, 3) == (gb.OK, gb.ALGO_IGEMM_FFMA)


def test_auto_picks_tensor_core_stem_for_fp32_stems():
    """fp32 3x3 stems (C <= 4) with 16 to 128 output channels go to the
    tensor-core stem; narrower and wider ones, other dtypes, C > 4 and the
    fused pool do not."""
    pick = lambda **kw: gb.select_algo(_desc(**kw), 2)[1]
    assert pick(C=3, OC=64, H=640, W=640, k=3, pad=1, stride=2) == gb.ALGO_DIRECT_TC
    assert pick(C=3, OC=128, H=64, W=64, k=3, pad=1, stride=1) == gb.ALGO_DIRECT_TC
    assert pick(C=3, OC=32, H=640, W=640, k=3, pad=1, stride=2) == gb.ALGO_DIRECT_TC
    assert pick(C=4, OC=16, H=64, W=64, k=3, pad=1, stride=1) == gb.ALGO_DIRECT_TC
    assert pick(C=3, OC=8, H=32, W=32, k=3, pad=1, stride=1) == gb.ALGO_DIRECT
    assert pick(C=5, OC=64, H=64, W=64, k=3, pad=1, stride=1) != gb.ALGO_DIRECT_TC
    assert pick(C=3, OC=32, H=64, W=64, k=3, pad=1, stride=2, pool=True) == gb.ALGO_DIRECT
    assert pick(C=3, OC=160, H=64, W=64, k=3, pad=1, stride=1) != gb.ALGO_DIRECT_TC
    assert pick(C=3, OC=64, H=64, W=64, k=3, pad=1, stride=1, dtype=gb.F16) != gb.ALGO_DIRECT_TC


def test_fused_maxpool_shapes_and_limits():
    """Pooled y is [OH/2][OW/2] (floor); the fused pool exists on the
    few-channel 3x3 direct kernel only."""
    mk = lambda **kw: _desc(**dict(dict(pool=True), **kw))
    assert gb.output_shape(mk(H=32, W=32), 2) == (gb.OK, (1, 16, 16))
    assert gb.output_shape(mk(H=9, W=11), 2) == (gb.OK, (1, 4, 5))
    assert gb.output_shape(mk(H=640, W=640, stride=2), 2) == (gb.OK, (1, 160, 160))
    assert gb.select_algo(mk(H=64, W=64, OC=64), 2) == (gb.OK, gb.ALGO_DIRECT)
    assert gb.select_algo(mk(algo=gb.ALGO_IGEMM_FFMA), 2)[0] == gb.ERR_ALGO
    assert gb.select_algo(mk(algo=gb.ALGO_DIRECT_TC, OC=64), 2)[0] == gb.ERR_ALGO
    assert gb.select_algo(mk(C=8), 2)[0] == gb.ERR_ALGO
    assert gb.select_algo(mk(k=5, pad=2), 2)[0] == gb.ERR_ALGO
    assert gb.output_shape(mk(H=1, W=8, pad=0, k=1), 2)[0] == gb.ERR_SHAPE
    d3 = gb.make_desc(1, 3, 8, 8, 4, 3, 1, 1, D=4, pool=True)
    assert gb.output_shape(d3, 3)[0] == gb.ERR_SHAPE


def test_fp32_tensor_core_gemm_workspace():
    """fp32 layers beyond the direct kernels' reach run on the tensor cores as
    three TF32 products: x and the packed weights carry a hi and a lo half of
    C rounded up to 32 channels each; the CUDA-core GEMM stays available."""
    L = synthetic.LAYERS[3]
    d = gb.make_desc(L.N, L.C, L.H, L.W, L.OC, L.k, L.pad, L.stride)
    assert gb.select_algo(d, 2) == (gb.OK, gb.ALGO_IGEMM_TC)
    Cs = (L.C + 31) // 32 * 32
    x_split = L.N * L.H * L.W * 2 * Cs * 4
    w_pk = 9 * L.OC * 2 * Cs * 4
    assert gb.weight_packed_size(d, 2) == (gb.OK, w_pk)
    assert gb.workspace_size(d, 2) == (gb.OK, (x_split + 255) // 256 * 256 + (w_pk + 255) // 256 * 256)
    d.algo = gb.ALGO_IGEMM_FFMA
    assert gb.select_algo(d, 2) == (gb.OK, gb.ALGO_IGEMM_FFMA)
    # C = 20 pads each half to 32 channels; channels-last fp32 still splits x in the workspace
    dc = gb.make_desc(2, 20, 9, 13, 40, 3, 1, 1, channels_last=True)
    assert gb.select_algo(dc, 2) == (gb.OK, gb.ALGO_IGEMM_TC)
    assert gb.workspace_size(dc, 2) == (gb.OK, (2 * 9 * 13 * 64 * 4 + 255) // 256 * 256 +
                                        (9 * 40 * 64 * 4 + 255) // 256 * 256)


def test_channels_last_algorithms_and_workspace():
    """Channels-last x and y: the tensor-core GEMM for 16-bit storage with C a
    multiple of 8 (reading x in place: no channels-last copy in the
    workspace), else the CUDA-core GEMM; the direct kernels and the fused pool
    refuse the flag."""
    cl = lambda **kw: _desc(**dict(dict(channels_last=True), **kw))
    pick = lambda d, nd=2: gb.select_algo(d, nd)
    assert pick(cl(C=64, OC=64, dtype=gb.F16)) == (gb.OK, gb.ALGO_IGEMM_TC)
    assert pick(cl(C=64, OC=64, dtype=gb.BF16)) == (gb.OK, gb.ALGO_IGEMM_TC)
    assert pick(cl(C=12, OC=64, dtype=gb.F16)) == (gb.OK, gb.ALGO_IGEMM_FFMA)
    assert pick(cl(C=3, OC=32, H=640, W=640, stride=2)) == (gb.OK, gb.ALGO_IGEMM_TC)
    assert pick(cl(C=64, OC=64)) == (gb.OK, gb.ALGO_IGEMM_TC)
    assert pick(cl(C=64, OC=64, algo=gb.ALGO_IGEMM_FFMA)) == (gb.OK, gb.ALGO_IGEMM_FFMA)
    assert pick(cl(C=3, OC=8, algo=gb.ALGO_DIRECT))[0] == gb.ERR_ALGO
    assert pick(cl(C=3, OC=32, algo=gb.ALGO_DIRECT_TC))[0] == gb.ERR_ALGO
    assert pick(cl(C=12, OC=64, dtype=gb.F16, algo=gb.ALGO_IGEMM_TC))[0] == gb.ERR_ALGO
    assert pick(cl(C=3, OC=32, pool=True))[0] == gb.ERR_ALGO
    d3 = gb.make_desc(1, 128, 128, 240, 128, 3, 1, 1, D=5, dtype=gb.F16, channels_last=True)
    assert pick(d3, 3) == (gb.OK, gb.ALGO_IGEMM_TC)
    assert gb.output_shape(d3, 3) == (gb.OK, (5, 128, 240))
    # workspace: packed weights only, and nothing once they are pre-packed
    w_pk = 27 * 128 * 128 * 2
    assert gb.workspace_size(d3, 3) == (gb.OK, (w_pk + 255) // 256 * 256)
    d3.w_layout = gb.W_PACKED
    assert gb.workspace_size(d3, 3) == (gb.OK, 0)
    # the tensor-core kernel reads x in place with TMA: 16-byte alignment
    dh = cl(C=64, OC=64, dtype=gb.F16, w_layout=gb.W_PACKED)
    assert gb.conv2d_fwd(dh, FAKE + 8, FAKE * 64, None, FAKE * 128, 0) == gb.ERR_ALIGN
    # the CUDA-core path takes element alignment
    df = cl(C=12, OC=64, dtype=gb.F16, w_layout=gb.W_PACKED)
    assert gb.conv2d_fwd(df, FAKE + 8, FAKE * 64, None, FAKE * 128, 0) != gb.ERR_ALIGN


def test_frame_padding_modes_shapes():
    """Causal: OD = floor((D-1)/s)+1; none: floor((D-k)/s)+1; H, W unchanged."""
    mk = lambda tp, s=1, D=5: gb.make_desc(1, 4, 6, 7, 2, k=3, pad=1, stride=s, D=D, tpad=tp)
    assert gb.output_shape(mk(gb.TPAD_CAUSAL), 3) == (gb.OK, (5, 6, 7))
    assert gb.output_shape(mk(gb.TPAD_CAUSAL, 2), 3) == (gb.OK, (3, 3, 4))
    assert gb.output_shape(mk(gb.TPAD_NONE), 3) == (gb.OK, (3, 6, 7))
    assert gb.output_shape(mk(gb.TPAD_NONE, 2, 9), 3) == (gb.OK, (4, 3, 4))
    assert gb.output_shape(mk(gb.TPAD_NONE, 1, 2), 3)[0] == gb.ERR_SHAPE
    assert gb.output_shape(mk(gb.TPAD_SYMMETRIC), 3) == (gb.OK, (5, 6, 7))


def test_conv3d_shapes():
    d = gb.make_desc(1, 4, 6, 7, 2, k=3, pad=1, stride=2, D=5)
    assert gb.output_shape(d, 3) == (gb.OK, (3, 3, 4))
    d1 = gb.make_desc(1, 4, 6, 7, 2, k=3, pad=0, stride=1, D=2)
    assert gb.output_shape(d1, 3)[0] == gb.ERR_SHAPE   # frames < k, no pad
    assert gb.output_shape(d1, 4)[0] == gb.ERR_SHAPE   # ndim must be 2 or 3


def test_status_and_algo_names():
    for s in range(0, 15):
        assert gb.status_string(s) and gb.status_string(s) != "unknown status"
    assert gb.status_string(99) == "unknown status"
    assert [gb.algo_name(a) for a in range(5)] == [
        "auto", "direct", "igemm_ffma", "igemm_tc", "direct_tc"]
    assert gb.set_wait_limit_ns(0) == gb.ERR_SHAPE
    assert gb.set_wait_limit_ns(2_000_000_000) == gb.OK


def test_torch_front_end_checks_what_pointers_cannot_say():
    # The C ABI takes raw pointers; the torch front end checks devices,
    # contiguity, dtypes and the weight/bias shapes before any call.
    from implicit_gemm_convolution_conv_gb300.torch_ops import Conv, check_tensors
    x, w, b = torch.zeros(1, 3, 8, 8), torch.zeros(4, 3, 3, 3), torch.zeros(4)
    assert check_tensors(x, w, b, require_cuda=False) == (4, 3)
    assert check_tensors(torch.zeros(1, 8, 8, 3), w, None, channels_last=True, require_cuda=False) == (4, 3)
    assert check_tensors(torch.zeros(1, 3, 4, 8, 8), torch.zeros(4, 3, 3, 3, 3), None,
                         require_cuda=False) == (4, 3)
    bad = [
        (x, torch.zeros(4, 2, 3, 3), b),             # channel count differs from x
        (x, torch.zeros(4, 3, 3, 5), b),             # non-square kernel
        (x, torch.zeros(4, 3, 3, 3, 3), b),          # conv3d weights for a 4-D x
        (x, w.half(), b),                            # dtype differs from x
        (x, w, torch.zeros(5)),                      # bias length
        (x, w, torch.zeros(4, dtype=torch.float64)), # bias dtype
        (x.transpose(2, 3), w, b),                   # non-contiguous x
        (x.long(), w.long(), b),                     # unsupported dtype
    ]
    for args in bad:
        with pytest.raises(ValueError):
            check_tensors(*args, require_cuda=False)
    with pytest.raises(TypeError):
        check_tensors(x, w.numpy(), b, require_cuda=False)
    with pytest.raises(ValueError, match="CUDA"):
        Conv(x, w, b)                                # CPU tensors: there is no CPU path


def test_make_desc_refuses_values_wider_than_a_c_int():
    # ctypes would wrap 2^32 + 1 to 1 without a word; the binding refuses it
    for kw in (dict(N=2**32 + 1), dict(C=-2**31 - 1), dict(OC=2**40)):
        args = dict(N=1, C=3, H=8, W=8, OC=4, k=3, pad=1, stride=1)
        args.update(kw)
        with pytest.raises(ValueError):
            gb.make_desc(**args)


@pytest.mark.skipif(HAVE_GPU, reason="checks the host-side log line on a machine without a GPU")
def test_gbconv_log_writes_the_kernel_choice_to_stderr():
    """GBCONV_LOG=1: a forward call writes one line with its shape, frame
    padding, algorithm, weight layout and workspace to stderr (here the call
    then stops at the device check, as there is no GPU). Without the
    variable nothing is written."""
    import sys
    code = (
        "import implicit_gemm_convolution_conv_gb300 as gb\n"
        "d = gb.make_desc(1, 128, 128, 240, 128, 3, 1, 1, D=5, dtype=gb.F16, tpad=gb.TPAD_CAUSAL,\n"
        "                 workspace=1 << 32, workspace_bytes=1 << 30)\n"
        "print(gb.conv3d_fwd(d, 1 << 20, 1 << 28, None, 1 << 29, 0))\n")
    env = dict(os.environ, GBCONV_LOG="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert int(r.stdout.strip()) == gb.ERR_UNSUPPORTED_DEVICE
    line = [l for l in r.stderr.splitlines() if l.startswith("gbconv: conv3d")]
    assert len(line) == 1, r.stderr
    assert "algo=igemm_tc" in line[0] and "frame_pad" in line[0] and "OD=5 OH=128 OW=240" in line[0]
    env.pop("GBCONV_LOG")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "gbconv:" not in r.stderr
