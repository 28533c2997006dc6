"""GPU parity on hand-picked edge shapes, through AUTO and every algorithm
the library accepts for each (the check of test_gpu_random_shapes): many
tiny images (tiles across images), one-row and one-column images, 1,024
output channels, 1,024 input channels with 1x1 kernels, k = 7 at stride 2
with more than 128 output channels, conv3d with causal frames at stride 2,
one output channel, a single pixel, padding wider than half the kernel, a
depth-1 conv3d with k = 7, stride 3 on odd extents, a 1920-pixel-wide
image, 200 channels-last images, and a three-channel stem with four output
channels."""
import pytest

import synthetic
from test_gpu_random_shapes import test_random_problem as check

pytestmark = pytest.mark.gpu


def L(name, **kw):
    base = dict(N=1, C=8, D=1, H=8, W=8, OC=8, k=3, pad=1, stride=1, dtype="f32", relu=False, ndim=2,
                x_dist="n01", w_dist="he", b_dist="u005", seed=5, tpad=0, cl=False)
    base.update(kw)
    return synthetic.Layer(name, **base)


CASES = [
    L("tiny_images", N=64, C=16, H=4, W=4, OC=32),
    L("tiny_images_f16", N=64, C=16, H=4, W=4, OC=32, dtype="f16"),
    L("one_row", C=1, H=1, W=3000, OC=8),
    L("one_row_f16", C=8, H=1, W=3000, OC=24, dtype="f16"),
    L("one_col", C=8, H=3000, W=1, OC=16),
    L("one_col_bf16", C=16, H=3000, W=1, OC=16, dtype="bf16"),
    L("oc1024_f16", N=2, C=256, H=16, W=16, OC=1024, dtype="f16"),
    L("c1024_1x1_f16", C=1024, H=8, W=8, OC=64, k=1, pad=0, dtype="f16"),
    L("c1024_1x1_f32", C=1024, H=8, W=8, OC=64, k=1, pad=0),
    L("k7_s2_oc300", C=3, H=64, W=64, OC=300, k=7, pad=3, stride=2),
    L("k7_s2_oc300_f16", C=3, H=64, W=64, OC=300, k=7, pad=3, stride=2, dtype="f16"),
    L("conv3d_causal_s2", C=32, D=16, H=16, W=16, OC=64, stride=2, ndim=3, tpad=1, dtype="f16"),
    L("conv3d_k5_s3_cl_f32", C=20, D=9, H=20, W=20, OC=40, k=5, pad=0, stride=3, ndim=3, cl=True),
    L("oc1_f16", C=64, H=32, W=32, OC=1, dtype="f16"),
    L("oc1_f32", C=64, H=32, W=32, OC=1),
    L("trivial", C=1, H=1, W=1, OC=1, k=1, pad=0),
    L("one_pixel_f16", C=64, H=1, W=1, OC=64, k=1, pad=0, dtype="f16"),
    L("pad_gt_half", C=16, H=5, W=5, OC=16, k=3, pad=3),
    L("pad_gt_half_f16_cl", C=16, H=5, W=5, OC=16, k=3, pad=3, dtype="f16", cl=True),
    L("bf16_3d_d1_k7_cl", C=24, D=1, H=20, W=20, OC=40, k=7, pad=3, ndim=3, dtype="bf16", cl=True),
    L("stride3_odd", C=32, H=31, W=29, OC=48, k=3, pad=0, stride=3, dtype="f16"),
    L("wide_image_f16", C=64, H=2, W=1920, OC=64, dtype="f16"),
    L("many_images_cl_f16", N=200, C=32, H=6, W=6, OC=64, dtype="f16", cl=True),
    L("c3_oc4_stem_f16", C=3, H=100, W=100, OC=4, dtype="f16"),
]


@pytest.mark.parametrize("L", CASES, ids=[c.name for c in CASES])
def test_edge_shape(L):
    check(L)
