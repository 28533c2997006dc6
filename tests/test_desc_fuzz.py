"""Seeded fuzzing of descriptor validation, host only (no GPU, no CUDA call).

Every field of `gbconv_desc` is drawn from a mix of valid values, boundary
values (0, 1, the limits and one past them) and wild ones (negative, 2^31 - 1),
and each descriptor goes through the host-only queries. The library must
answer every one with a status code, never crash, and answer consistently:
- the status of `select_algo`, `workspace_size`, `output_shape` and
  `weight_packed_size` is the same;
- an accepted descriptor has positive output extents within the limits, a
  resolved algorithm (never AUTO), and its output element count within
  GBCONV_MAX_ELEMS;
- an accepted descriptor stays accepted when its algorithm is forced to the
  one AUTO chose.
"""
import numpy as np
import pytest

import implicit_gemm_convolution_conv_gb300 as gb

MAX_DIM, MAX_K, MAX_STRIDE, MAX_ELEMS = 65535, 16, 8, 1 << 36
FAKE = 1 << 44            # a 256-byte-aligned address; never dereferenced


def _pick(rng, valid, extra):
    # mostly a valid value; now and then a boundary or wild one, so that a
    # draw holds zero, one or a few bad fields
    if rng.random() < 0.96:
        return int(rng.choice(valid))
    return int(rng.choice(extra))


def _draw(rng):
    dim_extra = [0, -1, MAX_DIM, MAX_DIM + 1, 2**31 - 1, -2**31]
    ndim = int(rng.choice([2, 3, 1, 4]) if rng.random() < 0.05 else rng.choice([2, 3]))
    f = dict(
        N=_pick(rng, [1, 2, 3, 16, 4096], dim_extra),
        C=_pick(rng, [1, 3, 8, 64, 256, 4096], dim_extra),
        D=_pick(rng, [1, 1, 3, 5, 64], dim_extra) if ndim == 3 else _pick(rng, [1], [0, 2]),
        H=_pick(rng, [1, 7, 32, 640, 4096], dim_extra),
        W=_pick(rng, [1, 9, 32, 640, 4096], dim_extra),
        OC=_pick(rng, [1, 8, 32, 128, 300], dim_extra),
        k=_pick(rng, [1, 3, 5, 7], [0, MAX_K, MAX_K + 1, -3]),
        pad=_pick(rng, [0, 1, 2], [-1, MAX_K, MAX_K + 1]),
        stride=_pick(rng, [1, 2, 3], [0, MAX_STRIDE, MAX_STRIDE + 1, -2]),
        dtype=_pick(rng, [gb.F32, gb.F16, gb.BF16], [3, -1]),
        act=_pick(rng, [gb.ACT_NONE, gb.ACT_RELU], [2, -5]),
        w_layout=_pick(rng, [gb.W_OIHW, gb.W_PACKED], [2]),
        algo=_pick(rng, [gb.ALGO_AUTO, gb.ALGO_AUTO, gb.ALGO_DIRECT, gb.ALGO_IGEMM_FFMA,
                         gb.ALGO_IGEMM_TC, gb.ALGO_DIRECT_TC], [5, -1]),
        flags=_pick(rng, [0, 0, 1, 2, 4, 8, 9], [3, 16, 1 << 30, -1]),
    )
    return ndim, f


def _desc(f):
    d = gb.make_desc(f["N"], f["C"], f["H"], f["W"], f["OC"], f["k"], f["pad"], f["stride"],
                     D=f["D"], dtype=f["dtype"], act=f["act"], w_layout=f["w_layout"],
                     algo=f["algo"])
    d.flags = f["flags"]
    return d


@pytest.mark.parametrize("seed", range(8))
def test_fuzzed_descriptors_get_consistent_answers(seed):
    rng = np.random.Generator(np.random.PCG64(1000 + seed))
    accepted = 0
    for _ in range(500):
        ndim, f = _draw(rng)
        d = _desc(f)
        st_a, algo = gb.select_algo(d, ndim)
        st_w, ws = gb.workspace_size(d, ndim)
        st_o, (od, oh, ow) = gb.output_shape(d, ndim)
        st_p, packed = gb.weight_packed_size(d, ndim)
        assert st_a == st_w == st_o == st_p, (ndim, f, st_a, st_w, st_o, st_p)
        if st_a != gb.OK:
            # the forward call rejects it the same way, before any CUDA call
            # (fake, aligned, non-overlapping pointers; nothing is read)
            if ndim in (2, 3):
                fwd = gb.conv3d_fwd if ndim == 3 else gb.conv2d_fwd
                assert fwd(d, FAKE, FAKE + (1 << 40), None, FAKE + (2 << 40), 0) == st_a, (ndim, f)
            continue
        accepted += 1
        assert algo != gb.ALGO_AUTO and algo in (gb.ALGO_DIRECT, gb.ALGO_IGEMM_FFMA,
                                                 gb.ALGO_IGEMM_TC, gb.ALGO_DIRECT_TC)
        assert 1 <= oh <= MAX_DIM + 2 * MAX_K and 1 <= ow <= MAX_DIM + 2 * MAX_K and od >= 1
        assert ws >= 0 and packed > 0
        assert f["N"] * f["OC"] * od * oh * ow <= MAX_ELEMS
        assert f["N"] * f["C"] * f["D"] * f["H"] * f["W"] <= MAX_ELEMS
        forced = _desc(dict(f, algo=algo))
        assert gb.select_algo(forced, ndim) == (gb.OK, algo), (ndim, f, algo)
    assert accepted > 40          # the draw mixes enough valid descriptors
