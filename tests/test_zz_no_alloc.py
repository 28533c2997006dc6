"""gbconv_conv_fwd_noalloc: the entry point for callers that cannot allocate.

Some callers cannot call cudaMalloc: code that runs while a stream is being
captured into a CUDA graph, loops that must never enter the allocator, and C
hosts without a caching allocator that do not want to manage a workspace.
This entry point takes no workspace; the scratch it needs (the packed
weights of the CUDA-core implicit-GEMM path) lives in a fixed array inside
the library.

The GPU test calls it through the C ABI on several layers in a row (fp32
conv2d NCHW, f16 conv3d, bf16 conv2d channels-last) and checks each output
against the fp64 oracle and against the regular entry point
(gbconv_conv2d_fwd / gbconv_conv3d_fwd, same kernel family, caller-provided
workspace), both within the tolerances of the parity tests; a last call
repeats the first and must reproduce it exactly, so nothing left in the
shared array by the calls in between leaks into the next one. This file is
collected last.
"""
import numpy as np
import pytest

import synthetic
import implicit_gemm_convolution_conv_gb300 as gb


def _desc(L, **kw):
    kw.setdefault("act", gb.ACT_RELU if L.relu else gb.ACT_NONE)
    return gb.make_desc(L.N, L.C, L.H, L.W, L.OC, L.k, L.pad, L.stride, D=L.D,
                        dtype=L.dtype, tpad=L.tpad, channels_last=L.cl, **kw)


def test_noalloc_rejects_what_it_cannot_hold():
    """Host-side checks, no GPU needed: too-large scratch, wrong algorithm,
    weight layout or activation, the fused pool, all rejected before any CUDA
    call."""
    big = synthetic.Layer("big", N=1, C=1024, H=8, W=8, OC=1024, k=3, pad=1,
                          stride=1)
    fake = 1 << 20
    assert 9 * 1024 * 1024 * 4 > gb.NOALLOC_SCRATCH_BYTES
    assert gb.conv_fwd_noalloc(_desc(big), 2, fake, fake * 64, None,
                               fake * 256, 0) == gb.ERR_TOO_LARGE
    L = synthetic.LAYERS[3]
    assert gb.conv_fwd_noalloc(_desc(L, algo=gb.ALGO_IGEMM_TC), 2, fake,
                               fake * 4, None, fake * 16, 0) == gb.ERR_ALGO
    assert gb.conv_fwd_noalloc(_desc(L, w_layout=gb.W_PACKED), 2, fake,
                               fake * 4, None, fake * 16, 0) == gb.ERR_LAYOUT
    assert gb.conv_fwd_noalloc(_desc(L, act=7), 2, fake, fake * 4, None,
                               fake * 16, 0) == gb.ERR_ACT
    # the fused max pool exists only in the direct kernel
    stem = synthetic.LAYERS[2]
    assert gb.conv_fwd_noalloc(_desc(stem, pool=True), 2, fake, fake * 4, None,
                               fake * 16, 0) == gb.ERR_ALGO


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_regular_entry_point_on_calls_in_a_row():
    import torch
    from gpu_helpers import assert_close, reference
    from implicit_gemm_convolution_conv_gb300.torch_ops import (Conv,
                                                                output_tensor,
                                                                to_device,
                                                                to_numpy)
    import oracle

    layers = [
        synthetic.LAYERS[3],                                   # conv2d fp32 NCHW
        synthetic.Layer("noalloc_3d_f16", N=1, C=24, D=5, H=12, W=20, OC=40,
                        k=3, pad=1, stride=1, dtype="f16", relu=True, ndim=3,
                        x_dist="n01", w_dist="he", b_dist="u005", seed=77,
                        tpad=gb.TPAD_CAUSAL),
        synthetic.Layer("noalloc_2d_bf16_channels_last", N=2, C=20, H=13, W=30,
                        OC=36, k=3, pad=1, stride=2, dtype="bf16", relu=True,
                        x_dist="n01", w_dist="he", b_dist="u005", seed=78,
                        cl=True),
    ]
    outs = []
    for L in layers + layers[:1]:
        inp = synthetic.make_inputs(L)
        x_host = np.ascontiguousarray(np.moveaxis(inp.x, 1, -1)) if L.cl else inp.x
        x = to_device(x_host, L.dtype)
        w = to_device(inp.w, L.dtype)
        b = torch.from_numpy(inp.b).cuda()
        d = _desc(L)
        y = output_tensor(d, L.ndim, x)
        st = gb.conv_fwd_noalloc(d, L.ndim, x, w, b, y)
        assert st == gb.OK, gb.status_string(st)
        regular = Conv(x, w, b, L.stride, L.pad, L.relu, algo=gb.ALGO_IGEMM_FFMA,
                       tpad=L.tpad, channels_last=L.cl)()
        torch.cuda.synchronize()
        got = oracle.widen(to_numpy(y), L.dtype)
        exp = oracle.widen(to_numpy(regular), L.dtype)
        if L.cl:
            got, exp = np.moveaxis(got, -1, 1), np.moveaxis(exp, -1, 1)
        assert_close(L.dtype, got, reference(inp), f"noalloc vs oracle, {L.name}")
        assert_close(L.dtype, got, exp, f"noalloc vs regular, {L.name}")
        outs.append(got)
    np.testing.assert_array_equal(outs[0], outs[-1])
    assert gb.check_device_error() == gb.OK
