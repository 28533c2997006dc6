"""BatchNorm folded into the convolution (lpnh.cn/news/2745477 section 3.1).

CPU: the oracle's fold is pinned to the BatchNorm definition applied after the
oracle's conv (a different formulation of the same result) and to the
identity BatchNorm. GPU: gbconv_fold_batchnorm against the fp64 fold, and a
forward call with the folded parameters against the oracle conv with the same
parameters.
"""
import numpy as np
import pytest

import oracle
import implicit_gemm_convolution_conv_gb300 as gb

FAKE = 1 << 20


def _bn_params(r, OC):
    gamma = r.uniform(0.5, 2.0, OC)
    beta = r.uniform(-0.5, 0.5, OC)
    mean = r.uniform(-0.3, 0.3, OC)
    var = r.uniform(0.1, 3.0, OC)
    return gamma, beta, mean, var


@pytest.mark.parametrize("ndim,relu", [(2, False), (3, False), (2, True)])
def test_fold_equals_batchnorm_after_conv(ndim, relu):
    """conv(x, w', b') = BN(conv(x, w, b)) (ReLU, when set, after both)."""
    r = np.random.Generator(np.random.PCG64(41 + ndim))
    x = r.standard_normal((2, 3) + (5,) * ndim)
    w = r.standard_normal((4, 3) + (3,) * ndim)
    b = r.standard_normal(4)
    g, bt, m, v = _bn_params(r, 4)
    eps = 1e-5
    wf, bf = oracle.fold_batchnorm(w, b, g, bt, m, v, eps)
    y = oracle.conv(x, wf, bf, stride=1, pad=1, relu=relu)
    ref = oracle.batchnorm(oracle.conv(x, w, b, stride=1, pad=1), g, bt, m, v, eps)
    if relu:
        ref = np.maximum(ref, 0.0)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_fold_without_bias_and_identity_batchnorm():
    r = np.random.Generator(np.random.PCG64(43))
    w = r.standard_normal((3, 2, 3, 3))
    var = r.uniform(0.2, 2.0, 3)
    mean = r.uniform(-1, 1, 3)
    eps = 1e-3
    # gamma = sqrt(var + eps), beta = mean: BN is the identity
    wf, bf = oracle.fold_batchnorm(w, None, np.sqrt(var + eps), mean, mean, var, eps)
    np.testing.assert_allclose(wf, w, rtol=1e-15)
    np.testing.assert_allclose(bf, np.zeros(3), atol=1e-15)


def test_fold_validation_without_gpu():
    d = gb.make_desc(1, 3, 8, 8, 4, 3, 1, 1)
    f = FAKE
    assert gb.fold_batchnorm(d, 2, 0, 0, f, f * 2, f * 3, f * 4, 1e-5, f * 5, f * 6, 0) == gb.ERR_NULL
    assert gb.fold_batchnorm(d, 2, f, 0, f * 2, f * 3, f * 4, f * 5, -1.0, f * 6, f * 7, 0) == gb.ERR_SHAPE
    assert gb.fold_batchnorm(d, 2, f + 2, 0, f * 2, f * 3, f * 4, f * 5, 1e-5, f * 6, f * 7, 0) == gb.ERR_ALIGN
    bad = gb.make_desc(1, 3, 8, 8, 4, 3, 1, 1, act=5)
    assert gb.fold_batchnorm(bad, 2, f, 0, f * 2, f * 3, f * 4, f * 5, 1e-5, f * 6, f * 7, 0) == gb.ERR_ACT


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,inplace", [("f32", False), ("f16", False), ("bf16", True), ("f32", True)])
def test_fold_on_gpu(dtype, inplace):
    import torch
    import synthetic
    from implicit_gemm_convolution_conv_gb300.torch_ops import Conv, to_device, to_numpy
    from gpu_helpers import assert_close
    L = synthetic.Layer("bn", N=2, C=24, H=12, W=20, OC=40, k=3, pad=1, stride=1, dtype=dtype,
                        relu=True, x_dist="n01", w_dist="he", b_dist="u11", seed=44)
    inp = synthetic.make_inputs(L)
    r = np.random.Generator(np.random.PCG64(45))
    g, bt, m, v = (a.astype(np.float32) for a in _bn_params(r, L.OC))
    eps = 1e-5
    x, w = to_device(inp.x, dtype), to_device(inp.w, dtype)
    b = torch.from_numpy(inp.b).cuda()
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    gd, btd, md, vd = dev(g), dev(bt), dev(m), dev(v)
    w_out = w if inplace else torch.empty_like(w)
    b_out = b if inplace else torch.empty_like(b)
    w_in, b_in = (w.clone(), b.clone()) if inplace else (w, b)
    d = gb.make_desc(L.N, L.C, L.H, L.W, L.OC, L.k, L.pad, L.stride, dtype=dtype)
    assert gb.fold_batchnorm(d, 2, w_out if inplace else w, b_out if inplace else b, gd, btd, md, vd,
                             eps, w_out, b_out) == gb.OK
    torch.cuda.synchronize()
    # the fold itself against fp64 (scale formed in fp32, product rounded to storage)
    wf, bf = oracle.fold_batchnorm(oracle.widen(inp.w, dtype), inp.b, g, bt, m, v, eps)
    got_w = oracle.widen(to_numpy(w_out), dtype)
    # relative: a few ulp of the storage type; absolute: one subnormal step
    ulp = {"f32": 2.0 ** -21, "f16": 2.0 ** -10, "bf16": 2.0 ** -7}[dtype]
    sub = {"f32": 2.0 ** -149, "f16": 2.0 ** -24, "bf16": 2.0 ** -133}[dtype]
    assert np.all(np.abs(got_w - wf) <= ulp * np.abs(wf) + sub)
    np.testing.assert_allclose(b_out.cpu().numpy(), bf, rtol=2e-6, atol=1e-6)
    # a forward call with the folded parameters = the oracle conv with them
    y = Conv(x, w_out, b_out, L.stride, L.pad, L.relu)()
    torch.cuda.synchronize()
    ref = oracle.conv(inp.x, to_numpy(w_out), b_out.cpu().numpy(), L.stride, L.pad, L.relu, dtype)
    assert_close(dtype, oracle.widen(to_numpy(y), dtype), ref, "bn-folded conv")
    if inplace:
        assert not torch.equal(w_in, w_out)
