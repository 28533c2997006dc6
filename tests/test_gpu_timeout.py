"""Bounded device waits: a wait that runs out is reported, not a hang or a crash.

githubissues.com/ysh329/OpenCL-101/52 ("init fault tolerance") asks a GPU
backend to report a failure through its API instead of crashing. The
tensor-core kernels bound every mbarrier wait by the SM cycle counter; when a
wait runs out, the kernel raises an abort flag that the CTA's other roles
see, stops issuing copies and MMAs, lets those already issued land (their
drain has a fixed bound of its own, independent of the limit set here),
frees its TMEM and returns, and gbconv_check_device_error reports
GBCONV_ERR_TIMEOUT.

Nothing here injects a fault or skips an arrive: the only lever is a wait
limit far below the time the work takes. The GEMM case is one tile whose
K loop (4096 channels x 9 taps) takes tens of microseconds, so the
epilogue's wait for its accumulator cannot finish within 1 us. After each
case the default limit is restored and an ordinary call must match the
oracle, i.e. the context and the library state stay usable.
"""
import pytest
import torch

import oracle
import synthetic
import implicit_gemm_convolution_conv_gb300 as gb
from implicit_gemm_convolution_conv_gb300.torch_ops import to_numpy
from gpu_helpers import assert_close, reference, run

pytestmark = pytest.mark.gpu

DEFAULT_LIMIT_NS = 2_000_000_000


@pytest.fixture(autouse=True)
def _restore_limit():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    assert gb.check_device_error() == gb.OK
    yield
    assert gb.set_wait_limit_ns(DEFAULT_LIMIT_NS) == gb.OK
    torch.cuda.synchronize()
    gb.check_device_error()


def _usable_afterwards():
    """The default limit back in place, an ordinary tensor-core call and a
    tensor-core stem call match the oracle and report no error."""
    assert gb.set_wait_limit_ns(DEFAULT_LIMIT_NS) == gb.OK
    L = synthetic.Layer("after_timeout_tc", N=1, C=64, H=16, W=40, OC=64, k=3, pad=1,
                        stride=1, dtype="f16", relu=True, x_dist="n01", w_dist="he",
                        b_dist="u005", seed=11)
    inp = synthetic.make_inputs(L)
    y, conv = run(inp, algo=gb.ALGO_IGEMM_TC)
    assert conv.algo == gb.ALGO_IGEMM_TC
    assert_close(L.dtype, y, reference(inp), L.name)
    S = synthetic.layer(2, H=64, W=96)
    inp = synthetic.make_inputs(S)
    y, conv = run(inp, algo=gb.ALGO_DIRECT_TC)
    assert_close(S.dtype, y, reference(inp), S.name)
    assert gb.check_device_error() == gb.OK


def test_gemm_wait_runs_out_and_is_reported():
    L = synthetic.Layer("long_k_single_tile", N=1, C=4096, H=4, W=64, OC=128, k=3, pad=1,
                        stride=1, dtype="f16", x_dist="n01", w_dist="he", b_dist="u005",
                        seed=12)
    inp = synthetic.make_inputs(L)
    # a full-limit call first: the same problem completes and is correct
    y, conv = run(inp, algo=gb.ALGO_IGEMM_TC)
    assert conv.algo == gb.ALGO_IGEMM_TC
    assert gb.check_device_error() == gb.OK
    assert_close(L.dtype, y, reference(inp), L.name)
    # 1 us: the epilogue's wait for the tile's accumulator runs out
    assert gb.set_wait_limit_ns(1000) == gb.OK
    conv()
    assert gb.check_device_error() == gb.ERR_TIMEOUT
    # the error word was cleared by the read
    assert gb.check_device_error() == gb.OK
    _usable_afterwards()


@pytest.mark.parametrize("limit_ns", [1, 200])
def test_short_limits_on_every_tensor_core_kernel_leave_the_context_usable(limit_ns):
    """Limits of 1 ns and 200 ns on the stem and the GEMM (16-bit and fp32,
    one and several tiles per CTA): each call either completes or reports
    GBCONV_ERR_TIMEOUT; either way the process carries on and later calls
    are correct."""
    layers = [
        (gb.ALGO_DIRECT_TC, synthetic.layer(2)),
        (gb.ALGO_DIRECT_TC, synthetic.Layer("stem_plain_loads", N=2, C=3, H=64, W=638, OC=32, k=3,
                                            pad=1, stride=2, dtype="f32", relu=True, x_dist="u01",
                                            w_dist="he", b_dist="u01_1", seed=13)),
        (gb.ALGO_IGEMM_TC, synthetic.layer(4)),
        (gb.ALGO_IGEMM_TC, synthetic.layer(3)),
        (gb.ALGO_IGEMM_TC, synthetic.Layer("many_tiles", N=16, C=64, H=40, W=64, OC=64, k=3, pad=1,
                                           stride=1, dtype="f16", x_dist="n01", w_dist="he",
                                           b_dist="u005", seed=14)),
    ]
    for algo, L in layers:
        inp = synthetic.make_inputs(L)
        _, conv = run(inp, algo=algo)
        assert conv.algo == algo
        assert gb.check_device_error() == gb.OK
        assert gb.set_wait_limit_ns(limit_ns) == gb.OK
        for _ in range(5):
            conv()
        st = gb.check_device_error()
        assert st in (gb.OK, gb.ERR_TIMEOUT), gb.status_string(st)
        assert gb.set_wait_limit_ns(DEFAULT_LIMIT_NS) == gb.OK
        # the same prepared call with the default limit is correct again
        y = conv()
        torch.cuda.synchronize()
        assert gb.check_device_error() == gb.OK
        assert_close(L.dtype, oracle.widen(to_numpy(y), L.dtype), reference(inp), L.name)
    _usable_afterwards()
