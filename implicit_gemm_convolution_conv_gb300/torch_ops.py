"""Torch-tensor front end of the C ABI: allocation and argument marshalling.

PyTorch provides device memory and the stream; `forward` allocates the output
and the workspace the library asks for, then calls gbconv_conv2d_fwd /
gbconv_conv3d_fwd. No arithmetic happens here.
"""
import copy

import numpy as np
import torch

from . import (ACT_NONE, ACT_RELU, ALGO_AUTO, BF16, F16, F32,
               FLAG_CHANNELS_LAST, W_OIHW, W_PACKED, GbconvError, check,
               conv2d_fwd, conv3d_fwd,
               make_desc, output_shape, select_algo, weight_pack,
               weight_packed_size, workspace_size)

TORCH_DTYPE = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}
CODE_OF = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}


def to_device(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """numpy storage array -> torch tensor on `device` (bf16 from uint16 bits)."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
        return t.view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_numpy(t: torch.Tensor) -> np.ndarray:
    """torch tensor -> numpy storage array (bf16 as uint16 bits)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _desc(x, OC, k, stride, pad, relu, algo, w_layout, tpad=0, pool=False,
          channels_last=False):
    nsp = x.dim() - 2
    if channels_last:
        # x is [N, H, W, C] or [N, D, H, W, C]
        N, C = x.shape[0], x.shape[-1]
        D, H, W = (1,) + tuple(x.shape[1:3]) if nsp == 2 else tuple(x.shape[1:4])
    elif nsp == 2:
        N, C, H, W = x.shape
        D = 1
    else:
        N, C, D, H, W = x.shape
    d = make_desc(N, C, H, W, OC, k=k, pad=pad, stride=stride, D=D,
                  dtype=CODE_OF[x.dtype], act=ACT_RELU if relu else ACT_NONE,
                  w_layout=w_layout, algo=algo, tpad=tpad, pool=pool,
                  channels_last=channels_last)
    return d, nsp


def check_tensors(x, w, b=None, channels_last=False, require_cuda=True):
    """The checks a raw-pointer ABI cannot make: x, w and b are contiguous
    tensors on one CUDA device, w has x's dtype and the shape [OC, C, k, k]
    (conv2d) or [OC, C, k, k, k] (conv3d) with C = x's channels, and b is
    fp32 with OC elements. Raises TypeError or ValueError; returns (OC, k)."""
    for name, t in (("x", x), ("w", w)) + ((("b", b),) if b is not None else ()):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if require_cuda and not t.is_cuda:
            raise ValueError(f"{name} must be on a CUDA device (there is no CPU path)")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device != x.device:
            raise ValueError(f"{name} is on {t.device}, x on {x.device}")
    if x.dtype not in CODE_OF:
        raise ValueError(f"x has dtype {x.dtype}; float32, float16 or bfloat16 expected")
    if x.dim() not in (4, 5):
        raise ValueError("x must be 4-D (conv2d) or 5-D (conv3d)")
    if w.dtype != x.dtype:
        raise ValueError(f"w has dtype {w.dtype}, x {x.dtype}")
    C = x.shape[-1] if channels_last else x.shape[1]
    nsp = x.dim() - 2
    if w.dim() != x.dim() or w.shape[1] != C or len(set(w.shape[2:])) != 1:
        raise ValueError(f"w has shape {tuple(w.shape)}; [OC, {C}] + {nsp} equal kernel sizes expected")
    OC, k = w.shape[0], w.shape[-1]
    if b is not None and (b.dtype != torch.float32 or b.numel() != OC):
        raise ValueError(f"b must be float32 with {OC} elements")
    return OC, k


def y_shape(desc, ndim):
    """y's shape for this desc, from gbconv_output_shape (frame padding,
    fused pool and channels-last included), not from a formula restated
    here."""
    st, (od, oh, ow) = output_shape(desc, ndim)
    check(st)
    sp = [oh, ow] if ndim == 2 else [od, oh, ow]
    if desc.flags & FLAG_CHANNELS_LAST:
        return [desc.N] + sp + [desc.OC]
    return [desc.N, desc.OC] + sp


def output_tensor(desc, ndim, x):
    """An uninitialised y for this desc, with x's dtype, on x's device."""
    return torch.empty(y_shape(desc, ndim), dtype=x.dtype, device=x.device)


class Conv:
    """A prepared convolution: descriptor, output and workspace allocated once.

    `w` is OIHW/OIDHW; with `prepack=True` it is packed once with
    gbconv_weight_pack and later calls pass w_layout PACKED. With
    `channels_last=True`, x is [N, (D,) H, W, C] and y [N, (OD,) OH, OW, OC].
    """

    def __init__(self, x, w, b=None, stride=1, pad=0, relu=False,
                 algo=ALGO_AUTO, prepack=False, out=None, workspace=None, tpad=0,
                 pool=False, channels_last=False):
        OC, k = check_tensors(x, w, b, channels_last)
        self.x, self.b = x, b
        layout = W_PACKED if prepack else W_OIHW
        self.channels_last = channels_last
        self.desc, self.nsp = _desc(x, OC, k, stride, pad, relu, algo, layout, tpad, pool,
                                    channels_last)
        st, self.algo = select_algo(self.desc, self.nsp)
        check(st)
        if prepack:
            st, nb = weight_packed_size(self.desc, self.nsp)
            check(st)
            self.w = torch.empty(nb + 256, dtype=torch.uint8, device=x.device)
            self.w = _aligned_view(self.w, nb)
            check(weight_pack(self.desc, self.nsp, w, self.w))
        else:
            self.w = w
        st, ws = workspace_size(self.desc, self.nsp)
        check(st)
        self.workspace_bytes = ws
        if ws:
            if workspace is None:
                raw = torch.empty(ws + 256, dtype=torch.uint8, device=x.device)
                workspace = _aligned_view(raw, ws)
            elif not (workspace.is_contiguous() and workspace.device == x.device):
                raise ValueError("workspace must be a contiguous tensor on x's device")
            self.desc.workspace = workspace.data_ptr()
            # the tensor's real size: the library refuses one that is too small
            self.desc.workspace_bytes = workspace.numel() * workspace.element_size()
        self.workspace = workspace
        shape = y_shape(self.desc, self.nsp)
        if out is None:
            out = torch.empty(shape, dtype=x.dtype, device=x.device)
        elif (list(out.shape) != shape or out.dtype != x.dtype or out.device != x.device or
              not out.is_contiguous()):
            raise ValueError(f"out must be a contiguous {x.dtype} tensor of shape {shape} on {x.device}")
        self.y = out
        self._fn = conv2d_fwd if self.nsp == 2 else conv3d_fwd

    def with_input(self, x):
        """The same prepared call (descriptor, weights, workspace) on another
        input tensor of the same shape, writing a new output tensor."""
        c = copy.copy(self)
        c.x = x
        c.y = torch.empty_like(self.y)
        return c

    def __call__(self, x=None, stream=None):
        if x is not None and (x.shape != self.x.shape or x.dtype != self.x.dtype or
                              x.device != self.x.device or not x.is_contiguous()):
            raise ValueError("x must match the prepared input's shape, dtype and device, contiguous")
        st = self._fn(self.desc, self.x if x is None else x, self.w, self.b,
                      self.y, stream)
        if st != 0:
            raise GbconvError(st)
        return self.y


def _aligned_view(raw: torch.Tensor, nbytes: int) -> torch.Tensor:
    off = (-raw.data_ptr()) % 256
    return raw[off:off + nbytes]


def forward(x, w, b=None, stride=1, pad=0, relu=False, algo=ALGO_AUTO,
            prepack=False, tpad=0, pool=False, channels_last=False):
    """One convolution call; returns y (allocated here)."""
    return Conv(x, w, b, stride, pad, relu, algo, prepack, tpad=tpad, pool=pool,
                channels_last=channels_last)()
