"""Torch-facing API over libfkl.so: the loss's forward and backward, both in one
call, the KL + cross-entropy mixture, the teacher top-K cache producer and the
autograd loss.

Every step of the loss runs in the library's CUDA kernels; this module only
checks tensor properties, allocates outputs and the workspace with torch, and
passes raw pointers plus the current CUDA stream.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _lib

STATUS_NAMES = {0: "FKL_OK", 1: "FKL_ERR_INVALID_ARG", 2: "FKL_ERR_WORKSPACE", 3: "FKL_ERR_INDEX",
                4: "FKL_ERR_CUDA", 5: "FKL_ERR_UNSUPPORTED", 6: "FKL_ERR_TIMEOUT"}


class FKLError(RuntimeError):
    def __init__(self, status: int, where: str):
        L = _lib.lib()
        msg = L.fkl_last_error().decode()
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({L.fkl_status_string(status).decode()}){': ' + msg if msg else ''}")
        self.status = status


def _check(st: int, where: str):
    if st != 0:
        raise FKLError(st, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _expect(t, name, dtype, ndim, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _expect_out(t, name, dtype, shape, device):
    """A caller-supplied output: its dtype, shape, device and layout as the library writes it."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    _expect(t, name, dtype, len(shape), device)


def _ws_bytes(ws, device) -> int:
    """Byte size of a caller-supplied workspace (any dtype), which must be contiguous device memory on h's device."""
    if not isinstance(ws, torch.Tensor):
        raise TypeError("ws must be a torch.Tensor")
    if not ws.is_cuda:
        raise ValueError("ws must be a CUDA tensor")
    if ws.device != device:
        raise ValueError(f"ws is on {ws.device}, expected {device}")
    if not ws.is_contiguous():
        raise ValueError("ws must be contiguous")
    return ws.numel() * ws.element_size()


def workspace_size(N: int, d: int, V: int, K: int, chunk: int = 0) -> int:
    n = _lib.lib().fkl_workspace_size(int(N), int(d), int(V), int(K), int(chunk))
    if n == 0:
        raise ValueError(f"invalid sizes N={N} d={d} V={V} K={K} chunk={chunk}")
    return int(n)


def alloc_workspace(N, d, V, K, chunk=0, device="cuda") -> torch.Tensor:
    return torch.empty(workspace_size(N, d, V, K, chunk), dtype=torch.uint8, device=device)


def _inputs(h, W, idx, tlogit, mask):
    _expect(h, "h", torch.bfloat16, 2)
    dev = h.device
    _expect(W, "W", torch.bfloat16, 2, dev)
    _expect(idx, "idx", torch.int32, 2, dev)
    _expect(tlogit, "tlogit", torch.float32, 2, dev)
    if mask is not None:
        _expect(mask, "mask", torch.uint8, 1, dev)
    N, d = h.shape
    V, d2 = W.shape
    if d2 != d:
        raise ValueError(f"h is [N,{d}] but W is [V,{d2}]")
    if idx.shape != tlogit.shape or idx.shape[0] != N:
        raise ValueError("idx and tlogit must both be [N,K]")
    if mask is not None and mask.shape[0] != N:
        raise ValueError("mask must be [N]")
    return N, d, V, idx.shape[1], dev


def _grad_scalar(g, device):
    """The upstream gradient as the library reads it: one fp32 value in device memory (or None = 1)."""
    if g is None:
        return None
    if not isinstance(g, torch.Tensor) or g.numel() != 1:
        raise ValueError("grad_loss must be a one-element tensor")
    g = g.reshape(1)
    _expect(g, "grad_loss", torch.float32, 1, device)
    return g


def _grad_outputs(dh, dW, N, d, V, device):
    if dh is None:
        dh = torch.empty((N, d), dtype=torch.bfloat16, device=device)
    _expect_out(dh, "dh", torch.bfloat16, (N, d), device)
    if dW is None:
        dW = torch.empty((V, d), dtype=torch.float32, device=device)
    _expect_out(dW, "dW", torch.float32, (V, d), device)
    return dh, dW


def forward(h, W, idx, tlogit, mask=None, T: float = 1.0, chunk: int = 0,
            ws: Optional[torch.Tensor] = None, loss: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Fused forward: returns (loss [1] fp32, lse [N] fp32) on h's device."""
    N, d, V, K, dev = _inputs(h, W, idx, tlogit, mask)
    if ws is None:
        ws = alloc_workspace(N, d, V, K, chunk, dev)
    ws_bytes = _ws_bytes(ws, dev)
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=dev)
    _expect_out(loss, "loss", torch.float32, (1,), dev)
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    _expect_out(lse, "lse", torch.float32, (N,), dev)
    with torch.cuda.device(dev):  # the library launches on the current device
        st = _lib.lib().fkl_forward(_ptr(h), _ptr(W), _ptr(idx), _ptr(tlogit), _ptr(mask), N, d, V, K,
                                    float(T), int(chunk), _ptr(loss), _ptr(lse), _ptr(ws), ws_bytes,
                                    _stream(dev))
    _check(st, "fkl_forward")
    return loss, lse


def backward(h, W, idx, tlogit, mask, T: float, lse: torch.Tensor,
             grad_loss: Optional[torch.Tensor] = None, chunk: int = 0,
             ws: Optional[torch.Tensor] = None, dh: Optional[torch.Tensor] = None,
             dW: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Fused backward: returns (dh [N,d] bf16, dW [V,d] fp32)."""
    N, d, V, K, dev = _inputs(h, W, idx, tlogit, mask)
    _expect_out(lse, "lse", torch.float32, (N,), dev)
    grad_loss = _grad_scalar(grad_loss, dev)
    if ws is None:
        ws = alloc_workspace(N, d, V, K, chunk, dev)
    ws_bytes = _ws_bytes(ws, dev)
    dh, dW = _grad_outputs(dh, dW, N, d, V, dev)
    with torch.cuda.device(dev):  # the library launches on the current device
        st = _lib.lib().fkl_backward(_ptr(h), _ptr(W), _ptr(idx), _ptr(tlogit), _ptr(mask), N, d, V, K,
                                     float(T), int(chunk), _ptr(lse), _ptr(grad_loss), _ptr(dh),
                                     _ptr(dW), _ptr(ws), ws_bytes, _stream(dev))
    _check(st, "fkl_backward")
    return dh, dW


def mix_forward(h, W, idx, tlogit, mask, label, T: float, alpha: float, chunk: int = 0,
                ws: Optional[torch.Tensor] = None):
    """KL + hard-label CE mixture, forward: (loss [1], lse [N], lse1 [N]) fp32."""
    N, d, V, K, dev = _inputs(h, W, idx, tlogit, mask)
    _expect_out(label, "label", torch.int32, (N,), dev)
    if ws is None:
        ws = alloc_workspace(N, d, V, K, chunk, dev)
    ws_bytes = _ws_bytes(ws, dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    lse1 = torch.empty(N, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):  # the library launches on the current device
        st = _lib.lib().fkl_mix_forward(_ptr(h), _ptr(W), _ptr(idx), _ptr(tlogit), _ptr(mask), _ptr(label), N, d, V,
                                        K, float(T), float(alpha), int(chunk), _ptr(loss), _ptr(lse), _ptr(lse1),
                                        _ptr(ws), ws_bytes, _stream(dev))
    _check(st, "fkl_mix_forward")
    return loss, lse, lse1


def mix_backward(h, W, idx, tlogit, mask, label, T: float, alpha: float, lse, lse1,
                 grad_loss: Optional[torch.Tensor] = None, chunk: int = 0, ws: Optional[torch.Tensor] = None):
    """KL + hard-label CE mixture, backward: (dh [N,d] bf16, dW [V,d] fp32)."""
    N, d, V, K, dev = _inputs(h, W, idx, tlogit, mask)
    _expect_out(label, "label", torch.int32, (N,), dev)
    _expect_out(lse, "lse", torch.float32, (N,), dev)
    _expect_out(lse1, "lse1", torch.float32, (N,), dev)
    grad_loss = _grad_scalar(grad_loss, dev)
    if ws is None:
        ws = alloc_workspace(N, d, V, K, chunk, dev)
    ws_bytes = _ws_bytes(ws, dev)
    dh, dW = _grad_outputs(None, None, N, d, V, dev)
    with torch.cuda.device(dev):  # the library launches on the current device
        st = _lib.lib().fkl_mix_backward(_ptr(h), _ptr(W), _ptr(idx), _ptr(tlogit), _ptr(mask), _ptr(label), N, d,
                                         V, K, float(T), float(alpha), int(chunk), _ptr(lse), _ptr(lse1),
                                         _ptr(grad_loss), _ptr(dh), _ptr(dW), _ptr(ws), ws_bytes, _stream(dev))
    _check(st, "fkl_mix_backward")
    return dh, dW


def forward_backward(h, W, idx, tlogit, mask, T: float, grad_loss: Optional[torch.Tensor] = None,
                     chunk: int = 0, ws: Optional[torch.Tensor] = None, loss: Optional[torch.Tensor] = None,
                     lse: Optional[torch.Tensor] = None, dh: Optional[torch.Tensor] = None,
                     dW: Optional[torch.Tensor] = None):
    """Loss and gradients in one call (logits kept per chunk, no recompute).

    Returns (loss [1] fp32, lse [N] fp32, dh [N,d] bf16, dW [V,d] fp32)."""
    N, d, V, K, dev = _inputs(h, W, idx, tlogit, mask)
    grad_loss = _grad_scalar(grad_loss, dev)
    if ws is None:
        ws = alloc_workspace(N, d, V, K, chunk, dev)
    ws_bytes = _ws_bytes(ws, dev)
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=dev)
    _expect_out(loss, "loss", torch.float32, (1,), dev)
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    _expect_out(lse, "lse", torch.float32, (N,), dev)
    dh, dW = _grad_outputs(dh, dW, N, d, V, dev)
    with torch.cuda.device(dev):  # the library launches on the current device
        st = _lib.lib().fkl_forward_backward(_ptr(h), _ptr(W), _ptr(idx), _ptr(tlogit), _ptr(mask), N, d, V, K,
                                             float(T), int(chunk), _ptr(grad_loss), _ptr(loss), _ptr(lse),
                                             _ptr(dh), _ptr(dW), _ptr(ws), ws_bytes, _stream(dev))
    _check(st, "fkl_forward_backward")
    return loss, lse, dh, dW


def topk_workspace_size(N: int, d: int, V: int, K: int, chunk: int = 0) -> int:
    n = _lib.lib().fkl_topk_workspace_size(int(N), int(d), int(V), int(K), int(chunk))
    if n == 0:
        raise ValueError(f"invalid sizes N={N} d={d} V={V} K={K} chunk={chunk}")
    return int(n)


def teacher_topk(h: torch.Tensor, W: torch.Tensor, K: int, chunk: int = 0,
                 ws: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Teacher top-K cache: (idx [N,K] int32, logit [N,K] fp32), logits descending."""
    _expect(h, "h", torch.bfloat16, 2)
    dev = h.device
    _expect(W, "W", torch.bfloat16, 2, dev)
    N, d = h.shape
    V, d2 = W.shape
    if d2 != d:
        raise ValueError(f"h is [N,{d}] but W is [V,{d2}]")
    L = _lib.lib()
    if ws is None:
        ws = torch.empty(topk_workspace_size(N, d, V, K, chunk), dtype=torch.uint8, device=dev)
    ws_bytes = _ws_bytes(ws, dev)
    idx = torch.empty((N, K), dtype=torch.int32, device=dev)
    logit = torch.empty((N, K), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):  # the library launches on the current device
        st = L.fkl_teacher_topk(_ptr(h), _ptr(W), N, d, V, int(K), int(chunk), _ptr(idx), _ptr(logit), _ptr(ws),
                                ws_bytes, _stream(dev))
    _check(st, "fkl_teacher_topk")
    return idx, logit


def get_status(ws: torch.Tensor) -> int:
    """Synchronises the current stream and returns the workspace's device status word."""
    with torch.cuda.device(ws.device):
        return int(_lib.lib().fkl_get_status(_ptr(ws), _stream(ws.device)))


def _raise_on_device_status(ws: torch.Tensor, where: str):
    """Reads the workspace's device status word (synchronising the stream) and raises on an error."""
    st = get_status(ws)
    if st != 0:
        raise FKLError(st, f"{where} (device status)")


class FKLLoss(torch.autograd.Function):
    """T^2 * mean over valid rows of KL(p_teacher || q_student); gradients for h and W."""

    @staticmethod
    def forward(ctx, h, W, idx, tlogit, mask, T, chunk, check_status=False):
        N, d, V, K, dev = _inputs(h, W, idx, tlogit, mask)
        ws = alloc_workspace(N, d, V, K, chunk, dev)
        loss, lse = forward(h, W, idx, tlogit, mask, T, chunk, ws=ws)
        if check_status:
            _raise_on_device_status(ws, "fkl_forward")
        ctx.save_for_backward(h, W, idx, tlogit, lse)
        ctx.mask, ctx.T, ctx.chunk, ctx.ws, ctx.check_status = mask, T, chunk, ws, check_status
        return loss.reshape(())

    @staticmethod
    def backward(ctx, g):
        h, W, idx, tlogit, lse = ctx.saved_tensors
        g = g.reshape(1).to(torch.float32).contiguous()
        dh, dW = backward(h, W, idx, tlogit, ctx.mask, ctx.T, lse, grad_loss=g, chunk=ctx.chunk,
                          ws=ctx.ws)
        if ctx.check_status:
            _raise_on_device_status(ctx.ws, "fkl_backward")
        ctx.ws = None
        return dh, dW.to(W.dtype), None, None, None, None, None, None


class FKLLossKeepLogits(torch.autograd.Function):
    """The same loss with its gradients formed during the forward (fkl_forward_backward:
    each chunk's logits kept instead of recomputed, 6 N d V tensor FLOP instead of 8);
    the backward only scales them by the upstream gradient (fkl_scale_grads).  dh and
    dW are allocated in the forward and held until the backward."""

    @staticmethod
    def forward(ctx, h, W, idx, tlogit, mask, T, chunk, check_status=False):
        N, d, V, K, dev = _inputs(h, W, idx, tlogit, mask)
        ws = alloc_workspace(N, d, V, K, chunk, dev)
        loss, _, dh, dW = forward_backward(h, W, idx, tlogit, mask, T, chunk=chunk, ws=ws)
        if check_status:
            _raise_on_device_status(ws, "fkl_forward_backward")
        ctx.save_for_backward(dh, dW)
        ctx.w_dtype = W.dtype
        return loss.reshape(())

    @staticmethod
    def backward(ctx, g):
        dh, dW = ctx.saved_tensors
        g = g.reshape(1).to(torch.float32).contiguous()
        N, d = dh.shape
        with torch.cuda.device(dh.device):  # the library launches on the current device
            st = _lib.lib().fkl_scale_grads(_ptr(dh), _ptr(dW), N, d, dW.shape[0], _ptr(g), _stream(dh.device))
        _check(st, "fkl_scale_grads")
        return dh, dW.to(ctx.w_dtype), None, None, None, None, None, None


def fkl_loss(h, W, idx, tlogit, mask=None, T: float = 1.0, chunk: int = 0,
             keep_logits: bool = False, check_status: bool = False) -> torch.Tensor:
    """Autograd-aware fused loss (scalar).

    keep_logits=False: fkl_forward now, fkl_backward (logits recomputed) in autograd's
    backward.  keep_logits=True: loss and gradients together in the forward, without
    the recompute; faster, with dh and dW held from the forward to the backward.

    Errors found on the device (a teacher id outside [0, V), a pipeline wait that
    timed out) only set the workspace's status word; the loss and the gradients are
    then undefined.  check_status=True reads that word after each library pass (one
    stream synchronisation each) and raises FKLError on an error; with the default
    False the caller is responsible for validating the teacher ids."""
    if keep_logits:
        return FKLLossKeepLogits.apply(h, W, idx, tlogit, mask, T, chunk, check_status)
    return FKLLoss.apply(h, W, idx, tlogit, mask, T, chunk, check_status)


# ---- measurement hooks -------------------------------------------------------
def profile_enable(on: bool = True):
    _lib.lib().fkl_profile_enable(1 if on else 0)


def profile_reset():
    _lib.lib().fkl_profile_reset()


def profile_read() -> dict:
    """{kernel name: (total ms, launches, algorithmic FLOP)} of the recorded launches."""
    L = _lib.lib()
    n = 64
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    fl = (ctypes.c_double * n)()
    k = L.fkl_profile_read(ms, cnt, fl, n)
    return {L.fkl_kernel_name(i).decode(): (ms[i], int(cnt[i]), fl[i]) for i in range(k) if cnt[i]}


def launch_count() -> int:
    return int(_lib.lib().fkl_launch_count())


def selftest_gemm(A: torch.Tensor, B: torch.Tensor, M: int, N: int, K: int, a_mn: int, b_mn: int,
                  bn: int = 256) -> torch.Tensor:
    """C = A . B^T on the library's tcgen05 pipeline (see fkl_selftest_gemm)."""
    C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    ws = torch.zeros(256, dtype=torch.uint8, device=A.device)
    with torch.cuda.device(A.device):  # the library launches on the current device
        st = _lib.lib().fkl_selftest_gemm(_ptr(A), _ptr(B), _ptr(C), M, N, K, a_mn, b_mn, bn, _ptr(ws),
                                          _stream(A.device))
    _check(st, "fkl_selftest_gemm")
    s = get_status(ws)
    if s != 0:
        raise FKLError(s, "fkl_selftest_gemm (device)")
    return C
