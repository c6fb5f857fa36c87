"""PyTorch-facing binding of the C ABI (``include/lce.h``).

PyTorch supplies device memory and the stream; every step of the computation runs in
``liblce.so``.  The functions keep the C names: ``lce_workspace_size``, ``lce_forward``,
``lce_backward``, ``lce_check_error``; ``linear_cross_entropy`` wraps the forward/backward pair
in a ``torch.autograd.Function``.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import _lib

_DT = {torch.bfloat16: "bf16", torch.float32: "f32"}
# Arithmetic for float32 inputs: "exact" fp32 products on the CUDA cores (LCE_F32), or "tf32x3"
# on the tensor cores, each product from three tf32 products of hi / lo parts (LCE_F32_TF32X3).
F32_MODES = {"exact": "f32", "tf32x3": "tf32x3"}


def _dtype_name(t: torch.Tensor, f32_mode: str = "exact") -> str:
    try:
        dt = _DT[t.dtype]
    except KeyError:
        raise TypeError(f"H and W must be bfloat16 or float32, got {t.dtype}") from None
    if f32_mode not in F32_MODES:
        raise ValueError(f"f32_mode must be one of {sorted(F32_MODES)}, got {f32_mode!r}")
    return F32_MODES[f32_mode] if dt == "f32" else dt


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(device: torch.device, stream: Optional[torch.cuda.Stream]) -> int:
    s = torch.cuda.current_stream(device) if stream is None else stream
    return s.cuda_stream


def _event_handle(e: Optional[torch.cuda.Event]) -> Optional[int]:
    """The cudaEvent_t of a torch event (torch creates the CUDA event at its first record)."""
    if e is None:
        return None
    if not e.cuda_event:
        e.record()
    return e.cuda_event


def _check_inputs(H, W, labels):
    if not (H.is_cuda and W.is_cuda and labels.is_cuda):
        raise ValueError("H, W and labels must be CUDA tensors")
    if H.dim() != 2 or W.dim() != 2 or labels.dim() != 1:
        raise ValueError("expected H [N, d], W [V, d], labels [N]")
    if H.shape[1] != W.shape[1] or labels.shape[0] != H.shape[0]:
        raise ValueError(f"shape mismatch H{tuple(H.shape)} W{tuple(W.shape)} "
                         f"labels{tuple(labels.shape)}")
    if H.dtype != W.dtype:
        raise TypeError("H and W must have the same dtype")
    if labels.dtype != torch.int64:
        raise TypeError("labels must be int64")
    if not (H.is_contiguous() and W.is_contiguous() and labels.is_contiguous()):
        raise ValueError("H, W and labels must be contiguous")


def lce_workspace_size(N: int, d: int, V: int, strip_V: int, dtype: str = "bf16") -> int:
    """Workspace bytes for these sizes (0 when a shape rule is broken)."""
    return int(_lib.load().lce_workspace_size(N, d, V, strip_V, _lib.DTYPES[dtype]))


def lce_strip_columns(V: int, strip_V: int, dtype: str = "bf16") -> int:
    """Width of the vocabulary strips for these sizes (0 on a bad argument)."""
    return int(_lib.load().lce_strip_columns(V, strip_V, _lib.DTYPES[dtype]))


def lce_forward(H, W, labels, *, ignore_index: int = -100, strip_V: int = 8192,
                reduction: str = "mean", workspace: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None, out=None, f32_mode: str = "exact"):
    """Run the forward entry point.  Returns (loss [] fp32, lse [N] fp32, n_valid [] int64,
    workspace).  ``out`` may supply preallocated (loss, lse, n_valid); ``f32_mode`` picks the
    arithmetic for float32 inputs ("exact" or "tf32x3")."""
    _check_inputs(H, W, labels)
    lib = _lib.load()
    N, d = H.shape
    V = W.shape[0]
    dt = _dtype_name(H, f32_mode)
    ws_bytes = lce_workspace_size(N, d, V, strip_V, dt)
    if ws_bytes == 0:
        raise _lib.LceError(2, "lce_workspace_size")
    dev = H.device
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    if out is None:
        loss = torch.empty((), dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        n_valid = torch.empty((), dtype=torch.int64, device=dev)
    else:
        loss, lse, n_valid = out
    with torch.cuda.device(dev):
        st = lib.lce_forward(_ptr(H), _ptr(W), _ptr(labels), N, d, V, ignore_index, strip_V,
                             _lib.REDUCTIONS[reduction], _lib.DTYPES[dt], _ptr(loss), _ptr(lse),
                             _ptr(n_valid), _ptr(workspace), workspace.numel(),
                             _stream_handle(dev, stream))
    _lib.check(st, "lce_forward")
    return loss, lse, n_valid, workspace


def lce_backward(H, W, labels, lse, n_valid, dloss, *, ignore_index: int = -100,
                 strip_V: int = 8192, reduction: str = "mean",
                 workspace: Optional[torch.Tensor] = None, dH=None, dW=None,
                 stream: Optional[torch.cuda.Stream] = None, f32_mode: str = "exact",
                 parts: str = "both"):
    """Run the backward entry point.  Returns (dH [N, d] fp32, dW [V, d] fp32, workspace).

    ``parts`` = "dh" or "dw" computes one gradient only (``lce_backward_parts``; the other is
    returned as None): the data gradient on the critical path now, the weight gradient later."""
    if parts not in _lib.GRAD_PARTS:
        raise ValueError(f"parts must be one of {sorted(_lib.GRAD_PARTS)}, got {parts!r}")
    _check_inputs(H, W, labels)
    lib = _lib.load()
    N, d = H.shape
    V = W.shape[0]
    dt = _dtype_name(H, f32_mode)
    ws_bytes = lce_workspace_size(N, d, V, strip_V, dt)
    if ws_bytes == 0:
        raise _lib.LceError(2, "lce_workspace_size")
    dev = H.device
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    want_dh, want_dw = parts in ("dh", "both"), parts in ("dw", "both")
    if dH is None and want_dh:
        dH = torch.empty(N, d, dtype=torch.float32, device=dev)
    if dW is None and want_dw:
        dW = torch.empty(V, d, dtype=torch.float32, device=dev)
    if not want_dh:
        dH = None
    if not want_dw:
        dW = None
    dloss = dloss.to(device=dev, dtype=torch.float32).contiguous()
    with torch.cuda.device(dev):
        if parts == "both":
            st = lib.lce_backward(_ptr(H), _ptr(W), _ptr(labels), _ptr(lse), _ptr(n_valid),
                                  _ptr(dloss), N, d, V, ignore_index, strip_V,
                                  _lib.REDUCTIONS[reduction], _lib.DTYPES[dt], _ptr(dH), _ptr(dW),
                                  _ptr(workspace), workspace.numel(), _stream_handle(dev, stream))
        else:
            st = lib.lce_backward_parts(_ptr(H), _ptr(W), _ptr(labels), _ptr(lse), _ptr(n_valid),
                                        _ptr(dloss), N, d, V, ignore_index, strip_V,
                                        _lib.REDUCTIONS[reduction], _lib.DTYPES[dt],
                                        _lib.GRAD_PARTS[parts], _ptr(dH), _ptr(dW),
                                        _ptr(workspace), workspace.numel(),
                                        _stream_handle(dev, stream))
    _lib.check(st, "lce_backward")
    return dH, dW, workspace


def lce_host_buffer_size(N: int, d: int, V: int, strip_V: int, dtype: str = "bf16") -> int:
    """Device-buffer bytes lce_forward_backward_host needs for these sizes (0 on a bad shape)."""
    return int(_lib.load().lce_host_buffer_size(N, d, V, strip_V, _lib.DTYPES[dtype]))


def lce_forward_backward_host(H, W, labels, dloss, *, device_buffer: torch.Tensor,
                              ignore_index: int = -100, strip_V: int = 8192,
                              reduction: str = "mean", f32_mode: str = "exact", loss=None,
                              lse=None, n_valid=None, dH=None, dW=None, flags=None,
                              stream: Optional[torch.cuda.Stream] = None,
                              compute_after: Optional[torch.cuda.Event] = None,
                              compute_done: Optional[torch.cuda.Event] = None):
    """Run the host-buffer entry point: H [N, d], W [V, d], labels [N] and dloss [] are CPU
    tensors (pinned for asynchronous copies); loss, lse, n_valid, dH, dW and flags are CPU
    tensors the results are copied into, or None to skip that copy.  device_buffer is a CUDA
    uint8 tensor of at least lce_host_buffer_size bytes.  compute_after / compute_done: events
    the call's kernels wait for / record when they are done (see include/lce.h).  Only enqueues
    work on the stream."""
    for t in (H, W, labels, dloss):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("H, W, labels and dloss must be contiguous CPU tensors")
    if H.dim() != 2 or W.dim() != 2 or labels.dim() != 1 or H.shape[1] != W.shape[1] or \
            labels.shape[0] != H.shape[0] or H.dtype != W.dtype or labels.dtype != torch.int64:
        raise ValueError("expected H [N, d], W [V, d] of one dtype and int64 labels [N]")
    if dloss.dtype != torch.float32 or dloss.numel() != 1:
        raise ValueError("dloss must be one float32 value")
    for t in (loss, lse, n_valid, dH, dW, flags):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError("outputs must be contiguous CPU tensors")
    if not device_buffer.is_cuda:
        raise ValueError("device_buffer must be a CUDA tensor")
    N, d = H.shape
    V = W.shape[0]
    dt = _dtype_name(H, f32_mode)
    dev = device_buffer.device
    with torch.cuda.device(dev):
        st = _lib.load().lce_forward_backward_host(
            _ptr(H), _ptr(W), _ptr(labels), _ptr(dloss), N, d, V, ignore_index, strip_V,
            _lib.REDUCTIONS[reduction], _lib.DTYPES[dt], _ptr(loss), _ptr(lse), _ptr(n_valid),
            _ptr(dH), _ptr(dW), _ptr(flags), _ptr(device_buffer), device_buffer.numel(),
            _stream_handle(dev, stream), _event_handle(compute_after),
            _event_handle(compute_done))
    _lib.check(st, "lce_forward_backward_host")


def lce_check_error(workspace: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Synchronise and raise if the device flagged a bad label or a timed-out wait."""
    with torch.cuda.device(workspace.device):
        st = _lib.load().lce_check_error(_ptr(workspace),
                                         _stream_handle(workspace.device, stream))
    _lib.check(st, "lce_check_error")


def lce_launch_count() -> int:
    return int(_lib.load().lce_launch_count())


class LinearCrossEntropy(torch.autograd.Function):
    """loss = CE(H W^T, labels) without the N x V logits; gradients for H and W."""

    @staticmethod
    def forward(ctx, H, W, labels, ignore_index, strip_V, reduction, f32_mode):
        loss, lse, n_valid, ws = lce_forward(H, W, labels, ignore_index=ignore_index,
                                             strip_V=strip_V, reduction=reduction,
                                             f32_mode=f32_mode)
        del ws  # the forward workspace is released before backward allocates its own
        ctx.save_for_backward(H, W, labels, lse, n_valid)
        ctx.cfg = (ignore_index, strip_V, reduction, f32_mode)
        return loss

    @staticmethod
    def backward(ctx, dloss):
        H, W, labels, lse, n_valid = ctx.saved_tensors
        ignore_index, strip_V, reduction, f32_mode = ctx.cfg
        dH, dW, _ = lce_backward(H, W, labels, lse, n_valid, dloss, ignore_index=ignore_index,
                                 strip_V=strip_V, reduction=reduction, f32_mode=f32_mode)
        return dH.to(H.dtype), dW.to(W.dtype), None, None, None, None, None


def linear_cross_entropy(H, W, labels, ignore_index: int = -100, strip_V: int = 8192,
                         reduction: str = "mean", f32_mode: str = "exact"):
    """Fused vocabulary projection + cross-entropy (autograd).  H [N, d], W [V, d] (bf16 or fp32),
    labels [N] int64; returns the fp32 scalar loss.  ``f32_mode`` ("exact" or "tf32x3") picks the
    arithmetic for float32 inputs."""
    return LinearCrossEntropy.apply(H, W, labels, ignore_index, strip_V, reduction, f32_mode)
