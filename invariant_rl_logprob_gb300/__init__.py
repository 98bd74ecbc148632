"""Batch-invariant selected-token logprob on GB300 (sm_103a).

Thin Python binding over the C-ABI library ``librk.so`` (see ``include/rk.h``).
This module only marshals arguments -- device pointers, sizes and the current
CUDA stream -- and allocates outputs and workspace with PyTorch; every step of
the computation runs in the library's CUDA kernels.  There is no CPU path: if
``librk.so`` is missing or no GPU is present the calls raise.

Operators (RL-Kernel issue #101, maintainer comment, P0 operator list):

* :func:`linear_logp`      -- ``logp[t] = z[t, target_t] - logsumexp_v z[t, v]``, ``z = h W^T``
* :func:`logp_from_logits` -- the same from materialised bf16 logits
* :func:`linear_logp_bwd`  -- ``dh[t] = g[t] (W[target_t] - softmax(z[t]) W)``

Each is bitwise invariant for a given logical row under changes of batch
size, row position, neighbour content, padding and varlen packing.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "RkError", "library_path", "load_library",
    "linear_logp", "linear_logp_workspace_size",
    "logp_from_logits",
    "linear_logp_bwd", "linear_logp_bwd_workspace_size", "linear_logp_bwd_min_workspace_size",
    "lm_head", "logp_from_logits_bwd", "grpo_token_loss", "linear_logp_grpo", "linear_greedy",
    "linear_logp_fwd_saved", "linear_logp_bwd_saved", "linear_logp_saved_size",
    "linear_logp_bwd_saved_workspace_size", "linear_logp_bwd_full_saved",
    "linear_greedy_workspace_size", "linear_logp_dw", "linear_logp_dw_workspace_size",
    "linear_logp_bwd_full", "linear_logp_bwd_full_workspace_size", "lm_head_workspace_size",
    "get_device_error", "selftest_wait_timeout", "set_row_blocks", "last_row_blocks", "DEVERR_TARGET_RANGE", "DEVERR_TIMEOUT", "DEVERR_LSE",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "librk.so")
_lib = None

RK_OK, RK_ERR_INVALID_ARG, RK_ERR_UNSUPPORTED, RK_ERR_WORKSPACE, RK_ERR_CUDA = range(5)
DEVERR_TARGET_RANGE = 0x1
DEVERR_TIMEOUT = 0x2
DEVERR_LSE = 0x4


class RkError(RuntimeError):
    def __init__(self, what: str, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        name = _lib.rk_status_string(status).decode() if _lib is not None else str(status)
        msg = f"{what} failed: {name}"
        if status == RK_ERR_CUDA:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)


def library_path() -> str:
    return _LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load librk.so (built by ``invariant_rl_logprob_gb300.build``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"{_LIB_PATH} is missing: build it with `python -m invariant_rl_logprob_gb300.build` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    lib.rk_linear_logp_workspace_size.argtypes = [i64, i64, i64]
    lib.rk_linear_logp_workspace_size.restype = sz
    lib.rk_linear_logp.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, vp, vp, vp, sz, vp]
    lib.rk_linear_logp.restype = ctypes.c_int
    lib.rk_logp_from_logits.argtypes = [vp, vp, vp, i32, i64, i64, vp, vp, vp]
    lib.rk_logp_from_logits.restype = ctypes.c_int
    lib.rk_linear_logp_bwd_workspace_size.argtypes = [i64, i64, i64]
    lib.rk_linear_logp_bwd_workspace_size.restype = sz
    lib.rk_linear_logp_bwd_min_workspace_size.argtypes = [i64, i64]
    lib.rk_linear_logp_bwd_min_workspace_size.restype = sz
    lib.rk_linear_logp_bwd.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, vp, vp, vp, vp, sz, vp]
    lib.rk_linear_logp_bwd.restype = ctypes.c_int
    lib.rk_lm_head.argtypes = [vp, vp, i64, i64, i64, vp, i64, vp, sz, vp]
    lib.rk_lm_head_workspace_size.argtypes = []
    lib.rk_lm_head_workspace_size.restype = sz
    lib.rk_lm_head.restype = ctypes.c_int
    lib.rk_logp_from_logits_bwd.argtypes = [vp, vp, vp, i32, i64, i64, vp, vp, vp, vp]
    lib.rk_logp_from_logits_bwd.restype = ctypes.c_int
    f32 = ctypes.c_float
    lib.rk_grpo_token_loss.argtypes = [vp, vp, vp, vp, vp, vp, i32, i64, f32, f32, f32, f32,
                                       vp, vp, vp, vp, vp]
    lib.rk_grpo_token_loss.restype = ctypes.c_int
    lib.rk_linear_greedy_workspace_size.argtypes = [i64, i64, i64]
    lib.rk_linear_greedy_workspace_size.restype = sz
    lib.rk_linear_greedy.argtypes = [vp, vp, vp, i32, i64, i64, i64, vp, vp, vp, vp, sz, vp]
    lib.rk_linear_greedy.restype = ctypes.c_int
    lib.rk_linear_logp_dw_workspace_size.argtypes = [i64, i64, i64]
    lib.rk_linear_logp_dw_workspace_size.restype = sz
    lib.rk_linear_logp_dw.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, vp, vp, vp, i64, vp, vp,
                                      sz, vp]
    lib.rk_linear_logp_dw.restype = ctypes.c_int
    lib.rk_linear_logp_bwd_full_workspace_size.argtypes = [i64, i64, i64]
    lib.rk_linear_logp_bwd_full_workspace_size.restype = sz
    lib.rk_linear_logp_bwd_full.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, vp, vp, vp, i64,
                                            vp, vp, vp, sz, vp]
    lib.rk_linear_logp_bwd_full.restype = ctypes.c_int
    lib.rk_selftest_wait_timeout.argtypes = [i64, vp]
    lib.rk_selftest_wait_timeout.restype = ctypes.c_int
    lib.rk_get_device_error.argtypes = [vp, ctypes.POINTER(i32)]
    lib.rk_get_device_error.restype = ctypes.c_int
    lib.rk_status_string.argtypes = [ctypes.c_int]
    lib.rk_status_string.restype = ctypes.c_char_p
    lib.rk_last_cuda_error.argtypes = []
    lib.rk_last_cuda_error.restype = ctypes.c_int
    lib.rk_version.argtypes = []
    lib.rk_version.restype = ctypes.c_char_p
    f32 = ctypes.c_float
    lib.rk_linear_logp_grpo.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, vp, vp, vp, f32, f32,
                                        f32, f32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.rk_linear_logp_grpo.restype = ctypes.c_int
    lib.rk_linear_logp_saved_size.argtypes = [i64, i64, i64]
    lib.rk_linear_logp_saved_size.restype = sz
    lib.rk_linear_logp_fwd_saved.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, vp, vp, vp, sz, vp]
    lib.rk_linear_logp_fwd_saved.restype = ctypes.c_int
    lib.rk_linear_logp_bwd_saved_workspace_size.argtypes = [i64, i64, i64]
    lib.rk_linear_logp_bwd_saved_workspace_size.restype = sz
    lib.rk_linear_logp_bwd_saved.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, vp, vp, vp, sz, vp,
                                             vp, sz, vp]
    lib.rk_linear_logp_bwd_saved.restype = ctypes.c_int
    lib.rk_linear_logp_bwd_full_saved.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, vp, vp, vp,
                                                  sz, vp, i64, vp, vp, vp, sz, vp]
    lib.rk_linear_logp_bwd_full_saved.restype = ctypes.c_int
    lib.rk_set_row_blocks.argtypes = [i32]
    lib.rk_set_row_blocks.restype = ctypes.c_int
    lib.rk_last_row_blocks.argtypes = [i32]
    lib.rk_last_row_blocks.restype = i32
    lib.rk_last_tile_order.argtypes = [i32]
    lib.rk_last_tile_order.restype = i32
    _lib = lib
    return lib


def _check(status: int, what: str) -> None:
    if status != RK_OK:
        raise RkError(what, status, _lib.rk_last_cuda_error() if status == RK_ERR_CUDA else 0)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path), got {t.device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _rows(targets, cu_seqlens, T, device):
    _need(targets, "targets", torch.int64, 1)
    if targets.shape[0] != T or targets.device != device:
        raise ValueError("targets must be [T] on the same device")
    if cu_seqlens is None:
        return None, 0
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    if cu_seqlens.device != device or cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens must be a non-empty int32 tensor on the same device")
    return cu_seqlens, cu_seqlens.numel() - 1


def linear_logp_workspace_size(T: int, H: int, V: int) -> int:
    return int(load_library().rk_linear_logp_workspace_size(T, H, V))


def linear_logp(h: torch.Tensor, W: torch.Tensor, targets: torch.Tensor,
                cu_seqlens: torch.Tensor | None = None, *, out: torch.Tensor | None = None,
                lse: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                stream: torch.cuda.Stream | None = None):
    """Selected-token logprob of ``h W^T``: returns ``(logp, lse)``, fp32 ``[T]``."""
    lib = load_library()
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    T, H = h.shape
    V = W.shape[0]
    if W.shape[1] != H or W.device != h.device:
        raise ValueError("W must be [V, H] on h's device")
    cu, ns = _rows(targets, cu_seqlens, T, h.device)
    if out is None:
        out = torch.empty(T, dtype=torch.float32, device=h.device)
    if lse is None:
        lse = torch.empty(T, dtype=torch.float32, device=h.device)
    need = int(lib.rk_linear_logp_workspace_size(T, H, V))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=h.device)
    st = lib.rk_linear_logp(_ptr(h), _ptr(W), _ptr(targets), _ptr(cu), ns, T, H, V,
                            _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                            _stream_handle(stream, h.device))
    _check(st, "rk_linear_logp")
    return out, lse


def logp_from_logits(logits: torch.Tensor, targets: torch.Tensor,
                     cu_seqlens: torch.Tensor | None = None, *, out: torch.Tensor | None = None,
                     lse: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None):
    """Selected-token logprob from bf16 logits ``[T, V]``: returns ``(logp, lse)``."""
    lib = load_library()
    _need(logits, "logits", torch.bfloat16, 2)
    T, V = logits.shape
    cu, ns = _rows(targets, cu_seqlens, T, logits.device)
    if out is None:
        out = torch.empty(T, dtype=torch.float32, device=logits.device)
    if lse is None:
        lse = torch.empty(T, dtype=torch.float32, device=logits.device)
    st = lib.rk_logp_from_logits(_ptr(logits), _ptr(targets), _ptr(cu), ns, T, V, _ptr(out),
                                 _ptr(lse), _stream_handle(stream, logits.device))
    _check(st, "rk_logp_from_logits")
    return out, lse


def linear_logp_bwd_workspace_size(T: int, H: int, V: int) -> int:
    return int(load_library().rk_linear_logp_bwd_workspace_size(T, H, V))


def linear_logp_bwd_min_workspace_size(H: int, V: int) -> int:
    return int(load_library().rk_linear_logp_bwd_min_workspace_size(H, V))


def linear_logp_bwd(h: torch.Tensor, W: torch.Tensor, targets: torch.Tensor, lse: torch.Tensor,
                    grad_logp: torch.Tensor, cu_seqlens: torch.Tensor | None = None, *,
                    dh: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                    stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """dh = g (W[target] - softmax(h W^T) W) in fp32 ``[T, H]``."""
    lib = load_library()
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    T, H = h.shape
    V = W.shape[0]
    if W.shape[1] != H or W.device != h.device:
        raise ValueError("W must be [V, H] on h's device")
    cu, ns = _rows(targets, cu_seqlens, T, h.device)
    _need(lse, "lse", torch.float32, 1)
    _need(grad_logp, "grad_logp", torch.float32, 1)
    if dh is None:
        dh = torch.empty((T, H), dtype=torch.float32, device=h.device)
    if workspace is None:
        need = int(lib.rk_linear_logp_bwd_workspace_size(T, H, V))
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=h.device)
    st = lib.rk_linear_logp_bwd(_ptr(h), _ptr(W), _ptr(targets), _ptr(cu), ns, T, H, V,
                                _ptr(lse), _ptr(grad_logp), _ptr(dh), _ptr(workspace),
                                workspace.numel(), _stream_handle(stream, h.device))
    _check(st, "rk_linear_logp_bwd")
    return dh


def lm_head_workspace_size() -> int:
    return int(load_library().rk_lm_head_workspace_size())


def lm_head(h: torch.Tensor, W: torch.Tensor, *, out: torch.Tensor | None = None,
            workspace: torch.Tensor | None = None,
            stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Dense path: bf16 logits ``[T, V]`` = bf16(h W^T) (fp32 accumulation).

    ``workspace`` (uint8, >= ``rk_lm_head_workspace_size()`` bytes) holds the
    tile counter; one is allocated when it is None."""
    lib = load_library()
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    T, H = h.shape
    V = W.shape[0]
    if W.shape[1] != H or W.device != h.device:
        raise ValueError("W must be [V, H] on h's device")
    ld = (V + 7) // 8 * 8
    if out is None:
        buf = torch.empty((T, ld), dtype=torch.bfloat16, device=h.device)
        out = buf[:, :V]
    else:
        if out.dtype != torch.bfloat16 or out.dim() != 2 or out.stride(1) != 1:
            raise ValueError("out must be a bf16 [T, V] view with unit column stride")
        ld = out.stride(0)
    if workspace is None:
        workspace = torch.empty(int(lib.rk_lm_head_workspace_size()), dtype=torch.uint8,
                                device=h.device)
    st = lib.rk_lm_head(_ptr(h), _ptr(W), T, H, V, _ptr(out), ld, _ptr(workspace),
                        workspace.numel(), _stream_handle(stream, h.device))
    _check(st, "rk_lm_head")
    return out


def logp_from_logits_bwd(logits: torch.Tensor, targets: torch.Tensor, lse: torch.Tensor,
                         grad_logp: torch.Tensor, cu_seqlens: torch.Tensor | None = None, *,
                         out: torch.Tensor | None = None,
                         stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """dlogits = g (onehot - softmax(logits)) in fp32 ``[T, V]``."""
    lib = load_library()
    _need(logits, "logits", torch.bfloat16, 2)
    T, V = logits.shape
    cu, ns = _rows(targets, cu_seqlens, T, logits.device)
    _need(lse, "lse", torch.float32, 1)
    _need(grad_logp, "grad_logp", torch.float32, 1)
    if out is None:
        out = torch.empty((T, V), dtype=torch.float32, device=logits.device)
    st = lib.rk_logp_from_logits_bwd(_ptr(logits), _ptr(targets), _ptr(cu), ns, T, V, _ptr(lse),
                                     _ptr(grad_logp), _ptr(out),
                                     _stream_handle(stream, logits.device))
    _check(st, "rk_logp_from_logits_bwd")
    return out


def grpo_token_loss(logp: torch.Tensor, logp_old: torch.Tensor, advantages: torch.Tensor,
                    targets: torch.Tensor, cu_seqlens: torch.Tensor | None = None, *,
                    logp_ref: torch.Tensor | None = None, eps_low: float = 0.2,
                    eps_high: float = 0.2, beta: float = 0.0, scale: float = 1.0,
                    stream: torch.cuda.Stream | None = None) -> dict:
    """Per-token GRPO loss: dict with fp32 ``loss``, ``grad`` (d loss/d logp),
    ``ratio`` and ``kl``, each ``[T]``."""
    lib = load_library()
    for name, t in (("logp", logp), ("logp_old", logp_old), ("advantages", advantages)):
        _need(t, name, torch.float32, 1)
    T = logp.shape[0]
    if logp_ref is not None:
        _need(logp_ref, "logp_ref", torch.float32, 1)
    cu, ns = _rows(targets, cu_seqlens, T, logp.device)
    out = {k: torch.empty(T, dtype=torch.float32, device=logp.device)
           for k in ("loss", "grad", "ratio", "kl")}
    st = lib.rk_grpo_token_loss(_ptr(logp), _ptr(logp_old), _ptr(logp_ref), _ptr(advantages),
                                _ptr(targets), _ptr(cu), ns, T, eps_low, eps_high, beta, scale,
                                _ptr(out["loss"]), _ptr(out["grad"]), _ptr(out["ratio"]),
                                _ptr(out["kl"]), _stream_handle(stream, logp.device))
    _check(st, "rk_grpo_token_loss")
    return out


def linear_logp_grpo(h: torch.Tensor, W: torch.Tensor, targets: torch.Tensor,
                     logp_old: torch.Tensor, advantages: torch.Tensor,
                     cu_seqlens: torch.Tensor | None = None, *,
                     logp_ref: torch.Tensor | None = None, eps_low: float = 0.2,
                     eps_high: float = 0.2, beta: float = 0.0, scale: float = 1.0,
                     workspace: torch.Tensor | None = None,
                     stream: torch.cuda.Stream | None = None) -> dict:
    """linear_logp with the per-token GRPO loss applied in its merge: dict of
    fp32 ``[T]`` tensors ``logp``, ``lse``, ``loss``, ``grad``, ``ratio``,
    ``kl`` (the same bits as linear_logp followed by grpo_token_loss)."""
    lib = load_library()
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    T, H = h.shape
    V = W.shape[0]
    if W.shape[1] != H or W.device != h.device:
        raise ValueError("W must be [V, H] on h's device")
    for name, t in (("logp_old", logp_old), ("advantages", advantages)):
        _need(t, name, torch.float32, 1)
    if logp_ref is not None:
        _need(logp_ref, "logp_ref", torch.float32, 1)
    cu, ns = _rows(targets, cu_seqlens, T, h.device)
    out = {k: torch.empty(T, dtype=torch.float32, device=h.device)
           for k in ("logp", "lse", "loss", "grad", "ratio", "kl")}
    need = int(lib.rk_linear_logp_workspace_size(T, H, V))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=h.device)
    st = lib.rk_linear_logp_grpo(_ptr(h), _ptr(W), _ptr(targets), _ptr(cu), ns, T, H, V,
                                 _ptr(logp_old), _ptr(logp_ref), _ptr(advantages), eps_low,
                                 eps_high, beta, scale, _ptr(out["logp"]), _ptr(out["lse"]),
                                 _ptr(out["loss"]), _ptr(out["grad"]), _ptr(out["ratio"]),
                                 _ptr(out["kl"]), _ptr(workspace), workspace.numel(),
                                 _stream_handle(stream, h.device))
    _check(st, "rk_linear_logp_grpo")
    return out


def linear_logp_saved_size(T: int, H: int, V: int) -> int:
    return int(load_library().rk_linear_logp_saved_size(T, H, V))


def linear_logp_bwd_saved_workspace_size(T: int, H: int, V: int) -> int:
    return int(load_library().rk_linear_logp_bwd_saved_workspace_size(T, H, V))


def linear_logp_fwd_saved(h: torch.Tensor, W: torch.Tensor, targets: torch.Tensor,
                          cu_seqlens: torch.Tensor | None = None, *,
                          out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                          saved: torch.Tensor | None = None,
                          stream: torch.cuda.Stream | None = None):
    """linear_logp that also keeps its softmax terms for
    :func:`linear_logp_bwd_saved`: returns ``(logp, lse, saved)``."""
    lib = load_library()
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    T, H = h.shape
    V = W.shape[0]
    if W.shape[1] != H or W.device != h.device:
        raise ValueError("W must be [V, H] on h's device")
    cu, ns = _rows(targets, cu_seqlens, T, h.device)
    if out is None:
        out = torch.empty(T, dtype=torch.float32, device=h.device)
    if lse is None:
        lse = torch.empty(T, dtype=torch.float32, device=h.device)
    if saved is None:
        saved = torch.empty(max(int(lib.rk_linear_logp_saved_size(T, H, V)), 1), dtype=torch.uint8,
                            device=h.device)
    st = lib.rk_linear_logp_fwd_saved(_ptr(h), _ptr(W), _ptr(targets), _ptr(cu), ns, T, H, V,
                                      _ptr(out), _ptr(lse), _ptr(saved), saved.numel(),
                                      _stream_handle(stream, h.device))
    _check(st, "rk_linear_logp_fwd_saved")
    return out, lse, saved


def linear_logp_bwd_saved(h: torch.Tensor, W: torch.Tensor, targets: torch.Tensor,
                          lse: torch.Tensor, grad_logp: torch.Tensor, saved: torch.Tensor,
                          cu_seqlens: torch.Tensor | None = None, *,
                          dh: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                          stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """dh fp32 ``[T, H]`` from the state :func:`linear_logp_fwd_saved` kept
    (which this call consumes)."""
    lib = load_library()
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    _need(lse, "lse", torch.float32, 1)
    _need(grad_logp, "grad_logp", torch.float32, 1)
    T, H = h.shape
    V = W.shape[0]
    cu, ns = _rows(targets, cu_seqlens, T, h.device)
    if dh is None:
        dh = torch.empty((T, H), dtype=torch.float32, device=h.device)
    if workspace is None:
        need = int(lib.rk_linear_logp_bwd_saved_workspace_size(T, H, V))
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=h.device)
    st = lib.rk_linear_logp_bwd_saved(_ptr(h), _ptr(W), _ptr(targets), _ptr(cu), ns, T, H, V,
                                      _ptr(lse), _ptr(grad_logp), _ptr(saved), saved.numel(),
                                      _ptr(dh), _ptr(workspace), workspace.numel(),
                                      _stream_handle(stream, h.device))
    _check(st, "rk_linear_logp_bwd_saved")
    return dh


def linear_logp_bwd_full_saved(h: torch.Tensor, W: torch.Tensor, targets: torch.Tensor,
                               lse: torch.Tensor, grad_logp: torch.Tensor, saved: torch.Tensor,
                               cu_seqlens: torch.Tensor | None = None, *,
                               row_order: torch.Tensor | None = None,
                               dh: torch.Tensor | None = None, dW: torch.Tensor | None = None,
                               workspace: torch.Tensor | None = None,
                               stream: torch.cuda.Stream | None = None):
    """(dh fp32 [T, H], dW fp32 [V, H]) from the state :func:`linear_logp_fwd_saved`
    kept (read only)."""
    lib = load_library()
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    T, H = h.shape
    V = W.shape[0]
    cu, ns = _rows(targets, cu_seqlens, T, h.device)
    if row_order is not None:
        _need(row_order, "row_order", torch.int64, 1)
        n = row_order.shape[0]
    else:
        n = T
    if dh is None:
        dh = torch.empty((T, H), dtype=torch.float32, device=h.device)
    if dW is None:
        dW = torch.empty((V, H), dtype=torch.float32, device=h.device)
    if workspace is None:
        need = int(lib.rk_linear_logp_bwd_full_workspace_size(n, H, V))
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=h.device)
    st = lib.rk_linear_logp_bwd_full_saved(_ptr(h), _ptr(W), _ptr(targets), _ptr(cu), ns, T, H, V,
                                           _ptr(lse), _ptr(grad_logp), _ptr(saved), saved.numel(),
                                           _ptr(row_order), n, _ptr(dh), _ptr(dW),
                                           _ptr(workspace), workspace.numel(),
                                           _stream_handle(stream, h.device))
    _check(st, "rk_linear_logp_bwd_full_saved")
    return dh, dW


def linear_greedy_workspace_size(T: int, H: int, V: int) -> int:
    return int(load_library().rk_linear_greedy_workspace_size(T, H, V))


def linear_greedy(h: torch.Tensor, W: torch.Tensor, cu_seqlens: torch.Tensor | None = None, *,
                  workspace: torch.Tensor | None = None,
                  stream: torch.cuda.Stream | None = None):
    """Greedy step: ``(token int64 [T], logp fp32 [T], lse fp32 [T])``."""
    lib = load_library()
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    T, H = h.shape
    V = W.shape[0]
    if W.shape[1] != H or W.device != h.device:
        raise ValueError("W must be [V, H] on h's device")
    cu, ns = (None, 0)
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
        cu, ns = cu_seqlens, cu_seqlens.numel() - 1
    token = torch.empty(T, dtype=torch.int64, device=h.device)
    logp = torch.empty(T, dtype=torch.float32, device=h.device)
    lse = torch.empty(T, dtype=torch.float32, device=h.device)
    if workspace is None:
        need = int(lib.rk_linear_greedy_workspace_size(T, H, V))
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=h.device)
    st = lib.rk_linear_greedy(_ptr(h), _ptr(W), _ptr(cu), ns, T, H, V, _ptr(token), _ptr(logp),
                              _ptr(lse), _ptr(workspace), workspace.numel(),
                              _stream_handle(stream, h.device))
    _check(st, "rk_linear_greedy")
    return token, logp, lse


def linear_logp_dw_workspace_size(n: int, H: int, V: int) -> int:
    return int(load_library().rk_linear_logp_dw_workspace_size(n, H, V))


def linear_logp_dw(h: torch.Tensor, W: torch.Tensor, targets: torch.Tensor, lse: torch.Tensor,
                   grad_logp: torch.Tensor, cu_seqlens: torch.Tensor | None = None, *,
                   row_order: torch.Tensor | None = None, dW: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None,
                   stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """dW fp32 ``[V, H]`` summed over the active rows in canonical order
    (``row_order``, int64 physical row indices; ascending rows by default)."""
    lib = load_library()
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    T, H = h.shape
    V = W.shape[0]
    if W.shape[1] != H or W.device != h.device:
        raise ValueError("W must be [V, H] on h's device")
    cu, ns = _rows(targets, cu_seqlens, T, h.device)
    _need(lse, "lse", torch.float32, 1)
    _need(grad_logp, "grad_logp", torch.float32, 1)
    n = T
    if row_order is not None:
        _need(row_order, "row_order", torch.int64, 1)
        n = row_order.numel()
    if dW is None:
        dW = torch.empty((V, H), dtype=torch.float32, device=h.device)
    if workspace is None:
        need = int(lib.rk_linear_logp_dw_workspace_size(n, H, V))
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=h.device)
    st = lib.rk_linear_logp_dw(_ptr(h), _ptr(W), _ptr(targets), _ptr(cu), ns, T, H, V, _ptr(lse),
                               _ptr(grad_logp), _ptr(row_order), n, _ptr(dW), _ptr(workspace),
                               workspace.numel(), _stream_handle(stream, h.device))
    _check(st, "rk_linear_logp_dw")
    return dW


def linear_logp_bwd_full_workspace_size(n: int, H: int, V: int) -> int:
    return int(load_library().rk_linear_logp_bwd_full_workspace_size(n, H, V))


def linear_logp_bwd_full(h: torch.Tensor, W: torch.Tensor, targets: torch.Tensor,
                         lse: torch.Tensor, grad_logp: torch.Tensor,
                         cu_seqlens: torch.Tensor | None = None, *,
                         row_order: torch.Tensor | None = None, dh: torch.Tensor | None = None,
                         dW: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                         stream: torch.cuda.Stream | None = None):
    """(dh fp32 [T, H], dW fp32 [V, H]) from one shared softmax pass."""
    lib = load_library()
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    T, H = h.shape
    V = W.shape[0]
    if W.shape[1] != H or W.device != h.device:
        raise ValueError("W must be [V, H] on h's device")
    cu, ns = _rows(targets, cu_seqlens, T, h.device)
    _need(lse, "lse", torch.float32, 1)
    _need(grad_logp, "grad_logp", torch.float32, 1)
    n = T
    if row_order is not None:
        _need(row_order, "row_order", torch.int64, 1)
        n = row_order.numel()
    if dh is None:
        dh = torch.empty((T, H), dtype=torch.float32, device=h.device)
    if dW is None:
        dW = torch.empty((V, H), dtype=torch.float32, device=h.device)
    if workspace is None:
        need = int(lib.rk_linear_logp_bwd_full_workspace_size(n, H, V))
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=h.device)
    st = lib.rk_linear_logp_bwd_full(_ptr(h), _ptr(W), _ptr(targets), _ptr(cu), ns, T, H, V,
                                     _ptr(lse), _ptr(grad_logp), _ptr(row_order), n, _ptr(dh),
                                     _ptr(dW), _ptr(workspace), workspace.numel(),
                                     _stream_handle(stream, h.device))
    _check(st, "rk_linear_logp_bwd_full")
    return dh, dW


def selftest_wait_timeout(limit_ns: int, stream: torch.cuda.Stream | None = None) -> None:
    """Launch a kernel whose bounded wait must time out after ``limit_ns``."""
    lib = load_library()
    _check(lib.rk_selftest_wait_timeout(int(limit_ns), _stream_handle(stream, None)),
           "rk_selftest_wait_timeout")


def set_row_blocks(n: int) -> None:
    """Row blocks per tile of the dh and dW GEMMs: 0 automatic (default), or
    1 / 2 forced for every later launch in the process (bits are unchanged)."""
    _check(load_library().rk_set_row_blocks(int(n)), "rk_set_row_blocks")


def last_row_blocks(gemm: str) -> int:
    """Row blocks per tile of the last ``"dh"`` or ``"dw"`` GEMM launched on
    this thread (0 before the first)."""
    return int(load_library().rk_last_row_blocks({"dh": 0, "dw": 1}[gemm]))


def last_tile_order(gemm: str) -> int:
    """Tile order of the last ``"dh"`` or ``"dw"`` GEMM launched on this
    thread: 2 rounds started together, 1 tiles from a counter, 0 before the
    first."""
    return int(load_library().rk_last_tile_order({"dh": 0, "dw": 1}[gemm]))


def get_device_error(stream: torch.cuda.Stream | None = None) -> int:
    """Read and clear the device error word (synchronises the stream)."""
    lib = load_library()
    v = ctypes.c_int32(0)
    _check(lib.rk_get_device_error(_stream_handle(stream, None), ctypes.byref(v)),
           "rk_get_device_error")
    return int(v.value)
