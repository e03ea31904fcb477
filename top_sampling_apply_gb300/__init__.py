"""Per-row vocabulary selection on GB300: thin Python binding of libtsa.so.

The three calls mirror the C ABI in include/tsa.h (logits-processor, "API";
lm-head-topk, "API").  This module only marshals arguments: it checks torch
tensors' device, dtype and contiguity, passes raw pointers and the current
CUDA stream, and maps status codes to exceptions.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Union

import torch

from . import _build

__all__ = ["apply_token_bitmask", "sample", "topk", "device_status", "max_vocab", "load_library",
           "TSAError"]

_DT = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
_lock = threading.Lock()
_lib = None
_workspaces = {}  # device index -> uint8 scratch tensor


class TSAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("%s (status %d)" % (msg, status))
        self.status = status


def load_library(path: Optional[str] = None):
    """Load libtsa.so (built by ``__graft_entry__.build()`` or
    ``python -m top_sampling_apply_gb300._build``).  Raises if it is missing:
    the product has no CPU path."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _build.LIB
        if not os.path.exists(p):
            raise RuntimeError("libtsa.so not built: run __graft_entry__.build() (nvcc, sm_103a)")
        lib = ctypes.CDLL(p)
        P, i64, i32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64
        f32, sz, ci = ctypes.c_float, ctypes.c_size_t, ctypes.c_int
        lib.tsa_apply_token_bitmask.argtypes = [P, ci, i64, i64, i64, P, i64, P]
        lib.tsa_sample.argtypes = [P, ci, i64, i64, i64, P, i64, P, f32, P, i32, P, f32, P, f32,
                                   u64, u64, P, P, P, sz, P]
        lib.tsa_sample_noalloc.argtypes = [P, ci, i64, i64, i64, P, i64, P, f32, P, i32, P, f32,
                                           P, f32, u64, u64, P, P, P]
        lib.tsa_topk.argtypes = [P, ci, i64, i64, i64, i32, P, P, P, sz, P]
        lib.tsa_sample_icdf.argtypes = [P, ci, i64, i64, i64, P, i64, P, f32, P, i32, P, f32, P,
                                        f32, P, P, P, P, sz, P]
        lib.tsa_bitmask_from_allowed.argtypes = [P, i64, i64, i64, P, i64, P]
        lib.tsa_sample_sequential.argtypes = [P, ci, i64, i64, i64, P, i64, P, f32, P, i32, P, f32,
                                              P, f32, u64, u64, P, P, P, sz, P]
        lib.tsa_sample_sequential_workspace_bytes.argtypes = [i64, i64, ci]
        lib.tsa_sample_sequential_workspace_bytes.restype = sz
        lib.tsa_lm_head_topk.argtypes = [P, i64, i64, i64, P, i64, i64, P, i32, P, P, P, sz, P]
        lib.tsa_lm_head_topk_workspace_bytes.argtypes = [i64, i64, i32]
        lib.tsa_lm_head_topk_workspace_bytes.restype = sz
        lib.tsa_selective_log_softmax.argtypes = [P, ci, i64, i64, i64, P, i64, P, f32, P, P, P]
        lib.tsa_sample_workspace_bytes.argtypes = [i64, i64, ci]
        lib.tsa_sample_workspace_bytes.restype = sz
        lib.tsa_topk_workspace_bytes.argtypes = [i64, i64, i32, ci]
        lib.tsa_topk_workspace_bytes.restype = sz
        lib.tsa_status_string.argtypes = [ci]
        lib.tsa_status_string.restype = ctypes.c_char_p
        lib.tsa_device_status.argtypes = [ci]
        lib.tsa_selftest_wait_timeout.argtypes = [ctypes.c_uint32, P]
        lib.tsa_max_vocab.argtypes = [ci]
        lib.tsa_max_vocab.restype = i64
        for fn in ("tsa_apply_token_bitmask", "tsa_sample", "tsa_sample_noalloc", "tsa_topk",
                   "tsa_sample_icdf", "tsa_bitmask_from_allowed", "tsa_sample_sequential", "tsa_lm_head_topk",
                   "tsa_device_status", "tsa_selftest_wait_timeout"):
            getattr(lib, fn).restype = ci
        _lib = lib
        return lib


def _check(status: int):
    if status != 0:
        lib = load_library()
        raise TSAError(status, lib.tsa_status_string(status).decode())


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _rows(logits: torch.Tensor):
    if not logits.is_cuda:
        raise ValueError("logits must be a CUDA tensor")
    if logits.dtype not in _DT:
        raise ValueError("logits dtype must be float32, float16 or bfloat16")
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be 2-D [B, V] with unit stride along V")
    return logits.shape[0], logits.shape[1], logits.stride(0)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _workspace(nbytes: int, device: torch.device) -> torch.Tensor:
    """A device workspace of at least ``nbytes``, cached per device (calls on
    different streams must not run concurrently on the same workspace)."""
    idx = device.index if device.index is not None else torch.cuda.current_device()
    ws = _workspaces.get(idx)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[idx] = ws
    return ws


def max_vocab(dtype: torch.dtype) -> int:
    return int(load_library().tsa_max_vocab(_DT[dtype]))


def apply_token_bitmask(logits: torch.Tensor, bitmask: torch.Tensor) -> torch.Tensor:
    """logits-processor, "API": set logits to -inf, in place, where the packed
    bit is 0 (bit 1 = allowed).  bitmask: int32 [B, >= ceil(V / 32)]."""
    lib = load_library()
    B, V, stride = _rows(logits)
    if bitmask.dtype != torch.int32 or not bitmask.is_cuda or bitmask.dim() != 2:
        raise ValueError("bitmask must be a CUDA int32 [B, W] tensor")
    if bitmask.shape[0] != B or bitmask.stride(1) != 1:
        raise ValueError("bitmask must have B rows and unit stride along W")
    if bitmask.shape[1] < (V + 31) // 32:
        raise ValueError("bitmask needs ceil(V / 32) words per row")
    _check(lib.tsa_apply_token_bitmask(_ptr(logits), _DT[logits.dtype], B, V, stride,
                                       _ptr(bitmask), bitmask.stride(0), _stream(logits)))
    return logits


Param = Union[float, int, torch.Tensor]


def _param(x: Param, B: int, dtype: torch.dtype, device):
    """(device pointer or None, scalar) for a per-row parameter."""
    if isinstance(x, torch.Tensor):
        if x.dim() == 0:
            return None, x.item()
        if x.shape != (B,) or x.dtype != dtype or x.device != device or not x.is_contiguous():
            raise ValueError("per-row parameter must be a contiguous %s [B] tensor on %s"
                             % (dtype, device))
        return x, 0
    return None, x


def sample(logits: torch.Tensor, temperature: Param = 1.0, top_k: Param = 0, top_p: Param = 1.0,
           min_p: Param = 0.0, seed: int = 0, offset: int = 0,
           bitmask: Optional[torch.Tensor] = None, return_min_kept: bool = False,
           out: Optional[torch.Tensor] = None, sequential: bool = False):
    """logits-processor, "API": one int64 token per row (-1 for a row with no
    allowed finite logit).  Each sampling parameter is a scalar or a [B]
    tensor (float32 for temperature / top_p / min_p, int32 for top_k).  With
    ``bitmask`` the mask is applied on load; the logits are not modified.
    ``sequential`` takes top-p over the softmax renormalised over the top-k
    survivors (the transformers processor chain) instead of the full one."""
    lib = load_library()
    B, V, stride = _rows(logits)
    dev = logits.device
    T, Ts = _param(temperature, B, torch.float32, dev)
    K, Ks = _param(top_k, B, torch.int32, dev)
    Pp, Ps = _param(top_p, B, torch.float32, dev)
    M, Ms = _param(min_p, B, torch.float32, dev)
    if bitmask is not None:
        if bitmask.dtype != torch.int32 or bitmask.device != dev or bitmask.dim() != 2:
            raise ValueError("bitmask must be an int32 [B, W] tensor on the logits' device")
        if bitmask.shape[0] != B or bitmask.stride(1) != 1 or bitmask.shape[1] < (V + 31) // 32:
            raise ValueError("bitmask must be [B, >= ceil(V / 32)] with unit stride along W")
        mstride = bitmask.stride(0)
    else:
        mstride = 0
    tokens = out if out is not None else torch.empty(B, dtype=torch.int64, device=dev)
    vstar = torch.empty(B, dtype=torch.float32, device=dev) if return_min_kept else None
    if sequential:
        nws = int(lib.tsa_sample_sequential_workspace_bytes(B, V, _DT[logits.dtype]))
        ws = _workspace(nws, dev) if nws > 0 else None
        call = lib.tsa_sample_sequential
    else:
        nws = int(lib.tsa_sample_workspace_bytes(B, V, _DT[logits.dtype]))
        ws = _workspace(nws, dev) if nws > 0 else None
        call = lib.tsa_sample
    _check(call(_ptr(logits), _DT[logits.dtype], B, V, stride, _ptr(bitmask), mstride,
                          _ptr(T), float(Ts), _ptr(K), int(Ks), _ptr(Pp), float(Ps), _ptr(M),
                          float(Ms), int(seed) & 0xFFFFFFFFFFFFFFFF,
                          int(offset) & 0xFFFFFFFFFFFFFFFF, _ptr(tokens), _ptr(vstar), _ptr(ws),
                          nws, _stream(logits)))
    return (tokens, vstar) if return_min_kept else tokens


def sample_icdf(logits: torch.Tensor, uniform: torch.Tensor, temperature: Param = 1.0, top_k: Param = 0,
                top_p: Param = 1.0, min_p: Param = 0.0, bitmask: Optional[torch.Tensor] = None,
                return_min_kept: bool = False, out: Optional[torch.Tensor] = None):
    """logits-mask-xpu, "Usage" / "Method": the inverse-CDF draw from the caller's
    ``uniform`` (float32 [B] in [0, 1) on the logits' device) over the keep set of
    ``sample``: the first kept token, in index order, whose running weight passes
    u W.  Parameters as ``sample`` (no seed: the draw is the uniform's)."""
    lib = load_library()
    B, V, stride = _rows(logits)
    dev = logits.device
    if uniform.dtype != torch.float32 or uniform.device != dev or uniform.shape != (B,) \
            or not uniform.is_contiguous():
        raise ValueError("uniform must be a contiguous float32 [B] tensor on the logits' device")
    T, Ts = _param(temperature, B, torch.float32, dev)
    K, Ks = _param(top_k, B, torch.int32, dev)
    Pp, Ps = _param(top_p, B, torch.float32, dev)
    M, Ms = _param(min_p, B, torch.float32, dev)
    mstride = _mask_stride(bitmask, B, V, dev)
    tokens = out if out is not None else torch.empty(B, dtype=torch.int64, device=dev)
    vstar = torch.empty(B, dtype=torch.float32, device=dev)
    nws = int(lib.tsa_sample_workspace_bytes(B, V, _DT[logits.dtype]))
    ws = _workspace(nws, dev) if nws > 0 else None
    _check(lib.tsa_sample_icdf(_ptr(logits), _DT[logits.dtype], B, V, stride, _ptr(bitmask), mstride,
                               _ptr(T), float(Ts), _ptr(K), int(Ks), _ptr(Pp), float(Ps), _ptr(M),
                               float(Ms), _ptr(uniform), _ptr(tokens), _ptr(vstar), _ptr(ws), nws,
                               _stream(logits)))
    return (tokens, vstar) if return_min_kept else tokens


def bitmask_from_allowed(allowed: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """logits-mask-xpu, "Usage": a CUDA bool [B, V] allow-set packed into int32
    [B, ceil(V / 32)] words (token i at bit i % 32 of word i // 32)."""
    lib = load_library()
    if allowed.dtype != torch.bool or not allowed.is_cuda or allowed.dim() != 2 or allowed.stride(1) != 1:
        raise ValueError("allowed must be a CUDA bool [B, V] tensor with unit stride along V")
    B, V = allowed.shape
    W = (V + 31) // 32
    bits = out if out is not None else torch.empty(B, W, dtype=torch.int32, device=allowed.device)
    if bits.dtype != torch.int32 or bits.device != allowed.device or bits.shape[0] != B \
            or bits.shape[1] < W or bits.stride(1) != 1:
        raise ValueError("out must be an int32 [B, >= ceil(V / 32)] tensor on the same device")
    _check(lib.tsa_bitmask_from_allowed(_ptr(allowed), B, V, allowed.stride(0), _ptr(bits),
                                        bits.stride(0), _stream(allowed)))
    return bits


def _mask_stride(bitmask: Optional[torch.Tensor], B: int, V: int, dev) -> int:
    if bitmask is None:
        return 0
    if bitmask.dtype != torch.int32 or bitmask.device != dev or bitmask.dim() != 2:
        raise ValueError("bitmask must be an int32 [B, W] tensor on the logits' device")
    if bitmask.shape[0] != B or bitmask.stride(1) != 1 or bitmask.shape[1] < (V + 31) // 32:
        raise ValueError("bitmask must be [B, >= ceil(V / 32)] with unit stride along W")
    return bitmask.stride(0)


def selective_log_softmax(logits: torch.Tensor, index: torch.Tensor, temperature: Param = 1.0,
                          bitmask: Optional[torch.Tensor] = None,
                          out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """selective_log_softmax, "Selective Log Softmax": one float per row, the
    log-softmax of the allowed, temperature-scaled row at ``index`` (int64
    [B]); T <= 0 uses T = 1.  -inf for a disallowed index, NaN for an index
    outside [0, V) or a row with no allowed finite logit.  Called with
    ``sample``'s tokens it gives their log-probabilities before filtering."""
    lib = load_library()
    B, V, stride = _rows(logits)
    dev = logits.device
    if index.dtype != torch.int64 or index.device != dev or index.shape != (B,) or not index.is_contiguous():
        raise ValueError("index must be a contiguous int64 [B] tensor on the logits' device")
    T, Ts = _param(temperature, B, torch.float32, dev)
    if bitmask is not None:
        if bitmask.dtype != torch.int32 or bitmask.device != dev or bitmask.dim() != 2:
            raise ValueError("bitmask must be an int32 [B, W] tensor on the logits' device")
        if bitmask.shape[0] != B or bitmask.stride(1) != 1 or bitmask.shape[1] < (V + 31) // 32:
            raise ValueError("bitmask must be [B, >= ceil(V / 32)] with unit stride along W")
        mstride = bitmask.stride(0)
    else:
        mstride = 0
    res = out if out is not None else torch.empty(B, dtype=torch.float32, device=dev)
    _check(lib.tsa_selective_log_softmax(_ptr(logits), _DT[logits.dtype], B, V, stride, _ptr(bitmask),
                                         mstride, _ptr(T), float(Ts), _ptr(index), _ptr(res),
                                         _stream(logits)))
    return res


def sample_noalloc(logits: torch.Tensor, tokens_out: torch.Tensor, temperature: Param = 1.0,
                   top_k: Param = 0, top_p: Param = 1.0, min_p: Param = 0.0, seed: int = 0,
                   offset: int = 0, bitmask: Optional[torch.Tensor] = None,
                   min_kept_out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """``sample`` for callers that cannot allocate device memory: the library
    uses its own fixed device scratch (at most
    ``sample_noalloc_max_bytes()`` of workspace), so nothing is allocated
    here; the caller passes the int64 [B] ``tokens_out`` (and optionally the
    float32 [B] ``min_kept_out``).  Calls overlapping on the GPU share that
    scratch and must not run concurrently."""
    lib = load_library()
    B, V, stride = _rows(logits)
    dev = logits.device
    T, Ts = _param(temperature, B, torch.float32, dev)
    K, Ks = _param(top_k, B, torch.int32, dev)
    Pp, Ps = _param(top_p, B, torch.float32, dev)
    M, Ms = _param(min_p, B, torch.float32, dev)
    if tokens_out is None:
        raise ValueError("tokens_out is required")
    for t, dt, name in ((tokens_out, torch.int64, "tokens_out"), (min_kept_out, torch.float32, "min_kept_out")):
        if t is not None and (t.shape != (B,) or t.dtype != dt or t.device != dev or not t.is_contiguous()):
            raise ValueError("%s must be a contiguous %s [B] tensor on %s" % (name, dt, dev))
    if bitmask is not None:
        if bitmask.dtype != torch.int32 or bitmask.device != dev or bitmask.dim() != 2:
            raise ValueError("bitmask must be an int32 [B, W] tensor on the logits' device")
        if bitmask.shape[0] != B or bitmask.stride(1) != 1 or bitmask.shape[1] < (V + 31) // 32:
            raise ValueError("bitmask must be [B, >= ceil(V / 32)] with unit stride along W")
        mstride = bitmask.stride(0)
    else:
        mstride = 0
    _check(lib.tsa_sample_noalloc(_ptr(logits), _DT[logits.dtype], B, V, stride, _ptr(bitmask),
                                  mstride, _ptr(T), float(Ts), _ptr(K), int(Ks), _ptr(Pp), float(Ps),
                                  _ptr(M), float(Ms), int(seed) & 0xFFFFFFFFFFFFFFFF,
                                  int(offset) & 0xFFFFFFFFFFFFFFFF, _ptr(tokens_out),
                                  _ptr(min_kept_out), _stream(logits)))
    return tokens_out


def sample_noalloc_max_bytes() -> int:
    """Size of the fixed scratch behind ``sample_noalloc``: a (B, V, dtype)
    whose ``tsa_sample_workspace_bytes`` exceeds it is rejected."""
    return 16 * 1024 * 1024


def lm_head_topk(hidden: torch.Tensor, weight: torch.Tensor, k: int, bias: Optional[torch.Tensor] = None):
    """lm-head-topk, "API" (the dense head): (values float32 [M, k], indices
    int64 [M, k]) of the exact top-k of hidden @ weight^T (+ bias), sorted
    descending, ties to the lower index; the score matrix is never written.
    hidden bf16 [M <= 4, H], weight bf16 [V, H] (unit stride along H)."""
    lib = load_library()
    for t, name in ((hidden, "hidden"), (weight, "weight")):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("%s must be a CUDA bfloat16 2-D tensor with unit stride along H" % name)
    M, H = hidden.shape
    V = weight.shape[0]
    if weight.shape[1] != H or weight.device != hidden.device:
        raise ValueError("weight must be [V, H] on the hidden rows' device")
    if bias is not None and (bias.dtype != torch.float32 or bias.shape != (V,) or bias.device != hidden.device
                             or not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous float32 [V] tensor on the same device")
    dev = hidden.device
    values = torch.empty(M, k, dtype=torch.float32, device=dev)
    indices = torch.empty(M, k, dtype=torch.int64, device=dev)
    nws = int(lib.tsa_lm_head_topk_workspace_bytes(M, V, k))
    ws = _workspace(nws, dev) if nws > 0 else None
    _check(lib.tsa_lm_head_topk(_ptr(hidden), M, H, hidden.stride(0), _ptr(weight), V, weight.stride(0), _ptr(bias),
                                int(k), _ptr(values), _ptr(indices), _ptr(ws), nws, _stream(hidden)))
    return values, indices


def topk(logits: torch.Tensor, k: int):
    """lm-head-topk, "API": (values float32 [B, k], indices int64 [B, k]),
    sorted by value descending, ties to the lower index; k <= 2048."""
    lib = load_library()
    B, V, stride = _rows(logits)
    values = torch.empty(B, k, dtype=torch.float32, device=logits.device)
    indices = torch.empty(B, k, dtype=torch.int64, device=logits.device)
    _check(lib.tsa_topk(_ptr(logits), _DT[logits.dtype], B, V, stride, int(k), _ptr(values),
                        _ptr(indices), None, 0, _stream(logits)))
    return values, indices


def device_status(clear: bool = True) -> int:
    """0, or TSA_ERR_DEVICE_TIMEOUT (-8) if a kernel's bounded wait ran out."""
    return int(load_library().tsa_device_status(1 if clear else 0))
