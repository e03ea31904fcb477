"""CPU oracle for per-row vocabulary selection -- TEST INFRASTRUCTURE ONLY.

A plain, slow, double-precision restatement of the calls the GPU library
exports (``apply_token_bitmask``, ``sample``, ``topk``, ``bitmask_from_allowed``,
``sample_icdf`` written in C in
``tsa_oracle.c`` and loaded here with ctypes; ``selective_log_softmax`` in
numpy float64 below).  It fully sorts every row and
computes cumulative masses as explicit running sums.  It shares no code with
the CUDA path, and only the tests, the package smoke check and the benchmark's
CPU baseline / reference arm may import it: the product never does.

Each function cites the page passage it follows (page title, section):
  * logits-processor, "API" / "Method"   -- bitmask, sample
  * logits-mask-xpu, "Method"            -- top_k == 1 is argmax; the inverse-CDF draw
  * logits-mask-xpu, "Usage"             -- bitmask_from_allowed; a caller uniform per row
  * lm-head-topk, "API" / "Method"       -- exact sorted top-k; the dense head's scores
  * selective_log_softmax, "Selective Log Softmax" -- log-probability at an index
  * Salmon et al., SC'11                 -- Philox4x32-10

Pins: every function here is checked against something other than itself in
``tests/test_oracle_*.py`` (torch.argmax / torch.topk on the CPU, brute force on
tiny rows, closed forms, an independent Philox implementation, mpmath).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tsa_oracle.c")
_LIB = os.path.join(_HERE, "libtsa_oracle.so")
_lock = threading.Lock()
_lib = None

DT_F32, DT_F16, DT_BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (plain -O2, no ISA flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, u64, u32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64, ctypes.c_uint32
        dbl = ctypes.c_double
        lib.tsao_philox4x32_10.argtypes = [P, P, P]
        lib.tsao_philox4x32_10.restype = None
        lib.tsao_rand_word.argtypes = [u64, u64, i64, i64]
        lib.tsao_rand_word.restype = u32
        lib.tsao_rand_words.argtypes = [u64, u64, i64, i64, i64, P]
        lib.tsao_rand_words.restype = None
        lib.tsao_uniform.argtypes = [u32]
        lib.tsao_uniform.restype = dbl
        lib.tsao_gumbel.argtypes = [u32]
        lib.tsao_gumbel.restype = dbl
        lib.tsao_apply_token_bitmask.argtypes = [P, ctypes.c_int, i64, i64, i64, P, i64]
        lib.tsao_apply_token_bitmask.restype = ctypes.c_int
        lib.tsao_sample.argtypes = [P, i64, i64, i64, P, i64, P, P, P, P, u64, u64, P, P, P,
                                    ctypes.c_int, ctypes.c_int]
        lib.tsao_sample.restype = ctypes.c_int
        lib.tsao_sample_row_detail.argtypes = [P, i64, P, dbl, i32, dbl, dbl, u64, u64, i64, P,
                                               P, P, P, P, ctypes.c_int]
        lib.tsao_sample_row_detail.restype = ctypes.c_int
        lib.tsao_topk.argtypes = [P, i64, i64, i64, i32, P, P, ctypes.c_int]
        lib.tsao_topk.restype = ctypes.c_int
        lib.tsao_bitmask_from_allowed.argtypes = [P, i64, i64, i64, P, i64]
        lib.tsao_bitmask_from_allowed.restype = ctypes.c_int
        lib.tsao_sample_icdf.argtypes = [P, i64, i64, i64, P, i64, P, P, P, P, P, P, P, P, P,
                                         ctypes.c_int]
        lib.tsao_sample_icdf.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(status: int, what: str):
    if status != 0:
        raise ValueError("oracle %s failed with status %d" % (what, status))


def selective_log_softmax(logits, index, temperature=1.0, bitmask=None) -> np.ndarray:
    """selective_log_softmax, "Selective Log Softmax": per row, the logit at
    ``index`` less the row's log-sum-exp, here over the allowed tokens of the
    temperature-scaled row, in float64:
        out[b] = (l[b, i] - m) / T - ln sum_{j allowed} exp((l[b, j] - m) / T),
    m the row's largest allowed logit.  T <= 0 is taken as 1 (the page's
    unscaled definition).  NaN logits count as -inf; a disallowed index gives
    -inf; an index outside [0, V) or a row with no allowed finite logit gives
    NaN.  ``bitmask``: int32 [B, >= ceil(V / 32)], bit 1 = allowed."""
    x = _as_f64_rows(logits)
    B, V = x.shape
    T = _per_row(temperature, B, np.float32, np.float64)
    idx = np.asarray(index.cpu().numpy() if hasattr(index, "cpu") else index, dtype=np.int64).reshape(B)
    allowed = np.ones((B, V), dtype=bool)
    if bitmask is not None:
        words = np.ascontiguousarray(
            np.asarray(bitmask.cpu().numpy() if hasattr(bitmask, "cpu") else bitmask).astype(np.uint32))
        # bit j & 31 of word j >> 5 (little-endian words, so byte-wise little-endian bits)
        allowed = np.unpackbits(words.view(np.uint8), axis=1, bitorder="little")[:, :V].astype(bool)
    out = np.empty(B, dtype=np.float64)
    for b in range(B):
        row = np.where(np.isnan(x[b]) | ~allowed[b], -np.inf, x[b])
        t = T[b] if T[b] > 0 else 1.0
        i = int(idx[b])
        if not (0 <= i < V) or not np.any(row > -np.inf):
            out[b] = np.nan
            continue
        m = row.max()
        if row[i] == -np.inf:
            out[b] = -np.inf
            continue
        z = np.sum(np.exp((row[row > -np.inf] - m) / t))
        out[b] = (row[i] - m) / t - np.log(z)
    return out


def _as_f64_rows(logits) -> np.ndarray:
    """Widen a [B, V] float array (numpy or torch CPU, any float dtype) to
    float64; the widening from f32 / f16 / bf16 is exact."""
    try:
        import torch

        if isinstance(logits, torch.Tensor):
            return np.ascontiguousarray(logits.detach().cpu().to(torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(logits, dtype=np.float64))


def _per_row(x, B: int, dtype, np_dtype):
    """A sampling parameter given as a scalar or a length-B sequence, rounded
    through the GPU's parameter type (float32 / int32) and widened back."""
    a = np.asarray(x.cpu().numpy() if hasattr(x, "cpu") else x)
    if a.ndim == 0:
        a = np.full(B, a.item())
    a = a.astype(dtype).astype(np_dtype)
    if a.shape != (B,):
        raise ValueError("per-row parameter must be a scalar or have shape [B]")
    return np.ascontiguousarray(a)


# --------------------------------------------------------------------------
def philox4x32_10(counter, key) -> np.ndarray:
    """Philox4x32-10 block function (Salmon et al., SC'11)."""
    lib = _load()
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    lib.tsao_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def rand_word(seed: int, offset: int, row: int, index: int) -> int:
    """Random word of token ``index`` in ``row`` for draw (seed, offset)."""
    return int(_load().tsao_rand_word(seed, offset, row, index))


def rand_words(seed: int, offset: int, row: int, start: int, n: int) -> np.ndarray:
    """Random words of tokens start .. start + n - 1 in ``row``."""
    out = np.zeros(n, dtype=np.uint32)
    _load().tsao_rand_words(seed, offset, row, start, n, _ptr(out))
    return out


def uniform(x: int) -> float:
    return float(_load().tsao_uniform(x))


def gumbel(x: int) -> float:
    return float(_load().tsao_gumbel(x))


def apply_token_bitmask(logits: np.ndarray, bitmask: np.ndarray, dtype_code: int) -> np.ndarray:
    """logits-processor, "API": return a copy of ``logits`` (a [B, V] array of
    raw element bits: uint32 for f32, uint16 for f16 / bf16) with disallowed
    entries replaced by the dtype's -inf bit pattern."""
    lib = _load()
    out = np.ascontiguousarray(logits).copy()
    B, V = out.shape
    m = np.ascontiguousarray(bitmask, dtype=np.int32)
    _check(lib.tsao_apply_token_bitmask(_ptr(out), dtype_code, B, V, V, _ptr(m), m.shape[1]),
           "apply_token_bitmask")
    return out


def sample(logits, temperature, top_k, top_p, min_p, seed: int, offset: int = 0,
           bitmask=None, nthreads: int = 1, sequential: bool = False):
    """logits-processor, "API": one token per row.  Returns (tokens int64 [B],
    vstar float64 [B] = smallest kept logit, gap float64 [B] = best minus
    second-best perturbed score in the keep set).  ``sequential`` takes top-p
    over the renormalised top-k survivors (logits-processor's opening: the
    transformers processor chain) instead of the full softmax."""
    lib = _load()
    x = _as_f64_rows(logits)
    B, V = x.shape
    T = _per_row(temperature, B, np.float32, np.float64)
    K = _per_row(top_k, B, np.int32, np.int32)
    Pp = _per_row(top_p, B, np.float32, np.float64)
    Mp = _per_row(min_p, B, np.float32, np.float64)
    if bitmask is not None:
        m = np.ascontiguousarray(np.asarray(bitmask.cpu().numpy() if hasattr(bitmask, "cpu")
                                            else bitmask, dtype=np.int32))
        mp, ms = _ptr(m), m.shape[1]
    else:
        m, mp, ms = None, None, 0
    tokens = np.zeros(B, dtype=np.int64)
    vstar = np.zeros(B, dtype=np.float64)
    gap = np.zeros(B, dtype=np.float64)
    _check(lib.tsao_sample(_ptr(x), B, V, V, mp, ms, _ptr(T), _ptr(K), _ptr(Pp), _ptr(Mp),
                           seed, offset, _ptr(tokens), _ptr(vstar), _ptr(gap), nthreads,
                           1 if sequential else 0),
           "sample")
    return tokens, vstar, gap


def sample_row_detail(row, temperature: float, top_k: int, top_p: float, min_p: float,
                      seed: int, offset: int, b: int, mask_row=None, sequential: bool = False) -> dict:
    """Every intermediate of one row of ``sample`` (for tolerance rules):
    token, m, Z, v_k, v_p, v_m, vstar, gap, n_allowed, n_kept, and per token
    M (mass strictly above, as a probability) and w = exp((l - m) / T)."""
    lib = _load()
    x = _as_f64_rows(np.asarray(row)[None, :] if isinstance(row, np.ndarray) else row.reshape(1, -1))[0]
    x = np.ascontiguousarray(x)
    V = x.shape[0]
    T = float(np.float32(temperature))
    p = float(np.float32(top_p))
    mp = float(np.float32(min_p))
    if mask_row is not None:
        mr = np.ascontiguousarray(np.asarray(mask_row, dtype=np.int32))
        mptr = _ptr(mr)
    else:
        mr, mptr = None, None
    token = np.zeros(1, dtype=np.int64)
    out7 = np.zeros(7, dtype=np.float64)
    counts = np.zeros(2, dtype=np.int64)
    M = np.zeros(V, dtype=np.float64)
    w = np.zeros(V, dtype=np.float64)
    _check(lib.tsao_sample_row_detail(_ptr(x), V, mptr, T, int(top_k), p, mp, seed, offset, b,
                                      _ptr(token), _ptr(out7), _ptr(counts), _ptr(M), _ptr(w),
                                      1 if sequential else 0),
           "sample_row_detail")
    return dict(token=int(token[0]), m=out7[0], Z=out7[1], v_k=out7[2], v_p=out7[3],
                v_m=out7[4], vstar=out7[5], gap=out7[6], n_allowed=int(counts[0]),
                n_kept=int(counts[1]), M=M, w=w)


def bitmask_from_allowed(allowed) -> np.ndarray:
    """logits-mask-xpu, "Usage": pack a [B, V] bool allow-set into [B, ceil(V/32)]
    int32 words, token i at bit i mod 32 of word i // 32, the bits past V zero."""
    lib = _load()
    a = np.ascontiguousarray(np.asarray(allowed.cpu().numpy() if hasattr(allowed, "cpu") else allowed,
                                        dtype=bool)).view(np.uint8)
    B, V = a.shape
    out = np.zeros((B, (V + 31) // 32), dtype=np.int32)
    _check(lib.tsao_bitmask_from_allowed(_ptr(a), B, V, V, _ptr(out), out.shape[1]), "bitmask_from_allowed")
    return out


def sample_icdf(logits, temperature, top_k, top_p, min_p, uniform, bitmask=None, nthreads: int = 1,
                with_cum: bool = False):
    """logits-mask-xpu, "Method" / "Usage": the inverse-CDF draw from a caller
    uniform u per row over the keep set of ``sample`` (index order, weights
    exp((l - m) / T)).  Returns (tokens int64 [B], vstar float64 [B], W float64
    [B] = the kept total weight, and with ``with_cum`` the running sums float64
    [B, V] at kept tokens, NaN elsewhere)."""
    lib = _load()
    x = _as_f64_rows(logits)
    B, V = x.shape
    T = _per_row(temperature, B, np.float32, np.float64)
    K = _per_row(top_k, B, np.int32, np.int32)
    Pp = _per_row(top_p, B, np.float32, np.float64)
    Mp = _per_row(min_p, B, np.float32, np.float64)
    U = _per_row(uniform, B, np.float32, np.float64)
    if bitmask is not None:
        m = np.ascontiguousarray(np.asarray(bitmask.cpu().numpy() if hasattr(bitmask, "cpu")
                                            else bitmask, dtype=np.int32))
        mp, ms = _ptr(m), m.shape[1]
    else:
        m, mp, ms = None, None, 0
    tokens = np.zeros(B, dtype=np.int64)
    vstar = np.zeros(B, dtype=np.float64)
    W = np.zeros(B, dtype=np.float64)
    cum = np.zeros((B, V), dtype=np.float64) if with_cum else None
    _check(lib.tsao_sample_icdf(_ptr(x), B, V, V, mp, ms, _ptr(T), _ptr(K), _ptr(Pp), _ptr(Mp), _ptr(U),
                                _ptr(tokens), _ptr(vstar), _ptr(W), _ptr(cum) if with_cum else None,
                                nthreads), "sample_icdf")
    return (tokens, vstar, W, cum) if with_cum else (tokens, vstar, W)


def lm_head_topk(hidden, weight, k: int, bias=None, nthreads: int = 1):
    """lm-head-topk, "API" / "Method" (the dense head): the exact top-k of the
    vocabulary projection scores = hidden @ weight^T (+ bias), without the
    GPU's chunking: the scores in float64 (a library matmul on the exactly
    widened bf16 inputs), then ``topk`` on them.  hidden [M, H], weight [V, H],
    bias [V] or None.  Returns (values float64 [M, k], indices int64 [M, k],
    scores float64 [M, V])."""
    h = np.asarray(hidden.float().cpu().numpy() if hasattr(hidden, "cpu") else hidden, dtype=np.float64)
    V = weight.shape[0]
    scores = np.empty((h.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, 8192):  # widened a block of rows at a time (a full bf16 head is 2.5 GB)
        wb = weight[v0:v0 + 8192]
        wb = np.asarray(wb.float().cpu().numpy() if hasattr(wb, "cpu") else wb, dtype=np.float64)
        scores[:, v0:v0 + wb.shape[0]] = h @ wb.T
    if bias is not None:
        scores = scores + np.asarray(bias.float().cpu().numpy() if hasattr(bias, "cpu") else bias,
                                     dtype=np.float64)[None, :]
    vals, idx = topk(scores, k, nthreads=nthreads)
    return vals, idx, scores


def topk(logits, k: int, nthreads: int = 1):
    """lm-head-topk, "API": (values float64 [B, k], indices int64 [B, k]),
    sorted by value descending, ties to the lower index."""
    lib = _load()
    x = _as_f64_rows(logits)
    B, V = x.shape
    values = np.zeros((B, k), dtype=np.float64)
    indices = np.zeros((B, k), dtype=np.int64)
    _check(lib.tsao_topk(_ptr(x), B, V, V, k, _ptr(values), _ptr(indices), nthreads), "topk")
    return values, indices
