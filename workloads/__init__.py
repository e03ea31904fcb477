"""Seeded synthetic inputs for per-row vocabulary selection.

This module only draws random inputs; it holds none of the selection
arithmetic, so both the CPU oracle and the GPU library can be fed from it.
Every generator is deterministic in its seed.  Tensors are returned on the CPU
(torch, so bf16 exists); callers move them to the device.

Workloads (restated from the selection problem's own benchmark shapes):
  tiny_case       B=4,    V=8,192   f32  N(0, 2^2), mask density 0.7
  decode_batch    B=256,  V=128,256 f32  3*N(0,1) + Zipf(s=1.1) log-rank head
  hetero_batch    B=1024, V=32,000  bf16 N(0, 1.5^2), per-row parameters
  topk_large      B=8,    V=248,320 f32  N(0,1), winners planted in one chunk
  peaked_batch    B=512,  V=256,000 bf16 N(0,1), one +10 token or a flat row
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Union

import numpy as np
import torch

Param = Union[float, int, torch.Tensor]


@dataclass
class SampleCase:
    name: str
    logits: torch.Tensor                  # [B, V] float32 / bfloat16 / float16, CPU
    bitmask: Optional[torch.Tensor]       # [B, ceil(V/32)] int32, CPU, or None
    temperature: Param
    top_k: Param
    top_p: Param
    min_p: Param
    seed: int = 0
    offset: int = 0
    info: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.logits.shape[0]

    @property
    def V(self) -> int:
        return self.logits.shape[1]


def mask_words(V: int) -> int:
    return (V + 31) // 32


def pack_allowed(allowed: np.ndarray) -> torch.Tensor:
    """[B, W*32] bool -> [B, W] int32, token i at bit (i & 31) of word i >> 5.
    Uses numpy.packbits (little bit order) and a little-endian word view."""
    B, nbits = allowed.shape
    assert nbits % 32 == 0
    packed = np.packbits(allowed.astype(np.uint8), axis=1, bitorder="little")
    words = packed.reshape(B, nbits // 32, 4).copy().view("<u4").reshape(B, nbits // 32)
    return torch.from_numpy(words.astype(np.uint32).view(np.int32).copy())


def random_bitmask(rng: np.random.Generator, B: int, V: int, density, force_one=True,
                   force_index: Optional[np.ndarray] = None) -> torch.Tensor:
    """Each bit allowed with probability ``density`` (scalar or per-row).  Bits
    at or beyond V are random too (the library must ignore them).  With
    ``force_one``, a row with no allowed token below V gets one random bit;
    ``force_index[b] >= 0`` forces that token allowed."""
    W = mask_words(V)
    dens = np.broadcast_to(np.asarray(density, dtype=np.float64), (B,))
    allowed = rng.random((B, W * 32)) < dens[:, None]
    if force_index is not None:
        for b in range(B):
            if force_index[b] >= 0:
                allowed[b, force_index[b]] = True
    if force_one:
        for b in range(B):
            if not allowed[b, :V].any():
                allowed[b, rng.integers(0, V)] = True
    return pack_allowed(allowed)


def tiny_case(seed: int = 0) -> SampleCase:
    """B=4, V=8,192, f32 N(0, 2^2); mask density 0.7 with one allowed token
    forced; T=0.7, top_k=50, top_p=0.9, min_p=0.05, seed=1, offset=0."""
    rng = np.random.default_rng(seed)
    B, V = 4, 8192
    logits = torch.from_numpy((2.0 * rng.standard_normal((B, V))).astype(np.float32))
    mask = random_bitmask(rng, B, V, 0.7)
    return SampleCase("tiny", logits, mask, 0.7, 50, 0.9, 0.05, seed=1, offset=0,
                      info={"topk_k": 10})


def zipf_rows(rng: np.random.Generator, B: int, V: int, s: float = 1.1,
              noise: float = 3.0) -> np.ndarray:
    """noise*N(0,1) plus a Zipf(s) log-rank head: the token of rank r (r = 1..V,
    a fresh random permutation per row) gets -s*ln(r)."""
    head = -s * np.log(np.arange(1, V + 1, dtype=np.float64))
    out = noise * rng.standard_normal((B, V))
    for b in range(B):
        out[b, rng.permutation(V)] += head
    return out.astype(np.float32)


DECODE_MODES = {
    # name: (temperature, top_k, top_p, min_p)
    "greedy": (0.0, 0, 1.0, 0.0),
    "unfiltered": (1.0, 0, 1.0, 0.0),
    "top_k": (1.0, 50, 1.0, 0.0),
    "top_p": (1.0, 0, 0.9, 0.0),
    "combined": (1.0, 50, 0.9, 0.05),
}


def decode_batch(mode: str = "combined", mask_density: Optional[float] = 0.7, B: int = 256,
                 V: int = 128256, seed: int = 0, rows: Optional[int] = None) -> SampleCase:
    """Decode batch: B=256, V=128,256, f32 3*N(0,1) + Zipf(1.1) head.  The
    fused headline adds a per-row mask at density 0.7; ``mask_density=None``
    gives the unmasked runs.  ``rows`` generates only the first rows (same
    values as the full batch)."""
    rng = np.random.default_rng(seed)
    nb = B if rows is None else rows
    logits = torch.from_numpy(zipf_rows(rng, nb, V))
    mask = None
    if mask_density is not None:
        mrng = np.random.default_rng(seed + 1)
        mask = random_bitmask(mrng, nb, V, mask_density)
    T, k, p, mp = DECODE_MODES[mode]
    return SampleCase("decode_" + mode, logits, mask, T, k, p, mp, seed=0, offset=0,
                      info={"mode": mode, "mask_density": mask_density})


def hetero_batch(seed: int = 0, B: int = 1024, V: int = 32000) -> SampleCase:
    """Heterogeneous continuous batch: bf16 N(0, 1.5^2); per-row T ~ U[0.3,1.5]
    with 10% of rows greedy (T=0); top_k uniform over {0..100}; top_p ~
    U[0.5,1]; min_p from {0, 0.02, 0.1}; mask density from {1%, 50%, 100%};
    5% of rows have the row maximum repeated at 2-4 indices in total."""
    rng = np.random.default_rng(seed)
    x = (1.5 * rng.standard_normal((B, V))).astype(np.float32)
    logits = torch.from_numpy(x).to(torch.bfloat16)
    T = rng.uniform(0.3, 1.5, B).astype(np.float32)
    T[rng.random(B) < 0.10] = 0.0
    top_k = rng.integers(0, 101, B).astype(np.int32)
    top_p = rng.uniform(0.5, 1.0, B).astype(np.float32)
    min_p = rng.choice(np.array([0.0, 0.02, 0.1], dtype=np.float32), B)
    dens = rng.choice(np.array([0.01, 0.5, 1.0]), B)
    mask = random_bitmask(rng, B, V, dens)
    dup_rows = np.nonzero(rng.random(B) < 0.05)[0]
    lv = logits.view(torch.int16)  # exact bit copies of the bf16 maximum
    for b in dup_rows:
        row = logits[b].float()
        amax = int(torch.argmax(row))
        copies = int(rng.integers(2, 5)) - 1
        others = rng.choice(np.setdiff1d(np.arange(V), [amax]), copies, replace=False)
        for j in others:
            lv[b, int(j)] = lv[b, amax]
    return SampleCase("hetero", logits, mask, torch.from_numpy(T), torch.from_numpy(top_k),
                      torch.from_numpy(top_p), torch.from_numpy(min_p), seed=0, offset=0,
                      info={"dup_rows": dup_rows.tolist()})


CHUNK = 2048


def topk_large(k: int, seed: int = 0, B: int = 8, V: int = 248320):
    """Exact top-k at a large vocabulary: f32 N(0,1), B=8, V=248,320 (121 full
    2,048-entry chunks and a 512-wide ragged one).  Rows 0..B/2-1 get +8.0 on k
    distinct positions of one random chunk-aligned 2,048-wide span.  In every
    row the k-th largest value is copied to one lower and one higher index
    outside the top k, so ties must resolve to the lower index."""
    rng = np.random.default_rng(seed + 1000 * k)
    x = rng.standard_normal((B, V)).astype(np.float32)
    nfull = V // CHUNK
    planted = []
    for b in range(B // 2):
        c = int(rng.integers(0, nfull))
        pos = c * CHUNK + rng.choice(CHUNK, min(k, CHUNK), replace=False)
        x[b, pos] += np.float32(8.0)
        planted.append((b, c))
    for b in range(B):
        order = np.lexsort((np.arange(V), -x[b].astype(np.float64)))
        ik = int(order[k - 1])
        vk = x[b, ik]
        rest = order[k:]
        lower = rest[rest < ik]
        higher = rest[rest > ik]
        if lower.size:
            x[b, int(rng.choice(lower))] = vk
        if higher.size:
            x[b, int(rng.choice(higher))] = vk
    return torch.from_numpy(x), {"planted": planted}


def peaked_batch(seed: int = 0, B: int = 512, V: int = 256000, rows: Optional[int] = None
                 ) -> SampleCase:
    """Large peaked batch: bf16 N(0,1); 90% of rows have one random token set
    to +10 (that token is kept allowed by the mask), 10% are flat (all 0.0);
    per-row mask at density 0.3; T=0.8, top_k=0, top_p=0.95, min_p=0.05."""
    rng = np.random.default_rng(seed)
    nb = B if rows is None else rows
    x = rng.standard_normal((nb, V)).astype(np.float32)
    flat = rng.random(nb) < 0.10
    peak = np.full(nb, -1, dtype=np.int64)
    for b in range(nb):
        if flat[b]:
            x[b, :] = 0.0
        else:
            peak[b] = int(rng.integers(0, V))
            x[b, peak[b]] = 10.0
    logits = torch.from_numpy(x).to(torch.bfloat16)
    mask = random_bitmask(rng, nb, V, 0.3, force_index=peak)
    return SampleCase("peaked", logits, mask, 0.8, 0, 0.95, 0.05, seed=0, offset=0,
                      info={"flat_rows": np.nonzero(flat)[0].tolist()})
