"""GPU-vs-oracle comparison under the selection tolerance rules.

Rules (all against the CPU oracle on the same seeded inputs):
  * greedy tokens (T <= 0 or top_k == 1), bitmask output, top-k keep sets and
    topk indices / values: bit-exact;
  * top-p / min-p keep sets: equal except tokens whose mass strictly above
    (top-p) or relative weight (min-p) lies within 1e-6 of the cut;
  * sampled tokens: equal, except rows whose two best perturbed scores differ
    by less than 1e-5, or whose keep sets differ (by exempt tokens only) in a
    way that includes either side's winner.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

MASS_BAND = 1e-6
GAP_BAND = 1e-5


def allowed_matrix(bitmask, V):
    if bitmask is None:
        return None
    m = bitmask.cpu().numpy() if isinstance(bitmask, torch.Tensor) else bitmask
    return np.unpackbits(np.ascontiguousarray(m).view(np.uint8), axis=1,
                         bitorder="little")[:, :V].astype(bool)


def per_row(x, B, dtype):
    if isinstance(x, torch.Tensor) and x.dim() == 1:
        return x.cpu().numpy().astype(dtype)
    v = x.item() if isinstance(x, torch.Tensor) else x
    return np.full(B, v, dtype=dtype)


def check_sample(logits_cpu, bitmask_cpu, T, K, P, MP, seed, offset, tok_g, vstar_g,
                 nthreads=8, rows=None, sequential=False):
    """Returns a list of failure strings (empty when the GPU result passes)."""
    B, V = logits_cpu.shape
    if rows is not None:
        logits_cpu = logits_cpu[rows]
        bitmask_cpu = None if bitmask_cpu is None else bitmask_cpu[rows]
        T, K, P, MP = [x[rows] if isinstance(x, torch.Tensor) and x.dim() == 1 else x
                       for x in (T, K, P, MP)]
        tok_g, vstar_g = tok_g[rows], vstar_g[rows]
        row_ids = np.asarray(rows)
    else:
        row_ids = np.arange(B)
    # the oracle keys every draw by the row's index in the launched batch
    fails = []
    n = logits_cpu.shape[0]
    Tn = per_row(T, n, np.float32)
    Kn = per_row(K, n, np.int32)
    Pn = per_row(P, n, np.float32)
    Mn = per_row(MP, n, np.float32)
    l = logits_cpu.double().numpy()
    allowed = allowed_matrix(bitmask_cpu, V)
    finite = np.isfinite(l) if allowed is None else (np.isfinite(l) & allowed)
    tok_o = np.zeros(n, np.int64)
    vstar_o = np.zeros(n)
    gap_o = np.zeros(n)
    if rows is None:
        tok_o, vstar_o, gap_o = oracle.sample(logits_cpu, Tn, Kn, Pn, Mn, seed, offset,
                                              bitmask=bitmask_cpu, nthreads=nthreads,
                                              sequential=sequential)
    else:
        for j, b in enumerate(row_ids):
            d = oracle.sample_row_detail(l[j], Tn[j], int(Kn[j]), Pn[j], Mn[j], seed, offset, int(b),
                                         mask_row=None if bitmask_cpu is None
                                         else bitmask_cpu[j].numpy(), sequential=sequential)
            tok_o[j], vstar_o[j], gap_o[j] = d["token"], d["vstar"], d["gap"]
    tok_g = tok_g.cpu().numpy() if isinstance(tok_g, torch.Tensor) else tok_g
    vstar_g = vstar_g.cpu().double().numpy() if isinstance(vstar_g, torch.Tensor) else vstar_g
    for j in range(n):
        b = int(row_ids[j])
        greedy = not (Tn[j] > 0) or Kn[j] == 1
        if tok_o[j] < 0:
            if tok_g[j] != -1:
                fails.append("row %d: empty row gave %d" % (b, tok_g[j]))
            continue
        if greedy:
            if tok_g[j] != tok_o[j]:
                fails.append("row %d: greedy %d != %d" % (b, tok_g[j], tok_o[j]))
            if vstar_g[j] != vstar_o[j]:
                fails.append("row %d: greedy max %r != %r" % (b, vstar_g[j], vstar_o[j]))
            continue
        kg = finite[j] & (l[j] >= vstar_g[j])
        ko = finite[j] & (l[j] >= vstar_o[j])
        if not (0 <= tok_g[j] < V) or not kg[tok_g[j]]:
            fails.append("row %d: token %d outside its own keep set" % (b, tok_g[j]))
            continue
        diff = kg ^ ko
        if diff.any():
            p_on, m_on = Pn[j] < 1, Mn[j] > 0
            if not (p_on or m_on):
                fails.append("row %d: top-k keep set differs (%d tokens)" % (b, diff.sum()))
                continue
            mrow = None if bitmask_cpu is None else bitmask_cpu[j].numpy()
            d = oracle.sample_row_detail(l[j], Tn[j], int(Kn[j]), Pn[j], Mn[j], seed, offset, b,
                                         mask_row=mrow, sequential=sequential)
            ex = np.zeros(V, bool)
            if p_on:
                ex |= np.abs(d["M"] - Pn[j]) < MASS_BAND
            if m_on:
                ex |= np.abs(d["w"] - Mn[j]) < MASS_BAND
            bad = diff & ~ex
            if bad.any():
                i = int(np.nonzero(bad)[0][0])
                fails.append("row %d: keep sets differ at %d (M=%.9g w=%.9g, %d tokens)"
                             % (b, i, d["M"][i], d["w"][i], bad.sum()))
                continue
        if tok_g[j] != tok_o[j]:
            if gap_o[j] < GAP_BAND:
                continue
            if diff.any() and (diff[tok_g[j]] or diff[tok_o[j]]):
                continue
            fails.append("row %d: token %d != oracle %d (gap %.3g)" % (b, tok_g[j], tok_o[j], gap_o[j]))
    return fails
