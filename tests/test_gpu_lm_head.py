"""GPU parity for the dense lm-head projection fused with top-k (lm-head-topk,
"API", "Method", "Correctness") against the oracle's float64 scores.

Rules: values are the GPU's fp32 sums of bf16 products, so each may differ
from the exact score by at most DELTA = H 2^-23 sum_h |h_h w_vh| (a bound on
fp32 accumulation).  Each returned value lies within DELTA of its index's
exact score; the returned set equals the oracle's except for entries whose
exact score is within 2 DELTA of the oracle's k-th value (near-ties that
rounding may order either way); values come sorted descending, equal values
by ascending index."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def tsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import top_sampling_apply_gb300 as lib

    lib.load_library()
    return lib


def _case(rng, M, H, V, wscale=0.05):
    h = torch.from_numpy(rng.standard_normal((M, H)).astype(np.float32)).to(torch.bfloat16)
    w = torch.from_numpy((wscale * rng.standard_normal((V, H))).astype(np.float32)).to(torch.bfloat16)
    return h, w


def _abs_dots(h, w):
    ha = np.abs(h.float().numpy().astype(np.float64))
    out = np.empty((ha.shape[0], w.shape[0]))
    for v0 in range(0, w.shape[0], 8192):
        wb = np.abs(w[v0:v0 + 8192].float().numpy().astype(np.float64))
        out[:, v0:v0 + wb.shape[0]] = ha @ wb.T
    return out


def _check(h, w, k, bias, vals_g, idx_g):
    M, H = h.shape
    _, idx_o, scores = oracle.lm_head_topk(h, w, k, bias=bias)
    delta = H * 2.0 ** -23 * _abs_dots(h, w) + (1e-6 if bias is not None else 0.0)
    vals_g, idx_g = vals_g.cpu().numpy().astype(np.float64), idx_g.cpu().numpy()
    fails = []
    for m in range(M):
        ig = idx_g[m]
        if not np.all((ig >= 0) & (ig < w.shape[0])) or len(set(ig.tolist())) != k:
            fails.append("row %d: invalid or repeated indices" % m)
            continue
        err = np.abs(vals_g[m] - scores[m, ig])
        if np.any(err > delta[m, ig]):
            j = int(np.argmax(err - delta[m, ig]))
            fails.append("row %d: value of %d off by %.3g (bound %.3g)" % (m, ig[j], err[j], delta[m, ig[j]]))
        if np.any(np.diff(vals_g[m]) > 0):
            fails.append("row %d: values not sorted descending" % m)
        same = np.diff(vals_g[m]) == 0
        if np.any(same & (np.diff(ig) < 0)):
            fails.append("row %d: equal values not in index order" % m)
        kth = scores[m, idx_o[m, -1]]
        for t in set(ig.tolist()) ^ set(idx_o[m].tolist()):
            if abs(scores[m, t] - kth) > 2 * delta[m, t] + 2 * delta[m, idx_o[m, -1]]:
                fails.append("row %d: set differs at %d (score %.9g, k-th %.9g)" % (m, t, scores[m, t], kth))
                break
    return fails


@pytest.mark.parametrize("M,H,V,k,with_bias", [(1, 512, 8192, 1, False), (2, 512, 8192, 50, True),
                                                (3, 2048, 128256, 100, False), (4, 1024, 8192 + 77, 50, True),
                                                (4, 512, 128256, 2048, False), (1, 2048, 1000, 1000, False)])
def test_lm_head_topk_matches_oracle(tsa, M, H, V, k, with_bias):
    rng = np.random.default_rng(M * 1000 + V + k)
    h, w = _case(rng, M, H, V)
    bias = torch.from_numpy(rng.standard_normal(V).astype(np.float32)) if with_bias else None
    vals, idx = tsa.lm_head_topk(h.to(DEV), w.to(DEV), k, bias=None if bias is None else bias.to(DEV))
    torch.cuda.synchronize()
    fails = _check(h, w, k, bias, vals, idx)
    assert not fails, fails[:3]
    assert tsa.device_status() == 0


def test_lm_head_topk_every_winner_in_one_chunk(tsa):
    """The page's planted test: all k winners inside one 512-entry chunk."""
    rng = np.random.default_rng(7)
    M, H, V, k = 1, 512, 16384, 100
    h, w = _case(rng, M, H, V)
    w32 = w.float()
    planted = 7 * 512 + rng.choice(512, k, replace=False)
    w32[planted] = 0.05 * h.float() * torch.from_numpy(rng.uniform(0.5, 1.5, (k, 1)).astype(np.float32))
    w = w32.to(torch.bfloat16)
    vals, idx = tsa.lm_head_topk(h.to(DEV), w.to(DEV), k)
    torch.cuda.synchronize()
    assert set(idx[0].cpu().tolist()) == set(planted.tolist())
    assert not _check(h, w, k, None, vals, idx)


def test_lm_head_topk_full_size(tsa):
    """V = 248,320, H = 5,120, k = 50 (lm-head-topk, "Measured"), one hidden row."""
    rng = np.random.default_rng(11)
    M, H, V, k = 1, 5120, 248320, 50
    h = torch.from_numpy(rng.standard_normal((M, H)).astype(np.float32)).to(torch.bfloat16)
    w = torch.empty(V, H, dtype=torch.bfloat16, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(5)
    w.normal_(0.0, 0.02, generator=g)
    vals, idx = tsa.lm_head_topk(h.to(DEV), w, k)
    torch.cuda.synchronize()
    fails = _check(h, w.cpu(), k, None, vals, idx)
    assert not fails, fails[:3]


def test_lm_head_topk_argument_checks(tsa):
    lib = tsa.load_library()
    h = torch.zeros(1, 512, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(100, 512, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(tsa.TSAError):
        tsa.lm_head_topk(h, w, 101)  # k > V
    with pytest.raises(tsa.TSAError):
        tsa.lm_head_topk(torch.zeros(5, 512, dtype=torch.bfloat16, device=DEV), w, 5)  # M > 4
    assert lib.tsa_lm_head_topk_workspace_bytes(0, 100, 5) == 0
