"""Pins for the oracle's dense lm-head top-k (lm-head-topk, "API", "Method",
"Correctness"): the scores against an explicit exactly-rounded dot product
(math.fsum) per entry, k = 1 against torch.argmax, the page's planted case
(every winner inside one 2,048-entry chunk) against torch.topk on the
materialised scores, and the bias term."""
import math

import numpy as np
import torch

import oracle


def _case(rng, M, H, V):
    h = torch.from_numpy(rng.standard_normal((M, H)).astype(np.float32)).to(torch.bfloat16)
    w = torch.from_numpy((0.05 * rng.standard_normal((V, H))).astype(np.float32)).to(torch.bfloat16)
    return h, w


def test_scores_are_exact_dot_products():
    rng = np.random.default_rng(0)
    h, w = _case(rng, 2, 64, 300)
    _, _, scores = oracle.lm_head_topk(h, w, 5)
    hf, wf = h.float().numpy().astype(np.float64), w.float().numpy().astype(np.float64)
    for m in range(2):
        for v in rng.choice(300, 40, replace=False):
            exact = math.fsum(float(a) * float(b) for a, b in zip(hf[m], wf[v]))
            assert abs(scores[m, v] - exact) <= 1e-12 * max(1.0, abs(exact))


def test_k1_is_argmax_and_planted_chunk_matches_torch_topk():
    rng = np.random.default_rng(1)
    M, H, V, k = 3, 128, 8192, 50
    h, w = _case(rng, M, H, V)
    vals, idx, scores = oracle.lm_head_topk(h, w, k)
    st = torch.from_numpy(scores)
    tv, ti = torch.topk(st, k, dim=1)
    assert torch.equal(torch.from_numpy(idx), ti)
    assert np.array_equal(vals, tv.numpy())
    v1, i1, _ = oracle.lm_head_topk(h, w, 1)
    assert torch.equal(torch.from_numpy(i1[:, 0]), torch.argmax(st, dim=1))
    # plant every winner of a one-row case in chunk 2 (entries 4,096 .. 6,143):
    # those rows point along the hidden vector
    h1 = h[:1]
    w32 = w.float()
    planted = 4096 + rng.choice(2048, 64, replace=False)
    w32[planted] = 0.25 * h1.float() * torch.from_numpy(rng.uniform(0.5, 1.5, (64, 1)).astype(np.float32))
    vals, idx, scores = oracle.lm_head_topk(h1, w32.to(torch.bfloat16), k)
    assert np.all((idx >= 4096) & (idx < 6144))
    tv, ti = torch.topk(torch.from_numpy(scores), k, dim=1)
    assert torch.equal(torch.from_numpy(idx), ti)


def test_bias_shifts_scores():
    rng = np.random.default_rng(2)
    h, w = _case(rng, 1, 32, 100)
    b = torch.from_numpy(rng.standard_normal(100).astype(np.float32))
    _, _, s0 = oracle.lm_head_topk(h, w, 3)
    _, _, s1 = oracle.lm_head_topk(h, w, 3, bias=b)
    assert np.allclose(s1 - s0, b.numpy().astype(np.float64)[None, :], rtol=0, atol=1e-12)
