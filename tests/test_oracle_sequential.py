"""Pins for the oracle's sequential reading of top-p (logits-processor's opening:
the transformers processor chain, where top-p sees the softmax renormalised
over the top-k survivors) against a closed form, the intersection reading it
must reduce to, a subset property, and brute force: the chain written as
explicit masks with scipy's softmax on tiny rows with ties."""
import numpy as np
import pytest
from scipy.special import softmax

import oracle


def _vstar(x, T, K, P, MP, sequential):
    _, vs, _ = oracle.sample(x[None, :], T, K, P, MP, seed=0, sequential=sequential)
    return vs[0]


def test_sequential_closed_form():
    """Logits 2, 1, 0, -1 at T = 1, top_k = 2, top_p = 0.7.  Over the full
    softmax the mass above the second token is 0.644 < 0.7, so both survive;
    renormalised over the two survivors it is 0.731 >= 0.7, so only the first."""
    x = np.array([2.0, 1.0, 0.0, -1.0])
    assert _vstar(x, 1.0, 2, 0.7, 0.0, False) == 1.0
    assert _vstar(x, 1.0, 2, 0.7, 0.0, True) == 2.0


def test_sequential_reduces_to_intersection_without_top_k_or_top_p():
    rng = np.random.default_rng(0)
    for _ in range(50):
        x = (2 * rng.standard_normal(300)).astype(np.float32).astype(np.float64)
        T = float(rng.uniform(0.5, 1.5))
        P = float(rng.uniform(0.3, 1.0))
        MP = float(rng.choice([0.0, 0.05]))
        assert _vstar(x, T, 0, P, MP, True) == _vstar(x, T, 0, P, MP, False)
        K = int(rng.integers(1, 100))
        assert _vstar(x, T, K, 1.0, MP, True) == _vstar(x, T, K, 1.0, MP, False)


def test_sequential_keep_set_inside_intersection_keep_set():
    rng = np.random.default_rng(1)
    for _ in range(100):
        x = (2 * rng.standard_normal(200)).astype(np.float32).astype(np.float64)
        T, K, P = float(rng.uniform(0.5, 1.5)), int(rng.integers(2, 60)), float(rng.uniform(0.3, 0.99))
        assert _vstar(x, T, K, P, 0.0, True) >= _vstar(x, T, K, P, 0.0, False)


def _chain_vstar(x, T, K, P, MP):
    """The processor chain on one row, mask by mask: temperature, top-k (ties at
    the k-th value kept), top-p on the softmax renormalised over the survivors
    (a token is kept while the mass of strictly larger survivors is < p; the
    largest always), then min-p (relative to the largest probability)."""
    n = len(x)
    keep = np.ones(n, bool)
    if 1 <= K < n:
        kth = np.sort(x)[::-1][K - 1]
        keep &= x >= kth
    if P < 1.0:
        p = np.zeros(n)
        p[keep] = softmax(x[keep] / T)
        above = np.array([p[keep & (x > x[i])].sum() for i in range(n)])
        keep &= (above < P) | (x == x[keep].max())
    if MP > 0.0:
        p = softmax(x / T)
        keep &= p >= MP * p.max()
    return x[keep].min()


@pytest.mark.parametrize("seed", range(6))
def test_sequential_matches_the_chain_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    for _ in range(200):
        n = int(rng.integers(2, 9))
        x = rng.integers(-3, 4, n).astype(np.float64) * 0.5  # small integers: many ties
        T = float(np.float32(rng.uniform(0.4, 1.6)))
        K = int(rng.integers(0, n + 1))
        P = float(np.float32(rng.uniform(0.2, 1.0)))
        MP = float(np.float32(rng.choice([0.0, 0.1, 0.3])))
        assert _vstar(x, T, K, P, MP, True) == _chain_vstar(x, T, K, P, MP), (x, T, K, P, MP)
