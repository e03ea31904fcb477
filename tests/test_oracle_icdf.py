"""Pins for the oracle's allow-set packer and inverse-CDF draw (logits-mask-xpu,
"Usage" and "Method") against what the pages and the mathematics fix:
numpy.packbits in little bit order (a library routine for the same packing),
a round trip through the pinned apply_token_bitmask oracle, the keep set of the
pinned sample oracle, closed forms (two tokens whose weights are 3:1), the
draw's first and only kept tokens, and the inverse-CDF law: uniform u mapped
through the draw lands on token i with probability w_i / W."""
import math

import numpy as np
import pytest

import oracle


def _allowed(rng, B, V, density):
    return rng.random((B, V)) < density


@pytest.mark.parametrize("V", [1, 31, 32, 33, 100, 1000])
def test_bitmask_from_allowed_matches_packbits(V):
    rng = np.random.default_rng(V)
    a = _allowed(rng, 5, V, 0.4)
    bits = oracle.bitmask_from_allowed(a)
    W = (V + 31) // 32
    padded = np.zeros((5, W * 32), dtype=bool)
    padded[:, :V] = a
    ref = np.packbits(padded, axis=1, bitorder="little").view("<u4").astype(np.uint32).view(np.int32)
    assert bits.shape == (5, W)
    assert np.array_equal(bits, ref)


def test_bitmask_from_allowed_round_trip_through_apply():
    """Applying the packed words masks exactly the disallowed tokens."""
    rng = np.random.default_rng(3)
    B, V = 4, 77
    a = _allowed(rng, B, V, 0.5)
    x = rng.standard_normal((B, V)).astype(np.float32)
    out = oracle.apply_token_bitmask(x.view(np.uint32), oracle.bitmask_from_allowed(a), oracle.DT_F32)
    y = out.view(np.float32)
    assert np.array_equal(np.isneginf(y), ~a)
    assert np.array_equal(y[a], x[a])


def test_icdf_closed_form_two_tokens():
    """Weights 1 and 1/3 (logits ln 3 and 0 at T = 1): the boundary sits at
    u = 3/4 when the heavier token comes first, at u = 1/4 when it comes last."""
    x = np.array([[math.log(3.0), 0.0], [0.0, math.log(3.0)]], dtype=np.float64)
    for u, want in [(0.0, [0, 0]), (0.2, [0, 0]), (0.3, [0, 1]), (0.74, [0, 1]), (0.76, [1, 1]),
                    (0.999, [1, 1])]:
        tok, vstar, W = oracle.sample_icdf(x, 1.0, 0, 1.0, 0.0, [u, u])
        assert list(tok) == want, (u, tok)
        assert np.allclose(W, 4.0 / 3.0)


def test_icdf_first_and_only_kept_tokens():
    rng = np.random.default_rng(5)
    V = 200
    x = rng.standard_normal((3, V))
    a = _allowed(rng, 3, V, 0.3)
    a[2] = False
    a[2, 123] = True  # one allowed token
    bits = oracle.bitmask_from_allowed(a)
    tok, vstar, W = oracle.sample_icdf(x, 0.7, 0, 1.0, 0.0, [0.0, 0.0, 0.0], bitmask=bits)
    first = [int(np.nonzero(a[b])[0][0]) for b in range(3)]
    assert list(tok) == first  # u = 0: the first kept token in index order
    for u in (0.25, 0.5, 0.9999):
        t2, _, _ = oracle.sample_icdf(x[2:], 0.7, 0, 1.0, 0.0, [u], bitmask=bits[2:])
        assert t2[0] == 123


def test_icdf_keep_set_is_sample_keep_set():
    """The draw's vstar is sample's, and every token drawn lies in that keep set."""
    rng = np.random.default_rng(11)
    B, V = 16, 500
    x = (2 * rng.standard_normal((B, V))).astype(np.float32)
    bits = oracle.bitmask_from_allowed(_allowed(rng, B, V, 0.6))
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    K = rng.integers(0, 60, B).astype(np.int32)
    P = rng.uniform(0.5, 1.0, B).astype(np.float32)
    MP = rng.choice(np.array([0.0, 0.05], np.float32), B)
    T[3] = 0.0
    K[4] = 1
    _, vs_ref, _ = oracle.sample(x, T, K, P, MP, seed=0, bitmask=bits)
    tg, _, _ = oracle.sample(x, T, K, P, MP, seed=0, bitmask=bits)
    allowed = np.unpackbits(bits.view(np.uint8), axis=1, bitorder="little")[:, :V].astype(bool)
    for u in (0.0, 0.37, 0.81, 0.999):
        tok, vstar, W = oracle.sample_icdf(x, T, K, P, MP, np.full(B, u, np.float32), bitmask=bits)
        assert np.array_equal(vstar, vs_ref)
        for b in range(B):
            assert allowed[b, tok[b]] and x[b, tok[b]] >= vstar[b]
        assert tok[3] == tg[3] and tok[4] == tg[4]  # greedy rows: the argmax


def test_icdf_law_on_a_fine_grid():
    """u on a fine midpoint grid lands on token i with frequency w_i / W, and
    the token never decreases as u grows (inverse-CDF law, checked against
    the sample oracle's keep set and weights, not the draw's own sums)."""
    rng = np.random.default_rng(2)
    V = 7
    x = rng.standard_normal(V)
    T, P = 0.8, 0.85
    d = oracle.sample_row_detail(x, T, 0, P, 0.0, 0, 0, 0)
    kept = x >= d["vstar"]
    w = np.where(kept, np.exp((x - d["m"]) / T), 0.0)
    N = 4000
    us = (np.arange(N) + 0.5) / N
    tok, _, _ = oracle.sample_icdf(np.tile(x, (N, 1)), T, 0, P, 0.0, us)
    assert np.all(np.diff(tok) >= 0)
    freq = np.bincount(tok, minlength=V) / N
    assert np.allclose(freq, w / w.sum(), atol=1.0 / N + 1e-12)


def test_icdf_rejects_uniform_outside_unit_interval():
    with pytest.raises(ValueError):
        oracle.sample_icdf(np.zeros((1, 4)), 1.0, 0, 1.0, 0.0, [1.0])
