"""Pins for the oracle's mask, keep sets, draw and top-k against what the pages
and the mathematics fix: torch.argmax / torch.sort / torch.topk on the CPU,
brute force on tiny rows (an O(V^2) definition of "mass strictly above"),
closed forms (the 1/2, 1/4, ... row; min-p as a logit offset), the pages'
stated checks (logits-mask-xpu "Validation", logits-processor "Correctness",
lm-head-topk "Correctness"), and the Gumbel-max law P(i) = softmax(s)_i."""
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(rng, B, V, scale=2.0, dup=False):
    x = (scale * rng.standard_normal((B, V))).astype(np.float32)
    if dup:
        for b in range(B):
            j = rng.choice(V, 3, replace=False)
            x[b, j] = x[b].max()
    return x


# ----------------------------------------------------------------- bitmask
@pytest.mark.parametrize("dtype_code,np_t,ninf", [(0, np.uint32, 0xFF800000),
                                                   (1, np.uint16, 0xFC00),
                                                   (2, np.uint16, 0xFF80)])
def test_bitmask_every_pattern_small_v(dtype_code, np_t, ninf):
    """Brute force over every mask pattern for V <= 10, with garbage in the
    bits at or beyond V (logits-processor "Correctness": exactly the
    disallowed logits become -inf, vocabularies not a multiple of 32)."""
    rng = np.random.default_rng(dtype_code)
    for V in range(1, 11):
        pats = np.arange(1 << V, dtype=np.int64)
        garbage = rng.integers(0, 1 << (32 - V), pats.size, dtype=np.int64) << V
        words = ((pats | garbage) & 0xFFFFFFFF).astype(np.uint32).view(np.int32)[:, None]
        bits = rng.integers(0, np.iinfo(np_t).max, (pats.size, V), dtype=np.int64).astype(np_t)
        out = oracle.apply_token_bitmask(bits, words, dtype_code)
        for r in range(pats.size):
            for i in range(V):
                allowed = (int(pats[r]) >> i) & 1
                expect = bits[r, i] if allowed else ninf
                assert out[r, i] == expect


@pytest.mark.parametrize("V", [1, 31, 32, 33, 95, 8191])
def test_bitmask_lsb_first_against_numpy_unpack(V):
    rng = np.random.default_rng(V)
    B = 5
    x = rng.standard_normal((B, V)).astype(np.float32)
    mask = workloads.random_bitmask(rng, B, V, 0.5, force_one=False).numpy()
    allowed = np.unpackbits(mask.view(np.uint8), axis=1, bitorder="little")[:, :V].astype(bool)
    out = oracle.apply_token_bitmask(x.view(np.uint32), mask, 0).view(np.float32)
    assert np.array_equal(out[allowed].view(np.uint32), x[allowed].view(np.uint32))
    assert np.all(np.isneginf(out[~allowed]))


# ----------------------------------------------------------------- greedy
def test_greedy_and_top_k_one_equal_torch_argmax(nthreads):
    """logits-processor "Correctness" / logits-mask-xpu "Validation": greedy
    (T <= 0) and top_k = 1 return torch.argmax (first index on ties)."""
    rng = np.random.default_rng(3)
    x = _rows(rng, 64, 1000, dup=True)
    ref = torch.argmax(torch.from_numpy(x), dim=1).numpy()
    for T, k in [(0.0, 0), (-1.0, 50), (0.7, 1), (1.0, 1)]:
        tok, vstar, _ = oracle.sample(x, T, k, 0.9, 0.05, seed=5, nthreads=nthreads)
        assert np.array_equal(tok, ref)
        assert np.array_equal(vstar, x.max(axis=1).astype(np.float64))


def test_masked_greedy_lands_in_allow_set():
    rng = np.random.default_rng(4)
    B, V = 32, 777
    x = _rows(rng, B, V)
    mask = workloads.random_bitmask(rng, B, V, 0.3).numpy()
    allowed = np.unpackbits(mask.view(np.uint8), axis=1, bitorder="little")[:, :V].astype(bool)
    tok, _, _ = oracle.sample(x, 0.0, 0, 1.0, 0.0, seed=0, bitmask=mask)
    xm = np.where(allowed, x, -np.inf)
    assert np.array_equal(tok, np.argmax(xm, axis=1))
    assert allowed[np.arange(B), tok].all()


def test_empty_row_gives_minus_one():
    x = np.zeros((2, 40), dtype=np.float32)
    mask = np.zeros((2, 2), dtype=np.int32)
    mask[1, 0] = 1 << 7
    tok, vstar, _ = oracle.sample(x, 1.0, 0, 1.0, 0.0, seed=0, bitmask=mask)
    assert tok[0] == -1 and math.isnan(vstar[0]) and tok[1] == 7
    y = np.full((1, 9), -np.inf, dtype=np.float32)
    tok, _, _ = oracle.sample(y, 0.0, 0, 1.0, 0.0, seed=0)
    assert tok[0] == -1


# ----------------------------------------------------------------- keep sets
def _brute_sets(l, T, k, p, mp):
    """Keep sets from the definitions, by O(V^2) brute force, for a row with
    no mask: top-k by counting strictly-greater entries, top-p by the mass
    strictly above each token, min-p by the weight relative to the max."""
    V = l.size
    s = l.astype(np.float64) / T
    prob = softmax(s)
    greater = (l[None, :] > l[:, None])  # greater[i, j] = l_j > l_i
    mass_above = (greater * prob[None, :]).sum(axis=1)
    is_max = l == l.max()
    n_greater = greater.sum(axis=1)
    Kk = np.ones(V, bool) if (k < 1 or k >= V) else (n_greater < k)
    Kp = np.ones(V, bool) if p >= 1 else ((mass_above < p) | is_max)
    Km = np.ones(V, bool) if mp <= 0 else ((prob / prob.max() >= mp) | is_max)
    return Kk, Kp, Km, mass_above, prob / prob.max()


def _kept(detail, l):
    return l.astype(np.float64) >= detail["vstar"]


def test_top_k_keep_set_brute_force():
    """k = 1..100 on tiny rows vs exhaustive sort (with ties kept whole)."""
    rng = np.random.default_rng(5)
    for trial in range(6):
        V = 120
        l = _rows(rng, 1, V, dup=(trial % 2 == 1))[0]
        if trial >= 4:
            l = np.round(l)  # many ties
        for k in range(2, 101):
            d = oracle.sample_row_detail(l, 1.0, k, 1.0, 0.0, 0, 0, 0)
            Kk, *_ = _brute_sets(l, 1.0, k, 1.0, 0.0)
            kept = _kept(d, l)
            assert np.array_equal(kept, Kk), (trial, k)
            assert kept.sum() >= k
            srt = np.sort(l)[::-1]
            assert d["v_k"] == srt[k - 1]
            if np.unique(l).size == V:
                assert kept.sum() == k


def test_top_p_keep_set_brute_force():
    rng = np.random.default_rng(6)
    for trial in range(40):
        V = int(rng.integers(2, 60))
        l = _rows(rng, 1, V, scale=float(rng.uniform(0.3, 4.0)))[0]
        if trial % 3 == 0:
            l = np.round(l * 2) / 2
        T = float(np.float32(rng.uniform(0.3, 2.0)))
        p = float(np.float32(rng.uniform(0.05, 0.99)))
        d = oracle.sample_row_detail(l, T, 0, p, 0.0, 0, 0, 0)
        _, Kp, _, mass_above, _ = _brute_sets(l, T, 0, p, 0.0)
        near = np.abs(mass_above - p) < 1e-9
        kept = _kept(d, l)
        assert np.array_equal(kept[~near], Kp[~near]), trial
        assert np.allclose(d["M"], mass_above, atol=1e-12)


def test_top_p_prefix_rule_scipy_cumsum():
    """With distinct values, top-p keeps the smallest descending prefix whose
    mass reaches p (np.cumsum over scipy's softmax)."""
    rng = np.random.default_rng(7)
    for _ in range(50):
        V = 200
        l = _rows(rng, 1, V)[0]
        p = float(np.float32(rng.uniform(0.1, 0.99)))
        d = oracle.sample_row_detail(l, 1.0, 0, p, 0.0, 0, 0, 0)
        order = np.argsort(-l.astype(np.float64), kind="stable")
        cs = np.cumsum(softmax(l.astype(np.float64))[order])
        n = int(np.searchsorted(cs, p, side="left")) + 1
        if abs(cs[n - 1] - p) < 1e-12 or (n >= 2 and abs(cs[n - 2] - p) < 1e-12):
            continue
        assert d["n_kept"] == min(n, V)


def test_top_p_golden_halving_row():
    path = os.path.join(GOLDEN, "top_p_halving.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    probs = np.array([float(v) for v in rows[0][1:]])
    assert abs(probs.sum() - 1.0) < 1e-15
    l = np.log(probs)
    for p_s, n_s in rows[1:]:
        d = oracle.sample_row_detail(l, 1.0, 0, float(p_s), 0.0, 0, 0, 0)
        assert d["n_kept"] == int(n_s), (p_s, d["n_kept"])


def test_min_p_closed_form():
    """min-p keeps w_i = exp((l_i - m)/T) >= min_p, i.e. l_i >= m + T ln(min_p)."""
    rng = np.random.default_rng(8)
    for _ in range(40):
        l = _rows(rng, 1, 300)[0]
        T = float(np.float32(rng.uniform(0.3, 2.0)))
        mp = float(np.float32(rng.choice([0.01, 0.05, 0.1, 0.3, 0.9])))
        d = oracle.sample_row_detail(l, T, 0, 1.0, mp, 0, 0, 0)
        cut = l.max() + T * math.log(mp)
        far = np.abs(l.astype(np.float64) - cut) > 1e-9
        assert np.array_equal(_kept(d, l)[far], (l.astype(np.float64) >= cut)[far])
        assert d["v_m"] <= l.max()
    # min_p > 1 and top_p <= 0 still keep the argmax class
    l = np.array([1.0, 3.0, 3.0, 2.0], dtype=np.float32)
    for (p, mp) in [(1.0, 2.0), (0.0, 0.0), (-1.0, 0.0)]:
        d = oracle.sample_row_detail(l, 1.0, 0, p, mp, 0, 0, 0)
        assert d["n_kept"] == 2 and d["vstar"] == 3.0


def test_intersection_and_mask_invariants():
    """K = K_k & K_p & K_m (the filters' intersection, logits-processor
    "Method"); the argmax is always kept; masked tokens never are."""
    rng = np.random.default_rng(9)
    for trial in range(60):
        V = int(rng.integers(2, 90))
        l = _rows(rng, 1, V, scale=float(rng.uniform(0.5, 3.0)))[0]
        T = float(np.float32(rng.uniform(0.3, 1.5)))
        k = int(rng.integers(0, V + 3))
        p = float(np.float32(rng.uniform(0.2, 1.0)))
        mp = float(np.float32(rng.choice([0.0, 0.02, 0.1, 0.5])))
        d = oracle.sample_row_detail(l, T, k, p, mp, 3, 1, 0)
        if k == 1:
            continue
        Kk, Kp, Km, mass_above, wrel = _brute_sets(l, T, k, p, mp)
        near = (np.abs(mass_above - p) < 1e-9) | (np.abs(wrel - mp) < 1e-9)
        kept = _kept(d, l)
        assert np.array_equal(kept[~near], (Kk & Kp & Km)[~near]), trial
        assert kept[np.argmax(l)]
        assert kept[d["token"]]
    # masked tokens are outside the allowed set
    x = _rows(rng, 16, 500)
    mask = workloads.random_bitmask(rng, 16, 500, 0.4).numpy()
    allowed = np.unpackbits(mask.view(np.uint8), axis=1, bitorder="little")[:, :500].astype(bool)
    for seed in range(10):
        tok, _, _ = oracle.sample(x, 1.0, 0, 1.0, 0.0, seed=seed, bitmask=mask)
        assert allowed[np.arange(16), tok].all()


# ----------------------------------------------------------------- draws
def _tv_expectation(p, n):
    return 0.5 * float(np.sum(np.sqrt(2 * p * (1 - p) / (math.pi * n))))


@pytest.mark.parametrize("case", ["skewed", "filtered"])
def test_gumbel_max_distribution_8_tokens(case, nthreads):
    """The empirical draw distribution over an 8-token vocabulary matches the
    renormalised filtered softmax (logits-processor "Correctness"): 100k draws
    as 1,000 identical rows x 100 offsets, TV <= 0.005."""
    l = np.array([2.0, 1.5, 1.0, 0.5, 0.0, -0.5, -1.0, -1.5], dtype=np.float32)
    x = np.tile(l, (1000, 1))
    if case == "skewed":
        T, k, p, mp = 1.0, 0, 1.0, 0.0
        target = softmax(l.astype(np.float64))
    else:
        T, k, p, mp = 0.8, 6, 0.9, 0.02
        q = softmax(l.astype(np.float64) / T)
        keep = np.zeros(8, bool)
        keep[:6] = True
        cum = np.concatenate([[0.0], np.cumsum(q)[:-1]])
        keep &= (cum < p)
        keep &= q / q.max() >= mp
        target = np.where(keep, q, 0.0)
        target /= target.sum()
    counts = np.zeros(8)
    for off in range(100):
        tok, _, _ = oracle.sample(x, T, k, p, mp, seed=11, offset=off, nthreads=nthreads)
        counts += np.bincount(tok, minlength=8)
    emp = counts / counts.sum()
    tv = 0.5 * np.abs(emp - target).sum()
    assert counts[target == 0].sum() == 0
    assert tv <= 0.005, (tv, _tv_expectation(target[target > 0], 100000))


def test_xpu_validation_cases():
    """logits-mask-xpu "Validation" checks, restated in tests/golden."""
    # top_p = 1 keeps the full support: every one of 8 tokens is drawn
    l = np.array([0.3, -0.2, 0.1, 0.0, -0.4, 0.2, -0.1, 0.05], dtype=np.float32)
    x = np.tile(l, (200, 1))
    seen = set()
    for off in range(100):
        seen |= set(oracle.sample(x, 1.0, 0, 1.0, 0.0, seed=1, offset=off)[0].tolist())
    assert seen == set(range(8))
    # top_p = 0.5 on a peaked row collapses to the mode in all 200 draws
    pk = np.array([4.0, 0.5, 0.2, 0.0, -0.3, 0.1, -1.0, 0.3], dtype=np.float32)
    tok = oracle.sample(np.tile(pk, (200, 1)), 1.0, 0, 0.5, 0.0, seed=2)[0]
    assert np.all(tok == 0)
    # top_k = 5 never selects outside the true top 5 (1000 trials)
    rng = np.random.default_rng(12)
    x = _rows(rng, 1000, 64)
    top5 = np.argsort(-x, axis=1)[:, :5]
    tok = oracle.sample(x, 1.0, 5, 1.0, 0.0, seed=3)[0]
    assert all(tok[b] in top5[b] for b in range(1000))


def test_draws_deterministic_and_keyed():
    rng = np.random.default_rng(13)
    x = _rows(rng, 64, 300)
    a = oracle.sample(x, 1.0, 0, 1.0, 0.0, seed=4, offset=9)[0]
    assert np.array_equal(a, oracle.sample(x, 1.0, 0, 1.0, 0.0, seed=4, offset=9, nthreads=4)[0])
    assert not np.array_equal(a, oracle.sample(x, 1.0, 0, 1.0, 0.0, seed=4, offset=10)[0])
    assert not np.array_equal(a, oracle.sample(x, 1.0, 0, 1.0, 0.0, seed=5, offset=9)[0])


def test_per_row_parameters_independent():
    """Per-row parameters are honoured independently (logits-processor
    "Correctness"): a heterogeneous batch equals its rows run one at a time."""
    rng = np.random.default_rng(14)
    B, V = 24, 200
    x = _rows(rng, B, V)
    T = rng.uniform(0.0, 1.5, B).astype(np.float32)
    K = rng.integers(0, 30, B).astype(np.int32)
    P = rng.uniform(0.3, 1.0, B).astype(np.float32)
    M = rng.choice(np.array([0.0, 0.05], np.float32), B)
    tok, vstar, _ = oracle.sample(x, T, K, P, M, seed=6, offset=2)
    for b in range(B):
        d = oracle.sample_row_detail(x[b], T[b], int(K[b]), P[b], M[b], 6, 2, b)
        assert d["token"] == tok[b] and d["vstar"] == vstar[b]


# ----------------------------------------------------------------- topk
def test_topk_matches_torch_stable_sort_with_ties(nthreads):
    """lm-head-topk "Method": sorted descending, ties to the lower index --
    the first k of torch.sort(descending, stable)."""
    rng = np.random.default_rng(15)
    x = np.round(_rows(rng, 12, 3000) * 4) / 4  # heavy ties
    for k in [1, 2, 10, 100, 2048]:
        vals, idx = oracle.topk(x, k, nthreads=nthreads)
        sv, si = torch.sort(torch.from_numpy(x).double(), dim=1, descending=True, stable=True)
        assert np.array_equal(idx, si[:, :k].numpy())
        assert np.array_equal(vals, sv[:, :k].numpy())


def test_topk_matches_torch_topk_distinct():
    """torch.topk on tie-free rows: indices torch.equal, values equal
    (lm-head-topk "Correctness"); k = 1 equals torch.argmax."""
    rng = np.random.default_rng(16)
    x = rng.standard_normal((8, 20000)).astype(np.float32)
    t = torch.from_numpy(x)
    for k in [1, 50, 100]:
        vals, idx = oracle.topk(x, k)
        rv, ri = torch.topk(t, k, dim=1)
        assert torch.equal(torch.from_numpy(idx), ri)
        assert np.array_equal(vals.astype(np.float32), rv.numpy())
    assert np.array_equal(oracle.topk(x, 1)[1][:, 0], torch.argmax(t, dim=1).numpy())


def test_topk_planted_in_one_chunk_and_ragged_tail():
    """Every winner inside one 2,048-wide chunk still equals brute force, and
    a ragged final chunk returns only valid indices (lm-head-topk
    "Correctness")."""
    rng = np.random.default_rng(17)
    V = 2048 * 5 + 300
    x = rng.standard_normal((4, V)).astype(np.float32)
    for b, c in enumerate([0, 2, 4, 5]):
        lo = c * 2048
        hi = min(V, lo + 2048)
        pos = rng.choice(np.arange(lo, hi), 50, replace=False)
        x[b, pos] += 8.0
    vals, idx = oracle.topk(x, 50)
    order = np.lexsort((np.tile(np.arange(V), (4, 1)), -x.astype(np.float64)), axis=1)
    assert np.array_equal(idx, order[:, :50])
    assert np.all((idx >= 0) & (idx < V))
    for b, c in enumerate([0, 2, 4, 5]):
        assert np.all(idx[b] // 2048 == c)


def test_topk_negative_zero_ties_by_index():
    x = np.array([[0.0, -0.0, -1.0, 0.0, -0.0]], dtype=np.float32)
    vals, idx = oracle.topk(x, 4)
    assert idx.tolist() == [[0, 1, 3, 4]]
    assert np.signbit(vals[0]).tolist() == [False, True, False, True]


def find_equal_uniform_pair(seed: int, offset: int, row: int, V: int):
    """Two tokens i < j of one row whose random words fall on the same lattice
    point (same x >> 9), so equal logits give exactly equal perturbed scores."""
    w = oracle.rand_words(seed, offset, row, 0, V) >> 9
    order = np.argsort(w, kind="stable")
    same = np.nonzero(w[order][1:] == w[order][:-1])[0]
    if same.size == 0:
        return None
    a, b = int(order[same[0]]), int(order[same[0] + 1])
    return min(a, b), max(a, b)


def test_exact_score_tie_goes_to_lower_index():
    """Gumbel-max with an exact score tie returns the lower index: a flat row
    whose mask allows only two tokens with the same uniform."""
    V = 16384
    found = None
    for row in range(8):
        pair = find_equal_uniform_pair(21, 0, row, V)
        if pair:
            found = (row, pair)
            break
    assert found is not None
    row, (i, j) = found
    B = row + 1
    x = np.zeros((B, V), dtype=np.float32)
    allowed = np.zeros((B, V), dtype=bool)
    allowed[:, :] = True
    allowed[row, :] = False
    allowed[row, [i, j]] = True
    mask = workloads.pack_allowed(allowed).numpy()
    tok, _, gap = oracle.sample(x, 1.0, 0, 1.0, 0.0, seed=21, offset=0, bitmask=mask)
    assert tok[row] == i and gap[row] == 0.0
