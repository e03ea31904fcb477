"""Pins of the oracle's selective log-softmax (selective_log_softmax, "Selective
Log Softmax"), each against something other than the oracle's own formula:
closed forms (two tokens: the softplus form; n equal logits: -ln n), the
normalisation of the distribution it defines, invariance to a shift of the
logits, and the special values the calls document."""
import math

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


@pytest.mark.parametrize("a,b,T", [(0.3, -1.2, 1.0), (5.0, 5.5, 0.4), (-20.0, 17.0, 2.5), (1e4, 1e4 + 3.0, 1.0)])
def test_two_tokens_closed_form(a, b, T):
    # p(0) = 1 / (1 + exp((b - a) / T)), so log p(0) = -softplus((b - a) / T)
    def softplus(z):
        return max(z, 0.0) + math.log1p(math.exp(-abs(z)))

    got = oracle.selective_log_softmax(np.array([[a, b], [a, b]]), [0, 1], T)
    T = float(np.float32(T))  # temperatures are float32 parameters, as on the GPU
    assert got[0] == pytest.approx(-softplus((b - a) / T), abs=1e-12)
    assert got[1] == pytest.approx(-softplus((a - b) / T), abs=1e-12)


@pytest.mark.parametrize("n", [1, 3, 1000])
def test_equal_logits_give_minus_ln_n(n):
    x = np.full((1, n), 0.7)
    assert oracle.selective_log_softmax(x, [n // 2], 0.9)[0] == pytest.approx(-math.log(n), abs=1e-12)


def test_probabilities_sum_to_one_over_allowed_tokens():
    rng = np.random.default_rng(3)
    V = 301
    x = rng.standard_normal(V) * 3
    words = rng.integers(0, 2**32, size=(1, (V + 31) // 32), dtype=np.uint64).astype(np.uint32).view(np.int32)
    allowed = [(int(words.view(np.uint32)[0, j >> 5]) >> (j & 31)) & 1 == 1 for j in range(V)]
    rows = np.tile(x, (V, 1))
    lp = oracle.selective_log_softmax(rows, np.arange(V), 0.8, np.tile(words, (V, 1)))
    assert all(lp[j] == -np.inf for j in range(V) if not allowed[j])
    assert sum(math.exp(lp[j]) for j in range(V) if allowed[j]) == pytest.approx(1.0, abs=1e-12)


def test_shift_invariance_and_temperature_floor():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((4, 50))
    idx = [0, 7, 13, 49]
    base = oracle.selective_log_softmax(x, idx, 1.3)
    assert np.allclose(oracle.selective_log_softmax(x + 123.5, idx, 1.3), base, atol=1e-12)
    # T <= 0 is the unscaled (T = 1) log-softmax
    assert np.allclose(oracle.selective_log_softmax(x, idx, 0.0), oracle.selective_log_softmax(x, idx, 1.0))
    assert np.allclose(oracle.selective_log_softmax(x, idx, -2.0), oracle.selective_log_softmax(x, idx, 1.0))


def test_special_values():
    x = np.array([[1.0, np.nan, 2.0, -np.inf],
                  [-np.inf, -np.inf, -np.inf, -np.inf],
                  [0.5, 0.25, 0.0, 1.0]])
    out = oracle.selective_log_softmax(x, [1, 0, 4], 1.0)
    assert out[0] == -np.inf          # a NaN logit counts as -inf
    assert math.isnan(out[1])         # no allowed finite logit
    assert math.isnan(out[2])         # index outside [0, V)
    # the NaN entry drops out of the normaliser: token 2 is then a two-way choice
    assert oracle.selective_log_softmax(x[:1], [2], 1.0)[0] == pytest.approx(-math.log1p(math.exp(-1.0)), abs=1e-12)
    masked = np.array([[0b1011]], dtype=np.int32)  # token 2 disallowed
    assert oracle.selective_log_softmax(x[2:], [2], 1.0, masked)[0] == -np.inf
