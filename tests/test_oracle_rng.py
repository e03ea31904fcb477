"""Pins for the oracle's random stream: Philox4x32-10 against an independent
implementation (NVIDIA curand's host generator), statistical balance, the
uniform lattice and the Gumbel transform against mpmath at high precision."""
import ctypes
import glob
import math
import os

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _curand():
    cands = []
    for root in [os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"]:
        if root:
            cands += sorted(glob.glob(os.path.join(root, "lib64", "libcurand.so*")))
    cands.append("libcurand.so")
    for c in cands:
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    return None


CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161


@pytest.mark.parametrize("seed", [0, 1, 0x123456789ABCDEF0, (1 << 64) - 1])
def test_philox_block_matches_curand_host_generator(seed):
    """curand's host Philox4_32_10 generator emits, for seed s, the blocks of
    counter (0, 0, j, 0) under key (s lo, s hi), j = 0, 1, ...  Matching 2,048
    blocks pins the round function, both multipliers and the key schedule."""
    lib = _curand()
    if lib is None:
        pytest.skip("libcurand not available")
    gen = ctypes.c_void_p()
    if lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) != 0:
        pytest.skip("curand host generator unavailable")
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        nblk = 2048
        ref = np.zeros(4 * nblk, dtype=np.uint32)
        assert lib.curandGenerate(gen, ref.ctypes.data_as(ctypes.c_void_p),
                                  ctypes.c_size_t(ref.size)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    mine = np.concatenate([oracle.philox4x32_10([0, 0, j, 0], key) for j in range(nblk)])
    assert np.array_equal(mine, ref)


def test_token_word_layout():
    """Token i of row b uses word i & 3 of the block with counter
    (i >> 2, b, offset lo, offset hi) and key (seed lo, seed hi)."""
    seed, offset = 0xDEADBEEF12345678, (7 << 32) | 11
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for b, i in [(0, 0), (3, 5), (255, 128255), (1023, 31999)]:
        blk = oracle.philox4x32_10([i >> 2, b, offset & 0xFFFFFFFF, offset >> 32], key)
        assert oracle.rand_word(seed, offset, b, i) == int(blk[i & 3])
    w = oracle.rand_words(seed, offset, 9, 100, 8)
    assert [int(v) for v in w] == [oracle.rand_word(seed, offset, 9, 100 + t) for t in range(8)]


def test_stream_balance():
    """Byte chi-square over 256 bins and per-bit balance over 2^20 words
    (4 rows x 2^18 tokens).  Bounds are ~5 sigma."""
    words = np.concatenate([oracle.rand_words(42, 3, b, 0, 1 << 18) for b in range(4)])
    n = words.size
    bits = ((words[:, None] >> np.arange(32, dtype=np.uint32)) & 1).sum(axis=0)
    assert np.all(np.abs(bits - n / 2) < 5 * math.sqrt(n / 4))
    by = words.view(np.uint8)
    counts = np.bincount(by, minlength=256)
    exp = by.size / 256
    chi2 = float(((counts - exp) ** 2 / exp).sum())
    # chi-square with 255 dof: mean 255, sd ~22.6
    assert chi2 < 255 + 5 * 22.6
    # distinct streams for distinct rows / offsets / seeds
    a = oracle.rand_words(1, 0, 0, 0, 64)
    assert not np.array_equal(a, oracle.rand_words(1, 0, 1, 0, 64))
    assert not np.array_equal(a, oracle.rand_words(1, 1, 0, 0, 64))
    assert not np.array_equal(a, oracle.rand_words(2, 0, 0, 0, 64))


def test_uniform_lattice():
    assert oracle.uniform(0) == 2.0 ** -24
    assert oracle.uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    rng = np.random.default_rng(0)
    for x in rng.integers(0, 1 << 32, 2000, dtype=np.uint64):
        u = oracle.uniform(int(x))
        k = u * 2.0 ** 24
        assert k == int(k) and int(k) % 2 == 1 and 0.0 < u < 1.0
        assert np.float32(u) == u  # exact in fp32
        assert int(k) == 2 * (int(x) >> 9) + 1


def test_gumbel_against_mpmath():
    """G(x) = -ln(-ln u(x)) evaluated by mpmath at 50 digits; the oracle's
    double evaluation must agree to ~1e-15 relative, including both ends of
    the lattice (G in [-2.8116, 16.6355])."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    xs = [0, 1 << 9, 0x7FFFFFFF, 0x80000000, 0xFFFFFE00, 0xFFFFFFFF]
    rng = np.random.default_rng(1)
    xs += [int(v) for v in rng.integers(0, 1 << 32, 300, dtype=np.uint64)]
    for x in xs:
        k = 2 * (x >> 9) + 1
        u = mpmath.mpf(k) / mpmath.mpf(2) ** 24
        ref = -mpmath.log(-mpmath.log(u))
        got = oracle.gumbel(x)
        assert abs(got - float(ref)) <= 4e-15 * max(1.0, abs(float(ref))), (x, got, ref)
    top = oracle.gumbel(0xFFFFFFFF)
    bot = oracle.gumbel(0)
    assert abs(top - 16.6355) < 1e-3 and abs(bot + 2.8116) < 1e-3


def test_gumbel_monotone():
    ks = np.arange(0, 1 << 23, 997, dtype=np.uint64)
    g = np.array([oracle.gumbel(int(k) << 9) for k in ks])
    assert np.all(np.diff(g) > 0)
