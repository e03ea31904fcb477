"""GPU parity for the allow-set packer and the inverse-CDF draw (logits-mask-xpu,
"Usage" and "Method") against the CPU oracle on the same seeded inputs.

Rules: the packed words are bit-exact.  The draw's v* is the sample call's,
bit for bit.  Its token equals the oracle's on rows whose keep set the oracle
reproduces (same v*).  The exception is a token whose boundary (running mass
before or after it) lies within ICDF_BAND of u W: the GPU sums in compensated
fp32 and the oracle in double, so such a boundary may fall on either side.
There the GPU token must still be kept, and u W must lie in its interval
widened by the band."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

from .parity import allowed_matrix

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
NT = max(1, min(16, os.cpu_count() or 1))
ICDF_BAND = 1e-5  # relative to W


@pytest.fixture(scope="module")
def tsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import top_sampling_apply_gb300 as lib

    lib.load_library()
    return lib


@pytest.mark.parametrize("B,V", [(1, 1), (3, 31), (5, 32), (7, 33), (64, 128256), (300, 1000)])
def test_bitmask_from_allowed_bit_exact(tsa, B, V):
    rng = np.random.default_rng(B * 7 + V)
    a = rng.random((B, V)) < 0.37
    bits = tsa.bitmask_from_allowed(torch.from_numpy(a).to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(bits.cpu(), torch.from_numpy(oracle.bitmask_from_allowed(a)))


def test_bitmask_from_allowed_strided_rows_and_wider_out(tsa):
    rng = np.random.default_rng(4)
    big = torch.from_numpy(rng.random((9, 700)) < 0.5).to(DEV)
    a = big[:, 3:653]  # rows 700 bytes apart, V = 650
    out = torch.full((9, 40), -1, dtype=torch.int32, device=DEV)
    tsa.bitmask_from_allowed(a, out=out)
    torch.cuda.synchronize()
    W = (650 + 31) // 32
    ref = oracle.bitmask_from_allowed(a.cpu().numpy())
    assert torch.equal(out[:, :W].cpu(), torch.from_numpy(ref))
    assert bool((out[:, W:] == -1).all())  # words past ceil(V/32) untouched


def _check_icdf(case_logits, bitmask, T, K, P, MP, u, tok_g, vstar_g, vstar_sample):
    """Failure strings for the GPU's inverse-CDF tokens (see the module rules)."""
    fails = []
    assert np.array_equal(vstar_g, vstar_sample, equal_nan=True), "v* differs from the sample call's"
    tok_o, vstar_o, W, cum = oracle.sample_icdf(case_logits, T, K, P, MP, u, bitmask=bitmask,
                                                 nthreads=NT, with_cum=True)
    l = case_logits.double().numpy() if isinstance(case_logits, torch.Tensor) else case_logits
    B = l.shape[0]
    allowed = allowed_matrix(bitmask, l.shape[1])
    for b in range(B):
        t = int(tok_g[b])
        if t == tok_o[b]:
            continue
        if not (vstar_g[b] == vstar_o[b]):
            # the keep sets differ (within sample's own rules, tested elsewhere):
            # the token must be kept under the GPU's v*
            ok = 0 <= t < l.shape[1] and l[b, t] >= vstar_g[b] and (allowed is None or allowed[b, t])
            if not ok:
                fails.append("row %d: token %d outside its keep set" % (b, t))
            continue
        if not (0 <= t < l.shape[1]) or np.isnan(cum[b, t]):
            fails.append("row %d: token %d not kept (oracle %d)" % (b, t, tok_o[b]))
            continue
        kept = np.nonzero(~np.isnan(cum[b]))[0]
        j = np.searchsorted(kept, t)
        excl = cum[b, kept[j - 1]] if j > 0 else 0.0
        incl = cum[b, t]
        target = float(np.float32(u[b])) * W[b]
        if not (excl - ICDF_BAND * W[b] <= target <= incl + ICDF_BAND * W[b]):
            fails.append("row %d: token %d (oracle %d), interval [%.9g, %.9g] of W=%.9g misses u W=%.9g"
                         % (b, t, tok_o[b], excl, incl, W[b], target))
    return fails


def _run(tsa, x, mask, T, K, P, MP, u):
    dp = lambda p: p.to(DEV) if isinstance(p, torch.Tensor) else p  # noqa: E731
    xd = x.to(DEV)
    md = None if mask is None else mask.to(DEV)
    ud = torch.from_numpy(np.asarray(u, np.float32)).to(DEV)
    tok, vstar = tsa.sample_icdf(xd, ud, dp(T), dp(K), dp(P), dp(MP), bitmask=md, return_min_kept=True)
    _, vs_sample = tsa.sample(xd, dp(T), dp(K), dp(P), dp(MP), seed=0, offset=0, bitmask=md,
                              return_min_kept=True)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), vstar.cpu().numpy(), vs_sample.cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B", [16, 160])
def test_icdf_mixed_batch_matches_oracle(tsa, dtype, B):
    """Split rows (B < 128) and one CTA per row (B >= 128); greedy, unfiltered
    and filtered rows side by side; a misaligned row stride."""
    rng = np.random.default_rng(B)
    V, S = 40000, 40003
    big = torch.from_numpy((2 * rng.standard_normal((B, S))).astype(np.float32)).to(dtype)
    x = big[:, :V]
    m = workloads.random_bitmask(rng, B, V, 0.8)
    T = rng.uniform(0.5, 1.2, B).astype(np.float32)
    K = rng.integers(0, 300, B).astype(np.int32)
    P = rng.uniform(0.6, 1.0, B).astype(np.float32)
    MP = rng.choice(np.array([0.0, 0.05], np.float32), B)
    T[0::7] = 0.0
    K[1::7], P[1::7], MP[1::7] = 0, 1.0, 0.0
    K[2::11] = 1
    u = rng.random(B).astype(np.float32)
    u[3] = 0.0
    T, K, P, MP = (torch.from_numpy(v) for v in (T, K, P, MP))
    tok, vstar, vs_sample = _run(tsa, x, m, T, K, P, MP, u)
    fails = _check_icdf(x.contiguous().float(), m, T, K, P, MP, u, tok, vstar, vs_sample)
    assert not fails, fails[:3]
    assert tsa.device_status() == 0


def test_icdf_decode_batch_full_size(tsa):
    """The masked decode batch, B=256 V=128,256 f32, combined filter, in the
    benchmark's launch configuration; the oracle checks a sample of rows."""
    case = workloads.decode_batch("combined", mask_density=0.7)
    rng = np.random.default_rng(9)
    u = rng.random(case.B).astype(np.float32)
    tok, vstar, vs_sample = _run(tsa, case.logits, case.bitmask, case.temperature, case.top_k, case.top_p,
                                 case.min_p, u)
    rows = np.arange(0, case.B, 16)
    fails = _check_icdf(case.logits[rows], case.bitmask[rows], case.temperature, case.top_k, case.top_p,
                        case.min_p, u[rows], tok[rows], vstar[rows], vs_sample[rows])
    assert not fails, fails[:3]


def test_icdf_edges(tsa):
    """u = 0 gives the first kept token; a row with one allowed token gives it
    for any u; an empty row gives -1; T = 0 gives the argmax."""
    rng = np.random.default_rng(1)
    B, V = 4, 5000
    x = torch.from_numpy(rng.standard_normal((B, V)).astype(np.float32))
    allowed = rng.random((B, V)) < 0.5
    allowed[1] = False
    allowed[1, 4321] = True
    allowed[2] = False
    m = torch.from_numpy(oracle.bitmask_from_allowed(allowed))
    T = torch.tensor([1.0, 1.0, 1.0, 0.0])
    for uu in (0.0, 0.5, 0.99999):
        u = np.full(B, uu, np.float32)
        tok, vstar, vs_sample = _run(tsa, x, m, T, 0, 1.0, 0.0, u)
        if uu == 0.0:
            assert tok[0] == int(np.nonzero(allowed[0])[0][0])
        assert tok[1] == 4321
        assert tok[2] == -1
        xa = np.where(allowed[3], x[3].numpy(), -np.inf)
        assert tok[3] == int(np.argmax(xa))


# ------------------------------------------------ sequential top-p (f1's flag)
from .parity import check_sample  # noqa: E402


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B", [16, 160])
@pytest.mark.parametrize("V,S", [(40000, 40003), (40001, 40008)])
def test_sequential_matches_oracle(tsa, dtype, B, V, S):
    """tsa_sample_sequential against the oracle's sequential reading: split rows
    and one CTA per row, mixed modes, under the sample tolerance rules.  Rows
    40,003 apart start misaligned (the survivors' mask is formed a token a
    lane); rows 40,008 apart start 16-byte aligned (a 16-byte vector a lane),
    with V = 40,001 ending inside a vector."""
    rng = np.random.default_rng(40 + B + V)
    big = torch.from_numpy((2 * rng.standard_normal((B, S))).astype(np.float32)).to(dtype)
    x = big[:, :V]
    xd = big.to(DEV)[:, :V]  # rows S apart on the device too
    m = workloads.random_bitmask(rng, B, V, 0.8)
    T = rng.uniform(0.5, 1.2, B).astype(np.float32)
    K = rng.integers(0, 300, B).astype(np.int32)
    P = rng.uniform(0.3, 1.0, B).astype(np.float32)
    MP = rng.choice(np.array([0.0, 0.05], np.float32), B)
    T[0::7] = 0.0
    K[1::7], P[1::7], MP[1::7] = 0, 1.0, 0.0
    K[2::11] = 1
    T, K, P, MP = (torch.from_numpy(v) for v in (T, K, P, MP))
    dp = lambda p: p.to(DEV)  # noqa: E731
    tok, vstar = tsa.sample(xd, dp(T), dp(K), dp(P), dp(MP), seed=5, offset=6, bitmask=m.to(DEV),
                            return_min_kept=True, sequential=True)
    torch.cuda.synchronize()
    fails = check_sample(x.contiguous().float(), m, T, K, P, MP, 5, 6, tok.cpu(), vstar.cpu(), nthreads=NT,
                         sequential=True)
    assert not fails, fails[:3]
    # and the readings do differ on some rows here
    _, vs_int = tsa.sample(xd, dp(T), dp(K), dp(P), dp(MP), seed=5, offset=6, bitmask=m.to(DEV),
                           return_min_kept=True)
    torch.cuda.synchronize()
    assert bool((vstar.cpu() > vs_int.cpu()).any())
    assert tsa.device_status() == 0


def test_sequential_decode_batch_full_size(tsa):
    case = workloads.decode_batch("combined", mask_density=0.7)
    x, m = case.logits.to(DEV), case.bitmask.to(DEV)
    tok, vstar = tsa.sample(x, case.temperature, case.top_k, case.top_p, case.min_p, seed=3, offset=4,
                            bitmask=m, return_min_kept=True, sequential=True)
    torch.cuda.synchronize()
    fails = check_sample(case.logits, case.bitmask, case.temperature, case.top_k, case.top_p, case.min_p, 3, 4,
                         tok.cpu(), vstar.cpu(), nthreads=NT, rows=list(range(0, case.B, 16)), sequential=True)
    assert not fails, fails[:3]
