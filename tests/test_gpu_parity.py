"""GPU parity: every call of the CUDA library (through its C ABI, via the
Python binding) against the CPU oracle on the same seeded inputs, at the
workloads' full sizes in the benchmark's launch configuration, plus edge
cases (empty rows, ragged and misaligned rows, V not a multiple of 32, ties,
maximum sizes)."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

from .parity import allowed_matrix, check_sample

pytestmark = pytest.mark.gpu

NT = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module")
def tsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import top_sampling_apply_gb300 as lib

    lib.load_library()
    return lib


DEV = "cuda:0"


def _run_sample(tsa, case, seed=None, offset=None, mask=True):
    x = case.logits.to(DEV)
    m = case.bitmask.to(DEV) if (mask and case.bitmask is not None) else None
    dev_param = lambda p: p.to(DEV) if isinstance(p, torch.Tensor) else p  # noqa: E731
    tok, vstar = tsa.sample(x, dev_param(case.temperature), dev_param(case.top_k),
                            dev_param(case.top_p), dev_param(case.min_p),
                            seed=case.seed if seed is None else seed,
                            offset=case.offset if offset is None else offset, bitmask=m,
                            return_min_kept=True)
    torch.cuda.synchronize()
    return tok.cpu(), vstar.cpu()


def _assert_sample(tsa, case, seed=None, offset=None, mask=True, rows=None):
    seed = case.seed if seed is None else seed
    offset = case.offset if offset is None else offset
    tok, vstar = _run_sample(tsa, case, seed, offset, mask)
    fails = check_sample(case.logits, case.bitmask if mask else None, case.temperature,
                         case.top_k, case.top_p, case.min_p, seed, offset, tok, vstar,
                         nthreads=NT, rows=rows)
    assert not fails, "%d rows fail, first: %s" % (len(fails), fails[:5])
    assert tsa.device_status() == 0
    return tok


# ------------------------------------------------------------------ bitmask
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("V", [1, 31, 33, 8191, 8192, 128257])
def test_bitmask_bit_exact(tsa, dtype, V):
    rng = np.random.default_rng(V)
    B = 5
    x = torch.from_numpy(rng.standard_normal((B, V)).astype(np.float32)).to(dtype)
    m = workloads.random_bitmask(rng, B, V, 0.6, force_one=False)
    y = x.to(DEV)
    tsa.apply_token_bitmask(y, m.to(DEV))
    torch.cuda.synchronize()
    code = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[dtype]
    raw = x.view(torch.int32 if dtype == torch.float32 else torch.int16).numpy()
    raw = raw.view(np.uint32 if dtype == torch.float32 else np.uint16)
    ref = oracle.apply_token_bitmask(raw, m.numpy(), code)
    got = y.cpu().view(torch.int32 if dtype == torch.float32 else torch.int16).numpy()
    assert np.array_equal(got.view(ref.dtype), ref)


def test_bitmask_strided_rows(tsa):
    rng = np.random.default_rng(1)
    B, V, S = 7, 1000, 1003  # odd row stride: misaligned rows
    big = torch.from_numpy(rng.standard_normal((B, S)).astype(np.float32))
    m = workloads.random_bitmask(rng, B, V, 0.5)
    mw = torch.zeros(B, 40, dtype=torch.int32)
    mw[:, : m.shape[1]] = m
    y = big.to(DEV)
    tsa.apply_token_bitmask(y[:, :V], mw.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.apply_token_bitmask(big[:, :V].contiguous().numpy().view(np.uint32), m.numpy(), 0)
    got = y.cpu().numpy()
    assert np.array_equal(got[:, :V].view(np.uint32), ref)
    assert np.array_equal(got[:, V:], big[:, V:].numpy())  # padding untouched


# ------------------------------------------------------------------ sample
def test_sample_tiny_case(tsa):
    case = workloads.tiny_case()
    _assert_sample(tsa, case)
    for t in range(4):
        _assert_sample(tsa, case, seed=t, offset=t)


@pytest.mark.parametrize("mode", list(workloads.DECODE_MODES))
def test_sample_decode_batch_modes(tsa, mode):
    case = workloads.decode_batch(mode, mask_density=None)
    for t in (0, 1, 31):
        _assert_sample(tsa, case, seed=t, offset=t)


def test_sample_decode_batch_fused_mask(tsa):
    case = workloads.decode_batch("combined", mask_density=0.7)
    for t in (0, 5, 31):
        _assert_sample(tsa, case, seed=t, offset=t)
    case2 = workloads.decode_batch("top_p", mask_density=0.7)
    _assert_sample(tsa, case2, seed=3, offset=3)


def test_sample_hetero_batch(tsa):
    case = workloads.hetero_batch()
    for t in (0, 1):
        _assert_sample(tsa, case, seed=t, offset=t)


def test_sample_peaked_batch(tsa):
    """All 512 rows (90% with one +10 token, 10% flat) at four of the 64
    steps, the last one included."""
    case = workloads.peaked_batch()
    for t in (0, 21, 42, 63):
        _assert_sample(tsa, case, seed=t, offset=t)


LARGE_MODES = {"top_p": (0, 0.9, 0.0), "min_p": (0, 1.0, 0.05), "combined": (50, 0.9, 0.05)}


@pytest.mark.parametrize("shift,T", [(40.0, 0.5), (40.0, 0.8), (-40.0, 0.5), (-40.0, 0.8)])
def test_sample_large_magnitude_logits(tsa, shift, T):
    """Logits of the size real models produce (the decode batch moved by
    +-40) at temperatures below 1: the normaliser's exponents are then large,
    and any rounding that scales Z moves the top-p cut by more than the 1e-6
    band.  Both the one-CTA-per-row kernel (256 rows) and the split-row
    kernels (32 rows), with and without the mask."""
    base = workloads.decode_batch("combined", mask_density=0.7)
    x = (base.logits + shift).contiguous()
    for B in (256, 32):
        for mode, (k, p, mp) in LARGE_MODES.items():
            for masked in (True, False):
                case = workloads.SampleCase("large_%s" % mode, x[:B].contiguous(),
                                            base.bitmask[:B].contiguous() if masked else None,
                                            T, k, p, mp)
                seed = int(abs(shift)) + B + k
                _assert_sample(tsa, case, seed=seed, offset=3)


def test_sample_hetero_batch_large_magnitude(tsa):
    """The heterogeneous bf16 batch moved by +30 (per-row temperatures down to
    0.3; bf16 at 30 has a spacing of 1/8, so ties are common)."""
    case = workloads.hetero_batch()
    case.logits = (case.logits.float() + 30.0).to(torch.bfloat16)
    for t in (0, 1):
        _assert_sample(tsa, case, seed=t, offset=t)


def test_greedy_equals_torch_argmax_with_ties(tsa):
    rng = np.random.default_rng(3)
    B, V = 64, 50000
    x = (2 * rng.standard_normal((B, V))).astype(np.float32)
    for b in range(B):
        j = rng.choice(V, 3, replace=False)
        x[b, j] = x[b].max()
    xt = torch.from_numpy(x)
    ref = torch.argmax(xt, dim=1)
    for T, k in [(0.0, 0), (0.8, 1)]:
        tok = tsa.sample(xt.to(DEV), T, k, 0.9, 0.1, seed=1)
        assert torch.equal(tok.cpu(), ref)


def test_top_k_five_never_leaves_true_top5(tsa):
    rng = np.random.default_rng(12)
    x = torch.from_numpy((2 * rng.standard_normal((1000, 4096))).astype(np.float32))
    top5 = torch.topk(x, 5, dim=1).indices
    for off in range(3):
        tok = tsa.sample(x.to(DEV), 1.0, 5, 1.0, 0.0, seed=3, offset=off).cpu()
        assert (top5 == tok[:, None]).any(dim=1).all()


def test_empty_and_tiny_rows(tsa):
    rng = np.random.default_rng(4)
    for V in [1, 2, 3, 5, 31, 32, 33, 63, 2049]:
        B = 6
        x = torch.from_numpy(rng.standard_normal((B, V)).astype(np.float32))
        allowed = rng.random((B, ((V + 31) // 32) * 32)) < 0.5
        allowed[0, :] = False  # row 0 empty
        allowed[1, :V] = True
        m = workloads.pack_allowed(allowed)
        for (T, k, p, mp) in [(0.0, 0, 1.0, 0.0), (1.0, 0, 1.0, 0.0), (0.7, 3, 0.8, 0.05),
                              (1.3, 0, 0.5, 0.0), (1.0, 2, 1.0, 0.0)]:
            tok, vstar = tsa.sample(x.to(DEV), T, k, p, mp, seed=7, offset=V, bitmask=m.to(DEV),
                                    return_min_kept=True)
            torch.cuda.synchronize()
            assert tok[0].item() == -1
            fails = check_sample(x, m, T, k, p, mp, 7, V, tok.cpu(), vstar.cpu())
            assert not fails, (V, T, k, p, mp, fails[:3])


def test_all_minus_inf_row(tsa):
    x = torch.full((3, 5000), float("-inf"))
    x[1, 17] = 0.5
    tok = tsa.sample(x.to(DEV), 1.0, 0, 0.9, 0.0, seed=1).cpu()
    assert tok.tolist() == [-1, 17, -1]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("V,S", [(8191, 8191), (8191, 8197), (128257, 128257), (40000, 40003)])
def test_sample_misaligned_and_ragged(tsa, dtype, V, S):
    """Odd vocabularies and row strides: rows start off 16-byte boundaries, so
    heads and tails are loaded outside the bulk copies."""
    rng = np.random.default_rng(V + S)
    B = 12
    big = torch.from_numpy((2 * rng.standard_normal((B, S))).astype(np.float32)).to(dtype)
    m = workloads.random_bitmask(rng, B, V, 0.8)
    x = big.to(DEV)[:, :V]
    T = torch.from_numpy(rng.uniform(0.5, 1.2, B).astype(np.float32))
    K = torch.from_numpy(rng.integers(0, 300, B).astype(np.int32))
    P = torch.from_numpy(rng.uniform(0.6, 1.0, B).astype(np.float32))
    MP = torch.from_numpy(rng.choice(np.array([0.0, 0.05], np.float32), B))
    tok, vstar = tsa.sample(x, T.to(DEV), K.to(DEV), P.to(DEV), MP.to(DEV), seed=9, offset=2,
                            bitmask=m.to(DEV), return_min_kept=True)
    torch.cuda.synchronize()
    fails = check_sample(big[:, :V].contiguous(), m, T, K, P, MP, 9, 2, tok.cpu(), vstar.cpu(),
                         nthreads=NT)
    assert not fails, fails[:3]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("V,S", [(8191, 8197), (40000, 40003), (1000, 1003), (3, 5)])
def test_row_kernel_misaligned_and_ragged_mixed_modes(tsa, dtype, V, S):
    """The one-CTA-per-row kernel (taken from 128 rows on): rows that start off
    16-byte boundaries (head and tail elements beside the bulk copies, mask bits
    straddling words), a short last stage, rows of one stage or none, and
    greedy, unfiltered and filtered rows side by side in one batch."""
    rng = np.random.default_rng(7 * V + S)
    B = 160
    big = torch.from_numpy((2 * rng.standard_normal((B, S))).astype(np.float32)).to(dtype)
    m = workloads.random_bitmask(rng, B, V, 0.8)
    x = big.to(DEV)[:, :V]
    T = rng.uniform(0.5, 1.2, B).astype(np.float32)
    K = rng.integers(0, 300, B).astype(np.int32)
    P = rng.uniform(0.6, 1.0, B).astype(np.float32)
    MP = rng.choice(np.array([0.0, 0.05], np.float32), B)
    T[0::7] = 0.0  # greedy rows
    K[1::7], P[1::7], MP[1::7] = 0, 1.0, 0.0  # unfiltered rows
    T, K, P, MP = (torch.from_numpy(v) for v in (T, K, P, MP))
    tok, vstar = tsa.sample(x, T.to(DEV), K.to(DEV), P.to(DEV), MP.to(DEV), seed=11, offset=3,
                            bitmask=m.to(DEV), return_min_kept=True)
    torch.cuda.synchronize()
    fails = check_sample(big[:, :V].contiguous(), m, T, K, P, MP, 11, 3, tok.cpu(), vstar.cpu(),
                         nthreads=NT)
    assert not fails, fails[:3]
    assert tsa.device_status() == 0


def test_row_kernel_edge_rows(tsa):
    """The one-CTA-per-row kernel on rows that leave its fast path: NaN logits
    (read as -inf; the normaliser is recomputed), a row of -inf only, a row
    with one finite logit, top_k above the thread-maximum bound (radix
    select), top_k = 300 on flat rows (a long candidate list), top-p alone."""
    rng = np.random.default_rng(21)
    B, V = 144, 20000
    x = (2 * rng.standard_normal((B, V))).astype(np.float32)
    nan_pos = np.zeros_like(x, dtype=bool)
    nan_pos[[3, 10]] = rng.random((2, V)) < 0.3
    x[nan_pos] = np.nan
    x[5] = -np.inf
    x[6] = -np.inf
    x[6, 123] = 0.25
    T = rng.uniform(0.6, 1.2, B).astype(np.float32)
    K = np.full(B, 50, np.int32)
    P = np.full(B, 0.9, np.float32)
    MP = np.zeros(B, np.float32)
    r = np.arange(B)
    K[r % 5 == 0] = 1500
    K[r % 5 == 1] = 300
    K[r % 5 == 2], P[r % 5 == 2] = 0, 0.5
    MP[r % 5 >= 3] = 0.05
    T, K, P, MP = (torch.from_numpy(v) for v in (T, K, P, MP))
    tok, vstar = tsa.sample(torch.from_numpy(x).to(DEV), T.to(DEV), K.to(DEV), P.to(DEV), MP.to(DEV),
                            seed=13, offset=1, return_min_kept=True)
    torch.cuda.synchronize()
    tok, vstar = tok.cpu(), vstar.cpu()
    assert int(tok[5]) == -1 and int(tok[6]) == 123
    clean = torch.from_numpy(np.where(nan_pos, -np.inf, x).astype(np.float32))
    rows = [i for i in range(B) if i != 5]
    fails = check_sample(clean, None, T, K, P, MP, 13, 1, tok, vstar, nthreads=NT, rows=rows)
    assert not fails, fails[:3]
    assert tsa.device_status() == 0


def _assert_logprob(got, ref):
    """NaN and -inf where the oracle has them; elsewhere within 1e-4 + 1e-6 |ref|
    (fp32 per-thread sums of a few hundred terms, then a block sum, bound the
    error of ln Z by a few 1e-5)."""
    got = got.double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    fin = np.isfinite(ref)
    err = np.abs(got[fin] - ref[fin])
    assert np.all(err <= 1e-4 + 1e-6 * np.abs(ref[fin])), err.max()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("V,S", [(128256, 128256), (8191, 8197), (3, 5)])
def test_selective_log_softmax_matches_oracle(tsa, dtype, V, S):
    rng = np.random.default_rng(V + 3 * S)
    B = 40
    big = torch.from_numpy((3 * rng.standard_normal((B, S))).astype(np.float32)).to(dtype)
    m = workloads.random_bitmask(rng, B, V, 0.7)
    x = big.to(DEV)[:, :V]
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    T[::9] = 0.0  # read as T = 1
    idx = rng.integers(0, V, B).astype(np.int64)
    idx[1], idx[2] = -1, V  # outside [0, V): NaN
    T = torch.from_numpy(T)
    tok = tsa.sample(x, T.to(DEV), 40, 0.9, 0.0, seed=3, bitmask=m.to(DEV)).cpu().numpy()
    idx[3::2] = tok[3::2]  # sampled tokens, allowed by construction
    got = tsa.selective_log_softmax(x, torch.from_numpy(idx).to(DEV), T.to(DEV), bitmask=m.to(DEV)).cpu()
    ref = oracle.selective_log_softmax(big[:, :V].float(), idx, T, m)
    _assert_logprob(got, ref)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_selective_log_softmax_edge_rows(tsa, dtype):
    """Rows that move every thread's reference many times (an ascending ramp over
    600 units at T = 0.3), logits near +-1e4, a fully masked row (NaN), NaN
    entries (read as -inf), a +inf entry (NaN), at a row start one element off
    16-byte alignment, each against the oracle."""
    rng = np.random.default_rng(17)
    B, V = 12, 20000
    base = (2 * rng.standard_normal((B, V + 1))).astype(np.float32)
    base[0, 1:] = np.linspace(-300.0, 300.0, V, dtype=np.float32)
    base[1, 1:] = np.where(rng.random(V) < 0.5, 1e4, -1e4).astype(np.float32) + rng.standard_normal(V).astype(np.float32)
    base[3, 1 + rng.choice(V, 50, replace=False)] = np.nan
    base[4, 1 + 777] = np.inf
    big = torch.from_numpy(base).to(dtype)
    x = big.to(DEV)[:, 1:]  # one element past a 16-byte boundary
    allowed = np.ones((B, V), bool)
    allowed[2] = False
    allowed[5:] = rng.random((B - 5, V)) < 0.6
    m = torch.from_numpy(oracle.bitmask_from_allowed(allowed))
    T = np.full(B, 1.0, np.float32)
    T[0] = 0.3
    idx = np.array([V - 1, 5, 7, 11, 13] + [int(np.nonzero(allowed[b])[0][3]) for b in range(5, B)], np.int64)
    idx[0] = V // 2
    got = tsa.selective_log_softmax(x, torch.from_numpy(idx).to(DEV), torch.from_numpy(T).to(DEV),
                                    bitmask=m.to(DEV)).cpu()
    ref = oracle.selective_log_softmax(big[:, 1:].float(), idx, torch.from_numpy(T), m)
    assert np.isnan(ref[2]) and np.isnan(ref[4]) and np.isfinite(ref[0]) and np.isfinite(ref[3])
    _assert_logprob(got, ref)


def test_selective_log_softmax_decode_batch(tsa):
    """The full decode batch, scored at the tokens ``sample`` draws from it."""
    case = workloads.decode_batch("combined", mask_density=0.7)
    x, mk = case.logits.to(DEV), case.bitmask.to(DEV)
    tok = tsa.sample(x, case.temperature, case.top_k, case.top_p, case.min_p, seed=5, offset=5, bitmask=mk)
    got = tsa.selective_log_softmax(x, tok, case.temperature, bitmask=mk).cpu()
    ref = oracle.selective_log_softmax(case.logits, tok.cpu().numpy(), case.temperature, case.bitmask)
    _assert_logprob(got, ref)
    assert np.all(np.isfinite(ref))


def test_nan_logits_treated_as_minus_inf(tsa):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((8, 3000)).astype(np.float32)
    nan_pos = rng.random(x.shape) < 0.3
    x[nan_pos] = np.nan
    xt = torch.from_numpy(x)
    for (T, k, p) in [(0.0, 0, 1.0), (1.0, 0, 1.0), (1.0, 20, 0.9)]:
        tok = tsa.sample(xt.to(DEV), T, k, p, 0.0, seed=2).cpu().numpy()
        assert not nan_pos[np.arange(8), tok].any()
    clean = np.where(nan_pos, -np.inf, x)
    tok = tsa.sample(xt.to(DEV), 0.0, 0, 1.0, 0.0, seed=0).cpu().numpy()
    assert np.array_equal(tok, np.argmax(clean, axis=1))


def test_large_k_uses_radix_path(tsa):
    """top_k above the thread-maximum bound and top_p alone take the cluster
    radix-select path; both must still match the oracle."""
    case = workloads.decode_batch("top_k", mask_density=None, rows=32)
    case.top_k = 1500
    _assert_sample(tsa, case, seed=4, offset=4)
    case.top_k = 0
    case.top_p = 0.5
    case.min_p = 0.0
    _assert_sample(tsa, case, seed=5, offset=5)


def test_maximum_vocabulary(tsa):
    for dtype in (torch.float32, torch.bfloat16):
        V = tsa.max_vocab(dtype)
        rng = np.random.default_rng(6)
        x = torch.from_numpy(rng.standard_normal((2, V)).astype(np.float32)).to(dtype)
        for (T, k, p, mp) in [(0.0, 0, 1.0, 0.0), (1.0, 40, 0.9, 0.0), (1.0, 0, 0.8, 0.0)]:
            tok, vstar = tsa.sample(x.to(DEV), T, k, p, mp, seed=1, return_min_kept=True)
            torch.cuda.synchronize()
            fails = check_sample(x, None, T, k, p, mp, 1, 0, tok.cpu(), vstar.cpu(), nthreads=NT)
            assert not fails, (dtype, fails[:3])
        with pytest.raises(tsa.TSAError):
            tsa.sample(torch.zeros(1, V + 16, dtype=dtype, device=DEV), 1.0)


def test_determinism_and_keying(tsa):
    case = workloads.decode_batch("unfiltered", mask_density=0.7, rows=64)
    a = _run_sample(tsa, case, 3, 8)[0]
    b = _run_sample(tsa, case, 3, 8)[0]
    assert torch.equal(a, b)
    assert not torch.equal(a, _run_sample(tsa, case, 3, 9)[0])
    assert not torch.equal(a, _run_sample(tsa, case, 4, 8)[0])


def test_per_row_parameters_match_broadcast(tsa):
    case = workloads.decode_batch("combined", mask_density=0.7, rows=48)
    x, m = case.logits.to(DEV), case.bitmask.to(DEV)
    B = case.B
    ref = tsa.sample(x, 0.9, 50, 0.9, 0.05, seed=2, offset=1, bitmask=m)
    per = tsa.sample(x, torch.full((B,), 0.9, device=DEV),
                     torch.full((B,), 50, dtype=torch.int32, device=DEV),
                     torch.full((B,), 0.9, device=DEV), torch.full((B,), 0.05, device=DEV),
                     seed=2, offset=1, bitmask=m)
    assert torch.equal(ref, per)


def test_exact_score_tie_goes_to_lower_index(tsa):
    from .test_oracle_select import find_equal_uniform_pair

    V = 16384
    for row in range(8):
        pair = find_equal_uniform_pair(21, 0, row, V)
        if pair:
            break
    i, j = pair
    B = row + 1
    allowed = np.ones((B, V), dtype=bool)
    allowed[row, :] = False
    allowed[row, [i, j]] = True
    m = workloads.pack_allowed(allowed)
    tok = tsa.sample(torch.zeros(B, V, device=DEV), 1.0, 0, 1.0, 0.0, seed=21, offset=0,
                     bitmask=m.to(DEV)).cpu()
    assert tok[row].item() == i


def test_draw_distribution_8_tokens(tsa):
    """100k draws (1,000 rows x 100 offsets) over 8 tokens: total variation
    against the filtered, renormalised softmax <= 0.005."""
    from scipy.special import softmax

    l = torch.tensor([2.0, 1.5, 1.0, 0.5, 0.0, -0.5, -1.0, -1.5])
    x = l.repeat(1000, 1).to(DEV)
    for (T, k, p, mp) in [(1.0, 0, 1.0, 0.0), (0.8, 6, 0.9, 0.02)]:
        counts = torch.zeros(8, dtype=torch.int64)
        for off in range(100):
            tok = tsa.sample(x, T, k, p, mp, seed=11, offset=off)
            counts += torch.bincount(tok.cpu(), minlength=8)
        q = softmax(l.double().numpy() / T)
        keep = np.arange(8) < (k if k > 0 else 8)
        keep &= np.concatenate([[0.0], np.cumsum(q)[:-1]]) < p
        keep &= q / q.max() >= mp
        target = np.where(keep, q, 0.0)
        target /= target.sum()
        emp = counts.numpy() / counts.sum().item()
        assert counts.numpy()[~keep].sum() == 0
        assert 0.5 * np.abs(emp - target).sum() <= 0.005


# ------------------------------------------------------------------ topk
@pytest.mark.parametrize("k", [1, 50, 100, 2048])
def test_topk_large_vocab_planted(tsa, k):
    x, info = workloads.topk_large(k)
    vals, idx = tsa.topk(x.to(DEV), k)
    torch.cuda.synchronize()
    v_o, i_o = oracle.topk(x, k, nthreads=NT)
    assert np.array_equal(idx.cpu().numpy(), i_o)
    assert np.array_equal(vals.cpu().double().numpy(), v_o)
    # winners strictly above the k-th value all sit in the planted chunk (the
    # tie plant may move boundary ties elsewhere; at k = 2048 the whole chunk
    # is planted and the background's tail can pass the chunk's minimum)
    for b, c in info["planted"] if k < 2048 else []:
        above = v_o[b] > v_o[b, -1]
        assert np.all(i_o[b][above] // 2048 == c)
    assert tsa.device_status() == 0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("V,S,k", [(1, 1, 1), (7, 9, 7), (2049, 2049, 2048), (8192, 8192, 10),
                                   (33333, 33335, 300), (128257, 128257, 50)])
def test_topk_shapes_and_ties(tsa, dtype, V, S, k):
    rng = np.random.default_rng(V + k)
    B = 6
    big = torch.from_numpy(np.round(rng.standard_normal((B, S)) * 8) / 8).float().to(dtype)
    big[0, : min(V, 5)] = -0.0
    big[1, :] = 1.0  # a whole row of ties
    x = big.to(DEV)[:, :V]
    vals, idx = tsa.topk(x, k)
    torch.cuda.synchronize()
    ref = big[:, :V].contiguous()
    v_o, i_o = oracle.topk(ref, k, nthreads=NT)
    assert np.array_equal(idx.cpu().numpy(), i_o)
    assert np.array_equal(vals.cpu().double().numpy(), v_o)
    # exact copies: the sign of zero survives
    got_bits = vals.cpu().numpy().view(np.uint32)
    ref_bits = ref.float().numpy()[np.arange(B)[:, None], i_o].view(np.uint32)
    assert np.array_equal(got_bits, ref_bits)


def test_topk_matches_torch_topk(tsa):
    rng = np.random.default_rng(16)
    x = torch.from_numpy(rng.standard_normal((8, 248320)).astype(np.float32))
    for k in [1, 50, 100]:
        v, i = tsa.topk(x.to(DEV), k)
        rv, ri = torch.topk(x, k, dim=1)
        assert torch.equal(i.cpu(), ri) and torch.equal(v.cpu(), rv)
    assert torch.equal(tsa.topk(x.to(DEV), 1)[1][:, 0].cpu(), torch.argmax(x, dim=1))


def test_topk_deterministic(tsa):
    x, _ = workloads.topk_large(100)
    xd = x.to(DEV)
    a = tsa.topk(xd, 100)
    b = tsa.topk(xd, 100)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ------------------------------------------------------------------ failure path
def test_bounded_wait_reports_timeout(tsa):
    """A kernel waiting on a barrier that nothing completes gives up after its
    limit, records the flag, and the context stays usable."""
    lib = tsa.load_library()
    assert tsa.device_status() == 0
    assert lib.tsa_selftest_wait_timeout(2000, None) == 0
    assert tsa.device_status(clear=True) == -8
    assert tsa.device_status() == 0
    tok = tsa.sample(torch.zeros(2, 100, device=DEV), 0.0)
    assert tok.cpu().tolist() == [0, 0]
