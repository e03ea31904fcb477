"""tsa_sample_noalloc: the sample call with the library's fixed device scratch
instead of a caller workspace, for callers that cannot allocate device
memory.  On the GPU it must give exactly what tsa_sample gives on the same
inputs, call after call, although every call reuses one scratch array that
still holds the previous call's contents.  Only batches under 128 rows use
the scratch (larger ones resolve every row on chip), so the consecutive calls
below are small batches of different shapes and element types.  This file is
named so that pytest collects it last; it passes alone in a fresh process as
well."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import workloads

from .parity import check_sample

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DEV = "cuda:0"
TSA_OK, TSA_ERR_NULL, TSA_ERR_SHAPE, TSA_ERR_STRIDE, TSA_ERR_WORKSPACE, TSA_ERR_ALIGN = 0, -1, -2, -5, -6, -9
FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every call below fails before device work
NT = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module")
def tsa():
    import __graft_entry__

    __graft_entry__.build()
    import top_sampling_apply_gb300 as lib

    lib.load_library()
    return lib


def _call(lib, B, V, dtype=0, logits=FAKE, tokens=FAKE, mask=None, mstride=0, stride=None):
    return lib.tsa_sample_noalloc(logits, dtype, B, V, V if stride is None else stride, mask, mstride,
                                  None, 1.0, None, 0, None, 1.0, None, 0.0, 0, 0, tokens, None, None)


def test_noalloc_limit_matches_header(tsa):
    text = open(os.path.join(ROOT, "include", "tsa.h")).read()
    m = re.search(r"#define TSA_SAMPLE_NOALLOC_SCRATCH_BYTES \((\d+)u \* 1024u \* 1024u\)", text)
    assert m and int(m.group(1)) * 1024 * 1024 == tsa.sample_noalloc_max_bytes()


def test_noalloc_rejects_sizes_beyond_its_scratch(tsa):
    """Checked before any device work, so this runs without a GPU."""
    lib = tsa.load_library()
    cap = tsa.sample_noalloc_max_bytes()
    refused = 0
    for dtype in (0, 1, 2):
        V = lib.tsa_max_vocab(dtype)
        for B in (1, 16, 64, 127):
            need = lib.tsa_sample_workspace_bytes(B, V, dtype)
            if need > cap:
                refused += 1
                assert _call(lib, B, V, dtype) == TSA_ERR_WORKSPACE, (dtype, B)
                # an invalid call reports what tsa_sample would, whatever its size
                assert _call(lib, B, V, dtype, logits=None) == TSA_ERR_NULL
                assert _call(lib, B, V, dtype, tokens=None) == TSA_ERR_NULL
                assert _call(lib, B, V, dtype, mask=FAKE, mstride=3) == TSA_ERR_STRIDE
                assert _call(lib, B, V, dtype, stride=V - 1) == TSA_ERR_SHAPE
                assert _call(lib, B, V, dtype, tokens=ctypes.c_void_p(0x10004)) == TSA_ERR_ALIGN
    assert refused > 0  # the limit is reachable: 64 rows of the largest vocabulary are refused
    # the documented example, and batches that need no scratch at all
    assert lib.tsa_sample_workspace_bytes(64, 800000, 0) > cap
    for B in (128, 256, 512, 4096):
        assert lib.tsa_sample_workspace_bytes(B, lib.tsa_max_vocab(0), 0) == 0
    assert lib.tsa_sample_workspace_bytes(127, 128256, 0) <= cap
    assert _call(lib, 0, 128256) == TSA_OK
    assert _call(lib, 4, 0) == TSA_ERR_SHAPE


def _on_device(case):
    dev_param = lambda p: p.to(DEV) if isinstance(p, torch.Tensor) else p  # noqa: E731
    return dict(logits=case.logits.to(DEV),
                bitmask=None if case.bitmask is None else case.bitmask.to(DEV),
                temperature=dev_param(case.temperature), top_k=dev_param(case.top_k),
                top_p=dev_param(case.top_p), min_p=dev_param(case.min_p))


def _bf16_large_vocab(B=16, V=248320, seed=31):
    """bf16 rows of a 248,320-entry vocabulary with per-row parameters and a
    half-density mask: its rows take 15 slices each in the scratch."""
    rng = np.random.default_rng(seed)
    x = torch.from_numpy((1.5 * rng.standard_normal((B, V))).astype(np.float32)).to(torch.bfloat16)
    mask = workloads.random_bitmask(rng, B, V, 0.5)
    T = rng.uniform(0.4, 1.2, B).astype(np.float32)
    T[0] = 0.0
    K = rng.integers(0, 80, B).astype(np.int32)
    P = rng.uniform(0.6, 1.0, B).astype(np.float32)
    MP = rng.choice(np.array([0.0, 0.05], np.float32), B)
    return workloads.SampleCase("bf16_v248320", x, mask, torch.from_numpy(T), torch.from_numpy(K),
                                torch.from_numpy(P), torch.from_numpy(MP))


@pytest.mark.gpu
def test_noalloc_equals_workspace_sample_on_consecutive_calls(tsa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = tsa.load_library()
    # batches under 128 rows (split rows: the scratch holds slice summaries and
    # candidates), one after another, each finding the previous call's
    # contents in the scratch; then the tiny case again
    cases = [(workloads.tiny_case(), 11, 5),
             (workloads.decode_batch("combined", mask_density=0.7, rows=32), 12, 6),
             (_bf16_large_vocab(), 13, 7),
             (workloads.tiny_case(), 14, 8)]
    for case, _, _ in cases:
        need = lib.tsa_sample_workspace_bytes(case.B, case.V, {torch.float32: 0, torch.float16: 1,
                                                               torch.bfloat16: 2}[case.logits.dtype])
        assert 0 < need <= tsa.sample_noalloc_max_bytes()
    inputs = [_on_device(c) for c, _, _ in cases]
    refs = []
    for d, (_, seed, offset) in zip(inputs, cases):
        tok, vstar = tsa.sample(d["logits"], d["temperature"], d["top_k"], d["top_p"], d["min_p"],
                                seed=seed, offset=offset, bitmask=d["bitmask"], return_min_kept=True)
        refs.append((tok, vstar))
    outs = [(torch.full((d["logits"].shape[0],), -7, dtype=torch.int64, device=DEV),
             torch.zeros(d["logits"].shape[0], dtype=torch.float32, device=DEV)) for d in inputs]
    torch.cuda.synchronize()
    before = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    for d, (_, seed, offset), (tok, vstar) in zip(inputs, cases, outs):
        tsa.sample_noalloc(d["logits"], tok, d["temperature"], d["top_k"], d["top_p"], d["min_p"],
                           seed=seed, offset=offset, bitmask=d["bitmask"], min_kept_out=vstar)
    torch.cuda.synchronize()
    assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == before
    for i, ((rt, rv), (t, v)) in enumerate(zip(refs, outs)):
        # the same kernels on the same inputs: tokens and v* agree exactly
        assert torch.equal(t, rt), "call %d: %d tokens differ" % (i, int((t != rt).sum()))
        torch.testing.assert_close(v, rv, rtol=0, atol=0, equal_nan=True)
    # and the 32 decode rows agree with the oracle under the parity rules
    case, seed, offset = cases[1]
    fails = check_sample(case.logits, case.bitmask, case.temperature, case.top_k, case.top_p, case.min_p,
                         seed, offset, outs[1][0].cpu(), outs[1][1].cpu(), nthreads=NT)
    assert not fails, fails[:3]
    assert tsa.device_status() == 0


@pytest.mark.gpu
def test_noalloc_large_peaked_batch_matches_oracle(tsa):
    """B=512, V=256,000 bf16 (one CTA per row, no scratch): accepted, and every
    row within the parity rules."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    case = workloads.peaked_batch()
    d = _on_device(case)
    tok = torch.empty(case.B, dtype=torch.int64, device=DEV)
    vstar = torch.empty(case.B, dtype=torch.float32, device=DEV)
    for t in (0, 63):
        tsa.sample_noalloc(d["logits"], tok, case.temperature, case.top_k, case.top_p, case.min_p,
                           seed=t, offset=t, bitmask=d["bitmask"], min_kept_out=vstar)
        torch.cuda.synchronize()
        fails = check_sample(case.logits, case.bitmask, case.temperature, case.top_k, case.top_p,
                             case.min_p, t, t, tok.cpu(), vstar.cpu(), nthreads=NT)
        assert not fails, fails[:3]
    assert tsa.device_status() == 0
