"""tsa_sample_noalloc: the sample call with the library's fixed device scratch
instead of a caller workspace, for callers that cannot allocate device
memory.  On the GPU it must give exactly what tsa_sample gives on the same
inputs, call after call, although every call reuses one scratch array that
still holds the previous call's contents.  This file is named so that pytest
collects it last; it passes alone in a fresh process as well."""
import os
import re

import pytest
import torch

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DEV = "cuda:0"
TSA_ERR_SHAPE, TSA_ERR_WORKSPACE = -2, -6


@pytest.fixture(scope="module")
def tsa():
    import __graft_entry__

    __graft_entry__.build()
    import top_sampling_apply_gb300 as lib

    lib.load_library()
    return lib


def _call(lib, B, V, dtype=0):
    return lib.tsa_sample_noalloc(None, dtype, B, V, V, None, 0, None, 1.0, None, 0, None, 1.0,
                                  None, 0.0, 0, 0, None, None, None)


def test_noalloc_limit_matches_header(tsa):
    text = open(os.path.join(ROOT, "include", "tsa.h")).read()
    m = re.search(r"#define TSA_SAMPLE_NOALLOC_SCRATCH_BYTES \((\d+)u \* 1024u \* 1024u\)", text)
    assert m and int(m.group(1)) * 1024 * 1024 == tsa.sample_noalloc_max_bytes()


def test_noalloc_rejects_sizes_beyond_its_scratch(tsa):
    """Checked before any device work, so this runs without a GPU."""
    lib = tsa.load_library()
    cap = tsa.sample_noalloc_max_bytes()
    for dtype, V in ((0, 128256), (2, 248320), (0, 4096)):
        B = 1
        while lib.tsa_sample_workspace_bytes(B, V, dtype) <= cap:
            B *= 2
        assert _call(lib, B, V, dtype) == TSA_ERR_WORKSPACE
    # the documented example: 508 rows of a 128256-entry fp32 vocabulary fit, 509 do not
    assert lib.tsa_sample_workspace_bytes(508, 128256, 0) <= cap
    assert _call(lib, 509, 128256) == TSA_ERR_WORKSPACE
    assert _call(lib, 0, 128256) == 0
    assert _call(lib, 4, 0) == TSA_ERR_SHAPE


def _on_device(case):
    dev_param = lambda p: p.to(DEV) if isinstance(p, torch.Tensor) else p  # noqa: E731
    return dict(logits=case.logits.to(DEV),
                bitmask=None if case.bitmask is None else case.bitmask.to(DEV),
                temperature=dev_param(case.temperature), top_k=dev_param(case.top_k),
                top_p=dev_param(case.top_p), min_p=dev_param(case.min_p))


@pytest.mark.gpu
def test_noalloc_equals_workspace_sample_on_consecutive_calls(tsa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    # the fused decode workload (B=256, V=128256 f32, mask density 0.7), then
    # a heterogeneous bf16 batch of different shape and per-row parameters,
    # then the first one again: each call finds the previous one's scratch
    cases = [(workloads.decode_batch("combined", mask_density=0.7), 11, 5),
             (workloads.hetero_batch(), 12, 6),
             (workloads.decode_batch("combined", mask_density=0.7), 13, 7)]
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
        # the same kernels on the same inputs: the tokens and v* agree exactly
        # (inside the oracle parity tolerance, which allows v* a few ulps)
        assert torch.equal(t, rt), "call %d: %d tokens differ" % (i, int((t != rt).sum()))
        torch.testing.assert_close(v, rv, rtol=0, atol=0, equal_nan=True)
    assert tsa.device_status() == 0
