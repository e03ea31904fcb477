"""Host-side checks of the C ABI (no GPU work): the library builds, loads and
exports every function include/tsa.h declares; argument validation returns
the documented status before anything is launched."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tsa.h")


@pytest.fixture(scope="module")
def lib():
    from top_sampling_apply_gb300 import _build

    _build.build()
    import top_sampling_apply_gb300 as tsa

    return tsa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tsa_[a-z0-9_]+)\s*\(", text)))


def status_codes():
    text = open(HEADER).read()
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"(TSA_[A-Z_]+)\s*=\s*(-?\d+)", text)}


S = status_codes()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"tsa_apply_token_bitmask", "tsa_sample", "tsa_topk"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for name, code in S.items():
        if name.startswith("TSA_ERR") or name == "TSA_OK":
            s = lib.tsa_status_string(code)
            assert s and s != b"unknown status", name
    assert lib.tsa_status_string(12345) == b"unknown status"


def test_workspace_queries(lib):
    # below 128 rows the rows are split across the GPU (slice summaries and
    # candidate lists); from 128 rows on one CTA resolves each row on chip
    n = lib.tsa_sample_workspace_bytes(127, 128256, 0)
    assert 0 < n < 64 << 20
    assert 0 < lib.tsa_sample_workspace_bytes(32, 128256, 0) < n
    assert 0 < lib.tsa_sample_workspace_bytes(1, 8192, 2)
    for B in (128, 129, 256, 512, 1024, 1 << 20):
        for dt, V in ((0, 128256), (2, 256000), (1, 32000)):
            assert lib.tsa_sample_workspace_bytes(B, V, dt) == 0, (B, V, dt)
    assert lib.tsa_sample_workspace_bytes(0, 128256, 0) == 0
    assert lib.tsa_sample_workspace_bytes(-1, 128256, 0) == 0
    assert lib.tsa_sample_workspace_bytes(4, 0, 0) == 0
    assert lib.tsa_topk_workspace_bytes(8, 248320, 2048, 0) == 0


def test_max_vocab(lib):
    f32, bf16 = lib.tsa_max_vocab(0), lib.tsa_max_vocab(2)
    assert f32 >= 800_000 and bf16 >= 1_600_000 and lib.tsa_max_vocab(1) == bf16


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first


def _sample(lib, logits=FAKE, dtype=0, B=4, V=100, stride=100, mask=None, mstride=0, tokens=FAKE,
            T=None, K=None, P=None, M=None, ws=None, nws=0):
    return lib.tsa_sample(logits, dtype, B, V, stride, mask, mstride, T, 1.0, K, 0, P, 1.0, M, 0.0,
                          0, 0, tokens, None, ws, nws, None)


def test_sample_validation(lib):
    assert _sample(lib, logits=None) == S["TSA_ERR_NULL"]
    assert _sample(lib, tokens=None) == S["TSA_ERR_NULL"]
    assert _sample(lib, dtype=7) == S["TSA_ERR_DTYPE"]
    assert _sample(lib, V=0) == S["TSA_ERR_SHAPE"]
    assert _sample(lib, B=-1) == S["TSA_ERR_SHAPE"]
    assert _sample(lib, stride=99) == S["TSA_ERR_SHAPE"]
    assert _sample(lib, V=lib.tsa_max_vocab(0) + 1, stride=10**7) == S["TSA_ERR_SHAPE"]
    assert _sample(lib, mask=FAKE, mstride=3) == S["TSA_ERR_STRIDE"]
    assert _sample(lib, logits=ctypes.c_void_p(0x10002)) == S["TSA_ERR_ALIGN"]
    assert _sample(lib, tokens=ctypes.c_void_p(0x10004)) == S["TSA_ERR_ALIGN"]
    assert _sample(lib, T=ctypes.c_void_p(0x10001)) == S["TSA_ERR_ALIGN"]
    assert _sample(lib, B=0) == S["TSA_OK"]  # empty batch: no launch
    # from 128 rows no workspace is needed, but every other check still holds
    assert _sample(lib, B=256, tokens=None) == S["TSA_ERR_NULL"]
    assert _sample(lib, B=256, mask=FAKE, mstride=3) == S["TSA_ERR_STRIDE"]
    need = lib.tsa_sample_workspace_bytes(4, 100, 0)
    assert _sample(lib) == S["TSA_ERR_WORKSPACE"]
    assert _sample(lib, ws=FAKE, nws=need - 1) == S["TSA_ERR_WORKSPACE"]
    assert _sample(lib, ws=ctypes.c_void_p(0x10010), nws=need) == S["TSA_ERR_ALIGN"]


def test_topk_validation(lib):
    def tk(k=10, V=100, B=2, vals=FAKE, idx=FAKE, dtype=0):
        return lib.tsa_topk(FAKE, dtype, B, V, V, k, vals, idx, None, 0, None)

    assert tk(k=0) == S["TSA_ERR_K_RANGE"]
    assert tk(k=2049, V=5000) == S["TSA_ERR_K_RANGE"]
    assert tk(k=101) == S["TSA_ERR_K_RANGE"]
    assert tk(vals=None) == S["TSA_ERR_NULL"]
    assert tk(idx=ctypes.c_void_p(0x10004)) == S["TSA_ERR_ALIGN"]
    assert tk(dtype=3) == S["TSA_ERR_DTYPE"]
    assert tk(B=0) == S["TSA_OK"]


def test_bitmask_validation(lib):
    f = lib.tsa_apply_token_bitmask
    assert f(FAKE, 0, 2, 100, 100, None, 4, None) == S["TSA_ERR_NULL"]
    assert f(FAKE, 0, 2, 100, 100, FAKE, 3, None) == S["TSA_ERR_STRIDE"]
    assert f(FAKE, 2, 2, 100, 100, ctypes.c_void_p(0x10002), 4, None) == S["TSA_ERR_ALIGN"]
    assert f(FAKE, 0, 0, 100, 100, FAKE, 4, None) == S["TSA_OK"]


def test_selective_log_softmax_validation(lib):
    def lp(B=2, V=100, stride=100, mask=None, mstride=0, T=None, idx=FAKE, out=FAKE, dtype=0, logits=FAKE):
        return lib.tsa_selective_log_softmax(logits, dtype, B, V, stride, mask, mstride, T, 1.0, idx, out, None)

    assert lp(idx=None) == S["TSA_ERR_NULL"]
    assert lp(out=None) == S["TSA_ERR_NULL"]
    assert lp(logits=None) == S["TSA_ERR_NULL"]
    assert lp(dtype=5) == S["TSA_ERR_DTYPE"]
    assert lp(stride=99) == S["TSA_ERR_SHAPE"]
    assert lp(mask=FAKE, mstride=3) == S["TSA_ERR_STRIDE"]
    assert lp(idx=ctypes.c_void_p(0x10004)) == S["TSA_ERR_ALIGN"]
    assert lp(out=ctypes.c_void_p(0x10002)) == S["TSA_ERR_ALIGN"]
    assert lp(B=0, idx=None, out=None) == S["TSA_OK"]


def test_binding_rejects_cpu_tensors():
    import torch

    import top_sampling_apply_gb300 as tsa

    with pytest.raises(ValueError):
        tsa.sample(torch.zeros(2, 10), 1.0)
    with pytest.raises(ValueError):
        tsa.topk(torch.zeros(2, 10), 3)
    with pytest.raises(ValueError):
        tsa.sample(torch.zeros(2, 10), 1.0, 5, 0.9, sequential=True)
    with pytest.raises(ValueError):
        tsa.sample_icdf(torch.zeros(2, 10), torch.rand(2))
    with pytest.raises(ValueError):
        tsa.bitmask_from_allowed(torch.zeros(2, 10, dtype=torch.bool))
    with pytest.raises(ValueError):
        tsa.lm_head_topk(torch.zeros(1, 64, dtype=torch.bfloat16), torch.zeros(100, 64, dtype=torch.bfloat16), 5)


def _a256(n):
    return (n + 255) // 256 * 256


def test_sequential_validation(lib):
    def seq(logits=FAKE, B=4, V=100, stride=100, mask=None, mstride=0, tokens=FAKE, ws=None, nws=0):
        return lib.tsa_sample_sequential(logits, 0, B, V, stride, mask, mstride, None, 1.0, None, 50, None, 0.9,
                                         None, 0.0, 0, 0, tokens, None, ws, nws, None)

    assert seq(logits=None) == S["TSA_ERR_NULL"]
    assert seq(tokens=None) == S["TSA_ERR_NULL"]
    assert seq(V=0) == S["TSA_ERR_SHAPE"]
    assert seq(stride=99) == S["TSA_ERR_SHAPE"]
    assert seq(mask=FAKE, mstride=3) == S["TSA_ERR_STRIDE"]
    assert seq(B=0) == S["TSA_OK"]
    # the survivors' bitmask (B ceil(V / 32) words) and the B top-k cuts, each
    # rounded up to 256 bytes, then the sample call's own workspace
    need = lib.tsa_sample_sequential_workspace_bytes(4, 100, 0)
    assert need == _a256(4 * 4 * 4) + _a256(4 * 4) + lib.tsa_sample_workspace_bytes(4, 100, 0)
    assert lib.tsa_sample_sequential_workspace_bytes(256, 128256, 0) == _a256(256 * 4008 * 4) + _a256(256 * 4)
    assert lib.tsa_sample_sequential_workspace_bytes(0, 100, 0) == 0
    assert seq() == S["TSA_ERR_WORKSPACE"]
    assert seq(ws=FAKE, nws=need - 1) == S["TSA_ERR_WORKSPACE"]
    assert seq(ws=ctypes.c_void_p(0x10010), nws=need) == S["TSA_ERR_ALIGN"]
    # from 128 rows the workspace holds only the bitmask and the cuts
    assert seq(B=256, V=128256, stride=128256) == S["TSA_ERR_WORKSPACE"]


def test_icdf_validation(lib):
    def icdf(logits=FAKE, B=4, u=FAKE, vout=FAKE, tokens=FAKE, ws=None, nws=0):
        return lib.tsa_sample_icdf(logits, 0, B, 100, 100, None, 0, None, 1.0, None, 0, None, 1.0, None, 0.0,
                                   u, tokens, vout, ws, nws, None)

    assert icdf(logits=None) == S["TSA_ERR_NULL"]
    assert icdf(u=None) == S["TSA_ERR_NULL"]
    assert icdf(vout=None) == S["TSA_ERR_NULL"]  # v* is the draw's keep-threshold
    assert icdf(u=ctypes.c_void_p(0x10002)) == S["TSA_ERR_ALIGN"]
    assert icdf(B=0, u=None, vout=None) == S["TSA_OK"]
    # below 128 rows the sample call that fixes v* needs its workspace
    assert icdf() == S["TSA_ERR_WORKSPACE"]


def test_bitmask_from_allowed_validation(lib):
    f = lib.tsa_bitmask_from_allowed
    assert f(FAKE, 2, 100, 100, None, 4, None) == S["TSA_ERR_NULL"]
    assert f(None, 2, 100, 100, FAKE, 4, None) == S["TSA_ERR_NULL"]
    assert f(FAKE, 2, 0, 100, FAKE, 4, None) == S["TSA_ERR_SHAPE"]
    assert f(FAKE, 2, 100, 99, FAKE, 4, None) == S["TSA_ERR_SHAPE"]
    assert f(FAKE, -1, 100, 100, FAKE, 4, None) == S["TSA_ERR_SHAPE"]
    assert f(FAKE, 2, 100, 100, FAKE, 3, None) == S["TSA_ERR_STRIDE"]
    assert f(FAKE, 2, 100, 100, ctypes.c_void_p(0x10002), 4, None) == S["TSA_ERR_ALIGN"]
    assert f(FAKE, 0, 100, 100, FAKE, 4, None) == S["TSA_OK"]


def test_lm_head_topk_validation(lib):
    def lh(hidden=FAKE, M=1, H=64, hs=64, weight=FAKE, V=1000, wst=64, bias=None, k=10, vals=FAKE, idx=FAKE,
           ws=None, nws=0):
        return lib.tsa_lm_head_topk(hidden, M, H, hs, weight, V, wst, bias, k, vals, idx, ws, nws, None)

    for kw in ({"M": 5}, {"M": -1}, {"H": 4}, {"H": 12}, {"H": 8200}, {"hs": 32}, {"wst": 32}, {"V": 0}):
        assert lh(**kw) == S["TSA_ERR_SHAPE"], kw
    assert lh(k=0) == S["TSA_ERR_K_RANGE"]
    assert lh(k=2049, V=5000) == S["TSA_ERR_K_RANGE"]
    assert lh(k=1001) == S["TSA_ERR_K_RANGE"]
    assert lh(M=0) == S["TSA_OK"]
    assert lh(hidden=None) == S["TSA_ERR_NULL"]
    assert lh(weight=None) == S["TSA_ERR_NULL"]
    assert lh(idx=None) == S["TSA_ERR_NULL"]
    assert lh(hidden=ctypes.c_void_p(0x10008)) == S["TSA_ERR_ALIGN"]  # rows are read in 16-byte vectors
    assert lh(hs=68) == S["TSA_ERR_ALIGN"]
    assert lh(idx=ctypes.c_void_p(0x10004)) == S["TSA_ERR_ALIGN"]
    need = lib.tsa_lm_head_topk_workspace_bytes(1, 1000, 10)
    assert need > 0
    assert lib.tsa_lm_head_topk_workspace_bytes(0, 1000, 10) == 0
    assert lib.tsa_lm_head_topk_workspace_bytes(5, 1000, 10) == 0
    assert lh() == S["TSA_ERR_WORKSPACE"]
    assert lh(ws=FAKE, nws=need - 1) == S["TSA_ERR_WORKSPACE"]
    assert lh(ws=ctypes.c_void_p(0x10010), nws=need) == S["TSA_ERR_ALIGN"]
