"""CPU-side checks of the C ABI: the library builds, loads without a GPU,
exports every entry point include/fa.h declares, and rejects bad arguments on
the host before touching the device."""
import ctypes
import os
import re

import pytest

import exact_io_aware_03_gb300 as fa
from exact_io_aware_03_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.load()


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names.update(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_status_string",
              "fa_get_last_device_error", "fa_bwd_preprocess", "fa_bwd_main",
              "fa_bwd_postprocess"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_status_strings(lib):
    for s in range(5):
        assert fa.fa_status_string(s).startswith("FA_")
    assert fa.fa_status_string(99) == "unknown fa_status"


def test_workspace_size(lib):
    B, H, Nq, Nk, d = 4, 16, 4096, 4096, 128
    rows = B * H * Nq
    r256 = lambda x: (x + 255) // 256 * 256
    # statistics, the fp32 dQ accumulator and 256 bytes for the main kernel's
    # work-item counter
    assert fa.fa_bwd_workspace_size(B, H, Nq, Nk, d) == 2 * r256(rows * 4) + r256(rows * d * 4) + 256
    assert fa.fa_bwd_workspace_size(0, 1, 1, 1, 64) == 0
    # per-row statistics are padded to 128 rows per head
    assert fa.fa_bwd_workspace_size(1, 1, 3, 1, 64) == 2 * 512 + 768 + 256
    assert fa.fa_bwd_workspace_size(2, 3, 129, 5, 128) == (2 * r256(6 * 256 * 4) + r256(6 * 129 * 512)
                                                           + 256)


FAKE = 1 << 20          # 16-byte aligned, never dereferenced: rejected before any launch


@pytest.mark.parametrize("args,expect", [
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=0), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nq=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nk=-1), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(dtype=7), fa.FA_ERR_INVALID_ARG),
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(o=None), fa.FA_ERR_INVALID_ARG),
    (dict(lse=None), fa.FA_ERR_INVALID_ARG),          # bf16 path always writes LSE
    (dict(k=FAKE + 8), fa.FA_ERR_INVALID_ARG),        # misaligned
    (dict(key_bias=FAKE + 2), fa.FA_ERR_INVALID_ARG),
    (dict(B=1 << 16, H=1 << 15), fa.FA_ERR_INVALID_ARG),
    (dict(Nq=1 << 25), fa.FA_ERR_INVALID_ARG),        # Nq * d overflows 31 bits
])
def test_fwd_rejects_bad_arguments_on_host(lib, args, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, key_bias=None, o=FAKE, lse=FAKE, B=1, H=1, Nq=16, Nk=16,
             d=64, scale=0.125, causal=0, dtype=fa.FA_DTYPE_BF16, stream=None)
    a.update(args)
    assert fa.fa_fwd(**a) == expect


@pytest.mark.parametrize("args,expect", [
    (dict(dtype=fa.FA_DTYPE_FP32), fa.FA_ERR_UNSUPPORTED),
    (dict(d=32), fa.FA_ERR_UNSUPPORTED),
    (dict(workspace=None), fa.FA_ERR_INVALID_ARG),
    (dict(workspace=FAKE + 16), fa.FA_ERR_INVALID_ARG),   # not 256-byte aligned
    (dict(workspace_bytes=100), fa.FA_ERR_INVALID_ARG),
    (dict(dO=None), fa.FA_ERR_INVALID_ARG),
    (dict(dv=FAKE + 4), fa.FA_ERR_INVALID_ARG),
    (dict(lse=FAKE + 2), fa.FA_ERR_INVALID_ARG),
])
@pytest.mark.parametrize("fn", ["fa_bwd", "fa_bwd_preprocess", "fa_bwd_main",
                                "fa_bwd_postprocess"])
def test_bwd_rejects_bad_arguments_on_host(lib, args, expect, fn):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dO=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
             key_bias=None, B=1, H=1, Nq=16, Nk=16, d=64, scale=0.125, causal=1,
             dtype=fa.FA_DTYPE_BF16, workspace=FAKE, workspace_bytes=1 << 20, stream=None)
    a.update(args)
    assert getattr(fa, fn)(**a) == expect


def test_binding_refuses_to_run_without_the_library(tmp_path):
    import importlib
    mod = importlib.import_module("exact_io_aware_03_gb300")
    saved = mod._lib
    try:
        mod._lib = None
        with pytest.raises(ImportError):
            mod.load(str(tmp_path / "missing.so"))
    finally:
        mod._lib = saved


def test_splitkv_workspace_and_validation(lib):
    B, H, Nq, Nk, d, S = 2, 3, 5, 1000, 128, 4
    rows = S * B * H * Nq
    r256 = lambda x: (x + 255) // 256 * 256
    assert fa.fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, S) == r256(rows * d * 4) + r256(rows * 4)
    assert fa.fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, 0) == 0
    assert fa.fa_fwd_splitkv_default_splits(B, H, Nq, Nk, d) >= 1
    a = dict(q=FAKE, k=FAKE, v=FAKE, key_bias=None, o=FAKE, lse=FAKE, B=B, H=H, H_kv=H, Nq=Nq,
             Nk=Nk, d=d, scale=0.1, causal=0, num_splits=S, workspace=FAKE,
             workspace_bytes=1 << 30, stream=None)
    for bad in (dict(num_splits=0), dict(workspace=None), dict(workspace_bytes=16),
                dict(workspace=FAKE + 64), dict(lse=None), dict(d=80), dict(H_kv=2)):
        b = dict(a)
        b.update(bad)
        st = fa.fa_fwd_splitkv(**b)
        assert st in (fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED), bad


def _sm_count():
    import torch
    if torch.cuda.is_available():
        return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return 148   # the library's count when it cannot query a device


@pytest.mark.parametrize("B,H,Nq,Nk,d", [(8, 32, 1, 32768, 128), (1, 32, 1, 8192, 128),
                                         (2, 16, 1, 65536, 128), (16, 32, 1, 4096, 128),
                                         (4, 8, 1, 16384, 64), (1, 1, 1, 300, 64),
                                         (4, 16, 2048, 2048, 64), (1, 2, 700, 100000, 128)])
def test_splitkv_default_split_count(lib, B, H, Nq, Nk, d):
    """The default split count: among 1 .. min(128, key tiles / 4) splits, the
    one with the least waves(s) * (key tiles per split + 3), where a wave is
    one CTA per SM and a CTA is one (head, query-tile pair, split); the
    smallest such count on ties."""
    sms = _sm_count()
    ctas = B * H * ((Nq + 255) // 256)
    n_kv = (Nk + 127) // 128
    max_s = max(1, min(128, n_kv // 4))
    cost = {s: -(-ctas * s // sms) * (-(-n_kv // s) + 3) for s in range(1, max_s + 1)}
    best = min(cost.values())
    want = min(s for s, c in cost.items() if c == best)
    got = fa.fa_fwd_splitkv_default_splits(B, H, Nq, Nk, d)
    assert 1 <= got <= max_s
    assert got == want, (got, want, cost[got], best)


@pytest.mark.parametrize("H,H_kv", [(8, 3), (8, 0), (4, 8), (4, -1)])
def test_gqa_rejects_bad_head_counts(lib, H, H_kv):
    a = dict(q=FAKE, k=FAKE, v=FAKE, key_bias=None, o=FAKE, lse=FAKE, B=1, H=H, H_kv=H_kv, Nq=16,
             Nk=16, d=64, scale=0.125, causal=0, dtype=fa.FA_DTYPE_BF16, stream=None)
    assert fa.fa_fwd_gqa(**a) == fa.FA_ERR_INVALID_ARG
    b = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dO=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
             key_bias=None, B=1, H=H, H_kv=H_kv, Nq=16, Nk=16, d=64, scale=0.125, causal=1,
             dtype=fa.FA_DTYPE_BF16, workspace=FAKE, workspace_bytes=1 << 20, stream=None)
    assert fa.fa_bwd_gqa(**b) == fa.FA_ERR_INVALID_ARG


def test_deterministic_backward_workspace_and_validation(lib):
    B, H, Nq, d = 2, 3, 129, 128
    r256 = lambda x: (x + 255) // 256 * 256
    # only D and the base-2 LSE, 128-row padded per head: no dQ accumulator
    assert fa.fa_bwd_deterministic_workspace_size(B, H, Nq, d) == 2 * r256(B * H * 256 * 4)
    assert fa.fa_bwd_deterministic_workspace_size(0, H, Nq, d) == 0
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dO=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
             key_bias=None, B=B, H=H, H_kv=H, Nq=Nq, Nk=300, d=d, scale=0.1, causal=1,
             dtype=fa.FA_DTYPE_BF16, workspace=FAKE,
             workspace_bytes=fa.fa_bwd_deterministic_workspace_size(B, H, Nq, d) - 1,
             stream=None)
    assert fa.fa_bwd_deterministic(**a) == fa.FA_ERR_INVALID_ARG       # workspace too small
    for bad, expect in ((dict(d=96), fa.FA_ERR_UNSUPPORTED), (dict(H_kv=2), fa.FA_ERR_INVALID_ARG),
                        (dict(workspace=FAKE + 64), fa.FA_ERR_INVALID_ARG),
                        (dict(dtype=fa.FA_DTYPE_FP32), fa.FA_ERR_UNSUPPORTED)):
        b = dict(a, workspace_bytes=1 << 30)
        b.update(bad)
        assert fa.fa_bwd_deterministic(**b) == expect, bad
    for stage in (0, 4, -1):
        assert fa.fa_bwd_deterministic_stage(**dict(a, workspace_bytes=1 << 30),
                                             stage=stage) == fa.FA_ERR_INVALID_ARG


def test_fp8_forward_workspace_and_validation(lib):
    B, H, Hkv, Nq, Nk, d = 2, 4, 2, 300, 517, 128
    nk16 = (Nk + 15) // 16 * 16
    r256 = lambda x: (x + 255) // 256 * 256
    want = (r256(4 * (B * H + 2 * B * Hkv)) + r256(B * H * Nq * d) + r256(B * Hkv * Nk * d)
            + r256(B * Hkv * d * nk16))
    assert fa.fa_fwd_fp8_workspace_size(B, H, Hkv, Nq, Nk, d) == want
    assert fa.fa_fwd_fp8_workspace_size(0, H, Hkv, Nq, Nk, d) == 0
    a = dict(q=FAKE, k=FAKE, v=FAKE, key_bias=None, o=FAKE, lse=FAKE, B=B, H=H, H_kv=Hkv, Nq=Nq,
             Nk=Nk, d=d, scale=0.1, causal=1, workspace=FAKE, workspace_bytes=want - 1, stream=None)
    assert fa.fa_fwd_fp8(**a) == fa.FA_ERR_INVALID_ARG           # workspace too small
    for bad, expect in ((dict(d=64), fa.FA_ERR_UNSUPPORTED), (dict(H_kv=3), fa.FA_ERR_INVALID_ARG),
                        (dict(lse=None), fa.FA_ERR_INVALID_ARG),
                        (dict(workspace=FAKE + 64), fa.FA_ERR_INVALID_ARG)):
        b = dict(a, workspace_bytes=1 << 30)
        b.update(bad)
        assert fa.fa_fwd_fp8(**b) == expect, bad
    for stage in (-1, 3):
        assert fa.fa_fwd_fp8_stage(**dict(a, workspace_bytes=1 << 30), stage=stage) == \
            fa.FA_ERR_INVALID_ARG
