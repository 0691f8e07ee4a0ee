"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (a runtime that plans all device memory ahead and hands kernels
only their buffers, code inside an allocator callback, a service that may not
call cudaMalloc on its request path) get the backward's workspace from a fixed
array inside the library instead of from their own allocation. These tests
call that entry point through the C ABI and check it against fa_bwd, which
takes a caller-allocated workspace, and against the fp64 oracle, on two calls
in a row (the array is shared and keeps the previous call's contents, which
must not leak into the result). The file is named to be collected last.
"""
import math

import numpy as np
import pytest
import torch

import exact_io_aware_03_gb300 as fa
import oracle
from parity import compare


@pytest.fixture(scope="module")
def lib():
    from exact_io_aware_03_gb300 import build
    build.build()
    return fa.load()


def _inputs(B, H, Nq, Nk, d, seed, pad):
    g = torch.Generator().manual_seed(seed)
    q, k, v, dO = (torch.randn(B, H, n, d, generator=g).to(torch.bfloat16)
                   for n in (Nq, Nk, Nk, Nq))
    bias = None
    if pad:
        L = torch.randint(Nk // 2, Nk + 1, (B,), generator=g)
        bias = torch.zeros(B, Nk)
        bias[torch.arange(Nk)[None, :] >= L[:, None]] = -math.inf
    return q, k, v, dO, bias


def _noalloc(q, k, v, o, lse, dO, bias, causal, scale):
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = fa.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), dO.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                           dv.data_ptr(), None if bias is None else bias.data_ptr(),
                           B, H, Nq, Nk, d, scale, int(causal), fa.FA_DTYPE_BF16,
                           torch.cuda.current_stream().cuda_stream)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return dq, dk, dv


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,pad", [
    (2, 4, 1000, 1500, 128, True, False),
    (2, 3, 700, 900, 64, False, True),
])
def test_noalloc_matches_fa_bwd_on_two_calls(lib, B, H, Nq, Nk, d, causal, pad):
    assert fa.fa_bwd_workspace_size(B, H, Nq, Nk, d) <= fa.FA_NOALLOC_SCRATCH_BYTES
    q, k, v, dO, bias = (None if t is None else t.cuda()
                         for t in _inputs(B, H, Nq, Nk, d, seed=Nq + d, pad=pad))
    scale = d ** -0.5
    o, lse = fa.fwd(q, k, v, key_bias=bias, causal=causal, scale=scale)
    ref = fa.bwd(q, k, v, o, lse, dO, key_bias=bias, causal=causal, scale=scale)
    fa.check_device_error()
    ref64 = [t.double().cpu().numpy() for t in ref]
    for call in range(2):
        got = _noalloc(q, k, v, o, lse, dO, bias, causal, scale)
        fa.check_device_error()
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref64):
            compare(name, g, r, extra="no-alloc call %d" % call)
        # dK and dV involve no cross-CTA accumulation: identical to fa_bwd's
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])


@pytest.mark.gpu
def test_noalloc_matches_the_oracle(lib):
    """The same entry point checked against the fp64 oracle directly (not only
    against fa_bwd), on a small causal key-padding case, twice in a row."""
    B, H, Nq, Nk, d, causal = 1, 2, 300, 300, 64, True
    q, k, v, dO, bias = _inputs(B, H, Nq, Nk, d, seed=4242, pad=True)
    scale = d ** -0.5
    qd, kd, vd, dOd, bd = (t.cuda() for t in (q, k, v, dO, bias))
    o, lse = fa.fwd(qd, kd, vd, key_bias=bd, causal=causal, scale=scale)
    ref = oracle.bwd(q, k, v, bias, dO, scale=scale, causal=causal)
    for call in range(2):
        got = _noalloc(qd, kd, vd, o, lse, dOd, bd, causal, scale)
        fa.check_device_error()
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            compare(name, g, r, extra="no-alloc vs oracle, call %d" % call)


def test_noalloc_rejects_problems_larger_than_its_array(lib):
    # 16 heads x 8192 rows x d=128 needs 16 * 8192 * (8 + 512) bytes > 32 MiB;
    # rejected on the host before any device work (no GPU needed).
    B, H, Nq, Nk, d = 1, 16, 8192, 8192, 128
    assert fa.fa_bwd_workspace_size(B, H, Nq, Nk, d) > fa.FA_NOALLOC_SCRATCH_BYTES
    fake = 1 << 20
    st = fa.fa_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, None,
                           B, H, Nq, Nk, d, 0.088, 1, fa.FA_DTYPE_BF16, None)
    assert st == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, None,
                             0, H, Nq, Nk, d, 0.088, 1, fa.FA_DTYPE_BF16, None) \
        == fa.FA_ERR_INVALID_ARG
