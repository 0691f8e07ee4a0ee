"""Grouped-query / multi-query attention (fa_fwd_gqa, fa_bwd_gqa) against the
fp64 oracle with head mapping."""
import math

import pytest
import torch

import exact_io_aware_03_gb300 as fa
import oracle
from parity import Guarded, compare, compare_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_io_aware_03_gb300 import build
    build.build()
    fa.load()


@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,d,causal,pad", [
    (2, 8, 2, 300, 400, 128, True, False),
    (1, 6, 1, 257, 257, 64, False, False),     # multi-query
    (2, 4, 4, 130, 520, 128, True, False),     # H_kv == H through the grouped entry
    (2, 8, 4, 200, 1000, 128, False, True),
    # more query-tile pairs x heads than the 152 SMs: the persistent forward,
    # with key/value heads shared by 8 and 10 query heads
    (2, 80, 10, 512, 512, 64, False, False),
    (1, 96, 12, 512, 700, 128, True, False),
])
def test_gqa_forward_and_backward(B, H, Hkv, Nq, Nk, d, causal, pad):
    g = torch.Generator().manual_seed(H * 100 + Hkv)
    q = torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, Nk, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, Nk, d, generator=g).to(torch.bfloat16)
    dO = torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16)
    bias = None
    if pad:
        L = torch.randint(1, Nk + 1, (B,), generator=g)
        bias = torch.zeros(B, Nk)
        bias[torch.arange(Nk)[None, :] >= L[:, None]] = -math.inf
    scale = d ** -0.5
    qd, kd, vd, dOd = (t.cuda() for t in (q, k, v, dO))
    bd = None if bias is None else bias.cuda()
    o, lse = fa.fwd(qd, kd, vd, key_bias=bd, causal=causal, scale=scale)
    gk, gv = Guarded(k.shape, torch.bfloat16), Guarded(v.shape, torch.bfloat16)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dOd, key_bias=bd, causal=causal, scale=scale,
                        dk=gk.t, dv=gv.t)
    fa.check_device_error()
    gk.check("dK")
    gv.check("dV")
    o_ref, lse_ref = oracle.fwd_gqa(q, k, v, bias=bias, scale=scale, causal=causal)
    dq_ref, dk_ref, dv_ref = oracle.bwd_gqa(q, k, v, bias, dO, scale=scale, causal=causal)
    tag = "(%d,%d,%d,%d,%d,%d,causal=%s)" % (B, H, Hkv, Nq, Nk, d, causal)
    compare("O", o.cpu(), o_ref, extra=tag)
    compare_lse(lse.cpu(), lse_ref, extra=tag)
    compare("dQ", dq.cpu(), dq_ref, extra=tag)
    compare("dK", dk.cpu(), dk_ref, extra=tag)
    compare("dV", dv.cpu(), dv_ref, extra=tag)


def test_gqa_splitkv_decode():
    B, H, Hkv, Nq, Nk, d = 2, 16, 2, 1, 9000, 128
    g = torch.Generator().manual_seed(5)
    q = torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, Nk, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, Nk, d, generator=g).to(torch.bfloat16)
    o, lse = fa.fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), num_splits=6)
    fa.check_device_error()
    o_ref, lse_ref = oracle.fwd_gqa(q, k, v, scale=d ** -0.5)
    compare("O", o.cpu(), o_ref)
    compare_lse(lse.cpu(), lse_ref)


def test_gqa_fp32_forward():
    B, H, Hkv, Nq, Nk, d = 1, 4, 2, 70, 90, 64
    g = torch.Generator().manual_seed(6)
    q = torch.randn(B, H, Nq, d, generator=g)
    k = torch.randn(B, Hkv, Nk, d, generator=g)
    v = torch.randn(B, Hkv, Nk, d, generator=g)
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    fa.check_device_error()
    o_ref, _ = oracle.fwd_gqa(q, k, v, scale=d ** -0.5, causal=True)
    compare("O", o.cpu(), o_ref, dtype="fp32")
