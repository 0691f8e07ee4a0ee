"""Split-KV (Flash-Decoding) forward against the fp64 oracle.

The split changes only how the key range is partitioned across CTAs and how
the partial softmax states are merged; the function is the oracle's, so every
case is compared with the plain definition, including splits that see no
visible key (their partial LSE is -inf and must drop out of the merge).
"""
import math

import numpy as np
import pytest
import torch

import exact_io_aware_03_gb300 as fa
import oracle
import workloads
from parity import Guarded, compare, compare_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_io_aware_03_gb300 import build
    build.build()
    fa.load()


def make(B, H, Nq, Nk, d, seed, pad=False):
    g = torch.Generator().manual_seed(seed)
    q, k, v = (torch.randn(B, H, n, d, generator=g).to(torch.bfloat16) for n in (Nq, Nk, Nk))
    bias = None
    if pad:
        L = torch.randint(1, Nk + 1, (B,), generator=g)
        bias = torch.zeros(B, Nk)
        bias[torch.arange(Nk)[None, :] >= L[:, None]] = -math.inf
    return q, k, v, bias


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,pad,splits", [
    (2, 4, 1, 5000, 128, False, False, 7),
    (2, 3, 7, 3000, 64, True, False, 4),
    (1, 2, 300, 4100, 128, True, False, 3),
    (3, 2, 4, 9000, 128, False, True, 8),      # padding: trailing splits see no key
    (1, 2, 5, 300, 128, False, False, 5),      # more splits than key tiles
    (2, 2, 1, 1, 64, False, False, 2),
    (1, 1, 2, 1000, 64, False, False, 1),      # one split: plain forward path
])
def test_splitkv_matches_oracle(B, H, Nq, Nk, d, causal, pad, splits):
    q, k, v, bias = make(B, H, Nq, Nk, d, seed=Nq * 31 + Nk, pad=pad)
    dev = "cuda"
    o = Guarded(q.shape, torch.bfloat16)
    lse = Guarded(q.shape[:3], torch.float32)
    ws_bytes = fa.fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, splits)
    ws = Guarded((ws_bytes,), torch.uint8)
    fa.fwd_splitkv(q.to(dev), k.to(dev), v.to(dev), key_bias=None if bias is None else bias.to(dev),
                   causal=causal, num_splits=splits, out=o.t, lse=lse.t, workspace=ws.t)
    fa.check_device_error()
    for g_, n in ((o, "O"), (lse, "LSE"), (ws, "workspace")):
        g_.check(n)
    o_ref, lse_ref = oracle.fwd(q, k, v, bias=bias, scale=d ** -0.5, causal=causal)
    tag = "(%d,%d,%d,%d,%d,causal=%s,pad=%s,splits=%d)" % (B, H, Nq, Nk, d, causal, pad, splits)
    compare("O", o.t.cpu(), o_ref, extra=tag)
    compare_lse(lse.t.cpu(), lse_ref, extra=tag)


def test_splitkv_decode_workload_full_parity():
    w = workloads.WORKLOADS["bf16_b8h32_q1_k32768_d128_decode"]
    x = workloads.make_inputs(w)
    o, lse = fa.fwd_splitkv(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=w.causal)
    fa.check_device_error()
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], scale=w.scale, causal=w.causal)
    compare("O", o.cpu(), o_ref, extra=w.name)
    compare_lse(lse.cpu(), lse_ref, extra=w.name)
    # and the plain forward agrees with the split one within the same tolerance
    o1, lse1 = fa.fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=w.causal)
    compare("O (unsplit)", o1.cpu(), o_ref, extra=w.name)
