"""GPU parity of the deterministic backward (fa_bwd_deterministic and its
varlen form, through the C ABI) against the fp64 oracle, and its bitwise
reproducibility.

The deterministic backward forms dQ in a query-outer kernel that adds the key
tiles in a fixed order, instead of reducing every key tile's share into a
shared accumulator ("flash-attention", Part VII: the deterministic option).
Same cases as the plain backward's parity tests, plus: two runs give
bit-identical dQ, dK, dV; its three stages run one by one equal the whole
call; grouped heads and packed ragged batches.
"""
import numpy as np
import pytest
import torch

import exact_io_aware_03_gb300 as fa
import oracle
import workloads
from parity import compare
from test_bwd_gpu import SMALL, make, run_fwd_bwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_io_aware_03_gb300 import build
    build.build()
    fa.load()
    torch.cuda.init()


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,bias", SMALL)
def test_det_bwd_small_full_parity(B, H, Nq, Nk, d, causal, bias):
    q, k, v, dO, b = make(B, H, Nq, Nk, d, seed=7 * B + Nq + 3 * Nk, bias=bias)
    scale = d ** -0.5
    dq, dk, dv = run_fwd_bwd(q, k, v, dO, b, causal, scale, deterministic=True)
    dq_r, dk_r, dv_r = oracle.bwd(q, k, v, b, dO, scale=scale, causal=causal)
    tag = "(%d,%d,%d,%d,%d,causal=%s,bias=%s) deterministic" % (B, H, Nq, Nk, d, causal, bias)
    compare("dQ", dq, dq_r, extra=tag)
    compare("dK", dk, dk_r, extra=tag)
    compare("dV", dv, dv_r, extra=tag)
    if b is not None:
        dead = torch.isinf(b)
        for bi in range(B):
            assert bool((dk[bi][:, dead[bi]] == 0).all()) and bool((dv[bi][:, dead[bi]] == 0).all())


@pytest.mark.parametrize("causal", [True, False])
def test_det_bwd_is_bitwise_reproducible(causal):
    q, k, v, dO, _ = make(2, 3, 1000, 1300, 128, seed=11)
    r1 = run_fwd_bwd(q, k, v, dO, None, causal, 128 ** -0.5, deterministic=True)
    r2 = run_fwd_bwd(q, k, v, dO, None, causal, 128 ** -0.5, deterministic=True)
    for a, b, n in zip(r1, r2, ("dQ", "dK", "dV")):
        assert torch.equal(a, b), n
    # dK and dV come from the same products as in the plain backward
    r0 = run_fwd_bwd(q, k, v, dO, None, causal, 128 ** -0.5)
    assert torch.equal(r0[2], r1[2])


def test_det_stages_equal_the_whole_call():
    q, k, v, dO, b = make(2, 2, 333, 700, 64, seed=5, bias="pad")
    dev = "cuda"
    qd, kd, vd, dOd, bd = (t.to(dev) for t in (q, k, v, dO, b))
    o, lse = fa.fwd(qd, kd, vd, key_bias=bd, causal=True)
    whole = fa.bwd(qd, kd, vd, o, lse, dOd, key_bias=bd, causal=True, deterministic=True)
    ws = torch.empty(fa.fa_bwd_deterministic_workspace_size(2, 2, 333, 64), dtype=torch.uint8,
                     device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    for stage in ("preprocess", "dkdv", "dq"):
        fa.bwd(qd, kd, vd, o, lse, dOd, key_bias=bd, causal=True, deterministic=True, stage=stage,
               workspace=ws, dq=dq, dk=dk, dv=dv)
    fa.check_device_error()
    for a, b_, n in zip(whole, (dq, dk, dv), ("dQ", "dK", "dV")):
        assert torch.equal(a, b_), n


@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,d,causal", [
    (2, 8, 2, 300, 450, 128, True),
    (1, 6, 1, 257, 129, 64, False),
])
def test_det_bwd_grouped_heads(B, H, Hkv, Nq, Nk, d, causal):
    g = torch.Generator().manual_seed(H * 31 + Nq)
    q, dO = (torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16) for _ in range(2))
    k, v = (torch.randn(B, Hkv, Nk, d, generator=g).to(torch.bfloat16) for _ in range(2))
    dev = "cuda"
    qd, kd, vd, dOd = (t.to(dev) for t in (q, k, v, dO))
    o, lse = fa.fwd(qd, kd, vd, causal=causal)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dOd, causal=causal, deterministic=True)
    fa.check_device_error()
    dq_r, dk_r, dv_r = oracle.bwd_gqa(q, k, v, None, dO, scale=d ** -0.5, causal=causal)
    tag = "GQA H=%d H_kv=%d deterministic" % (H, Hkv)
    compare("dQ", dq.cpu(), dq_r, extra=tag)
    compare("dK", dk.cpu(), dk_r, extra=tag)
    compare("dV", dv.cpu(), dv_r, extra=tag)


@pytest.mark.parametrize("lens_q,lens_k,H,Hkv,causal", [
    ([300, 0, 129, 1000], [300, 5, 0, 700], 2, 2, True),
    ([64, 513, 200], [640, 513, 17], 4, 2, False),
])
def test_det_bwd_varlen(lens_q, lens_k, H, Hkv, causal):
    d = 128
    g = torch.Generator().manual_seed(sum(lens_q) + H)
    tq, tk = sum(lens_q), sum(lens_k)
    q, dO = (torch.randn(H, tq, d, generator=g).to(torch.bfloat16) for _ in range(2))
    k, v = (torch.randn(Hkv, tk, d, generator=g).to(torch.bfloat16) for _ in range(2))
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32)
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32)
    dev = "cuda"
    qd, kd, vd, dOd, cqd, ckd = (t.to(dev) for t in (q, k, v, dO, cu_q, cu_k))
    o, lse = fa.fwd_varlen(qd, kd, vd, cqd, ckd, causal=causal)
    dq, dk, dv = fa.bwd_varlen(qd, kd, vd, o, lse, dOd, cqd, ckd, causal=causal,
                               deterministic=True)
    dq2, dk2, dv2 = fa.bwd_varlen(qd, kd, vd, o, lse, dOd, cqd, ckd, causal=causal,
                                  deterministic=True)
    fa.check_device_error()
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)
    dq_r, dk_r, dv_r = oracle.bwd_varlen(q, k, v, dO, cu_q.numpy(), cu_k.numpy(),
                                         scale=d ** -0.5, causal=causal)
    tag = "varlen %s/%s deterministic" % (lens_q, lens_k)
    compare("dQ", dq.cpu(), dq_r, extra=tag)
    compare("dK", dk.cpu(), dk_r, extra=tag)
    compare("dV", dv.cpu(), dv_r, extra=tag)


@pytest.mark.parametrize("name", ["bf16_b4h16_n4096_d128_causal_bwd",
                                  "bf16_b8h16_q1024_k16384_d128_keypad"])
def test_det_bwd_full_size_sampled(name):
    w = workloads.WORKLOADS[name]
    x = workloads.make_inputs(w, with_dO=True)
    dq, dk, dv = run_fwd_bwd(x["q"], x["k"], x["v"], x["dO"], x["bias"], w.causal, w.scale,
                             deterministic=True)
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())
    heads, rows = workloads.sample_rows(w, 48)
    dq_r = oracle.bwd_dq_rows(x["q"], x["k"], x["v"], x["bias"], x["dO"], heads, rows,
                              scale=w.scale, causal=w.causal)
    H = w.H
    dq_s = torch.stack([dq[h // H, h % H, r] for h, r in zip(heads, rows)])
    compare("dQ[sampled rows]", dq_s, dq_r, extra=name + " deterministic")
    whole = [0, w.B * w.H - 1]
    _, dk_r, dv_r = oracle.bwd_heads(x["q"], x["k"], x["v"], x["bias"], x["dO"], whole,
                                     scale=w.scale, causal=w.causal)
    dk_s = torch.stack([dk[h // H, h % H] for h in whole])
    dv_s = torch.stack([dv[h // H, h % H] for h in whole])
    compare("dK[sampled heads]", dk_s, dk_r, extra=name + " deterministic")
    compare("dV[sampled heads]", dv_s, dv_r, extra=name + " deterministic")
