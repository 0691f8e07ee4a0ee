"""GPU parity of the backward (fa_bwd through the C ABI) against the fp64 oracle.

The forward outputs O and LSE fed to fa_bwd come from fa_fwd on the same
inputs (that is the contract); the oracle recomputes everything from q, k, v.
Small problems are compared in full; the full-size workloads on sampled dQ
rows and on whole sampled heads for dK / dV.
"""
import math

import numpy as np
import pytest
import torch

import exact_io_aware_03_gb300 as fa
import oracle
import workloads
from parity import Guarded, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_io_aware_03_gb300 import build
    build.build()
    fa.load()
    torch.cuda.init()


def run_fwd_bwd(q, k, v, dO, bias, causal, scale, deterministic=False):
    dev = "cuda"
    qd, kd, vd, dOd = (t.to(dev) for t in (q, k, v, dO))
    bd = None if bias is None else bias.to(dev)
    o, lse = fa.fwd(qd, kd, vd, key_bias=bd, causal=causal, scale=scale)
    gq, gk, gv = Guarded(q.shape, q.dtype), Guarded(k.shape, k.dtype), Guarded(v.shape, v.dtype)
    B, H, Nq, d = q.shape
    ws_bytes = (fa.fa_bwd_deterministic_workspace_size(B, H, Nq, d) if deterministic
                else fa.fa_bwd_workspace_size(B, H, Nq, k.shape[2], d))
    ws = Guarded((ws_bytes,), torch.uint8)
    ws.t.fill_(0x7f)   # stale contents must not matter
    fa.bwd(qd, kd, vd, o, lse, dOd, key_bias=bd, causal=causal, scale=scale, workspace=ws.t,
           dq=gq.t, dk=gk.t, dv=gv.t, deterministic=deterministic)
    fa.check_device_error()
    for g, nm in ((gq, "dQ"), (gk, "dK"), (gv, "dV"), (ws, "workspace")):
        g.check(nm)
    return gq.t.cpu(), gk.t.cpu(), gv.t.cpu()


def make(B, H, Nq, Nk, d, seed=0, bias=None):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, H, Nk, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, H, Nk, d, generator=g).to(torch.bfloat16)
    dO = torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16)
    b = None
    if bias == "pad":
        L = torch.randint(1, Nk + 1, (B,), generator=g)
        b = torch.zeros(B, Nk)
        b[torch.arange(Nk)[None, :] >= L[:, None]] = -math.inf
    elif bias == "finite":
        b = torch.randn(B, Nk, generator=g)
        b[:, ::7] = -math.inf
    elif bias == "all_masked_first_batch":
        b = torch.randn(B, Nk, generator=g)
        b[0] = -math.inf
    elif bias == "zero_holes":
        # 0 / -inf, but not a plain padding mask: masked keys inside the
        # valid range, and a masked prefix in the second batch
        b = torch.zeros(B, Nk)
        b[:, 5::9] = -math.inf
        b[:, Nk - Nk // 3:] = -math.inf
        if B > 1:
            b[1, :Nk // 4] = -math.inf
    elif bias == "pad_mixed":
        # even batches keep their first 300 keys, odd ones all: runs of key
        # tiles with nothing to compute next to full ones
        b = torch.zeros(B, Nk)
        b[0::2, 300:] = -math.inf
    return q, k, v, dO, b


SMALL = [
    # B, H, Nq, Nk, d, causal, bias
    (1, 2, 256, 256, 128, True, None),
    (1, 2, 256, 256, 128, False, None),
    (2, 2, 384, 384, 64, False, None),
    (2, 2, 384, 384, 64, True, None),
    (1, 2, 300, 517, 128, True, None),        # ragged tails, Nq < Nk
    (2, 1, 700, 190, 64, True, None),         # Nq > Nk: rows with no visible key
    (2, 2, 129, 1000, 128, False, "pad"),
    (2, 2, 200, 333, 64, True, "finite"),
    (2, 1, 130, 260, 128, False, "all_masked_first_batch"),
    (2, 2, 300, 517, 128, True, "zero_holes"),
    (1, 1, 1, 1, 64, False, None),
    (1, 1, 1, 300, 128, True, None),
    (3, 1, 257, 1, 128, False, None),
    (1, 1, 64, 2048, 128, False, None),       # many key tiles: many dQ reductions per row
    (1, 1, 2048, 64, 128, False, None),       # many query tiles per key tile
    # more key tiles than SMs: several per persistent CTA, with runs of
    # fully masked ones between full ones (the dK/dV write-out hand-over)
    (2, 8, 256, 2048, 128, False, "pad_mixed"),
    (2, 8, 256, 2048, 64, True, "pad_mixed"),
    (1, 12, 384, 2048, 128, True, None),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,bias", SMALL)
def test_bwd_small_full_parity(B, H, Nq, Nk, d, causal, bias):
    q, k, v, dO, b = make(B, H, Nq, Nk, d, seed=7 * B + Nq + 3 * Nk, bias=bias)
    scale = d ** -0.5
    dq, dk, dv = run_fwd_bwd(q, k, v, dO, b, causal, scale)
    dq_r, dk_r, dv_r = oracle.bwd(q, k, v, b, dO, scale=scale, causal=causal)
    tag = "(%d,%d,%d,%d,%d,causal=%s,bias=%s)" % (B, H, Nq, Nk, d, causal, bias)
    compare("dQ", dq, dq_r, extra=tag)
    compare("dK", dk, dk_r, extra=tag)
    compare("dV", dv, dv_r, extra=tag)
    if b is not None:   # masked keys get exactly zero gradient
        dead = torch.isinf(b)
        for bi in range(B):
            assert bool((dk[bi][:, dead[bi]] == 0).all()) and bool((dv[bi][:, dead[bi]] == 0).all())


def test_bwd_dk_dv_deterministic():
    q, k, v, dO, _ = make(1, 2, 512, 512, 128, seed=3)
    r1 = run_fwd_bwd(q, k, v, dO, None, True, 128 ** -0.5)
    r2 = run_fwd_bwd(q, k, v, dO, None, True, 128 ** -0.5)
    assert torch.equal(r1[1], r2[1]) and torch.equal(r1[2], r2[2])
    assert float((r1[0].float() - r2[0].float()).abs().max()) <= 2 ** -7 * float(
        r1[0].float().abs().max())


def test_bwd_large_magnitude():
    """Scores with std ~16 (q, k scaled by 4): very peaked rows.

    The backward forms D_i = rowsum(dO_i o O_i) from the STORED bf16 output, as
    the method prescribes, so D carries the output's rounding error
    |dD_i| <= sum_c |dO_ic| |O_ic| 2^-8. Through dS = P o (dP - D) this adds at
    most scale * |dD_i| * max_j |K_jc| to dQ_ic (and scale * sum_i P_ij |dD_i|
    |Q_ic| to dK_jc). Those per-element bounds, computed from the exact P, are
    added to the max-abs and relative-L2 gates of dQ and dK; dV does not use D
    and keeps the plain gates.
    """
    q, k, v, dO, _ = make(1, 1, 384, 640, 128, seed=9)
    q = (q.float() * 4).to(torch.bfloat16)
    k = (k.float() * 4).to(torch.bfloat16)
    scale = 128 ** -0.5
    Nq, Nk = 384, 640
    dq, dk, dv = run_fwd_bwd(q, k, v, dO, None, True, scale)
    dq_r, dk_r, dv_r = oracle.bwd(q, k, v, None, dO, scale=scale, causal=True)
    o_r, lse_r = oracle.fwd(q, k, v, scale=scale, causal=True)
    # per-row bound on |D error| from the bf16 rounding of O, and its image in
    # dQ (scale dD_i sum_j P_ij |K_j|) and dK (scale sum_i P_ij dD_i |Q_i|)
    qd, kd = q[0, 0].double().numpy(), k[0, 0].double().numpy()
    dD = (np.abs(dO[0, 0].double().numpy()) * np.abs(o_r[0, 0])).sum(-1) * 2.0 ** -8
    s_ = scale * qd @ kd.T
    s_ = np.where(np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + Nk - Nq, s_, -np.inf)
    P = np.exp(s_ - lse_r[0, 0][:, None])
    b_q = scale * dD[:, None] * (P @ np.abs(kd))
    b_k = scale * (P * dD[:, None]).T @ np.abs(qd)
    from parity import BF16_ATOL, BF16_REL_L2, bf16_floor
    for name, got, ref, bnd in (("dQ", dq, dq_r, b_q), ("dK", dk, dk_r, b_k),
                                ("dV", dv, dv_r, np.zeros_like(dv_r[0, 0]))):
        g = got.double().numpy()
        err = np.abs(g - ref)[0, 0]
        assert float((err - bnd).max()) <= BF16_ATOL + bf16_floor(ref), name
        rel = float(np.linalg.norm(g - ref) / np.linalg.norm(ref))
        assert rel <= BF16_REL_L2 + float(np.linalg.norm(bnd) / np.linalg.norm(ref)), (name, rel)


@pytest.mark.parametrize("name,causal", [("bf16_b4h16_n4096_d128_causal_bwd", None),
                                         ("bf16_b8h16_q1024_k16384_d128_keypad", None),
                                         ("bf16_b4h16_n2048_d64", False),
                                         ("bf16_b4h16_n2048_d64", True)])
def test_bwd_full_size_sampled(name, causal):
    w = workloads.WORKLOADS[name]
    if causal is not None:   # the d = 64 workload is run both ways
        w = w.with_(causal=causal)
        name = name + (" causal" if causal else "")
    x = workloads.make_inputs(w, with_dO=True)
    dq, dk, dv = run_fwd_bwd(x["q"], x["k"], x["v"], x["dO"], x["bias"], w.causal, w.scale)
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())
    # dQ: 192 random rows plus the whole first and last query tiles of 2 heads;
    # dK, dV: 8 whole heads (the first, the last and 6 seeded others)
    heads, rows = workloads.sample_rows_dense(w, 192, n_tile_heads=2)
    dq_r = oracle.bwd_dq_rows(x["q"], x["k"], x["v"], x["bias"], x["dO"], heads, rows,
                              scale=w.scale, causal=w.causal)
    H = w.H
    dq_s = torch.stack([dq[h // H, h % H, r] for h, r in zip(heads, rows)])
    tag = name + " bwd"
    compare("dQ[sampled rows]", dq_s, dq_r, extra=tag)
    whole = workloads.sample_heads(w, 8)
    _, dk_r, dv_r = oracle.bwd_heads(x["q"], x["k"], x["v"], x["bias"], x["dO"], whole,
                                     scale=w.scale, causal=w.causal)
    dk_s = torch.stack([dk[h // H, h % H] for h in whole])
    dv_s = torch.stack([dv[h // H, h % H] for h in whole])
    compare("dK[8 heads]", dk_s, dk_r, extra=tag)
    compare("dV[8 heads]", dv_s, dv_r, extra=tag)
    if x["bias"] is not None:
        for h in whole:
            dead = torch.isinf(x["bias"][h // H])
            assert bool((dk[h // H, h % H][dead] == 0).all())
