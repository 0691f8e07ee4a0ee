"""FP8 forward (fa_fwd_fp8): e4m3 quantization and attention, against the
oracle.

The quantization step must equal the CPU quantization bit for bit (per-head
scale max|x| / 448, round to nearest even). The attention is compared with the
oracle on the dequantized inputs scale_x * e4m3(x / scale_x); the kernel then
rounds P to e4m3 (relative error <= 2^-4 for normal values, absolute <= 2^-10
for subnormal ones, in units of the running maximum), which bounds every output
element by
    |O - O_ref| <= 2^-4 sum_j P_ij |V_jc| + 2^-10 sum_j |V_jc| / l_i + 2^-8 |O_ref| + 1e-3,
(l_i = sum_j exp(s_ij - max_j s_ij) >= 1; the last terms: bf16 output rounding
and fp32 accumulation). The LSE comes from fp32 scores of exact e4m3
products: within 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import exact_io_aware_03_gb300 as fa
import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_io_aware_03_gb300 import build
    build.build()
    fa.load()


def r256(x):
    return (x + 255) // 256 * 256


def make(B, H, Hkv, Nq, Nk, seed, mag=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, Nq, 128, generator=g) * mag).to(torch.bfloat16)
    k = (torch.randn(B, Hkv, Nk, 128, generator=g) * mag).to(torch.bfloat16)
    v = torch.randn(B, Hkv, Nk, 128, generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("B,H,Hkv,Nq,Nk", [(2, 3, 3, 200, 333), (1, 4, 2, 129, 64)])
def test_fp8_quantization_matches_cpu(B, H, Hkv, Nq, Nk):
    q, k, v = make(B, H, Hkv, Nq, Nk, seed=Nq)
    ws = torch.zeros(fa.fa_fwd_fp8_workspace_size(B, H, Hkv, Nq, Nk, 128), dtype=torch.uint8,
                     device="cuda")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    fa.fwd_fp8(qd, kd, vd, workspace=ws, stage=1)
    fa.check_device_error()
    w = ws.cpu()
    nk16 = (Nk + 15) // 16 * 16
    amax = w[:4 * (B * H + 2 * B * Hkv)].view(torch.float32)
    o_q8 = r256(4 * (B * H + 2 * B * Hkv))
    o_k8 = o_q8 + r256(B * H * Nq * 128)
    o_vt = o_k8 + r256(B * Hkv * Nk * 128)
    for x, a in ((q, amax[:B * H]), (k, amax[B * H:B * H + B * Hkv]), (v, amax[B * H + B * Hkv:])):
        assert torch.equal(a, x.float().abs().amax(dim=(-1, -2)).reshape(-1))

    def cpu8(x):
        xf = x.float()
        sc = xf.abs().amax(dim=(-1, -2))
        sc = torch.where(sc > 0, sc / 448.0, torch.ones_like(sc))
        return (xf / sc[..., None, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(w[o_q8:o_q8 + B * H * Nq * 128].view(B, H, Nq, 128), cpu8(q))
    assert torch.equal(w[o_k8:o_k8 + B * Hkv * Nk * 128].view(B, Hkv, Nk, 128), cpu8(k))
    vt = w[o_vt:o_vt + B * Hkv * 128 * nk16].view(B, Hkv, 128, nk16)
    assert torch.equal(vt[..., :Nk], cpu8(v).transpose(-1, -2))
    assert int(vt[..., Nk:].sum()) == 0


def dequantized(x):
    x8, sc = oracle.quantize_e4m3(x)
    return x8.double() * sc.double()[..., None, None]


def bound_check(qd, kd, vd, o, lse, bias, causal, tag):
    """qd, kd, vd: the dequantized inputs (float64 tensors)."""
    scale = 128 ** -0.5
    if kd.shape[1] != qd.shape[1]:
        o_ref, lse_ref = oracle.fwd_gqa(qd, kd, vd, bias, scale=scale, causal=causal)
    else:
        o_ref, lse_ref = oracle.fwd(qd, kd, vd, bias, scale=scale, causal=causal)
    qd, kd, vd = qd.numpy(), kd.numpy(), vd.numpy()
    B, H, Nq, _ = qd.shape
    Hkv, Nk = kd.shape[1], kd.shape[2]
    g = H // Hkv
    got = o.double().cpu().numpy()
    worst = 0.0
    errs, bnds = [], []
    for b in range(B):
        for h in range(H):
            s = scale * qd[b, h] @ kd[b, h // g].T
            if bias is not None:
                s = s + bias[b].double().numpy()[None, :]
            if causal:
                s = np.where(np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + Nk - Nq, s, -np.inf)
            mx = s.max(axis=1, keepdims=True)
            ok = np.isfinite(mx[:, 0])
            e = np.where(ok[:, None], np.exp(s - np.where(ok[:, None], mx, 0)), 0.0)
            l = e.sum(axis=1, keepdims=True)
            P = np.where(ok[:, None], e / np.where(l > 0, l, 1), 0.0)
            av = np.abs(vd[b, h // g])
            bnd = 2.0 ** -4 * (P @ av) + 2.0 ** -10 * av.sum(axis=0)[None, :] / np.where(l > 0, l, 1) \
                + 2.0 ** -8 * np.abs(o_ref[b, h]) + 1e-3
            err = np.abs(got[b, h] - o_ref[b, h])
            worst = max(worst, float((err / bnd).max()))
            errs.append(err.mean())
            bnds.append(bnd.mean())
    assert worst <= 1.0, "%s: error / bound reaches %.3f" % (tag, worst)
    fin = np.isfinite(lse_ref)
    lg = lse.double().cpu().numpy()
    assert np.array_equal(np.isfinite(lg), fin), tag
    assert float(np.abs(lg[fin] - lse_ref[fin]).max()) <= 1e-3, tag
    return float(np.mean(errs)), float(np.mean(bnds))


@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,causal,pad", [
    (2, 2, 2, 300, 517, True, False),
    (1, 3, 3, 256, 256, False, False),
    (2, 2, 2, 129, 1000, False, True),
    (1, 4, 1, 200, 333, True, False),     # multi-query
    (1, 1, 1, 700, 190, True, False),     # rows with no visible key
])
def test_fp8_forward_within_derived_bound(B, H, Hkv, Nq, Nk, causal, pad):
    q, k, v = make(B, H, Hkv, Nq, Nk, seed=Nq + Nk)
    bias = None
    if pad:
        g = torch.Generator().manual_seed(11)
        L = torch.randint(Nk // 2, Nk + 1, (B,), generator=g)
        bias = torch.zeros(B, Nk)
        bias[torch.arange(Nk)[None, :] >= L[:, None]] = -math.inf
    o, lse = fa.fwd_fp8(q.cuda(), k.cuda(), v.cuda(), key_bias=None if bias is None else bias.cuda(),
                        causal=causal)
    fa.check_device_error()
    tag = "(%d,%d,%d,%d,%d,causal=%s,pad=%s)" % (B, H, Hkv, Nq, Nk, causal, pad)
    e, b = bound_check(dequantized(q), dequantized(k), dequantized(v), o.cpu(), lse.cpu(), bias,
                       causal, tag)
    assert e <= 0.5 * b, (tag, e, b)


def test_fp8_forward_large_magnitude_scores():
    # q, k scaled by 4: very peaked rows, P dominated by one key per row
    q, k, v = make(1, 2, 2, 256, 384, seed=9, mag=4.0)
    o, lse = fa.fwd_fp8(q.cuda(), k.cuda(), v.cuda(), causal=True)
    fa.check_device_error()
    bound_check(dequantized(q), dequantized(k), dequantized(v), o.cpu(), lse.cpu(), None, True,
                "large magnitude")


def test_fp8_long_context_sampled_rows():
    w = workloads.WORKLOADS["bf16_b2h32_n8192_d128_causal"]
    x = workloads.make_inputs(w, with_dO=False)
    o, lse = fa.fwd_fp8(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=True)
    fa.check_device_error()
    assert bool(torch.isfinite(o.float()).all())
    # rows of two heads, checked against the full oracle on those heads
    heads = [0, w.B * w.H - 1]
    qh = torch.stack([x["q"][h // w.H, h % w.H] for h in heads])[None]
    kh = torch.stack([x["k"][h // w.H, h % w.H] for h in heads])[None]
    vh = torch.stack([x["v"][h // w.H, h % w.H] for h in heads])[None]
    oh = torch.stack([o[h // w.H, h % w.H].cpu() for h in heads])[None]
    lh = torch.stack([lse[h // w.H, h % w.H].cpu() for h in heads])[None]
    # dequantized with the whole heads' scales; then the first 1024 rows,
    # which under the causal mask see only the first 1024 keys
    qd, kd, vd = dequantized(qh), dequantized(kh), dequantized(vh)
    sel = slice(0, 1024)
    bound_check(qd[:, :, sel], kd[:, :, sel], vd[:, :, sel], oh[:, :, sel], lh[:, :, sel], None,
                True, "long-context rows")
