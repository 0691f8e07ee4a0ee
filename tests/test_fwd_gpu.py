"""GPU parity of the forward (fa_fwd through the C ABI) against the fp64 oracle.

Small problems are compared element by element in full; they span several
128-row / 128-key tiles and ragged tails. The full-size workloads are
compared on sampled rows the oracle computes one by one, plus properties that
hold at any size (finite outputs, no writes outside the outputs).
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
    torch.cuda.init()


def run_fwd(q, k, v, bias, causal, scale):
    """Inputs on the CPU; returns (O, LSE) on the CPU, checking guard bands."""
    dev = "cuda"
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    bd = None if bias is None else bias.to(dev)
    o = Guarded(q.shape, q.dtype)
    lse = Guarded(q.shape[:3], torch.float32)
    fa.fwd(qd, kd, vd, key_bias=bd, causal=causal, scale=scale, out=o.t, lse=lse.t)
    fa.check_device_error()
    o.check("O")
    lse.check("LSE")
    return o.t.cpu(), lse.t.cpu()


def make(B, H, Nq, Nk, d, dtype=torch.bfloat16, seed=0, bias=None):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Nq, d, generator=g).to(dtype)
    k = torch.randn(B, H, Nk, d, generator=g).to(dtype)
    v = torch.randn(B, H, Nk, d, generator=g).to(dtype)
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
    return q, k, v, b


SMALL = [
    # B, H, Nq, Nk, d, causal, bias
    (1, 2, 256, 256, 128, False, None),
    (1, 2, 256, 256, 128, True, None),
    (2, 3, 384, 384, 64, True, None),
    (1, 2, 300, 517, 64, False, None),        # ragged query and key tails
    (2, 1, 300, 517, 128, True, None),        # Nq < Nk, bottom-right causal
    (1, 2, 700, 190, 128, True, None),        # Nq > Nk: leading rows see no key
    (2, 2, 129, 1000, 128, False, "pad"),     # key padding
    (2, 2, 200, 333, 64, True, "finite"),     # finite bias + causal
    (2, 1, 130, 260, 128, False, "all_masked_first_batch"),
    (2, 2, 200, 700, 128, False, "zero_holes"),
    (2, 2, 300, 517, 64, True, "zero_holes"),
    (1, 1, 1, 1, 64, False, None),            # degenerate sizes
    (1, 1, 1, 300, 128, True, None),
    (3, 1, 257, 1, 128, False, None),
    (1, 1, 64, 4096, 128, False, None),       # many key tiles: ring wrap-around
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,bias", SMALL)
def test_fwd_bf16_small_full_parity(B, H, Nq, Nk, d, causal, bias):
    q, k, v, b = make(B, H, Nq, Nk, d, seed=B * 1000 + Nq + Nk, bias=bias)
    scale = d ** -0.5
    o, lse = run_fwd(q, k, v, b, causal, scale)
    o_ref, lse_ref = oracle.fwd(q, k, v, bias=b, scale=scale, causal=causal)
    tag = "(%d,%d,%d,%d,%d,causal=%s,bias=%s)" % (B, H, Nq, Nk, d, causal, bias)
    compare("O", o, o_ref, extra=tag)
    compare_lse(lse, lse_ref, extra=tag)
    dead = np.isneginf(lse_ref)
    if dead.any():   # rows with no visible key are exactly zero
        assert bool((o.double().numpy()[dead] == 0).all())


def test_fwd_bf16_large_magnitude_rescaling():
    # scores of magnitude ~100s force the running max to move many times
    q, k, v, _ = make(1, 2, 256, 1024, 128, seed=5)
    q = (q.float() * 6).to(torch.bfloat16)
    k = (k.float() * 5).to(torch.bfloat16)
    for causal in (False, True):
        o, lse = run_fwd(q, k, v, None, causal, 128 ** -0.5)
        o_ref, lse_ref = oracle.fwd(q, k, v, scale=128 ** -0.5, causal=causal)
        compare("O", o, o_ref)
        compare_lse(lse, lse_ref)


def test_fwd_bf16_increasing_scores_force_every_rescale():
    # key j's score grows with j, so each new key tile raises the max by > 8 (log2)
    Nk, d = 1024, 64
    q = torch.zeros(1, 1, 128, d)
    q[..., 0] = 1.0
    k = torch.zeros(1, 1, Nk, d)
    k[0, 0, :, 0] = torch.arange(Nk, dtype=torch.float32) * 0.125
    v = torch.randn(1, 1, Nk, d, generator=torch.Generator().manual_seed(3))
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    o, lse = run_fwd(q, k, v, None, False, 1.0)
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=1.0)
    compare("O", o, o_ref)
    compare_lse(lse, lse_ref)


# More units (query-tile pairs x heads) than the GB300's 152 SMs and no
# bias: the persistent form, where each CTA claims further units from a
# counter kept in the LSE word of the last head's first row. Includes a last
# pair with one inactive query tile (Nq = 384, 640), Nq < Nk and Nq > Nk with
# ragged key tails, d = 64 and d = 128, causal and not.
PERSISTENT = [
    # B, H, Nq, Nk, d, causal
    (1, 80, 512, 512, 64, False),
    (1, 77, 384, 384, 128, False),
    (2, 40, 640, 1000, 128, False),
    (3, 30, 512, 300, 64, False),
    (1, 80, 512, 512, 64, True),
    (2, 40, 640, 1000, 128, True),
    # one query row per head (the pair's second tile inactive), 200 heads
    (1, 200, 1, 300, 64, False),
    (2, 100, 1, 257, 128, True),
    # a single ragged row past the last full tile pair
    (1, 160, 257, 129, 128, False),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", PERSISTENT)
def test_fwd_bf16_persistent_full_parity(B, H, Nq, Nk, d, causal):
    q, k, v, _ = make(B, H, Nq, Nk, d, seed=7 * H + Nq)
    scale = d ** -0.5
    o, lse = run_fwd(q, k, v, None, causal, scale)
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=scale, causal=causal)
    tag = "(%d,%d,%d,%d,%d,causal=%s)" % (B, H, Nq, Nk, d, causal)
    compare("O", o, o_ref, extra=tag)
    compare_lse(lse, lse_ref, extra=tag)


def test_fwd_bf16_persistent_counter_row_lse_zero():
    # The counter's word is the LSE of row 0 of the last head. Make that LSE
    # exactly 0 (one key, and q . k = 0 on that row): it is stored as -0.
    B, H, Nq, Nk, d = 1, 160, 256, 1, 64
    q, k, v, _ = make(B, H, Nq, Nk, d, seed=3)
    q[0, H - 1, 0] = 0
    o, lse = run_fwd(q, k, v, None, False, d ** -0.5)
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=d ** -0.5, causal=False)
    assert float(lse[0, H - 1, 0]) == 0.0 and lse_ref[0, H - 1, 0] == 0.0
    compare("O", o, o_ref)
    compare_lse(lse, lse_ref)


def test_fwd_bf16_persistent_counter_row_dead():
    # causal with Nq > Nk: the last head's first query tile sees no key, so
    # the counter's word ends as LSE = -inf (and that tile's O as 0)
    q, k, v, _ = make(2, 80, 384, 200, 64, seed=4)
    o, lse = run_fwd(q, k, v, None, True, 64 ** -0.5)
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=64 ** -0.5, causal=True)
    assert np.isneginf(lse_ref[1, 79, 0]) and np.isneginf(float(lse[1, 79, 0]))
    assert bool((o[1, 79, :128].float() == 0).all())
    compare("O", o, o_ref)
    compare_lse(lse, lse_ref)


def test_fwd_bf16_persistent_repeat_and_concurrent_streams():
    # the unit counter is reset on each launch's own stream and lives in that
    # launch's LSE: repeated launches and launches on two streams at once give
    # the same bits
    B, H, N, d = 2, 96, 512, 128
    q, k, v, _ = make(B, H, N, N, d, seed=11)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = fa.fwd(qd, kd, vd)
    torch.cuda.synchronize()
    fa.check_device_error()
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=d ** -0.5)
    compare("O", o1.cpu(), o_ref)
    compare_lse(l1.cpu(), lse_ref)
    s_a, s_b = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(s_a):
            oa, la = fa.fwd(qd, kd, vd)
        with torch.cuda.stream(s_b):
            ob, lb = fa.fwd(qd, kd, vd)
        outs += [(oa, la), (ob, lb)]
    torch.cuda.synchronize()
    fa.check_device_error()
    for o, l in outs:
        assert torch.equal(o, o1)
        assert torch.equal(l, l1)


def test_fwd_bf16_persistent_cuda_graph_replay():
    # the counter reset (a memset on the stream) is captured with the kernel:
    # every replay claims all units again
    B, H, N, d = 2, 96, 512, 64
    q, k, v, _ = make(B, H, N, N, d, seed=13)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(qd)
    lse = torch.empty(B, H, N, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fa.fwd(qd, kd, vd, out=o, lse=lse)   # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fa.fwd(qd, kd, vd, out=o, lse=lse)
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=d ** -0.5)
    for _ in range(3):
        o.zero_()
        lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        fa.check_device_error()
        compare("O", o.cpu(), o_ref)
        compare_lse(lse.cpu(), lse_ref)


def test_fwd_f32_workload_full_parity():
    w = workloads.WORKLOADS["f32_b1h1_n128_d64"]
    x = workloads.make_inputs(w)
    o, lse = run_fwd(x["q"], x["k"], x["v"], None, w.causal, w.scale)
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], scale=w.scale)
    compare("O", o, o_ref, dtype="fp32", extra=w.name + " fwd")
    assert float(np.abs(lse.double().numpy() - lse_ref).max()) <= 1e-5


@pytest.mark.parametrize("Nq,Nk,d,causal,bias", [
    (200, 333, 128, True, "finite"), (65, 70, 64, False, "pad"), (300, 130, 64, True, None)])
def test_fwd_f32_small_full_parity(Nq, Nk, d, causal, bias):
    q, k, v, b = make(2, 2, Nq, Nk, d, dtype=torch.float32, seed=11, bias=bias)
    o, lse = run_fwd(q, k, v, b, causal, d ** -0.5)
    o_ref, lse_ref = oracle.fwd(q, k, v, bias=b, scale=d ** -0.5, causal=causal)
    compare("O", o, o_ref, dtype="fp32")
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(lse.numpy()), ~fin)
    assert float(np.abs(lse.double().numpy()[fin] - lse_ref[fin]).max()) <= 1e-5


FULL = [("bf16_b4h16_n2048_d64", False), ("bf16_b4h16_n2048_d64", True),
        ("bf16_b2h32_n8192_d128_causal", True),
        ("bf16_b4h16_n4096_d128_causal_bwd", True),
        ("bf16_b8h16_q1024_k16384_d128_keypad", False)]


@pytest.mark.parametrize("name,causal", FULL)
def test_fwd_full_size_sampled_rows(name, causal):
    w = workloads.WORKLOADS[name]
    x = workloads.make_inputs(w, with_dO=False)
    o, lse = run_fwd(x["q"], x["k"], x["v"], x["bias"], causal, w.scale)
    # 512 random rows plus the whole first and last query tiles of 4 heads
    heads, rows = workloads.sample_rows_dense(w, 512, n_tile_heads=4)
    o_ref, lse_ref = oracle.fwd_rows(x["q"], x["k"], x["v"], x["bias"], heads, rows,
                                     scale=w.scale, causal=causal)
    H = w.H
    o_s = torch.stack([o[h // H, h % H, r] for h, r in zip(heads, rows)])
    l_s = torch.stack([lse[h // H, h % H, r] for h, r in zip(heads, rows)])
    tag = name + (" causal" if causal else "") + " fwd"
    compare("O[sampled]", o_s, o_ref, extra=tag)
    compare_lse(l_s, lse_ref, extra=tag)
    assert bool(torch.isfinite(o.float()).all())
