"""Pins for the fp64 oracle: values the pages print, closed forms, invariants,
an independent streaming implementation, a library witness, and finite
differences for the backward. None of these call the CUDA path.

Each check is chosen so that a plausible slip in the oracle (a dropped scale,
a missing max-subtraction, a wrong causal offset, a transposed operand, a sign
error in the softmax Jacobian) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden


def one_row_problem(scores, values):
    """Single query whose scaled scores against the keys are exactly `scores`
    (scale = 1, q = e_0, k_j = scores[j] * e_0), with value rows `values`."""
    values = np.atleast_2d(np.asarray(values, dtype=np.float64))
    if values.shape[0] == 1 and len(scores) > 1:
        values = values.T
    n, dv = values.shape
    D = max(dv, 1)
    q = np.zeros((1, 1, 1, D))
    q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, 1, n, D))
    k[0, 0, :, 0] = scores
    v = np.zeros((1, 1, n, D))
    v[0, 0, :, :dv] = values
    return q, k, v, dv


def row(scores, values, bias=None):
    q, k, v, dv = one_row_problem(scores, values)
    o, lse = oracle.fwd(q, k, v, bias=bias, scale=1.0)
    return o[0, 0, 0, :dv], lse[0, 0, 0]


def weights_of(scores):
    """Softmax weights read out through one-hot values (V = identity)."""
    n = len(scores)
    o, lse = row(scores, np.eye(n))
    return o, lse


# ---------------------------------------------------------------- pages' numbers

def test_worked_example_two_blocks_2d():
    g = read_golden("worked_example_two_blocks_2d.txt")
    o, lse = row(g["scores"], g["values"])
    m = max(g["scores"])
    l = math.exp(lse - m)
    assert abs(l - g["l"]) <= g["tol"]
    np.testing.assert_allclose(o, g["O"], rtol=0, atol=g["tol"])
    # unnormalised stable weights e^(s - m), read out through one-hot values
    w, lse_w = weights_of(g["scores"])
    np.testing.assert_allclose(w * math.exp(lse_w - m), g["weights_unnormalised"],
                               rtol=0, atol=g["weights_tol"])
    # state after block 1 alone: l1 = sum over block 1 relative to its own max
    o1, lse1 = row(g["block1"], np.asarray(g["values"])[:2])
    assert abs(math.exp(lse1 - max(g["block1"])) - g["l1"]) <= g["tol"]
    # accumulator after block 2 equals O * l (o = a / l at the end)
    np.testing.assert_allclose(o * l, g["a2"], rtol=0, atol=g["tol"] * 4)


def test_worked_example_eight_scores():
    g = read_golden("worked_example_eight_scores.txt")
    o, lse = row(g["scores"], g["values"])
    m = max(g["scores"])
    l = math.exp(lse - m)
    assert abs(l - g["l"]) <= g["tol4"]
    assert abs(o[0] - g["O"]) <= g["tol3"]
    assert abs(o[0] * l - g["O_unnormalised"]) <= g["tol3"]
    w, _ = weights_of(g["scores"])
    np.testing.assert_allclose(w, g["weights"], rtol=0, atol=g["tol4"])
    o1, lse1 = row(g["block1"], g["values"][:4])
    m1 = max(g["block1"])
    l1 = math.exp(lse1 - m1)
    assert abs(l1 - g["l1"]) <= g["tol4"]
    assert abs(o1[0] * l1 - g["O1_unnormalised"]) <= g["tol3"]
    assert abs(math.exp(m1 - m) - g["alpha"]) <= g["tol4"]


def test_worked_example_lse():
    g = read_golden("worked_example_lse.txt")
    _, lse = row(g["scores"], [0.0] * 4)
    assert abs(lse - g["LSE"]) <= g["tol"]
    _, lse1 = row(g["block1"], [0.0] * 2)
    assert abs(math.exp(lse1 - max(g["block1"])) - g["l1"]) <= g["tol"]
    assert abs(math.exp(lse - max(g["scores"])) - g["l2"]) <= g["tol"]


def test_overflow_guard():
    g = read_golden("overflow_guard.txt")
    w, lse = weights_of(g["scores"])
    assert np.all(np.isfinite(w)) and np.isfinite(lse)
    e = np.asarray(g["exp_shifted"])
    np.testing.assert_allclose(w, e / e.sum(), rtol=0, atol=g["tol"])
    np.testing.assert_allclose(w[1] / w[0], math.exp(g["shifted"][1]), rtol=1e-12)


# ---------------------------------------------------------------- closed forms

def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_single_key_gives_v():
    q, k, v = rand((2, 3, 5, 8), 1), rand((2, 3, 1, 8), 2), rand((2, 3, 1, 8), 3)
    o, lse = oracle.fwd(q, k, v, scale=0.7)
    np.testing.assert_allclose(o, np.broadcast_to(v, o.shape), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, 0.7 * np.einsum("bhid,bhjd->bhi", q, k), atol=1e-13)


def test_identical_keys_give_mean_of_v():
    q = rand((1, 2, 6, 4), 4)
    k = np.broadcast_to(rand((1, 2, 1, 4), 5), (1, 2, 9, 4)).copy()
    v = rand((1, 2, 9, 4), 6)
    o, lse = oracle.fwd(q, k, v, scale=0.5)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape),
                               atol=1e-14)
    s0 = 0.5 * np.einsum("bhid,bhd->bhi", q, k[:, :, 0])
    np.testing.assert_allclose(lse, s0 + math.log(9), atol=1e-13)


def test_causal_square_row0_is_v0_and_last_row_is_full():
    q, k, v = rand((1, 1, 7, 4), 7), rand((1, 1, 7, 4), 8), rand((1, 1, 7, 4), 9)
    oc, _ = oracle.fwd(q, k, v, scale=0.3, causal=True)
    on, _ = oracle.fwd(q, k, v, scale=0.3, causal=False)
    np.testing.assert_allclose(oc[0, 0, 0], v[0, 0, 0], atol=1e-15)
    np.testing.assert_allclose(oc[0, 0, -1], on[0, 0, -1], atol=1e-15)
    # row i sees exactly keys 0..i: same as a non-causal problem on K[:i+1]
    for i in range(7):
        oi, li = oracle.fwd(q[:, :, i:i + 1], k[:, :, :i + 1], v[:, :, :i + 1], scale=0.3)
        np.testing.assert_allclose(oc[0, 0, i], oi[0, 0, 0], atol=1e-14)


def test_causal_bottom_right_alignment():
    # Nq > Nk: query i sees keys j <= i - (Nq - Nk); the first rows see nothing.
    q, k, v = rand((1, 1, 5, 4), 10), rand((1, 1, 3, 4), 11), rand((1, 1, 3, 4), 12)
    o, lse = oracle.fwd(q, k, v, scale=1.0, causal=True)
    assert np.all(o[0, 0, :2] == 0.0) and np.all(np.isneginf(lse[0, 0, :2]))
    np.testing.assert_allclose(o[0, 0, 2], v[0, 0, 0], atol=1e-15)
    on, ln_ = oracle.fwd(q, k, v, scale=1.0)
    np.testing.assert_allclose(o[0, 0, 4], on[0, 0, 4], atol=1e-15)
    # Nq < Nk: the last query sees every key, the first sees Nk - Nq + 1 keys
    q, k, v = rand((1, 1, 2, 4), 13), rand((1, 1, 6, 4), 14), rand((1, 1, 6, 4), 15)
    o, lse = oracle.fwd(q, k, v, scale=1.0, causal=True)
    on, _ = oracle.fwd(q, k, v, scale=1.0)
    np.testing.assert_allclose(o[0, 0, 1], on[0, 0, 1], atol=1e-15)
    o0, _ = oracle.fwd(q[:, :, :1], k[:, :, :5], v[:, :, :5], scale=1.0)
    np.testing.assert_allclose(o[0, 0, 0], o0[0, 0, 0], atol=1e-15)


def test_fully_masked_rows_are_zero_with_neg_inf_lse():
    q, k, v = rand((2, 1, 3, 4), 16), rand((2, 1, 1, 4), 17), rand((2, 1, 1, 4), 18)
    bias = np.array([[-np.inf], [0.0]])
    o, lse = oracle.fwd(q, k, v, bias=bias, scale=1.0)
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(lse[0]))
    np.testing.assert_allclose(o[1, 0], np.broadcast_to(v[1, 0, 0], (3, 4)), atol=1e-15)


def test_key_padding_equals_truncation_and_ignores_masked_values():
    B, H, Nq, Nk, d = 3, 2, 5, 11, 6
    q, k, v = rand((B, H, Nq, d), 19), rand((B, H, Nk, d), 20), rand((B, H, Nk, d), 21)
    L = [11, 6, 1]
    bias = np.zeros((B, Nk))
    for b, Lb in enumerate(L):
        bias[b, Lb:] = -np.inf
        v[b, :, Lb:] = np.nan          # masked keys must get weight exactly 0
    o, lse = oracle.fwd(q, k, v, bias=bias, scale=0.4)
    assert np.all(np.isfinite(o))
    for b, Lb in enumerate(L):
        ot, lt = oracle.fwd(q[b:b + 1], k[b:b + 1, :, :Lb], v[b:b + 1, :, :Lb], scale=0.4)
        np.testing.assert_allclose(o[b], ot[0], atol=1e-15)
        np.testing.assert_allclose(lse[b], lt[0], atol=1e-15)


def test_finite_bias_shifts_scores_after_scaling():
    # S = scale * q.k + bias (bias NOT scaled): a constant bias leaves O unchanged
    # and shifts LSE by exactly that constant; a bias on one key equals scaling
    # its weight by e^bias.
    q, k, v = rand((1, 1, 4, 3), 22), rand((1, 1, 5, 3), 23), rand((1, 1, 5, 3), 24)
    o0, l0 = oracle.fwd(q, k, v, scale=0.25)
    o1, l1 = oracle.fwd(q, k, v, bias=np.full((1, 5), 2.5), scale=0.25)
    np.testing.assert_allclose(o1, o0, atol=1e-14)
    np.testing.assert_allclose(l1, l0 + 2.5, atol=1e-13)
    bias = np.zeros((1, 5))
    bias[0, 2] = math.log(3.0)
    o2, _ = oracle.fwd(q, k, v, bias=bias, scale=0.25)
    k3 = np.concatenate([k, k[:, :, 2:3], k[:, :, 2:3]], axis=2)   # key 2 three times
    v3 = np.concatenate([v, v[:, :, 2:3], v[:, :, 2:3]], axis=2)
    o3, _ = oracle.fwd(q, k3, v3, scale=0.25)
    np.testing.assert_allclose(o2, o3, atol=1e-14)


# ------------------------------------------------------------- invariants

def test_probabilities_rebuilt_from_lse_sum_to_one():
    B, H, Nq, Nk, d = 2, 2, 9, 13, 8
    q, k, v = rand((B, H, Nq, d), 25), rand((B, H, Nk, d), 26), rand((B, H, Nk, d), 27)
    for causal in (False, True):
        _, lse = oracle.fwd(q, k, v, scale=0.35, causal=causal)
        s = 0.35 * np.einsum("bhid,bhjd->bhij", q, k)
        if causal:
            i = np.arange(Nq)[:, None]
            j = np.arange(Nk)[None, :]
            s = np.where(j <= i + Nk - Nq, s, -np.inf)
        np.testing.assert_allclose(np.exp(s - lse[..., None]).sum(-1), 1.0, atol=1e-13)


def online_softmax_attention(s, V, block):
    """Independent one-pass streaming form of one attention row: running max m,
    running denominator l and unnormalised accumulator a, merged block by block
    and normalised once at the end ("Understanding FlashAttention Pt 1", §2.3-2.4)."""
    m, l, a = -np.inf, 0.0, np.zeros(V.shape[1])
    for j0 in range(0, len(s), block):
        sb, vb = s[j0:j0 + block], V[j0:j0 + block]
        mn = max(m, sb.max())
        alpha = math.exp(m - mn) if m != -np.inf else 0.0
        p = np.exp(sb - mn)
        l = alpha * l + p.sum()
        a = alpha * a + p @ vb
        m = mn
    return a / l, m + math.log(l)


@pytest.mark.parametrize("block", [1, 3, 4, 7, 64])
def test_two_pass_oracle_matches_streaming_recurrence(block):
    rng = np.random.default_rng(0)
    s = rng.standard_normal(64) * 3
    V = rng.standard_normal((64, 8))
    o_ref, lse_ref = online_softmax_attention(s, V, block)
    o, lse = row(s, V)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    assert abs(lse - lse_ref) < 1e-13


def test_library_witness_sdpa_float64():
    """torch's math SDPA in float64 on the CPU, with the same bottom-right causal
    mask and additive key bias, on small shapes."""
    torch.manual_seed(0)
    for (B, H, Nq, Nk, d, causal, use_bias) in [(2, 3, 17, 17, 16, False, False),
                                                (1, 2, 9, 23, 8, True, True),
                                                (2, 1, 20, 7, 4, True, False),
                                                (1, 1, 33, 40, 12, False, True)]:
        q = torch.randn(B, H, Nq, d, dtype=torch.float64)
        k = torch.randn(B, H, Nk, d, dtype=torch.float64)
        v = torch.randn(B, H, Nk, d, dtype=torch.float64)
        bias = None
        mask = torch.zeros(B, 1, Nq, Nk, dtype=torch.float64)
        if use_bias:
            bias = torch.randn(B, Nk, dtype=torch.float64)
            bias[:, -2:] = -math.inf
            mask = mask + bias[:, None, None, :]
        if causal:
            i = torch.arange(Nq)[:, None]
            j = torch.arange(Nk)[None, :]
            mask = mask.masked_fill(~(j <= i + Nk - Nq), -math.inf)
        rows_ok = torch.isfinite(mask).any(-1).expand(B, H, Nq)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                               scale=0.3)
        o, _ = oracle.fwd(q, k, v, bias=bias, scale=0.3, causal=causal)
        np.testing.assert_allclose(o[rows_ok.numpy()], ref.numpy()[rows_ok.numpy()],
                                   atol=1e-13)


def test_rows_api_matches_full():
    B, H, Nq, Nk, d = 2, 3, 20, 31, 8
    q, k, v = rand((B, H, Nq, d), 30), rand((B, H, Nk, d), 31), rand((B, H, Nk, d), 32)
    bias = np.zeros((B, Nk))
    bias[1, 25:] = -np.inf
    o, lse = oracle.fwd(q, k, v, bias=bias, scale=0.3, causal=True)
    heads = np.array([0, 5, 3, 5, 1])
    rows = np.array([0, 19, 7, 2, 13])
    orr, lrr = oracle.fwd_rows(q, k, v, bias, heads, rows, scale=0.3, causal=True)
    for t, (bh, i) in enumerate(zip(heads, rows)):
        b, h = divmod(bh, H)
        np.testing.assert_array_equal(orr[t], o[b, h, i])
        assert lrr[t] == lse[b, h, i] or (np.isneginf(lrr[t]) and np.isneginf(lse[b, h, i]))
    dO = rand((B, H, Nq, d), 33)
    dq, dk, dv = oracle.bwd(q, k, v, bias, dO, scale=0.3, causal=True)
    dqr = oracle.bwd_dq_rows(q, k, v, bias, dO, heads, rows, scale=0.3, causal=True)
    for t, (bh, i) in enumerate(zip(heads, rows)):
        b, h = divmod(bh, H)
        np.testing.assert_allclose(dqr[t], dq[b, h, i], atol=1e-15)
    hq, hk, hv = oracle.bwd_heads(q, k, v, bias, dO, [4, 1], scale=0.3, causal=True)
    np.testing.assert_allclose(hk[0], dk[1, 1], atol=1e-15)
    np.testing.assert_allclose(hv[1], dv[0, 1], atol=1e-15)


# ------------------------------------------------------------- backward

def fd_check(B, H, Nq, Nk, d, scale, causal, bias, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, Nq, d))
    k = rng.standard_normal((B, H, Nk, d))
    v = rng.standard_normal((B, H, Nk, d))
    G = rng.standard_normal((B, H, Nq, d))     # dO: loss = sum(O * G)

    def loss(q_, k_, v_):
        o, _ = oracle.fwd(q_, k_, v_, bias=bias, scale=scale, causal=causal)
        o = np.where(np.isfinite(o), o, 0.0)
        return float((o * G).sum())

    dq, dk, dv = oracle.bwd(q, k, v, bias, G, scale=scale, causal=causal)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy()
            xp[idx] += h
            xm = x.copy()
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name] = xp
            args_m[name] = xm
            num[idx] = (loss(**{a + "_": b for a, b in args_p.items()})
                        - loss(**{a + "_": b for a, b in args_m.items()})) / (2 * h)
        err = np.abs(num - g).max() / max(1.0, np.abs(g).max())
        assert err < 1e-6, (name, err)
    return dq, dk, dv


@pytest.mark.parametrize("case", [
    dict(B=1, H=1, Nq=6, Nk=6, d=4, scale=0.5, causal=False, bias=None),
    dict(B=1, H=2, Nq=7, Nk=7, d=3, scale=0.8, causal=True, bias=None),
    dict(B=2, H=1, Nq=5, Nk=9, d=4, scale=0.35, causal=True, bias="pad"),
    dict(B=1, H=1, Nq=9, Nk=4, d=2, scale=1.1, causal=True, bias=None),
    dict(B=2, H=1, Nq=4, Nk=8, d=5, scale=0.6, causal=False, bias="finite"),
])
def test_backward_finite_differences(case):
    case = dict(case)
    B, Nk = case["B"], case["Nk"]
    if case["bias"] == "pad":
        bias = np.zeros((B, Nk))
        bias[0, 6:] = -np.inf
        bias[1, 3:] = -np.inf
    elif case["bias"] == "finite":
        bias = np.random.default_rng(99).standard_normal((B, Nk))
    else:
        bias = None
    case["bias"] = bias
    dq, dk, dv = fd_check(seed=41, **case)
    if case["bias"] is not None and np.isneginf(bias).any():
        for b in range(B):
            masked = np.isneginf(bias[b])
            assert np.all(dk[b][:, masked] == 0.0) and np.all(dv[b][:, masked] == 0.0)


def test_backward_library_witness_autograd_float64():
    torch.manual_seed(1)
    B, H, Nq, Nk, d = 2, 2, 12, 15, 8
    q = torch.randn(B, H, Nq, d, dtype=torch.float64, requires_grad=True)
    k = torch.randn(B, H, Nk, d, dtype=torch.float64, requires_grad=True)
    v = torch.randn(B, H, Nk, d, dtype=torch.float64, requires_grad=True)
    G = torch.randn(B, H, Nq, d, dtype=torch.float64)
    i = torch.arange(Nq)[:, None]
    j = torch.arange(Nk)[None, :]
    mask = torch.zeros(Nq, Nk, dtype=torch.float64).masked_fill(~(j <= i + Nk - Nq), -math.inf)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=0.4)
    (o * G).sum().backward()
    dq, dk, dv = oracle.bwd(q, k, v, None, G, scale=0.4, causal=True)
    np.testing.assert_allclose(dq, q.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, k.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, v.grad.numpy(), atol=1e-12)


def test_rowsum_identity_D():
    # D_i = sum_c dO_ic O_ic equals sum_j P_ij dP_ij with dP = dO V^T
    # ("Understanding FlashAttention Pt 1", §3.6; "FlashAttention, Explained", §17).
    B, H, Nq, Nk, d = 1, 2, 10, 14, 6
    q, k, v = rand((B, H, Nq, d), 50), rand((B, H, Nk, d), 51), rand((B, H, Nk, d), 52)
    G = rand((B, H, Nq, d), 53)
    o, lse = oracle.fwd(q, k, v, scale=0.45, causal=True)
    s = 0.45 * np.einsum("bhid,bhjd->bhij", q, k)
    i = np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    s = np.where(j <= i + Nk - Nq, s, -np.inf)
    P = np.exp(s - lse[..., None])
    dP = np.einsum("bhid,bhjd->bhij", G, v)
    np.testing.assert_allclose((G * o).sum(-1), (P * dP).sum(-1), atol=1e-13)


def test_row_sampled_backward_sums_to_full_backward():
    B, H, Nq, Nk, d = 1, 1, 13, 17, 6
    q, k, v, G = rand((B, H, Nq, d), 60), rand((B, H, Nk, d), 61), rand((B, H, Nk, d), 62), \
        rand((B, H, Nq, d), 63)
    bias = np.zeros((B, Nk))
    bias[0, 15:] = -np.inf
    dq, dk, dv = oracle.bwd(q, k, v, bias, G, scale=0.5, causal=True)
    dk_acc, dv_acc = np.zeros((Nk, d)), np.zeros((Nk, d))
    parts = [np.arange(0, 5), np.arange(5, 13)]
    for rows in parts:
        dqr, _, _ = oracle.bwd_head_rows(q[0, 0], k[0, 0], v[0, 0], bias[0], G[0, 0], rows, 0.5,
                                         True, dk=dk_acc, dv=dv_acc)
        np.testing.assert_allclose(dqr, dq[0, 0, rows], atol=1e-15)
    np.testing.assert_allclose(dk_acc, dk[0, 0], atol=1e-14)
    np.testing.assert_allclose(dv_acc, dv[0, 0], atol=1e-14)
    o, l = oracle.fwd_head_rows(q[0, 0], k[0, 0], v[0, 0], bias[0], [3, 12], 0.5, True)
    of, lf = oracle.fwd(q, k, v, bias=bias, scale=0.5, causal=True)
    np.testing.assert_allclose(o, of[0, 0, [3, 12]], atol=1e-15)


# ------------------------------------------------------------- grouped heads

def test_gqa_oracle_is_per_head_attention_on_the_shared_head():
    B, H, Hkv, Nq, Nk, d = 2, 6, 2, 5, 9, 4
    q, k, v = rand((B, H, Nq, d), 70), rand((B, Hkv, Nk, d), 71), rand((B, Hkv, Nk, d), 72)
    o, lse = oracle.fwd_gqa(q, k, v, scale=0.5, causal=True)
    for b in range(B):
        for h in range(H):
            kv = h // (H // Hkv)
            oh, lh = oracle.fwd(q[b:b + 1, h:h + 1], k[b:b + 1, kv:kv + 1], v[b:b + 1, kv:kv + 1],
                                scale=0.5, causal=True)
            np.testing.assert_array_equal(o[b, h], oh[0, 0])
            np.testing.assert_array_equal(lse[b, h], lh[0, 0])
    o2, _ = oracle.fwd_gqa(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), scale=0.5,
                           causal=True)
    np.testing.assert_array_equal(o, o2)    # Hkv == H reduces to multi-head


def test_gqa_backward_finite_differences_on_shared_heads():
    B, H, Hkv, Nq, Nk, d = 1, 4, 2, 5, 6, 3
    rng = np.random.default_rng(73)
    q, k, v = (rng.standard_normal(s) for s in ((B, H, Nq, d), (B, Hkv, Nk, d), (B, Hkv, Nk, d)))
    G = rng.standard_normal((B, H, Nq, d))

    def loss(k_, v_):
        o, _ = oracle.fwd_gqa(q, k_, v_, scale=0.6, causal=True)
        return float((o * G).sum())

    _, dk, dv = oracle.bwd_gqa(q, k, v, None, G, scale=0.6, causal=True)
    h = 1e-6
    for name, x, g in (("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            lp = loss(xp, v) if name == "k" else loss(k, xp)
            lm = loss(xm, v) if name == "k" else loss(k, xm)
            num[idx] = (lp - lm) / (2 * h)
        assert np.abs(num - g).max() < 1e-6 * max(1.0, np.abs(g).max()), name


# ------------------------------------------------------------- packed sequences

def test_varlen_oracle_equal_lengths_is_the_dense_batch():
    B, H, N, d = 3, 2, 7, 4
    q, k, v = rand((B, H, N, d), 80), rand((B, H, N, d), 81), rand((B, H, N, d), 82)
    pack = lambda x: np.concatenate([x[b] for b in range(B)], axis=1)   # [H, B*N, d]
    cu = np.arange(0, (B + 1) * N, N)
    o, lse = oracle.fwd_varlen(pack(q), pack(k), pack(v), cu, cu, scale=0.4, causal=True)
    od, ld = oracle.fwd(q, k, v, scale=0.4, causal=True)
    np.testing.assert_array_equal(o, pack(od))
    np.testing.assert_array_equal(lse, np.concatenate([ld[b] for b in range(B)], axis=1))
    G = rand((B, H, N, d), 83)
    dq, dk, dv = oracle.bwd_varlen(pack(q), pack(k), pack(v), pack(G), cu, cu, scale=0.4,
                                   causal=True)
    dqd, dkd, dvd = oracle.bwd(q, k, v, None, G, scale=0.4, causal=True)
    np.testing.assert_allclose(dq, pack(dqd), atol=1e-15)
    np.testing.assert_allclose(dk, pack(dkd), atol=1e-15)


def test_varlen_oracle_sequences_do_not_interact():
    H, d = 2, 4
    lens = [3, 0, 5]
    total = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v = rand((H, total, d), 84), rand((H, total, d), 85), rand((H, total, d), 86)
    o, _ = oracle.fwd_varlen(q, k, v, cu, cu, scale=1.0)
    v2 = v.copy()
    v2[:, 3:] += 100.0            # change only the last sequence's values
    o2, _ = oracle.fwd_varlen(q, k, v2, cu, cu, scale=1.0)
    np.testing.assert_array_equal(o[:, :3], o2[:, :3])


# ---------------------------------------------------------------- e4m3 (FP8 forward)

def test_e4m3_value_set_from_definition():
    vals = oracle.e4m3_values()
    assert len(vals) == 253                      # 2 x 127 finite codes, +0 and -0 merged
    assert vals.max() == 448.0 and vals.min() == -448.0
    pos = vals[vals > 0]
    assert pos.min() == 2.0 ** -9                # smallest subnormal
    assert 1.0 in vals and 1.125 in vals and 1.0625 not in vals


def test_e4m3_conversion_rounds_to_nearest_even():
    """The library conversion behind oracle.quantize_e4m3 against the format:
    every value maps to itself, and any x in range to the nearest finite
    e4m3 value, a tie to the one with an even mantissa."""
    import torch
    vals = oracle.e4m3_values()
    t = torch.from_numpy(vals).float()
    assert torch.equal(t.to(torch.float8_e4m3fn).float(), t)
    # mantissa parity of each value (from its place in the ordered positive set)
    pos = vals[vals > 0]
    code = {v: i for i, v in enumerate(pos)}   # consecutive codes alternate mantissa parity
    g = np.random.default_rng(5)
    x = np.concatenate([g.uniform(-448, 448, 4000), g.uniform(-4, 4, 4000),
                        g.uniform(-2 ** -6, 2 ** -6, 2000),
                        (pos[:-1] + pos[1:]) / 2])              # exact midpoints (ties)
    got = torch.from_numpy(x).float().to(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    for xi, gi in zip(x, got):
        xa = abs(float(np.float32(xi)))
        d = np.abs(pos - xa)
        best = d.min()
        cands = pos[d == best]
        if xa < pos.min() / 2 or (xa == pos.min() / 2):
            want = 0.0
        elif len(cands) == 1:
            want = cands[0]
        else:   # tie: the even code (code 0 = 2^-9 is odd mantissa 1)
            want = [c for c in cands if (code[c] + 1) % 2 == 0][0]
        assert abs(gi) == want, (xi, gi, want)


def test_quantize_e4m3_scale_and_error():
    import torch
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(2, 3, 50, 128, generator=g) * 3).to(torch.bfloat16)
    x8, sc = oracle.quantize_e4m3(x)
    xf = x.float()
    amax = xf.abs().amax(dim=(-1, -2))
    assert torch.equal(sc, amax / 448.0)
    assert float(x8.abs().max()) <= 448.0
    # the head's largest |x| lands on 448 exactly; normal values round within 2^-4 relative
    assert torch.equal(x8.abs().amax(dim=(-1, -2)), torch.full_like(sc, 448.0))
    rel = ((x8 * sc[..., None, None] - xf).abs() / xf.abs().clamp_min(1e-30))
    normal = (xf / sc[..., None, None]).abs() >= 2.0 ** -6
    assert float(rel[normal].max()) <= 2.0 ** -4 + 1e-7
    zero = torch.zeros(1, 1, 4, 128)
    z8, zs = oracle.quantize_e4m3(zero)
    assert float(zs) == 1.0 and float(z8.abs().max()) == 0.0
