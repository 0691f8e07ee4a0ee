"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It computes the plain definition of
attention (materialised score rows, two-pass safe softmax, textbook softmax
Jacobian for the backward) in double precision; see ``oracle.c`` for the
formulas and the passages of the pages they follow. It shares no code with
the CUDA library.

All functions take torch tensors or numpy arrays of any float dtype in the
[B, H, N, d] layout (bias: [B, Nk]) and return float64 numpy arrays. The
widening to float64 is exact for bf16 and fp32 inputs.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lp = ctypes.POINTER(ctypes.c_long)
        ip = ctypes.POINTER(ctypes.c_int)
        ci, cd, cl = ctypes.c_int, ctypes.c_double, ctypes.c_long
        lib.oracle_fwd.argtypes = [dp, dp, dp, dp, dp, dp, ci, ci, ci, ci, ci, cd, ci]
        lib.oracle_fwd_rows.argtypes = [dp, dp, dp, dp, lp, ip, cl, dp, dp,
                                        ci, ci, ci, ci, ci, cd, ci]
        lib.oracle_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp,
                                   ci, ci, ci, ci, ci, cd, ci]
        lib.oracle_bwd_dq_rows.argtypes = [dp, dp, dp, dp, dp, lp, ip, cl, dp,
                                           ci, ci, ci, ci, ci, cd, ci]
        for f in (lib.oracle_fwd, lib.oracle_fwd_rows, lib.oracle_bwd,
                  lib.oracle_bwd_dq_rows):
            f.restype = ctypes.c_int
        lib.oracle_bwd_head_rows.argtypes = [dp, dp, dp, dp, dp, ip, ci, dp, dp, dp,
                                             ci, ci, ci, cd, ci, dp]
        lib.oracle_bwd_head_rows.restype = None
        lib.oracle_fwd_head_rows.argtypes = [dp, dp, dp, dp, ip, ci, dp, dp, ci, ci, ci, cd,
                                             ci, dp]
        lib.oracle_fwd_head_rows.restype = None
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(x):
    """Exact widening of a torch tensor / array to a contiguous float64 array."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shape4(q, k):
    B, H, Nq, d = q.shape
    Bk, Hk, Nk, dk = k.shape
    if (Bk, Hk, dk) != (B, H, d):
        raise ValueError("q and k/v must agree in B, H and d")
    return B, H, Nq, Nk, d


def num_threads() -> int:
    return _load().oracle_num_threads()


def fwd(q, k, v, bias=None, scale=None, causal=False):
    """O [B,H,Nq,d] and LSE [B,H,Nq] (natural log) of the full problem."""
    lib = _load()
    q, k, v, bias = _f64(q), _f64(k), _f64(v), _f64(bias)
    B, H, Nq, Nk, d = _shape4(q, k)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.empty((B, H, Nq, d))
    lse = np.empty((B, H, Nq))
    rc = lib.oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(o), _ptr(lse),
                        B, H, Nq, Nk, d, float(scale), int(bool(causal)))
    if rc:
        raise MemoryError("oracle_fwd: scratch allocation failed")
    return o, lse


def _head_groups(heads, rows):
    heads = np.asarray(heads, dtype=np.int64).reshape(-1)
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    if heads.shape != rows.shape:
        raise ValueError("heads and rows must have the same length")
    for h in np.unique(heads):
        idx = np.nonzero(heads == h)[0]
        yield int(h), idx, rows[idx]


def _head_slice(x, bh, H):
    """[N, d] float64 slice of head bh of a [B,H,N,d] tensor (converts one head only)."""
    b, h = divmod(bh, H)
    return _f64(x[b, h][None, None])


def fwd_rows(q, k, v, bias, heads, rows, scale=None, causal=False):
    """O [n,d] and LSE [n] for the (flat head b*H+h, query row) pairs given.

    Only the heads that are asked for are widened to float64, so this works
    at full problem sizes.
    """
    lib = _load()
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    heads_a = np.asarray(heads, dtype=np.int64).reshape(-1)
    o = np.empty((heads_a.size, d))
    lse = np.empty(heads_a.size)
    for bh, idx, r in _head_groups(heads, rows):
        qh, kh, vh = (_head_slice(t, bh, H) for t in (q, k, v))
        bh_bias = None if bias is None else _f64(bias[bh // H][None])
        n = idx.size
        hz = np.zeros(n, dtype=np.int64)                       # one head in the slice
        rr = np.ascontiguousarray(r, dtype=np.int32)
        oo = np.empty((n, d))
        ll = np.empty(n)
        rc = lib.oracle_fwd_rows(_ptr(qh), _ptr(kh), _ptr(vh), _ptr(bh_bias),
                                 hz.ctypes.data_as(ctypes.POINTER(ctypes.c_long)),
                                 rr.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), n,
                                 _ptr(oo), _ptr(ll), 1, 1, Nq, Nk, d,
                                 float(scale), int(bool(causal)))
        if rc:
            raise MemoryError("oracle_fwd_rows: scratch allocation failed")
        o[idx] = oo
        lse[idx] = ll
    return o, lse


def bwd(q, k, v, bias, dO, scale=None, causal=False):
    """dQ, dK, dV [B,H,N,d] of the full problem (loss gradient dO)."""
    lib = _load()
    q, k, v, bias, dO = _f64(q), _f64(k), _f64(v), _f64(bias), _f64(dO)
    B, H, Nq, Nk, d = _shape4(q, k)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.empty((B, H, Nq, d))
    dk = np.empty((B, H, Nk, d))
    dv = np.empty((B, H, Nk, d))
    rc = lib.oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(dO),
                        _ptr(dq), _ptr(dk), _ptr(dv), B, H, Nq, Nk, d,
                        float(scale), int(bool(causal)))
    if rc:
        raise MemoryError("oracle_bwd: scratch allocation failed")
    return dq, dk, dv


def bwd_heads(q, k, v, bias, dO, heads, scale=None, causal=False):
    """dQ, dK, dV of whole heads (flat indices b*H+h), each [n_heads, N, d].

    The selected heads are stacked as a batch of single-head problems so that
    they run in parallel (one OpenMP task per head).
    """
    H = q.shape[1]
    heads = [int(h) for h in heads]

    def sel(x):
        return np.stack([_f64(x[bh // H, bh % H]) for bh in heads])[:, None]

    bb = None if bias is None else np.stack([_f64(bias[bh // H]) for bh in heads])
    dq, dk, dv = bwd(sel(q), sel(k), sel(v), bb, sel(dO), scale=scale, causal=causal)
    return dq[:, 0], dk[:, 0], dv[:, 0]


def bwd_dq_rows(q, k, v, bias, dO, heads, rows, scale=None, causal=False):
    """dQ [n,d] for the (flat head, query row) pairs given."""
    lib = _load()
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    heads_a = np.asarray(heads, dtype=np.int64).reshape(-1)
    dq = np.empty((heads_a.size, d))
    for bh, idx, r in _head_groups(heads, rows):
        qh, kh, vh, doh = (_head_slice(t, bh, H) for t in (q, k, v, dO))
        bh_bias = None if bias is None else _f64(bias[bh // H][None])
        n = idx.size
        hz = np.zeros(n, dtype=np.int64)
        rr = np.ascontiguousarray(r, dtype=np.int32)
        out = np.empty((n, d))
        rc = lib.oracle_bwd_dq_rows(_ptr(qh), _ptr(kh), _ptr(vh), _ptr(bh_bias), _ptr(doh),
                                    hz.ctypes.data_as(ctypes.POINTER(ctypes.c_long)),
                                    rr.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), n,
                                    _ptr(out), 1, 1, Nq, Nk, d, float(scale),
                                    int(bool(causal)))
        if rc:
            raise MemoryError("oracle_bwd_dq_rows: scratch allocation failed")
        dq[idx] = out
    return dq


def bwd_head_rows(qh, kh, vh, bias_row, dOh, rows, scale, causal, dk=None, dv=None):
    """Backward contributions of the given query rows of one head (float64 arrays
    [N, d]; bias_row [Nk] or None), on the calling thread (releases the GIL).

    Returns dq [len(rows), d] and the dK, dV contributions [Nk, d] of those rows
    (accumulated into dk / dv when given). The same per-row work as ``bwd``.
    """
    lib = _load()
    Nq, d = qh.shape
    Nk = kh.shape[0]
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    dq = np.empty((rows.size, d))
    dk = np.zeros((Nk, d)) if dk is None else dk
    dv = np.zeros((Nk, d)) if dv is None else dv
    scratch = np.empty(2 * max(Nk, 1))
    lib.oracle_bwd_head_rows(_ptr(qh), _ptr(kh), _ptr(vh), _ptr(bias_row), _ptr(dOh),
                             rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), rows.size,
                             _ptr(dq), _ptr(dk), _ptr(dv), Nq, Nk, d, float(scale),
                             int(bool(causal)), _ptr(scratch))
    return dq, dk, dv


def fwd_head_rows(qh, kh, vh, bias_row, rows, scale, causal):
    """O [len(rows), d] and LSE of the given query rows of one head (float64 [N, d]),
    on the calling thread (releases the GIL)."""
    lib = _load()
    Nq, d = qh.shape
    Nk = kh.shape[0]
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    n = rows.size
    o = np.empty((n, d))
    lse = np.empty(n)
    scratch = np.empty(max(Nk, 1))
    lib.oracle_fwd_head_rows(_ptr(np.ascontiguousarray(qh)), _ptr(np.ascontiguousarray(kh)),
                             _ptr(np.ascontiguousarray(vh)), _ptr(bias_row),
                             rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), n,
                             _ptr(o), _ptr(lse), Nq, Nk, d, float(scale), int(bool(causal)),
                             _ptr(scratch))
    return o, lse


def _expand_kv(x, H):
    """[B, Hkv, N, d] -> [B, H, N, d]: query head h reads key/value head h // (H // Hkv)."""
    x = _f64(x)
    g = H // x.shape[1]
    return np.repeat(x, g, axis=1)


def fwd_gqa(q, k, v, bias=None, scale=None, causal=False):
    """Grouped-query attention: every query head attends its group's key/value
    head ("Understanding FlashAttention Pt 1", Part 4.1)."""
    H = q.shape[1]
    return fwd(q, _expand_kv(k, H), _expand_kv(v, H), bias=bias, scale=scale, causal=causal)


def bwd_gqa(q, k, v, bias, dO, scale=None, causal=False):
    """Backward of fwd_gqa: dK and dV of a shared head sum over its query heads."""
    B, H = q.shape[0], q.shape[1]
    Hkv = k.shape[1]
    dq, dk, dv = bwd(q, _expand_kv(k, H), _expand_kv(v, H), bias, dO, scale=scale, causal=causal)
    g = H // Hkv
    dk = dk.reshape(B, Hkv, g, *dk.shape[2:]).sum(axis=2)
    dv = dv.reshape(B, Hkv, g, *dv.shape[2:]).sum(axis=2)
    return dq, dk, dv


def fwd_varlen(q, k, v, cu_q, cu_k, scale=None, causal=False):
    """Packed sequences (q [H, total_q, d], k/v [H_kv, total_k, d], offsets [B+1]):
    each sequence is its own problem; returns O [H, total_q, d], LSE [H, total_q]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu_q = [int(x) for x in np.asarray(cu_q).reshape(-1)]
    cu_k = [int(x) for x in np.asarray(cu_k).reshape(-1)]
    H, total_q, d = q.shape
    o = np.zeros((H, total_q, d))
    lse = np.full((H, total_q), -np.inf)
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if q1 == q0:
            continue
        if k1 == k0:
            continue    # no key at all: O = 0, LSE = -inf
        ob, lb = fwd_gqa(q[None, :, q0:q1], k[None, :, k0:k1], v[None, :, k0:k1], scale=scale,
                         causal=causal)
        o[:, q0:q1] = ob[0]
        lse[:, q0:q1] = lb[0]
    return o, lse


def bwd_varlen(q, k, v, dO, cu_q, cu_k, scale=None, causal=False):
    """Backward of fwd_varlen: dQ [H, total_q, d], dK, dV [H_kv, total_k, d]."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    cu_q = [int(x) for x in np.asarray(cu_q).reshape(-1)]
    cu_k = [int(x) for x in np.asarray(cu_k).reshape(-1)]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if q1 == q0 or k1 == k0:
            continue
        gq, gk, gv = bwd_gqa(q[None, :, q0:q1], k[None, :, k0:k1], v[None, :, k0:k1], None,
                             dO[None, :, q0:q1], scale=scale, causal=causal)
        dq[:, q0:q1] = gq[0]
        dk[:, k0:k1] = gk[0]
        dv[:, k0:k1] = gv[0]
    return dq, dk, dv


# ---------------------------------------------------------------- e4m3
# The FP8 forward works on e4m3 copies of q, k, v with one scale per (batch,
# head): scale = max|x| / 448 (448 = the largest finite e4m3 value; 1 for an
# all-zero head) and x8 = e4m3(x / scale), round to nearest even ("FlashAttention,
# Explained", §21: low-precision operands with scaling factors). The rounding
# step is torch's float8_e4m3fn conversion (a library primitive, pinned in the
# tests against the e4m3 definition); everything here is on the CPU.

def e4m3_values():
    """All finite e4m3 values from the format's definition (1 sign bit, 4
    exponent bits with bias 7, 3 mantissa bits, subnormals, no infinity,
    exponent 15 with mantissa 7 = NaN)."""
    vals = []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
            vals.append(v)
    vals = sorted(set(vals))
    return np.array(sorted(set([-v for v in vals] + vals)))


def quantize_e4m3(x):
    """x: [..., N, d] bf16 or float CPU tensor, per-head scale over the last
    two dimensions. Returns (x8 as float32 values, scale [...] float32)."""
    import torch
    xf = x.float()
    amax = xf.abs().amax(dim=(-1, -2))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    x8 = (xf / scale[..., None, None]).to(torch.float8_e4m3fn)
    return x8.float(), scale


def fwd_fp8_dequantized(q, k, v, bias=None, scale=None, causal=False):
    """The attention the FP8 forward approximates: fwd on the dequantized
    scale_x * e4m3(x / scale_x) inputs (the rounding of P is the kernel's
    approximation on top, bounded separately)."""
    q8, sq = quantize_e4m3(q)
    k8, sk = quantize_e4m3(k)
    v8, sv = quantize_e4m3(v)
    qd = q8.double() * sq.double()[..., None, None]
    kd = k8.double() * sk.double()[..., None, None]
    vd = v8.double() * sv.double()[..., None, None]
    if k.shape[1] != q.shape[1]:
        return fwd_gqa(qd, kd, vd, bias, scale=scale, causal=causal)
    return fwd(qd, kd, vd, bias, scale=scale, causal=causal)
