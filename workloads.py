"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and describes problem shapes; it holds
none of the attention arithmetic, so the oracle and the CUDA path can both use
it without sharing any of the method.

Recipe (same for every consumer):
  * a CPU ``torch.Generator`` seeded with ``seed``; tensors are drawn in the
    order q, k, v, dO, then the per-batch valid key lengths;
  * q, k, v, dO are i.i.d. N(0, 1) in float32, then rounded to bfloat16 with
    round-to-nearest-even (``Tensor.to``), except for float32 problems;
  * key-padding problems: the valid key length of batch b is a uniform integer
    in [Nk/2, Nk] (inclusive); bias[b, j] = 0 for j < L_b and -inf otherwise.

The named workloads below are the problem shapes the benchmark and the parity
tests run; their seeds are 1001..1006 (the sixth, a decode step, exercises the
split-KV forward).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    dtype: str             # "bf16" or "fp32": storage/IO type of q, k, v, o
    causal: bool
    key_padding: bool      # additive [B, Nk] bias with -inf past a per-batch length
    backward: bool         # whether the workload includes the backward pass
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # single head, fp32, forward only
    "f32_b1h1_n128_d64": Workload("f32_b1h1_n128_d64", 1, 1, 128, 128, 64, "fp32",
                                  False, False, False, 1001),
    # short sequences, d=64, forward (run non-causal and causal)
    "bf16_b4h16_n2048_d64": Workload("bf16_b4h16_n2048_d64", 4, 16, 2048, 2048, 64, "bf16",
                                     False, False, False, 1002),
    # long-context causal forward, d=128
    "bf16_b2h32_n8192_d128_causal": Workload("bf16_b2h32_n8192_d128_causal", 2, 32, 8192, 8192,
                                             128, "bf16", True, False, False, 1003),
    # causal forward + backward, d=128
    "bf16_b4h16_n4096_d128_causal_bwd": Workload("bf16_b4h16_n4096_d128_causal_bwd", 4, 16, 4096,
                                                 4096, 128, "bf16", True, False, True, 1004),
    # cross-attention with key padding, forward + backward
    "bf16_b8h16_q1024_k16384_d128_keypad": Workload("bf16_b8h16_q1024_k16384_d128_keypad", 8, 16,
                                                    1024, 16384, 128, "bf16", False, True, True,
                                                    1005),
    # decode step with a long key/value context: one query row per head
    # (the split-KV forward's workload)
    "bf16_b8h32_q1_k32768_d128_decode": Workload("bf16_b8h32_q1_k32768_d128_decode", 8, 32, 1,
                                                 32768, 128, "bf16", False, False, False, 1006),
}


def make_inputs(w: Workload, with_dO: Optional[bool] = None, seed: Optional[int] = None):
    """Return a dict of CPU tensors: q, k, v, (dO), bias (or None), key_len (or None)."""
    if with_dO is None:
        with_dO = w.backward
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    dt = w.torch_dtype

    def draw(n):
        return torch.randn((w.B, w.H, n, w.d), generator=g, dtype=torch.float32).to(dt)

    out = {"q": draw(w.Nq), "k": draw(w.Nk), "v": draw(w.Nk), "dO": None,
           "bias": None, "key_len": None}
    if with_dO:
        out["dO"] = draw(w.Nq)
    if w.key_padding:
        lo = w.Nk // 2
        L = torch.randint(lo, w.Nk + 1, (w.B,), generator=g, dtype=torch.int64)
        j = torch.arange(w.Nk, dtype=torch.int64)
        bias = torch.zeros((w.B, w.Nk), dtype=torch.float32)
        bias[j[None, :] >= L[:, None]] = float("-inf")
        out["bias"] = bias
        out["key_len"] = L
    return out


def sample_rows(w: Workload, n: int, seed: int = 7):
    """n (flat head, query row) pairs drawn uniformly, plus every head's last row.

    Used to check full-size outputs element by element on a subset the
    oracle can afford.
    """
    g = torch.Generator().manual_seed(seed)
    heads = torch.randint(0, w.B * w.H, (n,), generator=g)
    rows = torch.randint(0, w.Nq, (n,), generator=g)
    heads = torch.cat([heads, torch.tensor([0, w.B * w.H - 1])])
    rows = torch.cat([rows, torch.tensor([w.Nq - 1, w.Nq - 1])])
    return heads.numpy(), rows.numpy()


def sample_rows_dense(w: Workload, n: int, n_tile_heads: int = 4, seed: int = 7, tile: int = 128):
    """``sample_rows(w, n)`` plus every row of the first and the last
    ``tile``-row query tile of ``n_tile_heads`` heads (the first, the last and
    seeded others). The first tile of a causal head holds row 0 (whose output
    is V_0) and the rows with the fewest keys, where outputs are largest.
    Returns (heads, rows) as int64 numpy arrays, duplicates removed."""
    import numpy as np
    heads, rows = sample_rows(w, n, seed)
    g = torch.Generator().manual_seed(seed + 1)
    BH = w.B * w.H
    picks = [0, BH - 1] + torch.randint(0, BH, (max(0, n_tile_heads - 2),), generator=g).tolist()
    extra_h, extra_r = [], []
    for h in dict.fromkeys(picks[:max(1, n_tile_heads)]):
        for r in list(range(min(tile, w.Nq))) + list(range(max(0, w.Nq - tile), w.Nq)):
            extra_h.append(h)
            extra_r.append(r)
    pairs = np.unique(np.stack([np.concatenate([heads, np.asarray(extra_h, dtype=np.int64)]),
                                np.concatenate([rows, np.asarray(extra_r, dtype=np.int64)])]),
                      axis=1)
    return pairs[0], pairs[1]


def sample_heads(w: Workload, n: int, seed: int = 11):
    """n distinct flat head indices b*H+h: the first, the last and seeded others."""
    g = torch.Generator().manual_seed(seed)
    BH = w.B * w.H
    out = [0, BH - 1]
    for h in torch.randperm(BH, generator=g).tolist():
        if len(out) >= min(n, BH):
            break
        if h not in out:
            out.append(h)
    return out[:min(n, BH)]


def varlen_lengths(n: int, seed: int, cap: int = 4096, lo: int = 64):
    """n sequence lengths drawn from a log-normal (median ~1000) clipped to
    [lo, cap] -- the ragged-batch shape used to compare packed and padded
    batches. Returns a list of ints."""
    g = torch.Generator().manual_seed(seed)
    x = torch.exp(torch.randn(n, generator=g, dtype=torch.float64) * 0.8 + math.log(1000.0))
    return [int(v) for v in x.clamp(lo, cap).round().tolist()]
