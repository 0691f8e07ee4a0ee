"""The largest shapes along each axis the tests afford: a 65,536-token causal
sequence (forward rows and dQ rows against the oracle, every output finite,
masked-key gradients exactly zero) and 2048 heads of a short sequence (in full).
These exercise the 64-bit row offsets and the grid orderings at sizes far from
the named workloads."""
import numpy as np
import pytest
import torch

import exact_io_aware_03_gb300 as fa
import oracle
from parity import compare, compare_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_io_aware_03_gb300 import build
    build.build()
    fa.load()


def test_long_sequence_forward_backward_sampled():
    N, d = 65536, 128
    g = torch.Generator().manual_seed(65536)
    q, k, v, dO = (torch.randn(1, 2, N, d, generator=g).to(torch.bfloat16) for _ in range(4))
    qd, kd, vd, dOd = (t.cuda() for t in (q, k, v, dO))
    o, lse = fa.fwd(qd, kd, vd, causal=True)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dOd, causal=True)
    fa.check_device_error()
    for t in (o, dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())
    rng = np.random.default_rng(1)
    heads = np.concatenate([rng.integers(0, 2, 24), [0, 1]])
    rows = np.concatenate([rng.integers(0, N, 24), [N - 1, 0]])
    o_r, lse_r = oracle.fwd_rows(q, k, v, None, heads, rows, scale=d ** -0.5, causal=True)
    oc, lc = o.cpu(), lse.cpu()
    compare("O[sampled rows, N=65536]", torch.stack([oc[0, h, r] for h, r in zip(heads, rows)]), o_r)
    compare_lse(torch.stack([lc[0, h, r] for h, r in zip(heads, rows)]), lse_r, extra="N=65536")
    dq_r = oracle.bwd_dq_rows(q, k, v, None, dO, heads[:8], rows[:8], scale=d ** -0.5, causal=True)
    dqc = dq.cpu()
    compare("dQ[sampled rows, N=65536]",
            torch.stack([dqc[0, h, r] for h, r in zip(heads[:8], rows[:8])]), dq_r)


def test_many_heads_full_parity():
    B, H, N, d = 2, 1024, 160, 64
    g = torch.Generator().manual_seed(2048)
    q, k, v, dO = (torch.randn(B, H, N, d, generator=g).to(torch.bfloat16) for _ in range(4))
    qd, kd, vd, dOd = (t.cuda() for t in (q, k, v, dO))
    o, lse = fa.fwd(qd, kd, vd, causal=True)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dOd, causal=True)
    fa.check_device_error()
    o_r, lse_r = oracle.fwd(q, k, v, scale=d ** -0.5, causal=True)
    compare("O[2048 heads]", o.cpu(), o_r)
    compare_lse(lse.cpu(), lse_r, extra="2048 heads")
    dq_r, dk_r, dv_r = oracle.bwd(q, k, v, None, dO, scale=d ** -0.5, causal=True)
    compare("dQ[2048 heads]", dq.cpu(), dq_r)
    compare("dK[2048 heads]", dk.cpu(), dk_r)
    compare("dV[2048 heads]", dv.cpu(), dv_r)
