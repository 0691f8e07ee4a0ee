"""The boundary's own entry points on the GPU: fa_fwd, fa_bwd_workspace_size and
fa_bwd called by their C names through ctypes, with device buffers that torch
only allocates, compared against the fp64 oracle.

The other GPU tests go through the binding's conveniences (which call these
same symbols for plain multi-head problems); here nothing but pointers,
sizes and a stream handle crosses the boundary.
"""
import ctypes
import math

import pytest
import torch

import exact_io_aware_03_gb300 as fa
import oracle
from parity import Guarded, compare, compare_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from exact_io_aware_03_gb300 import build
    build.build()
    torch.cuda.init()
    return fa.load()


CASES = [
    # B, H, Nq, Nk, d, causal, key padding
    (1, 2, 300, 300, 128, True, False),
    (2, 2, 200, 700, 64, False, True),
    (2, 1, 260, 520, 128, True, True),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,pad", CASES)
def test_c_abi_fa_fwd_fa_bwd_against_oracle(lib, B, H, Nq, Nk, d, causal, pad):
    g = torch.Generator().manual_seed(B * 7 + Nq + Nk + d)
    q, k, v, dO = (torch.randn(B, H, n, d, generator=g).to(torch.bfloat16)
                   for n in (Nq, Nk, Nk, Nq))
    bias = None
    if pad:
        L = torch.randint(Nk // 2, Nk + 1, (B,), generator=g)
        bias = torch.zeros(B, Nk)
        bias[torch.arange(Nk)[None, :] >= L[:, None]] = -math.inf
    scale = d ** -0.5
    dev = torch.device("cuda", 0)
    qd, kd, vd, dOd = (t.to(dev) for t in (q, k, v, dO))
    bd = None if bias is None else bias.to(dev)
    o, lse = Guarded(q.shape, torch.bfloat16), Guarded(q.shape[:3], torch.float32)
    dq, dk, dv = (Guarded(t.shape, torch.bfloat16) for t in (q, k, v))
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    p = lambda t: ctypes.c_void_p(None if t is None else t.data_ptr())

    st = lib.fa_fwd(p(qd), p(kd), p(vd), p(bd), p(o.t), p(lse.t), B, H, Nq, Nk, d,
                    ctypes.c_float(scale), int(causal), fa.FA_DTYPE_BF16, stream)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    ws_bytes = lib.fa_bwd_workspace_size(B, H, Nq, Nk, d)
    assert ws_bytes > 0
    ws = Guarded((ws_bytes,), torch.uint8)
    ws.t.fill_(0x5a)   # the workspace's contents on entry must not matter
    st = lib.fa_bwd(p(qd), p(kd), p(vd), p(o.t), p(lse.t), p(dOd), p(dq.t), p(dk.t), p(dv.t),
                    p(bd), B, H, Nq, Nk, d, ctypes.c_float(scale), int(causal),
                    fa.FA_DTYPE_BF16, p(ws.t), ctypes.c_size_t(ws_bytes), stream)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    assert lib.fa_get_last_device_error(stream) == fa.FA_OK
    for gb, name in ((o, "O"), (lse, "LSE"), (dq, "dQ"), (dk, "dK"), (dv, "dV"),
                     (ws, "workspace")):
        gb.check(name)

    o_ref, lse_ref = oracle.fwd(q, k, v, bias=bias, scale=scale, causal=causal)
    dq_ref, dk_ref, dv_ref = oracle.bwd(q, k, v, bias, dO, scale=scale, causal=causal)
    tag = "(%d,%d,%d,%d,%d,causal=%s,pad=%s)" % (B, H, Nq, Nk, d, causal, pad)
    compare("O", o.t, o_ref, extra=tag)
    compare_lse(lse.t, lse_ref, extra=tag)
    compare("dQ", dq.t, dq_ref, extra=tag)
    compare("dK", dk.t, dk_ref, extra=tag)
    compare("dV", dv.t, dv_ref, extra=tag)
