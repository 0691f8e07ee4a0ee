"""Packed variable-length batches (fa_fwd_varlen, fa_bwd_varlen) against the
fp64 oracle run sequence by sequence."""
import numpy as np
import pytest
import torch

import exact_io_aware_03_gb300 as fa
import oracle
from parity import Guarded, compare, compare_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_io_aware_03_gb300 import build
    build.build()
    fa.load()


def packed(H, lens, d, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(H, sum(lens), d, generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("lens_q,lens_k,H,Hkv,d,causal", [
    ([100, 300, 1, 0, 777], None, 4, 2, 128, True),
    ([100, 300, 5], [200, 150, 1000], 2, 2, 128, True),     # cross lengths, bottom-right
    ([129, 64, 513], None, 3, 1, 64, False),
    ([1000], [1], 2, 2, 128, False),
    ([7, 0, 300], [0, 50, 300], 2, 1, 128, True),           # a sequence with no key
])
def test_varlen_forward_backward(lens_q, lens_k, H, Hkv, d, causal):
    lens_k = lens_q if lens_k is None else lens_k
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    q = packed(H, lens_q, d, 1)
    k = packed(Hkv, lens_k, d, 2)
    v = packed(Hkv, lens_k, d, 3)
    dO = packed(H, lens_q, d, 4)
    scale = d ** -0.5
    cq, ck = torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda()
    qd, kd, vd, dOd = (t.cuda() for t in (q, k, v, dO))
    o = Guarded(q.shape, torch.bfloat16)
    lse = Guarded(q.shape[:2], torch.float32)
    fa.fwd_varlen(qd, kd, vd, cq, ck, causal=causal, scale=scale, out=o.t, lse=lse.t)
    gq, gk, gv = (Guarded(t.shape, torch.bfloat16) for t in (q, k, v))
    fa.bwd_varlen(qd, kd, vd, o.t, lse.t, dOd, cq, ck, causal=causal, scale=scale, dq=gq.t,
                  dk=gk.t, dv=gv.t)
    fa.check_device_error()
    for gd, n in ((o, "O"), (lse, "LSE"), (gq, "dQ"), (gk, "dK"), (gv, "dV")):
        gd.check(n)
    o_ref, lse_ref = oracle.fwd_varlen(q, k, v, cu_q, cu_k, scale=scale, causal=causal)
    dq_ref, dk_ref, dv_ref = oracle.bwd_varlen(q, k, v, dO, cu_q, cu_k, scale=scale,
                                               causal=causal)
    tag = "(lens_q=%s,lens_k=%s,H=%d,Hkv=%d,d=%d,causal=%s)" % (lens_q, lens_k, H, Hkv, d, causal)
    compare("O", o.t.cpu(), o_ref, extra=tag)
    compare_lse(lse.t.cpu(), lse_ref, extra=tag)
    compare("dQ", gq.t.cpu(), dq_ref, extra=tag)
    compare("dK", gk.t.cpu(), dk_ref, extra=tag)
    compare("dV", gv.t.cpu(), dv_ref, extra=tag)


def test_varlen_length_beyond_declared_maximum_is_reported():
    lens = [100, 300]
    cu = torch.tensor([0, 100, 400], dtype=torch.int32).cuda()
    q = packed(2, lens, 64, 5).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    assert fa.fa_get_last_device_error(stream) == fa.FA_OK
    # declare a maximum (200) smaller than the second sequence (300)
    fa.fwd_varlen(q, q, q, cu, cu, max_seqlen_q=200, max_seqlen_k=200)
    assert fa.fa_get_last_device_error(stream) == fa.FA_ERR_DEVICE
    assert fa.fa_get_last_device_error(stream) == fa.FA_OK
