"""Device-side failure path, exercised without faulting the GPU.

Every wait inside the kernels is bounded: when it runs out, the kernel records
a code in the device error word and returns, and the host reads it with
fa_get_last_device_error. This test makes such a wait run out on purpose
(a barrier nothing arrives at), then checks the status, that reading it
clears it, and that the context still computes correct results afterwards.
"""
import time

import numpy as np
import pytest
import torch

import exact_io_aware_03_gb300 as fa
import oracle
from parity import compare, compare_lse

pytestmark = pytest.mark.gpu


def test_bounded_wait_timeout_is_reported_and_context_stays_usable():
    from exact_io_aware_03_gb300 import build
    build.build()
    fa.load()
    stream = torch.cuda.current_stream().cuda_stream
    assert fa.fa_get_last_device_error(stream) == fa.FA_OK     # clean start
    t0 = time.time()
    assert fa.fa_selftest_device_timeout(stream) == fa.FA_OK   # launch succeeds
    assert fa.fa_get_last_device_error(stream) == fa.FA_ERR_DEVICE
    waited = time.time() - t0
    assert 0.5 < waited < 30.0, waited                         # the bounded wait, not a hang
    assert fa.fa_get_last_device_error(stream) == fa.FA_OK     # reading cleared it
    # the context is intact: a forward still matches the oracle
    g = torch.Generator().manual_seed(4)
    q, k, v = (torch.randn(1, 2, 200, 128, generator=g).to(torch.bfloat16) for _ in range(3))
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    fa.check_device_error()
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=128 ** -0.5, causal=True)
    compare("O", o.cpu(), o_ref)
    compare_lse(lse.cpu(), lse_ref)
