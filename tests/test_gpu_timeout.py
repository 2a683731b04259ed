"""Failure path of the attention kernel, without faulting the GPU: a
host-set flag makes the TMA producer skip its K/V copies, so the MMA and
softmax warps' bounded waits (short limit here) run out.  The kernel must
return on its own, report CPATTN_ERR_TIMEOUT through the device error word,
and leave the context usable: the next normal call is correct."""
import numpy as np
import pytest
import torch

import context_attention_partial_gb300 as cp
import oracle
from workloads import make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TIMEOUT = 9


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 64),
                                     (torch.float32, 128)])
def test_stalled_producer_times_out_and_recovers(dtype, d):
    lib = cp.load_library()
    q, k, v = make_qkv((1, 2, 300, d), dtype, seed=31, device=DEV)
    try:
        cp.set_wait_timeout_ns(20_000_000)          # 20 ms
        lib.cpattn_set_fault_injection(1)
        cp.ring(q, k, v, ring_degree=2)
        assert cp.last_device_status() == TIMEOUT
        assert cp.last_device_status() == 0          # the word was cleared
    finally:
        lib.cpattn_set_fault_injection(0)
        cp.set_wait_timeout_ns(2_000_000_000)
    out, lse = cp.ring(q, k, v, ring_degree=2)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    ro, rl = oracle.ring(q.cpu(), k.cpu(), v.cpu(), d ** -0.5, ring_degree=2)
    tol = 1e-2 if dtype == torch.bfloat16 else 2e-3
    assert np.abs(out.float().cpu().numpy() - ro).max() <= tol
    assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-3
