"""cpattn_ring_noalloc: the ring entry point for callers that cannot
allocate device memory (a fixed device-memory budget, a memory pool that
hands out no extra buffers, a plugin that only receives its input and output
pointers).  Its workspace is the library's own fixed device array, so the
caller passes inputs and outputs only.

This file is collected last on purpose.  The test calls the entry point
through the C ABI and checks its results against cpattn_ring (caller-given
workspace) on two calls in a row, within the tolerances of the other GPU
tests (identical kernel, so the results are expected to be bit-equal), and
checks that a problem whose workspace exceeds the fixed array is refused.
"""
import pytest
import torch

import context_attention_partial_gb300 as cp
from context_attention_partial_gb300 import _lib
from workloads import make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _call_noalloc(q, k, v, ring_degree, ring_anything, out, lse):
    lib = cp.load_library()
    d = lambda t, code: _lib.describe(t.data_ptr(), code, t.shape, t.stride())
    code = _lib.BF16 if q.dtype == torch.bfloat16 else _lib.F32
    return lib.cpattn_ring_noalloc(d(q, code), d(k, code), d(v, code), 0.0, ring_degree,
                                   int(ring_anything), d(out, code), d(lse, _lib.F32),
                                   torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("shape,R,anything,seeds", [
    ((1, 24, 4608, 128), 2, False, (0, 1)),     # the FLUX-like workload
    ((2, 3, 301, 128), 3, True, (2, 3)),        # ragged, uneven chunks
])
def test_noalloc_matches_ring_two_calls(shape, R, anything, seeds):
    lib = cp.load_library()
    assert lib.cpattn_ring_noalloc_max_workspace_bytes() == 64 << 20
    for seed in seeds:
        q, k, v = make_qkv(shape, torch.bfloat16, seed=seed, device=DEV)
        ref_o, ref_l = cp.ring(q, k, v, R, anything)
        out = torch.empty_like(q)
        lse = torch.empty(shape[:3], device=DEV, dtype=torch.float32)
        assert _call_noalloc(q, k, v, R, anything, out, lse) == 0
        torch.cuda.synchronize()
        assert cp.last_device_status() == 0
        assert (out.float() - ref_o.float()).abs().max().item() <= 1e-2
        assert (lse - ref_l).abs().max().item() <= 1e-3


def test_noalloc_rejects_oversized_workspace():
    # 1 x 24 x 32768 x 128 with ring_degree 8 needs ~406 MB of workspace
    q = torch.empty(1, 24, 32768, 128, device=DEV, dtype=torch.bfloat16)
    out = torch.empty_like(q)
    lse = torch.empty(1, 24, 32768, device=DEV, dtype=torch.float32)
    assert _call_noalloc(q, q, q, 8, False, out, lse) == 7   # CPATTN_ERR_WORKSPACE
