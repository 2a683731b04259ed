"""The workloads at full size, called exactly as bench.py calls them.

The oracle recomputes sampled query rows one by one (first and last rows,
tile and chunk boundaries, the ragged tail, random rows, several heads and
batches); every output row is also checked against properties that hold at
any size: finite values, and each output coordinate inside the [min, max]
of the V column it averages (a softmax-weighted mean).
"""
import numpy as np
import pytest
import torch

import context_attention_partial_gb300 as cp
import oracle
from context_attention_partial_gb300.workloads import WORKLOADS, make_qkv, make_workload

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def sample_rows(s, extra_seed=0, n_random=24):
    rows = {0, 1, 127, 128, 129, 255, 256, s // 2, s - 129, s - 128, s - 2, s - 1}
    rng = np.random.default_rng(1000 + extra_seed)
    rows |= set(int(r) for r in rng.integers(0, s, size=n_random))
    return sorted(r for r in rows if 0 <= r < s)


def check_convex(out, v, dims):
    """out[..., d] lies within [min_j v[j, d], max_j v[j, d]] (+ bf16 slack)."""
    vmin = v.float().amin(dim=dims, keepdim=True)
    vmax = v.float().amax(dim=dims, keepdim=True)
    o = out.float()
    slack = 1e-2
    assert torch.isfinite(o).all()
    assert bool((o >= vmin - slack).all()) and bool((o <= vmax + slack).all())


def check_ring_sampled(name, q, k, v, ring_degree, ring_anything, causal, heads_to_check):
    """cp.ring on q, k, v [B, H, S, D] against the oracle on sampled rows."""
    S, D = q.shape[2], q.shape[3]
    gq, gk, gv = q.to(DEV), k.to(DEV), v.to(DEV)
    out, lse = cp.ring(gq, gk, gv, ring_degree=ring_degree, ring_anything=ring_anything,
                       causal=causal)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    assert out.dtype == q.dtype and lse.dtype == torch.float32
    assert torch.isfinite(lse).all()
    check_convex(out, gv, dims=2)
    tol_o, tol_l = (2e-3, 1e-3) if q.dtype == torch.float32 else (1e-2, 1e-3)
    out_c, lse_c = out.cpu(), lse.cpu()
    for i, (b, h) in enumerate(heads_to_check):
        rows = sample_rows(S, i)
        if causal:
            # causal rows depend on their position: evaluate whole-sequence rows
            ro, rl = oracle.ring(q[b, h].unsqueeze(0), k[b, h].unsqueeze(0), v[b, h].unsqueeze(0),
                                 D ** -0.5, ring_degree=ring_degree,
                                 ring_anything=ring_anything, causal=True, rows=rows)
            ro, rl = ro[None], rl[None]
        else:
            ro, rl = oracle.ring(q[b, h, rows].unsqueeze(0), k[b, h].unsqueeze(0),
                                 v[b, h].unsqueeze(0), D ** -0.5,
                                 ring_degree=ring_degree, ring_anything=ring_anything)
        go = out_c[b, h, rows].float().numpy()
        gl = lse_c[b, h, rows].numpy()
        assert np.abs(go - ro[0]).max() <= tol_o, (name, b, h)
        assert np.abs(gl - rl[0]).max() <= tol_l, (name, b, h)


def run_ring_workload(name, heads_to_check):
    w, q, k, v = make_workload(name, seed=0)
    check_ring_sampled(name, q, k, v, w.ring_degree, w.ring_anything, w.causal, heads_to_check)


def test_tiny_ring_full():
    w, q, k, v = make_workload("tiny_ring", seed=0)
    out, lse = cp.ring(q.to(DEV), k.to(DEV), v.to(DEV), ring_degree=w.ring_degree)
    torch.cuda.synchronize()
    ro, rl = oracle.ring(q, k, v, w.head_dim ** -0.5, ring_degree=w.ring_degree)
    assert out.dtype == torch.float32
    assert np.abs(out.cpu().numpy() - ro).max() <= 2e-3
    assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-3


def test_flux_ring_sampled():
    run_ring_workload("flux_ring", [(0, 0), (0, 11), (0, 23)])


def test_uneven_ring_sampled():
    run_ring_workload("uneven_ring", [(0, 0), (1, 7), (1, 23)])


def test_flux_ring_causal_sampled():
    run_ring_workload("flux_ring_causal", [(0, 0), (0, 13), (0, 23)])


def test_ring_d64_many_waves_sampled():
    """bf16 at D = 64 (eight K/V stages, 16 KB running-state pieces) over
    864 CTAs, several waves: the final merge's shared-memory prefetch and the
    next wave's Q prefetch run across wave boundaries, ring degree 3."""
    q, k, v = make_qkv((2, 24, 4608, 64), torch.bfloat16, seed=61)
    check_ring_sampled("d64", q, k, v, 3, False, False, [(0, 0), (1, 12), (1, 23)])


def test_partial_flux_shape_sampled():
    """One partial (cpattn_partial) at the FLUX shape: bf16 inputs, fp32
    output written straight from the epilogue, fp32 LSE."""
    w, q, k, v = make_workload("flux_ring", seed=0)
    gv = v.to(DEV)
    out, lse = cp.partial(q.to(DEV), k.to(DEV), gv)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    assert out.dtype == torch.float32 and lse.dtype == torch.float32
    assert torch.isfinite(lse).all()
    check_convex(out, gv, dims=2)
    out_c, lse_c = out.cpu(), lse.cpu()
    for i, (b, h) in enumerate([(0, 0), (0, 9), (0, 23)]):
        rows = sample_rows(w.seq, 50 + i)
        ro, rl = oracle.partial(q[b, h, rows].unsqueeze(0), k[b, h].unsqueeze(0),
                                v[b, h].unsqueeze(0), w.head_dim ** -0.5)
        assert np.abs(out_c[b, h, rows].numpy() - ro[0]).max() <= 1e-2, (b, h)
        assert np.abs(lse_c[b, h, rows].numpy() - rl[0]).max() <= 1e-3, (b, h)


@pytest.mark.slow
def test_video_ring_sampled():
    run_ring_workload("video_ring", [(0, 0), (0, 17)])


def test_ulysses_sampled():
    w, q, k, v = make_workload("ulysses", seed=0)          # [B, S, H, D]
    gq, gk, gv = q.to(DEV), k.to(DEV), v.to(DEV)
    out, lse = cp.ulysses_attention(gq, gk, gv, w.ulysses_degree)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    assert out.shape == q.shape and out.dtype == q.dtype
    check_convex(out, gv, dims=1)
    out_c = out.cpu()
    lse_c = lse.cpu()                                         # [G*B, H/G, S]
    hg = w.heads // w.ulysses_degree
    for i, h in enumerate([0, 5, 6, 13, 23]):
        rows = sample_rows(w.seq, i, n_random=12)
        qs = q[0, rows, h].unsqueeze(0)
        ro, rl = oracle.attention(qs, k[0, :, h].unsqueeze(0), v[0, :, h].unsqueeze(0),
                                  w.head_dim ** -0.5)
        assert np.abs(out_c[0, rows, h].float().numpy() - ro[0]).max() <= 1e-2
        assert np.abs(lse_c[h // hg, h % hg, rows].numpy() - rl[0]).max() <= 1e-3


def test_unified_sampled():
    """Unified on the FLUX-like shape (ulysses_degree 2, ring_degree 2): each
    head's rows equal the ring schedule over that head's full sequence."""
    w, q, k, v = make_workload("unified", seed=0)          # [B, S, H, D]
    out, lse = cp.unified_attention(q.to(DEV), k.to(DEV), v.to(DEV), w.ulysses_degree,
                                    w.ring_degree)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    check_convex(out, v.to(DEV), dims=1)
    out_c, lse_c = out.cpu(), lse.cpu()
    hg = w.heads // w.ulysses_degree
    for i, h in enumerate([0, 11, 12, 23]):
        rows = sample_rows(w.seq, i, n_random=12)
        ro, rl = oracle.ring(q[0, rows, h].unsqueeze(0), k[0, :, h].unsqueeze(0),
                             v[0, :, h].unsqueeze(0), w.head_dim ** -0.5,
                             ring_degree=w.ring_degree)
        assert np.abs(out_c[0, rows, h].float().numpy() - ro[0]).max() <= 1e-2
        assert np.abs(lse_c[h // hg, h % hg, rows].numpy() - rl[0]).max() <= 1e-3


def test_ulysses_anything_sampled():
    """Ulysses Anything on the FLUX-like shape, 24 heads over 5 groups
    (5 5 5 5 4): each head's rows equal attention over that head's full
    sequence; heads on both sides of every group boundary are checked."""
    w, q, k, v = make_workload("ulysses_anything", seed=0)   # [B, S, H, D]
    out, lse = cp.ulysses_anything_attention(q.to(DEV), k.to(DEV), v.to(DEV), w.ulysses_degree)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    check_convex(out, v.to(DEV), dims=1)
    out_c, lse_c = out.cpu(), lse.cpu()
    start = oracle.ulysses_anything_heads(w.heads, w.ulysses_degree)
    for i, h in enumerate([0, 4, 5, 14, 15, 19, 20, 23]):
        g = max(j for j in range(w.ulysses_degree) if start[j] <= h)
        rows = sample_rows(w.seq, i, n_random=12)
        ro, rl = oracle.attention(q[0, rows, h].unsqueeze(0), k[0, :, h].unsqueeze(0),
                                  v[0, :, h].unsqueeze(0), w.head_dim ** -0.5)
        assert np.abs(out_c[0, rows, h].float().numpy() - ro[0]).max() <= 1e-2, h
        assert np.abs(lse_c[g, 0, h - start[g], rows].numpy() - rl[0]).max() <= 1e-3, h


def test_workload_table_flops():
    assert abs(WORKLOADS["flux_ring"].flops / 1e9 - 260.92) < 0.01
    assert abs(WORKLOADS["uneven_ring"].flops / 1e9 - 522.07) < 0.01
    assert abs(WORKLOADS["video_ring"].flops / 1e9 - 13194.1) < 0.1
