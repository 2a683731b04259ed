"""The workloads at full size, called exactly as bench.py calls them, with
EVERY output element compared against the oracle.

Expected values come from ``oracle/make_cache.py`` (fp64 oracle, stored as
float32 per machine; computed on first use, which takes a few seconds per
FLUX-size case and a few minutes for the video case on the host's cores).
Tolerances: bf16 outputs max-abs 1e-2, fp32 outputs of bf16 inputs 1e-2,
fp32 outputs of fp32 inputs 2e-3, LSE max-abs 1e-3 (N(0, 1) inputs).  The measured whole-tensor errors are
printed at the end of the session.

Fast fallback, for quick checks only: with CPATTN_PARITY=sampled the oracle
recomputes sampled query rows one by one instead (first and last rows, tile
and chunk boundaries, the ragged tail, random rows, several heads and
batches), and every other row is only checked to be finite and inside the
[min, max] of the V column it averages.
"""
import os

import numpy as np
import pytest
import torch

import context_attention_partial_gb300 as cp
import oracle
from oracle import make_cache
from workloads import WORKLOADS, make_workload

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SAMPLED = os.environ.get("CPATTN_PARITY", "full") == "sampled"
TOL_OUT, TOL_LSE = 1e-2, 1e-3


# ----------------------------------------------------------------------------
# whole-tensor comparison
# ----------------------------------------------------------------------------
def full_compare(case, out, lse, parity_report, lse_view=None, tol=(TOL_OUT, TOL_LSE)):
    """max |GPU - oracle| over every element of out and lse (on the GPU)."""
    eo, el = make_cache.expected(case)
    exp_o = torch.from_numpy(np.ascontiguousarray(eo)).to(DEV)
    exp_l = torch.from_numpy(np.ascontiguousarray(el)).to(DEV)
    got_l = lse if lse_view is None else lse_view(lse)
    assert tuple(out.shape) == tuple(exp_o.shape), (case, out.shape, exp_o.shape)
    assert tuple(got_l.shape) == tuple(exp_l.shape), (case, got_l.shape, exp_l.shape)
    assert torch.isfinite(out.float()).all() and torch.isfinite(got_l).all()
    err_o = (out.float() - exp_o).abs().max().item()
    err_l = (got_l.float() - exp_l).abs().max().item()
    parity_report[case] = {"elements": out.numel() + got_l.numel(), "max_abs_out": err_o,
                           "max_abs_lse": err_l, "tol": tuple(tol)}
    assert err_o <= tol[0], (case, err_o)
    assert err_l <= tol[1], (case, err_l)


# ----------------------------------------------------------------------------
# sampled fallback (CPATTN_PARITY=sampled)
# ----------------------------------------------------------------------------
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


def sampled_bhsd(q, k, v, out, lse, causal, heads_to_check):
    """Oracle full attention on sampled rows of [B, H, S, D] tensors."""
    S, D = q.shape[2], q.shape[3]
    check_convex(out, v.to(DEV), dims=2)
    out_c, lse_c = out.cpu(), lse.cpu()
    for i, (b, h) in enumerate(heads_to_check):
        rows = sample_rows(S, i)
        ro, rl = oracle.attention(q[b, h].unsqueeze(0), k[b, h].unsqueeze(0),
                                  v[b, h].unsqueeze(0), D ** -0.5, causal=causal, rows=rows)
        assert np.abs(out_c[b, h, rows].float().numpy() - ro).max() <= TOL_OUT, (b, h)
        assert np.abs(lse_c[b, h, rows].numpy() - rl).max() <= TOL_LSE, (b, h)


def sampled_bshd(q, k, v, out, lse_of_head, heads_to_check):
    """Oracle full attention on sampled rows of [B, S, H, D] tensors;
    lse_of_head(h) gives the GPU's LSE row of head h (batch 0)."""
    S, D = q.shape[1], q.shape[3]
    check_convex(out, v.to(DEV), dims=1)
    out_c = out.cpu()
    for i, h in enumerate(heads_to_check):
        rows = sample_rows(S, i, n_random=12)
        ro, rl = oracle.attention(q[0, rows, h].unsqueeze(0), k[0, :, h].unsqueeze(0),
                                  v[0, :, h].unsqueeze(0), D ** -0.5)
        assert np.abs(out_c[0, rows, h].float().numpy() - ro[0]).max() <= TOL_OUT, h
        assert np.abs(lse_of_head(h)[rows] - rl[0]).max() <= TOL_LSE, h


# ----------------------------------------------------------------------------
# the workloads
# ----------------------------------------------------------------------------
def run_ring(name, heads_to_check, parity_report):
    w, q, k, v = make_workload(name, seed=0)
    gq, gk, gv = q.to(DEV), k.to(DEV), v.to(DEV)
    out, lse = cp.ring(gq, gk, gv, ring_degree=w.ring_degree, ring_anything=w.ring_anything,
                       causal=w.causal)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    assert out.dtype == q.dtype and lse.dtype == torch.float32
    if SAMPLED:
        sampled_bhsd(q, k, v, out, lse, w.causal, heads_to_check)
    else:
        full_compare(name, out, lse, parity_report)


def test_tiny_ring_full(parity_report):
    """The tiny fp32 workload (tf32 tensor cores): output 2e-3, LSE 1e-3."""
    w, q, k, v = make_workload("tiny_ring", seed=0)
    out, lse = cp.ring(q.to(DEV), k.to(DEV), v.to(DEV), ring_degree=w.ring_degree)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    ro, rl = oracle.ring(q, k, v, w.head_dim ** -0.5, ring_degree=w.ring_degree)
    assert out.dtype == torch.float32
    err_o = float(np.abs(out.cpu().numpy() - ro).max())
    err_l = float(np.abs(lse.cpu().numpy() - rl).max())
    parity_report["tiny_ring"] = {"elements": out.numel() + lse.numel(), "max_abs_out": err_o,
                                  "max_abs_lse": err_l, "tol": (2e-3, 1e-3)}
    assert err_o <= 2e-3 and err_l <= 1e-3


def test_flux_ring(parity_report):
    run_ring("flux_ring", [(0, 0), (0, 11), (0, 23)], parity_report)


def test_uneven_ring(parity_report):
    run_ring("uneven_ring", [(0, 0), (1, 7), (1, 23)], parity_report)


def test_flux_ring_causal(parity_report):
    run_ring("flux_ring_causal", [(0, 0), (0, 13), (0, 23)], parity_report)


@pytest.mark.slow
def test_video_ring(parity_report):
    run_ring("video_ring", [(0, 0), (0, 17)], parity_report)


def test_ring_d64_many_waves(parity_report):
    """bf16 at D = 64 (eight K/V stages, 16 KB running-state pieces) over
    864 CTAs, several waves: the final merge's shared-memory prefetch and the
    next wave's Q prefetch run across wave boundaries, ring degree 3."""
    q, k, v = make_cache.inputs("d64_ring")
    out, lse = cp.ring(q.to(DEV), k.to(DEV), v.to(DEV), ring_degree=3)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    if SAMPLED:
        sampled_bhsd(q, k, v, out, lse, False, [(0, 0), (1, 12), (1, 23)])
    else:
        full_compare("d64_ring", out, lse, parity_report)


@pytest.mark.parametrize("case, ring_degree, anything, causal",
                         [("d64_causal", 2, False, True), ("d64_uneven", 3, True, False)])
def test_ring_d64_causal_and_uneven(parity_report, case, ring_degree, anything, causal):
    """bf16 D = 64, whose P has TMEM columns of its own (each query tile's
    next Q K^T goes out before its P V): causal over the FLUX-like length,
    and Ring Anything over 4609 keys in three uneven chunks."""
    q, k, v = make_cache.inputs(case)
    out, lse = cp.ring(q.to(DEV), k.to(DEV), v.to(DEV), ring_degree=ring_degree,
                       ring_anything=anything, causal=causal)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    if SAMPLED:
        sampled_bhsd(q, k, v, out, lse, causal, [(0, 0), (0, 23)])
    else:
        full_compare(case, out, lse, parity_report)


@pytest.mark.parametrize("case, ring_degree, anything, causal",
                         [("f32_d128_ring", 3, True, False), ("f32_d64_causal", 2, False, True)])
def test_ring_f32(parity_report, case, ring_degree, anything, causal):
    """fp32 inputs through the 3xTF32 path, every element against the
    oracle at the fp32 tolerances (output 2e-3, LSE 1e-3): D = 128 runs one
    128-row query tile per CTA against 64-key tiles (4609 rows: 37 CTAs per
    head, the last holding one row; three uneven chunks); D = 64 causal."""
    q, k, v = make_cache.inputs(case)
    out, lse = cp.ring(q.to(DEV), k.to(DEV), v.to(DEV), ring_degree=ring_degree,
                       ring_anything=anything, causal=causal)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    assert out.dtype == torch.float32
    if SAMPLED:
        sampled_bhsd(q, k, v, out, lse, causal, [(0, 0), (0, 7)])
    else:
        full_compare(case, out, lse, parity_report, tol=(2e-3, 1e-3))


def test_partial_flux_shape(parity_report):
    """One partial (cpattn_partial) at the FLUX shape: bf16 inputs, fp32
    output written straight from the epilogue, fp32 LSE; expected: full
    attention over every key (one chunk)."""
    w, q, k, v = make_workload("flux_ring", seed=0)
    out, lse = cp.partial(q.to(DEV), k.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    assert out.dtype == torch.float32 and lse.dtype == torch.float32
    if SAMPLED:
        sampled_bhsd(q, k, v, out, lse, False, [(0, 0), (0, 9), (0, 23)])
    else:
        report = {}
        full_compare("flux_ring", out, lse, report)
        parity_report["flux_partial"] = report["flux_ring"]


def test_ulysses(parity_report):
    w, q, k, v = make_workload("ulysses", seed=0)          # [B, S, H, D]
    out, lse = cp.ulysses_attention(q.to(DEV), k.to(DEV), v.to(DEV), w.ulysses_degree)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    assert out.shape == q.shape and out.dtype == q.dtype
    G, hg = w.ulysses_degree, w.heads // w.ulysses_degree
    if SAMPLED:
        lc = lse.cpu().numpy()                               # [G*B, H/G, S]
        sampled_bshd(q, k, v, out, lambda h: lc[h // hg, h % hg], [0, 5, 6, 13, 23])
    else:
        full_compare("ulysses", out, lse, parity_report,
                     lse_view=lambda l: l.reshape(G, w.batch, hg, w.seq))


def test_unified(parity_report):
    """Unified on the FLUX-like shape (ulysses_degree 2, ring_degree 2)."""
    w, q, k, v = make_workload("unified", seed=0)          # [B, S, H, D]
    out, lse = cp.unified_attention(q.to(DEV), k.to(DEV), v.to(DEV), w.ulysses_degree,
                                    w.ring_degree)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    G, hg = w.ulysses_degree, w.heads // w.ulysses_degree
    if SAMPLED:
        lc = lse.cpu().numpy()
        sampled_bshd(q, k, v, out, lambda h: lc[h // hg, h % hg], [0, 11, 12, 23])
    else:
        full_compare("unified", out, lse, parity_report,
                     lse_view=lambda l: l.reshape(G, w.batch, hg, w.seq))


def test_ulysses_anything(parity_report):
    """Ulysses Anything on the FLUX-like shape, 24 heads over 5 groups
    (5 5 5 5 4, padded to 5 slots); the padding slot's LSE is not compared."""
    w, q, k, v = make_workload("ulysses_anything", seed=0)   # [B, S, H, D]
    out, lse = cp.ulysses_anything_attention(q.to(DEV), k.to(DEV), v.to(DEV), w.ulysses_degree)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    start = oracle.ulysses_anything_heads(w.heads, w.ulysses_degree)
    if SAMPLED:
        lc = lse.cpu().numpy()                                 # [G, B, hm, S]

        def lse_of_head(h):
            g = max(j for j in range(w.ulysses_degree) if start[j] <= h)
            return lc[g, 0, h - start[g]]
        sampled_bshd(q, k, v, out, lse_of_head, [0, 4, 5, 14, 15, 19, 20, 23])
        return
    eo, el = make_cache.expected("ulysses_anything")
    exp_o = torch.from_numpy(np.ascontiguousarray(eo)).to(DEV)
    assert torch.isfinite(out.float()).all()
    err_o = (out.float() - exp_o).abs().max().item()
    err_l, n_l = 0.0, 0
    el = np.asarray(el)
    for g in range(w.ulysses_degree):
        hg = start[g + 1] - start[g]
        got = lse[g, :, :hg]
        exp_l = torch.from_numpy(np.ascontiguousarray(el[g, :, :hg])).to(DEV)
        assert torch.isfinite(got).all()
        err_l = max(err_l, (got - exp_l).abs().max().item())
        n_l += got.numel()
    parity_report["ulysses_anything"] = {"elements": out.numel() + n_l, "max_abs_out": err_o,
                                         "max_abs_lse": err_l, "tol": (TOL_OUT, TOL_LSE)}
    assert err_o <= TOL_OUT and err_l <= TOL_LSE, (err_o, err_l)


def test_workload_table_flops():
    assert abs(WORKLOADS["flux_ring"].flops / 1e9 - 260.92) < 0.01
    assert abs(WORKLOADS["uneven_ring"].flops / 1e9 - 522.07) < 0.01
    assert abs(WORKLOADS["video_ring"].flops / 1e9 - 13194.1) < 0.1
