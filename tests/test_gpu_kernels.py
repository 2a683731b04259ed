"""GPU parity of every kernel against the fp64 oracle on seeded inputs, at
sizes the oracle finishes in seconds that still span several tiles and a
ragged tail, plus the degenerate cases.

Tolerances: bf16 inputs -> output max-abs 1e-2, LSE max-abs 1e-3 (N(0,1)
inputs); fp32 inputs (tf32 tensor cores) -> output 2e-3, LSE 1e-3; the merge
(pure fp32 arithmetic) -> 2e-5 relative to the magnitudes involved; the
permute -> bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import context_attention_partial_gb300 as cp
import oracle
from workloads import make_partials, make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = {torch.bfloat16: (1e-2, 1e-3), torch.float32: (2e-3, 1e-3)}


def maxabs(a, b):
    a = a.detach().float().cpu().numpy() if hasattr(a, "detach") else np.asarray(a)
    return float(np.max(np.abs(a - b))) if np.size(b) else 0.0


def status_ok():
    assert cp.last_device_status() == 0


# ----------------------------------------------------------------------------
# Ulysses permute: bit-exact
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("shape,g,dtype", [
    ((1, 4608, 24, 128), 4, torch.bfloat16),      # the Ulysses workload's tensors
    ((2, 37, 12, 64), 3, torch.bfloat16),
    ((1, 5, 6, 8), 2, torch.float32),
    ((2, 3, 10, 3), 5, torch.bfloat16),           # 12-byte segments: element path
    ((1, 9, 7, 5), 7, torch.float32),             # 20-byte segments
    ((2, 17, 8, 128), 1, torch.bfloat16),         # G = 1 is the identity layout
])
def test_permute_bit_exact(shape, g, dtype):
    x = make_qkv(shape, dtype, seed=3)[0]
    y = cp.ulysses_permute(x.to(DEV), g, 1)
    torch.cuda.synchronize()
    ref = oracle.ulysses_permute(x, g, 1)
    assert tuple(y.shape) == tuple(ref.shape)
    assert torch.equal(y.cpu(), ref)
    back = cp.ulysses_permute(y, g, -1)
    torch.cuda.synchronize()
    assert torch.equal(back.cpu(), x)
    assert torch.equal(back.cpu(), oracle.ulysses_permute(ref, g, -1))


@pytest.mark.parametrize("shape,g,dtype,n", [
    ((1, 4608, 24, 128), 4, torch.bfloat16, 3),   # q, k, v of the Ulysses workload
    ((2, 37, 12, 64), 3, torch.bfloat16, 2),
    ((2, 3, 10, 3), 5, torch.bfloat16, 4),        # element path, the most tensors
    ((1, 9, 7, 5), 7, torch.float32, 1),
])
def test_permute_batch_bit_exact(shape, g, dtype, n):
    """n regroups in one launch equal n single regroups and the oracle."""
    xs = [make_qkv(shape, dtype, seed=70 + i)[0] for i in range(n)]
    ys = cp.ulysses_permute_batch([x.to(DEV) for x in xs], g, 1)
    torch.cuda.synchronize()
    for x, y in zip(xs, ys):
        assert torch.equal(y.cpu(), oracle.ulysses_permute(x, g, 1))
    backs = cp.ulysses_permute_batch(ys, g, -1)
    torch.cuda.synchronize()
    for x, back in zip(xs, backs):
        assert torch.equal(back.cpu(), x)


@pytest.mark.parametrize("shape,g,dtype,n", [
    ((1, 4608, 24, 128), 5, torch.bfloat16, 3),   # q, k, v of the Ulysses Anything workload
    ((2, 37, 7, 64), 3, torch.bfloat16, 2),
    ((2, 3, 5, 3), 2, torch.bfloat16, 4),         # element path
    ((1, 9, 2, 5), 4, torch.float32, 3),          # H < G
])
def test_anything_permute_batch_bit_exact(shape, g, dtype, n):
    xs = [make_qkv(shape, dtype, seed=80 + i)[0] for i in range(n)]
    H = shape[2]
    hm = -(-H // g)
    outs = [torch.full((g,) + shape[:2] + (hm, shape[3]), -3.0, dtype=dtype, device=DEV)
            for _ in range(n)]
    ys = cp.ulysses_anything_permute_batch([x.to(DEV) for x in xs], g, 1, outs=outs)
    torch.cuda.synchronize()
    start = oracle.ulysses_anything_heads(H, g)
    for x, y in zip(xs, ys):
        ref = oracle.ulysses_anything_permute(x, g, 1)
        yc = y.cpu()
        for gi in range(g):
            hg = start[gi + 1] - start[gi]
            assert torch.equal(yc[gi, :, :, :hg], ref[gi, :, :, :hg])
            assert torch.all(yc[gi, :, :, hg:] == -3.0)        # padding not written
    backs = cp.ulysses_anything_permute_batch(ys, g, -1, heads=H)
    torch.cuda.synchronize()
    for x, back in zip(xs, backs):
        assert torch.equal(back.cpu(), x)


def test_permute_rejects_indivisible_heads():
    x = torch.zeros(1, 4, 6, 8, device=DEV, dtype=torch.bfloat16)
    with pytest.raises(cp.CpattnError) as e:
        cp.ulysses_permute(x, 4, 1, out=torch.zeros(4, 1, 4, 1, 8, device=DEV, dtype=torch.bfloat16))
    assert e.value.name == "CPATTN_ERR_DIVISIBILITY"


# ----------------------------------------------------------------------------
# merge
# ----------------------------------------------------------------------------
def _merge_check(o_a, l_a, o_b, l_b, ga, gla):
    ro, rl = oracle.merge(o_a, l_a, o_b, l_b)
    scale = max(1.0, float(np.abs(o_a.numpy()).max()), float(np.abs(o_b.numpy()).max()))
    assert maxabs(ga, ro) <= 2e-5 * scale
    fin = np.isfinite(rl)
    g = gla.cpu().numpy()
    assert np.array_equal(np.isfinite(g), fin)
    assert np.max(np.abs(g[fin] - rl[fin]), initial=0.0) <= 2e-5 * max(1.0, np.abs(rl[fin]).max())
    assert np.all(g[~fin] == -np.inf)


@pytest.mark.parametrize("shape", [(1, 24, 4608, 128), (2, 3, 77, 64), (1, 1, 5, 4)])
def test_merge_matches_oracle(shape):
    o_a, l_a, o_b, l_b = make_partials(shape[:3], shape[3], seed=5)
    # empty partials: one side, the other side, both sides
    l_a[..., 0] = -math.inf
    if shape[2] > 2:
        l_b[..., 1] = -math.inf
        l_a[..., 2] = -math.inf
        l_b[..., 2] = -math.inf
        o_a[..., 2, :] = 0
        o_b[..., 2, :] = 0
    o_a[..., 0, :] = 0
    ga, gla = o_a.to(DEV), l_a.to(DEV)
    cp.merge(ga, gla, o_b.to(DEV), l_b.to(DEV))
    torch.cuda.synchronize()
    _merge_check(o_a, l_a, o_b, l_b, ga, gla)


def test_merge_strided_views():
    o_a, l_a, o_b, l_b = make_partials((2, 3, 40), 64, seed=6)
    big = torch.zeros(2, 3, 50, 64)
    big[:, :, 5:45] = o_a
    gbig = big.to(DEV)
    ga = gbig[:, :, 5:45]
    glbig = torch.zeros(2, 3, 50).to(DEV)
    glbig[:, :, 5:45] = l_a.to(DEV)
    gla = glbig[:, :, 5:45]
    cp.merge(ga, gla, o_b.to(DEV), l_b.to(DEV))
    torch.cuda.synchronize()
    _merge_check(o_a, l_a, o_b, l_b, ga, gla)
    assert torch.all(gbig[:, :, :5] == 0) and torch.all(gbig[:, :, 45:] == 0)


def test_merge_identity_and_self():
    o_a, l_a, _, _ = make_partials((1, 2, 33), 128, seed=7)
    ga, gla = o_a.to(DEV), l_a.to(DEV)
    cp.merge(ga, gla, torch.zeros_like(ga), torch.full_like(gla, -math.inf))
    torch.cuda.synchronize()
    assert torch.equal(ga.cpu(), o_a) and torch.equal(gla.cpu(), l_a)
    cp.merge(ga, gla, o_a.to(DEV), l_a.to(DEV))
    torch.cuda.synchronize()
    assert maxabs(ga, o_a.numpy()) <= 1e-6 * 4
    assert maxabs(gla, l_a.numpy() + math.log(2)) <= 1e-5


# ----------------------------------------------------------------------------
# partial (one chunk) and ring (chunk loop + merges in one kernel)
# ----------------------------------------------------------------------------
PARTIAL_CASES = [
    # (B, H, S_q, S_kv, D, dtype)
    (1, 2, 300, 333, 128, torch.bfloat16),
    (2, 3, 1, 1, 128, torch.bfloat16),
    (1, 2, 256, 128, 128, torch.bfloat16),
    (1, 1, 513, 700, 64, torch.bfloat16),
    (1, 2, 200, 257, 64, torch.float32),
    (1, 2, 200, 257, 128, torch.float32),         # fp32 D = 128: one query tile, 64-key tiles
    (2, 3, 1, 1, 128, torch.float32),
]


@pytest.mark.parametrize("case", PARTIAL_CASES, ids=lambda c: "x".join(map(str, c[:5])) + str(c[5])[-4:])
def test_partial_matches_oracle(case):
    B, H, Sq, Skv, D, dt = case
    g = torch.Generator("cpu").manual_seed(11)
    q = torch.randn(B, H, Sq, D, generator=g).to(dt)
    k = torch.randn(B, H, Skv, D, generator=g).to(dt)
    v = torch.randn(B, H, Skv, D, generator=g).to(dt)
    out, lse = cp.partial(q.to(DEV), k.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    status_ok()
    ro, rl = oracle.partial(q, k, v, D ** -0.5)
    to, tl = TOL[dt]
    assert out.dtype == torch.float32
    assert maxabs(out, ro) <= to
    assert maxabs(lse, rl) <= tl


RING_CASES = [
    # (B, H, S_q, S_kv, D, dtype, R, anything)
    (1, 2, 300, 300, 128, torch.bfloat16, 3, False),
    (1, 2, 300, 301, 128, torch.bfloat16, 3, True),      # 101/100/100
    (2, 2, 129, 1000, 128, torch.bfloat16, 5, False),
    (1, 3, 256, 256, 64, torch.bfloat16, 4, False),
    (1, 1, 77, 13, 128, torch.bfloat16, 13, True),       # one key per chunk
    (1, 2, 256, 256, 64, torch.float32, 4, False),       # the tiny workload's layout
    (1, 1, 130, 390, 64, torch.float32, 2, False),
    (1, 2, 64, 1024, 128, torch.bfloat16, 1, False),
    (1, 2, 256, 256, 128, torch.float32, 4, False),      # fp32 D = 128
    (1, 1, 130, 391, 128, torch.float32, 3, True),       # 131/130/130, ragged 64-key tiles
    (1, 24, 1030, 1030, 128, torch.float32, 2, False),   # 216 CTAs: more than one wave
]


@pytest.mark.parametrize("case", RING_CASES, ids=lambda c: "x".join(map(str, c[:5])) + f"R{c[6]}{'a' if c[7] else ''}{str(c[5])[-4:]}")
def test_ring_matches_oracle(case):
    B, H, Sq, Skv, D, dt, R, anything = case
    g = torch.Generator("cpu").manual_seed(13)
    q = torch.randn(B, H, Sq, D, generator=g).to(dt)
    k = torch.randn(B, H, Skv, D, generator=g).to(dt)
    v = torch.randn(B, H, Skv, D, generator=g).to(dt)
    out, lse = cp.ring(q.to(DEV), k.to(DEV), v.to(DEV), ring_degree=R, ring_anything=anything)
    torch.cuda.synchronize()
    status_ok()
    ro, rl = oracle.ring(q, k, v, D ** -0.5, ring_degree=R, ring_anything=anything)
    to, tl = TOL[dt]
    assert out.dtype == dt
    assert maxabs(out, ro) <= to
    assert maxabs(lse, rl) <= tl


@pytest.mark.parametrize("d,causal", [(128, False), (64, False), (64, True)])
def test_ring_large_scores_exercise_rescale(d, causal):
    """Scores with std ~12 make the running max grow by more than 2^8
    between key tiles, so the in-TMEM output rescale runs (at D = 64 after
    the wait for the tile's previous P V, P having TMEM of its own).  These
    inputs are not N(0, 1): the softmax is peaked, outputs reach |v| ~ 4, so
    the bound is the bf16 half-ulp at [2, 4) (2^-7) plus P's bf16 rounding
    (2^-9 relative) times max |v| (~4): 2e-2."""
    g = torch.Generator("cpu").manual_seed(17)
    sq = 1024 if causal else 256
    q = (torch.randn(1, 2, sq, d, generator=g) * 12).to(torch.bfloat16)
    k = torch.randn(1, 2, 1024, d, generator=g).to(torch.bfloat16)
    v = torch.randn(1, 2, 1024, d, generator=g).to(torch.bfloat16)
    out, lse = cp.ring(q.to(DEV), k.to(DEV), v.to(DEV), ring_degree=2, causal=causal)
    torch.cuda.synchronize()
    status_ok()
    ro, rl = oracle.ring(q, k, v, d ** -0.5, ring_degree=2, causal=causal)
    assert maxabs(out, ro) <= 2e-2
    # the LSE bound stays the stated 1e-3 absolute: the scores are exact
    # products of bf16 values summed in fp32 (error ~1e-5 at |lse| ~ 40)
    assert maxabs(lse, rl) <= 1e-3


def test_ring_closed_forms():
    g = torch.Generator("cpu").manual_seed(19)
    k = torch.randn(1, 2, 300, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(1, 2, 300, 128, generator=g).to(torch.bfloat16)
    q0 = torch.zeros(1, 2, 40, 128, dtype=torch.bfloat16)
    out, lse = cp.ring(q0.to(DEV), k.to(DEV), v.to(DEV), ring_degree=3)
    torch.cuda.synchronize()
    mean_v = v.double().mean(dim=2, keepdim=True).expand(1, 2, 40, 128).numpy()
    assert maxabs(out, mean_v) <= 1e-2
    assert maxabs(lse, np.full((1, 2, 40), math.log(300))) <= 1e-3
    c = torch.randn(1, 1, 1, 128, generator=g).to(torch.bfloat16).expand(1, 2, 300, 128).contiguous()
    q = torch.randn(1, 2, 40, 128, generator=g).to(torch.bfloat16)
    out, _ = cp.ring(q.to(DEV), k.to(DEV), c.to(DEV), ring_degree=2)
    torch.cuda.synchronize()
    assert maxabs(out, c[:, :, :40].double().numpy()) <= 1e-2


def test_ring_strided_bshd_inputs_equal_contiguous():
    g = torch.Generator("cpu").manual_seed(23)
    x = [torch.randn(1, 300, 4, 128, generator=g).to(torch.bfloat16).to(DEV) for _ in range(3)]
    views = [t.permute(0, 2, 1, 3) for t in x]           # [B, H, S, D] with stride H*D per token
    dense = [t.contiguous() for t in views]
    o1, l1 = cp.ring(*views, ring_degree=2)
    o2, l2 = cp.ring(*dense, ring_degree=2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_ring_empty_query_is_noop():
    k = torch.randn(1, 2, 64, 128, device=DEV).to(torch.bfloat16)
    q = torch.empty(1, 2, 0, 128, device=DEV, dtype=torch.bfloat16)
    out, lse = cp.ring(q, k, k, ring_degree=2)
    torch.cuda.synchronize()
    assert out.shape == (1, 2, 0, 128) and lse.shape == (1, 2, 0)


def test_ring_is_deterministic():
    q, k, v = make_qkv((1, 4, 700, 128), torch.bfloat16, seed=29, device=DEV)
    a = cp.ring(q, k, v, ring_degree=2)
    b = cp.ring(q, k, v, ring_degree=2)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("b,s,h,d,g,r,dt", [
    (1, 300, 8, 128, 2, 3, torch.bfloat16),
    (2, 256, 6, 64, 3, 2, torch.bfloat16),
    (1, 256, 4, 64, 2, 4, torch.float32),
    (1, 130, 4, 128, 4, 1, torch.bfloat16),
    (1, 256, 4, 128, 2, 2, torch.float32),
])
def test_unified_matches_oracle(b, s, h, d, g, r, dt):
    """Unified (Ulysses x Ring): regroup, ring inside each head group,
    inverse regroup -- against the oracle's composition of the same steps."""
    q, k, v = make_qkv((b, s, h, d), dt, seed=37)
    out, lse = cp.unified_attention(q.to(DEV), k.to(DEV), v.to(DEV), g, r)
    torch.cuda.synchronize()
    status_ok()
    ro, rl = oracle.unified(q, k, v, g, r, d ** -0.5)
    to, tl = TOL[dt]
    assert out.shape == q.shape and out.dtype == dt
    assert maxabs(out, ro) <= to
    assert maxabs(lse.reshape(g, b, h // g, s), rl) <= tl


CAUSAL_CASES = [
    # (B, H, S_q, S_kv, D, dtype, R, anything)
    (1, 2, 300, 300, 128, torch.bfloat16, 3, False),
    (1, 2, 301, 301, 128, torch.bfloat16, 3, True),      # 101/100/100
    (2, 2, 129, 1000, 128, torch.bfloat16, 5, False),    # S_q < S_kv: top-left aligned
    (1, 3, 256, 256, 64, torch.bfloat16, 4, False),
    (1, 2, 513, 513, 128, torch.bfloat16, 5, True),
    (1, 1, 700, 700, 128, torch.bfloat16, 1, False),
    (1, 2, 256, 256, 64, torch.float32, 4, False),
    (1, 1, 77, 13, 128, torch.bfloat16, 13, True),
    (1, 2, 300, 300, 128, torch.float32, 3, False),
]


@pytest.mark.parametrize("case", CAUSAL_CASES, ids=lambda c: "x".join(map(str, c[:5])) + f"R{c[6]}{'a' if c[7] else ''}{str(c[5])[-4:]}")
def test_ring_causal_matches_oracle(case):
    B, H, Sq, Skv, D, dt, R, anything = case
    g = torch.Generator("cpu").manual_seed(41)
    q = torch.randn(B, H, Sq, D, generator=g).to(dt)
    k = torch.randn(B, H, Skv, D, generator=g).to(dt)
    v = torch.randn(B, H, Skv, D, generator=g).to(dt)
    out, lse = cp.ring(q.to(DEV), k.to(DEV), v.to(DEV), ring_degree=R, ring_anything=anything,
                       causal=True)
    torch.cuda.synchronize()
    status_ok()
    ro, rl = oracle.ring(q, k, v, D ** -0.5, ring_degree=R, ring_anything=anything, causal=True)
    to, tl = TOL[dt]
    assert maxabs(out, ro) <= to
    assert maxabs(lse, rl) <= tl


def test_unified_causal_matches_oracle():
    q, k, v = make_qkv((1, 300, 8, 128), torch.bfloat16, seed=43)
    out, lse = cp.unified_attention(q.to(DEV), k.to(DEV), v.to(DEV), 2, 3, causal=True)
    torch.cuda.synchronize()
    ro, rl = oracle.unified(q, k, v, 2, 3, 128 ** -0.5, causal=True)
    assert maxabs(out, ro) <= 1e-2
    assert maxabs(lse.reshape(2, 1, 4, 300), rl) <= 1e-3


# ----------------------------------------------------------------------------
# Ulysses Anything: uneven head groups padded to ceil(H/G) slots
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("shape,g,dtype", [
    ((1, 4608, 24, 128), 5, torch.bfloat16),      # the Ulysses Anything workload's tensors
    ((1, 4608, 24, 128), 7, torch.bfloat16),      # groups 4 4 4 3 3 3 3
    ((2, 37, 7, 64), 3, torch.bfloat16),
    ((1, 5, 6, 8), 4, torch.float32),             # groups 2 2 1 1
    ((2, 3, 5, 3), 2, torch.bfloat16),            # 6-byte head rows: element path
    ((1, 9, 2, 5), 4, torch.float32),             # H < G: two groups hold no head
    ((2, 17, 8, 128), 4, torch.bfloat16),         # H % G == 0: plain Ulysses layout
])
def test_anything_permute_bit_exact(shape, g, dtype):
    x = make_qkv(shape, dtype, seed=5)[0]
    H = shape[2]
    hm = -(-H // g)
    sentinel = torch.full((g,) + shape[:2] + (hm, shape[3]), -3.0, dtype=dtype, device=DEV)
    y = cp.ulysses_anything_permute(x.to(DEV), g, 1, out=sentinel)
    torch.cuda.synchronize()
    ref = oracle.ulysses_anything_permute(x, g, 1)
    start = oracle.ulysses_anything_heads(H, g)
    yc = y.cpu()
    for gi in range(g):
        hg = start[gi + 1] - start[gi]
        assert torch.equal(yc[gi, :, :, :hg], ref[gi, :, :, :hg])
        assert torch.all(yc[gi, :, :, hg:] == -3.0)            # padding not written
    if H % g == 0:
        assert torch.equal(yc, oracle.ulysses_permute(x, g, 1))
    # the inverse does not read the padding: poison it first
    for gi in range(g):
        y[gi, :, :, start[gi + 1] - start[gi]:] = float("nan")
    back = cp.ulysses_anything_permute(y, g, -1, heads=H)
    torch.cuda.synchronize()
    assert torch.equal(back.cpu(), x)


@pytest.mark.parametrize("b,s,h,d,g,dt,causal", [
    (1, 300, 5, 128, 2, torch.bfloat16, False),    # groups 3 2
    (2, 257, 7, 64, 3, torch.bfloat16, False),     # groups 3 2 2
    (1, 256, 5, 64, 3, torch.float32, False),      # fp32 (3xTF32)
    (1, 200, 5, 128, 3, torch.float32, False),     # fp32, D = 128
    (1, 200, 2, 128, 4, torch.bfloat16, False),    # H < G
    (1, 300, 7, 128, 4, torch.bfloat16, True),     # causal, groups 2 2 2 1
    (1, 130, 8, 128, 4, torch.bfloat16, False),    # even split
])
def test_ulysses_anything_matches_oracle(b, s, h, d, g, dt, causal):
    q, k, v = make_qkv((b, s, h, d), dt, seed=47)
    out, lse = cp.ulysses_anything_attention(q.to(DEV), k.to(DEV), v.to(DEV), g, causal=causal)
    torch.cuda.synchronize()
    status_ok()
    ro, rl = oracle.ulysses_anything(q, k, v, g, d ** -0.5, causal=causal)
    to, tl = TOL[dt]
    assert out.shape == q.shape and out.dtype == dt
    assert maxabs(out, ro) <= to
    start = oracle.ulysses_anything_heads(h, g)
    lc = lse.cpu().numpy()
    for gi in range(g):
        hg = start[gi + 1] - start[gi]
        if hg:
            assert float(np.max(np.abs(lc[gi, :, :hg] - rl[gi, :, :hg]))) <= tl


def test_ulysses_anything_leaves_padding_slots_alone():
    """The attention launch skips padding head slots: out and lse keep what
    the caller put there."""
    b, s, h, d, g = 1, 256, 5, 128, 3                     # groups 2 2 1, 2 slots
    q, k, v = (x.to(DEV) for x in make_qkv((b, s, h, d), torch.bfloat16, seed=53))
    qg, kg, vg = (cp.ulysses_anything_permute(x, g, 1) for x in (q, k, v))
    og = torch.full_like(qg, 7.0)
    lse = torch.full((g, b, 2, s), 9.0, device=DEV)
    lib = cp.load_library()
    from context_attention_partial_gb300 import api
    rc = lib.cpattn_ulysses_anything_attention(api._desc(qg), api._desc(kg), api._desc(vg), 0.0, h,
                                               0, api._desc(og), api._desc(lse),
                                               torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    status_ok()
    assert torch.all(og[2, :, :, 1] == 7.0) and torch.all(lse[2, :, 1] == 9.0)
    assert torch.all(torch.isfinite(og[:2].float())) and not torch.any(lse[:2] == 9.0)


def test_prepared_calls_equal_plain_calls():
    """prepare_ring / prepare_unified / prepare_ulysses_anything issue the
    same library calls with descriptors built once: bit-equal results."""
    q, k, v = make_qkv((1, 3, 300, 128), torch.bfloat16, seed=59, device=DEV)
    ref = cp.ring(q, k, v, 3, causal=True)
    call = cp.prepare_ring(q, k, v, 3, causal=True)
    call()
    call()
    torch.cuda.synchronize()
    status_ok()
    assert torch.equal(call.out, ref[0]) and torch.equal(call.lse, ref[1])
    x = make_qkv((1, 258, 6, 64), torch.bfloat16, seed=61, device=DEV)
    ref = cp.unified_attention(*x, 2, 2)
    call = cp.prepare_unified(*x, 2, 2)
    call()
    torch.cuda.synchronize()
    assert torch.equal(call.out, ref[0]) and torch.equal(call.lse, ref[1])
    ref = cp.ulysses_anything_attention(*x, 4)
    call = cp.prepare_ulysses_anything(*x, 4)
    call()
    torch.cuda.synchronize()
    assert torch.equal(call.out, ref[0])
    start = oracle.ulysses_anything_heads(6, 4)
    for g in range(4):
        hg = start[g + 1] - start[g]
        assert torch.equal(call.lse[g, :, :hg], ref[1][g, :, :hg])


@pytest.mark.parametrize("skv,anything,causal", [
    (200, True, False),      # 64 chunks of 3 or 4 keys (Ring Anything)
    (128, False, False),     # 64 chunks of 2 keys
    (200, True, True),       # causal: most chunks past a tile's rows are skipped
])
def test_ring_at_the_maximum_ring_degree(skv, anything, causal):
    """ring_degree = CPATTN_MAX_RING_DEGREE (64): the chunk table at its
    largest, 63 in-kernel merges per query row."""
    g = torch.Generator("cpu").manual_seed(67)
    q = torch.randn(1, 2, skv, 128, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 2, skv, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(1, 2, skv, 128, generator=g).to(torch.bfloat16)
    out, lse = cp.ring(q.to(DEV), k.to(DEV), v.to(DEV), ring_degree=64, ring_anything=anything,
                       causal=causal)
    torch.cuda.synchronize()
    status_ok()
    ro, rl = oracle.ring(q, k, v, 128 ** -0.5, ring_degree=64, ring_anything=anything,
                         causal=causal)
    assert maxabs(out, ro) <= 1e-2
    assert maxabs(lse, rl) <= 1e-3
