"""Pins of the fp64 CPU oracle to facts other than itself.

Each ``pin_*`` function checks the oracle against something the pages or the
mathematics fix: hand-worked examples (tests/golden), closed forms, a library
routine (torch fp64 softmax / logsumexp, numpy array_split and transpose),
invariants of the ring method, and brute force on tiny inputs.  The last test
compiles copies of the oracle with plausible mistakes planted in them and
checks that every one of them fails at least one pin.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

RNG = np.random.default_rng(1234)


def _rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def _torch_sdpa(q, k, v, scale):
    """Library routine: softmax + matmul + logsumexp in torch float64."""
    q, k, v = (torch.from_numpy(np.asarray(x, dtype=np.float64)) for x in (q, k, v))
    s = scale * (q @ k.transpose(-1, -2))
    return (torch.softmax(s, dim=-1) @ v).numpy(), torch.logsumexp(s, dim=-1).numpy()


# --------------------------------------------------------------------------
# full attention (the definition)
# --------------------------------------------------------------------------
def pin_hand_examples():
    for name, scale, q, k, v, out, lse in read_golden("hand_attention.txt"):
        qa = np.array([[float(x) for x in q.split()]])
        ka = np.array([[float(x) for x in r.split()] for r in k.split(";")])
        va = np.array([[float(x) for x in r.split()] for r in v.split(";")])
        o, l = oracle.attention(qa, ka, va, scale=float(scale))
        assert np.allclose(o[0], [float(x) for x in out.split()], rtol=0, atol=1e-14), name
        assert abs(l[0] - float(lse)) < 1e-14, name


def pin_torch_fp64_crosscheck():
    for (lead, s_q, s_kv, d) in [((1,), 1, 1, 1), ((2, 3), 5, 7, 4), ((3,), 17, 9, 8),
                                 ((2, 2), 33, 64, 16), ((1,), 3, 130, 5)]:
        q, k, v = _rand(*lead, s_q, d), _rand(*lead, s_kv, d), _rand(*lead, s_kv, d)
        scale = 1.0 / math.sqrt(d)
        o, l = oracle.attention(q, k, v, scale)
        ro, rl = _torch_sdpa(q, k, v, scale)
        assert np.allclose(o, ro, rtol=0, atol=1e-12)
        assert np.allclose(l, rl, rtol=0, atol=1e-12)


def pin_closed_forms():
    d, s_kv = 6, 11
    v = _rand(2, s_kv, d)
    k = _rand(2, s_kv, d)
    # Q = 0: uniform weights -> mean of V, lse = log(S_kv)
    o, l = oracle.attention(np.zeros((2, 4, d)), k, v, 0.7)
    assert np.allclose(o, np.broadcast_to(v.mean(axis=1, keepdims=True), o.shape), atol=1e-14)
    assert np.allclose(l, math.log(s_kv), atol=1e-14)
    # K = 0: the same
    o, l = oracle.attention(_rand(2, 4, d), np.zeros_like(k), v, 0.7)
    assert np.allclose(o, np.broadcast_to(v.mean(axis=1, keepdims=True), o.shape), atol=1e-14)
    assert np.allclose(l, math.log(s_kv), atol=1e-14)
    # one key: out = v_0, lse = scale * q . k_0
    q1, k1, v1 = _rand(1, 3, d), _rand(1, 1, d), _rand(1, 1, d)
    o, l = oracle.attention(q1, k1, v1, 0.3)
    assert np.allclose(o, np.broadcast_to(v1, o.shape), atol=1e-15)
    assert np.allclose(l[0], 0.3 * (q1[0] @ k1[0, 0]), atol=1e-14)
    # all V rows equal c: out = c
    c = _rand(d)
    o, _ = oracle.attention(_rand(1, 5, d), _rand(1, s_kv, d), np.broadcast_to(c, (1, s_kv, d)), 1.1)
    assert np.allclose(o, np.broadcast_to(c, o.shape), atol=1e-14)
    # one score ahead of all others by > 800: e^-800 is 0 in double, so the
    # output is that key's V row and lse is that score, exactly
    q2 = np.zeros((1, 1, 2)); q2[0, 0, 0] = 1.0
    k2 = np.array([[[900.0, 0.0], [5.0, 1.0], [-3.0, 2.0]]])
    v2 = np.array([[[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]]])
    o, l = oracle.attention(q2, k2, v2, 1.0)
    assert np.array_equal(o[0, 0], [1.0, 2.0]) and l[0, 0] == 900.0


def pin_key_permutation_invariance():
    q, k, v = _rand(2, 9, 5), _rand(2, 13, 5), _rand(2, 13, 5)
    perm = RNG.permutation(13)
    o1, l1 = oracle.attention(q, k, v, 0.4)
    o2, l2 = oracle.attention(q, k[:, perm], v[:, perm], 0.4)
    assert np.allclose(o1, o2, atol=1e-13) and np.allclose(l1, l2, atol=1e-13)


def pin_brute_force_tiny():
    """S <= 3, D <= 2: every sum written out term by term with math.exp."""
    for s_q, s_kv, d in [(1, 1, 1), (2, 3, 2), (3, 2, 1)]:
        q, k, v = _rand(1, s_q, d), _rand(1, s_kv, d), _rand(1, s_kv, d)
        o, l = oracle.attention(q, k, v, 0.9)
        for i in range(s_q):
            e = [math.exp(0.9 * sum(q[0, i, t] * k[0, j, t] for t in range(d))) for j in range(s_kv)]
            z = sum(e)
            for t in range(d):
                assert abs(o[0, i, t] - sum(e[j] * v[0, j, t] for j in range(s_kv)) / z) < 1e-13
            assert abs(l[0, i] - math.log(z)) < 1e-13


def pin_rows_subset():
    q, k, v = _rand(3, 10, 4), _rand(3, 12, 4), _rand(3, 12, 4)
    o, l = oracle.attention(q, k, v, 0.5)
    rows = np.array([0, 7, 13, 29, 15])
    os_, ls_ = oracle.attention(q, k, v, 0.5, rows=rows)
    assert np.array_equal(os_, o.reshape(-1, 4)[rows]) and np.array_equal(ls_, l.reshape(-1)[rows])


# --------------------------------------------------------------------------
# the ring method: partials + merge == full attention
# --------------------------------------------------------------------------
def pin_partial_is_attention_on_the_range():
    q, k, v = _rand(2, 6, 4), _rand(2, 20, 4), _rand(2, 20, 4)
    o, l = oracle.partial(q, k, v, 0.6, 5, 13)
    ro, rl = oracle.attention(q, k[:, 5:13], v[:, 5:13], 0.6)
    assert np.allclose(o, ro, atol=1e-14) and np.allclose(l, rl, atol=1e-14)


def pin_ring_equals_full_every_degree():
    """Diffusers "Context parallelism", "Ring Attention": after one full loop
    every rank has seen every token's K/V, so the merged result is full
    attention."""
    s_kv = 23
    q, k, v = _rand(2, 7, 8), _rand(2, s_kv, 8), _rand(2, s_kv, 8)
    ro, rl = oracle.attention(q, k, v, 0.35)
    for r in range(1, s_kv + 1):
        o, l = oracle.ring(q, k, v, 0.35, ring_degree=r, ring_anything=True)
        assert np.allclose(o, ro, atol=1e-12) and np.allclose(l, rl, atol=1e-12), r
        if s_kv % r == 0:
            o2, l2 = oracle.ring(q, k, v, 0.35, ring_degree=r, ring_anything=False)
            assert np.array_equal(o, o2) and np.array_equal(l, l2)


def pin_ring_equals_full_on_workload_degrees():
    # tiny workload shape in full; the larger ones on a few sampled rows
    q, k, v = _rand(2, 256, 64), _rand(2, 256, 64), _rand(2, 256, 64)
    o, l = oracle.ring(q, k, v, 1 / 8, ring_degree=4)
    ro, rl = oracle.attention(q, k, v, 1 / 8)
    assert np.allclose(o, ro, atol=1e-12) and np.allclose(l, rl, atol=1e-12)
    for s, r, anything in [(4608, 2, False), (4609, 3, True)]:
        q, k, v = _rand(1, 4, 128), _rand(1, s, 128), _rand(1, s, 128)
        o, l = oracle.ring(q, k, v, 128 ** -0.5, ring_degree=r, ring_anything=anything)
        ro, rl = oracle.attention(q, k, v, 128 ** -0.5)
        assert np.allclose(o, ro, atol=1e-12) and np.allclose(l, rl, atol=1e-12)


# --------------------------------------------------------------------------
# merge
# --------------------------------------------------------------------------
def pin_merge_properties():
    n, d = 50, 7
    oa, ob, oc = _rand(n, d), _rand(n, d), _rand(n, d)
    la, lb, lc = _rand(n, scale=5), _rand(n, scale=5), _rand(n, scale=5)
    # commutative, exactly
    x = oracle.merge(oa, la, ob, lb)
    y = oracle.merge(ob, lb, oa, la)
    assert np.array_equal(x[0], y[0]) and np.array_equal(x[1], y[1])
    # associative and order-independent
    left = oracle.merge(*oracle.merge(oa, la, ob, lb), oc, lc)
    right = oracle.merge(oa, la, *oracle.merge(ob, lb, oc, lc))
    mid = oracle.merge(*oracle.merge(oc, lc, oa, la), ob, lb)
    for a in (right, mid):
        assert np.allclose(left[0], a[0], atol=1e-12) and np.allclose(left[1], a[1], atol=1e-12)
    # lse = -inf is the identity
    ninf = np.full(n, -np.inf)
    o, l = oracle.merge(oa, la, np.zeros((n, d)), ninf)
    assert np.array_equal(o, oa) and np.array_equal(l, la)
    o, l = oracle.merge(np.zeros((n, d)), ninf, ob, lb)
    assert np.array_equal(o, ob) and np.array_equal(l, lb)
    o, l = oracle.merge(np.zeros((n, d)), ninf, np.zeros((n, d)), ninf)
    assert np.all(o == 0) and np.all(l == -np.inf)
    # merging a partial with itself doubles its mass: lse + log 2
    o, l = oracle.merge(oa, la, oa, la)
    assert np.allclose(o, oa, atol=1e-14) and np.allclose(l, la + math.log(2), atol=1e-14)
    # closed form: lse = log(e^a + e^b), weights e^(a - lse)
    lse = np.logaddexp(la, lb)
    assert np.allclose(x[1], lse, atol=1e-13)
    w = np.exp(la - lse)[:, None]
    assert np.allclose(x[0], w * oa + (1 - w) * ob, atol=1e-13)
    # extreme gaps do not overflow
    o, l = oracle.merge(oa[:1], np.array([800.0]), ob[:1], np.array([-800.0]))
    assert np.allclose(o, oa[:1], atol=1e-300) and l[0] == 800.0


def pin_merge_of_disjoint_partials_is_full():
    q, k, v = _rand(3, 5, 6), _rand(3, 19, 6), _rand(3, 19, 6)
    a = oracle.partial(q, k, v, 0.8, 0, 8)
    b = oracle.partial(q, k, v, 0.8, 8, 19)
    o, l = oracle.merge(*a, *b)
    ro, rl = oracle.attention(q, k, v, 0.8)
    assert np.allclose(o, ro, atol=1e-13) and np.allclose(l, rl, atol=1e-13)


# --------------------------------------------------------------------------
# chunk partition
# --------------------------------------------------------------------------
def pin_chunk_bounds():
    for s, r, anything, expect in read_golden("chunk_bounds.txt"):
        s, r, anything = int(s), int(r), bool(int(anything))
        if expect.startswith("ERR"):
            with pytest.raises(oracle.OracleError):
                oracle.chunk_bounds(s, r, anything)
            continue
        b = oracle.chunk_bounds(s, r, anything)
        assert [b[i + 1] - b[i] for i in range(r)] == [int(x) for x in expect.split()], (s, r)
    # Ring Anything lengths equal numpy's array_split (first S mod R longer)
    for s in range(1, 40):
        for r in range(1, s + 1):
            b = oracle.chunk_bounds(s, r, True)
            lens = [len(a) for a in np.array_split(np.arange(s), r)]
            assert [b[i + 1] - b[i] for i in range(r)] == lens
            assert b[0] == 0 and b[-1] == s


# --------------------------------------------------------------------------
# Ulysses permute
# --------------------------------------------------------------------------
def pin_ulysses_permute():
    for (b, s, h, d, g) in [(1, 5, 4, 3, 2), (2, 3, 6, 4, 3), (1, 7, 24, 2, 4), (2, 2, 5, 2, 5),
                            (1, 3, 4, 8, 1)]:
        x = RNG.integers(-2 ** 31, 2 ** 31 - 1, size=(b, s, h, d), dtype=np.int64).astype(np.int32)
        y = oracle.ulysses_permute(x, g, 1)
        # library routine: split the head axis and move the group axis first
        ref = x.reshape(b, s, g, h // g, d).transpose(2, 0, 1, 3, 4)
        assert np.array_equal(y, ref)
        assert np.array_equal(oracle.ulysses_permute(y, g, -1), x)
        if g == 1:
            assert np.array_equal(y[0], x)
    # bf16 through torch, bit-exact round trip
    xt = torch.randn(2, 9, 12, 16).to(torch.bfloat16)
    yt = oracle.ulysses_permute(xt, 4, 1)
    assert yt.dtype == torch.bfloat16 and tuple(yt.shape) == (4, 2, 9, 3, 16)
    assert torch.equal(yt, xt.reshape(2, 9, 4, 3, 16).permute(2, 0, 1, 3, 4))
    assert torch.equal(oracle.ulysses_permute(yt, 4, -1), xt)
    with pytest.raises(oracle.OracleError):
        oracle.ulysses_permute(np.zeros((1, 2, 6, 4), np.int32), 4, 1)


def pin_unified_is_full_attention():
    """Diffusers "Context parallelism", "Unified Attention": regroup, ring on
    the result, reverse the regroup -- still every query meets every key of
    its head once, so the result is full attention per head."""
    for (b, s, h, d, g, r) in [(1, 12, 4, 3, 2, 3), (2, 8, 6, 4, 3, 2), (1, 10, 4, 2, 4, 5),
                               (1, 9, 2, 2, 1, 3), (1, 7, 6, 2, 6, 1)]:
        q, k, v = _rand(b, s, h, d), _rand(b, s, h, d), _rand(b, s, h, d)
        o, l = oracle.unified(q, k, v, g, r, 0.6)
        bhsd = lambda t: np.transpose(t, (0, 2, 1, 3))
        ro, rl = oracle.attention(bhsd(q), bhsd(k), bhsd(v), 0.6)   # [B, H, S, D]
        assert np.allclose(o, np.transpose(ro, (0, 2, 1, 3)), atol=1e-12)
        lg = l.reshape(g, b, h // g, s).transpose(1, 0, 2, 3).reshape(b, h, s)
        assert np.allclose(lg, rl, atol=1e-12)


# --------------------------------------------------------------------------
# Ulysses Anything (uneven head groups)
# --------------------------------------------------------------------------
def pin_ulysses_anything_heads():
    for h, g, expect in read_golden("ulysses_anything_heads.txt"):
        h, g = int(h), int(g)
        if expect.startswith("ERR"):
            with pytest.raises(oracle.OracleError):
                oracle.ulysses_anything_heads(h, g)
            continue
        st = oracle.ulysses_anything_heads(h, g)
        assert [st[i + 1] - st[i] for i in range(g)] == [int(x) for x in expect.split()], (h, g)
    # library routine: numpy's array_split deals out the same groups
    for h in range(1, 40):
        for g in range(1, 12):
            st = oracle.ulysses_anything_heads(h, g)
            groups = np.array_split(np.arange(h), g)
            assert st == [0] + list(np.cumsum([len(a) for a in groups]))


def pin_ulysses_anything_permute():
    for (b, s, h, d, g) in [(1, 5, 5, 3, 2), (2, 3, 7, 4, 3), (1, 4, 24, 2, 5), (1, 3, 24, 2, 7),
                            (2, 2, 2, 3, 4), (1, 3, 6, 2, 3), (1, 2, 4, 8, 1)]:
        x = RNG.integers(-2 ** 31, 2 ** 31 - 1, size=(b, s, h, d), dtype=np.int64).astype(np.int32)
        y = oracle.ulysses_anything_permute(x, g, 1, fill=-7)
        hm = -(-h // g)
        assert y.shape == (g, b, s, hm, d)
        # library routine: array_split of the head axis, each group padded
        for gi, heads in enumerate(np.array_split(np.arange(h), g)):
            assert np.array_equal(y[gi, :, :, :len(heads)], x[:, :, heads])
            assert np.all(y[gi, :, :, len(heads):] == -7)
        assert np.array_equal(oracle.ulysses_anything_permute(y, g, -1, heads=h), x)
        if h % g == 0:   # no padding: plain Ulysses
            assert np.array_equal(y, oracle.ulysses_permute(x, g, 1))
    # padding slots are never read by the inverse
    x = RNG.integers(0, 100, size=(1, 2, 5, 2)).astype(np.int32)
    y = oracle.ulysses_anything_permute(x, 3, 1)
    y[2, :, :, 1] = 12345
    assert np.array_equal(oracle.ulysses_anything_permute(y, 3, -1, heads=5), x)
    # bf16 through torch, bit-exact round trip
    xt = torch.randn(2, 9, 7, 16).to(torch.bfloat16)
    yt = oracle.ulysses_anything_permute(xt, 3, 1)
    assert yt.dtype == torch.bfloat16 and tuple(yt.shape) == (3, 2, 9, 3, 16)
    assert torch.equal(yt[2, :, :, :2], xt[:, :, 5:7])
    assert torch.equal(oracle.ulysses_anything_permute(yt, 3, -1, heads=7), xt)


def pin_ulysses_anything_is_full_attention():
    """Every head keeps its full sequence in exactly one group, so the
    composition is full attention per head, whatever the group sizes."""
    for (b, s, h, d, g, causal) in [(1, 9, 5, 3, 2, False), (2, 7, 7, 4, 3, False),
                                    (1, 6, 2, 2, 4, False), (1, 11, 5, 3, 3, True),
                                    (1, 8, 6, 2, 3, False)]:
        q, k, v = _rand(b, s, h, d), _rand(b, s, h, d), _rand(b, s, h, d)
        o, l = oracle.ulysses_anything(q, k, v, g, 0.7, causal=causal)
        bhsd = lambda t: np.transpose(t, (0, 2, 1, 3))
        ro, rl = oracle.attention(bhsd(q), bhsd(k), bhsd(v), 0.7, causal=causal)
        assert np.allclose(o, np.transpose(ro, (0, 2, 1, 3)), atol=1e-12)
        for gi, heads in enumerate(np.array_split(np.arange(h), g)):
            assert np.allclose(l[gi, :, :len(heads)], rl[:, heads], atol=1e-12)
            assert np.all(np.isnan(l[gi, :, len(heads):]))


# --------------------------------------------------------------------------
# causal (scaled_dot_product_attention's is_causal: query i attends keys j <= i)
# --------------------------------------------------------------------------
def pin_causal_torch_crosscheck():
    for (lead, s_q, s_kv, d) in [((2,), 7, 7, 3), ((1, 3), 12, 12, 5), ((2,), 5, 9, 4),
                                 ((1,), 9, 4, 2)]:
        q, k, v = _rand(*lead, s_q, d), _rand(*lead, s_kv, d), _rand(*lead, s_kv, d)
        o, l = oracle.attention(q, k, v, 0.45, causal=True)
        qt, kt, vt = (torch.from_numpy(x) for x in (q, k, v))
        sc = 0.45 * (qt @ kt.transpose(-1, -2))
        allowed = torch.ones(s_q, s_kv, dtype=torch.bool).tril()     # top-left aligned
        sc = sc.masked_fill(~allowed, float("-inf"))
        ro = torch.softmax(sc, dim=-1) @ vt
        rl = torch.logsumexp(sc, dim=-1)
        assert np.allclose(o, ro.numpy(), atol=1e-12) and np.allclose(l, rl.numpy(), atol=1e-12)


def pin_causal_closed_forms():
    q, k, v = _rand(2, 6, 4), _rand(2, 6, 4), _rand(2, 6, 4)
    o, l = oracle.attention(q, k, v, 0.8, causal=True)
    # the first query sees only the first key
    assert np.allclose(o[:, 0], v[:, 0], atol=1e-15)
    assert np.allclose(l[:, 0], 0.8 * np.einsum("bd,bd->b", q[:, 0], k[:, 0]), atol=1e-14)
    # the last query of a square problem sees every key: plain attention
    fo, fl = oracle.attention(q, k, v, 0.8)
    assert np.allclose(o[:, -1], fo[:, -1], atol=1e-14) and np.allclose(l[:, -1], fl[:, -1], atol=1e-14)
    # a key range entirely after a row gives that row the empty partial
    po, pl = oracle.partial(q, k, v, 0.8, 3, 6, causal=True)
    assert np.all(po[:, :3] == 0) and np.all(pl[:, :3] == -np.inf)
    assert np.all(np.isfinite(pl[:, 3:]))


def pin_causal_ring_equals_full():
    s = 19
    q, k, v = _rand(2, s, 6), _rand(2, s, 6), _rand(2, s, 6)
    ro, rl = oracle.attention(q, k, v, 0.5, causal=True)
    for r in range(1, s + 1):
        o, l = oracle.ring(q, k, v, 0.5, ring_degree=r, ring_anything=True, causal=True)
        assert np.allclose(o, ro, atol=1e-12) and np.allclose(l, rl, atol=1e-12), r


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# Plausible mistakes, each planted in a copy of the oracle source.  Every one
# must make at least one pin fail.
MUTANTS = {
    "dropped_max_shift": ("z += exp(s[j] - m);", "z += exp(s[j]);"),
    "wrong_exp_sign": ("double p = exp(scale * dot - m);", "double p = exp(m - scale * dot);"),
    "scale_dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "k_for_v": ("oi[e] += w * vb[j * d + e];", "oi[e] += w * kb[j * d + e];"),
    "head_offset_wrong": ("const double* kb = k + bh * s_kv * d;\n      const double* vb",
                          "const double* kb = k + 0 * bh * s_kv * d;\n      const double* vb"),
    "lse_log2": ("lse[r] = m + log(z);\n    }\n    free(s);", "lse[r] = m + log2(z);\n    }\n    free(s);"),
    "partial_no_normalise": ("for (int64_t e = 0; e < d; ++e) oi[e] /= z;", ""),
    "merge_weight_swapped": ("double wa = exp(a - l), wb = exp(b - l);",
                             "double wa = exp(b - l), wb = exp(a - l);"),
    "merge_no_log1p": ("double l = hi + log1p(exp(lo - hi));", "double l = hi + exp(lo - hi);"),
    "ring_skips_last_chunk": ("for (int64_t c = 1; c < ring_degree && rc == CPO_OK; ++c)",
                              "for (int64_t c = 1; c + 1 < ring_degree && rc == CPO_OK; ++c)"),
    "uneven_extra_at_end": ("bounds[c + 1] = bounds[c] + base + (c < extra ? 1 : 0);",
                            "bounds[c + 1] = bounds[c] + base + (c >= ring_degree - extra ? 1 : 0);"),
    "even_split_not_checked": ("if (!ring_anything && s_kv % ring_degree != 0) return CPO_ERR_DIVISIBILITY;", ""),
    "causal_excludes_diagonal": ("if (causal && i + 1 < s_kv) n_keys = i + 1;",
                                 "if (causal && i < s_kv) n_keys = i;"),
    "partial_causal_ignored": ("if (causal && i + 1 < k1) hi_key = i + 1;", ""),
    "anything_extra_heads_at_end": ("start[i + 1] = start[i] + base + (i < longer ? 1 : 0);",
                                    "start[i + 1] = start[i] + base + (i >= g - longer ? 1 : 0);"),
    "anything_dense_groups": ("int64_t grouped = (((gi * b + bi) * s + si) * hm + j) * d + e;",
                              "int64_t grouped = (((gi * b + bi) * s + si) * hg + j) * d + e;"),
    "anything_heads_reversed": ("int64_t bshd = ((bi * s + si) * h + start[gi] + j) * d + e;",
                                "int64_t bshd = ((bi * s + si) * h + start[gi + 1] - 1 - j) * d + e;"),
    "permute_group_index": ("int64_t bshd = ((bi * s + si) * h + gi * hg + hh) * d + e;",
                            "int64_t bshd = ((bi * s + si) * h + hh * g + gi) * d + e;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"mut_{name}.so"))
    failed = []
    with oracle.use_library(path):
        for pin in PINS:
            try:
                pin()
            except (AssertionError, oracle.OracleError, pytest.fail.Exception, Exception):
                failed.append(pin.__name__)
    assert failed, f"planted mistake {name} passed every pin"
