"""The bounds-checking build (libcpattn_check.so, -DCPATTN_CHECK), the
stand-in for compute-sanitizer, which the GPU pool these tests run on does
not offer.

Every global load and store of the kernels is tested in that build against
the extent of the buffer it belongs to; an access outside is skipped and
reported as CPATTN_ERR_BOUNDS, never trapped.  The tests run every entry
point through the check build on ragged shapes and require (1) no report
and (2) results bit-equal to the normal build's (the checks change no
arithmetic).  Then the testing hook cpattn_set_check_shrink makes every
output's extent 16 bytes smaller: the check build must report the writes to
those last bytes and leave them untouched, which shows that the checks run
and that a skipped write really is skipped.  No access ever leaves the real
buffers: the shrunken extents lie inside them.
"""
import pytest
import torch

import context_attention_partial_gb300 as cp
from context_attention_partial_gb300 import _lib, api
from context_attention_partial_gb300 import build as _build
from workloads import make_partials, make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
OK, BOUNDS = 0, 10
PATTERN = 0x5A


@pytest.fixture(scope="module")
def chk():
    lib = _lib.bind(_build.build(check=True))
    assert lib.cpattn_is_check_build() == 1
    assert cp.load_library().cpattn_is_check_build() == 0
    yield lib
    lib.cpattn_set_check_shrink(0)


def stream():
    return torch.cuda.current_stream().cuda_stream


def ring_with(lib, q, k, v, R, anything=False, causal=False, out=None, lse=None):
    B, H, S, D = q.shape
    out = torch.empty(B, H, S, D, device=DEV, dtype=q.dtype) if out is None else out
    lse = torch.empty(B, H, S, device=DEV, dtype=torch.float32) if lse is None else lse
    need = cp.ring_workspace_bytes(q, R)
    ws = torch.empty(max(need, 16), device=DEV, dtype=torch.uint8)
    fn = lib.cpattn_ring_causal if causal else lib.cpattn_ring
    rc = fn(api._desc(q), api._desc(k), api._desc(v), 0.0, R, int(anything), api._desc(out),
            api._desc(lse), ws.data_ptr(), need, stream())
    assert rc == OK
    return out, lse


RING_CASES = [
    # (B, H, S_q, S_kv, D, dtype, R, anything, causal)
    (1, 2, 301, 301, 128, torch.bfloat16, 3, True, False),
    (1, 2, 301, 301, 128, torch.bfloat16, 3, True, True),
    (2, 3, 77, 300, 64, torch.bfloat16, 2, False, False),
    (1, 2, 256, 256, 64, torch.float32, 4, False, False),
    (1, 2, 130, 390, 128, torch.float32, 3, False, False),
    (1, 4, 700, 700, 128, torch.bfloat16, 1, False, False),
]


@pytest.mark.parametrize("case", RING_CASES, ids=lambda c: f"q{c[2]}k{c[3]}d{c[4]}"
                         f"{str(c[5])[-4:]}R{c[6]}{'a' if c[7] else ''}{'c' if c[8] else ''}")
def test_ring_check_build_clean_and_equal(chk, case):
    B, H, Sq, Skv, D, dt, R, anything, causal = case
    g = torch.Generator("cpu").manual_seed(201)
    q = torch.randn(B, H, Sq, D, generator=g).to(dt).to(DEV)
    k = torch.randn(B, H, Skv, D, generator=g).to(dt).to(DEV)
    v = torch.randn(B, H, Skv, D, generator=g).to(dt).to(DEV)
    ref = ring_with(cp.load_library(), q, k, v, R, anything, causal)
    got = ring_with(chk, q, k, v, R, anything, causal)
    assert chk.cpattn_last_device_status(stream()) == OK
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])


def test_other_entry_points_check_build_clean_and_equal(chk):
    lib = cp.load_library()
    s = stream()
    # partial (fp32 output straight from the epilogue)
    q, k, v = make_qkv((1, 3, 129, 128), torch.bfloat16, seed=203, device=DEV)
    outs = []
    for L in (lib, chk):
        o = torch.empty(1, 3, 129, 128, device=DEV)
        l = torch.empty(1, 3, 129, device=DEV)
        assert L.cpattn_partial(api._desc(q), api._desc(k), api._desc(v), 0.0, api._desc(o),
                                api._desc(l), s) == OK
        outs.append((o, l))
    assert chk.cpattn_last_device_status(s) == OK
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    # merge on strided views
    o_a, l_a, o_b, l_b = (t.to(DEV) for t in make_partials((2, 3, 40), 64, seed=205))
    res = []
    for L in (lib, chk):
        big = torch.zeros(2, 3, 44, 68, device=DEV)
        a = big[:, :, 2:42, :64]
        a.copy_(o_a)
        la = l_a.clone()
        assert L.cpattn_merge(api._desc(a), api._desc(la), api._desc(o_b), api._desc(l_b), s) == OK
        res.append((a.clone(), la))
    assert chk.cpattn_last_device_status(s) == OK
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])
    # regroups: batched even and Ulysses Anything, forward and inverse
    xs = [make_qkv((1, 77, 7, 64), torch.bfloat16, seed=207 + i)[0].to(DEV) for i in range(3)]
    for anything, G in ((False, 7), (True, 3)):
        hm = -(-7 // G) if anything else 7 // G
        got = []
        for L in (lib, chk):
            ys = [torch.zeros(G, 1, 77, hm, 64, device=DEV, dtype=torch.bfloat16) for _ in xs]
            fn = L.cpattn_ulysses_anything_permute_batch if anything else L.cpattn_ulysses_permute_batch
            assert fn(3, api._descs(xs), G, 1, api._descs(ys), s) == OK
            backs = [torch.empty_like(x) for x in xs]
            assert fn(3, api._descs(ys), G, -1, api._descs(backs), s) == OK
            got.append((ys, backs))
        assert chk.cpattn_last_device_status(s) == OK
        for a, b in zip(got[0][0], got[1][0]):
            assert torch.equal(a, b)
        for x, b in zip(xs, got[1][1]):
            assert torch.equal(x, b)
    # Ulysses Anything attention over the padded grouped layout
    x = make_qkv((1, 200, 5, 128), torch.bfloat16, seed=211)
    grouped = [cp.ulysses_anything_permute(t.to(DEV), 3, 1) for t in x]
    got = []
    for L in (lib, chk):
        og = torch.zeros_like(grouped[0])
        lse = torch.zeros(3, 1, 2, 200, device=DEV)
        assert L.cpattn_ulysses_anything_attention(*(api._desc(t) for t in grouped), 0.0, 5, 0,
                                                   api._desc(og), api._desc(lse), s) == OK
        got.append((og, lse))
    assert chk.cpattn_last_device_status(s) == OK
    assert torch.equal(got[0][0], got[1][0]) and torch.equal(got[0][1], got[1][1])


def filled(shape, dtype):
    t = torch.empty(shape, dtype=dtype, device=DEV)
    t.view(torch.uint8).fill_(PATTERN)
    return t


def last_bytes_untouched(t, n=16):
    raw = t.contiguous().view(torch.uint8).flatten()
    return bool((raw[-n:] == PATTERN).all())


def test_shrunken_extents_are_reported_and_not_written(chk):
    s = stream()
    try:
        chk.cpattn_set_check_shrink(16)
        # ring, R = 2: out, lse and the workspace all lose their last 16 bytes
        q, k, v = make_qkv((1, 2, 256, 128), torch.bfloat16, seed=213, device=DEV)
        out = filled((1, 2, 256, 128), torch.bfloat16)
        lse = filled((1, 2, 256), torch.float32)
        need = cp.ring_workspace_bytes(q, 2)
        ws = torch.empty(need, device=DEV, dtype=torch.uint8)
        assert chk.cpattn_ring(api._desc(q), api._desc(k), api._desc(v), 0.0, 2, 0, api._desc(out),
                               api._desc(lse), ws.data_ptr(), need, s) == OK
        assert chk.cpattn_last_device_status(s) == BOUNDS
        assert last_bytes_untouched(out) and last_bytes_untouched(lse)
        assert not last_bytes_untouched(out, 32)           # the rest was written
        # merge: out_a and lse_a
        o_a, l_a, o_b, l_b = (t.to(DEV) for t in make_partials((1, 2, 64), 128, seed=215))
        a = filled((1, 2, 64, 128), torch.float32)
        la = filled((1, 2, 64), torch.float32)
        a[..., :-4].copy_(o_a[..., :-4])
        assert chk.cpattn_merge(api._desc(a), api._desc(la), api._desc(o_b), api._desc(l_b), s) == OK
        assert chk.cpattn_last_device_status(s) == BOUNDS
        assert last_bytes_untouched(a) and last_bytes_untouched(la)
        # regroup: the destination
        x = make_qkv((1, 64, 8, 128), torch.bfloat16, seed=217)[0].to(DEV)
        y = filled((4, 1, 64, 2, 128), torch.bfloat16)
        assert chk.cpattn_ulysses_permute(api._desc(x), 4, 1, api._desc(y), s) == OK
        assert chk.cpattn_last_device_status(s) == BOUNDS
        assert last_bytes_untouched(y)
    finally:
        chk.cpattn_set_check_shrink(0)
    # and with the real extents the same calls are clean again
    out2, lse2 = ring_with(chk, q, k, v, 2)
    assert chk.cpattn_last_device_status(s) == OK
    ref = ring_with(cp.load_library(), q, k, v, 2)
    assert torch.equal(out2, ref[0]) and torch.equal(lse2, ref[1])
