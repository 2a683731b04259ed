"""Out-of-bounds write checks by canaries (compute-sanitizer is not available
on the GPU pool this library is tested on).

Every output of a call is placed as an interior view of a larger buffer whose
bytes all start as a known pattern: padding before and after the sequence
axis, an extra head, and (for row-strided outputs) extra elements after each
row's D values.  After the call every byte outside the view must still hold
the pattern, and the view must equal the result of the same call with plain
contiguous outputs (the kernels are deterministic).  The ring workspace gets
guard bytes before and after it too.  Sizes are ragged on purpose: S_q = 1,
77, 300 and 4609 query rows, D = 64 and 128.
"""
import pytest
import torch

import context_attention_partial_gb300 as cp
from workloads import make_partials, make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
PATTERN = 0xA5


def guarded(shape, dtype, pad_front=3, pad_back=5, pad_row=None, extra_head=True):
    """A view of `shape` ([B, H, S, D] or [B, H, S]) inside a larger buffer
    filled with PATTERN bytes; returns (view, buffer, mask of the view)."""
    es = torch.tensor([], dtype=dtype).element_size()
    if pad_row is None:
        pad_row = 16 // es                 # keeps every row 16-byte aligned
    big_shape = list(shape)
    big_shape[1] += 1 if extra_head else 0
    big_shape[2] += pad_front + pad_back
    if len(shape) == 4:
        big_shape[3] += pad_row
    big = torch.empty(big_shape, dtype=dtype, device=DEV)
    big.view(torch.uint8).fill_(PATTERN)
    idx = [slice(None), slice(0, shape[1]), slice(pad_front, pad_front + shape[2])]
    if len(shape) == 4:
        idx.append(slice(0, shape[3]))
    view = big[tuple(idx)]
    mask = torch.zeros(big_shape, dtype=torch.bool, device=DEV)
    mask[tuple(idx)] = True
    return view, big, mask


def assert_outside_untouched(big, mask, what):
    es = big.element_size()
    raw = big.contiguous().view(torch.uint8).reshape(*big.shape, es)
    outside = raw[~mask]
    bad = int((outside != PATTERN).sum().item())
    assert bad == 0, f"{what}: {bad} bytes outside the output were written"


def guarded_workspace(nbytes, front=256, back=4096):
    buf = torch.full((front + nbytes + back,), PATTERN, dtype=torch.uint8, device=DEV)
    return buf[front:front + nbytes], buf, front, back


RING_CASES = [
    # (S_q, S_kv, D, dtype, R, ring_anything, causal)
    (1, 300, 128, torch.bfloat16, 3, False, False),
    (77, 300, 64, torch.bfloat16, 3, False, False),
    (300, 301, 128, torch.bfloat16, 3, True, False),
    (4609, 4609, 128, torch.bfloat16, 3, True, False),
    (4609, 4609, 64, torch.bfloat16, 2, True, False),
    (77, 256, 64, torch.float32, 4, False, False),
    (300, 301, 64, torch.float32, 3, True, False),
    (77, 300, 128, torch.float32, 3, False, False),
    (300, 300, 128, torch.float32, 2, False, True),
    (300, 300, 128, torch.bfloat16, 3, False, True),
    (4609, 4609, 128, torch.bfloat16, 3, True, True),
    (77, 77, 128, torch.bfloat16, 1, False, False),
]


@pytest.mark.parametrize("case", RING_CASES, ids=lambda c: f"q{c[0]}k{c[1]}d{c[2]}{str(c[3])[-4:]}"
                         f"R{c[4]}{'a' if c[5] else ''}{'c' if c[6] else ''}")
def test_ring_writes_only_its_outputs(case):
    S_q, S_kv, D, dt, R, anything, causal = case
    B, H = 1, 2
    g = torch.Generator("cpu").manual_seed(101)
    q = torch.randn(B, H, S_q, D, generator=g).to(dt).to(DEV)
    k = torch.randn(B, H, S_kv, D, generator=g).to(dt).to(DEV)
    v = torch.randn(B, H, S_kv, D, generator=g).to(dt).to(DEV)
    ref_o, ref_l = cp.ring(q, k, v, R, anything, causal=causal)
    out, big_o, mask_o = guarded((B, H, S_q, D), dt)
    lse, big_l, mask_l = guarded((B, H, S_q), torch.float32)
    need = cp.ring_workspace_bytes(q, R)
    ws = None
    if need:
        ws, ws_buf, front, back = guarded_workspace(need)
    cp.ring(q, k, v, R, anything, out=out, lse=lse, workspace=ws, causal=causal)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    assert_outside_untouched(big_o, mask_o, "out")
    assert_outside_untouched(big_l, mask_l, "lse")
    if need:
        assert bool((ws_buf[:front] == PATTERN).all()), "workspace underrun"
        assert bool((ws_buf[front + need:] == PATTERN).all()), "workspace overrun"


@pytest.mark.parametrize("S_q,S_kv,D,dt", [
    (1, 5, 128, torch.bfloat16), (77, 300, 64, torch.bfloat16),
    (4609, 1000, 128, torch.bfloat16), (300, 257, 64, torch.float32),
    (77, 130, 128, torch.float32),
])
def test_partial_writes_only_its_outputs(S_q, S_kv, D, dt):
    g = torch.Generator("cpu").manual_seed(103)
    q = torch.randn(2, 2, S_q, D, generator=g).to(dt).to(DEV)
    k = torch.randn(2, 2, S_kv, D, generator=g).to(dt).to(DEV)
    v = torch.randn(2, 2, S_kv, D, generator=g).to(dt).to(DEV)
    ref_o, ref_l = cp.partial(q, k, v)
    out, big_o, mask_o = guarded((2, 2, S_q, D), torch.float32)
    lse, big_l, mask_l = guarded((2, 2, S_q), torch.float32)
    cp.partial(q, k, v, out=out, lse=lse)
    torch.cuda.synchronize()
    assert cp.last_device_status() == 0
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    assert_outside_untouched(big_o, mask_o, "out")
    assert_outside_untouched(big_l, mask_l, "lse")


@pytest.mark.parametrize("S,D", [(1, 128), (77, 64), (300, 128), (4609, 64)])
def test_merge_writes_only_its_outputs(S, D):
    o_a, l_a, o_b, l_b = make_partials((2, 3, S), D, seed=107)
    ga, gla = o_a.to(DEV), l_a.to(DEV)
    cp.merge(ga, gla, o_b.to(DEV), l_b.to(DEV))
    out, big_o, mask_o = guarded((2, 3, S, D), torch.float32)
    lse, big_l, mask_l = guarded((2, 3, S), torch.float32)
    out.copy_(o_a.to(DEV))
    lse.copy_(l_a.to(DEV))
    cp.merge(out, lse, o_b.to(DEV), l_b.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(out, ga) and torch.equal(lse, gla)
    assert_outside_untouched(big_o, mask_o, "merged out")
    assert_outside_untouched(big_l, mask_l, "merged lse")


@pytest.mark.parametrize("shape,g,dt,anything", [
    ((1, 77, 24, 128), 4, torch.bfloat16, False),
    ((2, 300, 12, 64), 3, torch.bfloat16, False),
    ((1, 4609, 24, 128), 5, torch.bfloat16, True),
    ((1, 77, 7, 64), 3, torch.float32, True),
    ((2, 5, 10, 3), 5, torch.bfloat16, False),     # element path
])
def test_permute_writes_only_its_outputs(shape, g, dt, anything):
    """The regroup writes exactly its destination (a contiguous block placed
    inside a larger buffer), forward and inverse."""
    x = make_qkv(shape, dt, seed=109)[0].to(DEV)
    B, S, H, D = shape
    hm = -(-H // g)
    gshape = (g, B, S, hm if anything else H // g, D)
    n = 1
    for s in gshape:
        n *= s
    front, back = 40, 72                            # elements; keeps 16-byte alignment
    buf = torch.empty(front + n + back, dtype=dt, device=DEV)
    buf.view(torch.uint8).fill_(PATTERN)
    y = buf[front:front + n].view(gshape)
    if anything:
        cp.ulysses_anything_permute(x, g, 1, out=y)
        ref = cp.ulysses_anything_permute(x, g, 1)
    else:
        cp.ulysses_permute(x, g, 1, out=y)
        ref = cp.ulysses_permute(x, g, 1)
    torch.cuda.synchronize()
    raw = buf.view(torch.uint8)
    es = buf.element_size()
    assert bool((raw[:front * es] == PATTERN).all()) and bool((raw[(front + n) * es:] == PATTERN).all())
    if anything:
        from oracle import ulysses_anything_heads
        start = ulysses_anything_heads(H, g)
        for gi in range(g):
            hg = start[gi + 1] - start[gi]
            assert torch.equal(y[gi, :, :, :hg], ref[gi, :, :, :hg])
            pad = y[gi, :, :, hg:].contiguous().view(torch.uint8)
            assert bool((pad == PATTERN).all()), "padding slot written"
    else:
        assert torch.equal(y, ref)
    # inverse into a guarded destination
    m = x.numel()
    buf2 = torch.empty(front + m + back, dtype=dt, device=DEV)
    buf2.view(torch.uint8).fill_(PATTERN)
    back_view = buf2[front:front + m].view(shape)
    if anything:
        cp.ulysses_anything_permute(y, g, -1, out=back_view)
    else:
        cp.ulysses_permute(y, g, -1, out=back_view)
    torch.cuda.synchronize()
    raw2 = buf2.view(torch.uint8)
    assert bool((raw2[:front * es] == PATTERN).all()) and bool((raw2[(front + m) * es:] == PATTERN).all())
    assert torch.equal(back_view, x)
