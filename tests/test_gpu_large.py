"""The largest tensors: element and 16-byte-vector indices past 2^31 (and,
for the attention, past 2^32), where the kernels' 64-bit index paths run.

Every call goes first through the bounds-checking build
(libcpattn_check.so), which skips and reports any access outside the
caller's buffers instead of making it: it must report nothing.  Only then
does the normal build run the same call, and its result must be bit-equal
to the checked build's.  The oracle checks sampled rows (attention, merge)
or sampled sequence slices (regroups, byte-exact) at the start, the middle
and the far end of each tensor, where an index that wrapped would land.

Inputs come from torch's seeded generator on the device (tens of GB; the
host would take minutes); the oracle reads back the slices it checks.
The cases hold 15 to 105 GB on the device at once and are skipped on a GPU
with less free memory.
"""
import numpy as np
import pytest
import torch

import context_attention_partial_gb300 as cp
import oracle
from context_attention_partial_gb300 import _lib, api
from context_attention_partial_gb300 import build as _build

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
OK = 0
TOL_OUT, TOL_LSE = 1e-2, 1e-3


@pytest.fixture(scope="module")
def chk():
    lib = _lib.bind(_build.build(check=True))
    assert lib.cpattn_is_check_build() == 1
    yield lib


@pytest.fixture(autouse=True)
def release_memory():
    torch.cuda.empty_cache()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def need_free(gb):
    free, _ = torch.cuda.mem_get_info()
    if free < gb * 1e9:
        pytest.skip(f"needs {gb} GB free on the device, {free / 1e9:.0f} GB free")


def stream():
    return torch.cuda.current_stream().cuda_stream


def randn(shape, dtype, seed):
    """N(0, 1) from torch's seeded device generator, one leading slice at a
    time (no full-size fp32 temporary)."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    t = torch.empty(shape, dtype=dtype, device=DEV)
    for i in range(shape[0]):
        t[i] = torch.randn(shape[1:], generator=g, device=DEV, dtype=torch.float32).to(dtype)
    return t


def random_bits(n, seed):
    """n random int16 values (any bit pattern, NaNs included: the regroups
    move bytes, and results are compared as int16)."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randint(-32768, 32768, (n,), generator=g, device=DEV, dtype=torch.int16)


def edge_rows(s, n_random=6, seed=0):
    rows = {0, 1, 127, 128, s // 2, s - 129, s - 128, s - 2, s - 1}
    rng = np.random.default_rng(seed)
    rows |= set(int(r) for r in rng.integers(0, s, size=n_random))
    return sorted(rows)


def test_ring_past_2_to_the_32_elements(chk):
    """Ring Anything, R = 3, bf16 [16, 64, 32771, 128]: 4,295,360,512
    elements per tensor (past 2^32), a ragged last query block, and a
    17 GB fp32 running-state workspace."""
    need_free(60)
    B, H, S, D, R = 16, 64, 32771, 128, 3
    q = randn((B, H, S, D), torch.bfloat16, 301)
    k = randn((B, H, S, D), torch.bfloat16, 302)
    v = randn((B, H, S, D), torch.bfloat16, 303)
    assert q.numel() > 2 ** 32
    need = cp.ring_workspace_bytes(q, R)
    ws = torch.empty(need, device=DEV, dtype=torch.uint8)
    out = torch.empty_like(q)
    lse = torch.empty(B, H, S, device=DEV)
    args = (api._desc(q), api._desc(k), api._desc(v), 0.0, R, 1, api._desc(out), api._desc(lse),
            ws.data_ptr(), need, stream())
    assert chk.cpattn_ring(*args) == OK
    torch.cuda.synchronize()
    assert chk.cpattn_last_device_status(stream()) == OK
    out_chk, lse_chk = out.clone(), lse.clone()
    lib = cp.load_library()
    assert lib.cpattn_ring(*args) == OK
    torch.cuda.synchronize()
    assert lib.cpattn_last_device_status(stream()) == OK
    assert torch.equal(out, out_chk) and torch.equal(lse, lse_chk)
    del out_chk, lse_chk, ws
    for i, (b, h) in enumerate([(0, 0), (7, 31), (B - 1, H - 1), (B - 1, 0)]):
        rows = edge_rows(S, seed=i)
        ro, rl = oracle.ring(q[b, h].cpu().unsqueeze(0), k[b, h].cpu().unsqueeze(0),
                             v[b, h].cpu().unsqueeze(0), D ** -0.5, ring_degree=R,
                             ring_anything=True, rows=rows)
        got_o = out[b, h, rows].float().cpu().numpy()
        got_l = lse[b, h, rows].cpu().numpy()
        ro, rl = ro.reshape(len(rows), D), rl.reshape(len(rows))
        assert np.abs(got_o - ro).max() <= TOL_OUT, (b, h)
        assert np.abs(got_l - rl).max() <= TOL_LSE, (b, h)


def test_merge_past_2_to_the_31_elements(chk):
    """fp32 partials [16, 64, 32771, 128] (17.2 GB each; 4.3e9 elements)."""
    need_free(60)
    shape = (16, 64, 32771, 128)
    o_a = randn(shape, torch.float32, 311)
    o_b = randn(shape, torch.float32, 312)
    g = torch.Generator(device=DEV).manual_seed(313)
    l_a = torch.randn(shape[:3], generator=g, device=DEV) * 4 + 8
    l_b = torch.randn(shape[:3], generator=g, device=DEV) * 4 + 8
    picks = [(0, 0), (9, 40), (15, 63)]
    rows = edge_rows(shape[2])
    saved = [(o_a[b, h, rows].cpu(), l_a[b, h, rows].cpu(), o_b[b, h, rows].cpu(),
              l_b[b, h, rows].cpu()) for b, h in picks]
    # the checked build merges into copies of the first partial; the normal
    # build into the originals
    o_c, l_c = o_a.clone(), l_a.clone()
    assert chk.cpattn_merge(api._desc(o_c), api._desc(l_c), api._desc(o_b), api._desc(l_b),
                            stream()) == OK
    torch.cuda.synchronize()
    assert chk.cpattn_last_device_status(stream()) == OK
    cp.merge(o_a, l_a, o_b, l_b)
    torch.cuda.synchronize()
    assert cp.last_device_status() == OK
    assert torch.equal(o_a, o_c) and torch.equal(l_a, l_c)
    for (b, h), (ao, al, bo, bl) in zip(picks, saved):
        eo, el = oracle.merge(ao, al, bo, bl)
        assert np.abs(o_a[b, h, rows].cpu().numpy() - eo).max() <= 1e-5, (b, h)
        assert np.abs(l_a[b, h, rows].cpu().numpy() - el).max() <= 1e-5, (b, h)


def _permute_slices_match(x, y, degree, starts, width, anything=False):
    """y's sequence positions [s0, s0 + width) equal the oracle's regroup of
    x's, byte for byte (the regroup moves each sequence position alone)."""
    for s0 in starts:
        xs = x[:, s0:s0 + width].cpu().view(torch.int16)
        if anything:
            want = oracle.ulysses_anything_permute(xs, degree, 1)
        else:
            want = oracle.ulysses_permute(xs, degree, 1)
        want = want.numpy() if hasattr(want, "numpy") else np.asarray(want)
        got = y[:, :, s0:s0 + width].cpu().view(torch.int16).numpy()
        if anything:   # padding slots are not written
            h = x.shape[2]
            for g in range(degree):
                hg = h // degree + (1 if g < h % degree else 0)
                assert np.array_equal(got[g, :, :, :hg], want[g, :, :, :hg]), (s0, g)
        else:
            assert np.array_equal(got, want), s0


def test_regroup_past_2_to_the_31_vectors(chk):
    """Ulysses regroup, bf16 [1, 2^20 + 7, 128, 128], G = 4: 34.4 GB, more
    than 2^31 16-byte vectors (the 64-bit index form of the vector kernel),
    forward and inverse."""
    need_free(110)
    B, S, H, D, G = 1, 2 ** 20 + 7, 128, 128, 4
    x = random_bits(B * S * H * D, 321).view(torch.bfloat16).view(B, S, H, D)
    assert x.numel() * 2 // 16 > 2 ** 31
    y = torch.empty(G, B, S, H // G, D, device=DEV, dtype=torch.bfloat16)
    assert chk.cpattn_ulysses_permute(api._desc(x), G, 1, api._desc(y), stream()) == OK
    torch.cuda.synchronize()
    assert chk.cpattn_last_device_status(stream()) == OK
    y2 = cp.ulysses_permute(x, G, 1)
    torch.cuda.synchronize()
    assert cp.last_device_status() == OK
    assert torch.equal(y2.view(torch.int16), y.view(torch.int16))
    del y2
    starts = [0, S // 2, S - 64]
    _permute_slices_match(x, y, G, starts, 64)
    saved = {s0: x[:, s0:s0 + 64].clone() for s0 in starts}
    del x
    back = cp.ulysses_permute(y, G, -1)
    torch.cuda.synchronize()
    assert cp.last_device_status() == OK
    for s0, xs in saved.items():
        assert torch.equal(back[:, s0:s0 + 64].view(torch.int16), xs.view(torch.int16)), s0


def test_regroup_elementwise_past_2_to_the_31_elements(chk):
    """A bf16 regroup whose base is not 16-byte aligned (element kernel):
    [1, 2^21 + 3, 8, 128], 2^31 + 3072 elements, G = 2."""
    need_free(25)
    B, S, H, D, G = 1, 2 ** 21 + 3, 8, 128, 2
    n = B * S * H * D
    assert n > 2 ** 31
    buf = random_bits(n + 8, 331)
    x = buf[1:1 + n].view(torch.bfloat16).view(B, S, H, D)   # 2 bytes past alignment
    y = torch.empty(G, B, S, H // G, D, device=DEV, dtype=torch.bfloat16)
    assert chk.cpattn_ulysses_permute(api._desc(x), G, 1, api._desc(y), stream()) == OK
    torch.cuda.synchronize()
    assert chk.cpattn_last_device_status(stream()) == OK
    y2 = cp.ulysses_permute(x, G, 1)
    torch.cuda.synchronize()
    assert cp.last_device_status() == OK
    assert torch.equal(y2.view(torch.int16), y.view(torch.int16))
    del y2
    _permute_slices_match(x, y, G, [0, S // 3, S - 32], 32)


def test_anything_regroup_past_2_to_the_31_elements(chk):
    """Ulysses Anything regroup, H = 6 over G = 4 groups (2, 2, 1, 1 heads),
    bf16 [1, 2796205, 6, 128] at a base 2 bytes past alignment (element
    kernel): 2^31 + 2048 elements on the flat side, 2.9e9 on the padded
    grouped side."""
    need_free(30)
    B, S, H, D, G = 1, 2796205, 6, 128, 4
    n = B * S * H * D
    assert n > 2 ** 31
    buf = random_bits(n + 8, 341)
    x = buf[1:1 + n].view(torch.bfloat16).view(B, S, H, D)
    hm = -(-H // G)
    y = torch.zeros(G, B, S, hm, D, device=DEV, dtype=torch.bfloat16)
    assert chk.cpattn_ulysses_anything_permute(api._desc(x), G, 1, api._desc(y), stream()) == OK
    torch.cuda.synchronize()
    assert chk.cpattn_last_device_status(stream()) == OK
    y2 = torch.zeros_like(y)
    cp.ulysses_anything_permute(x, G, 1, out=y2)
    torch.cuda.synchronize()
    assert cp.last_device_status() == OK
    assert torch.equal(y2.view(torch.int16), y.view(torch.int16))
    del y2
    _permute_slices_match(x, y, G, [0, S // 2, S - 32], 32, anything=True)
    back = cp.ulysses_anything_permute(y, G, -1, heads=H)
    torch.cuda.synchronize()
    assert cp.last_device_status() == OK
    for s0 in (0, S // 2, S - 32):
        assert torch.equal(back[:, s0:s0 + 32].view(torch.int16),
                           x[:, s0:s0 + 32].view(torch.int16)), s0
