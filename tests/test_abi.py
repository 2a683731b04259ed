"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/cpattn.h declares, and rejects invalid arguments with
the documented status codes before launching anything."""
import ctypes
import os
import re

import pytest

import context_attention_partial_gb300 as cp
from context_attention_partial_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000   # a 16-byte aligned address that validation never dereferences

OK, NULL, DTYPE, SHAPE, DIV, LAYOUT, UNSUP, WS = 0, 1, 2, 3, 4, 5, 6, 7


def header_functions():
    text = open(os.path.join(ROOT, "include", "cpattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cpattn_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_header_symbol():
    lib = cp.load_library()
    names = header_functions()
    assert set(names) == set(_lib.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_library_is_in_tree_and_built_for_sm103a():
    assert os.path.dirname(_lib.LIB_PATH) == os.path.join(ROOT, "context_attention_partial_gb300")
    blob = open(_lib.LIB_PATH, "rb").read()
    assert b"sm_103a" in blob or b"sm_103" in blob


def t(shape, dtype=_lib.BF16, data=FAKE, stride=None):
    if stride is None:
        stride, acc = [], 1
        for s in reversed(shape):
            stride.insert(0, acc)
            acc *= s
    return _lib.describe(data, dtype, shape, stride)


def ring(q, k, v, R=1, anything=0, out=None, lse=None, ws=None, ws_bytes=0, scale=0.0):
    lib = cp.load_library()
    out = out if out is not None else t(tuple(q.shape[:4]), q.dtype)
    lse = lse if lse is not None else t(tuple(q.shape[:3]), _lib.F32)
    return lib.cpattn_ring(q, k, v, scale, R, anything, out, lse, ws, ws_bytes, None)


def test_status_strings():
    lib = cp.load_library()
    for code in range(10):
        assert lib.cpattn_status_string(code)
    assert lib.cpattn_status_string(0) == b"ok"


def test_ring_validation():
    q = t((1, 2, 256, 128)); kv = t((1, 2, 256, 128))
    lib = cp.load_library()
    assert lib.cpattn_ring(None, kv, kv, 0.0, 2, 0, q, t((1, 2, 256), _lib.F32), None, 0, None) == NULL
    assert ring(q, kv, kv, R=3) == DIV                                  # 256 % 3
    assert ring(q, t((1, 2, 3, 128)), t((1, 2, 3, 128)), R=4, anything=1) == SHAPE   # R > S
    assert ring(q, kv, kv, R=0) == SHAPE
    assert ring(q, kv, kv, R=65) == UNSUP
    assert ring(q, kv, t((1, 2, 256, 128), _lib.F32), R=1) == DTYPE
    assert ring(q, kv, t((1, 2, 255, 128)), R=1) == SHAPE
    assert ring(t((1, 2, 256, 96)), t((1, 2, 256, 96)), t((1, 2, 256, 96))) == UNSUP
    f = t((1, 2, 256, 96), _lib.F32)
    assert ring(f, f, f) == UNSUP                                       # D is 64 or 128
    f = t((1, 2, 256, 128), _lib.F32)
    assert ring(f, f, f, R=2) == WS                                     # f32 D = 128 is served
    # workspace required for R > 1
    assert ring(q, kv, kv, R=2) == WS
    lib_need = lib.cpattn_ring_workspace_bytes(q, 2)
    assert lib_need == 1 * 2 * 256 * (128 + 1) * 4
    assert lib.cpattn_ring_workspace_bytes(q, 1) == 0
    assert ring(q, kv, kv, R=2, ws=FAKE, ws_bytes=lib_need - 4) == WS
    assert ring(q, kv, kv, R=2, ws=FAKE + 8, ws_bytes=lib_need) == WS   # not 16-byte aligned
    # layout: inner stride must be 1; strides 16-byte multiples; aligned data
    assert ring(t((1, 2, 256, 128), stride=(65536, 32768, 128, 2)), kv, kv) == LAYOUT
    assert ring(t((1, 2, 256, 128), data=FAKE + 2), kv, kv) == LAYOUT
    assert ring(t((1, 2, 256, 64), stride=(2 * 256 * 68, 256 * 68, 68, 1)),
                t((1, 2, 256, 64)), t((1, 2, 256, 64))) == LAYOUT          # 136-byte rows
    # output dtype must match the input for ring, be f32 for partial
    assert ring(q, kv, kv, out=t((1, 2, 256, 128), _lib.F32)) == DTYPE
    assert lib.cpattn_partial(q, kv, kv, 0.0, t((1, 2, 256, 128)), t((1, 2, 256), _lib.F32), None) == DTYPE
    # empty query: a no-op that succeeds without touching memory
    e = t((1, 2, 0, 128), data=0)
    assert ring(e, kv, kv, out=t((1, 2, 0, 128), data=0), lse=t((1, 2, 0), _lib.F32, data=0)) == OK
    # keys must not be empty when there are queries
    assert lib.cpattn_partial(q, t((1, 2, 0, 128)), t((1, 2, 0, 128)), 0.0,
                              t((1, 2, 256, 128), _lib.F32), t((1, 2, 256), _lib.F32), None) == SHAPE


def test_merge_validation():
    lib = cp.load_library()
    o = t((1, 2, 8, 128), _lib.F32); l = t((1, 2, 8), _lib.F32)
    assert lib.cpattn_merge(None, l, o, l, None) == NULL
    assert lib.cpattn_merge(t((1, 2, 8, 128)), l, o, l, None) == DTYPE
    assert lib.cpattn_merge(o, l, t((1, 2, 9, 128), _lib.F32), l, None) == SHAPE
    assert lib.cpattn_merge(t((1, 2, 8, 96), _lib.F32), l, t((1, 2, 8, 96), _lib.F32), l, None) == UNSUP
    assert lib.cpattn_merge(t((1, 2, 8, 128), _lib.F32, data=FAKE + 4), l, o, l, None) == LAYOUT
    z = t((1, 2, 0, 128), _lib.F32, data=0); zl = t((1, 2, 0), _lib.F32, data=0)
    assert lib.cpattn_merge(z, zl, z, zl, None) == OK


def test_permute_validation():
    lib = cp.load_library()
    x = t((1, 16, 24, 128)); y = t((4, 1, 16, 6, 128), data=FAKE + (1 << 24))
    assert lib.cpattn_ulysses_permute(None, 4, 1, y, None) == NULL
    assert lib.cpattn_ulysses_permute(x, 5, 1, t((5, 1, 16, 4, 128)), None) == DIV
    assert lib.cpattn_ulysses_permute(x, 4, 2, y, None) == SHAPE
    assert lib.cpattn_ulysses_permute(x, 0, 1, y, None) == SHAPE
    assert lib.cpattn_ulysses_permute(x, 4, 1, t((4, 1, 16, 5, 128)), None) == SHAPE
    assert lib.cpattn_ulysses_permute(x, 4, 1, t((4, 1, 16, 6, 128), _lib.F32), None) == DTYPE
    # overlapping source and destination
    assert lib.cpattn_ulysses_permute(x, 4, 1, t((4, 1, 16, 6, 128), data=FAKE + 64), None) == LAYOUT
    # non-contiguous source
    assert lib.cpattn_ulysses_permute(t((1, 16, 24, 128), stride=(16 * 24 * 256, 24 * 256, 256, 1)),
                                      4, 1, y, None) == LAYOUT


def test_permute_batch_validation():
    """The batched regroups check every pair as the single call does, and
    that the pairs share one shape and dtype and no output overlaps another
    buffer of the call."""
    lib = cp.load_library()
    arr = lambda *ts: (_lib.CTensor * len(ts))(*ts)
    mb = 1 << 24
    for batch, h_slots, deg in ((lib.cpattn_ulysses_permute_batch, 6, 4),
                                (lib.cpattn_ulysses_anything_permute_batch, 5, 5)):
        gshape = (deg, 1, 16, h_slots, 128)
        xs = arr(*(t((1, 16, 24, 128), data=FAKE + i * mb) for i in range(3)))
        ys = arr(*(t(gshape, data=FAKE + (8 + i) * mb) for i in range(3)))
        assert batch(0, xs, deg, 1, ys, None) == SHAPE
        assert batch(5, xs, deg, 1, ys, None) == SHAPE
        assert batch(3, None, deg, 1, ys, None) == NULL
        # a pair whose shapes differ from pair 0's
        assert batch(3, xs, deg, 1, arr(ys[0], ys[1], t((deg, 1, 8, h_slots, 128),
                                                          data=FAKE + 10 * mb)), None) == SHAPE
        x_short = arr(xs[0], xs[1], t((1, 8, 24, 128), data=FAKE + 2 * mb))
        assert batch(3, x_short, deg, 1, arr(ys[0], ys[1], t((deg, 1, 8, h_slots, 128),
                                                            data=FAKE + 10 * mb)), None) == SHAPE
        # a pair of another dtype
        assert batch(2, arr(xs[0], t((1, 16, 24, 128), _lib.F32, data=FAKE + mb)), deg, 1,
                     arr(ys[0], t(gshape, _lib.F32, data=FAKE + 9 * mb)), None) == DTYPE
        # an output over another pair's input, or over another output
        assert batch(2, arr(xs[0], xs[1]), deg, 1, arr(ys[0], t(gshape, data=FAKE + 64)),
                     None) == LAYOUT
        assert batch(2, arr(xs[0], xs[1]), deg, 1, arr(ys[0], t(gshape, data=FAKE + 8 * mb + 64)),
                     None) == LAYOUT
        # every pair is checked like the single call
        assert batch(2, arr(xs[0], xs[1]), 0, 1, arr(ys[0], ys[1]), None) == SHAPE
        # nothing to move: accepted without a launch
        z = arr(t((1, 0, 24, 128), data=0), t((1, 0, 24, 128), data=0))
        zy = arr(t((deg, 1, 0, h_slots, 128), data=0), t((deg, 1, 0, h_slots, 128), data=0))
        assert batch(2, z, deg, 1, zy, None) == OK


def test_ulysses_anything_validation():
    lib = cp.load_library()
    x = t((1, 16, 24, 128)); y = t((5, 1, 16, 5, 128), data=FAKE + (1 << 24))
    perm = lib.cpattn_ulysses_anything_permute
    assert perm(None, 5, 1, y, None) == NULL
    assert perm(x, 0, 1, y, None) == SHAPE
    assert perm(x, 5, 2, y, None) == SHAPE
    assert perm(x, 5, 1, t((5, 1, 16, 4, 128), data=FAKE + (1 << 24)), None) == SHAPE  # not ceil(H/G)
    assert perm(x, 5, 1, t((5, 1, 16, 5, 128), _lib.F32, data=FAKE + (1 << 24)), None) == DTYPE
    assert perm(x, 5, 1, t((5, 1, 16, 5, 128), data=FAKE + 64), None) == LAYOUT        # overlap
    assert perm(t((1, 16, 24, 128), stride=(16 * 24 * 256, 24 * 256, 256, 1)), 5, 1, y, None) == LAYOUT
    z = t((1, 0, 24, 128), data=0)
    assert perm(z, 5, 1, t((5, 1, 0, 5, 128), data=0), None) == OK
    att = lib.cpattn_ulysses_anything_attention
    g = t((5, 1, 256, 5, 128)); lse = t((5, 1, 5, 256), _lib.F32)
    assert att(g, g, g, 0.0, 24, 0, g, None, None) == NULL
    assert att(g, g, g, 0.0, 26, 0, g, lse, None) == SHAPE          # ceil(26/5) = 6 slots
    assert att(g, g, g, 0.0, 0, 0, g, lse, None) == SHAPE
    assert att(g, g, t((5, 1, 255, 5, 128)), 0.0, 24, 0, g, lse, None) == SHAPE
    assert att(g, g, g, 0.0, 24, 0, g, t((5, 1, 256, 5), _lib.F32), None) == SHAPE
    assert att(g, g, g, 0.0, 24, 0, t((5, 1, 256, 5, 128), _lib.F32), lse, None) == DTYPE
    t96 = t((5, 1, 256, 5, 96))
    assert att(t96, t96, t96, 0.0, 24, 0, t96, lse, None) == UNSUP
    # the (group, batch) axes must merge into one batch axis
    gb = t((5, 2, 256, 5, 128), stride=(4 * 256 * 5 * 128, 256 * 5 * 128, 5 * 128, 128, 1))
    assert att(gb, gb, gb, 0.0, 24, 0, gb, t((5, 2, 5, 256), _lib.F32), None) == LAYOUT


def test_python_binding_rejects_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 4, 64)
    with pytest.raises(ValueError):
        cp.partial(q, q, q, out=torch.zeros(1, 1, 4, 64), lse=torch.zeros(1, 1, 4))


def test_normal_build_is_not_the_check_build():
    lib = cp.load_library()
    assert lib.cpattn_is_check_build() == 0
    lib.cpattn_set_check_shrink(0)                  # a no-op here
    assert lib.cpattn_status_string(10) == b"device-side bounds check failed (check build)"
