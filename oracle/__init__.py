"""fp64 CPU oracle for the context-parallel attention hot path.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import it; the library
package never does, and it imports nothing from the library.  It shares no
code with the CUDA path: the arithmetic lives in ``cpattn_oracle.c`` (plain C,
IEEE double); this module only converts arrays to contiguous float64, calls
the C routines through ctypes and returns numpy arrays.

Functions and the passages they follow (page title, section):

* ``attention``   -- the definition: softmax(scale * q k^T) v and its natural
  log-sum-exp.  ParaAttention README, "Run Unified Attention ... with
  torch.compile" (the sharded output must equal the matching slice of
  scaled_dot_product_attention).
* ``partial``     -- one ring step over a key range, emitting (out, lse).
  Diffusers "Context parallelism", "Ring Attention"; Diffusers "Parallelism"
  API, ContextParallelConfig ``convert_to_fp32`` ("output and LSE").
* ``merge``       -- LSE merge of two partials (same passages).
* ``chunk_bounds``-- the key partition: even split, or the Ring Anything
  uneven split.  Diffusers "Context parallelism", variants table and
  "Ring Anything Attention".
* ``ring``        -- partials over every chunk folded with ``merge``.
* ``ulysses_permute`` -- the head regroup of Diffusers "Context parallelism",
  "Ulysses Attention", as a layout permute.
* ``unified``     -- Diffusers "Context parallelism", "Unified Attention":
  regroup, ring within each group, inverse regroup (composition of the
  functions above).
* ``ulysses_anything_heads`` / ``ulysses_anything_permute`` /
  ``ulysses_anything`` -- Diffusers "Context parallelism", "Ulysses Anything
  Attention" (and the ``ulysses_anything`` parameter of the "Parallelism"
  API): the regroup without divisibility, heads dealt out with tensor_split
  rules into groups padded to ceil(H/G) slots; attention per group on its
  own heads; inverse regroup.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cpattn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libcpattn_oracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_DIVISIBILITY, ERR_SHAPE, ERR_ALLOC = 0, 1, 2, 3


class OracleError(ValueError):
    pass


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (IEEE double, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                        "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    d, i64, p = ctypes.c_double, ctypes.c_int64, ctypes.c_void_p
    ci = ctypes.c_int
    lib.cpo_attention_rows.argtypes = [p, p, p, i64, i64, i64, i64, d, p, i64, p, p, ci]
    lib.cpo_partial_rows.argtypes = [p, p, p, i64, i64, i64, i64, d, i64, i64, p, i64, p, p, ci]
    lib.cpo_merge.argtypes = [p, p, p, p, i64, i64]
    lib.cpo_merge.restype = None
    lib.cpo_chunk_bounds.argtypes = [i64, i64, ctypes.c_int, p]
    lib.cpo_ring_rows.argtypes = [p, p, p, i64, i64, i64, i64, d, i64, ctypes.c_int, p, i64, p, p, ci]
    lib.cpo_ulysses_permute.argtypes = [p, p, i64, i64, i64, i64, i64, ctypes.c_int, i64]
    lib.cpo_ulysses_anything_heads.argtypes = [i64, i64, p]
    lib.cpo_ulysses_anything_permute.argtypes = [p, p, i64, i64, i64, i64, i64, ctypes.c_int, i64]
    lib.cpo_num_threads.argtypes = []
    for name in ("cpo_attention_rows", "cpo_partial_rows", "cpo_chunk_bounds",
                 "cpo_ring_rows", "cpo_ulysses_permute", "cpo_ulysses_anything_heads",
                 "cpo_ulysses_anything_permute", "cpo_num_threads"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


class use_library:
    """Context manager: route every oracle call through another build of the
    C source (the tests use it to check that planted mistakes fail a pin)."""

    def __init__(self, path: str):
        self._path = path

    def __enter__(self):
        global _lib
        _load()
        with _lock:
            self._saved, _lib = _lib, _bind(self._path)
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self._saved
        return False


def compile_variant(source_text: str, out_path: str) -> str:
    """Compile a (modified) copy of the oracle source into ``out_path``."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
                    "-o", out_path, src, "-lm"], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _f64(x) -> np.ndarray:
    """Any torch tensor or array -> contiguous float64 numpy (values exact)."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu", torch.float64).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int):
    if rc == ERR_DIVISIBILITY:
        raise OracleError("sequence length not divisible by ring_degree")
    if rc == ERR_SHAPE:
        raise OracleError("invalid shape or degree")
    if rc == ERR_ALLOC:
        raise MemoryError("oracle allocation failed")


def _flatten(q, k, v):
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim < 2 or k.shape != v.shape or q.shape[:-2] != k.shape[:-2] or q.shape[-1] != k.shape[-1]:
        raise OracleError(f"incompatible shapes {q.shape} {k.shape} {v.shape}")
    lead = q.shape[:-2]
    nbh = int(np.prod(lead)) if lead else 1
    return q, k, v, lead, nbh, q.shape[-2], k.shape[-2], q.shape[-1]


def _rows(rows, nbh, s_q):
    if rows is None:
        return None, nbh * s_q
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).ravel())
    if r.size and (r.min() < 0 or r.max() >= nbh * s_q):
        raise OracleError("row index out of range")
    return r, r.size


def _shape_out(lead, s_q, d, rows, n, out, lse):
    if rows is None:
        return out.reshape(*lead, s_q, d), lse.reshape(*lead, s_q)
    return out.reshape(n, d), lse.reshape(n)


def attention(q, k, v, scale=None, rows=None, causal=False):
    """Full softmax attention (the definition).  q [..., S_q, D],
    k, v [..., S_kv, D].  ``rows``: optional flat indices into the
    [prod(...) * S_q] query rows; then out is [n, D] and lse [n].
    ``causal``: query i attends keys j <= i (is_causal)."""
    q, k, v, lead, nbh, s_q, s_kv, d = _flatten(q, k, v)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    r, n = _rows(rows, nbh, s_q)
    out = np.empty((n, d)); lse = np.empty(n)
    _check(_load().cpo_attention_rows(_ptr(q), _ptr(k), _ptr(v), nbh, s_q, s_kv, d,
                                      scale, None if r is None else _ptr(r), n,
                                      _ptr(out), _ptr(lse), int(bool(causal))))
    return _shape_out(lead, s_q, d, r, n, out, lse)


def partial(q, k, v, scale=None, k0=0, k1=None, rows=None, causal=False):
    """One ring step: attention over keys [k0, k1) only -> (out, lse)."""
    q, k, v, lead, nbh, s_q, s_kv, d = _flatten(q, k, v)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    k1 = s_kv if k1 is None else k1
    r, n = _rows(rows, nbh, s_q)
    out = np.empty((n, d)); lse = np.empty(n)
    _check(_load().cpo_partial_rows(_ptr(q), _ptr(k), _ptr(v), nbh, s_q, s_kv, d, scale,
                                    k0, k1, None if r is None else _ptr(r), n,
                                    _ptr(out), _ptr(lse), int(bool(causal))))
    return _shape_out(lead, s_q, d, r, n, out, lse)


def merge(o_a, lse_a, o_b, lse_b):
    """LSE merge of two partials; returns new arrays (inputs untouched)."""
    o = _f64(o_a).copy(); l = _f64(lse_a).copy()
    ob = _f64(o_b); lb = _f64(lse_b)
    if o.shape != ob.shape or l.shape != lb.shape or o.shape[:-1] != l.shape:
        raise OracleError("merge shape mismatch")
    d = o.shape[-1]
    _load().cpo_merge(_ptr(o), _ptr(l), _ptr(ob), _ptr(lb), l.size, d)
    return o, l


def chunk_bounds(s_kv: int, ring_degree: int, ring_anything: bool = False):
    """Chunk c of the key sequence is [b[c], b[c+1])."""
    b = np.empty(max(ring_degree, 0) + 1, dtype=np.int64)
    _check(_load().cpo_chunk_bounds(s_kv, ring_degree, int(bool(ring_anything)), _ptr(b)))
    return [int(x) for x in b]


def ring(q, k, v, scale=None, ring_degree=1, ring_anything=False, rows=None, causal=False):
    """The ring schedule: a partial per chunk, folded with ``merge`` in
    chunk order 0..R-1."""
    q, k, v, lead, nbh, s_q, s_kv, d = _flatten(q, k, v)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    r, n = _rows(rows, nbh, s_q)
    out = np.empty((n, d)); lse = np.empty(n)
    _check(_load().cpo_ring_rows(_ptr(q), _ptr(k), _ptr(v), nbh, s_q, s_kv, d, scale,
                                 ring_degree, int(bool(ring_anything)),
                                 None if r is None else _ptr(r), n, _ptr(out), _ptr(lse),
                                 int(bool(causal))))
    return _shape_out(lead, s_q, d, r, n, out, lse)


def ulysses_permute(x, degree: int, direction: int):
    """Head regroup as a byte-exact layout permute.
    direction +1: x [B, S, H, D] -> [G, B, S, H/G, D];
    direction -1: x [G, B, S, H/G, D] -> [B, S, H, D]."""
    is_torch = hasattr(x, "detach")
    if is_torch:
        import torch
        t = x.detach().cpu().contiguous()
        raw = t.view(torch.int16).numpy() if t.element_size() == 2 else (
            t.view(torch.int32).numpy() if t.element_size() == 4 else t.numpy())
    else:
        raw = np.ascontiguousarray(x)
    if direction == 1:
        if raw.ndim != 4:
            raise OracleError("forward permute takes [B, S, H, D]")
        b, s, h, d = raw.shape
        if degree < 1 or h % degree:
            raise OracleError("H must be divisible by the Ulysses degree")
        out_shape = (degree, b, s, h // degree, d)
    elif direction == -1:
        if raw.ndim != 5 or raw.shape[0] != degree:
            raise OracleError("inverse permute takes [G, B, S, H/G, D]")
        g, b, s, hg, d = raw.shape
        h = g * hg
        out_shape = (b, s, h, d)
    else:
        raise OracleError("direction must be +1 or -1")
    y = np.empty(out_shape, dtype=raw.dtype)
    _check(_load().cpo_ulysses_permute(_ptr(raw), _ptr(y), b, s, h, d, degree, direction,
                                       raw.dtype.itemsize))
    if is_torch:
        import torch
        yt = torch.from_numpy(y)
        return yt.view(x.dtype) if yt.dtype != x.dtype else yt
    return y


def unified(q, k, v, ulysses_degree: int, ring_degree: int = 1, scale=None, causal=False):
    """Unified (Ulysses x Ring) attention as the steps of Diffusers "Context
    parallelism", "Unified Attention": head regroup of q, k, v [B, S, H, D]
    into G groups (``ulysses_permute``), the ring schedule with ring_degree
    chunks over each group's full sequence (``ring``), inverse regroup of the
    output.  Returns (out [B, S, H, D] float64, lse [G, B, H/G, S])."""
    G, R = int(ulysses_degree), int(ring_degree)
    qg, kg, vg = (ulysses_permute(_f64(x), G, 1) for x in (q, k, v))   # [G, B, S, Hg, D]
    to_bhsd = lambda t: np.ascontiguousarray(np.transpose(t, (0, 1, 3, 2, 4)))   # [G, B, Hg, S, D]
    o, l = ring(to_bhsd(qg), to_bhsd(kg), to_bhsd(vg), scale, ring_degree=R, causal=causal)
    og = np.ascontiguousarray(np.transpose(o, (0, 1, 3, 2, 4)))        # [G, B, S, Hg, D]
    return ulysses_permute(og, G, -1), l


def ulysses_anything_heads(heads: int, degree: int):
    """Head groups of Ulysses Anything: group g holds heads
    [start[g], start[g+1]); returns start (length degree + 1)."""
    start = np.zeros(int(degree) + 1, dtype=np.int64)
    _check(_load().cpo_ulysses_anything_heads(int(heads), int(degree), _ptr(start)))
    return [int(x) for x in start]


def _raw(x):
    if hasattr(x, "detach"):
        import torch
        t = x.detach().cpu().contiguous()
        if t.element_size() == 2:
            return t.view(torch.int16).numpy()
        if t.element_size() == 4:
            return t.view(torch.int32).numpy()
        return t.numpy()
    return np.ascontiguousarray(x)


def ulysses_anything_permute(x, degree: int, direction: int, heads: int = None, fill=0):
    """Ulysses Anything regroup as a byte-exact layout permute.
    direction +1: x [B, S, H, D] -> [G, B, S, ceil(H/G), D]; padding slots
    hold ``fill``.  direction -1: x [G, B, S, ceil(H/G), D] -> [B, S, H, D];
    ``heads`` = H is required (padding slots are never read)."""
    raw = _raw(x)
    G = int(degree)
    if G < 1:
        raise OracleError("the Ulysses degree must be >= 1")
    if direction == 1:
        if raw.ndim != 4:
            raise OracleError("forward permute takes [B, S, H, D]")
        b, s, h, d = raw.shape
        out_shape = (G, b, s, -(-h // G), d)
        y = np.full(out_shape, fill, dtype=raw.dtype)
    elif direction == -1:
        if raw.ndim != 5 or raw.shape[0] != G or heads is None:
            raise OracleError("inverse permute takes [G, B, S, ceil(H/G), D] and H")
        _, b, s, hm, d = raw.shape
        h = int(heads)
        if hm != -(-h // G):
            raise OracleError("grouped tensor must have ceil(H/G) head slots")
        y = np.empty((b, s, h, d), dtype=raw.dtype)
    else:
        raise OracleError("direction must be +1 or -1")
    _check(_load().cpo_ulysses_anything_permute(_ptr(raw), _ptr(y), b, s, h, d, G, direction,
                                                raw.dtype.itemsize))
    if hasattr(x, "detach"):
        import torch
        yt = torch.from_numpy(y)
        return yt.view(x.dtype) if yt.dtype != x.dtype else yt
    return y


def ulysses_anything(q, k, v, degree: int, scale=None, causal=False):
    """Ulysses Anything attention as the steps of Diffusers "Context
    parallelism", "Ulysses Anything Attention": regroup q, k, v [B, S, H, D]
    into G head groups of tensor_split sizes (``ulysses_anything_permute``),
    attention of every group over its own heads and the full sequence
    (``attention``), inverse regroup.  Returns (out [B, S, H, D] float64,
    lse [G, B, ceil(H/G), S] with NaN in the padding slots)."""
    G = int(degree)
    B, S, H, D = np.shape(q)
    start = ulysses_anything_heads(H, G)
    qg, kg, vg = (ulysses_anything_permute(_f64(x), G, 1) for x in (q, k, v))
    hm = qg.shape[3]
    og = np.zeros_like(qg)
    lse = np.full((G, B, hm, S), np.nan)
    for g in range(G):
        hg = start[g + 1] - start[g]
        if hg == 0:
            continue
        to_bhsd = lambda t: np.ascontiguousarray(np.transpose(t[g, :, :, :hg], (0, 2, 1, 3)))
        o, l = attention(to_bhsd(qg), to_bhsd(kg), to_bhsd(vg), scale, causal=causal)
        og[g, :, :, :hg] = np.transpose(o, (0, 2, 1, 3))
        lse[g, :, :hg] = l
    return ulysses_anything_permute(og, G, -1, heads=H), lse


def num_threads() -> int:
    return int(_load().cpo_num_threads())
