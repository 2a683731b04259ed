"""PyTorch-facing binding of libcpattn.so.

Argument marshalling only: every function here allocates outputs with
PyTorch when the caller did not pass them, describes the tensors to the C ABI
and calls it on the current CUDA stream.  All computation runs in the CUDA
kernels; CPU tensors are rejected (there is no CPU path).
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _lib
from ._lib import CpattnError, check, describe

_DTYPES = {torch.float32: _lib.F32, torch.bfloat16: _lib.BF16}


def _code(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"dtype {t.dtype} is not supported (float32 or bfloat16)") from None


def _desc(t: torch.Tensor) -> _lib.CTensor:
    if not t.is_cuda:
        raise ValueError("cpattn runs on CUDA tensors only (no CPU path)")
    return describe(t.data_ptr(), _code(t), t.shape, t.stride())


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _scale(scale: Optional[float]) -> float:
    return 0.0 if scale is None else float(scale)


def partial(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: Optional[float] = None,
            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """One ring step: attention of q [B,H,S_q,D] against one K/V chunk
    [B,H,S_kv,D].  Returns (out f32 [B,H,S_q,D], lse f32 [B,H,S_q])."""
    lib = _lib.load()
    B, H, S, D = q.shape
    if out is None:
        out = torch.empty(B, H, S, D, device=q.device, dtype=torch.float32)
    if lse is None:
        lse = torch.empty(B, H, S, device=q.device, dtype=torch.float32)
    dq, dk, dv, do, dl = _desc(q), _desc(k), _desc(v), _desc(out), _desc(lse)
    check(lib.cpattn_partial(dq, dk, dv, _scale(scale), do, dl, _stream_handle(stream)),
          "cpattn_partial")
    return out, lse


def merge(out_a: torch.Tensor, lse_a: torch.Tensor, out_b: torch.Tensor, lse_b: torch.Tensor,
          stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """LSE merge of two f32 partials, in place into (out_a, lse_a)."""
    lib = _lib.load()
    da, la, db, lb = _desc(out_a), _desc(lse_a), _desc(out_b), _desc(lse_b)
    check(lib.cpattn_merge(da, la, db, lb, _stream_handle(stream)), "cpattn_merge")
    return out_a, lse_a


def ring_workspace_bytes(q: torch.Tensor, ring_degree: int) -> int:
    lib = _lib.load()
    return int(lib.cpattn_ring_workspace_bytes(describe(0, _code(q), q.shape, q.stride()),
                                               int(ring_degree)))


def ring(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, ring_degree: int = 1,
         ring_anything: bool = False, scale: Optional[float] = None,
         out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
         workspace: Optional[torch.Tensor] = None,
         stream: Optional[torch.cuda.Stream] = None,
         causal: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """The ring schedule on one GPU: q [B,H,S_q,D], k, v [B,H,S_kv,D].
    causal: query i attends keys j <= i (cpattn_ring_causal).
    Returns (out [B,H,S_q,D] in q's dtype, lse f32 [B,H,S_q])."""
    lib = _lib.load()
    B, H, S, D = q.shape
    if out is None:
        out = torch.empty(B, H, S, D, device=q.device, dtype=q.dtype)
    if lse is None:
        lse = torch.empty(B, H, S, device=q.device, dtype=torch.float32)
    need = ring_workspace_bytes(q, ring_degree)
    if workspace is None and need > 0:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    dq, dk, dv, do, dl = _desc(q), _desc(k), _desc(v), _desc(out), _desc(lse)
    fn = lib.cpattn_ring_causal if causal else lib.cpattn_ring
    check(fn(dq, dk, dv, _scale(scale), int(ring_degree), int(bool(ring_anything)),
             do, dl, ws_ptr, ws_bytes, _stream_handle(stream)),
          "cpattn_ring_causal" if causal else "cpattn_ring")
    return out, lse


def prepare_ring(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, ring_degree: int = 1,
                 ring_anything: bool = False, scale: Optional[float] = None,
                 out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None, causal: bool = False):
    """``ring`` with its argument descriptors built once: returns a callable
    that issues the same cpattn_ring (or cpattn_ring_causal) call on the
    same tensors and stream each time it is called, so repeated steps cost
    one foreign-function call of host time.  The callable's ``out`` and
    ``lse`` attributes are the output tensors; it keeps every tensor it was
    given alive."""
    lib = _lib.load()
    B, H, S, D = q.shape
    if out is None:
        out = torch.empty(B, H, S, D, device=q.device, dtype=q.dtype)
    if lse is None:
        lse = torch.empty(B, H, S, device=q.device, dtype=torch.float32)
    need = ring_workspace_bytes(q, ring_degree)
    if workspace is None and need > 0:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    fn = lib.cpattn_ring_causal if causal else lib.cpattn_ring
    name = "cpattn_ring_causal" if causal else "cpattn_ring"
    args = (_desc(q), _desc(k), _desc(v), _scale(scale), int(ring_degree),
            int(bool(ring_anything)), _desc(out), _desc(lse), ws_ptr, ws_bytes,
            _stream_handle(stream))

    def call():
        check(fn(*args), name)

    call.out, call.lse = out, lse
    call.keep = (q, k, v, out, lse, workspace)
    return call


def ring_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, ring_degree: int = 1,
                 ring_anything: bool = False, scale: Optional[float] = None,
                 out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """``ring`` without a workspace argument, for callers that cannot
    allocate device memory: the library's own fixed device array (see
    ``ring_noalloc_max_workspace_bytes``) holds the running merged result.
    Pass ``out`` and ``lse`` to avoid any allocation here as well.  Calls
    that overlap on the GPU share that array and race."""
    lib = _lib.load()
    B, H, S, D = q.shape
    if out is None:
        out = torch.empty(B, H, S, D, device=q.device, dtype=q.dtype)
    if lse is None:
        lse = torch.empty(B, H, S, device=q.device, dtype=torch.float32)
    dq, dk, dv, do, dl = _desc(q), _desc(k), _desc(v), _desc(out), _desc(lse)
    check(lib.cpattn_ring_noalloc(dq, dk, dv, _scale(scale), int(ring_degree),
                                  int(bool(ring_anything)), do, dl, _stream_handle(stream)),
          "cpattn_ring_noalloc")
    return out, lse


def ring_noalloc_max_workspace_bytes() -> int:
    return int(_lib.load().cpattn_ring_noalloc_max_workspace_bytes())


def ulysses_permute(x: torch.Tensor, degree: int, direction: int,
                    out: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """direction +1: [B,S,H,D] -> [G,B,S,H/G,D]; direction -1: the inverse."""
    lib = _lib.load()
    if out is None:
        if direction == 1:
            B, S, H, D = x.shape
            out = torch.empty(degree, B, S, H // max(degree, 1), D, device=x.device, dtype=x.dtype)
        else:
            G, B, S, Hg, D = x.shape
            out = torch.empty(B, S, G * Hg, D, device=x.device, dtype=x.dtype)
    dx, dy = _desc(x), _desc(out)
    check(lib.cpattn_ulysses_permute(dx, int(degree), int(direction), dy, _stream_handle(stream)),
          "cpattn_ulysses_permute")
    return out


def _descs(ts) -> ctypes.Array:
    arr = (_lib.CTensor * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = _desc(t)
    return arr


def ulysses_permute_batch(xs, degree: int, direction: int, outs=None,
                          stream: Optional[torch.cuda.Stream] = None) -> list:
    """ulysses_permute of up to 4 tensors of one shape and dtype in one
    launch (cpattn_ulysses_permute_batch); returns the outputs in order."""
    lib = _lib.load()
    outs = list(outs) if outs is not None else [None] * len(xs)
    for i, x in enumerate(xs):
        if outs[i] is None:
            if direction == 1:
                B, S, H, D = x.shape
                outs[i] = torch.empty(degree, B, S, H // max(degree, 1), D, device=x.device,
                                      dtype=x.dtype)
            else:
                G, B, S, Hg, D = x.shape
                outs[i] = torch.empty(B, S, G * Hg, D, device=x.device, dtype=x.dtype)
    check(lib.cpattn_ulysses_permute_batch(len(xs), _descs(xs), int(degree), int(direction),
                                           _descs(outs), _stream_handle(stream)),
          "cpattn_ulysses_permute_batch")
    return outs


def grouped_as_bhsd(t: torch.Tensor) -> torch.Tensor:
    """[G,B,S,H/G,D] -> strided view [G*B, H/G, S, D] (no copy)."""
    G, B, S, Hg, D = t.shape
    return t.view(G * B, S, Hg, D).permute(0, 2, 1, 3)


def unified_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, ulysses_degree: int,
                      ring_degree: int = 1, scale: Optional[float] = None,
                      stream: Optional[torch.cuda.Stream] = None,
                      buffers: Optional[dict] = None,
                      causal: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """Unified (Ulysses x Ring) attention on one GPU (Diffusers "Context
    parallelism", "Unified Attention": an all-to-all regroups heads and
    tokens, Ring Attention runs on the result, the all-to-all is reversed).
    q, k, v [B,S,H,D]: permute into G = ulysses_degree head groups, ring
    attention with ring_degree chunks over each group's full sequence (one
    launch for all groups), inverse permute of the output.  ring_degree 1 is
    plain Ulysses.  Returns (out [B,S,H,D], lse f32 [G*B, H/G, S]).
    `buffers` (a dict) keeps the grouped tensors and the ring workspace
    between calls."""
    B, S, H, D = q.shape
    G, R = int(ulysses_degree), int(ring_degree)
    bufs = buffers if buffers is not None else {}

    def buf(name, shape, dtype):
        t = bufs.get(name)
        if t is None or tuple(t.shape) != tuple(shape) or t.dtype != dtype:
            t = torch.empty(shape, device=q.device, dtype=dtype)
            bufs[name] = t
        return t

    gshape = (G, B, S, H // max(G, 1), D)
    # q, k and v regrouped by one launch
    qg, kg, vg = ulysses_permute_batch(
        (q, k, v), G, 1, outs=(buf("q", gshape, q.dtype), buf("k", gshape, q.dtype),
                               buf("v", gshape, q.dtype)), stream=stream)
    og = buf("o", gshape, q.dtype)
    lse = buf("lse", (G * B, H // G, S), torch.float32)
    qv = grouped_as_bhsd(qg)
    need = ring_workspace_bytes(qv, R)
    ws = buf("ws", (max(need, 16),), torch.uint8) if need > 0 else None
    ring(qv, grouped_as_bhsd(kg), grouped_as_bhsd(vg), R, False, scale,
         out=grouped_as_bhsd(og), lse=lse, workspace=ws, stream=stream, causal=causal)
    out = ulysses_permute(og, G, -1, out=buf("out", (B, S, H, D), q.dtype), stream=stream)
    return out, lse


def prepare_unified(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, ulysses_degree: int,
                    ring_degree: int = 1, scale: Optional[float] = None,
                    stream: Optional[torch.cuda.Stream] = None, causal: bool = False):
    """``unified_attention`` with its buffers allocated and its three calls'
    descriptors built once (batched regroup of q, k, v; ring over the grouped
    view; inverse regroup).  Returns a callable issuing the three calls; its
    ``out`` and ``lse`` attributes are the results."""
    lib = _lib.load()
    B, S, H, D = q.shape
    G, R = int(ulysses_degree), int(ring_degree)
    gshape = (G, B, S, H // max(G, 1), D)
    qg, kg, vg, og = (torch.empty(gshape, device=q.device, dtype=q.dtype) for _ in range(4))
    lse = torch.empty(G * B, H // G, S, device=q.device, dtype=torch.float32)
    out = torch.empty(B, S, H, D, device=q.device, dtype=q.dtype)
    h = _stream_handle(stream)
    fwd = (3, _descs((q, k, v)), G, 1, _descs((qg, kg, vg)), h)
    inner = prepare_ring(grouped_as_bhsd(qg), grouped_as_bhsd(kg), grouped_as_bhsd(vg), R, False,
                         scale, out=grouped_as_bhsd(og), lse=lse, stream=stream, causal=causal)
    inv = (_desc(og), G, -1, _desc(out), h)

    def call():
        check(lib.cpattn_ulysses_permute_batch(*fwd), "cpattn_ulysses_permute_batch")
        inner()
        check(lib.cpattn_ulysses_permute(*inv), "cpattn_ulysses_permute")

    call.out, call.lse = out, lse
    call.keep = (q, k, v, qg, kg, vg, og, inner)
    return call


def ulysses_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, degree: int,
                      scale: Optional[float] = None,
                      stream: Optional[torch.cuda.Stream] = None,
                      buffers: Optional[dict] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Ulysses on one GPU (Diffusers "Context parallelism", "Ulysses
    Attention"): permute q, k, v [B,S,H,D] into G head groups, full attention
    per group (one launch over all groups), inverse permute of the output.
    Returns (out [B,S,H,D], lse f32 [G*B, H/G, S])."""
    return unified_attention(q, k, v, degree, 1, scale, stream, buffers)


def ulysses_anything_permute(x: torch.Tensor, degree: int, direction: int,
                             heads: Optional[int] = None, out: Optional[torch.Tensor] = None,
                             stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Ulysses Anything regroup (cpattn_ulysses_anything_permute).
    direction +1: [B,S,H,D] -> [G,B,S,ceil(H/G),D] (padding slots untouched);
    direction -1: [G,B,S,ceil(H/G),D] -> [B,S,H,D], ``heads`` = H required
    unless ``out`` is given."""
    lib = _lib.load()
    G = int(degree)
    if out is None:
        if direction == 1:
            B, S, H, D = x.shape
            out = torch.empty(G, B, S, -(-H // max(G, 1)), D, device=x.device, dtype=x.dtype)
        else:
            if heads is None:
                raise ValueError("the inverse regroup needs heads (or out)")
            _, B, S, _, D = x.shape
            out = torch.empty(B, S, int(heads), D, device=x.device, dtype=x.dtype)
    dx, dy = _desc(x), _desc(out)
    check(lib.cpattn_ulysses_anything_permute(dx, G, int(direction), dy, _stream_handle(stream)),
          "cpattn_ulysses_anything_permute")
    return out


def ulysses_anything_permute_batch(xs, degree: int, direction: int, heads: Optional[int] = None,
                                   outs=None,
                                   stream: Optional[torch.cuda.Stream] = None) -> list:
    """ulysses_anything_permute of up to 4 tensors of one shape and dtype in
    one launch (cpattn_ulysses_anything_permute_batch); returns the outputs."""
    lib = _lib.load()
    G = int(degree)
    outs = list(outs) if outs is not None else [None] * len(xs)
    for i, x in enumerate(xs):
        if outs[i] is None:
            if direction == 1:
                B, S, H, D = x.shape
                outs[i] = torch.empty(G, B, S, -(-H // max(G, 1)), D, device=x.device,
                                      dtype=x.dtype)
            else:
                if heads is None:
                    raise ValueError("the inverse regroup needs heads (or outs)")
                _, B, S, _, D = x.shape
                outs[i] = torch.empty(B, S, int(heads), D, device=x.device, dtype=x.dtype)
    check(lib.cpattn_ulysses_anything_permute_batch(len(xs), _descs(xs), G, int(direction),
                                                    _descs(outs), _stream_handle(stream)),
          "cpattn_ulysses_anything_permute_batch")
    return outs


def ulysses_anything_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, degree: int,
                               scale: Optional[float] = None,
                               stream: Optional[torch.cuda.Stream] = None,
                               buffers: Optional[dict] = None,
                               causal: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """Ulysses Anything on one GPU (Diffusers "Context parallelism", "Ulysses
    Anything Attention": no divisibility of H or S by G; ring_degree 1).
    q, k, v [B,S,H,D]: regroup into G tensor_split head groups padded to
    ceil(H/G) slots, attention of every group over its own heads (one launch,
    padding slots skipped), inverse regroup.  Returns (out [B,S,H,D],
    lse f32 [G,B,ceil(H/G),S] whose padding slots are unspecified)."""
    lib = _lib.load()
    B, S, H, D = q.shape
    G = int(degree)
    hm = -(-H // max(G, 1))
    bufs = buffers if buffers is not None else {}

    def buf(name, shape, dtype):
        t = bufs.get(name)
        if t is None or tuple(t.shape) != tuple(shape) or t.dtype != dtype:
            t = torch.empty(shape, device=q.device, dtype=dtype)
            bufs[name] = t
        return t

    gshape = (G, B, S, hm, D)
    # q, k and v regrouped by one launch
    qg, kg, vg = ulysses_anything_permute_batch(
        (q, k, v), G, 1, outs=(buf("q", gshape, q.dtype), buf("k", gshape, q.dtype),
                               buf("v", gshape, q.dtype)), stream=stream)
    og = buf("o", gshape, q.dtype)
    lse = buf("lse", (G, B, hm, S), torch.float32)
    check(lib.cpattn_ulysses_anything_attention(_desc(qg), _desc(kg), _desc(vg), _scale(scale), H,
                                                int(bool(causal)), _desc(og), _desc(lse),
                                                _stream_handle(stream)),
          "cpattn_ulysses_anything_attention")
    out = ulysses_anything_permute(og, G, -1, out=buf("out", (B, S, H, D), q.dtype), stream=stream)
    return out, lse


def prepare_ulysses_anything(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, degree: int,
                             scale: Optional[float] = None,
                             stream: Optional[torch.cuda.Stream] = None, causal: bool = False):
    """``ulysses_anything_attention`` with its buffers allocated and its
    three calls' descriptors built once; returns a callable issuing them,
    whose ``out`` and ``lse`` attributes are the results."""
    lib = _lib.load()
    B, S, H, D = q.shape
    G = int(degree)
    hm = -(-H // max(G, 1))
    gshape = (G, B, S, hm, D)
    qg, kg, vg, og = (torch.empty(gshape, device=q.device, dtype=q.dtype) for _ in range(4))
    lse = torch.empty(G, B, hm, S, device=q.device, dtype=torch.float32)
    out = torch.empty(B, S, H, D, device=q.device, dtype=q.dtype)
    h = _stream_handle(stream)
    fwd = (3, _descs((q, k, v)), G, 1, _descs((qg, kg, vg)), h)
    attn = (_desc(qg), _desc(kg), _desc(vg), _scale(scale), H, int(bool(causal)), _desc(og),
            _desc(lse), h)
    inv = (_desc(og), G, -1, _desc(out), h)

    def call():
        check(lib.cpattn_ulysses_anything_permute_batch(*fwd),
              "cpattn_ulysses_anything_permute_batch")
        check(lib.cpattn_ulysses_anything_attention(*attn), "cpattn_ulysses_anything_attention")
        check(lib.cpattn_ulysses_anything_permute(*inv), "cpattn_ulysses_anything_permute")

    call.out, call.lse = out, lse
    call.keep = (q, k, v, qg, kg, vg, og)
    return call


def last_device_status(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronises the stream and returns (and clears) the device error word
    status: 0 = ok, 9 = a kernel-side wait timed out."""
    return int(_lib.load().cpattn_last_device_status(_stream_handle(stream)))


def set_wait_timeout_ns(ns: int) -> None:
    _lib.load().cpattn_set_wait_timeout_ns(int(ns))


__all__ = ["partial", "merge", "ring", "ring_workspace_bytes", "ring_noalloc", "prepare_ring",
           "prepare_unified", "prepare_ulysses_anything",
           "ring_noalloc_max_workspace_bytes", "ulysses_permute", "unified_attention",
           "ulysses_attention", "grouped_as_bhsd", "last_device_status", "set_wait_timeout_ns",
           "CpattnError"]
