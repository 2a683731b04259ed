"""Whole-tensor expected outputs of the full-size workloads, from the oracle.

TEST INFRASTRUCTURE ONLY.  This script calls nothing but the fp64 oracle of
this directory and the seeded input generator (``workloads.py``); it never
loads the CUDA library.  The GPU parity tests read what it writes and compare
every element of the CUDA path's outputs against it.

Each case is computed once per machine in fp64 and stored as float32 ``.npy``
files (out and lse) in a cache directory kept out of version control
(``$CPATTN_ORACLE_CACHE``, default ``_cache/oracle`` at the repository root).
A case is recomputed when its file is missing or when the oracle source, the
case's definition or the generated inputs themselves changed: the stored
fingerprint covers the bytes of q, k and v, because the seeded generator's
float32 draws are not bit-identical across CPU architectures and PyTorch
builds (a cache made on one machine is never trusted on another).  Storing
fp32 rounds the fp64 result by at most 2^-24 relative, far inside the
tolerances it is compared at (1e-2 or 2e-3, and 1e-3).

Expected values (page title, section):

* Ring workloads (plain, Ring Anything, causal) and the single partial: full
  softmax attention over every key, ``oracle.attention``: the definition the
  ring reaches exactly, since every query meets every key/value block once
  (Diffusers "Context parallelism", "Ring Attention"); the ParaAttention
  README's correctness script likewise compares the sharded result with full
  scaled_dot_product_attention.  The oracle's pins show that its chunked
  path equals this definition to 1e-12.
* Ulysses and Unified workloads: the oracle's composition of the pages'
  steps, ``oracle.unified`` (regroup, ring within each head group, inverse
  regroup; Diffusers "Context parallelism", "Ulysses Attention" and
  "Unified Attention").
* Ulysses Anything: ``oracle.ulysses_anything`` (same guide, "Ulysses
  Anything Attention").

Usage:  python oracle/make_cache.py [case ...]   (no argument: every case)
"""
from __future__ import annotations

import hashlib
import json
import os
import sys
import time

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(_HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from workloads import WORKLOADS, make_qkv  # noqa: E402

CACHE_DIR = os.environ.get("CPATTN_ORACLE_CACHE", os.path.join(ROOT, "_cache", "oracle"))

# case -> (input shape, dtype name, seed, how the expected value is computed)
#   ("attention", causal)                      full softmax attention, [B, H, S, D]
#   ("unified", ulysses_degree, ring_degree)   [B, S, H, D] inputs
#   ("ulysses_anything", ulysses_degree)       [B, S, H, D] inputs
CASES = {
    "flux_ring": (WORKLOADS["flux_ring"].shape, "bf16", 0, ("attention", False)),
    "flux_ring_causal": (WORKLOADS["flux_ring_causal"].shape, "bf16", 0, ("attention", True)),
    "uneven_ring": (WORKLOADS["uneven_ring"].shape, "bf16", 0, ("attention", False)),
    "video_ring": (WORKLOADS["video_ring"].shape, "bf16", 0, ("attention", False)),
    "ulysses": (WORKLOADS["ulysses"].shape, "bf16", 0, ("unified", 4, 1)),
    "unified": (WORKLOADS["unified"].shape, "bf16", 0, ("unified", 2, 2)),
    "ulysses_anything": (WORKLOADS["ulysses_anything"].shape, "bf16", 0,
                         ("ulysses_anything", 5)),
    # bf16 D = 64 over several waves of CTAs (not one of the named workloads)
    "d64_ring": ((2, 24, 4608, 64), "bf16", 61, ("attention", False)),
    # bf16 D = 64 (P in TMEM columns of its own): causal, and Ring Anything
    "d64_causal": ((1, 24, 4608, 64), "bf16", 63, ("attention", True)),
    "d64_uneven": ((2, 24, 4609, 64), "bf16", 65, ("attention", False)),
    # fp32 inputs (3xTF32): D = 128 (one 128-row query tile per CTA, 64-key
    # tiles) over four waves with a ragged tail, and D = 64 causal
    "f32_d128_ring": ((2, 8, 4609, 128), "f32", 71, ("attention", False)),
    "f32_d64_causal": ((1, 8, 4096, 64), "f32", 73, ("attention", True)),
}


def _torch_dtype(name):
    import torch
    return torch.float32 if name == "f32" else torch.bfloat16


def inputs(case: str):
    """The case's seeded q, k, v (CPU tensors in the case's dtype)."""
    shape, dt, seed, _ = CASES[case]
    return make_qkv(shape, _torch_dtype(dt), seed)


def _fingerprint(case: str, qkv=None) -> str:
    h = hashlib.sha256()
    for path in (os.path.join(_HERE, "cpattn_oracle.c"), os.path.join(_HERE, "__init__.py"),
                 os.path.join(ROOT, "workloads.py")):
        with open(path, "rb") as f:
            h.update(f.read())
    h.update(repr(CASES[case]).encode())
    import torch
    for t in (qkv if qkv is not None else inputs(case)):
        h.update(t.contiguous().view(torch.uint8).numpy().tobytes())
    return h.hexdigest()[:16]


def _paths(case: str):
    base = os.path.join(CACHE_DIR, case)
    return base + ".out.npy", base + ".lse.npy", base + ".json"


def _compute(case: str, qkv):
    shape, _, _, how = CASES[case]
    q, k, v = qkv
    if how[0] == "attention":
        d = shape[-1]
        return oracle.attention(q, k, v, d ** -0.5, causal=how[1])
    if how[0] == "unified":
        d = shape[-1]
        return oracle.unified(q, k, v, how[1], how[2], d ** -0.5)
    if how[0] == "ulysses_anything":
        d = shape[-1]
        return oracle.ulysses_anything(q, k, v, how[1], d ** -0.5)
    raise KeyError(case)


def fresh(case: str, qkv=None) -> bool:
    po, pl, pm = _paths(case)
    if not (os.path.exists(po) and os.path.exists(pl) and os.path.exists(pm)):
        return False
    with open(pm) as f:
        return json.load(f).get("fingerprint") == _fingerprint(case, qkv)


def make(case: str, verbose: bool = False) -> dict:
    """Compute and store one case (unless already fresh); returns its meta."""
    po, pl, pm = _paths(case)
    qkv = inputs(case)
    if fresh(case, qkv):
        with open(pm) as f:
            return json.load(f)
    os.makedirs(CACHE_DIR, exist_ok=True)
    t0 = time.perf_counter()
    out, lse = _compute(case, qkv)
    dt = time.perf_counter() - t0
    tag = f".{os.getpid()}.tmp"
    for arr, path in ((out, po), (lse, pl)):
        with open(path + tag, "wb") as f:
            np.save(f, np.asarray(arr, dtype=np.float32))
        os.replace(path + tag, path)
    meta = {"case": case, "fingerprint": _fingerprint(case, qkv), "oracle_seconds": dt,
            "threads": oracle.num_threads(), "out_shape": list(np.shape(out)),
            "lse_shape": list(np.shape(lse))}
    with open(pm + tag, "w") as f:
        json.dump(meta, f)
    os.replace(pm + tag, pm)
    if verbose:
        print(f"{case}: {dt:.1f} s on {meta['threads']} threads", flush=True)
    return meta


def expected(case: str):
    """(out, lse) float32 arrays of the case, computed first if needed."""
    make(case)
    po, pl, _ = _paths(case)
    return np.load(po, mmap_mode="r"), np.load(pl, mmap_mode="r")


def main(argv):
    cases = argv or list(CASES)
    for c in cases:
        if c not in CASES:
            raise SystemExit(f"unknown case {c!r}; cases: {', '.join(CASES)}")
    for c in cases:
        make(c, verbose=True)
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
