"""Benchmark of the context-parallel attention hot path on GB300.

One step = one pass of the hot path over one batch of the FLUX-like joint
attention workload (bf16 [1, 24, 4608, 128], ring_degree 2): the in-kernel
ring (chunk partition, Q K^T, online softmax, P V, per-chunk partial + fp32
LSE merge, epilogue) in one cpattn_ring launch.  Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload flux_ring] [--no-aux] [--no-cpu-baseline]
  python bench.py --sweep      # one JSON line per shape of a size sweep

Timing: CUDA events on the launching stream around each step; the L2 is
flushed (a 512 MiB write) between timed steps, outside the events.  Inputs
are resident in HBM before the timed region.  A step is one prepared library
call (descriptors built once).  nvidia-smi samples SM clocks and throttle
reasons from an untimed one-second soak of the same step through the end of
the timed region.  Under torchrun each rank runs
an independent replica on its own GPU (the hot path has no exchange step on
one GPU); value = all ranks' FLOPs / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 512 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in ("attn_fwd.cu", "ptx.cuh", "tmem_ops.cuh", "internal.h"):
        with open(os.path.join(ROOT, "context_attention_partial_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the attention kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"attn_fwd_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s+source_sha:\s*([0-9a-f]+)", text)
    if not m or m.group(2) != kernel_source_hash():
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            try:
                power.append(float(parts[3]))
            except ValueError:
                pass
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        # samples under load: power above half of the largest reading (an
        # idle GPU draws a small fraction of what this kernel does)
        if len(power) == len(sm) and power:
            loaded = [c for c, pw in zip(sm, power) if pw >= 0.5 * max(power)] or sm
        else:
            loaded = sm
        out = {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
               "samples": len(sm), "samples_under_load": len(loaded)}
        if power:
            out["power_w_median"] = statistics.median(power)
            out["power_w_max"] = max(power)
        return out


def dist_setup(n_gpus: int):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce_device():
    import torch.distributed as dist
    return "cpu" if dist.get_backend() == "gloo" else "cuda"


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time (timing is max over ranks)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], device=_reduce_device(), dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    """Work of all ranks together (value is the whole-job aggregate)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], device=_reduce_device(), dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def workload_config(w, world: int = 1) -> dict:
    """The workload the line is measured on (the same dict on both arms)."""
    return {"workload": w.description, "name": w.name, "batch": w.batch, "heads": w.heads,
            "seq_len": w.seq, "head_dim": w.head_dim, "ring_degree": w.ring_degree,
            "ring_anything": w.ring_anything,
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def time_steps(fn, steps: int, flush: torch.Tensor, stream):
    """Per-step CUDA events on `stream`; the L2 flush runs between steps,
    outside the events.  Returns the list of step times in ms."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for i in range(steps):
        flush.fill_(i & 0xFF)
        evs[i][0].record(stream)
        fn()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def ring_workload_step(name, dev):
    import context_attention_partial_gb300 as cp
    from workloads import make_workload
    w, q, k, v = make_workload(name, seed=0)
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], device=dev, dtype=torch.float32)
    need = cp.ring_workspace_bytes(q, w.ring_degree)
    ws = torch.empty(max(need, 16), device=dev, dtype=torch.uint8)
    # descriptors built once: a step is one call into the library, so host
    # marshalling stays far shorter than the L2 flush that precedes it
    step = cp.prepare_ring(q, k, v, w.ring_degree, w.ring_anything, out=out, lse=lse,
                           workspace=ws, causal=w.causal)
    return w, step, (q, k, v, out, lse, ws)


def ulysses_step(dev, name="ulysses"):
    """Ulysses (ring_degree 1), Unified (ring_degree > 1) or Ulysses Anything
    step: one batched regroup of q, k and v, one attention launch over all
    head groups, one inverse regroup."""
    import context_attention_partial_gb300 as cp
    from workloads import make_workload
    w, q, k, v = make_workload(name, seed=0)
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    if w.ulysses_anything:
        step = cp.prepare_ulysses_anything(q, k, v, w.ulysses_degree)
    else:
        step = cp.prepare_unified(q, k, v, w.ulysses_degree, w.ring_degree)
    return w, step, (q, k, v)


def e2e_ring(name, dev, steps, stream):
    """Same metric through the public API with HOST buffers: every step
    copies its q, k, v from pinned host memory to the device, calls the ring
    and copies out and lse back to pinned host memory, all inside the timed
    region.  Steps are pipelined the way a serving loop would run them: two
    device buffer sets, the host->device copies on one stream, the ring on a
    second and the device->host copies on a third, events guarding every
    buffer's reuse, so step i's copies overlap step i-1's attention."""
    import context_attention_partial_gb300 as cp
    from workloads import make_workload
    w, q, k, v = make_workload(name, seed=0)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    nbuf = 2
    dins = [tuple(torch.empty_like(hq, device=dev) for _ in range(3)) for _ in range(nbuf)]
    douts = [torch.empty_like(hq, device=dev) for _ in range(nbuf)]
    dlses = [torch.empty(q.shape[:3], device=dev, dtype=torch.float32) for _ in range(nbuf)]
    houts = [torch.empty_like(hq).pin_memory() for _ in range(nbuf)]
    hlses = [torch.empty(q.shape[:3], dtype=torch.float32).pin_memory() for _ in range(nbuf)]
    wss = [torch.empty(max(cp.ring_workspace_bytes(hq, w.ring_degree), 16), device=dev,
                       dtype=torch.uint8) for _ in range(nbuf)]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]
    ev_comp = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]
    used = [False] * nbuf

    def step(i):
        j = i % nbuf
        dq, dk, dv = dins[j]
        with torch.cuda.stream(s_in):
            if used[j]:
                s_in.wait_event(ev_comp[j])        # step i-2 has read these inputs
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            ev_in[j].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev_in[j])
            if used[j]:
                s_comp.wait_event(ev_out[j])       # step i-2's results have left
            cp.ring(dq, dk, dv, w.ring_degree, w.ring_anything, out=douts[j], lse=dlses[j],
                    workspace=wss[j], stream=s_comp)
            ev_comp[j].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[j])
            houts[j].copy_(douts[j], non_blocking=True)
            hlses[j].copy_(dlses[j], non_blocking=True)
            ev_out[j].record(s_out)
        used[j] = True

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for i in range(steps):
        step(i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_comp)
    end.record(s_out)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = houts[0].numel() * houts[0].element_size() + hlses[0].numel() * hlses[0].element_size()
    return ms, h2d, d2h, w.flops


def time_graph(fn, calls: int, flush: torch.Tensor, stream):
    """`calls` back-to-back calls captured into one CUDA graph (so host-side
    argument marshalling does not pace the GPU), replayed after an L2 flush
    between two CUDA events; returns ms per call.  Callers rotate buffer sets
    whose total exceeds L2, so every call streams from HBM."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(calls):
            fn()
    graph.replay()
    torch.cuda.synchronize()
    flush.fill_(7)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    graph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / calls


def aux_measurements(dev, stream, peaks):
    """Secondary lines: merge and permute HBM bandwidth, other workloads."""
    import context_attention_partial_gb300 as cp
    from workloads import make_partials
    aux = {}
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    # merge at the FLUX shape and the video shape; rotating sets > L2
    for label, shape in (("merge_flux", (1, 24, 4608)), ("merge_video", (1, 24, 32768))):
        sets = []
        n_sets = 4 if shape[2] < 10000 else 2
        for s in range(n_sets):
            o_a, l_a, o_b, l_b = make_partials(shape, 128, seed=s)
            sets.append((o_a.to(dev), l_a.to(dev), o_b.to(dev), l_b.to(dev)))
        rows = shape[0] * shape[1] * shape[2]
        nbytes = 3 * rows * 128 * 4 + 3 * rows * 4
        it = [0]

        def mstep():
            a = sets[it[0] % n_sets]
            it[0] += 1
            cp.merge(*a)
        for _ in range(5):
            mstep()
        ms = time_graph(mstep, 40, flush, stream)
        gbs = nbytes / (ms * 1e-3) / 1e9
        aux[label] = {"ms": ms, "GB/s": gbs, "bytes": nbytes, "frac_hbm": gbs / peaks["hbm_gbs"],
                      "timing": "40 calls in one CUDA graph over rotating sets > L2"}
        del sets
    # permute at the Ulysses workload, 8 rotating sets (453 MB > L2)
    from workloads import make_qkv
    xs = [make_qkv((1, 4608, 24, 128), torch.bfloat16, seed=s)[0].to(dev) for s in range(8)]
    ys = [torch.empty(4, 1, 4608, 6, 128, device=dev, dtype=torch.bfloat16) for _ in range(8)]
    it = [0]

    def pstep():
        i = it[0] % 8
        it[0] += 1
        cp.ulysses_permute(xs[i], 4, 1, out=ys[i])
    for _ in range(5):
        pstep()
    ms = time_graph(pstep, 80, flush, stream)
    nbytes = 2 * xs[0].numel() * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    aux["permute_ulysses"] = {"ms": ms, "GB/s": gbs, "bytes": nbytes,
                              "frac_hbm": gbs / peaks["hbm_gbs"],
                              "timing": "80 calls in one CUDA graph over 8 rotating sets > L2"}
    # q, k and v of a Ulysses step regrouped by one batched launch
    ys = [torch.empty(4, 1, 4608, 6, 128, device=dev, dtype=torch.bfloat16) for _ in range(8)]

    def bstep():
        # three sets the previous call did not touch: a set returns two calls
        # later at the earliest, after a whole other call's 170 MB (> L2)
        i = it[0]
        it[0] += 1
        sel = [(3 * i + j) % 8 for j in range(3)]
        cp.ulysses_permute_batch([xs[j] for j in sel], 4, 1, outs=[ys[j] for j in sel])
    for _ in range(5):
        bstep()
    ms = time_graph(bstep, 40, flush, stream)
    gbs = 3 * nbytes / (ms * 1e-3) / 1e9
    aux["permute_ulysses_qkv_batch"] = {"ms": ms, "GB/s": gbs, "bytes": 3 * nbytes,
                                        "frac_hbm": gbs / peaks["hbm_gbs"],
                                        "timing": "40 three-tensor calls in one CUDA graph, "
                                                  "each on 3 of 8 rotating sets that the "
                                                  "previous call did not touch"}
    # Ulysses Anything regroup (24 heads over 5 groups padded to 5 slots);
    # padding slots are not written, so the bytes are the same as above
    ys = [torch.empty(5, 1, 4608, 5, 128, device=dev, dtype=torch.bfloat16) for _ in range(8)]

    def astep():
        i = it[0] % 8
        it[0] += 1
        cp.ulysses_anything_permute(xs[i], 5, 1, out=ys[i])
    for _ in range(5):
        astep()
    ms = time_graph(astep, 80, flush, stream)
    gbs = nbytes / (ms * 1e-3) / 1e9
    aux["permute_ulysses_anything"] = {"ms": ms, "GB/s": gbs, "bytes": nbytes,
                                       "frac_hbm": gbs / peaks["hbm_gbs"],
                                       "timing": "80 calls in one CUDA graph over 8 rotating "
                                                 "sets > L2"}
    del xs, ys
    # the other attention workloads
    for name in ("uneven_ring", "video_ring", "tiny_ring", "flux_ring_causal"):
        w, step, keep = ring_workload_step(name, dev)
        for _ in range(3):
            step()
        times = time_steps(step, 10 if name == "video_ring" else 30, flush, stream)
        ms = statistics.median(times)
        aux[name] = {"ms": ms, "TFLOP/s": w.flops / (ms * 1e-3) / 1e12,
                     "frac_bf16_peak": w.flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"]}
        del keep
    for name in ("ulysses", "unified", "ulysses_anything"):
        w, step, keep = ulysses_step(dev, name)
        for _ in range(3):
            step()
        times = time_steps(step, 30, flush, stream)
        ms = statistics.median(times)
        aux[name] = {"ms": ms, "TFLOP/s": w.flops / (ms * 1e-3) / 1e12,
                     "launches_per_step": 3,
                     "frac_bf16_peak": w.flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"]}
        del keep
    return aux


def cpu_baseline(name, budget_s=12.0):
    """The oracle as it stands, on this host's cores, on a bounded sample of
    the workload: whole heads (every query row against all of that head's
    keys, through the ring path: partials per chunk + merge), as many heads
    as fit in about `budget_s` seconds."""
    import oracle
    from workloads import make_workload
    w, q, k, v = make_workload(name, seed=0)
    heads = [(b, h) for b in range(w.batch) for h in range(w.heads)]
    # calibrate on 256 rows of the first head
    b0, h0 = heads[0]
    t0 = time.perf_counter()
    oracle.ring(q[b0, h0:h0 + 1, :256], k[b0, h0:h0 + 1], v[b0, h0:h0 + 1],
                w.head_dim ** -0.5, w.ring_degree, w.ring_anything)
    per_head = (time.perf_counter() - t0) * w.seq / min(256, w.seq)
    n_heads = int(max(1, min(len(heads), budget_s / max(per_head, 1e-6))))
    t0 = time.perf_counter()
    for b, h in heads[:n_heads]:
        oracle.ring(q[b, h:h + 1], k[b, h:h + 1], v[b, h:h + 1], w.head_dim ** -0.5,
                    w.ring_degree, w.ring_anything)
    dt = time.perf_counter() - t0
    flops = 4.0 * n_heads * w.seq * w.seq * w.head_dim
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{n_heads} of {len(heads)} (batch, head) pairs of {name}, every query row "
                      f"against all {w.seq} keys (ring_degree {w.ring_degree}), fp64 C oracle, "
                      f"{dt:.1f} s"}


def run_ours(args):
    rank, world, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    import __graft_entry__
    __graft_entry__.build()
    peaks = load_peaks()
    stream = torch.cuda.current_stream()
    w, step, keep = ring_workload_step(args.workload, dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    import context_attention_partial_gb300 as cp
    assert cp.last_device_status() == 0

    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # clock soak: untimed steps for about args.soak_s seconds, so that
        # the sampler (one reading every 50 ms) sees the GPU under this
        # load; the timed region that follows is a few milliseconds long
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < args.soak_s:
            for _ in range(50):
                flush.fill_(2)
                step()
            torch.cuda.synchronize()
        t_soak = time.perf_counter() - t_soak
        t_wall = time.perf_counter()
        times = time_steps(step, args.steps, flush, stream)
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    torch.cuda.synchronize()
    total_ms = max_over_ranks(sum(times), world)
    ms_step = total_ms / args.steps
    flops_all = sum_over_ranks(w.flops * args.steps, world)
    value = flops_all / (total_ms * 1e-3) / 1e12
    kernel_ms = statistics.mean(times)
    achieved = w.flops / (kernel_ms * 1e-3) / 1e12
    traffic = profiled_traffic(args.workload)

    e2e = None
    if args.e2e:
        e2e_ms, h2d, d2h, fl = e2e_ring(args.workload, dev, max(5, min(args.steps, 50)), stream)
        e2e = {"value": fl / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "schedule": "pinned host buffers; copies in, ring, copies out on three streams, "
                           "two device buffer sets, step i's copies overlap step i-1's ring"}
    aux = aux_measurements(dev, stream, peaks) if (args.aux and rank == 0) else None
    cpu = cpu_baseline(args.workload) if (args.cpu_baseline and rank == 0 and world == 1) else None

    if rank == 0:
        line = {
            "metric": "ring-attention TFLOP/s (bf16, 1 GB300) and % of dense BF16 tensor peak",
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(w, world),
            "timing": {"l2": "flushed between timed steps (512 MiB write, outside the events)",
                       "events": "one CUDA event pair per step on the launching stream",
                       "step": "one prepared cpattn_ring call (descriptors built once)",
                       "clock_soak_s": t_soak},
            "roofline": {"bound": "tensor", "achieved": achieved,
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                         "peak_source": f"{peaks['source']} bf16 dense (burst)",
                         "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                         "kernel": "attn_fwd_kernel<bf16,128>",
                         "kernel_ms": kernel_ms},
            "e2e": e2e,
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
            "timed_wall_s": t_wall,
            "step_ms_percentiles": {f"p{q}": float(np.percentile(times, q))
                                    for q in (1, 10, 50, 90, 99)},
            "step_ms_max": float(max(times)),
            "steps_over_2x_median": int(sum(t > 2 * statistics.median(times) for t in times)),
        }
        if aux is not None:
            line["aux"] = aux
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------
# reference arm: the oracle as it stands, on the host cores
# ----------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    from workloads import make_workload
    oracle.build()
    w, q, k, v = make_workload(args.workload, seed=0)
    qh, kh, vh = q[0, 0:1], k[0, 0:1], v[0, 0:1]
    # each step: a bounded sample (rows of head 0 through the ring path),
    # sized so that warmup + steps take about a minute in total
    n = 64
    t0 = time.perf_counter()
    oracle.ring(qh[:, :n], kh, vh, w.head_dim ** -0.5, w.ring_degree, w.ring_anything)
    dt = max(time.perf_counter() - t0, 1e-4)
    per_step_budget = 60.0 / max(1, args.steps + args.warmup)
    n = int(min(w.seq, max(4, n * per_step_budget / dt)))
    for _ in range(args.warmup):
        oracle.ring(qh[:, :n], kh, vh, w.head_dim ** -0.5, w.ring_degree, w.ring_anything)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.ring(qh[:, :n], kh, vh, w.head_dim ** -0.5, w.ring_degree, w.ring_anything)
    dt = time.perf_counter() - t0
    flops = 4.0 * n * w.seq * w.head_dim * args.steps
    value = flops / dt / 1e12
    sample = (f"{n} query rows of head 0 against all {w.seq} keys of {w.name} per step "
              f"(ring_degree {w.ring_degree}), fp64 C oracle")
    print(json.dumps({
        "impl": "reference",
        "metric": "ring-attention TFLOP/s (bf16, 1 GB300) and % of dense BF16 tensor peak",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))
    return 0


# (batch, heads, seq, head_dim, dtype, ring_degree, ring_anything, causal)
SWEEP = [
    (1, 24, 1024, 128, "bf16", 1, False, False),
    (1, 24, 2048, 128, "bf16", 1, False, False),
    (1, 24, 4608, 128, "bf16", 1, False, False),
    (1, 24, 4608, 128, "bf16", 2, False, False),
    (1, 24, 4608, 128, "bf16", 4, False, False),
    (1, 24, 8192, 128, "bf16", 2, False, False),
    (1, 24, 16384, 128, "bf16", 4, False, False),
    (1, 24, 32768, 128, "bf16", 8, False, False),
    (4, 24, 4608, 128, "bf16", 2, False, False),
    (1, 24, 4609, 128, "bf16", 3, True, False),
    (1, 24, 4608, 128, "bf16", 2, False, True),
    (1, 24, 16384, 128, "bf16", 4, False, True),
    (1, 24, 4608, 64, "bf16", 2, False, False),
    (1, 24, 16384, 64, "bf16", 4, False, False),
    (1, 8, 4608, 128, "f32", 2, False, False),
    (1, 8, 4608, 64, "f32", 2, False, False),
]


def run_sweep(args):
    """Throughput of cpattn_ring over the SWEEP shapes: warm-up steps, then
    per-step CUDA events with the L2 flushed between steps; one JSON line
    per shape (inputs drawn on the device from a seeded generator)."""
    import context_attention_partial_gb300 as cp
    from workloads import Workload
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    peaks = load_peaks()
    steps = min(args.steps, 50)
    for (b, h, sq, d, dt, r, anything, causal) in SWEEP:
        w = Workload("sweep", b, h, sq, d, dt, ring_degree=r, ring_anything=anything,
                     causal=causal)
        g = torch.Generator(device=dev).manual_seed(7)
        q, k, v = (torch.randn(w.shape, generator=g, device=dev).to(w.torch_dtype)
                   for _ in range(3))
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], device=dev, dtype=torch.float32)
        need = cp.ring_workspace_bytes(q, r)
        ws = torch.empty(max(need, 16), device=dev, dtype=torch.uint8)
        step = cp.prepare_ring(q, k, v, r, anything, out=out, lse=lse, workspace=ws,
                               causal=causal)
        for _ in range(args.warmup):
            step()
        times = time_steps(step, steps, flush, stream)
        if cp.last_device_status() != 0:
            raise RuntimeError("device status after the sweep step")
        ms = statistics.median(times)
        tflops = w.flops / (ms * 1e-3) / 1e12
        print(json.dumps({"sweep": True, "shape": list(w.shape), "dtype": dt, "ring_degree": r,
                          "ring_anything": anything, "causal": causal, "ms_median": ms,
                          "TFLOP/s": tflops, "frac_bf16_peak": tflops / peaks["bf16_tflops"],
                          "steps": steps}), flush=True)
        del q, k, v, out, lse, ws, step
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="flux_ring")
    ap.add_argument("--no-aux", dest="aux", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--soak-s", type=float, default=1.0,
                    help="untimed steps before the timed region while clocks are sampled")
    ap.add_argument("--sweep", action="store_true",
                    help="time cpattn_ring over a list of shapes, one JSON line each")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
