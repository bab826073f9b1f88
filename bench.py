"""Benchmark of the rolling-KV hot path on B300.

One step = one pass of the whole hot path over one batch of synthetic input:
append one K/V pair per stream and layer (evicting the oldest), re-base the
origin, and attend every layer's queries over the window.  By default the
step is the fused rkv_step (one kernel: append + re-base + attend), followed
by rkv_rebase for stored-rotated keys with a re-basing epoch (the re-rotation
acts once per epoch), wherever the fused step applies (one new pair per
stream, bf16); otherwise, or with --path split, rkv_append + rkv_rebase +
rkv_attend.  Default workload: the 36-layer GQA 16/2 x 128 decoder, one
stream, window 4096, full (steady state: one pair evicted per step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...      # the float64 CPU oracle

Timing: K steps bracketed by a barrier + synchronize; each whole step is timed
with CUDA events on the launching stream.  Between steps, outside the events,
a 256 MiB buffer is written and another 256 MiB read, so every step starts on
a cold L2 that holds no dirty lines, and a short GPU spin gives the host time
to enqueue the whole step, so host launch latency never shows up between the
events.  ``value`` = K/V bytes read per step / event time per step (whole job:
all ranks' bytes over the slowest rank); the roofline object divides the same
bytes by the same events' time (the step's launches).  Prints one JSON line
(rank 0).
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "rolling-KV decode attention µs/step & achieved HBM GB/s (% of B300 peak)"
L2_FLUSH_BYTES = 256 << 20
HOST_SLACK_CYCLES = 400_000      # GPU spin (~0.2 ms) ahead of each timed step

WORKLOAD_TEXT = {
    "qwen3b": "36 layers, GQA 16 query / 2 KV heads, head_dim 128, bf16 K/V, window 4096, "
              "1 stream, 1 token per step, full window (one eviction per step)",
    "qwen3b_stored": "as qwen3b, stored-rotated keys: append + re-rotation of all retained "
                     "keys + attend",
    "qwen3b_epoch": "as qwen3b, stored-rotated keys re-based once every 4096 evictions "
                    "(rebase_epoch = W): append + re-base (a no-op until the lag reaches "
                    "W) + attend",
    "qwen3b_chunk6": "as qwen3b, 6 tokens per step (causal among the 6), 1% of k rows x2",
    "audio8": "8 layers, MHA 8 heads, head_dim 64, bf16 K/V, window 1024, 1 stream, 1 token "
              "per step, full window",
    "batch64": "64 streams, 36 layers, GQA 16/2 x 128, bf16, window 8192 each, fills uniform in "
               "[1, 8192], origins uniform in [0, 1e6), 1 token per stream per step",
    "encoder750": "causal audio encoder sliding window: 32 layers, 20 heads x 64 (MHA), bf16, "
                  "750 frames kept in 768 slots, 4 new frames per step (causal among the 4), "
                  "full window",
}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


def _workload(name):
    """(workload, key layout, re-basing epoch)."""
    from rkv_inputs import WORKLOADS
    if name == "qwen3b_stored":
        return WORKLOADS["qwen3b"], "stored_rotated", 0
    if name == "qwen3b_epoch":
        return WORKLOADS["qwen3b"], "stored_rotated", WORKLOADS["qwen3b"].capacity
    return WORKLOADS[name], "pre_rope", 0


def _kv_bytes_per_step(wl, fills):
    """Algorithmic K/V bytes the attention reads: every retained pair once."""
    return sum(fills) * wl.n_layers * wl.n_kv_heads * wl.head_dim * wl.elem_bytes * 2


# The source file each timed kernel is compiled from.
KERNEL_SOURCE = {
    "attend_mma": "rkv_attend_mma.cu", "attend_mma_step": "rkv_attend_mma.cu",
    "attend_mma_step_stored": "rkv_attend_mma.cu", "attend_mma_step_layer": "rkv_attend_mma.cu",
    "attend_mma_chunk": "rkv_attend_chunk.cu", "attend_fma": "rkv_attend_fma.cu",
    "attend_tc_chunk": "rkv_attend_tc.cu",
    "rerotate": "rkv_misc.cu",
}


def _sources(main):
    """`main` and the C-ABI entry points (which set the launch parameters and
    grid), with every library header they include, transitively.  The public
    header include/rkv.h (declarations and their documentation; no kernel
    includes it) is not part of a kernel's sources."""
    dirs = [os.path.join(ROOT, "rolling_kv_cache_buffer_b300", "csrc")]
    seen, todo = {}, [main, "rkv_api.cu"]
    while todo:
        name = todo.pop()
        if name in seen:
            continue
        path = next((os.path.join(d, name) for d in dirs if os.path.exists(os.path.join(d, name))),
                    None)
        if path is None:
            continue
        with open(path, "rb") as fh:
            seen[name] = fh.read()
        todo += re.findall(r'#include "([^"]+)"', seen[name].decode())
    return seen


def _code_only(text):
    """C/C++/CUDA source without its comments, whitespace runs collapsed."""
    text = re.sub(r"/\*.*?\*/", " ", text.decode(), flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split()).encode()


def kernel_hash(kernel_key):
    """Hash of the code (comments aside) a timed kernel is built from."""
    h = hashlib.sha256()
    for name, text in sorted(_sources(KERNEL_SOURCE[kernel_key]).items()):
        h.update(name.encode())
        h.update(_code_only(text))
    return h.hexdigest()[:16]


def _traffic(kernel_key, workload, alg_bytes_per_launch):
    """DRAM bytes per launch from the committed ncu summary (the record
    "<kernel>@<workload>" when there is one, else "<kernel>"), or None when
    the kernel's sources changed since the counters were taken or the counters
    were taken on another workload.  A record that states the algorithmic bytes
    of the launch it captured (a workload whose fills grow from step to step)
    is scaled to this line's algorithmic bytes per launch."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            d = json.load(f)
        ent = d.get(f"{kernel_key}@{workload}") or d.get(kernel_key)
        if (ent and ent.get("source_hash") == kernel_hash(kernel_key)
                and ent.get("workload", "").split(" ")[0] == workload):
            if ent.get("algorithmic_bytes"):
                return round(ent["bytes_per_launch"] * alg_bytes_per_launch
                             / ent["algorithmic_bytes"])
            return ent["bytes_per_launch"]
    except Exception:
        pass
    return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.tmp.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.tmp.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args, rank, world):
    import torch

    from rkv_inputs import initial_states, step_inputs
    from rolling_kv_cache_buffer_b300 import RollingKV

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl, layout, epoch = _workload(args.workload)
    c = wl.n_new
    cache = RollingKV(wl.n_streams, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                      wl.capacity, max_chunk=c, kv_dtype=wl.kv_dtype, layout=layout,
                      rope_theta=wl.rope_theta, attend_impl=args.attend_impl, device=dev,
                      rebase_epoch=epoch, window=wl.window or 0)
    # Steady-state windows: random contents (inputs of the path, not its work).
    gen = torch.Generator(device=dev).manual_seed(1234 + rank)
    cache.k_pool.normal_(generator=gen)
    cache.v_pool.normal_(generator=gen)
    if wl.random_state:
        origins, fills = initial_states(wl)
    else:
        origins, fills = [123_456] * wl.n_streams, [wl.retained] * wl.n_streams
    for s in range(wl.n_streams):
        cache.set_stream_state(s, origins[s], fills[s])
    dt = cache.kv_dtype

    # Pre-staged step inputs (a ring cycled by the timed loop).
    ring = []
    for t in range(args.ring):
        q, k, v = step_inputs(wl, 1 + t)
        ring.append((q.to(dt).to(dev), k.to(dt).to(dev), v.to(dt).to(dev)))
    out = torch.empty(ring[0][0].shape, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    drain = torch.zeros(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def cold():
        """Between steps, outside the events: a GPU spin (the host enqueues the
        step meanwhile), 256 MiB written (no line of the step's data stays in
        L2), then another 256 MiB read (the written lines are drained, so the
        step starts on a cold, clean L2)."""
        torch.cuda._sleep(HOST_SLACK_CYCLES)
        if not args.warm_l2:
            flush.zero_()
            torch.amax(drain)

    # Which calls make the step.  The fused decode step (rkv_step, one launch)
    # applies to pre-RoPE keys and to stored-rotated keys with a re-basing
    # epoch (then rkv_step + rkv_rebase, whose launch acts once per epoch),
    # one new pair, bf16; "auto" takes it wherever it applies (the faster path
    # measured on B300).
    fused = step_is_fused(wl, layout, epoch, args)

    per_layer = fused and (args.per_layer or args.graph)
    graphs = {}

    def layer_calls(q, k, v):
        for l in range(wl.n_layers):
            cache.step_layers(l, k[l:l + 1], v[l:l + 1], q[l:l + 1], out[l:l + 1],
                              last=(l == wl.n_layers - 1))

    def graph_of(i):
        """The per-layer calls of ring entry i, captured once in a CUDA graph."""
        if i not in graphs:
            q, k, v = ring[i]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="relaxed"):
                layer_calls(q, k, v)
            graphs[i] = g
        return graphs[i]

    def step(i, ev=None):
        q, k, v = ring[i % len(ring)]
        if args.graph and fused:
            g = graph_of(i % len(ring))      # captured outside the events
        if ev:
            ev[0].record(stream)
        if per_layer:
            if args.graph:
                g.replay()
            else:
                layer_calls(q, k, v)
        elif fused:
            cache.step(k, v, q, out)
            if layout == "stored_rotated":
                cache.rebase()
        else:
            cache.append(k, v)
            cache.rebase()
            cache.attend(q, out)
        if ev:
            ev[1].record(stream)

    if args.graph and fused:
        for i in range(len(ring)):
            graph_of(i)
    n_done = 0
    for i in range(args.warmup):
        cold()
        step(n_done)
        n_done += 1
    torch.cuda.synchronize(dev)
    # Stored-rotated keys with a re-basing epoch E: the re-rotation of the whole
    # key pool runs once every E evictions.  With fewer than E timed steps, lead
    # the streams (untimed steps) so that one re-rotation falls in the middle
    # of the timed region, which then carries more than its share of that work.
    if layout == "stored_rotated" and epoch:
        lead = max(0, epoch - args.steps // 2 - int(_lags(cache).max())) \
            if args.steps < epoch else 0
        for _ in range(lead):
            step(n_done)
            n_done += 1
        torch.cuda.synchronize(dev)
        lags = [int(x) for x in _lags(cache)]
    launches_per_step = ((wl.n_layers if per_layer else 1) +
                         (1 if layout == "stored_rotated" else 0)) if fused else \
        2 + (1 if layout == "stored_rotated" else 0)

    # Timed region: exactly `steps` whole steps, one event pair around each.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    fl = list(fills)
    for _ in range(n_done):
        fl = [min(wl.retained, f + c) for f in fl]
    bytes_per_step = []
    rerotations = 0
    with ClockSampler(dev.index) as clk:
        t0 = time.perf_counter()
        for i in range(args.steps):
            cold()
            step(n_done, evs[i])
            n_done += 1
            if layout == "stored_rotated" and epoch:
                lags = [g + max(0, f + c - wl.retained) for g, f in zip(lags, fl)]
                if max(lags) >= epoch:
                    rerotations += 1
                    lags = [0 if g >= epoch else g for g in lags]
            fl = [min(wl.retained, f + c) for f in fl]   # each step attends over fill'
            bytes_per_step.append(_kv_bytes_per_step(wl, fl))
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
    if world > 1:
        dist.barrier()
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]

    res_fills = fl
    total_bytes = sum(bytes_per_step)
    total_ms = sum(step_ms)
    assert torch.isfinite(out).all(), "non-finite attention output"

    # e2e: host buffers through the public API, copies inside the timed region.
    e2e = run_e2e(args, cache, ring, dev, wl, stream, fused, cold) if not args.no_e2e else \
        {"ms_per_step": float("nan"), "ms_mean": float("nan"), "steps": 0, "h2d": 0, "d2h": 0}

    res = dict(total_bytes=total_bytes, total_ms=total_ms, steps=args.steps, fused=fused,
               step_ms=step_ms, wall_s=wall,
               clocks=clk.summary(), launches=launches_per_step * args.steps,
               bytes_per_step=bytes_per_step, e2e=e2e, fills=res_fills,
               rerotations=rerotations if layout == "stored_rotated" and epoch else None)
    return res


TC_AUTO_MIN_ROWS = 16   # the library's choice under "auto": chunks of c*G >= 16 rows


def chunk_on_tc(attend_impl, rows):
    """Whether a chunk of `rows` = c*G query rows per KV head runs on the
    tcgen05 kernel for this attend_impl (the library's own rule)."""
    return attend_impl == "tc" or (attend_impl == "auto" and rows >= TC_AUTO_MIN_ROWS)


def step_is_fused(wl, layout, epoch, args):
    """Whether the timed step is the fused rkv_step (else the separate calls).
    The fused step applies to pre-RoPE keys and to stored-rotated keys with a
    re-basing epoch, one new pair, bf16, tensor-core kernels; "auto" takes the
    fused step wherever it applies (the faster path measured on B300: 39.9 us
    against 43.7 us for the separate calls on the 36-layer decoder;
    --per-layer and --graph are fused forms)."""
    fusable = (layout == "pre_rope" or epoch > 0) and wl.kv_dtype == "bf16" and \
        wl.n_new == 1 and args.attend_impl != "fma"
    path = "split" if args.no_fused else args.path
    if path == "auto":
        path = "fused"
    return fusable and path == "fused"


def _lags(cache):
    """Per-stream lag of stored-rotated keys behind the origin (int32 field 4
    of each 32-byte stream state record)."""
    import torch
    return cache.state.view(torch.int32)[: 8 * cache.S].view(cache.S, 8)[:, 4].cpu().numpy()


def _pack(ts, make):
    """One flat buffer (from make(numel, dtype)) holding the same-dtype tensors
    ts end to end, each starting on a 16-byte boundary; returns (flat, views)."""
    dt, esz = ts[0].dtype, ts[0].element_size()
    assert all(t.dtype == dt for t in ts)
    align = max(1, 16 // esz)
    offs, n = [], 0
    for t in ts:
        offs.append(n)
        n += -(-t.numel() // align) * align
    flat = make(n, dt)
    return flat, [flat[o:o + t.numel()].view(t.shape) for o, t in zip(offs, ts)]


def run_e2e(args, cache, ring, dev, wl, stream, fused, cold):
    """The step through the public API from host memory: each step's q, k and
    v sit in one pinned host buffer and go to the device in one copy (the
    library takes the three 16-byte-aligned views of the device buffer); the
    output comes back in one copy.  Same L2 regime as the main loop: the cold()
    flush runs between steps, outside the events; one event pair per step,
    at least 200 steps; the median and the mean are reported."""
    import torch
    host = []
    for q, k, v in ring[: min(len(ring), 16)]:
        hflat, views = _pack([q, k, v], lambda n, dt: torch.empty(n, dtype=dt).pin_memory())
        for h, t in zip(views, (q, k, v)):
            h.copy_(t.cpu())
        host.append(hflat)
    dflat, (dq, dk, dv) = _pack(list(ring[0]),
                                lambda n, dt: torch.empty(n, dtype=dt, device=dev))
    out = torch.empty(dq.shape, dtype=torch.float32, device=dev)
    hout = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    steps = max(200, args.steps // 4)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]

    def one(i):
        dflat.copy_(host[i % len(host)], non_blocking=True)
        if fused:
            cache.step(dk, dv, dq, out)
            if cache.stored:
                cache.rebase()
        else:
            cache.append(dk, dv)
            cache.rebase()
            cache.attend(dq, out)
        hout.copy_(out, non_blocking=True)

    for i in range(3):
        cold()
        one(i)
    torch.cuda.synchronize(dev)
    for i in range(steps):
        cold()
        evs[i][0].record(stream)
        one(i)
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    per = [e[0].elapsed_time(e[1]) for e in evs]
    h2d = host[0].numel() * host[0].element_size()
    d2h = hout.numel() * hout.element_size()
    return {"ms_per_step": statistics.median(per), "ms_mean": sum(per) / len(per),
            "steps": steps, "h2d": h2d, "d2h": d2h}


# ---------------------------------------------------------------------------
# CPU oracle (reported baseline and the reference arm)
# ---------------------------------------------------------------------------

class OracleRunner:
    """The float64 oracle (as it stands) on a bounded sample of the workload:
    at most two streams and `layers` of the layers, the window seeded to the
    workload's steady state.  One call of step() runs one whole step of the
    sample (append + re-rotation for stored-rotated + attend); its time is
    scaled to the full workload by streams x layers."""

    def __init__(self, wl_name, layers=2):
        from oracle import rkv_oracle as O
        from rkv_inputs import initial_states, initial_window
        self.wl, layout, epoch = _workload(wl_name)
        wl = self.wl
        self.S = min(wl.n_streams, 2)
        self.Ls = min(wl.n_layers, layers)
        self.stored = layout == "stored_rotated"
        if self.stored and epoch:
            self.orc = O.EpochRotatedOracle(self.S, self.Ls, wl.n_q_heads, wl.n_kv_heads,
                                            wl.head_dim, wl.capacity, theta=wl.rope_theta,
                                            epoch=epoch, window=wl.window)
        else:
            cls = O.StoredRotatedOracle if self.stored else O.RollingCacheOracle
            self.orc = cls(self.S, self.Ls, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                           wl.capacity, theta=wl.rope_theta, window=wl.window)
        if wl.random_state:
            origins, fills = initial_states(wl)
        else:
            origins, fills = [123_456] * wl.n_streams, [wl.retained] * wl.n_streams
        self.fills = fills
        for s in range(self.S):
            k, v = initial_window(wl, s, fills[s])
            self.orc.set_state(s, origins[s], fills[s], k[: self.Ls].double().numpy(),
                               v[: self.Ls].double().numpy())
        self.t = 0
        self.scale = (wl.n_streams / self.S) * (wl.n_layers / self.Ls)

    def step(self):
        """Runs one sampled step; returns its time scaled to the whole workload."""
        from rkv_inputs import step_inputs
        self.t += 1
        q, k, v = step_inputs(self.wl, self.t)
        Ls, S = self.Ls, self.S
        q = q[:Ls, :S].double().numpy()
        k = k[:Ls, :S].double().numpy()
        v = v[:Ls, :S].double().numpy()
        t0 = time.perf_counter()
        self.orc.append(k, v)
        if self.stored:
            self.orc.rebase()
        self.orc.attend(q)
        return (time.perf_counter() - t0) * self.scale

    def sample_text(self):
        return (f"{self.S} of {self.wl.n_streams} stream(s) x {self.Ls} of {self.wl.n_layers} "
                f"layers per step (float64 numpy), time scaled x{self.scale:g}")


def oracle_cores():
    """Threads the oracle's numpy BLAS runs on (bounded by the usable cores)."""
    cores = len(os.sched_getaffinity(0))
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
        return min(cores, threads)
    except ImportError:
        return cores


def combine_ranks(ms, e2e_ms, att_ms, bytes_local, world, device):
    """Whole-job numbers from every rank's own: the slowest rank's times (MAX)
    and the bytes all ranks processed (SUM).  Each rank runs its own streams
    (independent replicas), so this is the only cross-rank traffic."""
    if world <= 1:
        return ms, e2e_ms, att_ms, bytes_local
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms, e2e_ms, att_ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    b = torch.tensor([bytes_local], device=device, dtype=torch.float64)
    dist.all_reduce(b)
    ms, e2e_ms, att_ms = [float(x) for x in t.tolist()]
    return ms, e2e_ms, att_ms, float(b.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="qwen3b", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--attend-impl", default="auto", choices=["auto", "fma", "mma", "tc"])
    ap.add_argument("--ring", type=int, default=64)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", default="auto", choices=["auto", "fused", "split"],
                    help="fused: rkv_step where it applies; split: rkv_append + rkv_rebase + "
                         "rkv_attend; auto: the faster of the two for the layout")
    ap.add_argument("--no-fused", action="store_true", help="same as --path split")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer end-to-end loop (short runs under ncu)")
    ap.add_argument("--per-layer", action="store_true",
                    help="the fused step as one rkv_step_layers call per layer")
    ap.add_argument("--graph", action="store_true",
                    help="--per-layer, each step's calls replayed from a CUDA graph")
    ap.add_argument("--warm-l2", action="store_true",
                    help="no L2 flush between steps (reported alongside; the default is cold)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    wl, layout, _ = _workload(args.workload)
    peak, peak_kind = _peaks()
    tokens_per_step = wl.n_streams * wl.n_new

    if args.impl == "reference":
        if rank != 0:
            return
        # Each step samples one layer (of the workload's) when many steps are
        # asked for, so that the whole run stays within a few minutes.
        runner = OracleRunner(args.workload, layers=1 if args.steps > 200 else 2)
        for _ in range(args.warmup):
            runner.step()
        secs = [runner.step() for _ in range(args.steps)]
        sec = sum(secs) / len(secs)
        bps = _kv_bytes_per_step(wl, [min(wl.retained, f + wl.n_new) for f in runner.fills])
        val = bps / sec / 1e9
        line = {
            "impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "us_per_step": sec * 1e6,
            "tokens_per_s": tokens_per_step / sec, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT[args.workload]}"},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": oracle_cores(),
                             "kind": "oracle", "sample": runner.sample_text()},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", rank=rank, world_size=world)
    res = run_gpu(args, rank, world)
    ms_local = res["total_ms"] / res["steps"]
    bytes_local = res["total_bytes"] / res["steps"]
    e2e_ms_local = res["e2e"]["ms_per_step"]
    ms, e2e_ms, _, all_bytes = combine_ranks(ms_local, e2e_ms_local, ms_local, bytes_local,
                                             world, "cuda")
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    value = all_bytes / (ms * 1e-3) / 1e9
    # The roofline's kernel time is measured on the timed steps themselves, by
    # the same events: the step's launches are the kernel(s) it names, so
    # kernel_us <= us_per_step always holds (equality for a one-launch step).
    if res["fused"] and (args.per_layer or args.graph):
        # One launch per layer: the step's bytes over the step's time; kernel_us
        # is the average launch.
        kernel_key = "attend_mma_step_layer"
        scope = "rkv_step_layers, one launch per layer: the step's time over its launches"
        kern_us = ms_local * 1e3 / wl.n_layers
    elif res["fused"]:
        # The step is one launch of the fused kernel (for stored-rotated keys
        # followed by the re-base launch, which acts once per epoch): the
        # events bracket the kernel.
        stored = _workload(args.workload)[1] == "stored_rotated"
        kernel_key = "attend_mma_step_stored" if stored else "attend_mma_step"
        scope = "the fused step's one launch (events around it)" + \
            ("; the re-base launch acts once per epoch" if stored else "")
        kern_us = ms_local * 1e3
    else:
        kernel_key = "attend_fma" if args.attend_impl == "fma" or wl.kv_dtype != "bf16" else \
            ("attend_mma" if wl.n_new == 1 else
             "attend_tc_chunk" if chunk_on_tc(args.attend_impl, wl.n_new * wl.n_q_heads // wl.n_kv_heads)
             else "attend_mma_chunk")
        scope = ("the step's launches: rkv_append, then the attention launched with "
                 "programmatic dependent launch (its prologue overlaps the append); the "
                 "attention's own share of the device time is in the committed launch list")
        kern_us = ms_local * 1e3
    kern_launches = wl.n_layers if res["fused"] and (args.per_layer or args.graph) else 1
    achieved = bytes_local / (kern_us * kern_launches * 1e-6) / 1e9
    assert kern_us <= ms_local * 1e3 * (1 + 1e-9)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "us_per_step": ms * 1e3, "tokens_per_s": world * tokens_per_step / (ms * 1e-3),
        "pct_of_hbm_peak": 100.0 * value / (peak * world),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT[args.workload]}",
                   "kv_bytes_per_step": int(bytes_local),
                   "l2": ("warm: no flush between steps (inputs smaller than L2 may stay "
                          "resident)" if args.warm_l2 else
                          "between steps, outside the timed events: 256 MiB written, then "
                          "another 256 MiB read (cold L2, no dirty lines)"),
                   "attend_impl": args.attend_impl, "parallelism": f"replicas x{world}",
                   "step": (("rkv_step_layers x %d (one launch per layer%s)" %
                             (wl.n_layers, ", replayed from a CUDA graph" if args.graph else ""))
                            if res["fused"] and (args.per_layer or args.graph) else
                            ("rkv_step (append + attend, all layers, one launch) + rkv_rebase "
                             "(the re-rotation when due)" if args.workload.endswith("epoch") else
                             "rkv_step: append + attend (all layers), one launch")
                            if res["fused"] else
                            "rkv_append + rkv_attend (all layers; rkv_rebase launches nothing "
                            "for pre-RoPE keys)" if _workload(args.workload)[1] == "pre_rope" else
                            "rkv_append + rkv_rebase + rkv_attend (all layers)")},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} hbm_gbs",
                     "kernel": kernel_key,
                     "traffic": _traffic(kernel_key, args.workload,
                                         bytes_local / kern_launches),
                     "kernel_us": kern_us, "kernel_scope": scope},
        "e2e": ({"value": all_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                 "us_per_step": e2e_ms * 1e3, "us_per_step_mean": res["e2e"]["ms_mean"] * 1e3,
                 "steps": res["e2e"]["steps"], "statistic": "median of per-step events",
                 "l2": "cold, as the main loop (flush between steps, outside the events)",
                 "h2d_bytes_per_step": res["e2e"]["h2d"],
                 "d2h_bytes_per_step": res["e2e"]["d2h"]}
                if res["e2e"]["steps"] else
                {"value": None, "unit": "GB/s", "skipped": "--no-e2e",
                 "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}),
        "gpu_launches": res["launches"],
        **({"rerotations_in_timed_region": res["rerotations"]}
           if res["rerotations"] is not None else {}),
        "clocks": res["clocks"],
        "wall_s_timed_region": res["wall_s"],
    }
    if not args.no_cpu_baseline:
        runner = OracleRunner(args.workload)
        runner.step()
        secs, t0 = [], time.perf_counter()
        while len(secs) < 200 and (len(secs) < 3 or time.perf_counter() - t0 < args.cpu_budget):
            secs.append(runner.step())
        sec = sum(secs) / len(secs)
        cb = _kv_bytes_per_step(wl, [min(wl.retained, f + wl.n_new) for f in runner.fills])
        line["cpu_baseline"] = {
            "value": cb / sec / 1e9, "unit": "GB/s", "cores": oracle_cores(), "kind": "oracle",
            "sample": f"{len(secs)} steps of " + runner.sample_text(),
            "ms_per_step": sec * 1e3}
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
