#!/usr/bin/env python
"""Benchmark of the multi-adapter LoRA path on one GB300 (or N, one process each).

A step is one pass of the whole path over one batch of one configuration:

* tiny, prefill, hetero: lora_segments_build (grouping the batch's tokens by adapter,
  work lists) followed by the step's lora_apply call(s);
* decode (one token per request): lora_bgmv_ex, every token gathering its own adapter
  through the page table, shrink + scale + expand in place in y, one kernel; the ids
  and pools are uploaded once, so the calls pass LORA_BGMV_STATIC_ADAPTERS (a call
  stages its adapters while the call ahead of it finishes);
* backward (with --workload backward, and under per_config): lora_segments_build +
  lora_sgmv_backward on the prefill batch;
* mixed13b (the headline, the largest configuration that fits one GPU): one forward of
  the 13B-shaped mixed batch, one segment build and 40 layers x 7 projections, in four
  grouped calls per layer (lora_apply_multi for q, k, v on their shared input and for
  gate, up on theirs; lora_apply for o and down).

By default the printed JSON line is the 13B forward, with every other configuration
timed in the same process under "per_config" (each with its own roofline, CPU
baseline, end-to-end figure and parity sample).  `--workload NAME` times one
configuration alone.  `--impl reference` times the CPU fp64 oracle on the same
workload instead (the reference arm of this build: there is no runnable upstream
implementation).
"""

from __future__ import annotations

import argparse
import gc
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SGMV/BGMV adapter-path tokens/s and achieved HBM GB/s (% of roofline), 1×GB300"
UNIT = "tokens/s"
HEADLINE = "mixed13b"
# Decode first: a decode call is a chain of latencies (~5 us), and timed a few seconds into the
# process (after any other timing, another decode included) it reads ~0.45 us slower per call
# than timed first, with the memory and SM clocks unchanged; the other lines move by under 0.5 %.
OTHERS = ("decode", "tiny", "prefill", "hetero")

WORKLOAD_TEXT = {
    "decode": "decode BGMV: 64 tokens (1 per request), q_proj 4096->4096, 100 adapters rank 16, "
              "uniform adapter per token, bf16",
    "prefill": "prefill SGMV: 32 requests of U{64..512} tokens, 4096->4096, 200 adapters rank 16, "
               "Zipf(1.1) popularity, contiguous segments, bf16",
    "hetero": "heterogeneous ranks: 256 decode tokens, 500 adapters r in {8,16,32,64}, "
              "MLP up 4096->11008 and down 11008->4096 (two calls sharing the segments), "
              "paged 4096-element pages, bf16",
    "mixed13b": "13B-shaped mixed batch: 4 prefill requests of 1024 tokens + 128 decode tokens, "
                "d=5120, 40 layers x (q,k,v,o 5120->5120, gate,up 5120->13824, down 13824->5120), "
                "1000 adapters r in {16,32,64} Zipf(1.1)-popular, referenced ones resident in "
                "paged pools; a step is one forward: one segment build and 40 layers x 4 grouped "
                "calls ([q,k,v] on one x, [o], [gate,up] on one x, [down]) = 280 projections",
    "tiny": "tiny SGMV: d=256, 4 adapters rank 8, 16 tokens in segments [3,5,1,7]",
}

# timed steps of the configurations timed beside the headline (each well under a second)
OTHER_STEPS = {"tiny": 20000, "decode": 20000, "prefill": 2000, "hetero": 2000}
BACKWARD_STEPS = 500
BASE_STEPS = 100


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None,
                   help="timed steps of the headline (default 20 forwards of the 13B batch; "
                        "20000 for a small configuration timed alone)")
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["all", "backward", "base_fused"] + sorted(WORKLOAD_TEXT), default="all",
                   help="all (default): the 13B forward as the headline, every other "
                        "configuration under per_config; or one configuration alone "
                        "(backward: the adapter-training backward pass on the prefill batch)")
    p.add_argument("--cpu-seconds", type=float, default=5.0,
                   help="bounded CPU work per configuration for the oracle baseline (0 disables it)")
    p.add_argument("--e2e-steps", type=int, default=None,
                   help="end-to-end steps (default 500; 5 for the 13B forward)")
    p.add_argument("--soak-seconds", type=float, default=0.5,
                   help="untimed steady load before each timed region while clocks are sampled")
    args = p.parse_args(argv)
    head = HEADLINE if args.workload == "all" else args.workload
    if args.steps is None:
        args.steps = 20 if head == "mixed13b" else BACKWARD_STEPS if head == "backward" else \
            BASE_STEPS if head == "base_fused" else 20000
    return args


def default_e2e_steps(name: str, args) -> int:
    if args.e2e_steps is not None:
        return args.e2e_steps
    return 5 if name == "mixed13b" else 500


# ------------------------------------------------------------------ helpers --

def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.f = tempfile.NamedTemporaryFile("w", prefix="clocks_", suffix=".csv", delete=False)
        self.path = self.f.name
        self.proc = None
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "200"]
        if gpu_id:
            cmd[1:1] = ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            self.f.close()
            os.unlink(self.path)
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [c.strip() for c in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- workloads --

def make_workload(name: str, seed: int):
    from segmented_gather_gemm_lora_gb300 import workloads as W

    if name == "hetero":
        wl = W.hetero(seed, which="both")
    elif name == "mixed13b":  # one (layer, projection) on the host: the CPU sample
        wl = W.mixed13b(seed, layers=(0,), projections=("q",))
    else:
        wl = W.WORKLOADS[name](seed)
    return wl


def host_calls(wl, seed: int):
    """(pool, batch) of every projection call of one step on the host workload."""
    from segmented_gather_gemm_lora_gb300 import workloads as W

    calls = [(wl.pools[0], wl.batch)]
    if len(wl.pools) > 1:  # hetero: the down projection on the same ids
        p = wl.pools[1]
        bd = W.make_batch(np.random.default_rng([seed, 7]), wl.batch.ids, p.d_in, p.d_out)
        calls.append((p, bd))
    return calls


class _Shape:
    """What algorithmic_bytes / algorithmic_flops read of a pool."""

    def __init__(self, ranks, d_in, d_out):
        self.ranks, self.d_in, self.d_out = np.asarray(ranks), d_in, d_out


def device_pool(B, torch, dev, rng, ranks, d_in, d_out, page_elems=4096, alpha=16.0):
    """A paged pool drawn on the device (A ~ N(0, 1/d_in), B ~ N(0, 1/r) per page, physical
    pages in a random permutation) for configurations too large to draw on the host."""
    from segmented_gather_gemm_lora_gb300 import workloads as W

    P = page_elems
    ranks = np.asarray(ranks, dtype=np.int32)
    na = [(-(-int(r) * d_in // P)) if r > 0 else 0 for r in ranks]
    nb = [(-(-int(r) * d_out // P)) if r > 0 else 0 for r in ranks]
    n_list = int(sum(na) + sum(nb))
    n_pages = n_list + 3
    phys = rng.permutation(n_pages).astype(np.int32)
    desc = np.zeros(len(ranks), dtype=W.DESC_DTYPE)
    pscale = np.ones(n_pages, dtype=np.float32)
    cur = 0
    for i, r in enumerate(ranks):
        if r <= 0:
            continue
        desc[i] = (r, alpha / r, cur, cur + na[i])
        pscale[phys[cur:cur + na[i]]] = (1.0 / d_in) ** 0.5
        pscale[phys[cur + na[i]:cur + na[i] + nb[i]]] = (1.0 / r) ** 0.5
        cur += na[i] + nb[i]
    pool = (torch.randn(n_pages, P, device=dev) * torch.from_numpy(pscale).to(dev)[:, None]).to(torch.bfloat16)
    pl = torch.from_numpy(phys[:n_list].copy()).to(dev)
    dsc = torch.from_numpy(desc.view(np.uint8).copy()).to(dev)
    return B.PoolView(pool, pl, dsc, P, 64, d_in, d_out), _Shape(ranks, d_in, d_out)


def algorithmic_bytes(batch, pool, x_read: bool = True) -> int:
    """Bytes the fused apply must move at least once: every distinct adapter used (A and B
    at its own rank, no padding), x read (unless another projection of the same grouped
    call already counts it), y read and written (bf16)."""
    ids = batch.ids
    valid = ids >= 0
    distinct = np.unique(ids[valid])
    ranks = pool.ranks[distinct].astype(np.int64)
    adapters = int((ranks * (pool.d_in + pool.d_out)).sum()) * 2
    n = int(valid.sum())
    return adapters + (n * pool.d_in * 2 if x_read else 0) + n * pool.d_out * 2 * 2


def algorithmic_flops(batch, pool) -> int:
    ids = batch.ids
    r = pool.ranks[ids[ids >= 0]].astype(np.int64)
    return int((2 * r * (pool.d_in + pool.d_out)).sum())


# -------------------------------------------------------------- our arm --

def build_sets(name, rank, dev, l2, torch, B):
    """Input sets of the workload on the device.  Each set is one step's batch: its ids,
    segment buffer and projection calls (view, x, y and their algorithmic bytes / flops);
    sets rotate so that a pass over them exceeds 2x L2."""
    from segmented_gather_gemm_lora_gb300 import workloads as W

    def up(a):  # host bf16 bits -> device bf16
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    if name == "mixed13b":
        # One forward of 40 layers x 7 projections in 4 grouped calls per layer (q, k, v share
        # their input, as gate and up do); adapters and activations drawn on the device
        # (about 20 GB of adapter pages and 25 GB of activations, so nothing stays in L2
        # between calls).
        rng = np.random.default_rng(1000 * rank)
        ranks = W.mixed13b_ranks(rng)
        ids = W.mixed13b_ids(rng)
        resident = np.zeros_like(ranks)
        used = np.unique(ids)
        resident[used] = ranks[used]
        T = len(ids)
        proj = {p[0]: (i, p[1], p[2]) for i, p in enumerate(W.PROJ_13B)}
        calls = []
        for layer in range(40):
            for group in (("q", "k", "v"), ("o",), ("gate", "up"), ("down",)):
                d_in = proj[group[0]][1]
                x = torch.randn(T, d_in, device=dev).to(torch.bfloat16)
                views, ys, nbytes, nflops = [], [], 0, 0
                for k, pname in enumerate(group):
                    pi, _, d_out = proj[pname]
                    prng = np.random.default_rng([1000 * rank, 1 + layer, 1 + pi])
                    view, shape = device_pool(B, torch, dev, prng, resident, d_in, d_out)
                    bt = W.Batch(x=None, y0=None, ids=ids, d_in=d_in, d_out=d_out)
                    views.append(view)
                    ys.append(torch.randn(T, d_out, device=dev).to(torch.bfloat16))
                    nbytes += algorithmic_bytes(bt, shape, x_read=k == 0)
                    nflops += algorithmic_flops(bt, shape)
                calls.append(dict(views=views, x=x, ys=ys, bytes=nbytes, flops=nflops, layer=layer,
                                  name="+".join(group)))
        S = dict(calls=calls, ids=torch.from_numpy(ids).to(dev), seg=B.Segments(T, device=dev),
                 T=int((ids >= 0).sum()), host_ids=ids, wl=None, mode=0, n_ad=1000)
        set_bytes = sum(sum(v.pool.numel() * 2 for v in c["views"]) + c["x"].numel() * 2 +
                        sum(y.numel() * 2 for y in c["ys"]) for c in calls)
        return [S], set_bytes

    wl0 = make_workload(name, 1000 * rank)
    set_bytes = sum(p.pool.nbytes + b.x.nbytes + b.y0.nbytes for p, b in host_calls(wl0, 1000 * rank))
    n_sets = max(2, math.ceil(2 * l2 / max(set_bytes, 1)) + 1)
    sets = []
    for s in range(n_sets):
        seed = 1000 * rank + s
        wl = wl0 if s == 0 else make_workload(name, seed)
        calls = []
        for pool, b in host_calls(wl, seed):
            calls.append(dict(views=[B.PoolView.from_host(pool, device=dev)], x=up(b.x), ys=[up(b.y0)],
                              bytes=algorithmic_bytes(b, pool), flops=algorithmic_flops(b, pool),
                              hx=b.x, hy0=b.y0))
        sets.append(dict(calls=calls, ids=torch.from_numpy(wl.batch.ids).to(dev),
                         seg=B.Segments(wl.batch.T, device=dev), T=int((wl.batch.ids >= 0).sum()),
                         host_ids=wl.batch.ids, wl=wl, mode=wl.mode, n_ad=wl.n_adapters))
    return sets, set_bytes


def gpu_id_of(props) -> str:
    gpu_id = str(getattr(props, "uuid", "") or "")
    if gpu_id and not gpu_id.startswith("GPU-"):
        gpu_id = "GPU-" + gpu_id
    return gpu_id


def run_workload(name, steps, warmup, e2e_steps, soak_seconds, world, rank, local):
    """Time `steps` steps of one configuration (inputs resident in HBM), the step's
    projection calls alone, and the same step end to end from host buffers; returns the
    JSON fields of the configuration."""
    import torch

    from segmented_gather_gemm_lora_gb300 import binding as B

    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20)

    sets, set_bytes = build_sets(name, rank, dev, l2, torch, B)
    n_sets = len(sets)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    mode = sets[0]["mode"]
    n_ad = sets[0]["n_ad"]
    n_calls = len(sets[0]["calls"])

    bgmv = name == "decode"

    def run_call(c, ids, seg):
        if bgmv:
            # the ids and the pools are uploaded once and never written by a kernel
            B.lora_bgmv(c["x"], c["ys"][0], ids, c["views"][0], err=err, static_adapters=True)
        elif len(c["views"]) == 1:
            B.lora_apply(c["x"], c["ys"][0], seg, c["views"][0], err=err)
        else:
            B.lora_apply_multi(list(zip([c["x"]] * len(c["ys"]), c["ys"], c["views"])), seg, err=err)

    def calls_of(S):
        for c in S["calls"]:
            run_call(c, S["ids"], S["seg"])

    def step(k):
        S = sets[k % n_sets]
        if not bgmv:
            B.lora_segments_build(S["ids"], n_ad, S["seg"], mode=mode, err=err)
        calls_of(S)

    # warm-up (eager), then a CUDA graph of one pass over all sets.
    for k in range(max(warmup, 3)):
        step(k)
    torch.cuda.synchronize()
    g_steps = n_sets * max(1, 64 // (n_sets * n_calls))
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device=dev)
    launches0 = B.launch_count()
    with torch.cuda.graph(graph, stream=cap):
        for k in range(g_steps):
            step(k)
    launches_per_step = (B.launch_count() - launches0) / g_steps
    rem = steps % g_steps
    graph_rem = None
    if rem:
        graph_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_rem, stream=cap):
            for k in range(rem):
                step(k)
    reps = steps // g_steps
    graph.replay()
    torch.cuda.synchronize()

    # clocks: steady load before and during the timed region
    sampler = ClockSampler(gpu_id_of(props))
    t_end = time.perf_counter() + soak_seconds
    while time.perf_counter() < t_end:
        graph.replay()
        torch.cuda.synchronize()

    # ---- timed region: exactly `steps` steps ----
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    if graph_rem is not None:
        graph_rem.replay()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    ms_local = e0.elapsed_time(e1)
    ms = max_over_ranks(ms_local, world)
    assert int(err.item()) == 0, "device error word %d" % int(err.item())

    tokens_per_step = statistics.fmean(S["T"] for S in sets)  # sets are visited uniformly per pass
    per_pass = [sets[k % n_sets]["T"] for k in range(g_steps)]
    tokens_timed = reps * sum(per_pass) + sum(sets[k % n_sets]["T"] for k in range(rem))
    total_tokens = sum_over_ranks(tokens_timed, world)
    value = total_tokens / (ms / 1e3)

    # ---- duration of the step's projection calls alone (lora_bgmv / lora_apply) ----
    # A CUDA graph of those calls (segments built beforehand for every set), replayed back
    # to back and bracketed by CUDA events on the launching stream.
    if not bgmv:
        for S in sets:
            B.lora_segments_build(S["ids"], n_ad, S["seg"], mode=mode, err=err)
        torch.cuda.synchronize()

    call_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(call_graph, stream=cap):
        for k in range(g_steps):
            calls_of(sets[k % n_sets])
    call_graph.replay()
    torch.cuda.synchronize()
    call_reps = max(1, min(max(reps, 1), int(0.2 / max(ms / steps / 1e3 * g_steps, 1e-9))))
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record()
    for _ in range(call_reps):
        call_graph.replay()
    c1.record()
    torch.cuda.synchronize()
    calls_avg_s = c0.elapsed_time(c1) / (call_reps * g_steps) / 1e3

    # single-call latency (one eager call group on an idle GPU, not graph-amortised) and
    # the same calls with a warm L2 (one input set, back to back in a graph)
    lat = []
    for i in range(20):
        torch.cuda.synchronize()
        c0.record()
        calls_of(sets[i % n_sets])
        c1.record()
        torch.cuda.synchronize()
        lat.append(c0.elapsed_time(c1) * 1e3)
    single_us = statistics.median(lat)
    hot_us = None
    if name != "mixed13b":
        hot_graph = torch.cuda.CUDAGraph()
        n_hot = max(1, 64 // n_calls)
        with torch.cuda.graph(hot_graph, stream=cap):
            for _ in range(n_hot):
                calls_of(sets[0])
        hot_graph.replay()
        torch.cuda.synchronize()
        c0.record()
        for _ in range(5):
            hot_graph.replay()
        c1.record()
        torch.cuda.synchronize()
        hot_us = c0.elapsed_time(c1) * 1e3 / (5 * n_hot)
    bytes_avg = statistics.fmean(sum(c["bytes"] for c in sets[k % n_sets]["calls"]) for k in range(g_steps))
    flops_avg = statistics.fmean(sum(c["flops"] for c in sets[k % n_sets]["calls"]) for k in range(g_steps))
    hbm_peak, tc_peak, peak_kind = read_peaks()
    achieved_gbs = bytes_avg / calls_avg_s / 1e9

    # ---- end to end: host buffers in, result out, through the public API ----
    # Every step copies the ids and the projection calls' x and y0 from one pinned host
    # staging buffer into a device staging buffer (one copy), runs the step on views of
    # it through the public calls, and reads its y back into pinned host memory (one
    # copy).  The 13B forward stages layer 0's seven x / y0 in and reads layer 39's seven
    # y out.  When a step copies 8 MB or more in, the steps are pipelined as a serving
    # loop would run them: device staging slots take turns, the copies in and out run
    # on streams of their own, and step k + 1's copy in overlaps step k's calls and step
    # k - 1's read-back (both directions of the host link at once); a slot
    # is refilled once the step that last used it no longer needs what the copy
    # overwrites (its calls are done, and its outputs read back when they sit in the
    # staging buffer).  Smaller steps
    # (decode, tiny) are bound by the host's launches, where the extra streams and events
    # cost more than they hide: one slot, everything on the launching stream.  All of
    # every step's copies are inside the timed region.
    S0 = sets[0]
    if name == "mixed13b":
        ins = [c for c in S0["calls"] if c["layer"] == 0]
        outs_extra = [c for c in S0["calls"] if c["layer"] == 39]
    else:
        ins = S0["calls"]
        outs_extra = []
    pieces = [c["x"] for c in ins] + [y for c in ins for y in c["ys"]]
    offs, cur = [], 0
    for t in pieces:
        offs.append(cur)
        cur += (t.numel() * 2 + 255) // 256 * 256
    ids_off = cur
    cur += (S0["ids"].numel() * 4 + 255) // 256 * 256
    hstage = torch.empty(cur, dtype=torch.uint8).pin_memory()
    for t, o in zip(pieces, offs):  # the inputs' host copies
        hstage[o:o + t.numel() * 2].copy_(t.reshape(-1).view(torch.uint8).cpu())
    hstage[ids_off:ids_off + S0["ids"].numel() * 4].copy_(S0["ids"].view(torch.uint8).cpu())
    n_in = len(ins)
    y_lo, y_hi = offs[n_in], offs[-1] + pieces[-1].numel() * 2  # the staged y, contiguous
    pipelined = cur >= (8 << 20)
    # staging slots: three where the outputs sit in the staging buffer (a slot's read-back
    # then runs beside the next slot's copy in), two for the 13B forward (its outputs have
    # buffers of their own), one when not pipelined
    ns = (2 if name == "mixed13b" else 3) if pipelined else 1
    slots = []
    for _ in range(ns):
        dstage = torch.empty(cur, dtype=torch.uint8, device=dev)
        views = [dstage[o:o + t.numel() * 2].view(torch.bfloat16).view(t.shape) for t, o in zip(pieces, offs)]
        e_calls, k = [], n_in
        for i, c in enumerate(ins):
            e_calls.append(dict(c, x=views[i], ys=views[k:k + len(c["ys"])]))
            k += len(c["ys"])
        outs = []
        if name == "mixed13b":
            for c in S0["calls"]:
                if c["layer"] == 0:
                    continue
                if c["layer"] == 39:  # this slot's own outputs, read back while the other slot computes
                    ys = [y.clone() for y in c["ys"]]
                    outs += [(y, torch.empty(y.shape, dtype=torch.bfloat16).pin_memory()) for y in ys]
                    c = dict(c, ys=ys)
                e_calls.append(c)
        else:
            outs.append((dstage[y_lo:y_hi], torch.empty(y_hi - y_lo, dtype=torch.uint8).pin_memory()))
        e_ids = dstage[ids_off:ids_off + S0["ids"].numel() * 4].view(torch.int32)
        slots.append(dict(dstage=dstage, calls=e_calls, ids=e_ids, outs=outs, seg=B.Segments(S0["ids"].numel(), device=dev)
                          if not bgmv else None))
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(ns)]
    ev_comp = [torch.cuda.Event() for _ in range(ns)]
    ev_out = [torch.cuda.Event() for _ in range(ns)]
    e2e_steps = max(1, min(e2e_steps, steps))
    n_e2e = [0]

    def e2e_step():
        if not pipelined:
            sl = slots[0]
            sl["dstage"].copy_(hstage, non_blocking=True)
            if not bgmv:
                B.lora_segments_build(sl["ids"], n_ad, sl["seg"], mode=mode, err=err)
            for c in sl["calls"]:
                run_call(c, sl["ids"], sl["seg"])
            for d, h in sl["outs"]:
                h.copy_(d, non_blocking=True)
            return
        k = n_e2e[0]
        n_e2e[0] += 1
        q = k % ns
        sl = slots[q]
        with torch.cuda.stream(s_in):
            if k >= ns:
                # The step that last used this slot: once its calls are done its inputs are free,
                # unless its outputs sit in the staging buffer too, which must be read back first.
                # The 13B forward's outputs (layer 39's) do not, so its copy in runs beside the
                # read-back (the two directions of the host link at once).
                s_in.wait_event(ev_comp[q] if name == "mixed13b" else ev_out[q])
            sl["dstage"].copy_(hstage, non_blocking=True)
            ev_in[q].record(s_in)
        comp.wait_event(ev_in[q])
        if k >= ns and name == "mixed13b":
            comp.wait_event(ev_out[q])  # its outputs are read back before this step rewrites them
        if not bgmv:
            B.lora_segments_build(sl["ids"], n_ad, sl["seg"], mode=mode, err=err)
        for c in sl["calls"]:
            run_call(c, sl["ids"], sl["seg"])
        ev_comp[q].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[q])
            for d, h in sl["outs"]:
                h.copy_(d, non_blocking=True)
            ev_out[q].record(s_out)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e_value = sum_over_ranks(e2e_steps * S0["T"], world) / e2e_s
    h2d = cur
    d2h = sum(h.numel() * h.element_size() for _, h in slots[0]["outs"])

    grouped = any(len(c["views"]) > 1 for c in sets[0]["calls"])
    call = "lora_bgmv_ex (LORA_BGMV_STATIC_ADAPTERS)" if bgmv else \
        ("lora_apply / lora_apply_multi" if grouped else "lora_apply")
    kernels = "bgmv_kernel" if bgmv else ", ".join(B.apply_kernel_names())
    n_proj = sum(len(c["views"]) for c in sets[0]["calls"])
    out = {
        "value": value,
        "unit": UNIT,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": ms / steps,
        "config": {
            "workload": WORKLOAD_TEXT[name],
            "tokens_per_step": tokens_per_step,
            "segments": "none (one token per request)" if bgmv else ("GROUP" if mode == 0 else "CONTIGUOUS"),
            "step": ("%d x lora_bgmv_ex (LORA_BGMV_STATIC_ADAPTERS)" % n_calls) if bgmv else
                    ("lora_segments_build + %d grouped calls over %d projections" % (n_calls, n_proj) if grouped
                     else "lora_segments_build + %d x lora_apply" % n_calls),
            "l2": "inputs larger than L2: %d rotating input sets (%.0f MB in all, L2 %.0f MB)"
                  % (n_sets, n_sets * set_bytes / 1e6, l2 / 1e6),
            "timing": "CUDA graph of %d steps replayed; CUDA events on the launching stream" % g_steps,
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "%s x %d (%s)" % (call, n_calls, kernels),
            "achieved": achieved_gbs,
            "peak": hbm_peak,
            "unit": "GB/s",
            "frac": achieved_gbs / hbm_peak,
            "peak_kind": peak_kind + " (copy bandwidth, MEASURED_PEAKS.json)" if peak_kind == "measured"
            else peak_kind,
            "traffic": None,
            "traffic_note": "not measured in this run; DRAM bytes per call from ncu are summarised "
                            "under profiles/",
            "algorithmic_bytes_per_launch": bytes_avg,
            "avg_launch_us": calls_avg_s * 1e6,
            "calls_per_step": n_calls,
            "tflops": flops_avg / calls_avg_s / 1e12,
            "tensor_frac_of_bf16_peak": flops_avg / calls_avg_s / 1e12 / tc_peak,
        },
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "public calls, eager; every step's inputs copied in from pinned host memory and its y "
                        "read back inside the timed region; " +
                        ("pipelined over %d staging slots (step k + 1's copy in overlaps step k's calls and "
                         "step k - 1's read-back)" % ns if pipelined else "one slot, in order on the launching stream")},
        "call_timing": {"graph_us": calls_avg_s * 1e6, "single_launch_us": single_us, "hot_l2_us": hot_us,
                        "note": "the step's projection calls: graph-amortised over rotating sets (cold L2), "
                                "one eager launch group on an idle GPU, and one set repeated (warm L2)"},
        "gpu_launches": int(round(launches_per_step * steps)),
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                   "reasons": clocks["reasons"], "samples": clocks["samples"]},
    }
    del sets, graph, graph_rem, call_graph, slots, hstage
    gc.collect()
    torch.cuda.empty_cache()
    return out


def gpu_sample(name: str, local: int):
    """The CPU sample's projection calls on the GPU, from fresh copies of the same host
    inputs: y through lora_apply (bf16, in place) and through lora_apply_f32y (fp32)."""
    import torch

    from segmented_gather_gemm_lora_gb300 import binding as B

    dev = torch.device("cuda", local)
    wl, calls, _ = oracle_sample(name)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ids = torch.from_numpy(wl.batch.ids).to(dev)
    seg = B.Segments(wl.batch.T, device=dev)
    B.lora_segments_build(ids, wl.n_adapters, seg, mode=wl.mode, err=err)
    outs = []
    for pool, b in calls:
        view = B.PoolView.from_host(pool, device=dev)
        x = up(b.x)
        y = up(b.y0)
        yf = torch.empty(y.shape, dtype=torch.float32, device=dev)
        if name == "decode":
            B.lora_bgmv(x, y, ids, view, err=err)
        else:
            B.lora_apply(x, y, seg, view, err=err)
        B.lora_apply_f32y(x, up(b.y0), yf, seg, view, err=err)
        torch.cuda.synchronize()
        outs.append((y.view(torch.int16).cpu().numpy().view(np.uint16), yf.cpu().numpy()))
    assert int(err.item()) == 0, "device error word %d" % int(err.item())
    return outs


def parity_report(gpu_outs, oracle_ys, d_outs):
    """Raw max |err| and relative L2 of the GPU outputs against the oracle's, for the bf16
    output (gate: 2e-2 plus half a bf16 ulp of the oracle value) and the fp32 output
    (literal 2e-2)."""
    from segmented_gather_gemm_lora_gb300 import workloads as W

    mx16 = mx32 = 0.0
    num16 = num32 = den = 0.0
    gate_ok = True
    for (ybits, yf), ref, d_out in zip(gpu_outs, oracle_ys, d_outs):
        g16 = W.bf16_bits_to_f32(ybits[:, :d_out]).astype(np.float64)
        g32 = yf[:, :d_out].astype(np.float64)
        e16 = np.abs(g16 - ref)
        e32 = np.abs(g32 - ref)
        half_ulp = 0.5 * np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 7)
        gate_ok = gate_ok and bool((e16 <= 2e-2 + half_ulp).all())
        mx16 = max(mx16, float(e16.max(initial=0.0)))
        mx32 = max(mx32, float(e32.max(initial=0.0)))
        num16 += float((e16 ** 2).sum())
        num32 += float((e32 ** 2).sum())
        den += float((ref ** 2).sum())
    rel16 = math.sqrt(num16 / den) if den > 0 else 0.0
    rel32 = math.sqrt(num32 / den) if den > 0 else 0.0
    return {"bf16_y": {"max_abs_err": mx16, "rel_l2": rel16, "gate": "max|err| <= 2e-2 + half a bf16 ulp; "
                       "rel L2 <= 5e-3", "pass": gate_ok and rel16 <= 5e-3},
            "f32_y": {"max_abs_err": mx32, "rel_l2": rel32, "gate": "max|err| <= 2e-2; rel L2 <= 5e-3",
                      "pass": mx32 <= 2e-2 and rel32 <= 5e-3},
            "against": "the CPU fp64 oracle on the CPU baseline's sample"}


def backward_bytes(batch, pool) -> int:
    """Bytes one backward call must move at least once: x and dy read, dx read and
    written (bf16), every distinct adapter's A and B read (bf16) and their fp32
    gradients read and written."""
    ids = batch.ids
    valid = ids >= 0
    n = int(valid.sum())
    ranks = pool.ranks[np.unique(ids[valid])].astype(np.int64)
    elems = int((ranks * (pool.d_in + pool.d_out)).sum())
    return n * pool.d_in * 2 + n * pool.d_out * 2 + n * pool.d_in * 4 + elems * 2 + elems * 8


def pipelined_e2e(torch, dev, inputs, run, n_out, steps, world, tokens):
    """End to end through the public calls for the lines of one call per step:
    `inputs` (device tensors: the step's inputs, the ones it updates in place first)
    are copied in every step from one pinned host buffer into one of three device staging
    slots, `run(views)` enqueues the step on the current stream on that slot's copies,
    and the first `n_out` of them (the step's result) are read back into pinned host
    memory.  Step k + 1's copy in runs under step k's calls and beside step k - 1's
    read-back (the two directions of the host link at once), on streams of their own; a
    slot is refilled once the step that last used it has been read back.  Returns
    (tokens/s, bytes in, bytes out per step)."""
    offs, cur = [], 0
    for t in inputs:
        offs.append(cur)
        cur += (t.numel() * t.element_size() + 255) // 256 * 256
    hstage = torch.empty(cur, dtype=torch.uint8).pin_memory()
    for t, o in zip(inputs, offs):
        hstage[o:o + t.numel() * t.element_size()].copy_(t.reshape(-1).view(torch.uint8).cpu())
    out_end = offs[n_out - 1] + inputs[n_out - 1].numel() * inputs[n_out - 1].element_size()
    ns = 3
    slots = []
    for _ in range(ns):
        d = torch.empty(cur, dtype=torch.uint8, device=dev)
        views = [d[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(inputs, offs)]
        slots.append((d, views, torch.empty(out_end, dtype=torch.uint8).pin_memory()))
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(ns)]
    ev_comp = [torch.cuda.Event() for _ in range(ns)]
    ev_out = [torch.cuda.Event() for _ in range(ns)]

    def one(k):
        q = k % ns
        d, views, hout = slots[q]
        with torch.cuda.stream(s_in):
            if k >= ns:
                s_in.wait_event(ev_out[q])  # the step that last used this slot has been read back
            d.copy_(hstage, non_blocking=True)
            ev_in[q].record(s_in)
        comp.wait_event(ev_in[q])
        run(views)
        ev_comp[q].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[q])
            hout.copy_(d[:out_end], non_blocking=True)
            ev_out[q].record(s_out)

    for k in range(3):
        one(k)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for k in range(3, 3 + steps):
        one(k)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    del slots, hstage
    return sum_over_ranks(steps * tokens, world) / e2e_s, cur, out_end


def run_backward_line(steps, warmup, soak_seconds, world, rank, local):
    """The backward pass (adapter training) on the prefill-shaped batch: a step is
    lora_segments_build + lora_sgmv_backward (dA, dB into an fp32 gradient pool, dx
    in place); inputs rotate over enough sets to exceed 2x L2."""
    import torch

    from segmented_gather_gemm_lora_gb300 import binding as B
    from segmented_gather_gemm_lora_gb300 import workloads as W

    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    sets, k = [], 0
    while True:
        wl = W.prefill(1000 * rank + k)
        pool, b = wl.pools[0], wl.batch
        rng = np.random.default_rng([1000 * rank + k, 9])
        dy = W._normal_bf16(rng, (b.T, pool.d_out), 1.0)
        S = dict(view=B.PoolView.from_host(pool, device=dev), x=up(b.x), dy=up(dy),
                 dx=torch.zeros((b.T, pool.d_in), dtype=torch.bfloat16, device=dev),
                 grad=torch.zeros(pool.pool.shape, dtype=torch.float32, device=dev),
                 hu=torch.empty((2 * b.T, 64), dtype=torch.float32, device=dev),
                 ids=torch.from_numpy(b.ids).to(dev), seg=B.Segments(b.T, device=dev),
                 T=int((b.ids >= 0).sum()), n_ad=wl.n_adapters,
                 bytes=backward_bytes(b, pool), flops=3 * algorithmic_flops(b, pool))
        sets.append(S)
        k += 1
        if k >= 2 and sum(x["x"].numel() * 2 + x["dy"].numel() * 2 + x["dx"].numel() * 2 for x in sets) > 2 * l2:
            break
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(i):
        S = sets[i % len(sets)]
        B.lora_segments_build(S["ids"], S["n_ad"], S["seg"], mode=B.LORA_SEG_GROUP, err=err)
        B.lora_sgmv_backward(S["x"], S["dy"], S["dx"], S["grad"], S["hu"], S["seg"], S["view"], err=err)

    for i in range(max(warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    g_steps = len(sets) * max(1, 32 // len(sets))
    cap = torch.cuda.Stream(device=dev)
    graph = torch.cuda.CUDAGraph()
    launches0 = B.launch_count()
    with torch.cuda.graph(graph, stream=cap):
        for i in range(g_steps):
            step(i)
    launches_per_step = (B.launch_count() - launches0) / g_steps
    reps = max(1, steps // g_steps)
    graph.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_id_of(props))
    t_end = time.perf_counter() + soak_seconds
    while time.perf_counter() < t_end:
        graph.replay()
        torch.cuda.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    assert int(err.item()) == 0, "device error word %d" % int(err.item())
    S0 = sets[0]

    def run_bw(vw):  # dx (updated in place, read back), x, dy, ids
        B.lora_segments_build(vw[3], S0["n_ad"], S0["seg"], mode=B.LORA_SEG_GROUP, err=err)
        B.lora_sgmv_backward(vw[1], vw[2], vw[0], S0["grad"], S0["hu"], S0["seg"], S0["view"], err=err)

    e2e_value, e2e_in, e2e_out = pipelined_e2e(torch, dev, [S0["dx"], S0["x"], S0["dy"], S0["ids"]], run_bw, 1,
                                               min(steps, 50), world, S0["T"])
    n_steps = reps * g_steps
    tokens = sum_over_ranks(reps * sum(sets[i % len(sets)]["T"] for i in range(g_steps)), world)
    bytes_avg = statistics.fmean(sets[i % len(sets)]["bytes"] for i in range(g_steps))
    flops_avg = statistics.fmean(sets[i % len(sets)]["flops"] for i in range(g_steps))
    step_s = ms / n_steps / 1e3
    hbm_peak, tc_peak, peak_kind = read_peaks()
    achieved = bytes_avg / step_s / 1e9
    out = {
        "value": tokens / (ms / 1e3),
        "unit": UNIT,
        "steps": n_steps,
        "ms_per_step": ms / n_steps,
        "config": {"workload": "backward (adapter training) on the prefill SGMV batch: 32 requests of "
                               "U{64..512} tokens, 4096->4096, 200 rank-16 adapters, Zipf(1.1); dA, dB into an "
                               "fp32 gradient pool and dx in place, bf16 x and dy",
                   "step": "lora_segments_build + lora_sgmv_backward",
                   "l2": "inputs larger than L2: %d rotating input sets" % len(sets),
                   "timing": "CUDA graph of %d steps replayed; CUDA events on the launching stream" % g_steps},
        "roofline": {"bound": "hbm", "kernel": "lora_sgmv_backward (fused_tc shrink-only for h, fused_tc apply "
                                               "over the transposed adapters for u and dx, grad_kernel; gather "
                                               "for short segments)",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "peak_kind": peak_kind, "traffic": None,
                     "algorithmic_bytes_per_launch": bytes_avg, "avg_launch_us": step_s * 1e6,
                     "tflops": flops_avg / step_s / 1e12},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": e2e_in, "d2h_bytes_per_step": e2e_out,
                "note": "lora_segments_build + lora_sgmv_backward, eager; x, dy, dx and the ids copied in from "
                        "pinned host memory and dx read back every step (the gradient pool stays on the device "
                        "for the optimizer), pipelined over three staging slots"},
        "gpu_launches": int(round(launches_per_step * n_steps)),
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                   "reasons": clocks["reasons"], "samples": clocks["samples"]},
    }
    del sets, graph
    gc.collect()
    torch.cuda.empty_cache()
    return out


def run_base_line(steps, warmup, soak_seconds, world, rank, local):
    """The base projection with the adapter term in its epilogue on the prefill batch: a
    step is lora_segments_build + lora_base_apply (y = x W0^T + s_i (x A_i^T) B_i, y written
    once) with a random 4096 x 4096 W0; timed beside cuBLAS's x W0^T followed by
    lora_apply, the unfused way to the same y.  Two input sets rotate (each larger than L2)."""
    import torch

    from segmented_gather_gemm_lora_gb300 import binding as B
    from segmented_gather_gemm_lora_gb300 import workloads as W

    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    sets = []
    for k in range(2):
        wl = W.prefill(1000 * rank + k)
        pool, b = wl.pools[0], wl.batch
        g = torch.Generator(device=dev)
        g.manual_seed(1000 * rank + k)
        w0 = (torch.randn(pool.d_out, pool.d_in, generator=g, device=dev) / float(np.sqrt(pool.d_in))).to(torch.bfloat16)
        S = dict(view=B.PoolView.from_host(pool, device=dev), x=up(b.x), y=torch.empty((b.T, pool.d_out),
                 dtype=torch.bfloat16, device=dev), w0=w0, ids=torch.from_numpy(b.ids).to(dev),
                 seg=B.Segments(b.T, device=dev), T=b.T, n_ad=wl.n_adapters,
                 flops=2 * b.T * pool.d_in * pool.d_out + algorithmic_flops(b, pool))
        sets.append(S)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def fused(i):
        S = sets[i % 2]
        B.lora_segments_build(S["ids"], S["n_ad"], S["seg"], mode=B.LORA_SEG_CONTIGUOUS, err=err)
        B.lora_base_apply(S["x"], S["w0"], S["y"], S["ids"], S["seg"], S["view"], err=err)

    def unfused(i):
        S = sets[i % 2]
        B.lora_segments_build(S["ids"], S["n_ad"], S["seg"], mode=B.LORA_SEG_CONTIGUOUS, err=err)
        torch.matmul(S["x"], S["w0"].t(), out=S["y"])
        B.lora_apply(S["x"], S["y"], S["seg"], S["view"], err=err)

    def graph_of(fn, n):
        for i in range(max(warmup, 3)):
            fn(i)
        torch.cuda.synchronize()
        cap = torch.cuda.Stream(device=dev)
        gr = torch.cuda.CUDAGraph()
        l0 = B.launch_count()
        with torch.cuda.graph(gr, stream=cap):
            for i in range(n):
                fn(i)
        return gr, (B.launch_count() - l0) / n

    def timed(gr, reps, n):
        gr.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        barrier(world)
        e0.record()
        for _ in range(reps):
            gr.replay()
        e1.record()
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1), world) / (reps * n)

    n = 10
    reps = max(1, steps // n)
    g_f, launches_per_step = graph_of(fused, n)
    g_u, _ = graph_of(unfused, n)
    sampler = ClockSampler(gpu_id_of(props))
    t_end = time.perf_counter() + soak_seconds
    while time.perf_counter() < t_end:
        g_f.replay()
        torch.cuda.synchronize()
    ms_f = timed(g_f, reps, n)
    clocks = sampler.stop()
    ms_u = timed(g_u, reps, n)
    assert int(err.item()) == 0, "device error word %d" % int(err.item())
    S0 = sets[0]

    def run_base(vw):  # y (written, read back), x, ids
        B.lora_segments_build(vw[2], S0["n_ad"], S0["seg"], mode=B.LORA_SEG_CONTIGUOUS, err=err)
        B.lora_base_apply(vw[1], S0["w0"], vw[0], vw[2], S0["seg"], S0["view"], err=err)

    e2e_value, e2e_in, e2e_out = pipelined_e2e(torch, dev, [S0["y"], S0["x"], S0["ids"]], run_base, 1,
                                               min(steps, 50), world, S0["T"])
    tokens = sum_over_ranks(statistics.fmean(S["T"] for S in sets), world)
    flops = statistics.fmean(S["flops"] for S in sets)
    step_s = ms_f / 1e3
    hbm_peak, tc_peak, peak_kind = read_peaks()
    tc_sustained = tc_peak
    try:
        tc_sustained = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))).get("bf16_tflops_sustained",
                                                                                            tc_peak))
    except Exception:
        pass
    achieved = flops / step_s / 1e12
    out = {
        "value": tokens / step_s,
        "unit": UNIT,
        "steps": reps * n,
        "ms_per_step": ms_f,
        "config": {"workload": "base projection with the adapter term in its epilogue on the prefill SGMV batch: "
                               "32 requests of U{64..512} tokens, y = x W0^T + s_i (x A_i^T) B_i with a random "
                               "4096 x 4096 bf16 W0, 200 rank-16 adapters, Zipf(1.1), contiguous segments",
                   "step": "lora_segments_build + lora_base_apply (shrink, then the tcgen05 base GEMM with the "
                           "adapter term on the tensor cores into the same accumulator; y written once)",
                   "l2": "inputs larger than L2: 2 rotating input sets",
                   "timing": "CUDA graph of %d steps replayed; CUDA events on the launching stream" % n,
                   "unfused_ms_per_step": ms_u,
                   "unfused": "lora_segments_build + cuBLAS x W0^T (torch.matmul) + lora_apply, same inputs"},
        "roofline": {"bound": "tensor", "kernel": "lora_base_apply (base_gemm_kernel and the shrink before it)",
                     "achieved": achieved, "peak": tc_sustained, "unit": "TFLOP/s",
                     "frac": achieved / tc_sustained,
                     "peak_kind": "measured sustained bf16 (cuBLAS loop, MEASURED_PEAKS.json)", "traffic": None,
                     "flops_per_step": flops, "avg_launch_us": step_s * 1e6},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": e2e_in, "d2h_bytes_per_step": e2e_out,
                "note": "lora_segments_build + lora_base_apply, eager; x and the ids copied in from pinned host "
                        "memory and y read back every step (W0 and the adapters resident), pipelined over three "
                        "staging slots"},
        "gpu_launches": int(round(launches_per_step * reps * n)),
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                   "reasons": clocks["reasons"], "samples": clocks["samples"]},
    }
    del sets, g_f, g_u
    gc.collect()
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------ CPU oracle --

def oracle_sample(workload: str):
    """The host calls the CPU oracle runs for one step of `workload`, and how many calls of
    that size one step makes per sampled call (the 13B forward samples layer 0's q
    projection for its 280 calls)."""
    wl = make_workload(workload, 0)
    return wl, host_calls(wl, 0), (280 if workload == "mixed13b" else 1)


def oracle_pass(oracle, calls):
    return [oracle.lora_apply(b.x, b.y0, b.ids, pool)[0] for pool, b in calls]


def sample_text(wl, calls, scale, reps):
    if scale > 1:
        return ("layer 0's q projection (%d tokens) %d times; one forward counted as %d such calls"
                % (wl.batch.T, reps, scale))
    return "the full batch (%d tokens) through the step's %d projection call(s), %d times" % (
        wl.batch.T, len(calls), reps)


def _oracle_worker(workload: str, part: int, n_parts: int, seconds: float, start):
    """One process of the all-cores oracle timing: the step's calls on the tokens
    part, part + n_parts, ... of the batch (tokens are independent), repeated for a
    bounded time after every process is ready; (tokens, seconds)."""
    import oracle

    wl, calls, _ = oracle_sample(workload)
    sub = []
    for pool, b in calls:
        idx = np.arange(part, b.T, n_parts)
        sub.append((pool, b.x[idx], b.y0[idx], b.ids[idx]))
    n_tok = sum(int((ids >= 0).sum()) for _, _, _, ids in sub[:1])
    oracle.lora_apply(sub[0][1][:1], sub[0][2][:1], sub[0][3][:1], sub[0][0])
    start.wait()
    reps = 0
    t0 = time.perf_counter()
    while True:
        for pool, x, y0, ids in sub:
            oracle.lora_apply(x, y0, ids, pool)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return reps * n_tok, time.perf_counter() - t0


def oracle_all_cores(workload: str, seconds: float):
    """The oracle on every host core: one spawned process per core, each on an
    interleaved share of the batch's tokens; tokens/s summed over the processes."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor

    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        start = m.Barrier(n)
        with ProcessPoolExecutor(max_workers=n, mp_context=ctx) as ex:
            res = list(ex.map(_oracle_worker, [workload] * n, range(n), [n] * n, [seconds] * n, [start] * n))
    return sum(t / dt for t, dt in res), n


def cpu_baseline(workload: str, seconds: float):
    """The fp64 oracle as it stands, single-threaded, on the step's calls repeated for a
    bounded time; tokens/s.  Also the same oracle on every host core.  Returns the
    baseline and the oracle's outputs of one pass (for the parity sample)."""
    import oracle

    wl, calls, scale = oracle_sample(workload)
    b = wl.batch
    n_tok = int((b.ids >= 0).sum())
    oracle.lora_apply(b.x[:1], b.y0[:1], b.ids[:1], calls[0][0])  # load/compile outside the clock
    reps = 0
    ys = None
    t0 = time.perf_counter()
    while True:
        out = oracle_pass(oracle, calls)
        ys = out if ys is None else ys
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    res = {"value": reps * n_tok / dt / scale, "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": sample_text(wl, calls, scale, reps) + ", %.1f s" % dt}
    try:
        v, n = oracle_all_cores(workload, seconds)
        res["all_cores"] = {"value": v / scale, "cores": n,
                            "sample": "the same calls split by token over %d spawned processes, %.0f s each"
                                      % (n, seconds)}
    except (OSError, RuntimeError, EOFError) as e:  # a host without process support
        res["all_cores"] = {"unavailable": str(e)[:200]}
    return res, ys, [pool.d_out for pool, _ in calls]


def cpu_baseline_line(kind: str, seconds: float):
    """The fp64 oracle as it stands, single-threaded, for the backward ("backward":
    oracle.lora_backward) or the fused base projection ("base_fused": oracle.base_apply)
    on the first tokens of the same prefill batch, repeated for a bounded time; tokens/s.
    The sample is sized so that one pass takes about a quarter of the time."""
    import oracle
    from segmented_gather_gemm_lora_gb300 import workloads as W

    wl = W.prefill(0)
    pool, b = wl.pools[0], wl.batch
    rng = np.random.default_rng([0, 9])
    if kind == "backward":
        g = W._normal_bf16(rng, (b.T, pool.d_out), 1.0)
        run = lambda n: oracle.lora_backward(b.x[:n], g[:n], b.ids[:n], pool)
        what = "oracle.lora_backward (h, u, dA, dB, dx)"
    else:
        w0 = W.f32_to_bf16_bits((rng.standard_normal((pool.d_out, pool.d_in)) / 64.0).astype(np.float32))
        run = lambda n: oracle.base_apply(b.x[:n], w0, b.ids[:n], pool)
        what = "oracle.base_apply (x W0^T and the adapter term)"
    t1 = time.perf_counter()
    run(8)
    per_tok = (time.perf_counter() - t1) / 8
    n = int(min(b.T, max(8, seconds / 4 / max(per_tok, 1e-9))))
    n_tok = int((b.ids[:n] >= 0).sum())
    reps = 0
    t0 = time.perf_counter()
    while True:
        run(n)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": reps * n_tok / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "%s on the batch's first %d tokens, %d times, %.1f s" % (what, n, reps, dt)}


def run_reference(args, world, rank):
    """The reference arm: the CPU fp64 oracle, unchanged, over the step's calls on every
    host core (one spawned process per core, each on an interleaved share of the tokens),
    for about K steps' worth of work, bounded to a minute; the single-core rate alongside."""
    import oracle

    name = HEADLINE if args.workload == "all" else args.workload
    if name in ("backward", "base_fused"):  # the oracle's backward or base projection, on one core
        from segmented_gather_gemm_lora_gb300 import workloads as W

        step_tokens = W.prefill(0).batch.T
        base = cpu_baseline_line(name, min(60.0, max(5.0, float(args.steps))))
        return {"impl": "reference", "metric": METRIC, "value": base["value"], "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": step_tokens / base["value"] * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": name + " on the prefill SGMV batch",
                           "step": "the CPU fp64 oracle (%s)" % base["sample"]},
                "cpu_baseline": base,
                "e2e": {"value": base["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    wl, calls, scale = oracle_sample(name)
    b = wl.batch
    n_tok = int((b.ids >= 0).sum())
    oracle_pass(oracle, calls)  # load outside the clock
    t1 = time.perf_counter()
    oracle_pass(oracle, calls)
    one = time.perf_counter() - t1
    single = n_tok / one / scale
    try:
        n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        seconds = min(60.0, max(5.0, args.steps * one / max(n, 1)))
        value, n = oracle_all_cores(name, seconds)
        value /= scale
        how = "the step's calls split by token over %d spawned processes, %.0f s" % (n, seconds)
    except (OSError, RuntimeError, EOFError):  # a host without process support: one core
        n, value, seconds = 1, single, one
        how = "one pass of the step's calls on one core"
    ms = b.T / value * 1e3 if name != "mixed13b" else 4224 / value * 1e3
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[name],
                   "step": "the CPU fp64 oracle over the step's projection calls"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": n, "kind": "oracle",
                         "sample": how + "; one core: %.4g tokens/s (%s)" % (single, sample_text(wl, calls, scale, 1))},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------- main --

def config_line(name, args, world, rank, local, steps):
    out = run_workload(name, steps, args.warmup, default_e2e_steps(name, args), args.soak_seconds,
                       world, rank, local)
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        base, ys, d_outs = cpu_baseline(name, args.cpu_seconds)
        out["cpu_baseline"] = base
        out["parity"] = parity_report(gpu_sample(name, local), ys, d_outs)
    return out


def head_line(head, args, world, rank, local):
    """The line of the workload the JSON line leads with: the backward and base-projection
    lines have runners of their own (and their single-core oracle baseline, on rank 0 of a
    one-process run when --cpu-seconds is above zero); every other workload is a config line."""
    if head == "backward":
        h = run_backward_line(args.steps, args.warmup, args.soak_seconds, world, rank, local)
    elif head == "base_fused":
        h = run_base_line(args.steps, args.warmup, args.soak_seconds, world, rank, local)
    else:
        return config_line(head, args, world, rank, local, args.steps)
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        h["cpu_baseline"] = cpu_baseline_line(head, args.cpu_seconds)
    return h


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_info()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world, rank)), flush=True)
        return 0
    import torch

    if world > 1:
        import torch.distributed as dist

        dist.init_process_group(backend="nccl")
    torch.cuda.set_device(local)
    head = HEADLINE if args.workload == "all" else args.workload
    per_config = {}
    if args.workload == "all":
        for name in OTHERS:
            per_config[name] = config_line(name, args, world, rank, local, OTHER_STEPS[name])
        per_config["backward"] = run_backward_line(BACKWARD_STEPS, args.warmup, args.soak_seconds, world, rank,
                                                   local)
        per_config["base_fused"] = run_base_line(BASE_STEPS, args.warmup, args.soak_seconds, world, rank, local)
        if rank == 0 and world == 1 and args.cpu_seconds > 0:
            for k in ("backward", "base_fused"):
                per_config[k]["cpu_baseline"] = cpu_baseline_line(k, args.cpu_seconds)
    h = head_line(head, args, world, rank, local)
    out = {
        "metric": METRIC,
        "value": h["value"],
        "unit": UNIT,
        "n_gpus": world,
        "steps": h.get("steps", args.steps),
        "warmup": args.warmup,
        "ms_per_step": h["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
    }
    for k in ("config", "roofline", "e2e", "call_timing", "gpu_launches", "clocks", "cpu_baseline", "parity"):
        if k in h:
            out[k] = h[k]
    if per_config:
        out["per_config"] = per_config
        out["gpu_launches_all_configs"] = h["gpu_launches"] + sum(c["gpu_launches"] for c in per_config.values())
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
