#!/usr/bin/env python
"""Benchmark of the slot-cached MoE layer forward on GB300.

Default workload (one "step" = one full layer forward: route, permute,
expert_cache_manage, expert_cache_gather on a side stream, grouped SwiGLU
FFN, combine): a Qwen3-30B-A3B-shaped decode layer, T=64 tokens, hidden 2048,
128 experts, top-8, intermediate 768, bf16, 64 of 128 experts in the VRAM slot
pool, the rest in pinned host memory, LRU, expert-wave schedule (each missing
expert loaded at most once per step).  Each step gets a fresh seeded batch,
so the routing (near-uniform) changes every step and the cache sees a steady
miss stream.  Inputs are synthetic (no weights or traces exist here).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0), kept short; its last key, ``targets``, holds
the other workloads' figures (all-resident decode, prefill, token chunks,
W8A8, the 48-layer stack).  --impl reference times the CPU oracle on the host
cores on a bounded sample of the same workload.  N > 1 (under torchrun) runs
N independent replicas, one per GPU: the path has no exchange step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from typing import Optional

if "--impl" in sys.argv and "reference" in sys.argv:
    # the oracle leg: pin the BLAS pools before numpy loads, so "cores" is exact
    _thr = os.environ.get("MOE_ORACLE_THREADS", str(os.cpu_count() or 1))
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = _thr

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from harness import configs as C  # noqa: E402

# DRAM bytes (read + write) of gather_kernel per missed Qwen-shaped expert, from an ncu capture of
# the gather_T8 workload: 161,741,568 B written + 224,512 B read for a launch of 17 misses (the host
# side travels over NVLink-C2C and is not DRAM traffic).  Valid while the gather kernel is unchanged.
GATHER_DRAM_BYTES_PER_MISS = (161_741_568 + 224_512) / 17
METRIC = "MoE-layer tokens/s at 1 GB300; decode HBM GB/s vs roofline; prefill TFLOP/s"
UNIT = "tokens/s"
PROF_NAMES = ("route", "permute", "manage", "gather", "ffn_gateup", "ffn_down", "combine", "ffn_rows", "decode")


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ----------------------------------------------------------------------------

def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        return ws, rank, local, dist
    return 1, 0, local, None


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def _max_over_ranks(v: float, dist) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0])


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        time.sleep(0.25)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.f.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------
# workload setup
# ----------------------------------------------------------------------------

class Workload:
    """One layer's weights, slot pool, host store, cache state and input batches."""

    def __init__(self, cfg: C.LayerConfig, n_batches: int, dev: str, quant: bool = False):
        import expert_slot_cache_gb300 as M
        self.cfg, self.dev, self.M = cfg, dev, M
        self.quant = quant
        self.wr = C.draw_router(cfg, dev)
        slabs = torch.empty(cfg.E, cfg.slab_elems, dtype=torch.bfloat16, device=dev)
        C.draw_slabs(cfg, dev, out=slabs)
        if quant:  # W8A8 slabs (weights + slot-indexed scales)
            qs = M.quantize_slabs(slabs, cfg.H, cfg.I)
            del slabs
            slabs = qs
        self.slab_bytes = slabs[0].numel() * slabs.element_size()
        self.off = C.draw_logit_offset(cfg, dev)
        self.bias = None
        if cfg.bias_cap is not None:
            b, _ = C.draw_brightness(cfg)
            self.bias = M.bias_table(torch.from_numpy(b).to(dev), cfg.n_hot, cfg.bias_cap)
        if cfg.mode == C.MODE_RESIDENT:
            self.host, self.pool, self.state = None, slabs, None
        else:
            self.host = torch.empty(slabs.shape, dtype=slabs.dtype, pin_memory=True)
            self.host.copy_(slabs)
            s2e0 = C.initial_residency(cfg)
            self.pool = slabs[torch.from_numpy(s2e0.astype(np.int64)).to(dev)].contiguous()
            del slabs
            self.state = M.CacheState.from_slots(s2e0, cfg.E, dev)
        self.layer = M.SlotCachedMoELayer(self.wr, self.pool, cfg.k, cfg.I, cfg.mode, cfg.policy,
                                          host_slabs=self.host, state=self.state, logit_offset=self.off,
                                          sel_bias=self.bias, max_tokens=cfg.T, quant=int(quant),
                                          schedule=cfg.schedule)
        self.xs = [C.draw_x(cfg, dev, step=i) for i in range(n_batches)]
        self.out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=dev)
        self.out_res = self.out_miss = None
        if cfg.mode == C.MODE_ZERO_RETURN:
            self.out_res = torch.empty(cfg.T, cfg.H, dtype=torch.float32, device=dev)
            self.out_miss = torch.empty(cfg.T, cfg.H, dtype=torch.float32, device=dev)
        self.ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=dev)
        self.w = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=dev)

    def chunk(self) -> int:
        c = self.cfg
        if c.mode != C.MODE_GATHER or c.S >= c.E or c.T * c.k <= c.S or c.schedule == C.SCHED_WAVES:
            return c.T
        return c.S // c.k

    def step(self, i, prof=None, x=None):
        return self.layer.forward(self.xs[i] if x is None else x, out=self.out, ids=self.ids, w=self.w,
                                  out_res=self.out_res, out_miss=self.out_miss, prof=prof)

    def unique_per_chunk(self, ids: np.ndarray) -> int:
        C_ = self.chunk()
        return sum(len(np.unique(ids[t0:t0 + C_])) for t0 in range(0, ids.shape[0], C_))


class StackWorkload:
    """The 48-layer stack: per-layer router, experts, pool and cache state."""

    def __init__(self, cfg: C.LayerConfig, dev: str, layers: Optional[int] = None, steps: int = 0):
        import expert_slot_cache_gb300 as M
        self.cfg, self.dev, self.M = cfg, dev, M
        L = cfg.layers if layers is None else layers
        self.L = L
        self.hosts, self.layers = [], []
        for l in range(L):
            wr = C.draw_router(cfg, dev, l)
            slabs = torch.empty(cfg.E, cfg.slab_elems, dtype=torch.bfloat16, device=dev)
            C.draw_slabs(cfg, dev, l, out=slabs)
            if cfg.mode == C.MODE_RESIDENT:
                host, pool, state = None, slabs, None
            else:
                host = torch.empty(cfg.E, cfg.slab_elems, dtype=torch.bfloat16, pin_memory=True)
                host.copy_(slabs)
                s2e0 = C.initial_residency(cfg, l)
                pool = slabs[torch.from_numpy(s2e0.astype(np.int64)).to(dev)].contiguous()
                del slabs
                state = M.CacheState.from_slots(s2e0, cfg.E, dev)
            self.hosts.append(host)
            self.layers.append(M.SlotCachedMoELayer(wr, pool, cfg.k, cfg.I, cfg.mode, cfg.policy, host_slabs=host,
                                                    state=state, max_tokens=cfg.T, schedule=cfg.schedule))
        self.stack = M.LayerStack(self.layers, cfg.T)
        # inputs of every step and layer, drawn up front: [steps][L][T][H]
        self.inputs = torch.empty(max(steps, 1), L, cfg.T, cfg.H, dtype=torch.bfloat16, device=dev)
        for st in range(steps):
            for l in range(L):
                self.inputs[st, l].copy_(C.draw_x(cfg, dev, layer=l, step=st))

    def load_step(self, st: int):
        self.stack.x_all.copy_(self.inputs[st])


def stack_variant(dev: str, peaks: dict, cfg: "C.LayerConfig", steps: int = 8, warmup: int = 3) -> dict:
    """The 48-layer decode stack (288 experts per layer, top-8, H 2048, I 512,
    T = 32; all 48 layers as one CUDA-graph replay per step): tokens/s and,
    all-resident, HBM GB/s on unique expert bytes (Betelgeuse's single-graph
    decode over every layer).  Each step's inputs (48 x T x H) are copied into
    place inside the timed region; the unique experts per layer and chunk come
    from a second, untimed replay of the same steps."""
    wl = StackWorkload(cfg, dev, steps=warmup + steps)
    wl.load_step(0)
    wl.stack._run()
    torch.cuda.synchronize()
    wl.stack.capture()
    for st in range(warmup):
        wl.load_step(st)
        wl.stack.replay()
    torch.cuda.synchronize()
    misses0 = sum(int(l.stats[0]) for l in wl.layers)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for st in range(warmup, warmup + steps):
        wl.load_step(st)
        wl.stack.replay()
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e)
    misses = sum(int(l.stats[0]) for l in wl.layers) - misses0
    slots = sum(C.layer_S(cfg, l) for l in range(wl.L)) if cfg.mode != C.MODE_RESIDENT else wl.L * cfg.E
    out = {"config": f"{cfg.name}: {wl.L} layers x {cfg.E} experts, T={cfg.T}, k={cfg.k}, H={cfg.H}, I={cfg.I}, "
                     f"{slots} slots, {'all resident' if cfg.mode == C.MODE_RESIDENT else 'slot pool + pinned host'}",
           "tokens_per_s": cfg.T * steps / (ms * 1e-3), "ms_per_step": ms / steps,
           "expert_GB_in_hbm": slots * cfg.slab_bytes / 1e9}
    if cfg.mode == C.MODE_RESIDENT:
        units = 0
        C_ = cfg.T  # all-resident: one chunk per layer
        for st in range(warmup, warmup + steps):
            wl.load_step(st)
            wl.stack.replay()
            torch.cuda.synchronize()
            for l in range(wl.L):
                ids = wl.stack.ids[l].cpu().numpy()
                units += sum(len(np.unique(ids[t0:t0 + C_])) for t0 in range(0, cfg.T, C_))
        byts = units * cfg.slab_bytes
        out["unique_expert_GB_per_step"] = byts / steps / 1e9
        out["hbm"] = {"bound": "hbm", "achieved": byts / (ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                      "frac": byts / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], "of": "whole step (48 layers)"}
    else:
        out["misses_per_step"] = misses / steps
        out["host_link_GB_per_step"] = misses * cfg.slab_bytes / steps / 1e9
    del wl
    torch.cuda.empty_cache()
    return out


def w8a8_variants(dev: str, peaks: dict, steps: int = 10, warmup: int = 3, decode_kernels: int = 0) -> dict:
    """W8A8 experts (the vllm-expert-cache page's W8A8 model; scales
    slot-indexed inside the slab): the all-resident decode layer at T = 1, 8,
    64 (HBM GB/s on unique expert bytes, now 3HI + 4(2I+H) per expert) and the
    main workload's gather configuration (half the bytes over the host link)."""
    out = {}
    for T in (1, 8, 64):
        c = C.qwen(T, S=128, mode=C.MODE_RESIDENT)
        w = Workload(c, 2 * steps + warmup, dev, quant=True)
        w.layer.decode_kernels = decode_kernels
        r = time_steps(w, steps, warmup)
        units = count_unique_all(w, steps, warmup + steps)
        # T <= 8 runs the persistent W8A8 decode kernel: its whole launch counts
        t_ffn = (r["kern_ms"]["ffn_gateup"] + r["kern_ms"]["ffn_down"] + r["kern_ms"]["decode"]) * 1e-3
        ach = units * w.slab_bytes / t_ffn / 1e9 if t_ffn > 0 else 0.0
        layer_bytes = count_unique_all(w, steps, warmup) * w.slab_bytes
        out[f"resident_T{T}"] = {
            "tokens_per_s": T * steps / (r["ms"] * 1e-3), "ms_per_step": r["ms"] / steps,
            "ffn_hbm": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": ach / peaks["hbm_gbs"], "kernel": "decode_q8_kernel" if T <= 8 and not decode_kernels else "w8a8 stream (ffn_q8)",
                        "bytes_per_unit": w.slab_bytes,
                        "units": units},
            "layer_hbm_frac": layer_bytes / (r["ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"]}
        del w
        torch.cuda.empty_cache()
    c = main_config()
    w = Workload(c, 2 * steps + warmup, dev, quant=True)
    r = time_steps(w, steps, warmup)
    out["gather_T64"] = {"tokens_per_s": c.T * steps / (r["ms"] * 1e-3), "ms_per_step": r["ms"] / steps,
                         "misses_per_step": r["misses"] / steps,
                         "host_link_GB_per_step": r["gathered_bytes"] / steps / 1e9,
                         "gather_GBps": r["gathered_bytes"] / (r["kern_ms"]["gather"] * 1e-3) / 1e9
                         if r["kern_ms"]["gather"] > 0 else None}
    del w
    return out


def routing_variants(dev: str, steps: int = 10, warmup: int = 3) -> dict:
    """The Flash-Next zero-return layer (512 experts, top-10, the 192 brightest
    in VRAM slots, STATIC) under each way of using the brightness profile
    ("Nudge, don't cut": no bias, graded bias at two caps, a flat bias, a hard
    mask, damped weights, GLM's sigmoid router with a graded bias): step time
    and missing experts per step (each one a second-pass read over the host
    link)."""
    import expert_slot_cache_gb300 as M
    cfg = C.FLASH
    wl = Workload(cfg, 2 * steps + warmup, dev)
    b, _ = C.draw_brightness(cfg)
    bd = torch.from_numpy(b).to(dev)
    arms = [("none", None, None, 0), ("graded_cap-1", M.BIAS_GRADED, -1.0, 0),
            ("graded_cap-0.5", M.BIAS_GRADED, -0.5, 0), ("flat-0.5", M.BIAS_FLAT, -0.5, 0),
            ("hard_mask", M.BIAS_HARD, 0.0, 0), ("damped_graded_cap-1", M.BIAS_GRADED, -1.0, M.ROUTE_DAMPED),
            ("sigmoid_graded_cap-0.25", M.BIAS_GRADED, -0.25, M.ROUTE_SIGMOID)]
    out = {"workload": "flash-next-shaped zero-return layer, T=16, E=512, k=10, H=2048, I=512, S=192 STATIC "
                       "(the 192 brightest), Zipf(1.1) brightness"}
    for name, mode, val, rf in arms:
        wl.layer.sel_bias = None if mode is None else M.bias_table(bd, cfg.n_hot, val, mode=mode)
        wl.layer.route_flags = rf
        r = time_steps(wl, steps, warmup, profile=False)
        out[name] = {"ms_per_step": r["ms"] / steps, "tokens_per_s": cfg.T * steps / (r["ms"] * 1e-3),
                     "missing_experts_per_step": r["misses"] / steps,
                     "host_link_GB_per_step": r["misses"] / steps * cfg.slab_bytes / 1e9}
    del wl
    return out


def policy_replay(trace: np.ndarray, E: int, S: int, dev: str, slab_bytes: int) -> dict:
    """Replay one routing trace through expert_cache_manage under each policy
    ("Porting vllm-expert-cache to NVIDIA GPUs", "Measuring, without fooling
    yourself": count misses, not tokens).  STATIC keeps its seeded set; the
    hindsight baseline is STATIC with the S experts used most over the trace
    (the transcript's "oracle ... picked the best possible fixed set")."""
    import expert_slot_cache_gb300 as M
    steps, T, k = trace.shape
    ids_d = torch.from_numpy(trace).to(dev)
    seeded = C.initial_residency(C.TINY.with_(E=E, S=S, seed=E))
    counts = np.bincount(trace.reshape(-1), minlength=E)
    best = np.sort(np.argsort(-counts, kind="stable")[:S]).astype(np.int32)
    runs = {"lru": (C.POLICY_LRU, seeded), "lfu": (C.POLICY_LFU, seeded), "static": (C.POLICY_STATIC, seeded),
            "static_best_fixed": (C.POLICY_STATIC, best)}
    out = {}
    for name, (pol, s2e0) in runs.items():
        st = M.CacheState.from_slots(s2e0, E, dev)
        tot = torch.zeros(1, dtype=torch.int64, device=dev)
        for i in range(steps):
            tot += M.cache_manage(ids_d[i], st, pol).n_miss
        misses = int(tot.item())
        needed = sum(len(np.unique(trace[i])) for i in range(steps))
        out[name] = {"misses": misses, "hit_rate": 1.0 - misses / needed,
                     "host_link_GB": misses * slab_bytes / 1e9 if pol != C.POLICY_STATIC else 0.0,
                     "missed_expert_bytes_GB": misses * slab_bytes / 1e9}
    # STATIC with a periodic re-pick (the transcript's "every 500 tokens, have another look"): between
    # re-picks the set stays fixed (misses are served from host memory, zero-return); each re-pick loads
    # the experts that entered the set
    for every in (500, 2000):
        st = M.CacheState.from_slots(seeded, E, dev)
        counts = torch.zeros(E, dtype=torch.int32, device=dev)
        tot = torch.zeros(1, dtype=torch.int64, device=dev)
        loads = torch.zeros(1, dtype=torch.int64, device=dev)
        per = max(1, every // T)
        for i in range(steps):
            tot += M.cache_manage(ids_d[i], st, C.POLICY_STATIC).n_miss
            M.cache_count(ids_d[i], E, counts)
            if (i + 1) % per == 0:
                loads += M.cache_repick(counts, st).n_miss
        misses, n_loads = int(tot.item()), int(loads.item())
        needed = sum(len(np.unique(trace[i])) for i in range(steps))
        out[f"static_repick_every_{every}_tokens"] = {
            "misses": misses, "hit_rate": 1.0 - misses / needed, "repick_loads": n_loads,
            "host_link_GB": n_loads * slab_bytes / 1e9, "missed_expert_bytes_GB": misses * slab_bytes / 1e9}
    out["trace"] = {"steps": steps, "T": T, "k": k, "E": E, "S": S,
                    "recipe": "Zipf(1.1) popularity over a ranking drifting by 2 swaps per step"}
    return out


def graph_kernel_nodes(g) -> Optional[int]:
    """Kernel nodes of a captured torch CUDA graph (kept with keep_graph=True),
    counted with the driver API: the launches one replay of it makes."""
    import ctypes
    try:
        cu = ctypes.CDLL("libcuda.so.1")
        graph = ctypes.c_void_p(g.raw_cuda_graph())
        n = ctypes.c_size_t(0)
        if cu.cuGraphGetNodes(graph, None, ctypes.byref(n)) != 0:
            return None
        nodes = (ctypes.c_void_p * n.value)()
        if cu.cuGraphGetNodes(graph, nodes, ctypes.byref(n)) != 0:
            return None
        kinds = ctypes.c_int(0)
        count = 0
        for i in range(n.value):
            if cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(kinds)) != 0:
                return None
            count += kinds.value == 0  # CU_GRAPH_NODE_TYPE_KERNEL
        return count
    except Exception:
        return None


def _make_prof(M, pairs: int):
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * pairs)]
    for ev in evs:  # torch creates the underlying event lazily, on its first record
        ev.record()
    arr = (M.binding.c_void_p * (2 * pairs))(*[e.cuda_event for e in evs])
    tags = (M.binding.c_int32 * pairs)()
    p = M.binding.Prof(arr, 2 * pairs, 0, tags)
    return p, evs, arr, tags


def _prof_times(p, evs) -> dict:
    out = {n: [] for n in PROF_NAMES}
    for i in range(p.used // 2):
        out[PROF_NAMES[p.tags[i]]].append(evs[2 * i].elapsed_time(evs[2 * i + 1]))
    return out


def time_steps(wl: Workload, steps: int, warmup: int, dist=None, clocks=None, profile=True, graph=True):
    """K steps timed between CUDA events after W eager warm-ups.

    With ``graph`` the K steps are captured into one CUDA graph and the timed
    region is one replay (inputs differ per step; the cache state keeps
    evolving on the device).  The timed graph has no instrumentation.  With
    ``profile``, a second graph of the next K steps carries the timing events
    that the layer forward records around each of its launches; those give
    the per-kernel live times (the event nodes add a little latency, so that
    graph is not used for the step time).  That graph is replayed twice and
    the faster replay's times are kept, so that one disturbed replay (the
    host link or the GPU shared with another job for a moment) does not
    stand for the kernels' durations.
    """
    M = wl.M
    for i in range(warmup):
        wl.step(i)
    torch.cuda.synchronize()
    misses0, gathered0 = int(wl.layer.stats[0]), int(wl.layer.stats[2])

    nodes = [None]
    prof_times = [None]

    def run(first, prof_list):
        g = None
        if graph:
            g = torch.cuda.CUDAGraph(keep_graph=True)
            with torch.cuda.graph(g, capture_error_mode="relaxed"):
                for i in range(steps):
                    wl.step(first + i, prof=None if prof_list is None else prof_list[i][0])
            if prof_list is None:
                nodes[0] = graph_kernel_nodes(g)
            g.instantiate()
            torch.cuda.synchronize()
        best = None
        for rep in range(2 if (graph and prof_list is not None) else 1):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            if graph:
                g.replay()
            else:
                for i in range(steps):
                    wl.step(first + i, prof=None if prof_list is None else prof_list[i][0])
            e.record()
            torch.cuda.synchronize()
            t = s.elapsed_time(e)
            if prof_list is not None:
                times = [_prof_times(p, evs) for p, evs, _, _ in prof_list]
                if best is None or t < best[0]:
                    best = (t, times)
            else:
                best = (t, None)
        prof_times[0] = best[1]
        return best[0]

    _barrier(dist)
    if clocks:
        clocks.start()
    ms = run(warmup, None)
    cl = clocks.stop() if clocks else None
    _barrier(dist)
    ms = _max_over_ranks(ms, dist)
    misses = int(wl.layer.stats[0]) - misses0
    gathered = int(wl.layer.stats[2]) - gathered0
    kern = {n: 0.0 for n in PROF_NAMES}
    launches = {n: 0 for n in PROF_NAMES}
    per_launch = {n: [] for n in PROF_NAMES}
    ms_prof = None
    if profile:
        n_chunks = (wl.cfg.T + wl.chunk() - 1) // wl.chunk()
        profs = [_make_prof(M, 8 + 40 * n_chunks) for _ in range(steps)]
        ms_prof = run(warmup + steps, profs)
        for pt in prof_times[0]:
            for n, v in pt.items():
                kern[n] += sum(v)
                launches[n] += len(v)
                per_launch[n].extend(v)
    return {"ms": ms, "ms_instrumented": ms_prof, "kern_ms": kern, "launches": launches, "clocks": cl,
            "misses": misses, "gathered_bytes": gathered, "graph": graph, "kernel_nodes": nodes[0],
            "per_launch": per_launch}


def count_unique_all(wl: Workload, steps: int, warmup: int) -> int:
    """Expert-chunk units streamed by the FFN over the timed steps (re-run routing only)."""
    M = wl.M
    tot = 0
    for i in range(steps):
        ids, _ = M.route(wl.xs[warmup + i], wl.wr, wl.cfg.k, wl.off, wl.bias)
        tot += wl.unique_per_chunk(ids.cpu().numpy())
    return tot


def host_link_peak(dev: str, nbytes: int = 1 << 30) -> float:
    """Pinned host -> device copy bandwidth (GB/s), measured here with cudaMemcpyAsync."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d.copy_(h, non_blocking=True)
    torch.cuda.synchronize()
    best = 0.0
    for _ in range(3):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        d.copy_(h, non_blocking=True)
        e.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (s.elapsed_time(e) * 1e-3) / 1e9)
    del h, d
    return best


def e2e_steps(wl: Workload, steps: int, warmup: int, dist=None):
    """Same metric through the public API with host buffers: H2D of x and D2H of out in the timed region."""
    cfg = wl.cfg
    hx = [wl.xs[i].cpu().pin_memory() for i in range(warmup + steps)]
    hout = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, pin_memory=True)
    dx = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=wl.dev)
    for i in range(warmup):
        dx.copy_(hx[i], non_blocking=True)
        wl.step(0, x=dx)
        hout.copy_(wl.out, non_blocking=True)
    torch.cuda.synchronize()
    _barrier(dist)
    t0 = time.perf_counter()
    for i in range(steps):
        dx.copy_(hx[warmup + i], non_blocking=True)
        wl.step(0, x=dx)
        hout.copy_(wl.out, non_blocking=True)
    torch.cuda.synchronize()
    dt = _max_over_ranks(time.perf_counter() - t0, dist)
    nb = cfg.T * cfg.H * 2
    return {"value": cfg.T * steps / dt, "unit": UNIT, "h2d_bytes_per_step": nb, "d2h_bytes_per_step": nb}


# ----------------------------------------------------------------------------
# the CPU oracle leg
# ----------------------------------------------------------------------------

def oracle_sample(cfg: C.LayerConfig, steps: int, warmup: int, dev: str):
    """Time the oracle on ``steps`` layer forwards of the workload (after ``warmup``)."""
    import oracle as O
    gen_dev = dev if torch.cuda.is_available() else "cpu"
    wr = C.draw_router(cfg, gen_dev).float().cpu().numpy()
    host = torch.empty(cfg.E, cfg.slab_elems, dtype=torch.bfloat16)
    for e in range(cfg.E):
        host[e].copy_(C.draw_slab(cfg, e, gen_dev))

    class _S:
        def __getitem__(self, e):
            return host[int(e)].float().numpy()

    s2e0 = C.initial_residency(cfg)
    st = O.CacheState.from_slots(s2e0, cfg.E)
    mode = cfg.mode
    off = C.draw_logit_offset(cfg, gen_dev)
    off = None if off is None else off.cpu().numpy()
    xs = [C.draw_x(cfg, gen_dev, step=i).float().cpu().numpy() for i in range(warmup + steps)]
    for i in range(warmup):
        O.layer_forward(xs[i], wr, _S(), cfg.H, cfg.I, cfg.k, mode, cfg.policy, st, None, off,
                        schedule=cfg.schedule)
    t0 = time.perf_counter()
    for i in range(steps):
        O.layer_forward(xs[warmup + i], wr, _S(), cfg.H, cfg.I, cfg.k, mode, cfg.policy, st, None, off,
                        schedule=cfg.schedule)
    dt = time.perf_counter() - t0
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", "0") or 0) or os.cpu_count()
    return {"value": cfg.T * steps / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{steps} full layer forward(s) of the benchmarked workload (T={cfg.T}), after {warmup} "
                      f"warm-up; numpy oracle (python loops for top-k, permute and cache; the fp64 FFN "
                      f"matmuls in numpy's BLAS on {cores} thread(s))", "seconds": dt}


def run_reference(args, ws, rank, dist):
    if rank != 0:
        return
    cfg = main_config()
    steps = max(1, min(args.steps, 20))
    warm = min(args.warmup, 1)
    r = oracle_sample(cfg, steps, warm, "cuda:0")
    line = {"impl": "reference", "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": args.gpus,
            "steps": steps, "warmup": warm, "ms_per_step": 1e3 * r["seconds"] / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_obj(cfg), "cpu_baseline": r,
            "e2e": {"value": r["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# main
# ----------------------------------------------------------------------------

def main_config(schedule: int = C.SCHED_WAVES) -> C.LayerConfig:
    return C.qwen(64, S=64, mode=C.MODE_GATHER, policy=C.POLICY_LRU, schedule=schedule)


def config_obj(cfg: C.LayerConfig) -> dict:
    sched = "expert waves" if cfg.schedule == C.SCHED_WAVES else "token chunks"
    return {"workload": f"qwen3-30b-a3b-shaped MoE decode layer, T={cfg.T}, H={cfg.H}, E={cfg.E}, k={cfg.k}, "
                        f"I={cfg.I}, bf16, slot pool {cfg.S} of {cfg.E} (rest pinned host), LRU, gather, {sched}",
            "T": cfg.T, "H": cfg.H, "E": cfg.E, "k": cfg.k, "I": cfg.I, "S": cfg.S, "mode": "gather",
            "policy": "lru", "schedule": sched,
            "l2": "inputs larger than L2 (expert weights 1.21 GB; every step streams its experts)",
            "parallelism": "replicas"}


def ffn_roofline(wl: Workload, r: dict, units: int, peaks: dict) -> dict:
    cfg = wl.cfg
    bytes_per_unit = cfg.slab_bytes  # gate/up (4HI bytes) + down (2HI bytes) per expert-chunk unit
    t = (r["kern_ms"]["ffn_gateup"] + r["kern_ms"]["ffn_down"]) * 1e-3
    ach = units * bytes_per_unit / t / 1e9 if t > 0 else 0.0
    return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": ach / peaks["hbm_gbs"], "traffic": None, "kernel": "ffn_gateup+ffn_down",
            "bytes_per_unit": bytes_per_unit, "units": units, "peak_source": peaks["source"]}


def _r(v, d=4):
    """Round to d significant digits (keeps the JSON line short)."""
    if v is None or not isinstance(v, float):
        return v
    return float(f"{v:.{d}g}")


def resident_decode(dev: str, peaks: dict, T: int, quant: bool = False, steps: int = 10, warmup: int = 3) -> dict:
    """All-resident Qwen-shaped decode layer: step time, FFN and whole-layer HBM fractions on unique expert bytes."""
    c = C.qwen(T, S=128, mode=C.MODE_RESIDENT)
    w = Workload(c, 2 * steps + warmup, dev, quant=quant)
    r = time_steps(w, steps, warmup)
    units = count_unique_all(w, steps, warmup + steps)
    # the FFN kernels' live time; for the persistent decode kernel its whole launch (routing and combine
    # included, so the fraction is a lower bound for its weight streams)
    t_ffn = (r["kern_ms"]["ffn_gateup"] + r["kern_ms"]["ffn_down"] + r["kern_ms"]["decode"]) * 1e-3
    ffn = units * w.slab_bytes / t_ffn / 1e9 / peaks["hbm_gbs"] if t_ffn > 0 else 0.0
    layer = count_unique_all(w, steps, warmup) * w.slab_bytes / (r["ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"]
    del w
    torch.cuda.empty_cache()
    return {"us": 1e3 * r["ms"] / steps, "layer_hbm": layer, "ffn_hbm": ffn}


def prefill_line(dev: str, peaks: dict, steps: int = 3, warmup: int = 3) -> dict:
    """Prefill T=4096, all experts resident, skewed groups: FFN GEMMs against bf16 peak (and HBM)."""
    cp = C.PREFILL
    wp = Workload(cp, 2 * steps + warmup, dev)
    rp = time_steps(wp, steps, warmup)
    flops = 6.0 * cp.T * cp.k * cp.H * cp.I
    w_bytes = count_unique_all(wp, steps, warmup + steps) * cp.slab_bytes / steps
    t_ffn = (rp["kern_ms"]["ffn_gateup"] + rp["kern_ms"]["ffn_down"]) * 1e-3 / steps
    t_layer = rp["ms"] * 1e-3 / steps
    del wp
    torch.cuda.empty_cache()
    return {"ms": t_layer * 1e3, "tok_s": cp.T / t_layer, "ffn_tflops": flops / t_ffn / 1e12,
            "ffn_tc": flops / t_ffn / 1e12 / peaks["bf16_tflops"], "ffn_hbm": w_bytes / t_ffn / 1e9 / peaks["hbm_gbs"],
            "layer_tflops": flops / t_layer / 1e12}


def gather_line(dev: str, T: int, schedule: int, quant: bool = False, steps: int = 10, warmup: int = 3) -> dict:
    c = C.qwen(T, S=64, schedule=schedule)
    w = Workload(c, 2 * steps + warmup, dev, quant=quant)
    r = time_steps(w, steps, warmup, profile=False)
    del w
    torch.cuda.empty_cache()
    return {"tok_s": T * steps / (r["ms"] * 1e-3), "misses": r["misses"] / steps}


def targets(dev: str, peaks: dict) -> dict:
    """The figures the performance targets are stated in, one flat object."""
    t = {}
    for T in (1, 8, 64):
        d = resident_decode(dev, peaks, T)
        t[f"res_T{T}_us"], t[f"res_T{T}_layer_hbm"], t[f"res_T{T}_ffn_hbm"] = d["us"], d["layer_hbm"], d["ffn_hbm"]
    p = prefill_line(dev, peaks)
    t["prefill_ms"], t["prefill_ffn_tc"], t["prefill_ffn_tflops"], t["prefill_ffn_hbm"] = \
        p["ms"], p["ffn_tc"], p["ffn_tflops"], p["ffn_hbm"]
    for T in (1, 8, 32):
        g = gather_line(dev, T, C.SCHED_WAVES)
        t[f"gather_T{T}_tok_s"] = g["tok_s"]
    g = gather_line(dev, 64, C.SCHED_CHUNKS)
    t["gather_T64_chunks_tok_s"], t["gather_T64_chunks_misses"] = g["tok_s"], g["misses"]
    for T in (1, 8, 64):
        d = resident_decode(dev, peaks, T, quant=True)
        t[f"q8_res_T{T}_us"], t[f"q8_res_T{T}_layer_hbm"], t[f"q8_res_T{T}_ffn_hbm"] = \
            d["us"], d["layer_hbm"], d["ffn_hbm"]
    for T in (1, 8):  # one launch per step (the fused expert-cache step)
        t[f"q8_gather_T{T}_tok_s"] = gather_line(dev, T, C.SCHED_WAVES, quant=True)["tok_s"]
    t["q8_gather_T64_tok_s"] = gather_line(dev, 64, C.SCHED_WAVES, quant=True)["tok_s"]
    st = stack_variant(dev, peaks, C.STACK)
    t["stack48_tok_s"], t["stack48_hbm"] = st["tokens_per_s"], st["hbm"]["frac"]
    st = stack_variant(dev, peaks, C.STACK_SLOTS.with_(schedule=C.SCHED_WAVES), steps=4)
    t["stack48_slots_tok_s"], t["stack48_slots_link_GB"] = st["tokens_per_s"], st["host_link_GB_per_step"]
    st = stack_variant(dev, peaks, C.STACK_BUDGET, steps=4)
    t["stack48_budget_tok_s"], t["stack48_budget_link_GB"] = st["tokens_per_s"], st["host_link_GB_per_step"]
    return {k: _r(v) for k, v in t.items()}


def oracle_baselines(local: int) -> dict:
    """The oracle leg timed twice: numpy's BLAS on one thread and on every host core."""
    out = {}
    for thr in ("1", str(os.cpu_count() or 1)):
        env = dict(os.environ, MOE_ORACLE_THREADS=thr, WORLD_SIZE="1", RANK="0", LOCAL_RANK=str(local))
        p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                            "--warmup", "0"], capture_output=True, text=True, env=env)
        try:
            out[thr] = json.loads(p.stdout.strip().splitlines()[-1])["cpu_baseline"]
        except Exception:
            out[thr] = {"value": None, "error": (p.stderr or p.stdout)[-200:]}
    one, allc = out["1"], out[str(os.cpu_count() or 1)]
    best = allc if (allc.get("value") or 0) >= (one.get("value") or 0) else one
    return {"value": best.get("value"), "unit": UNIT, "cores": best.get("cores"), "kind": "oracle",
            "sample": best.get("sample", best.get("error")), "value_cores_1": _r(one.get("value")),
            "value_cores_all": _r(allc.get("value")), "cores_all": os.cpu_count()}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--separate-kernels", action="store_true",
                    help="single workloads: small all-resident and small expert-cache steps run as separate kernels, "
                         "not the persistent one")
    ap.add_argument("--workload", default="main",
                    help="main (default) | prefill | resident_T<n> | gather_T<n> | chunks_T<n> (each also as q8_<name>: "
                         "W8A8 experts) | routing_variants | "
                         "policy_replay | w8a8 | stack | stack_slots | stack_slots_chunks | stack_budget: one workload alone "
                         "(for profiling); prints its own JSON line")
    args = ap.parse_args()
    ws, rank, local, dist = _dist()
    if args.impl == "reference":
        run_reference(args, ws, rank, dist)
        return
    args.warmup = max(3, args.warmup)
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    peaks = _peaks()
    if args.workload == "w8a8":
        if rank == 0:
            print(json.dumps({"workload": "w8a8", **w8a8_variants(dev, _peaks(), args.steps, args.warmup,
                                                                    int(args.separate_kernels))}))
        return
    if args.workload == "routing_variants":
        if rank == 0:
            print(json.dumps({"workload": "routing_variants", **routing_variants(dev, args.steps, args.warmup)}))
        return
    if args.workload == "policy_replay":
        cfg = main_config()
        if rank == 0:
            print(json.dumps({"workload": "policy_replay",
                              **policy_replay(C.drifting_trace(cfg.E, cfg.k, 8, 400), cfg.E, cfg.S, dev,
                                              cfg.slab_bytes)}))
        return
    if args.workload in ("stack", "stack_slots", "stack_slots_chunks", "stack_budget"):
        cfg_s = {"stack": C.STACK, "stack_slots": C.STACK_SLOTS.with_(schedule=C.SCHED_WAVES),
                 "stack_slots_chunks": C.STACK_SLOTS, "stack_budget": C.STACK_BUDGET}[args.workload]
        if rank == 0:
            print(json.dumps({"workload": args.workload, **stack_variant(dev, peaks, cfg_s, args.steps, args.warmup)}))
        return
    if args.workload != "main":
        w = args.workload
        quant = w.startswith("q8_")  # the same workload with W8A8 experts
        if quant:
            w = w[3:]
        if w == "prefill":
            c = C.PREFILL
        elif w.startswith("resident_T"):
            c = C.qwen(int(w[len("resident_T"):]), S=128, mode=C.MODE_RESIDENT)
        elif w.startswith("gather_T"):
            c = C.qwen(int(w[len("gather_T"):]), S=64, schedule=C.SCHED_WAVES)
        elif w.startswith("chunks_T"):
            c = C.qwen(int(w[len("chunks_T"):]), S=64)
        else:
            raise SystemExit(f"unknown workload {w}")
        wl = Workload(c, 2 * args.steps + args.warmup, dev, quant=quant)
        wl.layer.decode_kernels = int(args.separate_kernels)
        r = time_steps(wl, args.steps, args.warmup, clocks=Clocks(local))
        if rank == 0:
            print(json.dumps({"workload": args.workload, "clocks": r["clocks"], "ms_per_step": r["ms"] / args.steps,
                              "ms_per_step_instrumented": r["ms_instrumented"] / args.steps,
                              "tokens_per_s": c.T * args.steps / (r["ms"] * 1e-3),
                              "misses_per_step": r["misses"] / args.steps,
                              "kernel_nodes_per_step": None if r["kernel_nodes"] is None
                              else r["kernel_nodes"] / args.steps,
                              "gather_launch_ms": [round(v, 4) for v in r["per_launch"]["gather"][:12]],
                              "kernels_ms_per_step": {n: v / args.steps for n, v in r["kern_ms"].items()}}))
        return
    cfg = main_config()
    K, W = args.steps, args.warmup

    wl = Workload(cfg, 2 * K + W, dev)
    clocks = Clocks(local)
    r = time_steps(wl, K, W, dist, clocks)
    value = ws * cfg.T * K / (r["ms"] * 1e-3)
    link_peak = host_link_peak(dev)
    kern = r["kern_ms"]
    dominant = max(kern, key=kern.get)
    if dominant == "gather":
        t = kern["gather"] * 1e-3
        ach = r["gathered_bytes"] / t / 1e9 if t > 0 else 0.0
        n_launch = max(1, r["launches"].get("gather", 0))
        roof = {"bound": "host-link", "achieved": _r(ach), "peak": _r(link_peak), "unit": "GB/s",
                "frac": _r(ach / link_peak), "traffic": _r(GATHER_DRAM_BYTES_PER_MISS * r["misses"] / n_launch),
                "kernel": "gather", "bytes_per_unit": cfg.slab_bytes, "units": r["misses"],
                "peak_source": "pinned-host->device cudaMemcpyAsync measured in this run"}
    else:
        units = count_unique_all(wl, K, W + K)
        roof = {k: _r(v) for k, v in ffn_roofline(wl, r, units, peaks).items()}
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": W,
            "ms_per_step": r["ms"] / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded, Irwin-Hall normal weights/activations)",
            "config": config_obj(cfg), "roofline": roof, "clocks": r["clocks"],
            "gpu_launches": r["kernel_nodes"] if r["kernel_nodes"] is not None else sum(r["launches"].values()),
            "timed_as": "one CUDA-graph replay of the K steps (eager warm-ups)",
            "misses_per_step": r["misses"] / K,
            "kernels_ms_per_step": {n: _r(v / K) for n, v in kern.items() if v > 0}}
    line["e2e"] = e2e_steps(wl, K, W, dist)
    del wl
    torch.cuda.empty_cache()
    tg = None
    if not args.no_variants:
        tg = targets(dev, peaks)
    if not args.no_cpu_baseline and rank == 0:
        line["cpu_baseline"] = oracle_baselines(local)
    if tg is not None:
        line["targets"] = tg  # last: the end of the line is what a truncated log keeps
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
