"""GPU parity of the persistent decode kernel on expert-cache steps: a small
GATHER step (T <= 8, T*k <= S, LRU or LFU) runs routing, the manage state
machine, the host-to-slot copy of the misses, both weight streams and the
combine in one cooperative launch.

"Porting vllm-expert-cache to NVIDIA GPUs", "1. Kernels" (a fused cache
manager, gather and expert kernel) and "What this package does" (victims among
the slots the step does not need, misses in ascending id); "Betelgeuse ... on
an RTX 3060", "What it actually does under the hood" (hits resolved in-stream
on the device, a decode pass replayed as one graph).  Every step is checked
against the oracle (ids bit for bit, weights within 1e-6, the output within the
bf16 tolerance, the cache state bit for bit) and against the separate kernels
(manage, gather, FFN, combine launches): the same state, statistics and slot
bytes, bit for bit.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from harness import configs as C
from tests._setup import HostSlabs, assert_out_close, stage_layer
from tests.test_gpu_parity import _check_state, _np
from tests.test_gpu_q8 import QHost

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _pair(cfg, s2e0, affinity=0.0, rflags=0, sel_bias=None, quant=0):
    """The persistent-kernel layer and the separate-kernel layer on the same inputs and starting state
    (W8A8 slabs, codes and scales, with quant=1)."""
    import expert_slot_cache_gb300 as M
    st = stage_layer(cfg)
    src, host = st["slabs_dev"], st["host"]
    if quant:
        src = M.quantize_slabs(st["slabs_dev"], cfg.H, cfg.I)
        host = torch.empty(src.shape, dtype=src.dtype, pin_memory=True)
        host.copy_(src)
        st["host_q"] = host
    layers = []
    for dk in (0, 1):
        pool = torch.zeros(cfg.S, src.shape[1], dtype=src.dtype, device=DEV)
        for s, e in enumerate(s2e0):
            if e >= 0:
                pool[s].copy_(src[e])
        state = M.CacheState.from_slots(s2e0, cfg.E)
        layers.append(M.SlotCachedMoELayer(st["wr"], pool, cfg.k, cfg.I, cfg.mode, cfg.policy, host_slabs=host,
                                           state=state, logit_offset=st["logit_offset"], max_tokens=cfg.T,
                                           affinity=affinity, route_flags=rflags, sel_bias=sel_bias, quant=quant,
                                           decode_kernels=dk))
    return st, layers


def _steps(cfg, s2e0, xs, affinity=0.0, rflags=0, quant=0):
    """Runs the steps on both layers and the oracle; returns the misses of each step."""
    import expert_slot_cache_gb300 as M
    bias_np = bias_d = None
    if cfg.bias_cap is not None:
        b, _ = C.draw_brightness(cfg)
        bias_np = O.bias_table(b, cfg.n_hot, cfg.bias_cap, O.BIAS_GRADED)
        bias_d = M.bias_table(torch.from_numpy(b).to(DEV), cfg.n_hot, cfg.bias_cap, mode=O.BIAS_GRADED)
    router = O.ROUTER_SIGMOID if rflags & M.ROUTE_SIGMOID else O.ROUTER_SOFTMAX
    st, (one, sep) = _pair(cfg, s2e0, affinity, rflags, bias_d, quant)
    ostate = O.CacheState.from_slots(s2e0, cfg.E)
    ohost = QHost(st["host"], cfg.H, cfg.I) if quant else HostSlabs(st["host"])
    slab_bytes = one.pool[0].numel() * one.pool.element_size()
    wr_np = _np(st["wr"].float())
    off_np = None if st["logit_offset"] is None else _np(st["logit_offset"])
    misses = []
    for step, x in enumerate(xs):
        r1 = one.forward(x)
        r2 = sep.forward(x)
        torch.cuda.synchronize()
        want = O.layer_forward(_np(x.float()), wr_np, ohost, cfg.H, cfg.I, cfg.k, cfg.mode,
                               cfg.policy, ostate, None, off_np, bias_np, affinity=affinity, router=router,
                               damped=bool(rflags & M.ROUTE_DAMPED), quant=bool(quant))
        assert np.array_equal(_np(r1["ids"]), want["ids"]), f"step {step}: ids"
        assert np.abs(_np(r1["w"]) - want["w"]).max() <= 1e-6, f"step {step}: w"
        assert torch.equal(r1["ids"], r2["ids"]) and torch.equal(r1["w"], r2["w"]), f"step {step}: routing"
        assert_out_close(_np(r1["out"].float()), want["out"], f"step {step}: out")
        if quant:  # the same exact integer sums and fp32 steps as the separate W8A8 kernels
            assert torch.equal(r1["out"], r2["out"]), f"step {step}: out differs from the separate kernels'"
        _check_state(one.state, ostate, f"step {step}")
        for f in ("e2s", "s2e", "prio", "stamp"):
            assert torch.equal(getattr(one.state, f), getattr(sep.state, f)), f"step {step}: {f}"
        assert torch.equal(one.stats, sep.stats), f"step {step}: stats"
        assert torch.equal(one.pool, sep.pool), f"step {step}: slot bytes"
        misses.append(sum(len(c["miss_e"]) for c in want["chunks"]))
    assert int(_np(one.dev_status)[0]) == 0 and int(_np(sep.dev_status)[0]) == 0
    # every occupied slot holds exactly its expert's bytes
    host = st["host_q"] if quant else st["host"]
    for s, e in enumerate(_np(one.state.s2e)):
        if e >= 0:
            assert torch.equal(one.pool[s].cpu(), host[int(e)]), f"slot {s}"
    stats = _np(one.stats)
    assert stats[0] == sum(misses) and stats[1] == len(xs) and stats[2] == sum(misses) * slab_bytes
    # the arrival and copy counters (start of the workspace) are back at zero
    assert int(one.workspace[: 4 * (cfg.E + 4 + 64)].count_nonzero()) == 0
    return misses


@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_decode_gather_qwen_lru(T):
    cfg = C.qwen(T)
    misses = _steps(cfg, C.initial_residency(cfg), [C.draw_x(cfg, DEV, step=s) for s in range(4)])
    assert sum(misses) > 0


@pytest.mark.parametrize("T", [1, 5, 8])
def test_decode_gather_w8a8_qwen_lru(T):
    # W8A8 slabs (codes and slot-indexed scales) copied host-to-slot in the persistent W8A8 kernel
    cfg = C.qwen(T)
    misses = _steps(cfg, C.initial_residency(cfg), [C.draw_x(cfg, DEV, step=s) for s in range(4)], quant=1)
    assert sum(misses) > 0


def test_decode_gather_w8a8_empty_pool_lfu_and_tiny():
    cfg = C.qwen(8, policy=C.POLICY_LFU)
    x0 = C.draw_x(cfg, DEV)
    _steps(cfg, np.full(cfg.S, -1, dtype=np.int32), [x0, x0, C.draw_x(cfg, DEV, step=1)], quant=1)
    cfg = C.TINY.with_(mode=C.MODE_GATHER, S=12, T=6, logit_offset=True, bias_cap=-0.5, n_hot=6, zipf_s=1.1)
    _steps(cfg, C.initial_residency(cfg), [C.draw_x(cfg, DEV, step=s) for s in range(3)], quant=1)


def test_decode_gather_qwen_lfu():
    cfg = C.qwen(8, policy=C.POLICY_LFU)
    _steps(cfg, C.initial_residency(cfg), [C.draw_x(cfg, DEV, step=s) for s in range(4)])


def test_decode_gather_empty_pool_all_misses():
    # an empty pool: every routed expert of the first step misses; identical tokens then hit every expert
    cfg = C.qwen(8)
    x0 = C.draw_x(cfg, DEV)
    misses = _steps(cfg, np.full(cfg.S, -1, dtype=np.int32), [x0, x0, C.draw_x(cfg, DEV, step=1)])
    ids = O.select_topk(O.router_logits(_np(x0.float()), _np(C.draw_router(cfg, DEV).float())), cfg.k)
    assert misses[0] == len(np.unique(ids)) and misses[1] == 0


def test_decode_gather_most_misses():
    # eight tokens whose 64 picks are all different, into an empty pool of 64 slots: 64 misses, every slot a
    # victim.  The tokens are picked greedily from seeded candidates, routed by the oracle.
    cfg = C.qwen(8)
    wr = _np(C.draw_router(cfg, DEV).float())
    rng = np.random.default_rng(5)
    cand = torch.from_numpy(rng.standard_normal((4096, cfg.H)).astype(np.float32)).to(torch.bfloat16)
    picks = O.select_topk(O.router_logits(cand.float().numpy(), wr), cfg.k)
    chosen, used = [], set()
    for i in range(cand.shape[0]):
        if not used.intersection(picks[i].tolist()):
            chosen.append(i)
            used.update(picks[i].tolist())
            if len(chosen) == cfg.T:
                break
    assert len(chosen) == cfg.T and len(used) == cfg.T * cfg.k
    x = cand[chosen].contiguous().to(DEV)
    misses = _steps(cfg, np.full(cfg.S, -1, dtype=np.int32), [x])
    assert misses == [cfg.T * cfg.k]


def test_decode_gather_pool_holds_every_expert():
    # S = E: no misses after the first loads, so no CTA copies and every CTA streams
    cfg = C.qwen(4, S=128)
    misses = _steps(cfg, C.initial_residency(cfg), [C.draw_x(cfg, DEV, step=s) for s in range(3)])
    assert misses == [0, 0, 0]


def test_decode_gather_with_affinity():
    # live-cache affinity reads the cache state as it stood before the step's manage call
    cfg = C.qwen(8)
    _steps(cfg, C.initial_residency(cfg), [C.draw_x(cfg, DEV, step=s) for s in range(3)], affinity=0.5)


@pytest.mark.parametrize("variant", ["softmax", "sigmoid", "damped"])
def test_decode_gather_offset_bias_and_router_variants(variant):
    # a per-expert logit offset, a graded selection bias, and the sigmoid router or damped weights
    import expert_slot_cache_gb300 as M
    rflags = {"softmax": 0, "sigmoid": M.ROUTE_SIGMOID, "damped": M.ROUTE_DAMPED}[variant]
    cfg = C.TINY.with_(mode=C.MODE_GATHER, S=12, T=6, logit_offset=True, bias_cap=-0.5, n_hot=6, zipf_s=1.1,
                       policy=C.POLICY_LFU if variant == "damped" else C.POLICY_LRU)
    _steps(cfg, C.initial_residency(cfg), [C.draw_x(cfg, DEV, step=s) for s in range(4)], rflags=rflags)


def test_decode_gather_tiny_and_widest_shapes():
    # tiny: 16 experts, slabs of eight 24 KB pieces; widest: 256 experts and 256 slots (the largest state copy)
    cfg = C.TINY.with_(mode=C.MODE_GATHER, S=8)
    _steps(cfg, C.initial_residency(cfg), [C.draw_x(cfg, DEV, step=s) for s in range(4)])
    cfg = C.qwen(8, S=256).with_(E=256, H=512, I=256)
    _steps(cfg, np.full(cfg.S, -1, dtype=np.int32), [C.draw_x(cfg, DEV, step=s) for s in range(2)])


def test_decode_gather_is_one_launch():
    import expert_slot_cache_gb300 as M
    cfg = C.qwen(2)
    _, (layer, _) = _pair(cfg, C.initial_residency(cfg))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
    for ev in evs:
        ev.record()
    arr = (ctypes.c_void_p * 8)(*[e.cuda_event for e in evs])
    tags = (ctypes.c_int32 * 4)()
    prof = M.binding.Prof(arr, 8, 0, tags)
    layer.forward(C.draw_x(cfg, DEV), prof=prof)
    torch.cuda.synchronize()
    assert prof.used == 2 and tags[0] == 8  # one (start, end) pair: MOE_PROF_DECODE


def test_decode_gather_graph_replay():
    # one captured step replayed over new inputs: the cache state moves on at every replay, as the oracle's
    cfg = C.qwen(8)
    s2e0 = C.initial_residency(cfg)
    st, (layer, _) = _pair(cfg, s2e0)
    ostate = O.CacheState.from_slots(s2e0, cfg.E)
    xs = [C.draw_x(cfg, DEV, step=i) for i in range(5)]
    x = torch.empty_like(xs[0])
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=DEV)
    ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=DEV)
    w = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=DEV)
    wr_np = _np(st["wr"].float())
    off_np = None if st["logit_offset"] is None else _np(st["logit_offset"])
    x.copy_(xs[0])
    layer.forward(x, out=out, ids=ids, w=w)  # eager first step
    torch.cuda.synchronize()
    O.layer_forward(_np(x.float()), wr_np, HostSlabs(st["host"]), cfg.H, cfg.I, cfg.k, cfg.mode, cfg.policy, ostate,
                    None, off_np)
    g = torch.cuda.CUDAGraph()
    snap = layer.state.clone()
    pool0 = layer.pool.clone()
    stats0 = layer.stats.clone()
    with torch.cuda.graph(g):  # capture runs nothing
        layer.forward(x, out=out, ids=ids, w=w)
    torch.cuda.synchronize()
    assert torch.equal(layer.state.e2s, snap.e2s) and torch.equal(layer.pool, pool0)
    assert torch.equal(layer.stats, stats0)
    for i in range(1, 5):
        x.copy_(xs[i])
        g.replay()
        torch.cuda.synchronize()
        want = O.layer_forward(_np(x.float()), wr_np, HostSlabs(st["host"]), cfg.H, cfg.I, cfg.k, cfg.mode,
                               cfg.policy, ostate, None, off_np)
        assert np.array_equal(_np(ids), want["ids"]), f"replay {i}: ids"
        assert_out_close(_np(out.float()), want["out"], f"replay {i}: out")
        _check_state(layer.state, ostate, f"replay {i}")
    assert int(_np(layer.dev_status)[0]) == 0
    assert int(layer.workspace[: 4 * (cfg.E + 4 + 64)].count_nonzero()) == 0
