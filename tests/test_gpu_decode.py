"""GPU parity of the persistent decode kernel: a small all-resident step (T <= 8,
T*k <= 64, E <= 256) runs the whole layer -- router logits, top-k, grouping,
both weight streams and the combine -- in one cooperative launch.

"Betelgeuse ... on an RTX 3060", "What it actually does under the hood" (hits
resolved in-stream, the decode pass as one CUDA graph) and "Porting
vllm-expert-cache to NVIDIA GPUs", "1. Kernels" (a fused cache-and-expert
kernel).  Every step is compared with the oracle: logits and ids bit for bit,
weights within 1e-6, the output within the bf16 tolerance; the launch is
checked to be that one kernel; a CUDA graph replays it over several steps (its
arrival counters go back to zero after every launch).
"""
import ctypes

import numpy as np
import pytest
import torch

from harness import configs as C
import oracle as O
from tests._setup import HostSlabs, assert_out_close, stage_layer
from tests.test_gpu_parity import _np, _run_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_decode_qwen_resident(T):
    _run_layer(C.qwen(T, S=128, mode=C.MODE_RESIDENT), steps=3)


def test_decode_one_token_small_shape():
    # one token on the small shape: two tiles per projection, fewer weight stages than CTAs
    _run_layer(C.TINY.with_(T=1), steps=4)


def test_decode_tiny_resident_with_offset_and_bias():
    cfg = C.TINY.with_(T=7, logit_offset=True, bias_cap=-0.5, n_hot=6, zipf_s=1.1)
    _run_layer(cfg, steps=3)


def test_decode_sigmoid_router_and_damped_weights():
    cfg = C.TINY.with_(T=6, bias_cap=-0.25, n_hot=8, zipf_s=1.1)
    import expert_slot_cache_gb300 as M
    _run_layer(cfg, steps=2, rflags=M.ROUTE_SIGMOID)
    _run_layer(cfg, steps=2, rflags=M.ROUTE_DAMPED)


def test_decode_separate_kernels_agree():
    _run_layer(C.qwen(4, S=128, mode=C.MODE_RESIDENT), steps=2, decode_kernels=1)


@pytest.mark.parametrize("T", [1, 8])
def test_decode_routing_equals_router_kernels_bitwise(T):
    # the persistent kernel's ids and weights are those of the router kernels, bit for bit
    cfg = C.qwen(T, S=128, mode=C.MODE_RESIDENT)
    st = stage_layer(cfg)
    import expert_slot_cache_gb300 as M
    lay = [M.SlotCachedMoELayer(st["wr"], st["slabs_dev"], cfg.k, cfg.I, C.MODE_RESIDENT, max_tokens=T,
                                decode_kernels=dk) for dk in (0, 1)]
    for step in range(3):
        x = C.draw_x(cfg, DEV, step=step)
        r1, r2 = lay[0].forward(x), lay[1].forward(x)
        torch.cuda.synchronize()
        assert torch.equal(r1["ids"], r2["ids"]) and torch.equal(r1["w"], r2["w"]), step
        assert_out_close(_np(r1["out"].float()), _np(r2["out"].float()).astype(np.float64), f"step {step}")


def _layer(cfg, st):
    import expert_slot_cache_gb300 as M
    return M.SlotCachedMoELayer(st["wr"], st["slabs_dev"], cfg.k, cfg.I, C.MODE_RESIDENT,
                                logit_offset=st["logit_offset"], max_tokens=cfg.T)


def test_decode_is_one_launch():
    import expert_slot_cache_gb300 as M
    cfg = C.qwen(2, S=128, mode=C.MODE_RESIDENT)
    st = stage_layer(cfg)
    layer = _layer(cfg, st)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
    for ev in evs:
        ev.record()
    arr = (ctypes.c_void_p * 8)(*[e.cuda_event for e in evs])
    tags = (ctypes.c_int32 * 4)()
    prof = M.binding.Prof(arr, 8, 0, tags)
    layer.forward(C.draw_x(cfg, DEV), prof=prof)
    torch.cuda.synchronize()
    assert prof.used == 2 and tags[0] == 8  # one (start, end) pair: MOE_PROF_DECODE


def test_decode_graph_replay_matches_oracle_every_step():
    cfg = C.qwen(3, S=128, mode=C.MODE_RESIDENT)
    st = stage_layer(cfg)
    layer = _layer(cfg, st)
    xs = [C.draw_x(cfg, DEV, step=i) for i in range(4)]
    x = torch.empty_like(xs[0])
    x.copy_(xs[0])
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=DEV)
    ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=DEV)
    w = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=DEV)
    layer.forward(x, out=out, ids=ids, w=w)  # eager first call
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(x, out=out, ids=ids, w=w)
    wr_np = _np(st["wr"].float())
    off_np = None if st["logit_offset"] is None else _np(st["logit_offset"])
    for i in range(4):
        x.copy_(xs[i])
        g.replay()
        torch.cuda.synchronize()
        want = O.layer_forward(_np(x.float()), wr_np, HostSlabs(st["host"]), cfg.H, cfg.I, cfg.k, O.RESIDENT,
                               logit_offset=off_np)
        assert np.array_equal(_np(ids), want["ids"]), f"replay {i}: ids"
        assert np.abs(_np(w) - want["w"]).max() <= 1e-6
        assert_out_close(_np(out.float()), want["out"], f"replay {i}: out")
    assert int(_np(layer.dev_status)[0]) == 0
    # the arrival counters (start of the workspace) are back at zero
    assert int(layer.workspace[: 4 * (cfg.E + 4)].count_nonzero()) == 0


def test_decode_with_a_remapped_pool():
    # all experts resident, but in a shuffled slot order (e2s): the kernel reads each expert from its slot
    import expert_slot_cache_gb300 as M
    cfg = C.qwen(4, S=128, mode=C.MODE_RESIDENT)
    st = stage_layer(cfg)
    perm = np.random.default_rng(9).permutation(cfg.E).astype(np.int32)  # slot s holds expert perm[s]
    pool = st["slabs_dev"][torch.from_numpy(perm.astype(np.int64)).to(DEV)].contiguous()
    state = M.CacheState.from_slots(perm, cfg.E)
    layer = M.SlotCachedMoELayer(st["wr"], pool, cfg.k, cfg.I, C.MODE_RESIDENT, state=state,
                                 logit_offset=st["logit_offset"], max_tokens=cfg.T)
    wr_np = _np(st["wr"].float())
    for step in range(2):
        x = C.draw_x(cfg, DEV, step=step)
        r = layer.forward(x)
        torch.cuda.synchronize()
        want = O.layer_forward(_np(x.float()), wr_np, HostSlabs(st["host"]), cfg.H, cfg.I, cfg.k, O.RESIDENT)
        assert np.array_equal(_np(r["ids"]), want["ids"]), step
        assert_out_close(_np(r["out"].float()), want["out"], f"step {step}")
    assert int(_np(layer.dev_status)[0]) == 0


def _check_bf16(cfg, x):
    import expert_slot_cache_gb300 as M
    st = stage_layer(cfg)
    layer = M.SlotCachedMoELayer(st["wr"], st["slabs_dev"], cfg.k, cfg.I, C.MODE_RESIDENT, max_tokens=cfg.T)
    r = layer.forward(x)
    torch.cuda.synchronize()
    want = O.layer_forward(_np(x.float()), _np(st["wr"].float()), HostSlabs(st["host"]), cfg.H, cfg.I, cfg.k,
                           O.RESIDENT)
    assert np.array_equal(_np(r["ids"]), want["ids"])
    assert np.abs(_np(r["w"]) - want["w"]).max() <= 1e-6
    assert_out_close(_np(r["out"].float()), want["out"], "out")
    assert int(_np(layer.dev_status)[0]) == 0
    return want


def test_decode_identical_tokens_give_every_expert_eight_rows():
    # every token routes to the same k experts: each routed expert has T = 8 rows (the widest batch)
    cfg = C.qwen(8, S=128, mode=C.MODE_RESIDENT)
    x = C.draw_x(cfg, DEV)[:1].repeat(cfg.T, 1).contiguous()
    want = _check_bf16(cfg, x)
    assert all(len(set(want["ids"][:, j])) == 1 for j in range(cfg.k))


def test_decode_256_experts():
    # the most experts the persistent kernel takes: eight router expert groups, the widest rank loop
    cfg = C.qwen(8, S=256, mode=C.MODE_RESIDENT).with_(E=256, H=512, I=256)
    _check_bf16(cfg, C.draw_x(cfg, DEV))
