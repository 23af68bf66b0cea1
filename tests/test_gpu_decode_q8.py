"""GPU parity of the persistent W8A8 decode kernel: a small all-resident step
(T <= 8, T*k <= 64, E <= 256) of W8A8 experts -- router logits, top-k,
grouping, the tokens' 8-bit codes, both weight streams, h quantised per row and
the combine -- in one cooperative launch.

"Porting vllm-expert-cache to NVIDIA GPUs" (the W8A8 model; weights and scales
slot-indexed; "1. Kernels", a fused cache-and-expert kernel) and "Betelgeuse
... on an RTX 3060", "What it actually does under the hood" (the decode pass
resolved on the device as one graph).  Against the oracle: ids bit for bit,
weights within 1e-6, the output within the bf16 tolerance.  Against the
separate W8A8 kernels: the output bit for bit (the same exact integer sums and
the same fp32 steps), so the single-launch path changes nothing but the time.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from harness import configs as C
from tests._setup import assert_out_close, stage_layer
from tests.test_gpu_q8 import QHost

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _np(t):
    return t.detach().cpu().numpy()


def _q8_layer(cfg, rflags=0, decode_kernels=0, perm=None, sel_bias=None):
    import expert_slot_cache_gb300 as M
    st = stage_layer(cfg)
    q = M.quantize_slabs(st["slabs_dev"], cfg.H, cfg.I)
    qh = QHost(st["host"], cfg.H, cfg.I)
    state = None
    if perm is not None:  # slot s holds expert perm[s]
        q = q[torch.from_numpy(perm.astype(np.int64)).to(DEV)].contiguous()
        state = M.CacheState.from_slots(perm, cfg.E)
    layer = M.SlotCachedMoELayer(st["wr"], q, cfg.k, cfg.I, C.MODE_RESIDENT, state=state,
                                 logit_offset=st["logit_offset"], sel_bias=sel_bias, max_tokens=cfg.T,
                                 route_flags=rflags, quant=1, decode_kernels=decode_kernels)
    return st, qh, layer


def _check(cfg, steps=2, rflags=0, bias_cap=None, perm=None):
    """The persistent kernel against the oracle and, bit for bit, against the separate kernels."""
    import expert_slot_cache_gb300 as M
    sel_bias = None
    bias_np = None
    if cfg.bias_cap is not None:
        b, _ = C.draw_brightness(cfg)
        bias_np = O.bias_table(b, cfg.n_hot, cfg.bias_cap, O.BIAS_GRADED)
        sel_bias = M.bias_table(torch.from_numpy(b).to(DEV), cfg.n_hot, cfg.bias_cap, mode=O.BIAS_GRADED)
    st, qh, one = _q8_layer(cfg, rflags, 0, perm, sel_bias)
    _, _, sep = _q8_layer(cfg, rflags, 1, perm, sel_bias)
    wr_np = _np(st["wr"].float())
    off_np = None if st["logit_offset"] is None else _np(st["logit_offset"])
    router = O.ROUTER_SIGMOID if rflags & M.ROUTE_SIGMOID else O.ROUTER_SOFTMAX
    for step in range(steps):
        x = C.draw_x(cfg, DEV, step=step)
        r1 = one.forward(x)
        r2 = sep.forward(x)
        torch.cuda.synchronize()
        want = O.layer_forward(_np(x.float()), wr_np, qh, cfg.H, cfg.I, cfg.k, O.RESIDENT, logit_offset=off_np,
                               bias=bias_np, router=router, damped=bool(rflags & M.ROUTE_DAMPED), quant=True)
        assert np.array_equal(_np(r1["ids"]), want["ids"]), f"step {step}: ids"
        assert np.abs(_np(r1["w"]) - want["w"]).max() <= 1e-6, f"step {step}: w"
        assert_out_close(_np(r1["out"].float()), want["out"], f"step {step}: out")
        assert np.array_equal(_np(r1["ids"]), _np(r2["ids"]))
        assert torch.equal(r1["w"], r2["w"]), f"step {step}: weights differ from the router kernels'"
        assert torch.equal(r1["out"], r2["out"]), f"step {step}: persistent and separate kernels differ"
    assert int(_np(one.dev_status)[0]) == 0 and int(_np(sep.dev_status)[0]) == 0
    return one


@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_decode_q8_qwen_resident(T):
    _check(C.qwen(T, S=128, mode=C.MODE_RESIDENT), steps=3)


def test_decode_q8_tiny_shape_offset_and_bias():
    # 16 experts, H 256, I 128: fewer quads and column pairs than CTAs, so many CTAs own no work
    _check(C.TINY.with_(T=7, logit_offset=True, bias_cap=-0.5, n_hot=6, zipf_s=1.1), steps=3)
    _check(C.TINY.with_(T=1), steps=3)


def test_decode_q8_sigmoid_router_and_damped_weights():
    import expert_slot_cache_gb300 as M
    cfg = C.TINY.with_(T=6, bias_cap=-0.25, n_hot=8, zipf_s=1.1)
    _check(cfg, steps=2, rflags=M.ROUTE_SIGMOID)
    _check(cfg, steps=2, rflags=M.ROUTE_DAMPED)


def test_decode_q8_remapped_pool():
    cfg = C.qwen(4, S=128, mode=C.MODE_RESIDENT)
    perm = np.random.default_rng(11).permutation(cfg.E).astype(np.int32)
    _check(cfg, steps=2, perm=perm)


def test_decode_q8_is_one_launch():
    import expert_slot_cache_gb300 as M
    cfg = C.qwen(2, S=128, mode=C.MODE_RESIDENT)
    _, _, layer = _q8_layer(cfg)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
    for ev in evs:
        ev.record()
    arr = (ctypes.c_void_p * 8)(*[e.cuda_event for e in evs])
    tags = (ctypes.c_int32 * 4)()
    prof = M.binding.Prof(arr, 8, 0, tags)
    layer.forward(C.draw_x(cfg, DEV), prof=prof)
    torch.cuda.synchronize()
    assert prof.used == 2 and tags[0] == 8  # one (start, end) pair: MOE_PROF_DECODE


def test_decode_q8_graph_replay_counters_back_to_zero():
    cfg = C.qwen(3, S=128, mode=C.MODE_RESIDENT)
    st, qh, layer = _q8_layer(cfg)
    xs = [C.draw_x(cfg, DEV, step=i) for i in range(4)]
    x = torch.empty_like(xs[0])
    x.copy_(xs[0])
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=DEV)
    ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=DEV)
    w = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=DEV)
    layer.forward(x, out=out, ids=ids, w=w)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(x, out=out, ids=ids, w=w)
    wr_np = _np(st["wr"].float())
    for i in range(4):
        x.copy_(xs[i])
        g.replay()
        torch.cuda.synchronize()
        want = O.layer_forward(_np(x.float()), wr_np, qh, cfg.H, cfg.I, cfg.k, O.RESIDENT, quant=True)
        assert np.array_equal(_np(ids), want["ids"]), f"replay {i}: ids"
        assert_out_close(_np(out.float()), want["out"], f"replay {i}: out")
    assert int(_np(layer.dev_status)[0]) == 0
    # the arrival counters (start of the workspace) are back at zero
    assert int(layer.workspace[: 4 * (cfg.E + 4)].count_nonzero()) == 0


def _check_q8_x(cfg, x):
    """One step on the given x: the oracle, and bit for bit the separate W8A8 kernels."""
    st, qh, one = _q8_layer(cfg)
    _, _, sep = _q8_layer(cfg, decode_kernels=1)
    r1, r2 = one.forward(x), sep.forward(x)
    torch.cuda.synchronize()
    want = O.layer_forward(_np(x.float()), _np(st["wr"].float()), qh, cfg.H, cfg.I, cfg.k, O.RESIDENT, quant=True)
    assert np.array_equal(_np(r1["ids"]), want["ids"])
    assert_out_close(_np(r1["out"].float()), want["out"], "out")
    assert torch.equal(r1["out"], r2["out"])
    assert int(_np(one.dev_status)[0]) == 0
    return want


def test_decode_q8_identical_tokens_give_every_expert_eight_rows():
    # every routed expert has T = 8 rows: the stage loops compiled for eight rows, h of eight rows a segment
    cfg = C.qwen(8, S=128, mode=C.MODE_RESIDENT)
    x = C.draw_x(cfg, DEV)[:1].repeat(cfg.T, 1).contiguous()
    want = _check_q8_x(cfg, x)
    assert all(len(set(want["ids"][:, j])) == 1 for j in range(cfg.k))


def test_decode_q8_256_experts():
    cfg = C.qwen(8, S=256, mode=C.MODE_RESIDENT).with_(E=256, H=512, I=256)
    _check_q8_x(cfg, C.draw_x(cfg, DEV))
