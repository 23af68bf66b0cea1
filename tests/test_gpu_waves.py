"""GPU parity of the expert-wave schedule (each missing expert loaded at most
once per step) against the oracle, through the layer forward of the C ABI.

"Porting vllm-expert-cache to NVIDIA GPUs", "What this package does" (victims
among slots the step does not need) and "Measuring, without fooling
yourself" (count misses, not tokens).  Every step: ids bit-exact, routing
weights within 1e-6, the cache state (e2s, s2e, prio, stamp) bit-exact, the
loads and manage calls counted exactly, every occupied slot holding its
expert's bytes, and the output within the bf16 tolerance.
"""
import numpy as np
import pytest

from harness import configs as C
from tests.test_gpu_parity import _run_layer

pytestmark = pytest.mark.gpu
W = C.SCHED_WAVES


@pytest.mark.parametrize("T", [8, 32, 64])
def test_waves_qwen_lru(T):
    _run_layer(C.qwen(T, schedule=W), steps=3)


def test_waves_qwen_lfu_single_stream():
    _run_layer(C.qwen(64, policy=C.POLICY_LFU, schedule=W), steps=3, side=False)


def test_waves_tiny_many_waves():
    # E = 16, S = 5, T*k = 12: up to two later waves per step
    _run_layer(C.TINY.with_(T=6, S=5, mode=C.MODE_GATHER, schedule=W), steps=6)


def test_waves_pool_smaller_than_top_k():
    # S = 1 < k = 2: token chunks cannot serve this; waves load one expert per call
    _run_layer(C.TINY.with_(T=3, S=1, mode=C.MODE_GATHER, schedule=W), steps=3)


def test_waves_stack_shape():
    # one layer of the 48-layer slot variant: 288 experts, 144 slots, T = 32, top-8
    _run_layer(C.STACK_SLOTS.with_(schedule=W), steps=2)


def test_waves_step_that_fits_equals_token_chunks():
    # T*k <= S: one manage call under either schedule, the same state
    a = _run_layer(C.qwen(8, S=64, schedule=W), steps=2)
    b = _run_layer(C.qwen(8, S=64), steps=2)
    for f in ("e2s", "s2e", "prio", "stamp"):
        assert np.array_equal(getattr(a.state, f).cpu().numpy(), getattr(b.state, f).cpu().numpy()), f


def test_waves_with_live_cache_affinity():
    # affinity reads the expert -> slot table before the step's first manage call
    import expert_slot_cache_gb300 as M
    import oracle as O
    import torch
    from tests._setup import HostSlabs, assert_out_close, stage_layer
    from tests.test_gpu_parity import _check_state, _np
    cfg = C.qwen(64, schedule=W)
    st = stage_layer(cfg)
    s2e0 = C.initial_residency(cfg)
    pool = st["slabs_dev"][torch.from_numpy(s2e0.astype(np.int64)).to("cuda")].contiguous()
    gstate = M.CacheState.from_slots(s2e0, cfg.E)
    ostate = O.CacheState.from_slots(s2e0, cfg.E)
    layer = M.SlotCachedMoELayer(st["wr"], pool, cfg.k, cfg.I, cfg.mode, cfg.policy, host_slabs=st["host"],
                                 state=gstate, max_tokens=cfg.T, affinity=0.5, schedule=W)
    for step in range(3):
        x = C.draw_x(cfg, "cuda", step=step)
        r = layer.forward(x)
        torch.cuda.synchronize()
        want = O.layer_forward(_np(x.float()), _np(st["wr"].float()), HostSlabs(st["host"]), cfg.H, cfg.I, cfg.k,
                               cfg.mode, cfg.policy, ostate, affinity=0.5, schedule=O.SCHED_WAVES)
        assert np.array_equal(_np(r["ids"]), want["ids"]), step
        assert_out_close(_np(r["out"].float()), want["out"], f"step {step}")
        _check_state(gstate, ostate, f"step {step}")
    assert int(layer.dev_status.item()) == 0
