"""The persistent decode kernels' bounded grid-wide waits: a wait that runs out
sets MOE_DEV_TIMEOUT, the kernel finishes (its later phases skip their work but
keep their arrivals, so no other wait depends on the lost one), the last CTA
out puts the counters back to zero, and the next call on the same workspace is
correct.  On an expert-cache step whose router wait runs out, the cache state,
the statistics and the pool stay as they were.  The failing wait is made on the
host: the router's arrival counter is set far below zero before the call, so its
grid-wide arrival never completes (nothing on the GPU faults or hangs; the wait
gives up after its bounded polls).
"""
import numpy as np
import pytest
import torch

import oracle as O
from harness import configs as C
from tests._setup import HostSlabs, assert_out_close, stage_layer
from tests.test_gpu_q8 import QHost

pytestmark = pytest.mark.gpu
DEV = "cuda"
MOE_DEV_TIMEOUT = 3
CTR_LOGITS = 0  # the router's arrival counter, right after the E per-expert counters


def _np(t):
    return t.detach().cpu().numpy()


@pytest.mark.parametrize("quant", [0, 1], ids=["bf16", "w8a8"])
def test_decode_wait_that_runs_out_reports_timeout_and_recovers(quant):
    import expert_slot_cache_gb300 as M
    cfg = C.qwen(2, S=128, mode=C.MODE_RESIDENT)
    st = stage_layer(cfg)
    pool, host = st["slabs_dev"], HostSlabs(st["host"])
    if quant:
        pool = M.quantize_slabs(st["slabs_dev"], cfg.H, cfg.I)
        host = QHost(st["host"], cfg.H, cfg.I)
    layer = M.SlotCachedMoELayer(st["wr"], pool, cfg.k, cfg.I, C.MODE_RESIDENT, max_tokens=cfg.T, quant=quant)
    ctr = layer.workspace.view(torch.int32)
    x = C.draw_x(cfg, DEV)
    ctr[cfg.E + CTR_LOGITS] = -(1 << 30)  # an arrival count that G arrivals never bring to G
    layer.forward(x)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == MOE_DEV_TIMEOUT
    assert int(ctr[: cfg.E + 4].count_nonzero()) == 0  # the last CTA out reset every counter
    layer.dev_status.zero_()
    r = layer.forward(x)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    want = O.layer_forward(_np(x.float()), _np(st["wr"].float()), host, cfg.H, cfg.I, cfg.k, O.RESIDENT,
                           quant=bool(quant))
    assert np.array_equal(_np(r["ids"]), want["ids"])
    assert_out_close(_np(r["out"].float()), want["out"], "after the timeout")


def test_decode_gather_wait_that_runs_out_leaves_the_cache_as_it_was():
    import expert_slot_cache_gb300 as M
    cfg = C.qwen(2)
    st = stage_layer(cfg)
    s2e0 = C.initial_residency(cfg)
    pool = st["slabs_dev"][torch.from_numpy(s2e0.astype(np.int64)).to(DEV)].contiguous()
    state = M.CacheState.from_slots(s2e0, cfg.E)
    layer = M.SlotCachedMoELayer(st["wr"], pool, cfg.k, cfg.I, cfg.mode, cfg.policy, host_slabs=st["host"],
                                 state=state, max_tokens=cfg.T)
    ctr = layer.workspace.view(torch.int32)
    snap, pool0, stats0 = state.clone(), pool.clone(), layer.stats.clone()
    x = C.draw_x(cfg, DEV)
    ctr[cfg.E + CTR_LOGITS] = -(1 << 30)
    layer.forward(x)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == MOE_DEV_TIMEOUT
    assert int(ctr[: cfg.E + 4 + 64].count_nonzero()) == 0
    for f in ("e2s", "s2e", "prio", "stamp"):
        assert torch.equal(getattr(state, f), getattr(snap, f)), f
    assert torch.equal(layer.stats, stats0) and torch.equal(pool, pool0)
    # the next call on the same state and workspace is the oracle's first step
    layer.dev_status.zero_()
    r = layer.forward(x)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    ostate = O.CacheState.from_slots(s2e0, cfg.E)
    want = O.layer_forward(_np(x.float()), _np(st["wr"].float()), HostSlabs(st["host"]), cfg.H, cfg.I, cfg.k,
                           cfg.mode, cfg.policy, ostate)
    assert np.array_equal(_np(r["ids"]), want["ids"])
    assert_out_close(_np(r["out"].float()), want["out"], "after the timeout")
    assert _np(state.e2s).tolist() == ostate.e2s.tolist() and _np(state.s2e).tolist() == ostate.s2e.tolist()
    assert int(layer.stats[0]) == len(want["chunks"][0]["miss_e"])
