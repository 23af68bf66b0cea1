"""The 48-layer stack (288 experts per layer, top-8, H 2048, I 512), slot
variant: 144 of each layer's experts in VRAM slots, the rest pinned in host
memory, T = 32 tokens, chunks of 18 tokens.  Step 0 runs eagerly, steps 1-2
replay one CUDA graph over all 48 layers.  Sampled layers are checked against
the oracle every step: ids bit-exact, outputs within tolerance, cache state
bit-exact, and every occupied slot holds its expert's bytes.
"""
import numpy as np
import pytest
import torch

import oracle as O
from harness import configs as C
from tests._setup import HostSlabs, assert_out_close

pytestmark = pytest.mark.gpu
SAMPLED = (0, 23, 47)
STEPS = 3


def test_stack48_slots_graph_replay():
    import bench
    cfg = C.STACK_SLOTS
    wl = bench.StackWorkload(cfg, "cuda", steps=STEPS)
    ostates = {l: O.CacheState.from_slots(C.initial_residency(cfg, l), cfg.E) for l in SAMPLED}
    wr = {l: wl.layers[l].w_router.float().cpu().numpy() for l in SAMPLED}
    for st in range(STEPS):
        wl.load_step(st)
        if st == 0:
            wl.stack._run()
            torch.cuda.synchronize()
            wl.stack.capture()
        else:
            wl.stack.replay()
        torch.cuda.synchronize()
        for l in SAMPLED:
            x = wl.inputs[st, l].float().cpu().numpy()
            want = O.layer_forward(x, wr[l], HostSlabs(wl.hosts[l]), cfg.H, cfg.I, cfg.k, O.GATHER, O.LRU,
                                   ostates[l])
            assert len(want["chunks"]) == 2
            assert np.array_equal(wl.stack.ids[l].cpu().numpy(), want["ids"]), (st, l)
            assert_out_close(wl.stack.outs[l].float().cpu().numpy(), want["out"], f"step {st} layer {l}")
            gs = wl.layers[l].state
            assert gs.e2s.cpu().numpy().tolist() == ostates[l].e2s.tolist(), (st, l)
            assert gs.s2e.cpu().numpy().tolist() == ostates[l].s2e.tolist(), (st, l)
            assert (gs.prio.cpu().numpy().astype(np.uint32)).tolist() == ostates[l].prio.tolist(), (st, l)
    for l in SAMPLED:
        s2e = wl.layers[l].state.s2e.cpu().numpy()
        pool = wl.layers[l].pool
        for s in range(0, cfg.S, 13):
            assert torch.equal(pool[s].cpu(), wl.hosts[l][s2e[s]])
        assert int(wl.layers[l].dev_status.item()) == 0


def test_stack48_per_layer_slot_budgets_expert_waves():
    # "Betelgeuse ... on an RTX 3060", "Arrival-Slack VRAM Slot Pool": more slots on the first layers,
    # fewer in the middle and at the tail; every layer owns its pool and cache state
    import bench
    cfg = C.STACK_BUDGET
    sampled = (0, 4, 5, 30, 43, 47)
    assert len({C.layer_S(cfg, l) for l in sampled}) == 3
    wl = bench.StackWorkload(cfg, "cuda", steps=STEPS)
    ostates = {l: O.CacheState.from_slots(C.initial_residency(cfg, l), cfg.E) for l in sampled}
    wr = {l: wl.layers[l].w_router.float().cpu().numpy() for l in sampled}
    for st in range(STEPS):
        wl.load_step(st)
        if st == 0:
            wl.stack._run()
            torch.cuda.synchronize()
            wl.stack.capture()
        else:
            wl.stack.replay()
        torch.cuda.synchronize()
        for l in sampled:
            assert wl.layers[l].S == C.layer_S(cfg, l)
            x = wl.inputs[st, l].float().cpu().numpy()
            want = O.layer_forward(x, wr[l], HostSlabs(wl.hosts[l]), cfg.H, cfg.I, cfg.k, O.GATHER, O.LRU,
                                   ostates[l], schedule=O.SCHED_WAVES)
            assert np.array_equal(wl.stack.ids[l].cpu().numpy(), want["ids"]), (st, l)
            assert_out_close(wl.stack.outs[l].float().cpu().numpy(), want["out"], f"step {st} layer {l}")
            gs = wl.layers[l].state
            assert gs.e2s.cpu().numpy().tolist() == ostates[l].e2s.tolist(), (st, l)
            assert gs.s2e.cpu().numpy().tolist() == ostates[l].s2e.tolist(), (st, l)
            assert (gs.prio.cpu().numpy().astype(np.uint32)).tolist() == ostates[l].prio.tolist(), (st, l)
            assert int(gs.stamp.item()) == ostates[l].stamp, (st, l)
    for l in sampled:
        s2e = wl.layers[l].state.s2e.cpu().numpy()
        pool = wl.layers[l].pool
        for s in range(0, C.layer_S(cfg, l), 7):
            assert torch.equal(pool[s].cpu(), wl.hosts[l][s2e[s]])
        assert int(wl.layers[l].dev_status.item()) == 0
