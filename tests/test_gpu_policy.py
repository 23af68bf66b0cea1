"""Policy replay: one drifting Zipf routing trace through expert_cache_manage
under LRU, LFU and STATIC; per-step misses and the final cache state match
the oracle replay exactly."""
import numpy as np
import pytest
import torch

import oracle as O
from harness import configs as C

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("policy", [0, 1, 2], ids=["lru", "lfu", "static"])
def test_policy_replay_matches_oracle(policy):
    import expert_slot_cache_gb300 as M
    E, S, T, k = 128, 64, 8, 8
    trace = C.drifting_trace(E, k, T, 150, seed=11)
    s2e0 = C.initial_residency(C.TINY.with_(E=E, S=S, seed=E))
    gst = M.CacheState.from_slots(s2e0, E)
    ost = O.CacheState.from_slots(s2e0, E)
    ids_d = torch.from_numpy(trace).cuda()
    got, want = [], []
    for i in range(trace.shape[0]):
        got.append(M.cache_manage(ids_d[i], gst, policy).n_miss)
        want.append(len(O.manage(ost, trace[i], policy).miss_e))
    got = torch.cat(got).cpu().numpy()
    assert got.tolist() == want
    assert gst.s2e.cpu().numpy().tolist() == ost.s2e.tolist()
    assert (gst.prio.cpu().numpy().astype(np.uint32)).tolist() == ost.prio.tolist()


def test_policy_replay_bench_helper_reports_fewer_misses_for_recency_than_static():
    import bench
    trace = C.drifting_trace(128, 8, 8, 100, seed=3)
    r = bench.policy_replay(trace, 128, 64, "cuda", 9437184)
    assert r["lru"]["misses"] < r["static"]["misses"]
    assert r["static_best_fixed"]["misses"] <= r["static"]["misses"]


# ----------------------------------------------------------------------------
# Periodic re-pick of a STATIC pool (transcript: "every 500 tokens, say, have
# another look. Swap out whatever's gone cold")
# ----------------------------------------------------------------------------

def test_repick_golden_on_gpu():
    import json
    import os
    import expert_slot_cache_gb300 as M
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "repick_traces.json")))
    for c in g["cases"]:
        st = M.CacheState.from_slots(np.array(c["s2e"], dtype=np.int32), c["E"])
        counts = torch.tensor(c["counts"], dtype=torch.int32, device="cuda")
        r = M.cache_repick(counts, st)
        n = int(r.n_miss.item())
        assert r.miss_e[:n].cpu().tolist() == c["miss_e"] and r.miss_s[:n].cpu().tolist() == c["miss_s"], c["name"]
        assert st.s2e.cpu().tolist() == c["s2e_after"], c["name"]
        assert not counts.any()


@pytest.mark.parametrize("E,S", [(16, 5), (128, 64), (512, 192), (288, 288), (40, 100)])
def test_repick_random_states_match_oracle(E, S):
    import expert_slot_cache_gb300 as M
    rng = np.random.default_rng(E * 7 + S)
    for trial in range(20):
        s2e = np.full(S, -1, dtype=np.int32)
        n_res = int(rng.integers(0, min(S, E) + 1))
        s2e[rng.permutation(S)[:n_res]] = rng.permutation(E)[:n_res]
        counts = rng.integers(0, 3 if trial % 2 else 50, size=E).astype(np.int32)
        gst, ost = M.CacheState.from_slots(s2e, E), O.CacheState.from_slots(s2e, E)
        cd = torch.from_numpy(counts).cuda()
        r = M.cache_repick(cd, gst)
        want = O.repick(ost, counts.astype(np.int64))
        n = int(r.n_miss.item())
        assert r.miss_e[:n].cpu().tolist() == want.miss_e and r.miss_s[:n].cpu().tolist() == want.miss_s
        assert gst.s2e.cpu().tolist() == ost.s2e.tolist() and gst.e2s.cpu().tolist() == ost.e2s.tolist()
        assert not cd.any()


def test_window_count_matches_bincount():
    import expert_slot_cache_gb300 as M
    rng = np.random.default_rng(4)
    ids = rng.integers(0, 288, size=(3, 4096)).astype(np.int32)
    counts = torch.zeros(288, dtype=torch.int32, device="cuda")
    for i in range(3):
        M.cache_count(torch.from_numpy(ids[i]).cuda(), 288, counts)
    assert counts.cpu().numpy().tolist() == np.bincount(ids.reshape(-1), minlength=288).tolist()


def test_zero_return_layer_with_periodic_repick_matches_oracle():
    """Flash-Next zero-return layer (STATIC): window counts from the layer,
    a re-pick + gather every 2 steps; ids, outputs, cache state and slot bytes
    against the oracle replay of the same schedule."""
    import expert_slot_cache_gb300 as M
    from tests._setup import HostSlabs, assert_out_close, stage_layer
    cfg = C.FLASH.with_(T=4)
    st = stage_layer(cfg)
    b, _ = C.draw_brightness(cfg)
    bias_np = O.bias_table(b, cfg.n_hot, cfg.bias_cap)
    bias_d = M.bias_table(torch.from_numpy(b).cuda(), cfg.n_hot, cfg.bias_cap)
    s2e0 = C.initial_residency(cfg)
    pool = torch.empty(cfg.S, cfg.slab_elems, dtype=torch.bfloat16, device="cuda")
    for s, e in enumerate(s2e0):
        pool[s].copy_(st["slabs_dev"][e])
    gst, ost = M.CacheState.from_slots(s2e0, cfg.E), O.CacheState.from_slots(s2e0, cfg.E)
    counts = torch.zeros(cfg.E, dtype=torch.int32, device="cuda")
    ocounts = np.zeros(cfg.E, dtype=np.int64)
    layer = M.SlotCachedMoELayer(st["wr"], pool, cfg.k, cfg.I, cfg.mode, cfg.policy, host_slabs=st["host"],
                                 state=gst, sel_bias=bias_d, max_tokens=cfg.T, window_counts=counts)
    slabs = HostSlabs(st["host"])
    wr = st["wr"].float().cpu().numpy()
    loads = 0
    for step in range(6):
        x = C.draw_x(cfg, "cuda", step=step)
        res = layer.forward(x)
        torch.cuda.synchronize()
        want = O.layer_forward(x.float().cpu().numpy(), wr, slabs, cfg.H, cfg.I, cfg.k, O.ZERO_RETURN, O.STATIC,
                               ost, None, None, bias_np)
        O.window_count(ocounts, want["ids"])
        assert np.array_equal(res["ids"].cpu().numpy(), want["ids"]), step
        assert_out_close(res["out"].float().cpu().numpy(), want["out"], f"step {step}")
        assert counts.cpu().numpy().tolist() == ocounts.tolist(), step
        if step % 2 == 1:
            r = layer.repick()
            torch.cuda.synchronize()
            wr_ = O.repick(ost, ocounts)
            n = int(r.n_miss.item())
            loads += n
            assert r.miss_e[:n].cpu().tolist() == wr_.miss_e and r.miss_s[:n].cpu().tolist() == wr_.miss_s
    assert loads > 0
    assert gst.s2e.cpu().tolist() == ost.s2e.tolist()
    s2e = gst.s2e.cpu().numpy()
    for s in range(0, cfg.S, 7):
        assert torch.equal(pool[s].cpu(), st["host"][s2e[s]])
    assert int(layer.dev_status.item()) == 0
