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
