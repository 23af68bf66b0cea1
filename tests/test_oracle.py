"""Pins for the CPU oracle, independent of the oracle itself.

Each test checks the oracle against something it does not compute from:
hand-derived fixtures (tests/golden), closed forms, exact integer sums,
error bounds, library routines (numpy/torch sort, topk, matmul), a second
cache model written differently, and brute-force dense evaluation.
"""
import itertools
import json
import math
import os
from collections import OrderedDict
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from harness import configs as C

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _bf16(a):
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


# ----------------------------------------------------------------------------
# Router logits
# ----------------------------------------------------------------------------

def test_logit_order_golden():
    g = _gold("logit_order.json")
    assert O.LOGIT_BLOCK == g["block"]
    for case in g["cases"]:
        x = np.zeros((1, case["H"]), dtype=np.float32)
        for h, v in case["x"].items():
            x[0, int(h)] = v
        w = np.ones((case["H"], 1), dtype=np.float32)
        assert O.router_logits(x, w)[0, 0] == np.float32(case["logit"])
        assert case["exact_sum"] == float(x.astype(np.float64).sum())


def test_logits_exact_on_small_integers():
    rng = np.random.default_rng(7)
    x = rng.integers(-8, 9, size=(5, 64)).astype(np.float32)
    w = rng.integers(-8, 9, size=(64, 12)).astype(np.float32)
    exact = [[sum(int(x[t, h]) * int(w[h, e]) for h in range(64)) for e in range(12)] for t in range(5)]
    assert np.array_equal(O.router_logits(x, w), np.array(exact, dtype=np.float32))


def test_logits_within_sequential_error_bound():
    rng = np.random.default_rng(8)
    T, H, E = 3, 512, 9
    x = _bf16(rng.normal(0, 1, (T, H)))
    w = _bf16(rng.normal(0, 0.02, (H, E)))
    got = O.router_logits(x, w)
    u = 2.0 ** -24
    gam = H * u / (1 - H * u)
    for t in range(T):
        for e in range(E):
            prods = [Fraction(float(x[t, h])) * Fraction(float(w[h, e])) for h in range(H)]
            exact = sum(prods)
            bound = gam * float(sum(abs(p) for p in prods))
            assert abs(float(got[t, e]) - float(exact)) <= bound


def test_logit_offset_added_after_sum():
    x = np.array([[1.0, 2.0]], dtype=np.float32)
    w = np.array([[1.0, 0.5], [0.25, 2.0]], dtype=np.float32)
    off = np.array([10.0, -1.0], dtype=np.float32)
    assert np.array_equal(O.router_logits(x, w, off), np.array([[11.5, 3.5]], dtype=np.float32))


# ----------------------------------------------------------------------------
# Top-k, weights, bias
# ----------------------------------------------------------------------------

def test_route_examples_golden():
    g = _gold("route_examples.json")
    logits = np.array([g["logits"]], dtype=np.float32)
    for case in g["cases"]:
        bias = None if case["bias"] is None else np.array(case["bias"], dtype=np.float32)
        ids = O.select_topk(logits, g["k"], bias)
        assert ids[0].tolist() == case["ids"]
        w = O.route_weights(logits, ids)
        assert np.allclose(w[0], case["w"], atol=1e-9)


def _topk_by_counting(scores, k):
    # rank(e) = number of experts ahead of e; the expert of rank j is the j-th pick
    E = len(scores)
    rank = [sum(1 for f in range(E) if scores[f] > scores[e] or (scores[f] == scores[e] and f < e)) for e in range(E)]
    return [rank.index(j) for j in range(k)]


def test_topk_matches_counting_definition_with_ties():
    rng = np.random.default_rng(3)
    for _ in range(50):
        E, k = int(rng.integers(4, 20)), int(rng.integers(1, 4))
        s = rng.integers(-3, 4, size=(2, E)).astype(np.float32)  # many ties
        ids = O.select_topk(s, k)
        for t in range(2):
            assert ids[t].tolist() == _topk_by_counting(s[t].tolist(), k)


def test_topk_matches_torch_on_distinct_scores():
    rng = np.random.default_rng(4)
    s = rng.normal(size=(16, 128)).astype(np.float32)
    ids = O.select_topk(s, 8)
    ref = torch.topk(torch.from_numpy(s), 8, dim=1, sorted=True).indices.numpy()
    assert np.array_equal(ids, ref)


def test_weights_closed_forms():
    rng = np.random.default_rng(5)
    logits = rng.normal(size=(6, 32)).astype(np.float32)
    ids = O.select_topk(logits, 5)
    w = O.route_weights(logits, ids)
    assert np.allclose(w.sum(1), 1.0, atol=1e-12)
    for t in range(6):
        for a, b in itertools.combinations(range(5), 2):
            r = math.exp(float(logits[t, ids[t, a]]) - float(logits[t, ids[t, b]]))
            assert w[t, a] / w[t, b] == pytest.approx(r, rel=1e-12)
    ids1 = O.select_topk(logits, 1)
    assert np.all(O.route_weights(logits, ids1) == 1.0)


def test_bias_table_golden():
    g = _gold("bias_table.json")
    b = np.array(g["b"], dtype=np.float32)
    got = O.bias_table(b, g["n_hot"], g["cap"])
    assert np.allclose(got, g["bias"], atol=1e-6)
    assert np.array_equal(O.bias_table(b, g["n_hot"], 0.0), np.array(g["cap_zero_bias"], dtype=np.float32))
    assert np.zeros((48, 512), dtype=np.float32).nbytes == g["table_bytes_48x512_fp32"]


def test_bias_rounding_is_one_fp32_round_of_fp64():
    rng = np.random.default_rng(9)
    b = rng.random(64).astype(np.float32) ** 3
    got = O.bias_table(b, 16, -2.0)
    hot = sorted(range(64), key=lambda e: (-float(b[e]), e))[:16]
    edge = min(float(b[e]) for e in hot)
    for e in range(64):
        want = 0.0 if e in hot else max(-2.0, math.log(float(b[e]) / edge))
        assert got[e] == np.float32(want)


def test_zero_bias_reproduces_unbiased_topk():
    cfg = C.FLASH.with_(T=8, H=256, E=64, k=10, I=64)
    x = C.draw_x(cfg).float().numpy()
    wr = C.draw_router(cfg).float().numpy()
    logits = O.router_logits(x, wr)
    b, _ = C.draw_brightness(cfg)
    bias0 = O.bias_table(b, 16, 0.0)
    assert np.all(bias0 == 0.0)
    assert np.array_equal(O.select_topk(logits, 10, bias0), O.select_topk(logits, 10))
    # a real bias moves picks towards the hot set but leaves the weights the router's own
    bias = O.bias_table(b, 16, -1.0)
    ids_b = O.select_topk(logits, 10, bias)
    w_b = O.route_weights(logits, ids_b)
    for t in range(8):
        l = np.array([float(logits[t, e]) for e in ids_b[t]])
        assert np.allclose(w_b[t], np.exp(l - l.max()) / np.exp(l - l.max()).sum())


# ----------------------------------------------------------------------------
# Permute
# ----------------------------------------------------------------------------

def test_permute_matches_stable_sort():
    rng = np.random.default_rng(11)
    for T, k, E in [(1, 1, 4), (7, 3, 5), (64, 8, 128), (33, 10, 512)]:
        ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
        count, offset, rows, pos = O.permute(ids, E)
        flat = ids.reshape(-1)
        assert np.array_equal(rows, np.argsort(flat, kind="stable"))
        assert np.array_equal(count, np.bincount(flat, minlength=E))
        assert offset[0] == 0 and offset[E] == T * k
        assert np.array_equal(rows[pos], np.arange(T * k))
        for e in range(E):
            assert np.all(flat[rows[offset[e]:offset[e + 1]]] == e)


# ----------------------------------------------------------------------------
# Manage / gather
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("trace", _gold("manage_traces.json")["traces"], ids=lambda t: t["name"])
def test_manage_golden_traces(trace):
    st = O.CacheState.from_slots(trace["s2e0"], trace["E"])
    for step in trace["steps"]:
        r = O.manage(st, np.array(step["ids"]), trace["policy"])
        assert r.miss_e == step["miss_e"]
        assert r.miss_s == step["miss_s"]
        assert r.hit_e == step["hit_e"]
        assert r.sid.tolist() == step["sid"]
        assert st.s2e.tolist() == step["s2e"]
        assert st.e2s.tolist() == step["e2s"]
        assert st.prio.tolist() == step["prio"]
        assert st.stamp == step["stamp"]


class _SecondModel:
    """An independently written cache model: per-slot records, greedy victim picking."""

    def __init__(self, s2e0, E, policy):
        self.E, self.policy = E, policy
        self.occ = OrderedDict((s, int(e)) for s, e in enumerate(s2e0))
        self.score = {s: 0 for s in self.occ}
        self.calls = 0

    def step(self, ids):
        self.calls += 1
        want = sorted(set(int(e) for e in ids))
        where = {e: s for s, e in self.occ.items() if e >= 0}
        hits = [e for e in want if e in where]
        miss = [e for e in want if e not in where]
        for e in hits:
            if self.policy == O.LRU:
                self.score[where[e]] = self.calls
            elif self.policy == O.LFU:
                self.score[where[e]] += 1
        taken = {where[e] for e in hits}
        placed = []
        for e in miss:
            if self.policy == O.STATIC:
                placed.append(-1)
                continue
            free = [s for s, v in self.occ.items() if v < 0 and s not in taken]
            if free:
                s = min(free)
            else:
                s = min((s for s in self.occ if s not in taken), key=lambda s: (self.score[s], s))
            self.occ[s] = e
            self.score[s] = self.calls if self.policy == O.LRU else 1
            taken.add(s)
            placed.append(s)
        return miss, placed

    def tables(self):
        s2e = [self.occ[s] for s in range(len(self.occ))]
        e2s = [-1] * self.E
        for s, e in enumerate(s2e):
            if e >= 0:
                e2s[e] = s
        return s2e, e2s, [self.score[s] for s in range(len(self.occ))]


def _zipf_ids(rng, steps, T, k, E, s=1.1):
    p = np.arange(1, E + 1, dtype=np.float64) ** -s
    p /= p.sum()
    perm = rng.permutation(E)
    out = []
    for _ in range(steps):
        rows = [perm[rng.choice(E, size=k, replace=False, p=p)] for _ in range(T)]
        out.append(np.array(rows, dtype=np.int32))
    return out


@pytest.mark.parametrize("policy", [O.LRU, O.LFU, O.STATIC])
@pytest.mark.parametrize("dist", ["uniform", "zipf"])
def test_manage_matches_second_model(policy, dist):
    rng = np.random.default_rng(100 + policy)
    E, S, T, k = 32, 12, 3, 4
    s2e0 = rng.permutation(E)[:S].astype(np.int32)
    s2e0[rng.integers(0, S)] = -1
    st = O.CacheState.from_slots(s2e0, E)
    m = _SecondModel(s2e0, E, policy)
    if dist == "zipf":
        traces = _zipf_ids(rng, 60, T, k, E)
    else:
        traces = [np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32) for _ in range(60)]
    for ids in traces:
        r = O.manage(st, ids, policy)
        miss, placed = m.step(ids.reshape(-1))
        assert r.miss_e == miss and r.miss_s == placed
        s2e, e2s, score = m.tables()
        assert st.s2e.tolist() == s2e and st.e2s.tolist() == e2s
        assert st.prio.tolist() == score


@pytest.mark.parametrize("policy", [O.LRU, O.LFU])
def test_manage_invariants(policy):
    rng = np.random.default_rng(200 + policy)
    E, S, T, k = 64, 24, 3, 8
    st = O.CacheState.from_slots(rng.permutation(E)[:S], E)
    for ids in _zipf_ids(rng, 80, T, k, E):
        before = set(int(e) for e in np.nonzero(st.e2s >= 0)[0])
        need = set(int(e) for e in ids.reshape(-1))
        used_slots = {int(st.e2s[e]) for e in need & before}
        r = O.manage(st, ids, policy)
        assert len(r.miss_e) == len(need - before)
        assert not (set(r.miss_s) & used_slots)
        assert all(st.e2s[e] >= 0 for e in need)
        for s, e in enumerate(st.s2e):
            if e >= 0:
                assert st.e2s[e] == s
        assert np.sum(st.e2s >= 0) == np.sum(st.s2e >= 0)
        assert np.array_equal(r.sid, st.e2s[ids])


def test_manage_all_resident_never_misses():
    E = 16
    st = O.CacheState.from_slots(np.arange(E), E)
    rng = np.random.default_rng(1)
    for _ in range(20):
        r = O.manage(st, rng.integers(0, E, size=(4, 2)), O.LRU)
        assert r.miss_e == []
        assert np.array_equal(st.s2e, np.arange(E))


def test_manage_capacity_and_chunking():
    st = O.CacheState.from_slots(np.arange(4), 8)
    with pytest.raises(O.CapacityError):
        O.manage(st, np.arange(5).reshape(1, 5), O.LRU)
    assert O.chunk_tokens(64, 8, 64, 128) == 8
    assert O.chunk_tokens(8, 8, 64, 128) == 8
    assert O.chunk_tokens(64, 8, 128, 128) == 64
    with pytest.raises(O.CapacityError):
        O.chunk_tokens(4, 8, 6, 128)


def _state(tr):
    st = O.CacheState.from_slots(np.array(tr["s2e0"], dtype=np.int32), tr["E"])
    st.prio[:] = tr["prio0"]
    st.stamp = tr["stamp0"]
    return st


@pytest.mark.parametrize("trace", _gold("wave_traces.json")["traces"], ids=lambda t: t["name"])
def test_wave_golden_traces(trace):
    st = _state(trace)
    waves = O.manage_waves(st, np.array(trace["ids"], dtype=np.int32), trace["policy"])
    assert len(waves) == len(trace["waves"])
    # replay the calls one at a time to compare the state after each
    st = _state(trace)
    first = True
    left = []
    for r, want in zip(waves, trace["waves"]):
        assert r.hit_e == want["hit_e"] and r.miss_e == want["miss_e"] and r.miss_s == want["miss_s"]
        if first:
            got = O.manage(st, np.array(trace["ids"], dtype=np.int32), trace["policy"], defer=True)
            left = list(got.deferred)
            assert got.deferred == want["deferred"]
            first = False
        else:
            O.manage(st, np.array(left[:trace["S"]], dtype=np.int32), trace["policy"])
            left = left[trace["S"]:]
        assert st.s2e.tolist() == want["s2e"] and st.prio.tolist() == want["prio"] and st.stamp == want["stamp"]
    if "loads_token_chunks" in trace:
        st = _state(trace)
        ids = np.array(trace["ids"], dtype=np.int32)
        C_ = O.chunk_tokens(ids.shape[0], trace["k"], trace["S"], trace["E"])
        loads = sum(len(O.manage(st, ids[t0:t0 + C_], trace["policy"]).miss_e) for t0 in range(0, ids.shape[0], C_))
        assert loads == trace["loads_token_chunks"]
        assert sum(len(w["miss_e"]) for w in trace["waves"]) < loads


def _second_model_waves(m, ids, S):
    """The expert-wave schedule on the second cache model, written from the reading
    independently of manage_waves: greedy victims per load, deferral when the
    step's free slots run out, then batches of at most S."""
    m.calls += 1
    want = sorted(set(int(e) for e in ids))
    where = {e: s for s, e in m.occ.items() if e >= 0}
    hits = [e for e in want if e in where]
    for e in hits:
        m.score[where[e]] = m.calls if m.policy == O.LRU else m.score[where[e]] + 1
    busy = {where[e] for e in hits}
    waves = [[]]
    deferred = []
    for e in (e for e in want if e not in where):
        pool = [s for s in m.occ if s not in busy]
        if not pool:
            deferred.append(e)
            continue
        s = min(pool, key=lambda s: (m.occ[s] >= 0, m.score[s] if m.occ[s] >= 0 else 0, s))
        m.occ[s], m.score[s] = e, (m.calls if m.policy == O.LRU else 1)
        busy.add(s)
        waves[0].append((e, s))
    for b0 in range(0, len(deferred), S):
        m.calls += 1
        busy = set()
        waves.append([])
        for e in deferred[b0:b0 + S]:
            s = min((s for s in m.occ if s not in busy), key=lambda s: (m.occ[s] >= 0, m.score[s], s))
            m.occ[s], m.score[s] = e, (m.calls if m.policy == O.LRU else 1)
            busy.add(s)
            waves[-1].append((e, s))
    return hits, waves


@pytest.mark.parametrize("policy", [O.LRU, O.LFU])
@pytest.mark.parametrize("dist", ["uniform", "zipf"])
def test_waves_match_second_model_and_load_each_miss_once(policy, dist):
    rng = np.random.default_rng(300 + 3 * policy + (dist == "zipf"))
    E, k = 40, 4
    for S in (3, 7, 16):
        s2e0 = rng.permutation(E)[:S].astype(np.int32)
        s2e0[rng.integers(0, S)] = -1
        st = O.CacheState.from_slots(s2e0, E)
        m = _SecondModel(s2e0, E, policy)
        T = 6
        traces = _zipf_ids(rng, 30, T, k, E) if dist == "zipf" else \
            [np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32) for _ in range(30)]
        for ids in traces:
            before = {int(e) for e in np.nonzero(st.e2s >= 0)[0]}
            need = {int(e) for e in ids.reshape(-1)}
            waves = O.manage_waves(st, ids, policy)
            hits, mw = _second_model_waves(m, ids.reshape(-1), S)
            assert waves[0].hit_e == hits
            assert [list(zip(w.miss_e, w.miss_s)) for w in waves] == mw
            s2e, e2s, score = m.tables()
            assert st.s2e.tolist() == s2e and st.e2s.tolist() == e2s and st.prio.tolist() == score
            loaded = [e for w in waves for e in w.miss_e]
            assert sorted(loaded) == sorted(need - before)  # each missing expert loaded exactly once
            assert all(len(w.miss_e) <= S for w in waves) and all(len(w.miss_e) > 0 for w in waves[1:])
            assert set(waves[0].hit_e) | set(loaded) == need


def test_waves_never_load_more_than_token_chunks():
    rng = np.random.default_rng(77)
    E, k, T = 32, 4, 12
    for S in (4, 9, 16):
        s2e0 = rng.permutation(E)[:S].astype(np.int32)
        a, b = O.CacheState.from_slots(s2e0, E), O.CacheState.from_slots(s2e0, E)
        C_ = O.chunk_tokens(T, k, S, E)
        la = lb = 0
        for ids in _zipf_ids(rng, 25, T, k, E):
            la += sum(len(w.miss_e) for w in O.manage_waves(a, ids, O.LRU))
            lb += sum(len(O.manage(b, ids[t0:t0 + C_], O.LRU).miss_e) for t0 in range(0, T, C_))
        assert la < lb


def test_wave_layer_equals_resident_layer_and_fills_slots():
    cfg = C.TINY.with_(T=6, S=5, mode=C.MODE_GATHER)
    rng = np.random.default_rng(5)
    H, I, E, k, T = cfg.H, cfg.I, cfg.E, cfg.k, cfg.T
    x = _bf16(rng.standard_normal((T, H)))
    wr = _bf16(rng.standard_normal((H, E)) * 0.02)
    host = _bf16(rng.standard_normal((E, 3 * H * I)) * 0.02)
    s2e0 = rng.permutation(E)[:cfg.S].astype(np.int32)
    st = O.CacheState.from_slots(s2e0, E)
    pool = host[s2e0].copy()
    res = O.layer_forward(x, wr, host, H, I, k, O.GATHER, O.LRU, st, pool, schedule=O.SCHED_WAVES)
    ref = O.layer_forward(x, wr, host, H, I, k, O.RESIDENT)
    assert np.array_equal(res["out"], ref["out"]) and np.array_equal(res["ids"], ref["ids"])
    waves = res["chunks"][0]["waves"]
    assert len(waves) >= 2  # the step needs more experts than the pool holds
    for s, e in enumerate(st.s2e):
        if e >= 0:
            assert np.array_equal(pool[s], host[e])
    # a step that fits the pool is one manage call, as in the token-chunk schedule
    st2 = O.CacheState.from_slots(s2e0, E)
    st3 = O.CacheState.from_slots(s2e0, E)
    r2 = O.layer_forward(x[:2], wr, host, H, I, k, O.GATHER, O.LRU, st2, schedule=O.SCHED_WAVES)
    r3 = O.layer_forward(x[:2], wr, host, H, I, k, O.GATHER, O.LRU, st3)
    assert r2["chunks"][0]["miss_e"] == r3["chunks"][0]["miss_e"]
    assert np.array_equal(st2.s2e, st3.s2e) and np.array_equal(st2.prio, st3.prio) and st2.stamp == st3.stamp


def test_gather_copies_bytes():
    rng = np.random.default_rng(2)
    host = rng.integers(0, 2 ** 16, size=(8, 40), dtype=np.uint16)
    pool = np.zeros((3, 40), dtype=np.uint16)
    O.gather(host, pool, [5, 1], [2, 0])
    assert np.array_equal(pool[2], host[5]) and np.array_equal(pool[0], host[1])
    assert not pool[1].any()


# ----------------------------------------------------------------------------
# FFN and combine
# ----------------------------------------------------------------------------

def test_silu_closed_forms():
    z = np.array([0.0, math.log(3.0), -math.log(3.0)])
    assert np.allclose(O.silu(z), [0.0, 0.75 * math.log(3.0), -0.25 * math.log(3.0)], rtol=1e-15, atol=0)


def test_swiglu_closed_form():
    H, I = 8, 4
    a = [0.0, math.log(3.0), -math.log(3.0), 2.0]
    bu = [1.0, 2.0, -4.0, 0.5]
    c = [3.0, 1.0, 2.0, -1.0]
    wg = np.zeros((H, I)); wu = np.zeros((H, I)); wd = np.zeros((I, H))
    wg[0] = a
    wu[0] = bu
    for i in range(I):
        wd[i, i + 2] = c[i]
    slab = np.concatenate([wg.ravel(), wu.ravel(), wd.ravel()])
    x = np.zeros((1, H)); x[0, 0] = 1.0
    y = O.swiglu_expert(x, slab, H, I)[0]
    want = np.zeros(H)
    for i in range(I):
        s = a[i] / (1.0 + math.exp(-a[i]))
        want[i + 2] = s * bu[i] * c[i]
    assert np.allclose(y, want, rtol=1e-14, atol=1e-15)
    assert y[4] == pytest.approx(-0.25 * math.log(3.0) * -4.0 * 2.0, rel=1e-14)


def test_swiglu_matches_explicit_loops():
    rng = np.random.default_rng(12)
    H, I, n = 6, 5, 3
    slab = rng.normal(size=3 * H * I)
    x = rng.normal(size=(n, H))
    y = O.swiglu_expert(x, slab, H, I)
    for r in range(n):
        h = []
        for i in range(I):
            g = sum(x[r, q] * slab[q * I + i] for q in range(H))
            u = sum(x[r, q] * slab[H * I + q * I + i] for q in range(H))
            h.append(g / (1 + math.exp(-g)) * u)
        for o in range(H):
            yo = sum(h[i] * slab[2 * H * I + i * H + o] for i in range(I))
            assert y[r, o] == pytest.approx(yo, rel=1e-12, abs=1e-14)


def _tiny_inputs(cfg=C.TINY):
    x = C.draw_x(cfg).float().numpy()
    wr = C.draw_router(cfg).float().numpy()
    host = C.draw_slabs(cfg).float().numpy()
    return x, wr, host


def test_layer_matches_dense_bruteforce():
    """Tiny config: evaluate every expert on every token, mask to the top-k, weight."""
    cfg = C.TINY
    x, wr, host = _tiny_inputs(cfg)
    res = O.layer_forward(x, wr, host, cfg.H, cfg.I, cfg.k, O.RESIDENT)
    logits = O.router_logits(x, wr)
    dense = np.stack([O.swiglu_expert(x, host[e], cfg.H, cfg.I) for e in range(cfg.E)])  # [E][T][H]
    ids = O.select_topk(logits, cfg.k)
    want = np.zeros((cfg.T, cfg.H))
    for t in range(cfg.T):
        mask = np.zeros(cfg.E, dtype=bool)
        mask[ids[t]] = True
        l = logits[t].astype(np.float64)
        p = np.where(mask, np.exp(l - l[mask].max()), 0.0)
        p /= p.sum()
        want[t] = (p[:, None] * dense[:, t, :]).sum(0)
    assert np.allclose(res["out"], want, rtol=1e-12, atol=1e-14)
    assert np.abs(want).max() > 0.01


def test_ffn_matches_torch_fp64_matmul():
    cfg = C.TINY
    x, wr, host = _tiny_inputs(cfg)
    e = 3
    xt = torch.from_numpy(x).double()
    s = torch.from_numpy(host[e]).double()
    n = cfg.H * cfg.I
    wg, wu, wd = s[:n].view(cfg.H, cfg.I), s[n:2 * n].view(cfg.H, cfg.I), s[2 * n:].view(cfg.I, cfg.H)
    ref = torch.matmul(torch.nn.functional.silu(xt @ wg) * (xt @ wu), wd).numpy()
    assert np.allclose(O.swiglu_expert(x, host[e], cfg.H, cfg.I), ref, rtol=1e-12, atol=1e-14)


def test_zero_return_partials_sum_to_full():
    cfg = C.TINY.with_(S=6)
    x, wr, host = _tiny_inputs(cfg)
    full = O.layer_forward(x, wr, host, cfg.H, cfg.I, cfg.k, O.RESIDENT)
    st = O.CacheState.from_slots(C.initial_residency(cfg.with_(S=6)), cfg.E)
    zr = O.layer_forward(x, wr, host, cfg.H, cfg.I, cfg.k, O.ZERO_RETURN, O.STATIC, st)
    assert np.allclose(zr["out_res"] + zr["out_miss"], full["out"], rtol=1e-12, atol=1e-14)
    assert np.abs(zr["out_miss"]).max() > 0 and np.abs(zr["out_res"]).max() > 0
    st_all = O.CacheState.from_slots(np.arange(cfg.E), cfg.E)
    zr_all = O.layer_forward(x, wr, host, cfg.H, cfg.I, cfg.k, O.ZERO_RETURN, O.STATIC, st_all)
    assert np.all(zr_all["out_miss"] == 0.0)
    assert np.array_equal(zr_all["out_res"], zr_all["out"])


def test_gather_mode_chunked_equals_resident():
    cfg = C.TINY.with_(T=9, S=5, k=2)
    x = C.draw_x(cfg).float().numpy()
    wr = C.draw_router(cfg).float().numpy()
    host = C.draw_slabs(cfg).float().numpy()
    full = O.layer_forward(x, wr, host, cfg.H, cfg.I, cfg.k, O.RESIDENT)
    s2e0 = C.initial_residency(cfg)
    st = O.CacheState.from_slots(s2e0, cfg.E)
    pool = host[s2e0].copy()
    g = O.layer_forward(x, wr, host, cfg.H, cfg.I, cfg.k, O.GATHER, O.LRU, st, pool)
    assert len(g["chunks"]) == 5  # floor(5/2) = 2 tokens per chunk
    assert np.allclose(g["out"], full["out"], rtol=1e-12, atol=1e-14)
    for s, e in enumerate(st.s2e):
        assert np.array_equal(pool[s], host[e])


def test_affinity_golden():
    g = _gold("affinity_example.json")
    logits = np.array([g["logits"]], dtype=np.float32)
    ids = O.select_topk(logits, g["k"], resident=np.array(g["resident"]), affinity=g["affinity"])
    assert ids[0].tolist() == g["ids"]
    assert O.select_topk(logits, g["k"])[0].tolist() == g["ids_without"]
    assert np.allclose(O.route_weights(logits, ids)[0], g["w"], atol=1e-9)


def test_affinity_zero_or_nothing_resident_is_plain_topk():
    rng = np.random.default_rng(21)
    logits = rng.normal(size=(6, 40)).astype(np.float32)
    res = rng.random(40) < 0.5
    plain = O.select_topk(logits, 5)
    assert np.array_equal(O.select_topk(logits, 5, resident=res, affinity=0.0), plain)
    assert np.array_equal(O.select_topk(logits, 5, resident=np.zeros(40, bool), affinity=0.7), plain)
    # a large affinity picks only resident experts while at least k are resident
    ids = O.select_topk(logits, 5, resident=res, affinity=100.0)
    assert res[ids].all()


# ----------------------------------------------------------------------------
# Routing variants ("Nudge, don't cut": hard mask, flat bias, damped weights,
# GLM's sigmoid router)
# ----------------------------------------------------------------------------

def _ulp32(v):
    v = np.abs(np.asarray(v, dtype=np.float64))
    return np.spacing(v.astype(np.float32)).astype(np.float64)


def test_exp32_within_two_ulp_of_the_exact_exponential():
    xs = np.concatenate([np.linspace(-80.0, 88.0, 400001, dtype=np.float32),
                         np.array([0.0, 1.0, -1.0, 0.5, 1e-8, -1e-8, 0.34657, -0.34657, 0.6931472], np.float32)])
    got = O.exp32(xs).astype(np.float64)
    want = np.exp(xs.astype(np.float64))
    assert np.all(np.abs(got - want) <= 2 * _ulp32(want))
    assert O.exp32(np.float32(0.0)) == np.float32(1.0)
    assert O.exp32(np.float32(89.0)) == np.float32(np.inf) and O.exp32(np.float32(-81.0)) == 0.0


def test_sigmoid32_within_three_ulp_and_symmetric():
    ls = np.linspace(-30.0, 30.0, 200001, dtype=np.float32)
    got = O.sigmoid32(ls).astype(np.float64)
    want = 1.0 / (1.0 + np.exp(-ls.astype(np.float64)))
    assert np.all(np.abs(got - want) <= 3 * _ulp32(want))
    assert O.sigmoid32(np.float32(0.0)) == np.float32(0.5)
    assert np.all(np.abs(O.sigmoid32(ls).astype(np.float64) + O.sigmoid32(-ls).astype(np.float64) - 1.0) < 2e-7)


def test_bias_modes_golden():
    g = _gold("route_variants.json")["bias_modes"]
    b = np.array(g["b"], dtype=np.float32)
    assert O.bias_table(b, g["n_hot"], g["flat_value"], O.BIAS_FLAT).tolist() == g["flat"]
    hard = O.bias_table(b, g["n_hot"], -1.0, O.BIAS_HARD)
    want = [float(v) for v in g["hard"]]
    assert hard.tolist() == want


def test_hard_mask_picks_the_top_k_of_the_hot_set():
    rng = np.random.default_rng(5)
    E, k, n_hot = 40, 6, 12
    b = rng.random(E).astype(np.float32)
    bias = O.bias_table(b, n_hot, -1.0, O.BIAS_HARD)
    hot = np.isfinite(bias)
    logits = rng.normal(size=(9, E)).astype(np.float32)
    ids = O.select_topk(logits, k, bias)
    masked = np.where(hot[None, :], logits.astype(np.float64), -np.inf)
    want = np.argsort(-masked, axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids, want)


def test_damped_and_selection_only_weights_golden():
    g = _gold("route_variants.json")["damped"]
    logits = np.array([g["logits"]], dtype=np.float32)
    bias = np.array(g["bias"], dtype=np.float32)
    ids, w, _ = _route_from_logits(logits, g["k"], bias, damped=True)
    assert ids[0].tolist() == g["ids"]
    assert np.allclose(w[0], g["w_damped"], rtol=0, atol=1e-12)
    ids, w, _ = _route_from_logits(logits, g["k"], bias, damped=False)
    assert np.allclose(w[0], g["w_select_only"], rtol=0, atol=1e-12)


def test_sigmoid_router_golden():
    g = _gold("route_variants.json")["sigmoid"]
    logits = np.array([g["logits"]], dtype=np.float32)
    bias = np.array(g["bias"], dtype=np.float32)
    ids, w, _ = _route_from_logits(logits, g["k"], bias, router=O.ROUTER_SIGMOID)
    assert ids[0].tolist() == g["ids_sigmoid"]
    assert np.allclose(w[0], g["w_sigmoid"], rtol=0, atol=1e-12)
    ids, _, _ = _route_from_logits(logits, g["k"], bias, router=O.ROUTER_SOFTMAX)
    assert ids[0].tolist() == g["ids_softmax"]


def _route_from_logits(logits, k, bias, router=0, damped=False):
    ids = O.select_topk(logits, k, bias, router=router)
    return ids, O.route_weights(logits, ids, router, bias, damped), logits


# ----------------------------------------------------------------------------
# Periodic re-pick of a STATIC pool (transcript: "every 500 tokens, say, have
# another look. Swap out whatever's gone cold")
# ----------------------------------------------------------------------------

def test_repick_golden_traces():
    g = _gold("repick_traces.json")
    for c in g["cases"]:
        st = O.CacheState.from_slots(np.array(c["s2e"], dtype=np.int32), c["E"])
        counts = np.array(c["counts"], dtype=np.int64)
        r = O.repick(st, counts)
        assert r.miss_e == c["miss_e"] and r.miss_s == c["miss_s"], c["name"]
        assert st.s2e.tolist() == c["s2e_after"], c["name"]
        assert sorted(e for e in st.s2e.tolist() if e >= 0) == sorted(c["new_set"]), c["name"]
        assert not counts.any()


def test_repick_matches_lexsort_top_s_and_keeps_stayers_in_place():
    rng = np.random.default_rng(12)
    for trial in range(200):
        E = int(rng.integers(4, 40))
        S = int(rng.integers(1, E + 1))
        perm = rng.permutation(E)
        s2e = np.full(S, -1, dtype=np.int32)
        n_res = int(rng.integers(0, S + 1))
        s2e[rng.permutation(S)[:n_res]] = perm[:n_res]
        st = O.CacheState.from_slots(s2e, E)
        counts = rng.integers(0, 4, size=E)
        old_e2s = st.e2s.copy()
        resident = old_e2s >= 0
        # independent ranking: lexsort keys (last key is primary)
        order = np.lexsort((np.arange(E), (~resident).astype(int), -counts))
        want = set(order[:S].tolist())
        r = O.repick(st, counts.copy())
        now = {int(e) for e in st.s2e if e >= 0}
        assert now == want
        assert len(r.miss_e) == len(want - {e for e in range(E) if resident[e]})
        for e in want:
            if resident[e]:
                assert st.e2s[e] == old_e2s[e]  # experts that stay never move
        assert all(st.s2e[st.e2s[e]] == e for e in range(E) if st.e2s[e] >= 0)


# ----------------------------------------------------------------------------
# W8A8 experts ("Porting vllm-expert-cache to NVIDIA GPUs": W8A8 model;
# weights and their scales indexed by the same id)
# ----------------------------------------------------------------------------

def test_quantize_cols_worked_example():
    # column scales 254/127 = 2, 0 (all zero), 127/127 = 1; codes rint(v / s), halves to even
    W = np.array([[254.0, 0.0, -127.0], [-127.0, 0.0, 63.5], [63.0, 0.0, 0.0]], dtype=np.float32)
    q, sc = O.quantize_cols(W)
    assert sc.tolist() == [2.0, 0.0, 1.0]
    assert q.tolist() == [[127, 0, -127], [-64, 0, 64], [32, 0, 0]]


def test_quantization_error_within_half_a_step():
    rng = np.random.default_rng(8)
    W = (rng.standard_normal((300, 40)) * rng.random(40) * 3).astype(np.float32)
    q, sc = O.quantize_cols(W)
    assert np.abs(q).max() <= 127 and (np.abs(q) == 127).any(axis=0).all()
    err = np.abs(W.astype(np.float64) - q.astype(np.float64) * sc.astype(np.float64))
    assert np.all(err <= 0.5 * sc.astype(np.float64) * (1 + 1e-5) + 1e-30)


def test_q8_slab_layout_by_index_formula():
    rng = np.random.default_rng(9)
    H, I = 16, 8
    slab = (rng.standard_normal(3 * H * I) * 0.02).astype(np.float32)
    b = O.quantize_slab(slab, H, I)
    assert b.size == O.q8_slab_bytes(H, I) == 3 * H * I + 4 * (2 * I + H)
    qg, qu, qd, sg, su, sd = O.unpack_q8_slab(b, H, I)
    wg = slab[:H * I].reshape(H, I)
    q_ref, s_ref = O.quantize_cols(wg)
    assert np.array_equal(sg, s_ref) and np.array_equal(qg, q_ref)
    raw = b.view(np.int8)
    for k in range(H):
        for n in range(I):
            assert raw[((k >> 2) * I + n) * 4 + (k & 3)] == q_ref[k, n]
    wd = slab[2 * H * I:].reshape(I, H)
    assert np.array_equal(qd, O.quantize_cols(wd)[0]) and np.array_equal(sd, O.quantize_cols(wd)[1])


def test_q8_expert_exact_integer_sums_and_zero_row():
    from oracle import moe_oracle as MO
    rng = np.random.default_rng(10)
    H, I = 32, 16
    slab = (rng.standard_normal(3 * H * I) * 0.02).astype(np.float32)
    b = O.quantize_slab(slab, H, I)
    qg, qu, qd, sg, su, sd = O.unpack_q8_slab(b, H, I)
    x = rng.standard_normal((3, H)).astype(np.float32)
    x[1] = 0.0
    qx, sx = O.quantize_rows(x)
    # integer sums with Python ints (exact), then the defined fp32 steps
    for r in range(3):
        for n in range(I):
            acc = sum(int(qx[r, kk]) * int(qg[kk, n]) for kk in range(H))
            g = np.float32(np.float32(acc) * sg[n]) * sx[r]
            assert np.float32(g) == MO._dequant(qx[r:r + 1].astype(np.int64) @ qg.astype(np.int64), sg, sx[r:r + 1])[0, n]
    y = O.swiglu_expert_q8(x, b, H, I)
    assert np.all(y[1] == 0.0) and sx[1] == 0.0


def test_q8_expert_close_to_the_bf16_expert():
    # three 8-bit quantisations (weights per channel, x and h per row), each a
    # relative noise of about (amax/rms)/127/sqrt(12) ~ 1% for Gaussian data:
    # the output's relative L2 error is a few percent at most
    rng = np.random.default_rng(11)
    H, I = 256, 128
    slab = (rng.standard_normal(3 * H * I) * 0.02).astype(np.float32)
    x = rng.standard_normal((6, H)).astype(np.float32)
    yq = O.swiglu_expert_q8(x, O.quantize_slab(slab, H, I), H, I)
    y = O.swiglu_expert(x, slab, H, I)
    assert np.linalg.norm(yq - y) / np.linalg.norm(y) < 4e-2


def _q8_hand_slab(g, wd_factor=1.0):
    """bf16 slab values (code x scale, exact in bf16) of the hand-worked W8A8 expert."""
    wg = np.array(g["qg"], dtype=np.float32) * np.float32(g["weight_scale_g"])
    wu = np.array(g["qu"], dtype=np.float32) * np.float32(g["weight_scale_u"])
    wd = np.array(g["qd"], dtype=np.float32) * np.float32(g["weight_scale_d"] * wd_factor)
    slab = np.concatenate([wg.reshape(-1), wu.reshape(-1), wd.reshape(-1)])
    assert np.array_equal(_bf16(slab), slab)  # the slab is exactly representable in bf16
    return slab


def test_q8_expert_hand_worked_example():
    g = _gold("q8_example.json")
    H, I = g["H"], g["I"]
    b = O.quantize_slab(_q8_hand_slab(g), H, I)
    qg, qu, qd, sg, su, sd = O.unpack_q8_slab(b, H, I)
    assert qg.tolist() == g["qg"] and qu.tolist() == g["qu"] and qd.tolist() == g["qd"]
    assert np.all(sg == g["weight_scale_g"]) and np.all(su == g["weight_scale_u"])
    assert np.all(sd == g["weight_scale_d"])
    x = np.array(g["x"], dtype=np.float32)
    qx, sx = O.quantize_rows(x)
    assert qx.tolist() == g["x_codes"] and sx.tolist() == g["x_scales"]
    qh, sh = O.quantize_rows(np.array(g["h"], dtype=np.float32))
    assert qh.tolist() == g["h_codes"] and sh.tolist() == g["h_scales"]
    y = O.swiglu_expert_q8(x, b, H, I)
    assert y.dtype == np.float32 and y.tolist() == g["y"]  # every step is exact for this example


def test_q8_hand_example_tells_row_from_column_quantisation_of_h():
    # the planted mistake: h quantised per column instead of per routing row
    g = _gold("q8_example.json")
    h = np.array(g["h"], dtype=np.float32)
    qh_col, sh_col = O.quantize_cols(h)
    qd = np.array(g["qd"], dtype=np.float64)
    y_col = (qh_col.astype(np.float64) * sh_col.astype(np.float64)[None, :]) @ qd * g["weight_scale_d"]
    assert sh_col.tolist() != g["h_scales"]
    assert np.abs(y_col - np.array(g["y"])).max() > 1.0


def test_grouped_q8_ffn_hand_example():
    # two experts: expert 0 is the hand-worked one, expert 1 the same with Wd doubled (same codes,
    # doubled down scales, so exactly twice its y); token 0 -> [1, 0], token 1 -> [0, 1]
    g = _gold("q8_example.json")
    H, I, k = g["H"], g["I"], 2
    qslabs = [O.quantize_slab(_q8_hand_slab(g, f), H, I) for f in (1.0, 2.0)]
    ids = np.array([[1, 0], [0, 1]], dtype=np.int32)
    count, offset, rows, pos = O.permute(ids, 2)
    assert rows.tolist() == [1, 2, 0, 3]
    y = O.expert_ffn_q8(np.array(g["x"], dtype=np.float32), rows, offset, k, qslabs, H, I)
    want = np.array(g["y"], dtype=np.float32)
    for t in range(2):
        for j in range(k):
            assert y[pos[t * k + j]].tolist() == (want[t] * (1 + ids[t, j])).tolist()
    left_out = O.expert_ffn_q8(np.array(g["x"], dtype=np.float32), rows, offset, k, qslabs, H, I, experts={0})
    assert np.isnan(left_out[offset[1]:offset[2]]).all() and not np.isnan(left_out[offset[0]:offset[1]]).any()


def test_layer_forward_quant_hand_example():
    # a zero router gives equal logits: ties pick [0, 1] and the weights are 1/2 each, so
    # out[t] = y0[t] / 2 + y1[t] / 2 = 1.5 y[t] exactly
    g = _gold("q8_example.json")
    H, I = g["H"], g["I"]
    qslabs = [O.quantize_slab(_q8_hand_slab(g, f), H, I) for f in (1.0, 2.0)]
    res = O.layer_forward(np.array(g["x"], dtype=np.float32), np.zeros((H, 2), dtype=np.float32), qslabs, H, I, 2,
                          O.RESIDENT, quant=True)
    assert res["ids"].tolist() == [[0, 1], [0, 1]] and res["w"].tolist() == [[0.5, 0.5], [0.5, 0.5]]
    assert res["out"].tolist() == (1.5 * np.array(g["y"], dtype=np.float64)).tolist()


def test_layer_forward_quant_equals_per_routing_experts_combined_by_hand():
    cfg = C.TINY
    rng = np.random.default_rng(21)
    H, I, E, k, T = cfg.H, cfg.I, cfg.E, cfg.k, cfg.T
    x = _bf16(rng.standard_normal((T, H)))
    wr = _bf16(rng.standard_normal((H, E)) * 0.02)
    qslabs = [O.quantize_slab(_bf16(rng.standard_normal(3 * H * I) * 0.02), H, I) for _ in range(E)]
    res = O.layer_forward(x, wr, qslabs, H, I, k, O.RESIDENT, quant=True)
    want = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            # per-row activation scales: one routing row alone gives the same codes as inside its group
            y = O.swiglu_expert_q8(x[t:t + 1], qslabs[int(res["ids"][t, j])], H, I)[0]
            want[t] += res["w"][t, j] * y.astype(np.float64)
    assert np.array_equal(res["out"], want)


def test_window_count_golden():
    g = _gold("window_count.json")
    counts = np.array(g["counts_before"], dtype=np.int64)
    O.window_count(counts, np.array(g["ids"], dtype=np.int32))
    assert counts.tolist() == g["counts_after"]
    # the window count is a histogram of the routings: adding traces in pieces gives the same counts
    rng = np.random.default_rng(22)
    ids = rng.integers(0, 7, size=(9, 3))
    a = np.zeros(7, dtype=np.int64)
    for t in range(9):
        O.window_count(a, ids[t:t + 1])
    assert a.tolist() == np.bincount(ids.reshape(-1), minlength=7).tolist()
