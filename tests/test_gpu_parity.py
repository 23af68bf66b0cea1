"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Integer results (ids, groups, cache state, miss lists, gathered bytes) must
match bit for bit; floating outputs within max-abs 2e-2 and relative L2 1e-2
(bf16 outputs), relative L2 1e-5 (fp32 intermediates) or 5e-3 (y from a path
that hands h to the down projection in bf16).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
from harness import configs as C
from tests._setup import ATOL_OUT, RL2_Y_BF16_H, HostSlabs, assert_f32_close, assert_out_close, rel_l2, stage_layer

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import expert_slot_cache_gb300 as M

GOLD = os.path.join(os.path.dirname(__file__), "golden")
DEV = "cuda"


def _np(t):
    return t.detach().cpu().numpy()


# ----------------------------------------------------------------------------
# Bias table and routing
# ----------------------------------------------------------------------------

def test_bias_table_bit_exact():
    for cfg, cap in [(C.FLASH, -1.0), (C.FLASH, -0.25), (C.FLASH, 0.0), (C.STACK.with_(n_hot=144, zipf_s=1.1), -0.5)]:
        b, _ = C.draw_brightness(cfg)
        got = M.bias_table(torch.from_numpy(b).to(DEV), cfg.n_hot, cap)
        want = O.bias_table(b, cfg.n_hot, cap)
        assert np.array_equal(_np(got), want)
    g = json.load(open(os.path.join(GOLD, "bias_table.json")))
    b = np.array(g["b"], dtype=np.float32)
    got = M.bias_table(torch.from_numpy(b).to(DEV), g["n_hot"], g["cap"])
    assert np.allclose(_np(got), g["bias"], atol=1e-6)


ROUTE_CASES = [
    ("tiny", C.TINY, None, False),
    ("qwen_T1", C.qwen(1), None, False),
    ("qwen_T8", C.qwen(8), None, False),
    ("qwen_T37_ragged", C.qwen(37), None, False),
    ("qwen_T64", C.qwen(64), None, False),
    ("flash_T16_bias", C.FLASH, -1.0, False),
    ("stack_T32_E288", C.STACK, None, False),
    ("prefill_T4096_offset", C.PREFILL, None, True),
    # enough tokens for the (64 tokens x 64 experts x 128 rows) tile path: ragged token and expert tiles
    ("qwen_T300_tiles", C.qwen(300), None, False),
    ("stack_T200_E288_tiles", C.STACK.with_(T=200), None, False),
    # enough tokens for the (64 tokens x 64 experts) tiles over all of H: ragged token and expert tiles,
    # and a ragged last 128-row block
    ("stack_T2500_E288_full", C.STACK.with_(T=2500), None, False),
    ("qwen_T2600_H1000_full", C.qwen(2600).with_(H=1000, logit_offset=True), None, True),
]


@pytest.mark.parametrize("blocked", [True, False], ids=["block_ctas", "ring"])
@pytest.mark.parametrize("name,cfg,cap,offset", ROUTE_CASES, ids=[c[0] for c in ROUTE_CASES])
def test_route_parity(name, cfg, cap, offset, blocked):
    x = C.draw_x(cfg, DEV)
    wr = C.draw_router(cfg, DEV)
    off = C.draw_logit_offset(cfg, DEV) if offset else None
    bias_np = bias_d = None
    if cap is not None:
        b, _ = C.draw_brightness(cfg)
        bias_np = O.bias_table(b, cfg.n_hot, cap)
        bias_d = M.bias_table(torch.from_numpy(b).to(DEV), cfg.n_hot, cap)
    ids, w, logits = M.route(x, wr, cfg.k, off, bias_d, return_logits=True, blocked=blocked)
    torch.cuda.synchronize()
    want_logits = O.router_logits(_np(x.float()), _np(wr.float()), None if off is None else _np(off))
    assert np.array_equal(_np(logits), want_logits), "logits differ"
    want_ids = O.select_topk(want_logits, cfg.k, bias_np)
    assert np.array_equal(_np(ids), want_ids), "ids differ"
    want_w = O.route_weights(want_logits, want_ids)
    assert np.abs(_np(w) - want_w).max() <= 1e-6
    if cap is not None:  # the bias moved some picks, and the weights stay the router's own
        assert not np.array_equal(want_ids, O.select_topk(want_logits, cfg.k))


# ----------------------------------------------------------------------------
# Permute
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("chunked", [True, False], ids=["chunked", "one_cta"])
@pytest.mark.parametrize("n,E", [(1, 16), (7, 5), (64, 128), (640, 512), (1024, 128), (1025, 16), (3001, 288),
                                 (32768, 128)])
def test_permute_parity(n, E, chunked):
    rng = np.random.default_rng(n * 7 + E)
    ids = rng.integers(0, E, size=n).astype(np.int32)
    g = M.permute(torch.from_numpy(ids).to(DEV), E, chunked=chunked)
    torch.cuda.synchronize()
    count, offset, rows, pos = O.permute(ids.reshape(1, -1), E)
    assert np.array_equal(_np(g.count), count)
    assert np.array_equal(_np(g.offset), offset)
    assert np.array_equal(_np(g.rows), rows)
    assert np.array_equal(_np(g.pos), pos)
    act = np.nonzero(count)[0]
    assert int(_np(g.n_act)[0]) == len(act)
    assert np.array_equal(_np(g.act_e)[: len(act)], act)


def test_permute_flags_bad_ids():
    ids = torch.tensor([0, 3, 9, 1], dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    g = M.permute(ids, 4, dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 1
    assert _np(g.offset)[4] == 3 and _np(g.pos)[2] == -1


# ----------------------------------------------------------------------------
# Manage / gather
# ----------------------------------------------------------------------------

def _check_state(gs, os_, what):
    assert _np(gs.e2s).tolist() == os_.e2s.tolist(), f"{what}: e2s"
    assert _np(gs.s2e).tolist() == os_.s2e.tolist(), f"{what}: s2e"
    assert (_np(gs.prio).astype(np.uint32)).tolist() == os_.prio.tolist(), f"{what}: prio"
    assert int(_np(gs.stamp)[0]) == os_.stamp, f"{what}: stamp"


def _check_manage(mo, r, what):
    nm = int(_np(mo.n_miss)[0])
    nh = int(_np(mo.n_hit)[0])
    assert _np(mo.miss_e)[:nm].tolist() == r.miss_e, f"{what}: miss_e"
    assert _np(mo.miss_s)[:nm].tolist() == r.miss_s, f"{what}: miss_s"
    assert _np(mo.hit_e)[:nh].tolist() == r.hit_e, f"{what}: hit_e"
    assert np.array_equal(_np(mo.sid), r.sid), f"{what}: sid"


def test_manage_golden_traces_on_gpu():
    g = json.load(open(os.path.join(GOLD, "manage_traces.json")))
    for tr in g["traces"]:
        st = M.CacheState.from_slots(tr["s2e0"], tr["E"])
        for i, step in enumerate(tr["steps"]):
            ids = torch.tensor(step["ids"], dtype=torch.int32, device=DEV)
            mo = M.cache_manage(ids, st, tr["policy"])
            torch.cuda.synchronize()
            nm = int(_np(mo.n_miss)[0])
            assert _np(mo.miss_e)[:nm].tolist() == step["miss_e"], (tr["name"], i)
            assert _np(mo.miss_s)[:nm].tolist() == step["miss_s"], (tr["name"], i)
            assert _np(mo.sid).tolist() == step["sid"], (tr["name"], i)
            assert _np(st.s2e).tolist() == step["s2e"], (tr["name"], i)
            assert _np(st.e2s).tolist() == step["e2s"], (tr["name"], i)
            assert _np(st.prio).tolist() == step["prio"], (tr["name"], i)


def _zipf_trace(rng, steps, T, k, E, s=1.1):
    p = np.arange(1, E + 1, dtype=np.float64) ** -s
    p /= p.sum()
    perm = rng.permutation(E)
    return [np.stack([perm[rng.choice(E, k, replace=False, p=p)] for _ in range(T)]).astype(np.int32)
            for _ in range(steps)]


@pytest.mark.parametrize("policy", [0, 1, 2], ids=["lru", "lfu", "static"])
@pytest.mark.parametrize("E,S,T,k,dist", [(128, 64, 8, 8, "uniform"), (128, 64, 8, 8, "zipf"),
                                          (512, 192, 16, 10, "zipf"), (288, 144, 18, 8, "uniform"),
                                          (16, 16, 4, 2, "uniform")])
def test_manage_parity_every_step(policy, E, S, T, k, dist):
    rng = np.random.default_rng(E + S + policy)
    if dist == "zipf":
        trace = _zipf_trace(rng, 40, T, k, E)
    else:
        trace = [np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32) for _ in range(40)]
    s2e0 = C.initial_residency(C.TINY.with_(E=E, S=S, seed=E))
    ost = O.CacheState.from_slots(s2e0, E)
    gst = M.CacheState.from_slots(s2e0, E)
    for i, ids in enumerate(trace):
        mo = M.cache_manage(torch.from_numpy(ids).to(DEV), gst, policy)
        torch.cuda.synchronize()
        r = O.manage(ost, ids, policy)
        _check_manage(mo, r, f"step {i}")
        _check_state(gst, ost, f"step {i}")


def test_manage_capacity_error():
    st = M.CacheState.from_slots(np.arange(4), 8)
    ids = torch.arange(5, dtype=torch.int32, device=DEV)
    with pytest.raises(M.MoeError) as ei:
        M.cache_manage(ids, st, 0)
    assert ei.value.code == -2


def test_gather_bytes():
    E, S, n = 12, 5, 4099 * 8  # slab not a multiple of the 32 KB chunk
    rng = np.random.default_rng(5)
    host = torch.from_numpy(rng.integers(-2 ** 15, 2 ** 15, size=(E, n), dtype=np.int16)).pin_memory()
    pool = torch.zeros(S, n, dtype=torch.int16, device=DEV)
    miss_e = torch.tensor([7, 2, 11, 0], dtype=torch.int32, device=DEV)
    miss_s = torch.tensor([3, 0, 4, 1], dtype=torch.int32, device=DEV)
    n_miss = torch.tensor([3], dtype=torch.int32, device=DEV)  # the 4th entry is not copied
    M.cache_gather(host, pool, miss_e, miss_s, n_miss, 4)
    torch.cuda.synchronize()
    p = _np(pool)
    assert np.array_equal(p[3], host[7].numpy()) and np.array_equal(p[0], host[2].numpy())
    assert np.array_equal(p[4], host[11].numpy())
    assert not p[1].any() and not p[2].any()


def test_gather_rejects_unpinned_host():
    host = torch.zeros(2, 64, dtype=torch.int16)
    pool = torch.zeros(2, 64, dtype=torch.int16, device=DEV)
    z = torch.zeros(2, dtype=torch.int32, device=DEV)
    with pytest.raises(M.MoeError) as ei:
        M.cache_gather(host, pool, z, z, z[:1], 2)
    assert ei.value.code == -4


# ----------------------------------------------------------------------------
# Expert FFN and combine
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("cfg,T", [(C.TINY, 4), (C.qwen(8), 8), (C.qwen(64), 64), (C.FLASH, 16)],
                         ids=["tiny", "qwen_T8", "qwen_T64", "flash_T16"])
def test_expert_ffn_parity(cfg, T):
    rng = np.random.default_rng(T)
    E = cfg.E
    # a skewed routing so groups span 1..many tokens (batches of 1, 2, 4, 8 and more)
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.2
    p /= p.sum()
    ids = np.stack([rng.choice(E, cfg.k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    count, offset, rows, pos = O.permute(ids, E)
    x = C.draw_x(cfg, DEV, T=T)
    host = torch.empty(E, cfg.slab_elems, dtype=torch.bfloat16, pin_memory=True)
    used = np.nonzero(count)[0]
    for e in used:
        host[e].copy_(C.draw_slab(cfg, int(e), DEV))
    # half the used experts in slots (pool), the rest read straight from the host store
    S = max(1, len(used) // 2)
    pool = torch.empty(S, cfg.slab_elems, dtype=torch.bfloat16, device=DEV)
    e2s = np.full(E, -1, dtype=np.int32)
    for s, e in enumerate(used[:S]):
        e2s[e] = s
        pool[s].copy_(host[e])
    lst = torch.from_numpy(used.astype(np.int32)).to(DEV)
    g = M.permute(torch.from_numpy(ids).to(DEV), E)
    y = M.expert_ffn(x, cfg.k, cfg.I, E, g.offset, g.rows, lst, torch.tensor([len(used)], dtype=torch.int32,
                     device=DEV), len(used), pool, torch.from_numpy(e2s).to(DEV), host)
    torch.cuda.synchronize()
    want = O.expert_ffn(_np(x.float()), rows, offset, cfg.k, HostSlabs(host), cfg.H, cfg.I)
    assert_f32_close(_np(y), want, "y")




STREAM_CASES = [
    ("tiny_T4", C.TINY, 4, 1.2),
    ("qwen_T1", C.qwen(1), 1, 1.2),
    ("qwen_T8", C.qwen(8), 8, 1.2),
    ("qwen_T37_uniform", C.qwen(37), 37, 0.0),
    ("qwen_T64_skewed", C.qwen(64), 64, 1.2),
    ("qwen_T64_same8", C.qwen(64), 64, None),
    ("flash_T16", C.FLASH, 16, 1.1),
    ("stack_T32", C.STACK, 32, 1.2),
]


@pytest.mark.parametrize("name,cfg,T,skew", STREAM_CASES, ids=[c[0] for c in STREAM_CASES])
def test_expert_ffn_stream_parity(name, cfg, T, skew):
    """Decode-sized groups with every listed expert in a VRAM slot (the stream
    path over full weight rows).  Slots are assigned in reverse so the slot
    remap is exercised; groups span 1..T tokens (several token batches per
    expert); "same8" routes every token to experts 0..7, so few experts carry
    all the rows and the parts-per-expert cap limits the CTAs used."""
    rng = np.random.default_rng(T + 17)
    E = cfg.E
    if skew is None:
        ids = np.tile(np.arange(cfg.k, dtype=np.int32), (T, 1))
        for t in range(T):
            rng.shuffle(ids[t])
    else:
        p = np.arange(1, E + 1, dtype=np.float64) ** -skew
        p /= p.sum()
        ids = np.stack([rng.choice(E, cfg.k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    count, offset, rows, pos = O.permute(ids, E)
    x = C.draw_x(cfg, DEV, T=T)
    used = np.nonzero(count)[0]
    S = len(used)
    host = torch.empty(E, cfg.slab_elems, dtype=torch.bfloat16, pin_memory=True)
    pool = torch.empty(S, cfg.slab_elems, dtype=torch.bfloat16, device=DEV)
    e2s = np.full(E, -1, dtype=np.int32)
    for i, e in enumerate(used):
        sl = S - 1 - i
        e2s[e] = sl
        pool[sl].copy_(C.draw_slab(cfg, int(e), DEV))
        host[e].copy_(pool[sl])
    lst = torch.from_numpy(used.astype(np.int32)).to(DEV)
    g = M.permute(torch.from_numpy(ids).to(DEV), E)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = M.expert_ffn(x, cfg.k, cfg.I, E, g.offset, g.rows, lst, torch.tensor([S], dtype=torch.int32, device=DEV),
                     S, pool, torch.from_numpy(e2s).to(DEV), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want = O.expert_ffn(_np(x.float()), rows, offset, cfg.k, HostSlabs(host), cfg.H, cfg.I)
    # the down projection reads h in bf16 (as the tensor-core prefill path does)
    got = _np(y)
    assert rel_l2(got, want) <= RL2_Y_BF16_H
    for e in used:
        a, b = offset[e], offset[e + 1]
        assert rel_l2(got[a:b], want[a:b]) <= 2 * RL2_Y_BF16_H, f"expert {e} ({b - a} rows)"


def test_combine_parity_split():
    rng = np.random.default_rng(3)
    T, k, H, E = 5, 3, 128, 9
    y = rng.normal(size=(T * k, H)).astype(np.float32)
    w = rng.random((T, k)).astype(np.float32)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    pos = rng.permutation(T * k).astype(np.int32)
    e2s = np.where(rng.random(E) < 0.5, -1, np.arange(E)).astype(np.int32)
    t = lambda a: torch.from_numpy(a).to(DEV)
    out = M.combine(t(y), t(w), t(pos), T, k, E)
    out_s, res, miss = M.combine(t(y), t(w), t(pos), T, k, E, ids=t(ids), e2s=t(e2s), split=True)
    torch.cuda.synchronize()
    want = O.combine(y, w, pos, T, k)
    wo, wr_, wm = O.combine(y, w, pos, T, k, resident=e2s[ids] >= 0)
    assert_out_close(_np(out.float()), want)
    assert_out_close(_np(out_s.float()), wo)
    assert_f32_close(_np(res), wr_, "out_res")
    assert_f32_close(_np(miss), wm, "out_miss")


# ----------------------------------------------------------------------------
# Whole layer
# ----------------------------------------------------------------------------

def _run_layer(cfg, steps=1, side=True, policy=None, T=None, bias_mode=O.BIAS_GRADED, rflags=0, schedule=None,
               decode_kernels=0):
    T = cfg.T if T is None else T
    policy = cfg.policy if policy is None else policy
    schedule = cfg.schedule if schedule is None else schedule
    st = stage_layer(cfg)
    bias_np = bias_d = None
    if cfg.bias_cap is not None:
        b, _ = C.draw_brightness(cfg)
        bias_np = O.bias_table(b, cfg.n_hot, cfg.bias_cap, bias_mode)
        bias_d = M.bias_table(torch.from_numpy(b).to(DEV), cfg.n_hot, cfg.bias_cap, mode=bias_mode)
    router = O.ROUTER_SIGMOID if rflags & M.ROUTE_SIGMOID else O.ROUTER_SOFTMAX
    damped = bool(rflags & M.ROUTE_DAMPED)
    s2e0 = C.initial_residency(cfg)
    if cfg.mode == C.MODE_RESIDENT:
        pool, gstate, ostate, opool = st["slabs_dev"], None, None, None
    else:
        pool = torch.empty(cfg.S, cfg.slab_elems, dtype=torch.bfloat16, device=DEV)
        for s, e in enumerate(s2e0):
            if e >= 0:
                pool[s].copy_(st["slabs_dev"][e])
        gstate = M.CacheState.from_slots(s2e0, cfg.E)
        ostate = O.CacheState.from_slots(s2e0, cfg.E)
        opool = None
    layer = M.SlotCachedMoELayer(st["wr"], pool, cfg.k, cfg.I, cfg.mode, policy,
                                 host_slabs=None if cfg.mode == C.MODE_RESIDENT else st["host"], state=gstate,
                                 logit_offset=st["logit_offset"], sel_bias=bias_d, max_tokens=T, side_stream=side,
                                 route_flags=rflags, schedule=schedule, decode_kernels=decode_kernels)
    wr_np = _np(st["wr"].float())
    off_np = None if st["logit_offset"] is None else _np(st["logit_offset"])
    slabs = HostSlabs(st["host"])
    total_miss = total_calls = 0
    for step in range(steps):
        x = C.draw_x(cfg, DEV, step=step, T=T)
        res = layer.forward(x)
        torch.cuda.synchronize()
        want = O.layer_forward(_np(x.float()), wr_np, slabs, cfg.H, cfg.I, cfg.k, cfg.mode, policy, ostate,
                               opool, off_np, bias_np, router=router, damped=damped, schedule=schedule)
        assert np.array_equal(_np(res["ids"]), want["ids"]), f"step {step}: ids"
        assert np.abs(_np(res["w"]) - want["w"]).max() <= 1e-6
        assert_out_close(_np(res["out"].float()), want["out"], f"step {step}: out")
        if cfg.mode == C.MODE_ZERO_RETURN:
            # resident experts run the stream path (bf16 h); missing ones read host memory in fp32
            assert rel_l2(_np(res["out_res"]), want["out_res"]) <= RL2_Y_BF16_H
            assert_f32_close(_np(res["out_miss"]), want["out_miss"], "out_miss")
            if bias_mode != O.BIAS_HARD:
                assert np.abs(want["out_miss"]).max() > 0
        if ostate is not None:
            _check_state(gstate, ostate, f"step {step}")
            total_miss += sum(len(c["miss_e"]) for c in want["chunks"])
            total_calls += sum(len(c.get("waves", [None])) for c in want["chunks"])
    assert int(_np(layer.dev_status)[0]) == 0
    if ostate is not None:
        stats = _np(layer.stats)
        assert stats[0] == total_miss
        assert stats[1] == total_calls  # manage calls (an empty wave is no call)
        if cfg.mode == C.MODE_GATHER:
            assert stats[2] == total_miss * cfg.slab_bytes
            # every occupied slot holds exactly its expert's bytes
            s2e = _np(gstate.s2e)
            for s, e in enumerate(s2e):
                assert torch.equal(pool[s].cpu(), st["host"][e]), f"slot {s}"
    return layer


def test_layer_tiny_resident():
    _run_layer(C.TINY, steps=2)


def test_layer_largest_expert_count_and_top_k():
    """The largest shapes the library takes: E = 1024 experts and top-16, all resident."""
    _run_layer(C.TINY.with_(E=1024, k=16, S=1024, T=6), steps=2)


def test_layer_top_k_equals_expert_count():
    """Degenerate routing: every token picks every expert (k = E), so top-k is a full sort and each
    expert's group holds every token."""
    _run_layer(C.TINY.with_(E=16, k=16, S=16, T=5), steps=2)


def test_layer_gather_one_token_per_chunk():
    """A pool exactly k slots deep: every chunk is one token (floor(S / k) = 1), each managing,
    gathering and computing on its own; 1024 experts, top-16."""
    _run_layer(C.TINY.with_(E=1024, k=16, S=16, T=3, mode=C.MODE_GATHER), steps=2)


@pytest.mark.parametrize("T", [1, 8, 32, 64])
def test_layer_qwen_gather_lru(T):
    _run_layer(C.qwen(T), steps=2)


def test_layer_qwen_gather_lfu_single_stream():
    _run_layer(C.qwen(8, policy=C.POLICY_LFU), steps=3, side=False)


def test_layer_qwen_all_resident():
    _run_layer(C.qwen(64, S=128, mode=C.MODE_RESIDENT), steps=1)


def test_layer_flash_zero_return():
    _run_layer(C.FLASH, steps=2)


def test_layer_stack_shape_all_resident():
    # 288 experts, all in the pool, T=32: up to 256 listed experts in one stream pass
    _run_layer(C.STACK, steps=2)


def test_layer_stack_shape_all_resident_174_experts():
    """Layer 24 of the stack, steps 0 and 1 (the second routes to 174 experts):
    the stream FFN must see the permute's complete lists (programmatic
    dependent launches along the layer)."""
    cfg = C.STACK
    l = 24
    wr = C.draw_router(cfg, DEV, l)
    slabs = torch.empty(cfg.E, cfg.slab_elems, dtype=torch.bfloat16, device=DEV)
    C.draw_slabs(cfg, DEV, l, out=slabs)
    layer = M.SlotCachedMoELayer(wr, slabs, cfg.k, cfg.I, cfg.mode, cfg.policy, max_tokens=cfg.T)
    wr_np = _np(wr.float())
    slabs_h = HostSlabs(slabs.cpu())
    for st in range(2):
        x = C.draw_x(cfg, DEV, layer=l, step=st)
        res = layer.forward(x)
        torch.cuda.synchronize()
        assert int(_np(layer.dev_status)[0]) == 0, f"step {st}"
        want = O.layer_forward(_np(x.float()), wr_np, slabs_h, cfg.H, cfg.I, cfg.k, cfg.mode, cfg.policy)
        assert np.array_equal(_np(res["ids"]), want["ids"]), f"step {st}: ids"
        assert_out_close(_np(res["out"].float()), want["out"], f"step {st}: out")
    assert len(np.unique(_np(res["ids"]))) == 174


def test_layer_stack_shape_gather_chunked():
    _run_layer(C.STACK_SLOTS, steps=2)


def test_layer_prefill_sampled_tokens():
    cfg = C.PREFILL
    st = stage_layer(cfg)
    layer = M.SlotCachedMoELayer(st["wr"], st["slabs_dev"], cfg.k, cfg.I, cfg.mode, max_tokens=cfg.T,
                                 logit_offset=st["logit_offset"])
    x = C.draw_x(cfg, DEV)
    res = layer.forward(x)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    tok = np.sort(rng.choice(cfg.T, 48, replace=False))
    tok[-1] = cfg.T - 1
    xs = _np(x.float())[tok]
    want = O.layer_forward(xs, _np(st["wr"].float()), HostSlabs(st["host"]), cfg.H, cfg.I, cfg.k, cfg.mode,
                           logit_offset=_np(st["logit_offset"]))
    assert np.array_equal(_np(res["ids"])[tok], want["ids"])
    assert_out_close(_np(res["out"].float())[tok], want["out"])
    # groups are uneven under the logit offset
    counts = np.bincount(_np(res["ids"]).ravel(), minlength=cfg.E)
    assert counts.max() > 2 * counts.mean()




@pytest.mark.parametrize("T,skew", [(512, 1.2), (520, 0.0)], ids=["T512_skewed", "T520_uniform_ragged"])
def test_expert_ffn_tensor_core_parity(T, skew):
    """Groups large enough for the tcgen05 grouped GEMMs (T*k >= 4096)."""
    cfg = C.qwen(T, S=128, mode=C.MODE_RESIDENT)
    E = cfg.E
    rng = np.random.default_rng(T)
    p = np.arange(1, E + 1, dtype=np.float64) ** -skew
    p /= p.sum()
    ids = np.stack([rng.choice(E, cfg.k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    count, offset, rows, pos = O.permute(ids, E)
    x = C.draw_x(cfg, DEV, T=T)
    st = stage_layer(cfg)
    used = np.nonzero(count)[0]
    lst = torch.from_numpy(used.astype(np.int32)).to(DEV)
    g = M.permute(torch.from_numpy(ids).to(DEV), E)
    y = M.expert_ffn(x, cfg.k, cfg.I, E, g.offset, g.rows, lst, torch.tensor([len(used)], dtype=torch.int32,
                     device=DEV), len(used), st["slabs_dev"])
    torch.cuda.synchronize()
    want = O.expert_ffn(_np(x.float()), rows, offset, cfg.k, HostSlabs(st["host"]), cfg.H, cfg.I)
    got = _np(y)
    assert rel_l2(got, want) <= RL2_Y_BF16_H
    # every group, including ragged last tiles and single-row groups, is right
    for e in used:
        a, b = offset[e], offset[e + 1]
        assert rel_l2(got[a:b], want[a:b]) <= 2 * RL2_Y_BF16_H, f"expert {e} ({b - a} rows)"


def test_expert_ffn_tensor_core_tile_edges():
    """Group sizes on the grouped GEMMs' tile edges: 1 row, N rounding to 16
    (15, 16, 17), one or two 128-row boxes per tile (127, 128, 129), one or
    two 256-row tiles (255, 256, 257), several tiles (511 .. 513)."""
    cfg = C.qwen(560, S=128, mode=C.MODE_RESIDENT)
    T, E, k = cfg.T, cfg.E, cfg.k
    edges = [1, 15, 16, 17, 31, 33, 127, 128, 129, 255, 256, 257, 511, 512, 513]
    rng = np.random.default_rng(11)
    counts = np.zeros(E, dtype=np.int64)
    perm = rng.permutation(E)
    counts[perm[:len(edges)]] = edges
    rest = perm[len(edges):len(edges) + 60]  # the other experts stay empty
    left = T * k - counts.sum()
    counts[rest] = left // len(rest)
    counts[rest[: left % len(rest)]] += 1
    assert counts.sum() == T * k and counts.max() <= T
    # expert-sorted list dealt column-wise: token t takes entries t, T + t, ... (distinct experts, as every run <= T)
    lst = np.repeat(np.arange(E, dtype=np.int32), counts)
    ids = np.ascontiguousarray(lst.reshape(k, T).T)
    assert all(len(set(r)) == k for r in ids)
    count, offset, rows, pos = O.permute(ids, E)
    assert np.array_equal(count, counts)
    x = C.draw_x(cfg, DEV, T=T)
    st = stage_layer(cfg)
    used = np.nonzero(count)[0]
    g = M.permute(torch.from_numpy(ids).to(DEV), E)
    y = M.expert_ffn(x, k, cfg.I, E, g.offset, g.rows, torch.from_numpy(used.astype(np.int32)).to(DEV),
                     torch.tensor([len(used)], dtype=torch.int32, device=DEV), len(used), st["slabs_dev"])
    torch.cuda.synchronize()
    want = O.expert_ffn(_np(x.float()), rows, offset, k, HostSlabs(st["host"]), cfg.H, cfg.I)
    got = _np(y)
    for e in used:
        a, b = offset[e], offset[e + 1]
        assert rel_l2(got[a:b], want[a:b]) <= 2 * RL2_Y_BF16_H, f"expert {e} ({b - a} rows)"
        assert np.abs(got[a:b] - want[a:b]).max() <= ATOL_OUT, f"expert {e} ({b - a} rows)"


# ----------------------------------------------------------------------------
# Live-cache affinity ("Nudge, don't cut", "Then Maya's own knob beat ours")
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("blocked", [True, False], ids=["block_ctas", "ring"])
def test_route_affinity_parity(blocked):
    cfg = C.qwen(16)
    x = C.draw_x(cfg, DEV)
    wr = C.draw_router(cfg, DEV)
    e2s = np.full(cfg.E, -1, dtype=np.int32)
    s2e = C.initial_residency(cfg)
    e2s[s2e] = np.arange(cfg.S, dtype=np.int32)
    ids, w, logits = M.route(x, wr, cfg.k, return_logits=True, blocked=blocked,
                             e2s=torch.from_numpy(e2s).to(DEV), affinity=0.3)
    torch.cuda.synchronize()
    want_logits = O.router_logits(_np(x.float()), _np(wr.float()))
    want = O.select_topk(want_logits, cfg.k, resident=e2s >= 0, affinity=0.3)
    assert np.array_equal(_np(ids), want)
    assert not np.array_equal(want, O.select_topk(want_logits, cfg.k))
    assert np.abs(_np(w) - O.route_weights(want_logits, want)).max() <= 1e-6


def test_layer_gather_with_affinity_matches_oracle_and_misses_less():
    cfg = C.qwen(8)
    st = stage_layer(cfg)
    s2e0 = C.initial_residency(cfg)
    res = {}
    for lam in (0.0, 0.5):
        pool = st["slabs_dev"][torch.from_numpy(s2e0.astype(np.int64)).to(DEV)].contiguous()
        gstate = M.CacheState.from_slots(s2e0, cfg.E)
        ostate = O.CacheState.from_slots(s2e0, cfg.E)
        layer = M.SlotCachedMoELayer(st["wr"], pool, cfg.k, cfg.I, cfg.mode, cfg.policy, host_slabs=st["host"],
                                     state=gstate, max_tokens=cfg.T, affinity=lam)
        misses = 0
        for step in range(4):
            x = C.draw_x(cfg, DEV, step=step)
            r = layer.forward(x)
            torch.cuda.synchronize()
            want = O.layer_forward(_np(x.float()), _np(st["wr"].float()), HostSlabs(st["host"]), cfg.H, cfg.I, cfg.k,
                                   cfg.mode, cfg.policy, ostate, affinity=lam)
            assert np.array_equal(_np(r["ids"]), want["ids"]), (lam, step)
            assert_out_close(_np(r["out"].float()), want["out"], f"affinity {lam} step {step}")
            _check_state(gstate, ostate, f"affinity {lam} step {step}")
            misses += sum(len(c["miss_e"]) for c in want["chunks"])
        assert int(layer.stats[0]) == misses
        res[lam] = misses
    assert res[0.5] < res[0.0]


# ----------------------------------------------------------------------------
# Routing variants ("Nudge, don't cut": hard mask, flat bias, damped weights,
# GLM's sigmoid router)
# ----------------------------------------------------------------------------

def test_bias_table_modes_bit_exact():
    cfg = C.FLASH
    b, _ = C.draw_brightness(cfg)
    bd = torch.from_numpy(b).to(DEV)
    for mode, val in ((O.BIAS_GRADED, -1.0), (O.BIAS_FLAT, -0.5), (O.BIAS_HARD, 0.0)):
        got = _np(M.bias_table(bd, cfg.n_hot, val, mode=mode))
        want = O.bias_table(b, cfg.n_hot, val, mode)
        assert np.array_equal(got, want), mode
    assert np.isneginf(_np(M.bias_table(bd, cfg.n_hot, 0.0, mode=O.BIAS_HARD))).sum() == cfg.E - cfg.n_hot


ROUTE_VARIANT_CASES = [
    ("flash_flat", C.FLASH, O.BIAS_FLAT, -0.5, 0),
    ("flash_hard_mask", C.FLASH, O.BIAS_HARD, 0.0, 0),
    ("flash_damped", C.FLASH, O.BIAS_GRADED, -1.0, 2),
    ("glm_stack_sigmoid_graded", C.STACK.with_(n_hot=144, zipf_s=1.1), O.BIAS_GRADED, -0.25, 1),
    ("qwen_T300_sigmoid_flat_tiles", C.qwen(300).with_(n_hot=64, zipf_s=1.1), O.BIAS_FLAT, -0.05, 1),
    ("prefill_sigmoid_offset", C.PREFILL, None, None, 1),
]


@pytest.mark.parametrize("blocked", [True, False], ids=["block_ctas", "ring"])
@pytest.mark.parametrize("name,cfg,mode,val,rflags", ROUTE_VARIANT_CASES, ids=[c[0] for c in ROUTE_VARIANT_CASES])
def test_route_variant_parity(name, cfg, mode, val, rflags, blocked):
    x = C.draw_x(cfg, DEV)
    wr = C.draw_router(cfg, DEV)
    off = C.draw_logit_offset(cfg, DEV)
    bias_np = bias_d = None
    if mode is not None:
        b, _ = C.draw_brightness(cfg)
        bias_np = O.bias_table(b, cfg.n_hot, val, mode)
        bias_d = M.bias_table(torch.from_numpy(b).to(DEV), cfg.n_hot, val, mode=mode)
    ids, w, logits = M.route(x, wr, cfg.k, off, bias_d, return_logits=True, blocked=blocked, rflags=rflags)
    torch.cuda.synchronize()
    want_logits = O.router_logits(_np(x.float()), _np(wr.float()), None if off is None else _np(off))
    assert np.array_equal(_np(logits), want_logits), "logits differ"
    router = O.ROUTER_SIGMOID if rflags & 1 else O.ROUTER_SOFTMAX
    want_ids = O.select_topk(want_logits, cfg.k, bias_np, router=router)
    assert np.array_equal(_np(ids), want_ids), "ids differ"
    want_w = O.route_weights(want_logits, want_ids, router, bias_np, bool(rflags & 2))
    assert np.abs(_np(w) - want_w).max() <= 1e-6
    if mode == O.BIAS_HARD:
        assert np.isfinite(bias_np[want_ids]).all()  # every pick in the hot set
    if rflags & 2:  # damped weights differ from the selection-only ones where a cold expert was picked
        assert np.abs(want_w - O.route_weights(want_logits, want_ids)).max() > 1e-3


def test_route_flags_rejected():
    cfg = C.TINY
    x, wr = C.draw_x(cfg, DEV), C.draw_router(cfg, DEV)
    for bad in (3, 4):
        with pytest.raises(M.MoeError) as ei:
            M.route(x, wr, cfg.k, rflags=bad)
        assert ei.value.code == -1


def test_layer_gather_sigmoid_router_flat_bias():
    _run_layer(C.qwen(8).with_(n_hot=64, bias_cap=-0.05, zipf_s=1.1), steps=2, bias_mode=O.BIAS_FLAT, rflags=M.ROUTE_SIGMOID)


def test_layer_flash_zero_return_damped_weights():
    _run_layer(C.FLASH, steps=1, rflags=M.ROUTE_DAMPED)


def test_layer_flash_zero_return_hard_mask_never_misses():
    layer = _run_layer(C.FLASH, steps=1, bias_mode=O.BIAS_HARD)
    assert int(_np(layer.stats)[0]) == 0  # the hot set is the pool: a hard mask never picks a missing expert
