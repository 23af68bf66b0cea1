"""The allocation-free FFN entry point gives the same result as the workspace one.

moe_expert_ffn_noalloc exists for callers that cannot allocate device memory
where they run the FFN (host callbacks, plug-ins that must not touch their
host's memory pool, runtimes with a frozen allocator): it keeps the FFN's
intermediate activations in a fixed array inside the library.  These tests
call it through the C ABI, twice in a row with different shapes and routings
on the identity slot map, then on a half-sized pool with a seeded slot remap,
with and without experts served from pinned host memory.  Each result is
compared with moe_expert_ffn's on the same inputs (within the error of the
bf16 h that the workspace path's tensor-core down projection reads, or within
fp32 summation error where both keep h in fp32) and with the oracle (the
allocation-free path keeps h in fp32).  They also check that an oversized
request is refused with a clear status and that a slot outside the pool is
flagged, not read.  The file name makes pytest collect it last.
"""
from ctypes import c_int, c_void_p

import numpy as np
import pytest
import torch

from harness import configs as C
import oracle as O
from tests._setup import RL2_F32, RL2_Y_BF16_H, HostSlabs, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc_fn():
    import expert_slot_cache_gb300 as M
    f = M.lib.moe_expert_ffn_noalloc
    V, I = c_void_p, c_int
    f.argtypes = [V, I, I, I, I, I, V, V, V, V, I, V, I, V, V, V, V, V]
    f.restype = c_int
    return f


def _routing(cfg, T, seed):
    rng = np.random.default_rng(seed)
    E = cfg.E
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.1
    p /= p.sum()
    return np.stack([rng.choice(E, cfg.k, replace=False, p=p) for _ in range(T)]).astype(np.int32), rng


def _case(cfg, T, seed):
    import expert_slot_cache_gb300 as M
    ids, _ = _routing(cfg, T, seed)
    used = np.unique(ids)
    x = C.draw_x(cfg, DEV, step=seed, T=T)
    pool = torch.empty(cfg.E, cfg.slab_elems, dtype=torch.bfloat16, device=DEV)
    for e in used:
        pool[e].copy_(C.draw_slab(cfg, int(e), DEV))
    g = M.permute(torch.from_numpy(ids).to(DEV), cfg.E)
    lst = torch.from_numpy(used.astype(np.int32)).to(DEV)
    n_list = torch.tensor([len(used)], dtype=torch.int32, device=DEV)
    return x, pool, g, lst, n_list, len(used)


def _p(t):
    return None if t is None else c_void_p(t.data_ptr())


def _call_noalloc(f, cfg, x, T, g, lst, n_list, n_used, pool, y, status, e2s=None, host=None):
    return f(_p(x), T, cfg.H, cfg.I, cfg.k, cfg.E, _p(g.offset), _p(g.rows), _p(lst), _p(n_list), n_used, _p(pool),
             pool.shape[0], _p(e2s), _p(host), _p(y), _p(status), c_void_p(torch.cuda.current_stream().cuda_stream))


def _oracle_y(x, g, cfg, slabs):
    rows, offset = g.rows.cpu().numpy(), g.offset.cpu().numpy()
    return O.expert_ffn(x.float().cpu().numpy(), rows, offset, cfg.k, HostSlabs(slabs), cfg.H, cfg.I)


def test_noalloc_ffn_matches_workspace_ffn_on_two_calls():
    import expert_slot_cache_gb300 as M
    f = _noalloc_fn()
    for call, (cfg, T) in enumerate([(C.qwen(8), 8), (C.qwen(64), 64)]):
        x, pool, g, lst, n_list, n_used = _case(cfg, T, seed=11 + call)
        y_ref = M.expert_ffn(x, cfg.k, cfg.I, cfg.E, g.offset, g.rows, lst, n_list, n_used, pool)
        y = torch.full((T * cfg.k, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        rc = _call_noalloc(f, cfg, x, T, g, lst, n_list, n_used, pool, y, status)
        assert rc == 0, M.status_str(rc)
        torch.cuda.synchronize()
        assert int(status[0]) == 0
        got, want = y.cpu().numpy(), y_ref.cpu().numpy()
        assert np.isfinite(got).all(), f"call {call}: rows left unwritten"
        assert rel_l2(got, want) <= RL2_Y_BF16_H, f"call {call}"
        assert rel_l2(got, _oracle_y(x, g, cfg, pool.cpu())) <= RL2_F32, f"call {call} vs oracle"


@pytest.mark.parametrize("with_host", [False, True])
def test_noalloc_ffn_on_a_remapped_half_pool(with_host):
    # S = 64 of 128 slots; used experts sit in seeded slots (e2s), and with a host store
    # every third used expert is left out of the pool and read from pinned host memory
    import expert_slot_cache_gb300 as M
    f = _noalloc_fn()
    cfg = C.qwen(8)
    T, S = 8, 64
    ids, rng = _routing(cfg, T, seed=31 + int(with_host))
    used = np.unique(ids)
    assert len(used) <= S
    slabs = torch.empty(cfg.E, cfg.slab_elems, dtype=torch.bfloat16, device=DEV)
    C.draw_slabs(cfg, DEV, out=slabs)
    host = None
    in_pool = used if not with_host else np.array([e for i, e in enumerate(used) if i % 3 != 0])
    if with_host:
        host = torch.empty(cfg.E, cfg.slab_elems, dtype=torch.bfloat16, pin_memory=True)
        host.copy_(slabs)
    e2s_np = np.full(cfg.E, -1, dtype=np.int32)
    e2s_np[in_pool] = rng.permutation(S)[:len(in_pool)]
    pool = torch.zeros(S, cfg.slab_elems, dtype=torch.bfloat16, device=DEV)
    for e in in_pool:
        pool[int(e2s_np[e])].copy_(slabs[int(e)])
    e2s = torch.from_numpy(e2s_np).to(DEV)
    x = C.draw_x(cfg, DEV, step=5, T=T)
    g = M.permute(torch.from_numpy(ids).to(DEV), cfg.E)
    lst = torch.from_numpy(used.astype(np.int32)).to(DEV)
    n_list = torch.tensor([len(used)], dtype=torch.int32, device=DEV)
    y_ref = M.expert_ffn(x, cfg.k, cfg.I, cfg.E, g.offset, g.rows, lst, n_list, len(used), pool, e2s=e2s,
                         host_slabs=host)
    for call in range(2):
        y = torch.full((T * cfg.k, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        rc = _call_noalloc(f, cfg, x, T, g, lst, n_list, len(used), pool, y, status, e2s=e2s, host=host)
        assert rc == 0, M.status_str(rc)
        torch.cuda.synchronize()
        assert int(status[0]) == 0
        got = y.cpu().numpy()
        assert np.isfinite(got).all(), f"call {call}: rows left unwritten"
        # with a host store both entry points run the host-weights kernel (fp32 h) on the same inputs
        tol = RL2_F32 if with_host else RL2_Y_BF16_H
        assert rel_l2(got, y_ref.cpu().numpy()) <= tol, f"call {call}"
        assert rel_l2(got, _oracle_y(x, g, cfg, slabs.cpu())) <= RL2_F32, f"call {call} vs oracle"


def test_noalloc_ffn_flags_a_slot_outside_the_pool():
    # one listed expert is mapped to slot S: the kernel's own check skips it and reports
    # MOE_DEV_BAD_SLOT; every other expert's rows are still computed
    import expert_slot_cache_gb300 as M
    f = _noalloc_fn()
    cfg = C.qwen(1)
    T, S = 1, 16
    ids = np.arange(cfg.k, dtype=np.int32).reshape(1, -1)
    slabs = torch.empty(cfg.k, cfg.slab_elems, dtype=torch.bfloat16, device=DEV)
    for e in range(cfg.k):
        slabs[e].copy_(C.draw_slab(cfg, e, DEV))
    pool = torch.zeros(S, cfg.slab_elems, dtype=torch.bfloat16, device=DEV)
    pool[:cfg.k].copy_(slabs)
    e2s_np = np.full(cfg.E, -1, dtype=np.int32)
    e2s_np[:cfg.k] = np.arange(cfg.k)
    e2s_np[cfg.k - 1] = S  # past the end of the pool
    e2s = torch.from_numpy(e2s_np).to(DEV)
    x = C.draw_x(cfg, DEV, step=3, T=T)
    g = M.permute(torch.from_numpy(ids).to(DEV), cfg.E)
    lst = torch.arange(cfg.k, dtype=torch.int32, device=DEV)
    n_list = torch.tensor([cfg.k], dtype=torch.int32, device=DEV)
    y = torch.full((T * cfg.k, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rc = _call_noalloc(f, cfg, x, T, g, lst, n_list, cfg.k, pool, y, status, e2s=e2s)
    assert rc == 0, M.status_str(rc)
    torch.cuda.synchronize()
    assert int(status[0]) == 2  # MOE_DEV_BAD_SLOT
    got = y.cpu().numpy()
    want = _oracle_y(x, g, cfg, torch.cat([slabs.cpu(), torch.zeros(cfg.E - cfg.k, cfg.slab_elems,
                                                                     dtype=torch.bfloat16)]))
    ok = np.arange(cfg.k - 1)  # grouped position p holds expert p (one token, ids 0..k-1)
    assert rel_l2(got[ok], want[ok]) <= RL2_F32


def test_noalloc_ffn_refuses_oversized_request():
    import expert_slot_cache_gb300 as M
    f = _noalloc_fn()
    cfg = C.qwen(8)
    T = (1 << 20) // (cfg.k * cfg.I) + 1  # one token more than the scratch holds
    x = torch.zeros(T, cfg.H, dtype=torch.bfloat16, device=DEV)
    z = torch.zeros(cfg.E + 1, dtype=torch.int32, device=DEV)
    rows = torch.zeros(T * cfg.k, dtype=torch.int32, device=DEV)
    pool = torch.zeros(cfg.E, 16, dtype=torch.bfloat16, device=DEV)
    y = torch.zeros(16, dtype=torch.float32, device=DEV)
    rc = f(_p(x), T, cfg.H, cfg.I, cfg.k, cfg.E, _p(z), _p(rows), _p(z), _p(z), 1, _p(pool), cfg.E, None, None,
           _p(y), None, c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -7
    assert "scratch" in M.status_str(rc)
