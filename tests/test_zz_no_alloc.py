"""The allocation-free FFN entry point gives the same result as the workspace one.

moe_expert_ffn_noalloc exists for callers that cannot allocate device memory
where they run the FFN (host callbacks, plug-ins that must not touch their
host's memory pool, runtimes with a frozen allocator): it keeps the FFN's
intermediate activations in a fixed array inside the library.  This test
calls it through the C ABI twice in a row, with different shapes and
routings, and compares each result with moe_expert_ffn's on the same inputs
(within the error of the bf16 h that the workspace path's tensor-core down
projection reads) and with the oracle (within fp32 summation error: the
allocation-free path keeps h in fp32).
It also checks that an oversized request is refused with a clear status.
The file name makes pytest collect it last.
"""
import ctypes
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
    f.argtypes = [V, I, I, I, I, I, V, V, V, V, I, V, V, V, V, V, V]
    f.restype = c_int
    return f


def _case(cfg, T, seed):
    import expert_slot_cache_gb300 as M
    rng = np.random.default_rng(seed)
    E = cfg.E
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.1
    p /= p.sum()
    ids = np.stack([rng.choice(E, cfg.k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    used = np.unique(ids)
    x = C.draw_x(cfg, DEV, step=seed, T=T)
    pool = torch.empty(E, cfg.slab_elems, dtype=torch.bfloat16, device=DEV)
    for e in used:
        pool[e].copy_(C.draw_slab(cfg, int(e), DEV))
    g = M.permute(torch.from_numpy(ids).to(DEV), E)
    lst = torch.from_numpy(used.astype(np.int32)).to(DEV)
    n_list = torch.tensor([len(used)], dtype=torch.int32, device=DEV)
    return x, pool, g, lst, n_list, len(used)


def _call_noalloc(f, cfg, x, T, g, lst, n_list, n_used, pool, y, status):
    p = lambda t: c_void_p(t.data_ptr())
    return f(p(x), T, cfg.H, cfg.I, cfg.k, cfg.E, p(g.offset), p(g.rows), p(lst), p(n_list), n_used, p(pool),
             None, None, p(y), p(status), c_void_p(torch.cuda.current_stream().cuda_stream))


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
        rows, offset = g.rows.cpu().numpy(), g.offset.cpu().numpy()
        ref = O.expert_ffn(x.float().cpu().numpy(), rows, offset, cfg.k, HostSlabs(pool.cpu()), cfg.H, cfg.I)
        assert rel_l2(got, ref) <= RL2_F32, f"call {call} vs oracle"


def test_noalloc_ffn_refuses_oversized_request():
    import expert_slot_cache_gb300 as M
    f = _noalloc_fn()
    cfg = C.qwen(8)
    T = (1 << 20) // (cfg.k * cfg.I) + 1  # one token more than the scratch holds
    x = torch.zeros(T, cfg.H, dtype=torch.bfloat16, device=DEV)
    z = torch.zeros(cfg.E + 1, dtype=torch.int32, device=DEV)
    rows = torch.zeros(T * cfg.k, dtype=torch.int32, device=DEV)
    pool = torch.zeros(1, 16, dtype=torch.bfloat16, device=DEV)
    y = torch.zeros(16, dtype=torch.float32, device=DEV)
    p = lambda t: c_void_p(t.data_ptr())
    rc = f(p(x), T, cfg.H, cfg.I, cfg.k, cfg.E, p(z), p(rows), p(z), p(z), 1, p(pool), None, None, p(y), None,
           c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -7
    assert "scratch" in M.status_str(rc)
