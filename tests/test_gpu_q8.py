"""W8A8 experts ("Porting vllm-expert-cache to NVIDIA GPUs": the W8A8 model;
weights and their scales indexed by the same id, so both slot-indexed).

The quantised slabs, the FFN output y and the layer's ids are compared with
the oracle bit for bit: both sides take every fp32 step in the same order
(codes, dequantisation, SiLU on the op-by-op exp), and the dot products are
exact integer sums.  The oracle quantises the bf16 weights itself; the GPU's
quantised bytes are checked equal to its own before they are used."""
import numpy as np
import pytest
import torch

import oracle as O
from harness import configs as C
from tests._setup import HostSlabs, assert_out_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


class QHost:
    """Lazy expert -> the oracle's quantised slab of a bf16 [E][3HI] tensor."""

    def __init__(self, slabs, H, I):
        self.f = HostSlabs(slabs)
        self.H, self.I = H, I
        self.cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = O.quantize_slab(self.f[e].astype(np.float32), self.H, self.I)
        return self.cache[e]


@pytest.mark.parametrize("cfg", [C.TINY, C.qwen(8), C.FLASH], ids=["tiny", "qwen", "flash"])
def test_quantize_slabs_bit_exact(cfg):
    import expert_slot_cache_gb300 as M
    slabs = torch.stack([C.draw_slab(cfg, e, DEV) for e in range(3)])
    q = M.quantize_slabs(slabs, cfg.H, cfg.I).cpu().numpy()
    for e in range(3):
        want = O.quantize_slab(slabs[e].float().cpu().numpy(), cfg.H, cfg.I)
        assert np.array_equal(q[e], want), e


Q8_CASES = [
    ("tiny_T4", C.TINY, 4, 1.2),
    ("qwen_T1", C.qwen(1), 1, 1.2),
    ("qwen_T8", C.qwen(8), 8, 1.2),
    ("qwen_T37_uniform", C.qwen(37), 37, 0.0),
    ("qwen_T64_skewed", C.qwen(64), 64, 1.2),
    ("flash_T16", C.FLASH, 16, 1.1),
]


@pytest.mark.parametrize("name,cfg,T,skew", Q8_CASES, ids=[c[0] for c in Q8_CASES])
def test_expert_ffn_q8_bit_exact(name, cfg, T, skew):
    import expert_slot_cache_gb300 as M
    rng = np.random.default_rng(T + 29)
    E = cfg.E
    p = np.arange(1, E + 1, dtype=np.float64) ** -skew
    p /= p.sum()
    ids = np.stack([rng.choice(E, cfg.k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    count, offset, rows, pos = O.permute(ids, E)
    x = C.draw_x(cfg, DEV, T=T)
    used = np.nonzero(count)[0]
    S = len(used)
    bf = torch.empty(E, cfg.slab_elems, dtype=torch.bfloat16)
    e2s = np.full(E, -1, dtype=np.int32)
    slabs = torch.stack([C.draw_slab(cfg, int(e), DEV) for e in used])
    qd = M.quantize_slabs(slabs, cfg.H, cfg.I)
    pool = torch.empty_like(qd)
    for i, e in enumerate(used):
        sl = S - 1 - i
        e2s[e] = sl
        pool[sl].copy_(qd[i])
        bf[e].copy_(slabs[i].cpu())
    lst = torch.from_numpy(used.astype(np.int32)).to(DEV)
    g = M.permute(torch.from_numpy(ids).to(DEV), E)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = M.expert_ffn_q8(x, cfg.k, cfg.I, E, g.offset, g.rows, lst, torch.tensor([S], dtype=torch.int32, device=DEV),
                        S, pool, torch.from_numpy(e2s).to(DEV), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    qh = QHost(bf, cfg.H, cfg.I)
    for i, e in enumerate(used[:4]):
        assert np.array_equal(qd[i].cpu().numpy(), qh[e])
    want = O.expert_ffn_q8(x.float().cpu().numpy(), rows, offset, cfg.k, qh, cfg.H, cfg.I)
    got = y.cpu().numpy()
    assert np.array_equal(got, want), f"max |diff| {np.nanmax(np.abs(got - want))}"


@pytest.mark.parametrize("mode,T,sched", [(C.MODE_GATHER, 8, C.SCHED_CHUNKS), (C.MODE_GATHER, 32, C.SCHED_CHUNKS),
                                          (C.MODE_GATHER, 64, C.SCHED_WAVES), (C.MODE_RESIDENT, 64, C.SCHED_CHUNKS)],
                         ids=["gather_T8", "gather_T32_chunked", "gather_T64_waves", "resident_T64"])
def test_layer_w8a8(mode, T, sched):
    import expert_slot_cache_gb300 as M
    cfg = C.qwen(T, S=64 if mode == C.MODE_GATHER else 128, mode=mode, schedule=sched)
    wr = C.draw_router(cfg, DEV)
    bf_dev = torch.empty(cfg.E, cfg.slab_elems, dtype=torch.bfloat16, device=DEV)
    C.draw_slabs(cfg, DEV, out=bf_dev)
    q_dev = M.quantize_slabs(bf_dev, cfg.H, cfg.I)
    bf_host = bf_dev.cpu()
    qh = QHost(bf_host, cfg.H, cfg.I)
    if mode == C.MODE_RESIDENT:
        pool, gst, ost, host_q = q_dev, None, None, None
    else:
        s2e0 = C.initial_residency(cfg)
        host_q = torch.empty(cfg.E, q_dev.shape[1], dtype=torch.uint8, pin_memory=True)
        host_q.copy_(q_dev)
        pool = q_dev[torch.from_numpy(s2e0.astype(np.int64)).to(DEV)].contiguous()
        gst, ost = M.CacheState.from_slots(s2e0, cfg.E), O.CacheState.from_slots(s2e0, cfg.E)
    del bf_dev
    layer = M.SlotCachedMoELayer(wr, pool, cfg.k, cfg.I, cfg.mode, cfg.policy, host_slabs=host_q, state=gst,
                                 max_tokens=T, quant=1, schedule=sched)
    wr_np = wr.float().cpu().numpy()
    for step in range(2):
        x = C.draw_x(cfg, DEV, step=step)
        res = layer.forward(x)
        torch.cuda.synchronize()
        want = O.layer_forward(x.float().cpu().numpy(), wr_np, qh, cfg.H, cfg.I, cfg.k, cfg.mode, cfg.policy, ost,
                               None, quant=True, schedule=sched)
        assert np.array_equal(res["ids"].cpu().numpy(), want["ids"]), step
        assert_out_close(res["out"].float().cpu().numpy(), want["out"], f"step {step}")
        if ost is not None:
            assert gst.s2e.cpu().numpy().tolist() == ost.s2e.tolist()
            assert gst.prio.cpu().numpy().astype(np.uint32).tolist() == ost.prio.tolist()
            assert int(gst.stamp.item()) == ost.stamp
    assert int(layer.dev_status.item()) == 0
    if mode == C.MODE_GATHER:
        s2e = gst.s2e.cpu().numpy()
        for s in range(0, cfg.S, 9):
            assert torch.equal(pool[s].cpu(), host_q[s2e[s]])
