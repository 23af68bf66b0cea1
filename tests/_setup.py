"""Shared helpers for the tests: tolerance checks and input staging.

The CUDA side and the oracle side receive the same seeded inputs (drawn by
``harness``); nothing here computes any part of the MoE layer.
"""
from __future__ import annotations

import numpy as np
import torch

from harness import configs as C

# Output tolerance (bf16 outputs): both max-abs <= 2e-2 and relative L2 <= 1e-2.
ATOL_OUT = 2e-2
RL2_OUT = 1e-2
# fp32 intermediates (h, y, partial sums) against the fp64 oracle: fp32
# accumulation over <= 2048 terms of random sign gives relative errors of a
# few 1e-7 per element; 1e-5 in relative L2 leaves a wide margin while still
# catching any dropped or misplaced term.
RL2_F32 = 1e-5


def rel_l2(got, want) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def assert_out_close(got, want, what="out"):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    ma = float(np.abs(got - want).max()) if got.size else 0.0
    rl = rel_l2(got, want)
    assert ma <= ATOL_OUT and rl <= RL2_OUT, f"{what}: max-abs {ma:.3e} rel-L2 {rl:.3e}"


# The tensor-core FFN paths hand h to the down projection in bf16: rounding
# h (relative 2^-9, random sign) gives y a relative L2 error of about
# 2^-9 / sqrt(3) ~ 1.1e-3.
RL2_Y_BF16_H = 5e-3


def assert_f32_close(got, want, what="y"):
    rl = rel_l2(got, want)
    assert rl <= RL2_F32, f"{what}: rel-L2 {rl:.3e}"


class HostSlabs:
    """Lazy expert -> fp32 numpy slab view of a bf16 [E][3HI] tensor (for the oracle)."""

    def __init__(self, slabs: torch.Tensor):
        self.slabs = slabs

    def __getitem__(self, e):
        return self.slabs[int(e)].float().numpy()

    def __len__(self):
        return self.slabs.shape[0]


def stage_layer(cfg: C.LayerConfig, layer: int = 0, device="cuda", pinned=True):
    """Draw one layer's inputs; returns a dict of device tensors + the pinned host store."""
    wr = C.draw_router(cfg, device, layer)
    slabs_dev = torch.empty(cfg.E, cfg.slab_elems, dtype=torch.bfloat16, device=device)
    C.draw_slabs(cfg, device, layer, out=slabs_dev)
    host = torch.empty(cfg.E, cfg.slab_elems, dtype=torch.bfloat16, pin_memory=pinned)
    host.copy_(slabs_dev)
    off = C.draw_logit_offset(cfg, device, layer)
    return {"wr": wr, "slabs_dev": slabs_dev, "host": host, "logit_offset": off}
