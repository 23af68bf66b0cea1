"""The layer configurations and the seeded inputs drawn for them.

Shapes follow the models the pages measure on: a Qwen3-30B-A3B-shaped layer
(128 experts, top-8, hidden 2048, intermediate 768), a Flash-Next-shaped
layer (512 experts, top-10, intermediate 512) and a GLM-like 288-expert
stack.  No page ships weights, routing traces or brightness profiles, so
every tensor below is synthetic: expert and router weights ~N(0, 0.02),
activations ~N(0, 1) (Irwin-Hall approximations, see ``harness.gen``), a
per-expert logit offset ~N(0, 1) for the prefill case, and a Zipf(1.1)
brightness over a seeded ranking for the soft-bias case.

Expert slab storage (one contiguous block per expert, bf16):
    [ Wg (H x I) | Wu (H x I) | Wd (I x H) ]   each stored input-major
so ``g = x @ Wg``, ``u = x @ Wu`` and ``y = h @ Wd``.  The block is drawn as
one stream of 3*H*I values in storage order.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from . import gen

MODE_RESIDENT = 0
MODE_GATHER = 1
MODE_ZERO_RETURN = 2
POLICY_LRU = 0
POLICY_LFU = 1
POLICY_STATIC = 2
SCHED_CHUNKS = 0
SCHED_WAVES = 1

W_SIGMA = 0.02
X_SIGMA = 1.0


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    S: int
    seed: int
    x_seed: int
    mode: int = MODE_RESIDENT
    policy: int = POLICY_LRU
    logit_offset: bool = False
    # soft selection bias (max(cap, ln(b/b_edge)) on cold experts)
    bias_cap: Optional[float] = None
    n_hot: int = 0
    zipf_s: float = 0.0
    layers: int = 1
    steps: int = 1
    # GATHER steps larger than the pool: token chunks or expert waves
    schedule: int = SCHED_CHUNKS
    # per-layer slot counts of a stack (None: every layer has S slots)
    s_per_layer: Optional[tuple] = None

    @property
    def slab_elems(self) -> int:
        return 3 * self.H * self.I

    @property
    def slab_bytes(self) -> int:
        return 2 * self.slab_elems

    def with_(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)


TINY = LayerConfig("tiny", T=4, H=256, E=16, k=2, I=128, S=16, seed=1, x_seed=1001)

QWEN = LayerConfig("qwen3-30b-a3b-decode", T=8, H=2048, E=128, k=8, I=768, S=64,
                   seed=2, x_seed=2008, mode=MODE_GATHER, policy=POLICY_LRU)


def qwen(T: int, S: int = 64, mode: int = MODE_GATHER, policy: int = POLICY_LRU,
         schedule: int = SCHED_CHUNKS) -> LayerConfig:
    return QWEN.with_(T=T, S=S, x_seed=2000 + T, mode=mode, policy=policy, schedule=schedule)


FLASH = LayerConfig("flash-next-zero-return", T=16, H=2048, E=512, k=10, I=512, S=192,
                    seed=3, x_seed=3016, mode=MODE_ZERO_RETURN, policy=POLICY_STATIC,
                    bias_cap=-1.0, n_hot=192, zipf_s=1.1)

PREFILL = LayerConfig("prefill", T=4096, H=2048, E=128, k=8, I=768, S=128, seed=4,
                      x_seed=4096, mode=MODE_RESIDENT, logit_offset=True)

STACK = LayerConfig("stack48", T=32, H=2048, E=288, k=8, I=512, S=288, seed=5, x_seed=5000,
                    mode=MODE_RESIDENT, layers=48, steps=64)

STACK_SLOTS = STACK.with_(name="stack48-slots", S=144, mode=MODE_GATHER, policy=POLICY_LRU)


def budget_slots(E: int, layers: int) -> tuple:
    """Non-uniform slots per layer after "Betelgeuse ... on an RTX 3060", "Arrival-Slack VRAM Slot Pool":
    240 slots per layer on layers 0-4 (no compute slack there), 92 on the middle layers, 60 on the tail
    layers, for 512 experts per layer and about 5,000 slots in all -- which puts 38 layers in the middle
    and 5 at the tail of 48.  Here the same fractions of E per layer: E*240/512 on the first 5 layers,
    E*60/512 on the last 5, E*92/512 between."""
    early, tail = 5, 5
    return tuple(round(E * (240 if l < early else 60 if l >= layers - tail else 92) / 512) for l in range(layers))


STACK_BUDGET = STACK_SLOTS.with_(name="stack48-budget", schedule=SCHED_WAVES, s_per_layer=budget_slots(288, 48))


def layer_S(cfg: LayerConfig, layer: int = 0) -> int:
    """Slots of one layer of a stack."""
    return cfg.s_per_layer[layer] if cfg.s_per_layer else cfg.S


# ----------------------------------------------------------------------------
# Draws
# ----------------------------------------------------------------------------

def draw_x(cfg: LayerConfig, device="cpu", layer: int = 0, step: int = 0, T: Optional[int] = None) -> torch.Tensor:
    """Activations [T][H] bf16."""
    T = cfg.T if T is None else T
    s = gen.stream_id(gen.KIND_X if step == 0 else gen.KIND_STEPX, layer, step)
    return gen.normal_bf16(cfg.x_seed + layer, s, T * cfg.H, X_SIGMA, device).view(T, cfg.H)


def draw_router(cfg: LayerConfig, device="cpu", layer: int = 0) -> torch.Tensor:
    """Router weight [H][E] bf16."""
    s = gen.stream_id(gen.KIND_ROUTER, layer)
    return gen.normal_bf16(cfg.seed, s, cfg.H * cfg.E, W_SIGMA, device).view(cfg.H, cfg.E)


def draw_slab(cfg: LayerConfig, e: int, device="cpu", layer: int = 0) -> torch.Tensor:
    """One expert's slab, flat bf16 [3*H*I] in storage order."""
    s = gen.stream_id(gen.KIND_EXPERT, layer, e)
    return gen.normal_bf16(cfg.seed, s, cfg.slab_elems, W_SIGMA, device)


def draw_slabs(cfg: LayerConfig, device="cpu", layer: int = 0, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """All experts' slabs [E][3*H*I] bf16 (into ``out`` when given)."""
    if out is None:
        out = torch.empty(cfg.E, cfg.slab_elems, dtype=torch.bfloat16, device=device)
    for e in range(cfg.E):
        out[e].copy_(draw_slab(cfg, e, out.device, layer))
    return out


def draw_logit_offset(cfg: LayerConfig, device="cpu", layer: int = 0) -> Optional[torch.Tensor]:
    """Per-expert additive logit offset ~N(0,1) fp32 (prefill skew), or None."""
    if not cfg.logit_offset:
        return None
    s = gen.stream_id(gen.KIND_OFFSET, layer)
    return gen.normal_f32(cfg.seed, s, cfg.E, 1.0, device)


def draw_brightness(cfg: LayerConfig, layer: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """Zipf brightness over a seeded ranking.

    Returns ``(b, rank)``: ``rank`` is a permutation of 1..E, and
    ``b[e] = rank[e]**-s / sum_j rank[j]**-s`` as fp32.
    """
    perm = gen.permutation(cfg.seed, gen.stream_id(gen.KIND_BRIGHT, layer), cfg.E)
    rank = np.empty(cfg.E, dtype=np.int64)
    rank[perm] = np.arange(1, cfg.E + 1)
    raw = rank.astype(np.float64) ** (-cfg.zipf_s)
    b = (raw / raw.sum()).astype(np.float32)
    return b, rank


def initial_residency(cfg: LayerConfig, layer: int = 0) -> np.ndarray:
    """Initial slot contents ``s2e[S]`` (int32, -1 = empty).

    Slot-pool configs: the experts of a seeded permutation's first S entries,
    sorted, in slots 0..S-1.  Soft-bias configs: the n_hot experts ranked
    brightest (rank <= n_hot), sorted.  S >= E: expert e in slot e.
    """
    S, E = layer_S(cfg, layer), cfg.E
    s2e = np.full(S, -1, dtype=np.int32)
    if S >= E:
        s2e[:E] = np.arange(E, dtype=np.int32)
        return s2e
    if cfg.n_hot > 0:
        _, rank = draw_brightness(cfg, layer)
        hot = np.sort(np.nonzero(rank <= cfg.n_hot)[0])[:S]
        s2e[: len(hot)] = hot
        return s2e
    perm = gen.permutation(cfg.seed, gen.stream_id(gen.KIND_RESIDENCY, layer), E)
    s2e[:] = np.sort(perm[:S])
    return s2e


def e2s_from_s2e(s2e: np.ndarray, E: int) -> np.ndarray:
    e2s = np.full(E, -1, dtype=np.int32)
    for s, e in enumerate(s2e):
        if e >= 0:
            e2s[e] = s
    return e2s


# ----------------------------------------------------------------------------
# Routing traces for policy replay
# ----------------------------------------------------------------------------

def drifting_trace(E: int, k: int, T: int, steps: int, seed: int = 7, s: float = 1.1,
                   swaps_per_step: int = 2) -> np.ndarray:
    """Synthetic routing ids [steps][T][k] with a popularity that drifts.

    Expert popularity is Zipf(s) over a ranking that changes slowly: after
    each step, ``swaps_per_step`` random pairs of ranks trade places, so the
    hot set drifts while any short window keeps temporal locality (the
    transcript's "the useful set drifts").  Each token draws k distinct
    experts from that popularity.  numpy's seeded Generator: a test input,
    drawn once on the host.
    """
    rng = np.random.default_rng(seed)
    p = np.arange(1, E + 1, dtype=np.float64) ** -s
    p /= p.sum()
    order = rng.permutation(E)  # order[r] = expert at rank r
    out = np.empty((steps, T, k), dtype=np.int32)
    for st in range(steps):
        for t in range(T):
            out[st, t] = order[rng.choice(E, size=k, replace=False, p=p)]
        for _ in range(swaps_per_step):
            a, b = rng.integers(0, E, size=2)
            order[a], order[b] = order[b], order[a]
    return out
