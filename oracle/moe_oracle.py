"""CPU oracle for the MoE layer with an expert slot cache.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plain statement of what
the hot path computes.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import it; the library never does, and it shares no
code with the CUDA path.

Sources (web pages; cited by title and section):
  [SGB]   "Nudge, don't cut" (PGO-SGB), section "The method in five lines":
          bias[l][e] = max(cap, ln(b[l][e] / b_edge[l])) on cold experts, 0 on
          hot ones; pick top-k by logit + bias; weights are the router's own
          softmax over the k picked, from the unbiased logits (selection only).
  [PORT]  "Porting vllm-expert-cache to NVIDIA GPUs", sections "What this
          package does" (manage picks victims among slots the step does not
          need and emits a miss list; gather copies missing experts host to
          slot; routing ids are remapped to slot space), "Prove it is correct
          before measuring" (fields: expert-to-slot table, cold map, slot
          contents, priorities, miss list; deterministic, no atomics;
          16-byte slabs), "Measuring, without fooling yourself" (sizing trap:
          a step is served from slots only when tokens x top_k <= slots).
  [ZERO]  "RTX 3060 runs a 35B MoE with llama.cpp" (video transcript), chapter
          "Designing a fixed expert cache with zero-return for missing
          experts": a missing expert returns zeros; a second pass over the
          missing experts is added, which gives exactly the full result.
  [REPICK] transcript, the chapter on code and chat profiles: the hot set is
          static, yet the useful set drifts; "every 500 tokens, say, have
          another look. Swap out whatever's gone cold and then leave it alone
          again", paying for transfers once per window.
  [Q8]    "Porting vllm-expert-cache to NVIDIA GPUs": the measured model is
          Qwen3-30B-A3B W8A8 (8-bit weights and activations); "weights and
          their scales are indexed by the same id, so both must be
          slot-indexed" (section on traps in a new backend).
  [SGB2]  same PGO-SGB page, introduction (two ways to use a profile: a hard
          mask, cold experts can never be picked; or a soft bias) and the KL
          comparison of a graded bias against a flat one (a flat -0.75,
          -0.5, -1); "Qwen on Strata" (selection-only against damped
          weights: the bias also enters the weights); "The same idea on
          GLM-5.3-Flash" (GLM's router is a sigmoid and the bias is added
          after the sigmoid, in probability space).

Precision.  Router logits decide integers (the top-k ids), so they are taken
in fp32 in one fixed order that the kernels follow as well: h is cut into
consecutive blocks of LOGIT_BLOCK = 128; within block b, part_b = 0 then
part_b = fma(x[t][h], Wr[h][e], part_b) for h ascending; then
logit = 0 + part_0 + part_1 + ... in block order (fp32 adds).  A bf16 x bf16
product is exact in fp32, so "multiply then add in fp32" is that same fma.
Selection compares fp32 scores logit + bias (one IEEE add).  Everything else
(softmax weights, the SwiGLU expert FFN, the combine) is evaluated in fp64.

Readings of points the pages leave open (each listed in the design notes):
  * top-k order: descending score, equal scores -> lower expert id first;
  * softmax over the k picked (equal to a full softmax renormalised);
  * hot set = the n_hot brightest experts (ties -> lower id); b_edge = the
    smallest brightness in it; bias computed in fp64, rounded to fp32; b = 0
    gives the cap;
  * SwiGLU: h = silu(x Wg) * (x Wu), silu(z) = z / (1 + exp(-z)), y = h Wd,
    no biases; slab = [Wg (HxI) | Wu (HxI) | Wd (IxH)] input-major;
  * manage: stamp += 1 per call.  LRU: prio = stamp on hit or load.  LFU:
    prio += 1 on a hit (once per call), prio = 1 on load.  STATIC: no
    eviction, no priority change; misses listed with slot -1.  Victims are
    slots not needed by the call: empty slots first (ascending slot), then
    ascending prio, then ascending slot.  The i-th missing expert (ascending
    id) takes the i-th victim.  Eviction clears the old expert's entry.
  * a step larger than the pool (T*k > S while S < E), token-chunk schedule:
    split into chunks of floor(S/k) consecutive tokens, each chunk managed,
    gathered and computed in turn; S < k cannot be served.
  * the same, expert-wave schedule (each missing expert loaded at most once
    per step; [PORT] "Measuring, without fooling yourself": count misses, not
    tokens): one manage call over the whole step updates the hits and loads
    as many misses (ascending id) as there are slots the step does not need;
    the misses left over are deferred.  The hits and the loaded misses are
    computed; then the deferred experts are taken in ascending id, at most S
    at a time, each batch one manage call whose victims may be any slot (every
    expert already resident has been computed: the rest of the step no longer
    needs it), gathered and computed in turn.  An empty batch is no call.
  * zero-return: residency is e2s[e] >= 0 after a STATIC manage; the output is
    the sum of the resident partial and the missing partial.
  * bias modes: graded (the formula above), flat (every cold expert gets one
    constant), hard mask (cold experts get -inf, so they are never picked
    while k hot experts exist).
  * damped weights: w = softmax over the k picked of logit + bias (the bias
    table only; affinity stays selection-only).
  * periodic re-pick (STATIC pool): every routing adds 1 to its expert's
    window count; a re-pick takes the S experts with the largest counts
    (ties: resident before cold, then lower id) as the new set, loads the
    new members into the slots of experts that left it (empty slots first,
    then ascending slot; new members in ascending id), and clears the counts.
  * W8A8 experts: symmetric int8, scale = amax / 127 (fp32), code =
    rint(v / scale) clamped to [-127, 127] (a zero amax gives scale 0 and
    code 0); weights per output channel (offline), activations per routing
    row (x before gate/up, h before down).  Products are exact int32 sums;
    g = (float(acc) * s_w[n]) * s_x[row], likewise u and y; h = silu(g) * u
    with silu(g) = g / (1 + exp32(-g)); all of it fp32, one operation at a
    time, so the codes of h and the output y are reproducible bit for bit.
    A quantised slab holds [Wg | Wu | Wd] as int8 with every 4 consecutive
    input rows of a column packed together (byte (k, n) at
    ((k div 4) * N + n) * 4 + k mod 4), then the fp32 scales sg[I], su[I],
    sd[H]; the scales travel with the weights, so they are slot-indexed too.
  * sigmoid router: s = sigmoid(logit); pick top-k by s + bias; weights =
    the picked experts' sigmoid values normalised to sum 1 (the router's own
    probabilities).  So that the ids are reproducible bit for bit, the fp32
    sigmoid is defined operation by operation (exp32 below).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

LRU, LFU, STATIC = 0, 1, 2
RESIDENT, GATHER, ZERO_RETURN = 0, 1, 2


# ----------------------------------------------------------------------------
# Routing  [SGB "The method in five lines"]
# ----------------------------------------------------------------------------

LOGIT_BLOCK = 128


def router_logits(x: np.ndarray, wr: np.ndarray, logit_offset=None) -> np.ndarray:
    """logit[t][e] = sum_h x[t][h] * Wr[h][e] in fp32, blocked order (see above).

    ``x`` [T][H] and ``wr`` [H][E] hold bf16 values (as float32 arrays).  The
    optional per-expert ``logit_offset`` [E] is added after the sum.
    """
    x = np.asarray(x, dtype=np.float32)
    wr = np.asarray(wr, dtype=np.float32)
    T, H = x.shape
    acc = np.zeros((T, wr.shape[1]), dtype=np.float32)
    for h0 in range(0, H, LOGIT_BLOCK):
        part = np.zeros_like(acc)
        for h in range(h0, min(H, h0 + LOGIT_BLOCK)):
            part += x[:, h:h + 1] * wr[h:h + 1, :]
        acc += part
    if logit_offset is not None:
        acc = acc + np.asarray(logit_offset, dtype=np.float32)[None, :]
    return acc


BIAS_GRADED, BIAS_FLAT, BIAS_HARD = 0, 1, 2


def bias_table(b: np.ndarray, n_hot: int, cap: float, mode: int = BIAS_GRADED) -> np.ndarray:
    """Selection bias for one layer: 0 on the hot set; on cold experts
    max(cap, ln(b/b_edge)) (graded, [SGB]), the constant ``cap`` (flat) or
    -inf (hard mask) [SGB2]."""
    b = np.asarray(b, dtype=np.float32)
    E = b.shape[0]
    order = sorted(range(E), key=lambda e: (-float(b[e]), e))
    hot = set(order[:n_hot])
    b_edge = min(float(b[e]) for e in hot)
    out = np.zeros(E, dtype=np.float32)
    for e in range(E):
        if e in hot:
            continue
        if mode == BIAS_FLAT:
            out[e] = np.float32(cap)
        elif mode == BIAS_HARD:
            out[e] = np.float32(-np.inf)
        else:
            be = float(b[e])
            val = cap if be <= 0.0 else max(cap, float(np.log(be / b_edge)))
            out[e] = np.float32(val)
    return out


# fp32 exp, defined operation by operation (each an IEEE fp32 multiply, add or
# subtract, none fused), after Cody and Waite's argument reduction: n = the
# integer nearest x*log2(e), r = x - n*ln2 with ln2 split into a short high
# part (n*LN2_HI is exact) and a low part, then the degree-7 Taylor polynomial
# of e^r in Horner form, scaled by 2^n.  exp32(x) = +inf above 88 and 0 below
# -80 (the sigmoid saturates there); in between 2^n stays a normal number.
_F = np.float32
_LOG2E = _F(float.fromhex("0x1.715476p+0"))
_LN2_HI = _F(float.fromhex("0x1.63p-1"))
_LN2_LO = _F(float.fromhex("-0x1.bd0106p-13"))
_TAYLOR = [_F(float.fromhex(h)) for h in ("0x1.a01a02p-13", "0x1.6c16c2p-10", "0x1.111112p-7",
                                           "0x1.555556p-5", "0x1.555556p-3", "0x1p-1", "0x1p+0", "0x1p+0")]


def exp32(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        n = np.rint(x * _LOG2E).astype(np.float32)
        r = (x - n * _LN2_HI).astype(np.float32)
        r = (r - n * _LN2_LO).astype(np.float32)
        p = _TAYLOR[0]
        for c in _TAYLOR[1:]:
            p = (p * r).astype(np.float32)
            p = (p + c).astype(np.float32)
        ni = np.clip(n, -126, 127).astype(np.int32)
        scale = ((ni + 127).astype(np.uint32) << np.uint32(23)).view(np.float32)
        out = (p * scale).astype(np.float32)
    out = np.where(x > _F(88.0), _F(np.inf), out)
    out = np.where(x < _F(-80.0), _F(0.0), out)
    return out.astype(np.float32)


def sigmoid32(l) -> np.ndarray:
    """fp32 sigmoid 1 / (1 + exp32(-l)): one fp32 add and one IEEE fp32 divide."""
    l = np.asarray(l, dtype=np.float32)
    with np.errstate(over="ignore"):
        d = (_F(1.0) + exp32(-l)).astype(np.float32)
        return (_F(1.0) / d).astype(np.float32)


ROUTER_SOFTMAX, ROUTER_SIGMOID = 0, 1


def select_topk(logits: np.ndarray, k: int, bias=None, resident=None, affinity: float = 0.0,
                router: int = ROUTER_SOFTMAX) -> np.ndarray:
    """ids[t][0..k-1]: the k largest fp32 scores, descending, ties -> lower id.

    score = logit (softmax router) or sigmoid32(logit) (sigmoid router, [SGB2]),
    + bias when a bias is given, then + affinity for experts resident in VRAM
    right now (live-cache affinity: "Nudge, don't cut", "Then Maya's own knob
    beat ours"), each add in fp32.
    """
    logits = np.asarray(logits, dtype=np.float32)
    base = sigmoid32(logits) if router == ROUTER_SIGMOID else logits
    scores = base if bias is None else (base + np.asarray(bias, dtype=np.float32)[None, :]).astype(np.float32)
    if resident is not None and affinity != 0.0:
        lam = np.where(np.asarray(resident, dtype=bool), np.float32(affinity), np.float32(0.0)).astype(np.float32)
        scores = np.where(lam[None, :] != 0, scores + lam[None, :], scores).astype(np.float32)
    T, E = scores.shape
    ids = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(scores[t, e]), e))
        ids[t] = order[:k]
    return ids


def route_weights(logits: np.ndarray, ids: np.ndarray, router: int = ROUTER_SOFTMAX, bias=None,
                  damped: bool = False) -> np.ndarray:
    """Routing weights over the k picked, fp64.

    softmax router: w[t][j] = exp(z_j) / sum_j' exp(z_j'), z = the unbiased
    logit (selection-only, [SGB]) or logit + bias (damped weights, [SGB2]);
    sigmoid router: w[t][j] = s_j / sum_j' s_j', s = sigmoid(logit) [SGB2].
    """
    T, k = ids.shape
    w = np.empty((T, k), dtype=np.float64)
    bz = None if (bias is None or not damped) else np.asarray(bias, dtype=np.float64)
    for t in range(T):
        l = np.array([float(logits[t, e]) for e in ids[t]], dtype=np.float64)
        if router == ROUTER_SIGMOID:
            sv = 1.0 / (1.0 + np.exp(-l))
            w[t] = sv / sv.sum()
            continue
        if bz is not None:
            l = l + np.array([bz[e] for e in ids[t]])
        p = np.exp(l - l.max())
        w[t] = p / p.sum()
    return w


def route(x, wr, k, logit_offset=None, bias=None, resident=None, affinity=0.0, router=ROUTER_SOFTMAX,
          damped=False):
    if router == ROUTER_SIGMOID and damped:
        raise ValueError("damped weights are defined for the softmax router only")
    logits = router_logits(x, wr, logit_offset)
    ids = select_topk(logits, k, bias, resident, affinity, router)
    return ids, route_weights(logits, ids, router, bias, damped), logits


# ----------------------------------------------------------------------------
# Permutation into per-expert groups
# ----------------------------------------------------------------------------

def permute(ids: np.ndarray, E: int):
    """Group the flat routing slots t*k+j by expert, stable in the flat index.

    Returns count[E], offset[E+1] (exclusive prefix), rows[T*k] (the flat
    index at each grouped position) and pos[T*k] (grouped position of each
    flat index).
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    n = flat.shape[0]
    count = np.zeros(E, dtype=np.int32)
    for e in flat:
        count[e] += 1
    offset = np.zeros(E + 1, dtype=np.int32)
    for e in range(E):
        offset[e + 1] = offset[e] + count[e]
    rows = np.array(sorted(range(n), key=lambda i: (int(flat[i]), i)), dtype=np.int32)
    pos = np.empty(n, dtype=np.int32)
    for p, i in enumerate(rows):
        pos[i] = p
    return count, offset, rows, pos


# ----------------------------------------------------------------------------
# Slot cache  [PORT "What this package does", "Prove it is correct ..."]
# ----------------------------------------------------------------------------

@dataclass
class CacheState:
    e2s: np.ndarray            # int32 [E], -1 = cold (host only)
    s2e: np.ndarray            # int32 [S], -1 = empty slot
    prio: np.ndarray           # uint32 [S]
    stamp: int = 0

    @staticmethod
    def from_slots(s2e, E: int) -> "CacheState":
        s2e = np.asarray(s2e, dtype=np.int32).copy()
        e2s = np.full(E, -1, dtype=np.int32)
        for s, e in enumerate(s2e):
            if e >= 0:
                e2s[e] = s
        return CacheState(e2s, s2e, np.zeros(len(s2e), dtype=np.uint32), 0)

    def copy(self) -> "CacheState":
        return CacheState(self.e2s.copy(), self.s2e.copy(), self.prio.copy(), self.stamp)


@dataclass
class ManageResult:
    miss_e: list = field(default_factory=list)
    miss_s: list = field(default_factory=list)
    hit_e: list = field(default_factory=list)
    sid: np.ndarray = None
    deferred: list = field(default_factory=list)


class CapacityError(ValueError):
    pass


def manage(state: CacheState, ids: np.ndarray, policy: int, defer: bool = False) -> ManageResult:
    """One expert_cache_manage call on the flat routing ids of a step (updates ``state``).

    With ``defer`` a call that needs more experts than the pool holds is
    allowed: the misses (ascending id) take the victims in order while they
    last, and the rest are listed in ``deferred`` and left cold (the first
    call of the expert-wave schedule).
    """
    flat = [int(e) for e in np.asarray(ids).reshape(-1)]
    S = state.s2e.shape[0]
    state.stamp += 1
    stamp = state.stamp
    needed = sorted(set(flat))
    if policy != STATIC and len(needed) > S and not defer:
        raise CapacityError(f"{len(needed)} experts needed, {S} slots")
    hits = [e for e in needed if state.e2s[e] >= 0]
    misses = [e for e in needed if state.e2s[e] < 0]
    res = ManageResult(miss_e=list(misses), hit_e=list(hits))
    if policy == LRU:
        for e in hits:
            state.prio[state.e2s[e]] = stamp
    elif policy == LFU:
        for e in hits:
            state.prio[state.e2s[e]] += 1
    if policy == STATIC:
        res.miss_s = [-1] * len(misses)
    else:
        used = {int(state.e2s[e]) for e in hits}
        cands = [s for s in range(S) if s not in used]
        empty = [s for s in cands if state.s2e[s] < 0]
        full = sorted((s for s in cands if state.s2e[s] >= 0), key=lambda s: (int(state.prio[s]), s))
        victims = (empty + full)[: len(misses)]
        res.deferred = misses[len(victims):]
        res.miss_e = misses[:len(victims)]
        for e, s in zip(misses, victims):
            old = int(state.s2e[s])
            if old >= 0:
                state.e2s[old] = -1
            state.s2e[s] = e
            state.e2s[e] = s
            state.prio[s] = stamp if policy == LRU else 1
        res.miss_s = list(victims)
    res.sid = np.array([state.e2s[e] for e in flat], dtype=np.int32).reshape(np.asarray(ids).shape)
    return res


def window_count(counts: np.ndarray, ids: np.ndarray) -> None:
    """Add one per routing to its expert's window count [REPICK]."""
    for e in np.asarray(ids).reshape(-1):
        counts[int(e)] += 1


def repick(state: CacheState, counts: np.ndarray) -> ManageResult:
    """Re-pick the resident set of a STATIC pool from the window counts [REPICK].

    New set: the S experts ranked first by (count descending, resident before
    cold, id ascending).  Its members that are not resident (ascending id) take,
    in order, the slots that are empty or hold an expert outside the new set
    (empty slots first, then ascending slot).  Priorities and stamp are left
    alone (STATIC); the counts are cleared.
    """
    E = state.e2s.shape[0]
    S = state.s2e.shape[0]
    resident = state.e2s >= 0
    order = sorted(range(E), key=lambda e: (-int(counts[e]), 0 if resident[e] else 1, e))
    new = set(order[:min(S, E)])
    miss_e = [e for e in range(E) if e in new and not resident[e]]
    empty = [s for s in range(S) if state.s2e[s] < 0]
    leaving = [s for s in range(S) if state.s2e[s] >= 0 and int(state.s2e[s]) not in new]
    victims = (empty + leaving)[:len(miss_e)]
    for e, s in zip(miss_e, victims):
        old = int(state.s2e[s])
        if old >= 0:
            state.e2s[old] = -1
        state.s2e[s] = e
        state.e2s[e] = s
    counts[:] = 0
    return ManageResult(miss_e=list(miss_e), miss_s=list(victims))


def gather(host: np.ndarray, pool: np.ndarray, miss_e, miss_s) -> None:
    """Copy each missing expert's slab bytes from the host store into its slot."""
    for e, s in zip(miss_e, miss_s):
        pool[s] = host[e]


def manage_waves(state: CacheState, ids: np.ndarray, policy: int) -> list:
    """The manage calls of one step under the expert-wave schedule (see the
    readings above): wave 0 over the whole step with deferral, then one call
    per batch of at most S deferred experts.  Returns the ManageResults in
    order; wave 0's ``hit_e`` and ``miss_e`` and each later wave's ``miss_e``
    are the expert lists computed after that wave's gather."""
    S = state.s2e.shape[0]
    first = manage(state, ids, policy, defer=True)
    waves = [first]
    left = list(first.deferred)
    for b0 in range(0, len(left), S):
        waves.append(manage(state, np.array(left[b0:b0 + S], dtype=np.int32), policy))
    return waves


def chunk_tokens(T: int, k: int, S: int, E: int) -> int:
    """Tokens per chunk so that every chunk fits the pool (sizing trap reading)."""
    if S >= E or T * k <= S:
        return T
    if S < k:
        raise CapacityError(f"S={S} < k={k}")
    return S // k


# ----------------------------------------------------------------------------
# Expert FFN and combine (fp64)
# ----------------------------------------------------------------------------

def unpack_slab(slab: np.ndarray, H: int, I: int):
    """Split a flat slab into Wg [H][I], Wu [H][I], Wd [I][H] (fp64)."""
    s = np.asarray(slab, dtype=np.float64).reshape(-1)
    n = H * I
    return s[:n].reshape(H, I), s[n:2 * n].reshape(H, I), s[2 * n:3 * n].reshape(I, H)


def silu(z):
    return z / (1.0 + np.exp(-z))


# ----------------------------------------------------------------------------
# W8A8 experts  [Q8]
# ----------------------------------------------------------------------------

def q8_slab_bytes(H: int, I: int) -> int:
    return 3 * H * I + 4 * (2 * I + H)


def quantize_cols(W: np.ndarray):
    """Per-column symmetric int8 of an fp32 [K][N] matrix: (codes int8 [K][N], scales fp32 [N])."""
    W = np.asarray(W, dtype=np.float32)
    amax = np.max(np.abs(W), axis=0).astype(np.float32)
    sc = (amax / _F(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(sc[None, :] > 0, np.rint((W / sc[None, :]).astype(np.float32)), _F(0.0))
    return np.clip(q, -127, 127).astype(np.int8), sc


def quantize_rows(X: np.ndarray):
    """Per-row symmetric int8 of an fp32 [R][K] matrix: (codes int8 [R][K], scales fp32 [R])."""
    q, sc = quantize_cols(np.asarray(X, dtype=np.float32).T)
    return np.ascontiguousarray(q.T), sc


def _pack_quads(q: np.ndarray) -> np.ndarray:
    K, N = q.shape
    return np.ascontiguousarray(q.reshape(K // 4, 4, N).transpose(0, 2, 1)).reshape(-1)


def _unpack_quads(b: np.ndarray, K: int, N: int) -> np.ndarray:
    return np.ascontiguousarray(b.reshape(K // 4, N, 4).transpose(0, 2, 1)).reshape(K, N)


def quantize_slab(slab: np.ndarray, H: int, I: int) -> np.ndarray:
    """bf16 slab (values as fp32 [3HI]) -> quantised slab bytes (uint8 [q8_slab_bytes])."""
    v = np.asarray(slab, dtype=np.float32).reshape(-1)
    n = H * I
    parts = []
    scales = []
    for W in (v[:n].reshape(H, I), v[n:2 * n].reshape(H, I), v[2 * n:3 * n].reshape(I, H)):
        q, sc = quantize_cols(W)
        parts.append(_pack_quads(q).view(np.uint8))
        scales.append(sc.view(np.uint8))
    return np.concatenate(parts + scales)


def unpack_q8_slab(b: np.ndarray, H: int, I: int):
    """-> (qg [H][I], qu [H][I], qd [I][H]) int8 and (sg [I], su [I], sd [H]) fp32."""
    b = np.asarray(b, dtype=np.uint8).reshape(-1)
    n = H * I
    qg = _unpack_quads(b[:n].view(np.int8), H, I)
    qu = _unpack_quads(b[n:2 * n].view(np.int8), H, I)
    qd = _unpack_quads(b[2 * n:3 * n].view(np.int8), I, H)
    o = 3 * n
    sg = b[o:o + 4 * I].view(np.float32)
    su = b[o + 4 * I:o + 8 * I].view(np.float32)
    sd = b[o + 8 * I:o + 8 * I + 4 * H].view(np.float32)
    return qg, qu, qd, sg, su, sd


def _dequant(acc: np.ndarray, s_w: np.ndarray, s_r: np.ndarray) -> np.ndarray:
    """(float(acc) * s_w[n]) * s_r[row], fp32, one rounding per operation."""
    a = np.asarray(acc, dtype=np.int64).astype(np.float32)
    return ((a * s_w[None, :]).astype(np.float32) * s_r[:, None]).astype(np.float32)


def swiglu_expert_q8(x_rows: np.ndarray, qslab: np.ndarray, H: int, I: int) -> np.ndarray:
    """W8A8 SwiGLU for a block of rows x [n][H] (fp32 values) -> y fp32 [n][H]  [Q8]."""
    qg, qu, qd, sg, su, sd = unpack_q8_slab(qslab, H, I)
    qx, sx = quantize_rows(np.asarray(x_rows, dtype=np.float32))
    xi = qx.astype(np.int64)
    g = _dequant(xi @ qg.astype(np.int64), sg, sx)
    u = _dequant(xi @ qu.astype(np.int64), su, sx)
    with np.errstate(over="ignore"):
        d = (_F(1.0) + exp32(-g)).astype(np.float32)
        h = ((g / d).astype(np.float32) * u).astype(np.float32)
    qh, sh = quantize_rows(h)
    return _dequant(qh.astype(np.int64) @ qd.astype(np.int64), sd, sh)


def expert_ffn_q8(x, rows, offset, k, qslabs, H, I, experts=None) -> np.ndarray:
    """Grouped W8A8 FFN (fp32 outputs, NaN for rows of experts left out)."""
    x = np.asarray(x, dtype=np.float32)
    E = len(offset) - 1
    y = np.full((len(rows), H), np.nan, dtype=np.float32)
    for e in range(E):
        a, b = int(offset[e]), int(offset[e + 1])
        if a == b or (experts is not None and e not in experts):
            continue
        tok = np.asarray(rows[a:b]) // k
        y[a:b] = swiglu_expert_q8(x[tok], qslabs[e], H, I)
    return y


def swiglu_expert(x_rows: np.ndarray, slab: np.ndarray, H: int, I: int) -> np.ndarray:
    """y = (silu(x Wg) * (x Wu)) Wd for a block of rows x [n][H]."""
    wg, wu, wd = unpack_slab(slab, H, I)
    xr = np.asarray(x_rows, dtype=np.float64)
    return (silu(xr @ wg) * (xr @ wu)) @ wd


def expert_ffn(x, rows, offset, k, slabs, H, I, experts=None) -> np.ndarray:
    """Grouped FFN.  y[p] for grouped position p of expert e uses token rows[p] // k.

    ``slabs`` maps expert id -> flat slab (an [E][3HI] array works).  Rows of
    experts not in ``experts`` (when given) are left as NaN.
    """
    x = np.asarray(x, dtype=np.float64)
    E = len(offset) - 1
    y = np.full((len(rows), H), np.nan, dtype=np.float64)
    for e in range(E):
        a, b = int(offset[e]), int(offset[e + 1])
        if a == b or (experts is not None and e not in experts):
            continue
        tok = np.asarray(rows[a:b]) // k
        y[a:b] = swiglu_expert(x[tok], slabs[e], H, I)
    return y


def combine(y, w, pos, T, k, resident=None):
    """out[t] = sum_j w[t][j] y[pos[t*k+j]], j ascending (fp64).

    With ``resident`` (bool [T][k]) also returns the resident and missing
    partial sums; the output is then their sum.
    """
    y = np.asarray(y, dtype=np.float64)
    H = y.shape[1]
    out = np.zeros((T, H))
    if resident is None:
        for t in range(T):
            for j in range(k):
                out[t] += w[t][j] * y[pos[t * k + j]]
        return out
    res = np.zeros((T, H))
    miss = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            term = w[t][j] * y[pos[t * k + j]]
            if resident[t][j]:
                res[t] += term
            else:
                miss[t] += term
    return res + miss, res, miss


# ----------------------------------------------------------------------------
# Whole layer
# ----------------------------------------------------------------------------

SCHED_CHUNKS, SCHED_WAVES = 0, 1


def layer_forward(x, wr, host, H, I, k, mode, policy=LRU, state=None, pool=None,
                  logit_offset=None, bias=None, affinity=0.0, router=ROUTER_SOFTMAX, damped=False, quant=False,
                  schedule=SCHED_CHUNKS):
    """One MoE layer forward with the slot cache.

    ``host`` [E][3HI] holds every expert (authoritative copy); ``pool``
    [S][3HI] the slot contents (updated by the gather); ``state`` the cache
    state (updated).  Returns a dict with the routing, the per-chunk cache
    results and the outputs (fp64).  In GATHER mode ``schedule`` picks token
    chunks or expert waves for a step larger than the pool; with waves the
    step is one chunk and its record carries ``waves``: per manage call the
    loaded experts, their slots and the cache state after the call.
    """
    if mode == GATHER and schedule == SCHED_WAVES:
        return _layer_forward_waves(x, wr, host, H, I, k, policy, state, pool, logit_offset, bias, affinity,
                                    router, damped, quant)
    x = np.asarray(x, dtype=np.float32)
    T = x.shape[0]
    E = wr.shape[1]
    resident = None if (state is None or affinity == 0.0) else state.e2s >= 0
    ids, w, logits = route(x, wr, k, logit_offset, bias, resident, affinity, router, damped)
    out = np.zeros((T, H))
    out_res = np.zeros((T, H))
    out_miss = np.zeros((T, H))
    chunks = []
    if mode == RESIDENT:
        C = T
    else:
        S = state.s2e.shape[0]
        C = T if policy == STATIC else chunk_tokens(T, k, S, E)
    for t0 in range(0, T, C):
        t1 = min(T, t0 + C)
        cids = ids[t0:t1]
        count, offset, rows, pos = permute(cids, E)
        rec = {"t0": t0, "t1": t1, "count": count, "offset": offset, "rows": rows, "pos": pos}
        if mode != RESIDENT:
            mr = manage(state, cids, policy)
            rec.update(miss_e=mr.miss_e, miss_s=mr.miss_s, hit_e=mr.hit_e, sid=mr.sid,
                       e2s=state.e2s.copy(), s2e=state.s2e.copy(), prio=state.prio.copy(),
                       stamp=state.stamp)
            if mode == GATHER and pool is not None:
                gather(host, pool, mr.miss_e, mr.miss_s)
        if quant:  # host / pool hold quantised slabs [Q8]
            y = expert_ffn_q8(x[t0:t1], rows, offset, k, host, H, I).astype(np.float64)
        else:
            y = expert_ffn(x[t0:t1], rows, offset, k, host, H, I)
        if mode == ZERO_RETURN:
            resident = state.e2s[cids] >= 0
            o, r, m = combine(y, w[t0:t1], pos, t1 - t0, k, resident)
            out[t0:t1], out_res[t0:t1], out_miss[t0:t1] = o, r, m
        else:
            out[t0:t1] = combine(y, w[t0:t1], pos, t1 - t0, k)
        chunks.append(rec)
    res = {"ids": ids, "w": w, "logits": logits, "out": out, "chunks": chunks}
    if mode == ZERO_RETURN:
        res["out_res"], res["out_miss"] = out_res, out_miss
    return res


def _layer_forward_waves(x, wr, host, H, I, k, policy, state, pool, logit_offset, bias, affinity, router, damped,
                         quant):
    """GATHER mode, expert-wave schedule: route and group the whole step once,
    run the manage calls of ``manage_waves`` (gathering each call's loads),
    then the expert FFN of every routed expert and one combine."""
    x = np.asarray(x, dtype=np.float32)
    T = x.shape[0]
    E = wr.shape[1]
    resident = None if affinity == 0.0 else state.e2s >= 0
    ids, w, logits = route(x, wr, k, logit_offset, bias, resident, affinity, router, damped)
    count, offset, rows, pos = permute(ids, E)
    waves = []
    for r in manage_waves(state, ids, policy):
        if pool is not None:
            gather(host, pool, r.miss_e, r.miss_s)
        waves.append({"hit_e": r.hit_e, "miss_e": r.miss_e, "miss_s": r.miss_s, "deferred": r.deferred,
                      "e2s": state.e2s.copy(), "s2e": state.s2e.copy(), "prio": state.prio.copy(),
                      "stamp": state.stamp})
    if quant:
        y = expert_ffn_q8(x, rows, offset, k, host, H, I).astype(np.float64)
    else:
        y = expert_ffn(x, rows, offset, k, host, H, I)
    out = combine(y, w, pos, T, k)
    rec = {"t0": 0, "t1": T, "count": count, "offset": offset, "rows": rows, "pos": pos, "waves": waves,
           "miss_e": [e for wv in waves for e in wv["miss_e"]], "miss_s": [s for wv in waves for s in wv["miss_s"]],
           "hit_e": waves[0]["hit_e"], "e2s": state.e2s.copy(), "s2e": state.s2e.copy(),
           "prio": state.prio.copy(), "stamp": state.stamp}
    return {"ids": ids, "w": w, "logits": logits, "out": out, "chunks": [rec]}
