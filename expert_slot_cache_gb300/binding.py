"""ctypes binding of libmoeslot.so (argument marshalling only).

Every computation runs in the library's CUDA kernels; this module allocates
output tensors with PyTorch, passes raw pointers and the current CUDA stream,
and turns a negative status into an exception.  There is no fallback: if the
library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int, c_int32, c_size_t, c_void_p
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmoeslot.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is not built; run `python __graft_entry__.py` "
        "(or __graft_entry__.build()) first")

lib = ctypes.CDLL(LIB_PATH)

MODE_RESIDENT, MODE_GATHER, MODE_ZERO_RETURN = 0, 1, 2
POLICY_LRU, POLICY_LFU, POLICY_STATIC = 0, 1, 2
DEV_BAD_EXPERT, DEV_BAD_SLOT = 1, 2


PROF_CLASSES = ("route", "permute", "manage", "gather", "ffn_gateup", "ffn_down", "combine", "ffn_rows")


class Prof(ctypes.Structure):
    _fields_ = [("events", POINTER(c_void_p)), ("capacity", c_int32), ("used", c_int32),
                ("tags", POINTER(c_int32))]


class LayerArgs(ctypes.Structure):
    _fields_ = [("T", c_int32), ("H", c_int32), ("E", c_int32), ("k", c_int32), ("I", c_int32), ("S", c_int32),
                ("mode", c_int32), ("policy", c_int32),
                ("x", c_void_p), ("w_router", c_void_p), ("logit_offset", c_void_p), ("sel_bias", c_void_p),
                ("pool", c_void_p), ("host_slabs", c_void_p),
                ("e2s", c_void_p), ("s2e", c_void_p), ("prio", c_void_p), ("stamp", c_void_p),
                ("ids", c_void_p), ("w", c_void_p), ("out", c_void_p), ("out_res", c_void_p),
                ("out_miss", c_void_p), ("stats", c_void_p), ("dev_status", c_void_p),
                ("workspace", c_void_p), ("workspace_bytes", c_size_t), ("prof", POINTER(Prof)),
                ("affinity", c_float), ("route_flags", c_int32), ("window_counts", c_void_p), ("quant", c_int32),
                ("schedule", c_int32), ("decode_kernels", c_int32)]


def _sig(name, argtypes, restype=c_int):
    f = getattr(lib, name)
    f.argtypes = argtypes
    f.restype = restype
    return f


V = c_void_p
I32 = c_int
_status_str = _sig("moe_status_str", [c_int], ctypes.c_char_p)
_bias_table = _sig("moe_bias_table", [V, I32, I32, c_float, V, V])
_bias_table_mode = _sig("moe_bias_table_mode", [V, I32, I32, I32, c_float, V, V])
_route = _sig("moe_route", [V, V, V, V, V, c_float, I32, I32, I32, I32, V, V, V, V, V])
_route_ex = _sig("moe_route_ex", [V, V, V, V, V, c_float, I32, I32, I32, I32, I32, V, V, V, V, V])

BIAS_GRADED, BIAS_FLAT, BIAS_HARD = 0, 1, 2
SCHED_CHUNKS, SCHED_WAVES = 0, 1
ROUTE_SIGMOID, ROUTE_DAMPED = 1, 2
_route_scratch = _sig("moe_route_scratch_bytes", [I32, I32, I32], c_size_t)
_permute = _sig("moe_permute", [V, I32, I32, V, V, V, V, V, V, V, V, V])
_permute_scratch = _sig("moe_permute_scratch_bytes", [I32, I32], c_size_t)
_manage = _sig("moe_cache_manage", [V, I32, I32, I32, I32, V, V, V, V, V, V, V, V, V, V, V, V])
_gather = _sig("moe_cache_gather", [V, V, c_size_t, I32, I32, V, V, V, I32, V, V])
_count = _sig("moe_cache_count", [V, I32, I32, V, V, V])
_q8_slab = _sig("moe_q8_slab_bytes", [I32, I32], c_size_t)
_quantize = _sig("moe_quantize_slabs", [V, I32, I32, I32, V, V])
_ffn_q8_ws = _sig("moe_ffn_q8_workspace_bytes", [I32, I32, I32, I32], c_size_t)
_ffn_q8 = _sig("moe_expert_ffn_q8", [V, I32, I32, I32, I32, I32, V, V, V, V, I32, V, I32, V, V, V, c_size_t, V, V])
_repick = _sig("moe_cache_repick", [V, I32, I32, V, V, V, V, V, V])
_ffn = _sig("moe_expert_ffn", [V, I32, I32, I32, I32, I32, V, V, V, V, I32, V, I32, V, V, V, V, c_size_t, V, V])
_ffn_ws = _sig("moe_ffn_workspace_bytes", [I32, I32, I32, I32], c_size_t)
_combine = _sig("moe_combine", [V, V, V, V, V, I32, I32, I32, I32, I32, V, V, V, V])
_layer = _sig("moe_layer_forward", [POINTER(LayerArgs), V, V])
_layer_ws = _sig("moe_layer_workspace_bytes", [I32, I32, I32, I32, I32, I32], c_size_t)


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_str(code)} ({code})")


def status_str(code: int) -> str:
    return _status_str(code).decode()


def _ck(rc: int, where: str) -> None:
    if rc != 0:
        raise MoeError(rc, where)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else c_void_p(t.data_ptr())


def _ptr(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.data_ptr()


def _s(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return c_void_p(s.cuda_stream)


# ---------------------------------------------------------------------------
# Single calls
# ---------------------------------------------------------------------------

def bias_table(b: torch.Tensor, n_hot: int, cap: float, stream=None, mode: int = BIAS_GRADED) -> torch.Tensor:
    out = torch.empty_like(b)
    if mode == BIAS_GRADED:
        _ck(_bias_table(_p(b), b.numel(), n_hot, cap, _p(out), _s(stream)), "moe_bias_table")
    else:
        _ck(_bias_table_mode(_p(b), b.numel(), n_hot, mode, cap, _p(out), _s(stream)), "moe_bias_table_mode")
    return out


def route(x, w_router, k, logit_offset=None, sel_bias=None, return_logits=False, stream=None, blocked=True,
          e2s=None, affinity=0.0, rflags=0):
    T, H = x.shape
    E = w_router.shape[1]
    ids = torch.empty(T, k, dtype=torch.int32, device=x.device)
    w = torch.empty(T, k, dtype=torch.float32, device=x.device)
    logits = torch.empty(T, E, dtype=torch.float32, device=x.device)
    nb = int(_route_scratch(T, H, E)) if blocked else 0
    scratch = torch.empty(max(nb // 4, 1), dtype=torch.float32, device=x.device) if nb else None
    if rflags:
        _ck(_route_ex(_p(x), _p(w_router), _p(logit_offset), _p(sel_bias), _p(e2s), affinity, rflags, T, H, E, k,
                      _p(logits), _p(scratch), _p(ids), _p(w), _s(stream)), "moe_route_ex")
    else:
        _ck(_route(_p(x), _p(w_router), _p(logit_offset), _p(sel_bias), _p(e2s), affinity, T, H, E, k,
                   _p(logits), _p(scratch), _p(ids), _p(w), _s(stream)), "moe_route")
    return (ids, w, logits) if return_logits else (ids, w)


@dataclass
class Groups:
    count: torch.Tensor
    offset: torch.Tensor
    rows: torch.Tensor
    pos: torch.Tensor
    act_e: torch.Tensor
    n_act: torch.Tensor


def permute(ids: torch.Tensor, E: int, dev_status: Optional[torch.Tensor] = None, stream=None,
            chunked: bool = True) -> Groups:
    n = ids.numel()
    i32 = dict(dtype=torch.int32, device=ids.device)
    g = Groups(torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(n, **i32), torch.empty(n, **i32),
               torch.empty(E, **i32), torch.empty(1, **i32))
    nb = int(_permute_scratch(n, E)) if chunked else 0
    scratch = torch.empty(max(nb // 4, 1), **i32) if nb else None
    _ck(_permute(_p(ids), n, E, _p(g.count), _p(g.offset), _p(g.rows), _p(g.pos), _p(g.act_e), _p(g.n_act),
                 _p(scratch), _p(dev_status), _s(stream)), "moe_permute")
    return g


@dataclass
class CacheState:
    e2s: torch.Tensor    # int32 [E]
    s2e: torch.Tensor    # int32 [S]
    prio: torch.Tensor   # uint32 [S], held as int32
    stamp: torch.Tensor  # uint32 [1], held as int32

    @staticmethod
    def from_slots(s2e, E: int, device="cuda") -> "CacheState":
        s2e_t = torch.as_tensor(s2e, dtype=torch.int32).clone().cpu()
        e2s = torch.full((E,), -1, dtype=torch.int32)
        for s, e in enumerate(s2e_t.tolist()):
            if e >= 0:
                e2s[e] = s
        S = s2e_t.numel()
        return CacheState(e2s.to(device), s2e_t.to(device), torch.zeros(S, dtype=torch.int32, device=device),
                          torch.zeros(1, dtype=torch.int32, device=device))

    def clone(self) -> "CacheState":
        return CacheState(self.e2s.clone(), self.s2e.clone(), self.prio.clone(), self.stamp.clone())


@dataclass
class ManageOut:
    miss_e: torch.Tensor
    miss_s: torch.Tensor
    n_miss: torch.Tensor
    hit_e: torch.Tensor
    n_hit: torch.Tensor
    sid: torch.Tensor


def cache_manage(ids: torch.Tensor, state: CacheState, policy: int, dev_status=None, stream=None) -> ManageOut:
    n = ids.numel()
    E, S = state.e2s.numel(), state.s2e.numel()
    lmax = min(n, E)
    i32 = dict(dtype=torch.int32, device=ids.device)
    o = ManageOut(torch.empty(lmax, **i32), torch.empty(lmax, **i32), torch.empty(1, **i32),
                  torch.empty(lmax, **i32), torch.empty(1, **i32), torch.empty(ids.shape, **i32))
    _ck(_manage(_p(ids), n, E, S, policy, _p(state.e2s), _p(state.s2e), _p(state.prio), _p(state.stamp),
                _p(o.miss_e), _p(o.miss_s), _p(o.n_miss), _p(o.hit_e), _p(o.n_hit), _p(o.sid), _p(dev_status),
                _s(stream)), "moe_cache_manage")
    return o


def cache_gather(host_slabs, pool, miss_e, miss_s, n_miss, max_miss, dev_status=None, stream=None) -> None:
    E = host_slabs.shape[0]
    S = pool.shape[0]
    slab_bytes = pool[0].numel() * pool.element_size()
    _ck(_gather(_p(host_slabs), _p(pool), slab_bytes, E, S, _p(miss_e), _p(miss_s), _p(n_miss), max_miss,
                _p(dev_status), _s(stream)), "moe_cache_gather")


def cache_count(ids, E, counts, dev_status=None, stream=None) -> None:
    """counts[e] += number of routings of expert e in ``ids`` (window counts for a re-pick)."""
    _ck(_count(_p(ids), ids.numel(), E, _p(counts), _p(dev_status), _s(stream)), "moe_cache_count")


@dataclass
class RepickResult:
    miss_e: torch.Tensor
    miss_s: torch.Tensor
    n_miss: torch.Tensor


def cache_repick(counts, state: "CacheState", stream=None) -> RepickResult:
    """Re-pick a STATIC pool's resident set from the window counts (clears them)."""
    E, S = state.e2s.numel(), state.s2e.numel()
    i32 = dict(dtype=torch.int32, device=counts.device)
    r = RepickResult(torch.empty(min(S, E), **i32), torch.empty(min(S, E), **i32), torch.zeros(1, **i32))
    _ck(_repick(_p(counts), E, S, _p(state.e2s), _p(state.s2e), _p(r.miss_e), _p(r.miss_s), _p(r.n_miss),
                _s(stream)), "moe_cache_repick")
    return r


def q8_slab_bytes(H: int, I: int) -> int:
    return int(_q8_slab(H, I))


def quantize_slabs(slabs: torch.Tensor, H: int, I: int, stream=None) -> torch.Tensor:
    """bf16 slabs [n][3HI] (device) -> W8A8 slabs uint8 [n][q8_slab_bytes] (device)."""
    n = slabs.shape[0]
    out = torch.empty(n, q8_slab_bytes(H, I), dtype=torch.uint8, device=slabs.device)
    _ck(_quantize(_p(slabs), n, H, I, _p(out), _s(stream)), "moe_quantize_slabs")
    return out


def expert_ffn_q8(x, k, I, E, offset, rows, list_e, n_list, max_list, pool_q, e2s=None, y=None, workspace=None,
                  dev_status=None, stream=None) -> torch.Tensor:
    T, H = x.shape
    if y is None:
        y = torch.zeros(T * k, H, dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty(int(_ffn_q8_ws(T, H, k, I)), dtype=torch.uint8, device=x.device)
    _ck(_ffn_q8(_p(x), T, H, I, k, E, _p(offset), _p(rows), _p(list_e), _p(n_list), max_list, _p(pool_q),
                pool_q.shape[0], _p(e2s), _p(y), _p(workspace), workspace.numel(), _p(dev_status), _s(stream)),
        "moe_expert_ffn_q8")
    return y


def ffn_workspace_bytes(T: int, H: int, k: int, I: int) -> int:
    return int(_ffn_ws(T, H, k, I))


def expert_ffn(x, k, I, E, offset, rows, list_e, n_list, max_list, pool, e2s=None, host_slabs=None,
               y=None, workspace=None, dev_status=None, stream=None) -> torch.Tensor:
    T, H = x.shape
    if y is None:
        y = torch.zeros(T * k, H, dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty(ffn_workspace_bytes(T, H, k, I), dtype=torch.uint8, device=x.device)
    _ck(_ffn(_p(x), T, H, I, k, E, _p(offset), _p(rows), _p(list_e), _p(n_list), max_list, _p(pool),
             pool.shape[0], _p(e2s),
             _p(host_slabs), _p(y), _p(workspace), workspace.numel(), _p(dev_status), _s(stream)),
        "moe_expert_ffn")
    return y


def combine(y, w, pos, T, k, E, ids=None, e2s=None, split=False, stream=None):
    H = y.shape[1]
    out = torch.empty(T, H, dtype=torch.bfloat16, device=y.device)
    out_res = torch.empty(T, H, dtype=torch.float32, device=y.device) if split else None
    out_miss = torch.empty(T, H, dtype=torch.float32, device=y.device) if split else None
    _ck(_combine(_p(y), _p(w), _p(pos), _p(ids), _p(e2s), T, k, H, E, int(split), _p(out), _p(out_res),
                 _p(out_miss), _s(stream)), "moe_combine")
    return (out, out_res, out_miss) if split else out


def layer_workspace_bytes(T, H, E, k, I, S) -> int:
    return int(_layer_ws(T, H, E, k, I, S))


# ---------------------------------------------------------------------------
# Whole layer
# ---------------------------------------------------------------------------

class SlotCachedMoELayer:
    """One layer's router, slot pool, host store, cache state and workspace.

    ``host_slabs`` (pinned host, [E][3HI] bf16) is the authoritative copy of
    every expert; ``pool`` ([S][3HI] bf16, device) holds the slot contents.
    In RESIDENT mode the pool holds every expert and no host store is needed.
    """

    def __init__(self, w_router, pool, k, I, mode, policy=POLICY_LRU, host_slabs=None, state=None,
                 logit_offset=None, sel_bias=None, max_tokens=64, side_stream=True, affinity=0.0,
                 route_flags=0, window_counts=None, quant=0, schedule=0, decode_kernels=0):
        self.w_router, self.pool, self.k, self.I = w_router, pool, k, I
        self.H, self.E = w_router.shape
        self.S = pool.shape[0]
        self.mode, self.policy = mode, policy
        self.host_slabs, self.state = host_slabs, state
        self.logit_offset, self.sel_bias = logit_offset, sel_bias
        self.affinity = float(affinity)
        self.route_flags = int(route_flags)
        self.window_counts = window_counts
        self.quant = int(quant)  # pool / host hold W8A8 slabs (quantize_slabs)
        self.schedule = int(schedule)  # SCHED_CHUNKS or SCHED_WAVES (GATHER steps larger than the pool)
        self.decode_kernels = int(decode_kernels)  # 0: persistent decode kernel where it applies, 1: separate
        dev = pool.device
        self.stats = torch.zeros(4, dtype=torch.int64, device=dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.max_tokens = max_tokens
        # zero-filled once: the persistent decode kernel's counters live at its start
        self.workspace = torch.zeros(layer_workspace_bytes(max_tokens, self.H, self.E, k, I, self.S),
                                     dtype=torch.uint8, device=dev)
        self.side = torch.cuda.Stream(device=dev) if side_stream else None

    def forward(self, x, out=None, ids=None, w=None, out_res=None, out_miss=None, stream=None, prof=None):
        T = x.shape[0]
        if T > self.max_tokens:
            raise ValueError(f"T={T} > max_tokens={self.max_tokens}")
        dev = x.device
        ids = torch.empty(T, self.k, dtype=torch.int32, device=dev) if ids is None else ids
        w = torch.empty(T, self.k, dtype=torch.float32, device=dev) if w is None else w
        out = torch.empty(T, self.H, dtype=torch.bfloat16, device=dev) if out is None else out
        if self.mode == MODE_ZERO_RETURN:
            out_res = torch.empty(T, self.H, dtype=torch.float32, device=dev) if out_res is None else out_res
            out_miss = torch.empty(T, self.H, dtype=torch.float32, device=dev) if out_miss is None else out_miss
        st = self.state
        a = LayerArgs(T, self.H, self.E, self.k, self.I, self.S, self.mode, self.policy,
                      x.data_ptr(), self.w_router.data_ptr(), _ptr(self.logit_offset), _ptr(self.sel_bias),
                      self.pool.data_ptr(), _ptr(self.host_slabs),
                      _ptr(st.e2s if st else None), _ptr(st.s2e if st else None),
                      _ptr(st.prio if st else None), _ptr(st.stamp if st else None),
                      ids.data_ptr(), w.data_ptr(), out.data_ptr(), _ptr(out_res), _ptr(out_miss),
                      self.stats.data_ptr(), self.dev_status.data_ptr(), self.workspace.data_ptr(),
                      self.workspace.numel(), ctypes.pointer(prof) if prof is not None else None, self.affinity,
                      self.route_flags, _ptr(self.window_counts), self.quant, self.schedule,
                      self.decode_kernels)
        main = torch.cuda.current_stream() if stream is None else stream
        # the library forks to and joins back from the side stream itself
        _ck(_layer(ctypes.byref(a), c_void_p(main.cuda_stream),
                   c_void_p(self.side.cuda_stream) if self.side is not None else None), "moe_layer_forward")
        res = {"out": out, "ids": ids, "w": w}
        if self.mode == MODE_ZERO_RETURN:
            res["out_res"], res["out_miss"] = out_res, out_miss
        return res

    def repick(self, stream=None) -> RepickResult:
        """Re-pick the resident set from ``window_counts`` and copy the new members into their slots."""
        r = cache_repick(self.window_counts, self.state, stream)
        cache_gather(self.host_slabs, self.pool, r.miss_e, r.miss_s, r.n_miss, r.miss_e.numel(), self.dev_status,
                     stream)
        return r


class LayerStack:
    """Several layers' forwards replayed as one CUDA graph.

    "Betelgeuse ... on an RTX 3060", "What it actually does under the hood":
    with hits resolved on the device and no host sync inside a layer, a whole
    decode pass over all layers replays as a single CUDA graph.  Each layer
    reads its own input buffer ``xs[l]`` and writes ``outs[l]``; the caller
    refreshes the inputs between replays.  Cache state and slot pools evolve
    on the device across replays.
    """

    def __init__(self, layers, T: int):
        self.layers = layers
        dev = layers[0].pool.device
        H = layers[0].H
        # one contiguous [L][T][H] input block, so a step's inputs arrive in one copy
        self.x_all = torch.zeros(len(layers), T, H, dtype=torch.bfloat16, device=dev)
        self.xs = list(self.x_all.unbind(0))
        self.out_all = torch.empty(len(layers), T, H, dtype=torch.bfloat16, device=dev)
        self.outs = list(self.out_all.unbind(0))
        self.ids = [torch.empty(T, l.k, dtype=torch.int32, device=dev) for l in layers]
        self.ws = [torch.empty(T, l.k, dtype=torch.float32, device=dev) for l in layers]
        self.graph = None

    def _run(self, prof=None):
        for i, l in enumerate(self.layers):
            l.forward(self.xs[i], out=self.outs[i], ids=self.ids[i], w=self.ws[i],
                      prof=None if prof is None else prof[i])

    def capture(self, prof=None):
        """Capture one pass over all layers (run one eager pass first to set up)."""
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, capture_error_mode="relaxed"):
            self._run(prof)
        return self.graph

    def replay(self):
        if self.graph is None:
            raise RuntimeError("capture() first")
        self.graph.replay()
