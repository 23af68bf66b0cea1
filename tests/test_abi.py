"""The C-ABI library loads, exports every declared entry point, and rejects
bad arguments on the host (no GPU needed: these paths return before any
CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    b = __graft_entry__._build_module()
    b.build()
    return ctypes.CDLL(b.LIB)


def _declared():
    src = open(os.path.join(ROOT, "include", "moeslot.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    lib.moe_status_str.restype = ctypes.c_char_p
    for code in range(0, -7, -1):
        assert lib.moe_status_str(code) and lib.moe_status_str(code) != b"unknown status"


def test_host_side_argument_errors(lib):
    buf = (ctypes.c_int32 * 64)()
    p = ctypes.cast(buf, ctypes.c_void_p)
    null = ctypes.c_void_p(0)
    # NULL inputs
    f0 = ctypes.c_float(0.0)
    assert lib.moe_route(null, null, null, null, null, f0, 4, 256, 16, 2, null, null, null, null, null) == -1
    # k > E
    assert lib.moe_route(p, p, null, null, null, f0, 4, 256, 8, 9, p, null, p, p, null) == -1
    # logits buffer is required
    assert lib.moe_route(p, p, null, null, null, f0, 4, 256, 16, 2, null, null, p, p, null) == -1
    # a step larger than the pool when the policy can evict
    assert lib.moe_cache_manage(p, 65, 128, 64, 0, p, p, p, p, p, p, p, null, null, null, null, null) == -2
    # bad policy
    assert lib.moe_cache_manage(p, 8, 128, 64, 7, p, p, p, p, p, p, p, null, null, null, null, null) == -1
    # slab not a 16-byte multiple
    assert lib.moe_cache_gather(p, p, ctypes.c_size_t(24), 4, 2, p, p, p, 2, null, null) == -3
    # shapes the FFN does not take (H % 64 != 0)
    assert lib.moe_expert_ffn(p, 4, 100, 128, 2, 16, p, p, p, p, 4, p, 16, null, null, p, p,
                              ctypes.c_size_t(1 << 20), null, null) == -1


def test_workspace_sizes(lib):
    lib.moe_layer_workspace_bytes.restype = ctypes.c_size_t
    lib.moe_ffn_workspace_bytes.restype = ctypes.c_size_t
    ws = lib.moe_layer_workspace_bytes(64, 2048, 128, 8, 768, 64)
    # h (n*I fp32) and y (n*H fp32) dominate
    assert ws >= 4 * 512 * (768 + 2048)
    # decode-sized groups add the stream path's buffers: partial sums in two
    # equal halves, each the larger of (gate/up parts x n x 2I) and (down
    # parts x n x H) fp32, parts per expert = 64 MiB // (n * N * 4) clamped to
    # [3, 160]; then x grouped by expert (bf16 n x H) and h (bf16 n x I)
    n = 512
    jg, jd = max(3, min((64 << 20) // (n * 1536 * 4), 160)), max(3, min((64 << 20) // (n * 2048 * 4), 160))
    half = max(jg * n * 1536 * 4, jd * n * 2048 * 4)
    stream = 2 * half + n * 2048 * 2 + n * 768 * 2
    assert lib.moe_ffn_workspace_bytes(64, 2048, 8, 768) == 4 * 512 * 768 + 256 + stream
    # the tensor-core path adds bf16 grouped x and bf16 h
    assert lib.moe_ffn_workspace_bytes(4096, 2048, 8, 768) == 4 * 32768 * 768 + 2 * 32768 * (2048 + 768)


def test_layer_forward_rejects_bad_arguments_on_the_host():
    """moe_layer_forward checks shapes, buffers and mode/policy pairs before any CUDA call: gather
    evicts (LRU or LFU), zero-return keeps a STATIC pool, a resident pool smaller than E needs a slot
    table, and the quantised path is on or off."""
    import expert_slot_cache_gb300.binding as b
    buf = (ctypes.c_int32 * 64)()
    p = ctypes.cast(buf, ctypes.c_void_p).value

    def args(**kw):
        a = b.LayerArgs()
        a.T, a.H, a.E, a.k, a.I, a.S = 4, 256, 16, 2, 128, 16
        for f in ("x", "w_router", "pool", "ids", "w", "out", "workspace"):
            setattr(a, f, p)
        for key, val in kw.items():
            setattr(a, key, val)
        return a

    def call(a):
        return b._layer(ctypes.byref(a), None, None)

    assert call(args(mode=9)) == -1                    # no such mode
    assert call(args(mode=1, policy=2)) == -1          # gather with a pool that never evicts
    assert call(args(mode=2, policy=0)) == -1          # zero-return with an evicting policy
    assert call(args(mode=1, policy=0)) == -1          # gather without cache state / host store
    assert call(args(S=8)) == -1                       # resident, fewer slots than experts, no table
    assert call(args(T=0)) == -1
    assert call(args(k=17)) == -1                      # top-k above the largest supported
    assert call(args(H=100)) == -1                     # H not a multiple of 64
    assert call(args(x=None)) == -1
    assert call(args(quant=3)) == -1
    assert b._layer(None, None, None) == -1
    assert b._layer_ws(0, 2048, 128, 8, 768, 64) == 0  # no workspace for an empty step
