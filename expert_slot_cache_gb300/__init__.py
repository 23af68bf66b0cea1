"""Slot-cached MoE layer for GB300 (sm_103a): C-ABI library + thin binding.

The MoE layer forward -- route, permute, expert_cache_manage,
expert_cache_gather (or zero-return), grouped SwiGLU FFN, combine -- runs in
the CUDA kernels of ``libmoeslot.so`` (declared in ``include/moeslot.h``).
This package only marshals arguments.  Build the library first with
``python __graft_entry__.py`` (it calls build()).
"""
from .binding import (MODE_GATHER, MODE_RESIDENT, MODE_ZERO_RETURN, POLICY_LFU, POLICY_LRU,  # noqa: F401
                      POLICY_STATIC, CacheState, LayerArgs, MoeError, SlotCachedMoELayer, bias_table,
                      cache_gather, cache_manage, combine, expert_ffn, ffn_workspace_bytes, layer_workspace_bytes,
                      lib, permute, route, status_str, LayerStack, BIAS_GRADED, BIAS_FLAT, BIAS_HARD,
                      ROUTE_SIGMOID, ROUTE_DAMPED, cache_count, cache_repick,
                      q8_slab_bytes, quantize_slabs, expert_ffn_q8, SCHED_CHUNKS, SCHED_WAVES)
