// The expert_cache_manage state machine of one call, on one thread block.
//
// "Porting vllm-expert-cache to NVIDIA GPUs", "What this package does": a
// manage call updates the hits' priorities, picks victims for the misses among
// the slots this call does not need (empty slots first, then ascending
// priority, then ascending slot) and remaps the loaded experts; "Prove it is
// correct before measuring": deterministic, no atomics, no order-dependent
// reduction.  Used by the manage kernel (cache.cu) and by the persistent
// decode kernel's fused gather step (decode.cu).
#pragma once

#include "internal.cuh"

namespace moe {

struct ManageCounts {
  int nm;  // missing experts
  int nh;  // hit experts
  int nl;  // missing experts that get a slot (all of them unless deferred)
};

// In shared memory: need[E] (1 where the call needs expert e) and the state e2s[E], s2e[S], prio[S], updated
// in place; work arrays mrank[E], hrank[E], cand[S], vict[S].  stamp is the call's new stamp.  With defer,
// the misses beyond the candidate slots are not loaded: they go, in ascending id, to def_e.  Outputs (any
// address space, each may be null except miss_e / miss_s): hit_e in ascending id, miss_e / miss_s for the
// nl loaded misses in ascending id (slot -1 under STATIC), ev_e: the expert each load evicted (-1 for an
// empty slot).  Every thread of the block calls this; blockDim.x is a multiple of 32.
__device__ __forceinline__ ManageCounts manage_block(int E, int S, int policy, bool defer, uint32_t stamp, int* need,
                                                     int* e2s, int* s2e, uint32_t* prio, int* mrank, int* hrank,
                                                     int* cand, int* vict, int32_t* hit_e, int32_t* miss_e,
                                                     int32_t* miss_s, int32_t* def_e, int32_t* ev_e,
                                                     int32_t* status) {
  __shared__ int tmp[33];
  __shared__ int s_nmiss, s_nhit;
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int s = tid; s < S; s += nt) vict[s] = -1;

  // Ranks of misses and hits in ascending expert order.
  int carry_m = 0, carry_h = 0;
  for (int e0 = 0; e0 < E; e0 += nt) {
    const int e = e0 + tid;
    const bool nd = e < E && need[e];
    const bool res = nd && e2s[e] >= 0 && e2s[e] < S;
    int tm, th;
    const int xm = block_exclusive_scan(nd && !res ? 1 : 0, tmp, &tm);
    const int xh = block_exclusive_scan(res ? 1 : 0, tmp, &th);
    if (e < E) {
      mrank[e] = nd && !res ? carry_m + xm : -1;
      hrank[e] = res ? carry_h + xh : -1;
    }
    carry_m += tm;
    carry_h += th;
  }
  if (tid == 0) {
    s_nmiss = carry_m;
    s_nhit = carry_h;
  }
  // Candidate slots: not holding an expert this call needs.
  int carry_c = 0;
  for (int s0 = 0; s0 < S; s0 += nt) {
    const int s = s0 + tid;
    int c = 0;
    if (s < S) {
      const int e = s2e[s];
      c = !(e >= 0 && e < E && need[e]);
      cand[s] = c;
    }
    int tc;
    block_exclusive_scan(c, tmp, &tc);
    carry_c += tc;
  }
  __syncthreads();
  const int nm = s_nmiss, nh = s_nhit;
  // misses that get a slot: all of them, or with deferral as many as there are candidates
  const int nl = (defer && policy != MOE_POLICY_STATIC) ? min(nm, carry_c) : nm;

  if (policy != MOE_POLICY_STATIC) {
    // Victim rank of each candidate: empty first (ascending slot), then
    // ascending prio, then ascending slot.
    for (int s = tid; s < S; s += nt) {
      if (!cand[s]) continue;
      const bool es = s2e[s] < 0;
      const uint32_t ps = prio[s];
      int r = 0;
      for (int q = 0; q < S; ++q) {
        if (!cand[q] || q == s) continue;
        const bool eq = s2e[q] < 0;
        bool before;
        if (eq != es)
          before = eq;
        else if (es)
          before = q < s;
        else
          before = prio[q] < ps || (prio[q] == ps && q < s);
        r += before;
      }
      if (r < nm) vict[r] = s;
    }
  }
  __syncthreads();

  // Apply.  Hit slots and victim slots are disjoint; evicted experts are
  // resident, missing experts are not, so no two writes touch one entry.
  for (int e = tid; e < E; e += nt) {
    if (hrank[e] >= 0) {
      const int s = e2s[e];
      if (policy == MOE_POLICY_LRU) prio[s] = stamp;
      else if (policy == MOE_POLICY_LFU) prio[s] = prio[s] + 1u;
      if (hit_e) hit_e[hrank[e]] = e;
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += nt) {
    const int r = mrank[e];
    if (r < 0) continue;
    if (r >= nl) {  // deferred to a later wave: stays cold
      def_e[r - nl] = e;
      continue;
    }
    miss_e[r] = e;
    if (policy == MOE_POLICY_STATIC) {
      miss_s[r] = -1;
      continue;
    }
    const int s = vict[r];
    miss_s[r] = s;
    if (s < 0) {  // cannot happen when the call fits the pool (checked on the host)
      set_status(status, MOE_DEV_BAD_SLOT);
      if (ev_e) ev_e[r] = -1;
      continue;
    }
    const int old = s2e[s];
    if (old >= 0 && old < E) e2s[old] = -1;
    if (ev_e) ev_e[r] = old >= 0 && old < E ? old : -1;
    s2e[s] = e;
    e2s[e] = s;
    prio[s] = policy == MOE_POLICY_LRU ? stamp : 1u;
  }
  __syncthreads();
  return ManageCounts{nm, nh, nl};
}

}  // namespace moe
