// Grouping of a small batch of routing slots by expert, done by one CTA of
// 256 threads: count[e], exclusive offset[e] (E + 1 entries), rows[] = slot
// indices t*k + j sorted by expert (ties by slot index, i.e. stable), pos[] =
// the inverse, act_e[] = experts with count > 0 in ascending id, n_act.
// ("Porting vllm-expert-cache to NVIDIA GPUs", "What this package does": the
// expert GEMM runs on tokens grouped per expert.)  Used by the permute kernel
// for small n, and by the top-k kernel when one CTA routes the whole batch.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kSmallN = 256;  // routing slots one CTA groups

struct PermOut {
  int32_t *count, *offset, *rows, *pos, *act_e, *n_act, *status;
};

// ids[0..n) must be complete and visible to the block; every thread of the block calls this.
__device__ __forceinline__ void permute_small_block(const int32_t* ids, int n, int E, const PermOut& o) {
  __shared__ int sid[kSmallN];
  __shared__ int soff[kMaxE];
  __shared__ int tmp[33];
  const int tid = threadIdx.x;
  if (tid < n) {
    int e = ids[tid];
    if (e < 0 || e >= E) {
      set_status(o.status, MOE_DEV_BAD_EXPERT);
      e = -1;
    }
    sid[tid] = e;
  }
  __syncthreads();
  int carry = 0, carry_act = 0;
  for (int e0 = 0; e0 < E; e0 += 256) {
    const int e = e0 + tid;
    int c = 0;
    if (e < E)
      for (int i = 0; i < n; ++i) c += sid[i] == e;
    int tot, tot_act;
    const int ex = block_exclusive_scan(c, tmp, &tot);
    const int exa = block_exclusive_scan(c > 0 ? 1 : 0, tmp, &tot_act);
    if (e < E) {
      soff[e] = carry + ex;
      o.offset[e] = carry + ex;
      o.count[e] = c;
      if (c > 0) o.act_e[carry_act + exa] = e;
    }
    carry += tot;
    carry_act += tot_act;
  }
  if (tid == 0) {
    o.offset[E] = carry;
    *o.n_act = carry_act;
  }
  __syncthreads();
  if (tid < n) {
    const int e = sid[tid];
    if (e >= 0) {
      int r = 0;
      for (int i = 0; i < tid; ++i) r += sid[i] == e;
      const int p = soff[e] + r;
      o.rows[p] = tid;
      o.pos[tid] = p;
    } else {
      o.pos[tid] = -1;
    }
  }
}

}  // namespace moe
