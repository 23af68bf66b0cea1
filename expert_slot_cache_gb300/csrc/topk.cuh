// Top-k of one token by one warp, shared by the router kernels and the
// persistent decode kernel.
//
// Method: "Nudge, don't cut" (PGO-SGB), section "The method in five lines":
// pick the top-k by logit + bias; the weights are the router's own softmax
// over the k picked, from the unbiased logits.
#pragma once

#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "fp32def.cuh"

namespace moe {

// Sigmoid router score ("Nudge, don't cut", "The same idea on GLM-5.3-Flash":
// the bias is added after the sigmoid): sigmoid32_def (fp32def.cuh).

// ---------------------------------------------------------------------------
// One warp routes token t: k rounds of a warp-wide argmax over the scores, then the weights.
template <int NQ>
__device__ __forceinline__ void topk_token_impl(float* __restrict__ logits, const float* __restrict__ bias,
                                                const int32_t* __restrict__ e2s, float affinity, int E, int k,
                                                int rflags, int t, int warp, int lane,
                                                float (*sel_l)[kMaxK], int (*sel_i)[kMaxK],
                                                int32_t* __restrict__ ids, float* __restrict__ wout) {
  float* lrow = logits + (size_t)t * E;
  // the token's scores, loaded once: lane holds experts lane + 32q
  float sc[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const int e = lane + 32 * q;
    float v = 0.f;
    if (e < E) {
      const float base = (rflags & MOE_ROUTE_SIGMOID) ? sigmoid32_def(lrow[e]) : lrow[e];
      v = bias ? __fadd_rn(base, bias[e]) : base;
      if (e2s && affinity != 0.f && e2s[e] >= 0) v = v + affinity;  // live-cache affinity
    }
    sc[q] = v;
  }
  unsigned taken = 0;
  for (int j = 0; j < k; ++j) {
    float best = -INFINITY;
    int bi = INT_MAX;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int e = lane + 32 * q;
      if (e >= E || ((taken >> q) & 1u)) continue;
      const float sv = sc[q];
      if (bi == INT_MAX || sv > best || (sv == best && e < bi)) {
        best = sv;
        bi = e;
      }
    }
#pragma unroll
    for (int d = 16; d; d >>= 1) {
      const float ob = __shfl_xor_sync(MOE_FULL_MASK, best, d);
      const int oi = __shfl_xor_sync(MOE_FULL_MASK, bi, d);
      if (oi != INT_MAX && (bi == INT_MAX || ob > best || (ob == best && oi < bi))) {
        best = ob;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == 0) sel_i[warp][j] = bi;
  }
  __syncwarp();
  if (lane < k) {
    const int e = sel_i[warp][lane];
    float z = lrow[e];
    if (rflags & MOE_ROUTE_SIGMOID) z = sigmoid32_def(z);
    else if ((rflags & MOE_ROUTE_DAMPED) && bias) z = z + bias[e];  // damped: the bias enters the weights too
    sel_l[warp][lane] = z;
  }
  __syncwarp();
  if (lane == 0 && (rflags & MOE_ROUTE_SIGMOID)) {
    // the router's own probabilities of the picked k, normalised
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum += sel_l[warp][j];
    const size_t base = (size_t)t * k;
    for (int j = 0; j < k; ++j) {
      ids[base + j] = sel_i[warp][j];
      wout[base + j] = sel_l[warp][j] / sum;
    }
  } else if (lane == 0) {
    float mx = sel_l[warp][0];
    for (int j = 1; j < k; ++j) mx = fmaxf(mx, sel_l[warp][j]);
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum += expf(sel_l[warp][j] - mx);
    const size_t base = (size_t)t * k;
    for (int j = 0; j < k; ++j) {
      ids[base + j] = sel_i[warp][j];
      wout[base + j] = expf(sel_l[warp][j] - mx) / sum;
    }
  }
}


}  // namespace moe
