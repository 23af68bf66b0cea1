// Router (logits, soft-biased top-k, softmax weights) and the soft-bias table.
//
// Method: "Nudge, don't cut" (PGO-SGB), section "The method in five lines":
// experts outside the hot set get bias max(cap, ln(b / b_edge)); the top-k
// is picked by logit + bias; the weights are the router's own softmax over
// the k picked, from the unbiased logits.
#include <limits.h>
#include <math.h>

#include "common.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Bias table: one CTA of >= E threads (E <= 1024).  Runs once per layer.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) bias_table_kernel(const float* __restrict__ b, int E, int n_hot,
                                                          float cap, float* __restrict__ bias) {
  __shared__ float sb[kMaxE];
  __shared__ int shot[kMaxE];
  const int e = threadIdx.x;
  if (e < E) sb[e] = b[e];
  __syncthreads();
  if (e < E) {
    // rank among all experts by (brightness desc, id asc)
    const float be = sb[e];
    int r = 0;
    for (int f = 0; f < E; ++f) r += (sb[f] > be) || (sb[f] == be && f < e);
    shot[e] = r < n_hot;
  }
  __syncthreads();
  if (e < E) {
    float edge = INFINITY;
    for (int f = 0; f < E; ++f)
      if (shot[f]) edge = fminf(edge, sb[f]);
    float v = 0.f;
    if (!shot[e]) {
      const double be = sb[e];
      v = be <= 0.0 ? cap : (float)fmax((double)cap, log(be / (double)edge));
    }
    bias[e] = v;
  }
}

// ---------------------------------------------------------------------------
// Route kernel.  One CTA = TT tokens x all E experts, 256 threads.
//
// Logits: each output (t, e) is one fp32 chain acc = fma(x[t][h], Wr[h][e], acc)
// over h = 0..H-1 in order (the order the oracle follows).  A thread owns up
// to kMG chains.  When every chain of a thread has the same expert, one Wr
// load feeds all of them.
//
// Top-k: one warp per token.  k rounds of a warp-wide argmax over
// score = logit + bias (ties -> lower id); the winner is marked taken.
// ---------------------------------------------------------------------------
constexpr int kMG = 8;
constexpr int kRouteThreads = 256;

inline int route_tt(int E) {
  const int tt = (kRouteThreads * kMG) / E;
  int p = 1;
  while (p * 2 <= tt) p *= 2;
  return p;
}

template <bool kSameE>
__device__ __forceinline__ void route_logits(const uint16_t* __restrict__ xs, const uint16_t* __restrict__ wr,
                                             const float* __restrict__ off, int TT, int nt, int H, int E,
                                             float* __restrict__ ls) {
  constexpr int kPF = 8;  // router rows loaded ahead of the fma chains
  const int tid = threadIdx.x;
  int tm[kMG], em[kMG];
  bool vm[kMG];
#pragma unroll
  for (int m = 0; m < kMG; ++m) {
    const int o = tid + kRouteThreads * m;
    tm[m] = o / E;
    em[m] = o - tm[m] * E;
    vm[m] = (o < TT * E) && (tm[m] < nt);
    if (!vm[m]) {  // keep idle chains in bounds; their results are discarded
      tm[m] = 0;
      em[m] = 0;
    }
  }
  float acc[kMG];
#pragma unroll
  for (int m = 0; m < kMG; ++m) acc[m] = 0.f;

  bool any = false;
#pragma unroll
  for (int m = 0; m < kMG; ++m) any |= vm[m];
  if (!any) return;
  const int Hm = H - H % kPF;
  for (int h0 = 0; h0 < Hm; h0 += kPF) {
    if (kSameE) {
      // every chain of this thread has expert em[0]: one router load per h
      float wv[kPF];
#pragma unroll
      for (int u = 0; u < kPF; ++u) wv[u] = bf16_to_f32(__ldg(wr + (size_t)(h0 + u) * E + em[0]));
#pragma unroll
      for (int u = 0; u < kPF; ++u)
#pragma unroll
        for (int m = 0; m < kMG; ++m) acc[m] = fmaf(bf16_to_f32(xs[tm[m] * H + h0 + u]), wv[u], acc[m]);
    } else {
      float wv[kPF][kMG];
#pragma unroll
      for (int u = 0; u < kPF; ++u)
#pragma unroll
        for (int m = 0; m < kMG; ++m)
          wv[u][m] = vm[m] ? bf16_to_f32(__ldg(wr + (size_t)(h0 + u) * E + em[m])) : 0.f;
#pragma unroll
      for (int u = 0; u < kPF; ++u)
#pragma unroll
        for (int m = 0; m < kMG; ++m) acc[m] = fmaf(bf16_to_f32(xs[tm[m] * H + h0 + u]), wv[u][m], acc[m]);
    }
  }
  for (int h = Hm; h < H; ++h) {
#pragma unroll
    for (int m = 0; m < kMG; ++m)
      acc[m] = fmaf(bf16_to_f32(xs[tm[m] * H + h]), bf16_to_f32(__ldg(wr + (size_t)h * E + em[m])), acc[m]);
  }
#pragma unroll
  for (int m = 0; m < kMG; ++m) {
    if (vm[m]) ls[tm[m] * E + em[m]] = off ? acc[m] + off[em[m]] : acc[m];
  }
}

__global__ void __launch_bounds__(kRouteThreads) route_kernel(const uint16_t* __restrict__ x,
                                                              const uint16_t* __restrict__ wr,
                                                              const float* __restrict__ off,
                                                              const float* __restrict__ bias, int T, int H,
                                                              int E, int k, int TT, int same_e,
                                                              float* __restrict__ logits,
                                                              int32_t* __restrict__ ids, float* __restrict__ wout) {
  extern __shared__ __align__(16) unsigned char route_smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(route_smem);                 // [TT][H] bf16
  float* ls = reinterpret_cast<float*>(route_smem + (size_t)TT * H * 2);  // [TT][E]
  __shared__ float sel_l[kRouteThreads / 32][kMaxK];
  __shared__ int sel_i[kRouteThreads / 32][kMaxK];

  const int t0 = blockIdx.x * TT;
  const int nt = min(TT, T - t0);
  for (int i = threadIdx.x; i < nt * H; i += blockDim.x) xs[i] = x[(size_t)t0 * H + i];
  for (int i = nt * H + threadIdx.x; i < TT * H; i += blockDim.x) xs[i] = 0;
  __syncthreads();

  if (same_e)
    route_logits<true>(xs, wr, off, TT, nt, H, E, ls);
  else
    route_logits<false>(xs, wr, off, TT, nt, H, E, ls);
  __syncthreads();

  if (logits) {
    for (int i = threadIdx.x; i < nt * E; i += blockDim.x) logits[(size_t)t0 * E + i] = ls[i];
  }

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int t = warp; t < nt; t += kRouteThreads / 32) {
    const float* lrow = ls + t * E;
    unsigned taken = 0;
    for (int j = 0; j < k; ++j) {
      float best = -INFINITY;
      int bi = INT_MAX;
      for (int q = 0; lane + 32 * q < E; ++q) {
        if ((taken >> q) & 1u) continue;
        const int e = lane + 32 * q;
        const float s = bias ? lrow[e] + bias[e] : lrow[e];
        if (bi == INT_MAX || s > best || (s == best && e < bi)) {
          best = s;
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
      if (lane == 0) {
        sel_i[warp][j] = bi;
        sel_l[warp][j] = lrow[bi];
      }
    }
    __syncwarp();
    if (lane == 0) {
      float mx = sel_l[warp][0];
      for (int j = 1; j < k; ++j) mx = fmaxf(mx, sel_l[warp][j]);
      float sum = 0.f;
      for (int j = 0; j < k; ++j) sum += expf(sel_l[warp][j] - mx);
      const size_t base = (size_t)(t0 + t) * k;
      for (int j = 0; j < k; ++j) {
        ids[base + j] = sel_i[warp][j];
        wout[base + j] = expf(sel_l[warp][j] - mx) / sum;
      }
    }
    __syncwarp();
  }
}

}  // namespace moe

using namespace moe;

extern "C" int moe_bias_table(const float* b, int E, int n_hot, float cap, float* bias, moe_stream_t stream) {
  if (!b || !bias || E < 1 || E > kMaxE || n_hot < 1 || n_hot > E) return MOE_ERR_ARG;
  const int threads = ((E + 31) / 32) * 32;
  bias_table_kernel<<<1, threads, 0, (cudaStream_t)stream>>>(b, E, n_hot, cap, bias);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

extern "C" int moe_route(const void* x, const void* w_router, const float* logit_offset, const float* sel_bias,
                         int T, int H, int E, int k, float* logits, int32_t* ids, float* w, moe_stream_t stream) {
  if (!x || !w_router || !ids || !w) return MOE_ERR_ARG;
  if (T < 1 || H < 1 || E < 1 || E > kMaxE || k < 1 || k > kMaxK || k > E) return MOE_ERR_ARG;
  constexpr int kSmemCap = 160 * 1024;
  int sms = 0, dev = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  // Enough CTAs to cover the SMs first, then up to kMG chains per thread.
  int TT = route_tt(E);
  while (TT > 1 && (T + TT - 1) / TT < sms) TT /= 2;
  auto smem_of = [&](int tt) { return (size_t)tt * H * 2 + (size_t)tt * E * 4; };
  while (TT > 1 && smem_of(TT) > (size_t)kSmemCap) TT /= 2;
  if (smem_of(TT) > (size_t)kSmemCap) return MOE_ERR_ARG;
  const int same_e = (kRouteThreads % E == 0) && (TT * E == kRouteThreads * kMG);
  static bool attr_done[64] = {};
  MOE_CUDA_TRY(ensure_smem(route_kernel, kSmemCap, attr_done));
  const int grid = (T + TT - 1) / TT;
  route_kernel<<<grid, kRouteThreads, smem_of(TT), (cudaStream_t)stream>>>(
      (const uint16_t*)x, (const uint16_t*)w_router, logit_offset, sel_bias, T, H, E, k, TT, same_e, logits, ids,
      w);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}
