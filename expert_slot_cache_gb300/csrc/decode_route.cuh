// Routing phases shared by the persistent decode kernels (bf16 and W8A8 experts).
//
// "Porting vllm-expert-cache to NVIDIA GPUs", "What this package does" (router
// logits in fp32, softmax over the picked experts, top-k with the optional
// selection bias) and "Betelgeuse ... on an RTX 3060", "What it actually does
// under the hood" (the routing of a decode step resolved on the device, inside
// the same graph as the experts).
//
//  route_logit_parts: units (128-row block b, 32 experts, token t) over all
//    warps of the grid; part_b = fma chain from 0 over the block's rows in
//    order -- the fp32 order of the router kernels; parts to lpart[b][t][e].
//  route_pick_group (after a grid-wide arrival on the parts): every CTA adds
//    the parts in block order (+ the offset), ranks the scores (top-k), forms
//    the weights and groups the step's routings by expert in shared memory.
//    From a few tokens up (a template parameter), CTA t routes token t alone
//    and publishes its ids and weights; every CTA reads them back after one
//    more grid-wide wait.
#pragma once

#include "fp32def.cuh"
#include "internal.cuh"
#include "tma.cuh"

namespace moe {

constexpr int kRStage = 8192 + 256;  // one warp's router staging: Wr [128][32] bf16 + x [128] bf16
constexpr int kRSpin = 1 << 20;      // polls of a grid-wide wait (about 1 us each) before it gives up: ~1 s

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void add_release(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Bounded wait until *p >= target; on giving up, flags the call and returns false.
__device__ __forceinline__ bool wait_count(const int32_t* p, int target, int32_t* status) {
  for (int i = 0; i < kRSpin; ++i) {
    if (ld_acquire(p) >= target) return true;
    __nanosleep(32);
  }
  set_status(status, MOE_DEV_TIMEOUT);
  return false;
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void cp_async_16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// sum_{j < J} p[j * stride] in j order, from 0; the loads of up to 16 parts are in flight together.
__device__ __forceinline__ float sum_parts(const float* p, size_t stride, int J) {
  float s = 0.f;
  for (int j0 = 0; j0 < J; j0 += 16) {
    float v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) v[u] = j0 + u < J ? __ldcg(p + (size_t)(j0 + u) * stride) : 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u)
      if (j0 + u < J) s += v[u];
  }
  return s;
}

struct RouteIO {
  const uint16_t* x;   // bf16 [T][H]
  const uint16_t* wr;  // bf16 [H][E]
  const float* off;    // fp32 [E] or NULL
  const float* bias;   // fp32 [E] or NULL
  const int32_t* e2s;  // [E] or NULL: live-cache affinity reads it
  float affinity;
  int rflags;
  int T, H, E, k;
  float* lpart;        // fp32 [H/128][T][E]
  float* logits;       // fp32 [T][E]
  int32_t* ids;        // [T][k]
  float* w;            // [T][k]
  int32_t* ctr_route;  // grid-wide arrival counter of the spread routing (zero on entry)
  int32_t* status;
};

// Shared-memory results of the routing: ids / weights in (t, j) order, per-expert counts, offsets
// and list index (-1: not routed), the list of routed experts, and the grouped order (rows: routing
// slot of position p; pos: position of routing slot i).
struct RouteSm {
  float* slog;  // [T][E] scratch
  float* ssc;   // [T][E] scratch
  int* ids;
  float* w;
  int* cnt;
  int* off;  // [E + 1]
  int* act;
  int* li;
  int* rows;
  int* pos;
  int* tmp;  // >= 33 ints
  int* nact;
  volatile int* abort_flag;
};

// Phase 1: this CTA's share of the router's block parts.  `stage` holds NT / 32 warps x kRStage bytes.
template <int NT>
__device__ __forceinline__ void route_logit_parts(const RouteIO& r, unsigned char* stage) {
  constexpr int NW = NT / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, G = gridDim.x;
  const int T = r.T, H = r.H, E = r.E;
  const int nblk = H / 128, neg = (E + 31) / 32;
  const int units = nblk * neg * T;
  // the warp's staging area: Wr rows [128][32 experts] bf16 (8 KB), then the x row (256 B)
  unsigned char* wst = stage + warp * kRStage;
  const uint16_t* ws16 = reinterpret_cast<const uint16_t*>(wst);
  // unit u goes to CTA u % G, so a small step's units spread over the grid before a CTA takes a second
  for (int u = warp * G + blockIdx.x; u < units; u += G * NW) {
    const int b = u % nblk, rest = u / nblk, eg = rest % neg, t = rest / neg;
    const int e0 = eg * 32, e = e0 + lane;
    for (int c = lane; c < 128 * 4; c += 32) {  // 16-byte pieces: row c / 4, experts e0 + 8 (c % 4) ..
      const int row = c >> 2, q = c & 3;
      if (e0 + 8 * q < E) cp_async_16(wst + row * 64 + q * 16, r.wr + (size_t)(b * 128 + row) * E + e0 + 8 * q);
    }
    if (lane < 16) cp_async_16(wst + 8192 + lane * 16, r.x + (size_t)t * H + b * 128 + 8 * lane);
    cp_async_wait_all();
    __syncwarp();
    const uint16_t* xs16 = ws16 + 4096;
    float acc = 0.f;
#pragma unroll 8
    for (int row = 0; row < 128; ++row) acc = fmaf(bf16_to_f32(xs16[row]), bf16_to_f32(ws16[row * 32 + lane]), acc);
    if (e < E) r.lpart[((size_t)b * T + t) * E + e] = acc;
    __syncwarp();
  }
}

// Phase 2 (every part of the logits in place): top-k, weights and the grouping by expert.  From
// SPREAD_T tokens up CTA t routes token t alone and publishes it (one more grid-wide wait); below that
// every CTA routes every token.
template <int NT, int SPREAD_T = 3>
__device__ __forceinline__ void route_pick_group(const RouteIO& r, const RouteSm& sm) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = r.T, E = r.E, k = r.k, n = T * k, nblk = r.H / 128;
  float* slog = sm.slog;
  float* ssc = sm.ssc;
  const bool spread = T >= SPREAD_T;
  const int t_lo = spread ? blockIdx.x : 0, t_hi = spread ? min((int)blockIdx.x + 1, T) : T;
  if (t_lo < t_hi) {
    for (int v = t_lo * E + tid; v < t_hi * E; v += NT) {
      const int e = v % E;
      float l = sum_parts(r.lpart + v, (size_t)T * E, nblk);  // part b of (t, e) at [b][t][e]
      if (r.off) l = l + r.off[e];
      slog[v] = l;
      // selection score: as the router's top-k (sigmoid router, bias, live-cache affinity)
      const float base = (r.rflags & MOE_ROUTE_SIGMOID) ? sigmoid32_def(l) : l;
      float sc = r.bias ? __fadd_rn(base, r.bias[e]) : base;
      if (r.e2s && r.affinity != 0.f && r.e2s[e] >= 0) sc = sc + r.affinity;
      ssc[v] = sc;
    }
    __syncthreads();
    if (spread || blockIdx.x == 0)
      for (int v = t_lo * E + tid; v < t_hi * E; v += NT) r.logits[v] = slog[v];
    // top-k by rank: expert e of token t is the r-th pick, r = the number of experts ranked before it
    // (higher score, or an equal score and a lower id); ranks below k are the picks, in order
    for (int v = t_lo * E + tid; v < t_hi * E; v += NT) {
      const int t = v / E, e = v - t * E;
      const float4* row4 = reinterpret_cast<const float4*>(ssc + t * E);  // E % 8 == 0
      const float se = ssc[v];
      int rk = 0;
#pragma unroll 4
      for (int f4 = 0; f4 < E / 4; ++f4) {
        const float4 q = row4[f4];
        const int f = 4 * f4;
        rk += (q.x > se) || (q.x == se && f < e);
        rk += (q.y > se) || (q.y == se && f + 1 < e);
        rk += (q.z > se) || (q.z == se && f + 2 < e);
        rk += (q.w > se) || (q.w == se && f + 3 < e);
      }
      if (rk < k) sm.ids[t * k + rk] = e;
    }
    __syncthreads();
    // the weights of token t over its k picks (the router's softmax, or its sigmoids normalised): one
    // warp per token, lane j for pick j; the sum runs in pick order from 0, as in the router's top-k
    // kernel, so both paths give the same weights bit for bit
    for (int t = t_lo + warp; t < t_hi; t += NW) {
      float zj = 0.f;
      if (lane < k) {
        const int e = sm.ids[t * k + lane];
        zj = slog[t * E + e];
        if (r.rflags & MOE_ROUTE_SIGMOID) zj = sigmoid32_def(zj);
        else if ((r.rflags & MOE_ROUTE_DAMPED) && r.bias) zj = zj + r.bias[e];
      }
      float mx = lane < k ? zj : -INFINITY;
#pragma unroll
      for (int d = 16; d; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(MOE_FULL_MASK, mx, d));
      const bool sig = (r.rflags & MOE_ROUTE_SIGMOID) != 0;
      const float num = lane < k ? (sig ? zj : expf(zj - mx)) : 0.f;
      float sum = 0.f;
      for (int j = 0; j < k; ++j) sum += __shfl_sync(MOE_FULL_MASK, num, j);
      if (lane < k) sm.w[t * k + lane] = num / sum;
    }
    __syncthreads();
    if (spread || blockIdx.x == 0)
      for (int i = t_lo * k + tid; i < t_hi * k; i += NT) {
        r.ids[i] = sm.ids[i];
        r.w[i] = sm.w[i];
      }
  }
  if (spread) {
    __syncthreads();
    if (tid == 0) {
      if (t_lo < t_hi) add_release(r.ctr_route, 1);
      if (!wait_count(r.ctr_route, T, r.status)) *sm.abort_flag = 1;
    }
    __syncthreads();
    for (int i = tid; i < n; i += NT) {
      sm.ids[i] = __ldcg(r.ids + i);
      sm.w[i] = __ldcg(r.w + i);
    }
    __syncthreads();
  }
  {
    int carry = 0, carry_act = 0;
    for (int e0 = 0; e0 < E; e0 += NT) {
      const int e = e0 + tid;
      int c = 0;
      if (e < E)
        for (int i = 0; i < n; ++i) c += sm.ids[i] == e;
      int tp;  // count in the low 16 bits, active flag in the high 16 (n <= 64, E <= 256: no carry)
      const int xp = block_exclusive_scan(c | ((c > 0 ? 1 : 0) << 16), sm.tmp, &tp);
      const int ex = xp & 0xffff, exa = xp >> 16, tot = tp & 0xffff, tota = tp >> 16;
      if (e < E) {
        sm.cnt[e] = c;
        sm.off[e] = carry + ex;
        sm.li[e] = c > 0 ? carry_act + exa : -1;
        if (c > 0) sm.act[carry_act + exa] = e;
      }
      carry += tot;
      carry_act += tota;
    }
    if (tid == 0) {
      sm.off[E] = carry;
      *sm.nact = carry_act;
    }
  }
  __syncthreads();
  if (tid < n) {
    const int e = sm.ids[tid];
    int rk = 0;
    for (int i = 0; i < tid; ++i) rk += sm.ids[i] == e;
    const int p = sm.off[e] + rk;
    sm.rows[p] = tid;
    sm.pos[tid] = p;
  }
  __syncthreads();
}

}  // namespace moe
