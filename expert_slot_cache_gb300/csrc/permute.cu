// Permute: group the flat routing slots t*k+j by expert (histogram, prefix
// sum, stable scatter).  One CTA of 1024 threads; any n.
//
// The grouped FFN needs every expert's token rows contiguous ("Porting
// vllm-expert-cache to NVIDIA GPUs", "What this package does": the fused MoE
// GEMM runs on grouped, slot-remapped ids).  Within an expert the order is
// ascending flat index, so the result is unique and checked bit for bit.
#include "common.cuh"

namespace moe {

constexpr int kPermThreads = 1024;

// Shared memory: cnt[E] | base[E] | wtab[32][E]
// wtab[w][e] = (tile << 16) | (number of ids == e in warp w of this tile)
__global__ void __launch_bounds__(kPermThreads) permute_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                               int32_t* __restrict__ count,
                                                               int32_t* __restrict__ offset,
                                                               int32_t* __restrict__ rows,
                                                               int32_t* __restrict__ pos,
                                                               int32_t* __restrict__ act_e,
                                                               int32_t* __restrict__ n_act,
                                                               int32_t* __restrict__ status) {
  extern __shared__ int perm_smem[];
  int* cnt = perm_smem;
  int* base = cnt + E;
  int* wtab = base + E;
  __shared__ int tmp[33];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int e = tid; e < E; e += kPermThreads) cnt[e] = 0;
  for (int i = tid; i < 32 * E; i += kPermThreads) wtab[i] = -1;
  __syncthreads();

  // Histogram (integer counts: the result does not depend on the order).
  for (int i = tid; i < n; i += kPermThreads) {
    const int e = ids[i];
    if (e < 0 || e >= E) {
      set_status(status, MOE_DEV_BAD_EXPERT);
      continue;
    }
    atomicAdd(&cnt[e], 1);
  }
  __syncthreads();

  // Exclusive prefix over experts, and the list of active experts.
  int carry = 0, carry_act = 0;
  for (int e0 = 0; e0 < E; e0 += kPermThreads) {
    const int e = e0 + tid;
    const int c = e < E ? cnt[e] : 0;
    int tot, tot_act;
    const int ex = block_exclusive_scan(c, tmp, &tot);
    const int exa = block_exclusive_scan(c > 0 ? 1 : 0, tmp, &tot_act);
    if (e < E) {
      base[e] = carry + ex;
      offset[e] = carry + ex;
      count[e] = c;
      if (c > 0) act_e[carry_act + exa] = e;
    }
    carry += tot;
    carry_act += tot_act;
  }
  if (tid == 0) {
    offset[E] = carry;
    *n_act = carry_act;
  }
  __syncthreads();

  // Stable scatter, one tile of 1024 ids at a time.
  for (int t0 = 0, tile = 0; t0 < n; t0 += kPermThreads, ++tile) {
    const int i = t0 + tid;
    int e = i < n ? ids[i] : -1;
    if (e >= E || e < 0) e = -1;
    const unsigned peers = __match_any_sync(MOE_FULL_MASK, e);
    const int wrank = __popc(peers & lanemask_lt());
    if (e >= 0 && lane == __ffs(peers) - 1) wtab[warp * E + e] = (tile << 16) | __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int pre = 0;
      for (int w2 = 0; w2 < warp; ++w2) {
        const int v = wtab[w2 * E + e];
        if ((v >> 16) == tile) pre += v & 0xffff;
      }
      const int p = base[e] + pre + wrank;
      rows[p] = i;
      pos[i] = p;
    } else if (i < n) {
      pos[i] = -1;
    }
    __syncthreads();
    for (int ee = tid; ee < E; ee += kPermThreads) {
      int s = 0;
      for (int w2 = 0; w2 < 32; ++w2) {
        const int v = wtab[w2 * E + ee];
        if ((v >> 16) == tile) s += v & 0xffff;
      }
      base[ee] += s;
    }
    __syncthreads();
  }
}

}  // namespace moe

using namespace moe;

extern "C" int moe_permute(const int32_t* ids, int n, int E, int32_t* count, int32_t* offset, int32_t* rows,
                           int32_t* pos, int32_t* act_e, int32_t* n_act, int32_t* dev_status,
                           moe_stream_t stream) {
  if (!ids || !count || !offset || !rows || !pos || !act_e || !n_act) return MOE_ERR_ARG;
  if (n < 1 || n >= (1 << 25) || E < 1 || E > kMaxE) return MOE_ERR_ARG;
  const size_t smem = (size_t)(2 * E + 32 * E) * sizeof(int);
  static bool attr_done[64] = {};
  MOE_CUDA_TRY(ensure_smem(permute_kernel, (int)((2 + 32) * kMaxE * sizeof(int)), attr_done));
  permute_kernel<<<1, kPermThreads, smem, (cudaStream_t)stream>>>(ids, n, E, count, offset, rows, pos, act_e,
                                                                   n_act, dev_status);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}
