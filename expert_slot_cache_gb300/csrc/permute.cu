// Permute: group the flat routing slots t*k+j by expert (histogram, prefix
// sum, stable scatter).  One CTA of 1024 threads; any n.
//
// The grouped FFN needs every expert's token rows contiguous ("Porting
// vllm-expert-cache to NVIDIA GPUs", "What this package does": the fused MoE
// GEMM runs on grouped, slot-remapped ids).  Within an expert the order is
// ascending flat index, so the result is unique and checked bit for bit.
#include "common.cuh"
#include "perm_small.cuh"

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
  pdl_trigger();
  pdl_wait();  // launched as a dependent: the ids (or the previous permute step) are complete
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

// ---------------------------------------------------------------------------
// Large n: the same grouping in three launches over chunks of 1024 ids.
//   hist:    hist[p][e] = ids == e in chunk p
//   scan:    offset/count/act_e, and base[p][e] = offset[e] + sum_{p'<p} hist[p'][e]
//   scatter: chunk p places its ids stably after base[p][e]
// Within a chunk the order is the flat index and chunks are taken in order,
// so rows/pos are identical to the one-CTA kernel's.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPermThreads) permute_hist_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                                    int32_t* __restrict__ hist,
                                                                    int32_t* __restrict__ status) {
  pdl_trigger();
  pdl_wait();  // launched as a dependent: the ids (or the previous permute step) are complete
  extern __shared__ int ph_smem[];
  const int p = blockIdx.x, tid = threadIdx.x;
  for (int e = tid; e < E; e += kPermThreads) ph_smem[e] = 0;
  __syncthreads();
  const int i = p * kPermThreads + tid;
  if (i < n) {
    const int e = ids[i];
    if (e < 0 || e >= E) set_status(status, MOE_DEV_BAD_EXPERT);
    else atomicAdd(&ph_smem[e], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kPermThreads) hist[(size_t)p * E + e] = ph_smem[e];
}

__global__ void __launch_bounds__(kPermThreads) permute_scan_kernel(const int32_t* __restrict__ hist, int P, int E,
                                                                    int32_t* __restrict__ count,
                                                                    int32_t* __restrict__ offset,
                                                                    int32_t* __restrict__ act_e,
                                                                    int32_t* __restrict__ n_act,
                                                                    int32_t* __restrict__ base) {
  pdl_trigger();
  pdl_wait();  // launched as a dependent: the ids (or the previous permute step) are complete
  __shared__ int tmp[33];
  const int tid = threadIdx.x;
  int carry = 0, carry_act = 0;
  for (int e0 = 0; e0 < E; e0 += kPermThreads) {
    const int e = e0 + tid;
    int c = 0;
    if (e < E)
      for (int p = 0; p < P; ++p) c += hist[(size_t)p * E + e];
    int tot, tot_act;
    const int ex = block_exclusive_scan(c, tmp, &tot);
    const int exa = block_exclusive_scan(c > 0 ? 1 : 0, tmp, &tot_act);
    if (e < E) {
      const int off = carry + ex;
      offset[e] = off;
      count[e] = c;
      if (c > 0) act_e[carry_act + exa] = e;
      int run = off;
      for (int p = 0; p < P; ++p) {
        base[(size_t)p * E + e] = run;
        run += hist[(size_t)p * E + e];
      }
    }
    carry += tot;
    carry_act += tot_act;
  }
  if (tid == 0) {
    offset[E] = carry;
    *n_act = carry_act;
  }
}

__global__ void __launch_bounds__(kPermThreads) permute_scatter_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                                       const int32_t* __restrict__ base,
                                                                       int32_t* __restrict__ rows,
                                                                       int32_t* __restrict__ pos) {
  pdl_trigger();
  pdl_wait();  // launched as a dependent: the ids (or the previous permute step) are complete
  extern __shared__ int ps_smem[];  // wtab[32][E]
  const int p = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* wtab = ps_smem;
  for (int v = tid; v < 32 * E; v += kPermThreads) wtab[v] = 0;
  __syncthreads();
  const int i = p * kPermThreads + tid;
  int e = i < n ? ids[i] : -1;
  if (e >= E || e < 0) e = -1;
  const unsigned peers = __match_any_sync(MOE_FULL_MASK, e);
  const int wrank = __popc(peers & lanemask_lt());
  if (e >= 0 && lane == __ffs(peers) - 1) wtab[warp * E + e] = __popc(peers);
  __syncthreads();
  if (e >= 0) {
    int pre = 0;
    for (int w2 = 0; w2 < warp; ++w2) pre += wtab[w2 * E + e];
    const int q = base[(size_t)p * E + e] + pre + wrank;
    rows[q] = i;
    pos[i] = q;
  } else if (i < n) {
    pos[i] = -1;
  }
}

}  // namespace moe

using namespace moe;

namespace moe {
// Small n (decode batches): one CTA, stable rank by counting (perm_small.cuh).
__global__ void __launch_bounds__(256) permute_small_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                            const PermOut o) {
  pdl_trigger();
  pdl_wait();  // launched as a dependent: the ids (or the previous permute step) are complete
  permute_small_block(ids, n, E, o);
}
}  // namespace moe

namespace moe {
int launch_permute(const int32_t* ids, int n, int E, int32_t* count, int32_t* offset, int32_t* rows, int32_t* pos,
                   int32_t* act_e, int32_t* n_act, int32_t* dev_status, int32_t* scratch, cudaStream_t s) {
  const int P = (n + kPermThreads - 1) / kPermThreads;
  if (n <= kSmallN) {
    const PermOut o{count, offset, rows, pos, act_e, n_act, dev_status};
    MOE_CUDA_TRY(launch_pdl(permute_small_kernel, dim3(1), dim3(256), 0, s, ids, n, E, o));
    return MOE_OK;
  }
  if (P > 1 && scratch) {
    int32_t* hist = scratch;
    int32_t* base = scratch + (size_t)P * E;
    static bool d1[64] = {}, d3[64] = {};
    MOE_CUDA_TRY(ensure_smem(permute_hist_kernel, (int)(kMaxE * sizeof(int)), d1));
    MOE_CUDA_TRY(ensure_smem(permute_scatter_kernel, (int)(32 * kMaxE * sizeof(int)), d3));
    MOE_CUDA_TRY(launch_pdl(permute_hist_kernel, dim3(P), dim3(kPermThreads), (size_t)E * sizeof(int), s, ids, n, E,
                            hist, dev_status));
    MOE_CUDA_TRY(launch_pdl(permute_scan_kernel, dim3(1), dim3(kPermThreads), 0, s, (const int32_t*)hist, P, E, count,
                            offset, act_e, n_act, base));
    MOE_CUDA_TRY(launch_pdl(permute_scatter_kernel, dim3(P), dim3(kPermThreads), (size_t)32 * E * sizeof(int), s, ids,
                            n, E, (const int32_t*)base, rows, pos));
    return MOE_OK;
  }
  const size_t smem = (size_t)(2 * E + 32 * E) * sizeof(int);
  static bool attr_done[64] = {};
  MOE_CUDA_TRY(ensure_smem(permute_kernel, (int)((2 + 32) * kMaxE * sizeof(int)), attr_done));
  MOE_CUDA_TRY(launch_pdl(permute_kernel, dim3(1), dim3(kPermThreads), smem, s, ids, n, E, count, offset, rows, pos,
                          act_e, n_act, dev_status));
  return MOE_OK;
}
}  // namespace moe

extern "C" size_t moe_permute_scratch_bytes(int n, int E) {
  if (n < 1 || E < 1) return 0;
  const size_t P = ((size_t)n + kPermThreads - 1) / kPermThreads;
  return P > 1 ? 2 * P * (size_t)E * sizeof(int32_t) : 0;
}

extern "C" int moe_permute(const int32_t* ids, int n, int E, int32_t* count, int32_t* offset, int32_t* rows,
                           int32_t* pos, int32_t* act_e, int32_t* n_act, int32_t* scratch, int32_t* dev_status,
                           moe_stream_t stream) {
  if (!ids || !count || !offset || !rows || !pos || !act_e || !n_act) return MOE_ERR_ARG;
  if (n < 1 || n >= (1 << 25) || E < 1 || E > kMaxE) return MOE_ERR_ARG;
  return launch_permute(ids, n, E, count, offset, rows, pos, act_e, n_act, dev_status, scratch, (cudaStream_t)stream);
}
