// expert_cache_manage and expert_cache_gather.
//
// "Porting vllm-expert-cache to NVIDIA GPUs", "What this package does": per
// MoE layer and step, manage picks victims among the slots this step does not
// need and emits a miss list; gather copies the missing experts host-to-slot;
// routing ids are remapped to slot space.  "Prove it is correct before
// measuring": the manager must stay deterministic (no atomics, no
// order-dependent reduction), the gather reads host memory from the device,
// and per-expert slabs are 16-byte multiples.  "Betelgeuse ... on an RTX
// 3060", "What it actually does under the hood": hits are resolved by an
// in-stream kernel on the device, with no host synchronisation.
#include <algorithm>

#include "internal.cuh"
#include "manage_core.cuh"

namespace moe {

constexpr int kManageThreads = 1024;
constexpr int kMaxS = 4096;

// kept list of a manage call: the experts of keep.in0 and keep.in1 that none of the call's nev loads
// evicted (keep.ev_e[0 .. nev), written by this block before the call), ascending id.  flag: E ints of
// shared memory; every thread of the block calls it.
__device__ void write_kept(int* flag, int E, const ManageKeep& keep, int nev) {
  __shared__ int ktmp[33];
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) flag[e] = 0;
  __syncthreads();
  const int n0 = keep.n_in0 ? *keep.n_in0 : 0, n1 = keep.n_in1 ? *keep.n_in1 : 0;
  for (int i = tid; i < n0; i += blockDim.x) {
    const int e = keep.in0[i];
    if (e >= 0 && e < E) flag[e] = 1;
  }
  for (int i = tid; i < n1; i += blockDim.x) {
    const int e = keep.in1[i];
    if (e >= 0 && e < E) flag[e] = 1;
  }
  __syncthreads();
  for (int r = tid; r < nev; r += blockDim.x) {
    const int e = keep.ev_e[r];
    if (e >= 0 && e < E) flag[e] = 0;
  }
  __syncthreads();
  int carry = 0;
  for (int e0 = 0; e0 < E; e0 += blockDim.x) {
    const int e = e0 + tid;
    const int f = e < E ? flag[e] : 0;
    int tot;
    const int x = block_exclusive_scan(f, ktmp, &tot);
    if (f) keep.kept_e[carry + x] = e;
    carry += tot;
  }
  if (tid == 0) *keep.n_kept = carry;
}

// Shared memory (dynamic): need[E] | e2s[E] | mrank[E] | hrank[E] | s2e[S] | prio[S] | cand[S] | vict[S]
//
// ids[0 .. n) are the call's routing ids.  With n_dev the call reads
// ids[n_off .. n_off + m) instead, m = clamp(*n_dev - n_off, 0, n): a batch of
// a device-side list (the later waves of the expert-wave schedule); m = 0 is
// no call (nothing changes, stamp included).  With def_e (wave 0 of that
// schedule) the misses beyond the available victims are not loaded: they go,
// in ascending id, to def_e / *n_def, and *n_miss counts the loaded ones.
__global__ void __launch_bounds__(kManageThreads) manage_kernel(
    const int32_t* __restrict__ ids, int n, const int32_t* __restrict__ n_dev, int n_off, int E, int S, int policy,
    int32_t* __restrict__ e2s_g, int32_t* __restrict__ s2e_g, uint32_t* __restrict__ prio_g,
    uint32_t* __restrict__ stamp_g, int32_t* __restrict__ miss_e, int32_t* __restrict__ miss_s,
    int32_t* __restrict__ n_miss, int32_t* __restrict__ hit_e, int32_t* __restrict__ n_hit,
    int32_t* __restrict__ sid, int32_t* __restrict__ def_e, int32_t* __restrict__ n_def,
    int32_t* __restrict__ sub_n, const SubBatches sub, const ManageKeep keep, int64_t* __restrict__ stats,
    int32_t* __restrict__ status) {
  extern __shared__ int man_smem[];
  int* need = man_smem;
  int* e2s = need + E;
  int* mrank = e2s + E;
  int* hrank = mrank + E;
  int* s2e = hrank + E;
  uint32_t* prio = reinterpret_cast<uint32_t*>(s2e + S);
  int* cand = reinterpret_cast<int*>(prio + S);
  int* vict = cand + S;
  const int tid = threadIdx.x;
  if (n_dev) {
    n = min(max(*n_dev - n_off, 0), n);
    ids += n_off;
    if (n == 0) {
      if (tid == 0) {
        *n_miss = 0;
        if (n_hit) *n_hit = 0;
        if (n_def) *n_def = 0;
        if (sub_n)
          for (int b = 0; b < sub.n; ++b) sub_n[b] = 0;
      }
      if (keep.kept_e) write_kept(mrank, E, keep, 0);  // nothing evicted
      return;
    }
  }

  for (int e = tid; e < E; e += kManageThreads) {
    need[e] = 0;
    e2s[e] = e2s_g[e];
  }
  for (int s = tid; s < S; s += kManageThreads) {
    s2e[s] = s2e_g[s];
    prio[s] = prio_g[s];
  }
  __syncthreads();
  for (int i = tid; i < n; i += kManageThreads) {
    const int e = ids[i];
    if (e < 0 || e >= E) {
      set_status(status, MOE_DEV_BAD_EXPERT);
      continue;
    }
    need[e] = 1;  // same value from every writer
  }
  __syncthreads();
  const uint32_t stamp = *stamp_g + 1u;
  const ManageCounts mc = manage_block(E, S, policy, def_e != nullptr, stamp, need, e2s, s2e, prio, mrank, hrank,
                                       cand, vict, hit_e, miss_e, miss_s, def_e, keep.ev_e, status);
  const int nm = mc.nm, nl = mc.nl;
  __syncthreads();
  if (keep.kept_e) write_kept(mrank, E, keep, nl);  // mrank is free from here on
  for (int e = tid; e < E; e += kManageThreads) e2s_g[e] = e2s[e];
  for (int s = tid; s < S; s += kManageThreads) {
    s2e_g[s] = s2e[s];
    prio_g[s] = prio[s];
  }
  if (sid) {
    for (int i = tid; i < n; i += kManageThreads) {
      const int e = ids[i];
      sid[i] = (e >= 0 && e < E) ? e2s[e] : -1;
    }
  }
  if (tid == 0) {
    *stamp_g = stamp;
    *n_miss = nl;
    if (n_hit) *n_hit = mc.nh;
    if (n_def) *n_def = nm - nl;
    if (sub_n)
      for (int b = 0; b < sub.n; ++b) sub_n[b] = min(max(nl - sub.off[b], 0), sub.off[b + 1] - sub.off[b]);
    if (stats) {
      stats[0] += nl;
      stats[1] += 1;
    }
  }
}

// Gather: each (miss, chunk) work item copies one chunk of a slab with
// 16-byte loads from mapped pinned host memory.  Grid-stride over items; the
// number of misses is read on the device.
constexpr int kGatherThreads = 256;
constexpr int kGatherUnroll = 8;
constexpr int kGatherChunkVec = kGatherThreads * kGatherUnroll;  // 32 KB per item

__global__ void __launch_bounds__(kGatherThreads) gather_kernel(const uint4* __restrict__ host,
                                                                uint4* __restrict__ pool, size_t slab_vec,
                                                                int E, int S, const int32_t* __restrict__ miss_e,
                                                                const int32_t* __restrict__ miss_s,
                                                                const int32_t* __restrict__ n_miss,
                                                                int64_t* __restrict__ stats,
                                                                int32_t* __restrict__ status) {
  const int nm = *n_miss;
  const size_t chunks = (slab_vec + kGatherChunkVec - 1) / kGatherChunkVec;
  const size_t items = (size_t)nm * chunks;
  for (size_t it = blockIdx.x; it < items; it += gridDim.x) {
    const int m = (int)(it / chunks);
    const size_t c = it - (size_t)m * chunks;
    const int e = miss_e[m], s = miss_s[m];
    if (e < 0 || e >= E || s < 0 || s >= S) {
      if (threadIdx.x == 0) set_status(status, e < 0 || e >= E ? MOE_DEV_BAD_EXPERT : MOE_DEV_BAD_SLOT);
      continue;
    }
    const uint4* src = host + (size_t)e * slab_vec + c * kGatherChunkVec;
    uint4* dst = pool + (size_t)s * slab_vec + c * kGatherChunkVec;
    const size_t lim = min((size_t)kGatherChunkVec, slab_vec - c * kGatherChunkVec);
    uint4 v[kGatherUnroll];
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      const size_t j = threadIdx.x + (size_t)u * kGatherThreads;
      if (j < lim) v[u] = ldg_stream(src + j);
    }
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      const size_t j = threadIdx.x + (size_t)u * kGatherThreads;
      if (j < lim) dst[j] = v[u];
    }
  }
  if (stats && blockIdx.x == 0 && threadIdx.x == 0) stats[2] += (int64_t)nm * (int64_t)slab_vec * 16;
}

// ---------------------------------------------------------------------------
// Periodic re-pick of a STATIC pool.  "RTX 3060 runs a 35B MoE with
// llama.cpp" (video transcript), chapter on code and chat profiles: the hot
// set is chosen once, yet the useful set drifts; "every 500 tokens, say, have
// another look. Swap out whatever's gone cold and then leave it alone again".
// Every routing adds one to its expert's window count; a re-pick keeps the S
// experts ranked first by (count desc, resident first, id asc), loads the new
// members (ascending id) into empty slots first and then into the slots of
// experts that left (ascending slot), and clears the counts.  One CTA, rank by
// compare and block scans: no atomics, deterministic.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kManageThreads) window_count_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                                      int32_t* __restrict__ counts,
                                                                      int32_t* __restrict__ status) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int e = ids[i];
    if (e < 0 || e >= E) {
      set_status(status, MOE_DEV_BAD_EXPERT);
      continue;
    }
    atomicAdd(&counts[e], 1);  // integer sums: the result does not depend on the order
  }
}

__global__ void __launch_bounds__(kManageThreads) window_add_kernel(const int32_t* __restrict__ count, int E,
                                                                    int32_t* __restrict__ counts) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[e] += count[e];
}

// Shared memory (dynamic): cnt[E] | res[E] | mlist[E] | innew[E] | s2e[S]
__global__ void __launch_bounds__(kManageThreads) repick_kernel(int32_t* __restrict__ counts, int E, int S,
                                                                int32_t* __restrict__ e2s_g,
                                                                int32_t* __restrict__ s2e_g,
                                                                int32_t* __restrict__ miss_e,
                                                                int32_t* __restrict__ miss_s,
                                                                int32_t* __restrict__ n_miss) {
  extern __shared__ int rp_smem[];
  int* cnt = rp_smem;
  int* res = cnt + E;
  int* mlist = res + E;
  int* innew = mlist + E;
  int* s2e = innew + E;
  __shared__ int tmp[33];
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int e = tid; e < E; e += nt) {
    cnt[e] = counts[e];
    res[e] = e2s_g[e] >= 0;
  }
  for (int q = tid; q < S; q += nt) s2e[q] = s2e_g[q];
  __syncthreads();
  const int keep = min(S, E);
  int mine = 0;
  if (tid < E) {  // E <= blockDim
    const int c = cnt[tid], r = res[tid];
    int rank = 0;
    for (int f = 0; f < E; ++f) {
      const int cf = cnt[f], rf = res[f];
      rank += (cf > c) || (cf == c && (rf > r || (rf == r && f < tid)));
    }
    innew[tid] = rank < keep;
    mine = rank < keep && !r;
  }
  __syncthreads();
  int nmiss = 0;
  const int mi = block_exclusive_scan(mine, tmp, &nmiss);
  if (mine) mlist[mi] = tid;
  __syncthreads();
  // victims: empty slots first, then slots whose expert left the set, each in ascending slot order
  int base = 0;
  for (int pass = 0; pass < 2; ++pass) {
    for (int q0 = 0; q0 < S; q0 += nt) {
      const int q = q0 + tid;
      int fl = 0;
      if (q < S) fl = pass == 0 ? s2e[q] < 0 : (s2e[q] >= 0 && !innew[s2e[q]]);
      int tot = 0;
      const int idx = block_exclusive_scan(fl, tmp, &tot);
      if (fl && base + idx < nmiss) {
        const int v = base + idx, e = mlist[v], old = s2e[q];
        if (old >= 0) e2s_g[old] = -1;  // the leaving expert is outside the new set: no other thread writes it
        s2e_g[q] = e;
        e2s_g[e] = q;
        miss_e[v] = e;
        miss_s[v] = q;
      }
      base += tot;
    }
  }
  for (int e = tid; e < E; e += nt) counts[e] = 0;
  if (tid == 0) *n_miss = nmiss;
}

int launch_window_add(const int32_t* count, int E, int32_t* counts, cudaStream_t stream) {
  window_add_kernel<<<1, 256, 0, stream>>>(count, E, counts);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

int launch_manage(const int32_t* ids, int n, int E, int S, int policy, int32_t* e2s, int32_t* s2e, uint32_t* prio,
                  uint32_t* stamp, int32_t* miss_e, int32_t* miss_s, int32_t* n_miss, int32_t* hit_e,
                  int32_t* n_hit, int32_t* sid, int64_t* stats, int32_t* dev_status, cudaStream_t stream,
                  const ManageWave* wave) {
  const size_t smem = (size_t)4 * E * sizeof(int) + (size_t)4 * S * sizeof(int);
  static bool attr_done[64] = {};
  MOE_CUDA_TRY(ensure_smem(manage_kernel, (int)(4 * kMaxE * 4 + 4 * kMaxS * 4), attr_done));
  const ManageWave nw{};
  const ManageWave& w = wave ? *wave : nw;
  manage_kernel<<<1, kManageThreads, smem, stream>>>(ids, n, w.n_dev, w.n_off, E, S, policy, e2s, s2e, prio, stamp,
                                                     miss_e, miss_s, n_miss, hit_e, n_hit, sid, w.def_e, w.n_def,
                                                     w.sub_n, w.sub, w.keep, stats, dev_status);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

int check_host_accessible(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_NOT_DEVICE_ACCESSIBLE;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return MOE_OK;
  if (a.type == cudaMemoryTypeHost && a.devicePointer == p) return MOE_OK;
  return MOE_ERR_NOT_DEVICE_ACCESSIBLE;
}

int launch_gather(const void* host_slabs, void* pool, size_t slab_bytes, int E, int S, const int32_t* miss_e,
                  const int32_t* miss_s, const int32_t* n_miss, int max_miss, int64_t* stats, int32_t* dev_status,
                  cudaStream_t stream) {
  if (max_miss <= 0) return MOE_OK;
  const size_t slab_vec = slab_bytes / 16;
  const size_t chunks = (slab_vec + kGatherChunkVec - 1) / kGatherChunkVec;
  // The host link, not the SMs, bounds the copy: on GB300 (NVLink-C2C, pinned memory) 24 CTAs of 256
  // threads with 32 KB each in flight already reach the link's 211 GB/s (16: 201, 8: 133).  Twice that
  // leaves the other SMs to the FFN that runs beside the gather on the main stream.
  constexpr size_t kGatherCtas = 48;
  const size_t items = (size_t)max_miss * chunks;
  const int grid = (int)std::min<size_t>(items, kGatherCtas);
  gather_kernel<<<grid, kGatherThreads, 0, stream>>>((const uint4*)host_slabs, (uint4*)pool, slab_vec, E, S,
                                                      miss_e, miss_s, n_miss, stats, dev_status);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" int moe_cache_manage(const int32_t* ids, int n, int E, int S, int policy, int32_t* e2s, int32_t* s2e,
                                uint32_t* prio, uint32_t* stamp, int32_t* miss_e, int32_t* miss_s,
                                int32_t* n_miss, int32_t* hit_e, int32_t* n_hit, int32_t* sid,
                                int32_t* dev_status, moe_stream_t stream) {
  if (!ids || !e2s || !s2e || !prio || !stamp || !miss_e || !miss_s || !n_miss) return MOE_ERR_ARG;
  if ((hit_e == nullptr) != (n_hit == nullptr)) return MOE_ERR_ARG;
  if (n < 1 || E < 1 || E > kMaxE || S < 1 || S > kMaxS) return MOE_ERR_ARG;
  if (policy < MOE_POLICY_LRU || policy > MOE_POLICY_STATIC) return MOE_ERR_ARG;
  if (policy != MOE_POLICY_STATIC && S < E && n > S) return MOE_ERR_CAPACITY;
  return launch_manage(ids, n, E, S, policy, e2s, s2e, prio, stamp, miss_e, miss_s, n_miss, hit_e, n_hit, sid,
                       nullptr, dev_status, (cudaStream_t)stream);
}

extern "C" int moe_cache_gather(const void* host_slabs, void* pool, size_t slab_bytes, int E, int S,
                                const int32_t* miss_e, const int32_t* miss_s, const int32_t* n_miss,
                                int max_miss, int32_t* dev_status, moe_stream_t stream) {
  if (!host_slabs || !pool || !miss_e || !miss_s || !n_miss) return MOE_ERR_ARG;
  if (E < 1 || S < 1 || max_miss < 0 || slab_bytes == 0) return MOE_ERR_ARG;
  if (slab_bytes % 16 || (uintptr_t)host_slabs % 16 || (uintptr_t)pool % 16) return MOE_ERR_ALIGN;
  const int acc = check_host_accessible(host_slabs);
  if (acc != MOE_OK) return acc;
  return launch_gather(host_slabs, pool, slab_bytes, E, S, miss_e, miss_s, n_miss, max_miss, nullptr, dev_status,
                       (cudaStream_t)stream);
}

extern "C" int moe_cache_count(const int32_t* ids, int n, int E, int32_t* counts, int32_t* dev_status,
                               moe_stream_t stream) {
  if (!ids || !counts || n < 0 || E < 1 || E > kMaxE) return MOE_ERR_ARG;
  if (n == 0) return MOE_OK;
  const int grid = std::min((n + kManageThreads - 1) / kManageThreads, 64);
  window_count_kernel<<<grid, kManageThreads, 0, (cudaStream_t)stream>>>(ids, n, E, counts, dev_status);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

extern "C" int moe_cache_repick(int32_t* counts, int E, int S, int32_t* e2s, int32_t* s2e, int32_t* miss_e,
                                int32_t* miss_s, int32_t* n_miss, moe_stream_t stream) {
  if (!counts || !e2s || !s2e || !miss_e || !miss_s || !n_miss) return MOE_ERR_ARG;
  if (E < 1 || E > kMaxE || S < 1 || S > kMaxS) return MOE_ERR_ARG;
  const size_t smem = (size_t)4 * E * sizeof(int) + (size_t)S * sizeof(int);
  static bool attr_done[64] = {};
  MOE_CUDA_TRY(ensure_smem(repick_kernel, (int)(4 * kMaxE * 4 + kMaxS * 4), attr_done));
  repick_kernel<<<1, kManageThreads, smem, (cudaStream_t)stream>>>(counts, E, S, e2s, s2e, miss_e, miss_s, n_miss);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}
