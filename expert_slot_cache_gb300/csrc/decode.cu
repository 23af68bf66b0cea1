// One persistent kernel for a small all-resident decode step.
//
// The whole layer of a decode batch of a few tokens -- router logits, top-k,
// grouping by expert, the gate/up and down weight streams on tcgen05, and the
// weighted combine -- runs as one cooperative launch with one CTA per SM.
// "Betelgeuse: Running Qwen 3.8 Flash Next ... on an RTX 3060", "What it
// actually does under the hood": hits are resolved in-stream on the device and
// a decode pass replays as one CUDA graph; "Porting vllm-expert-cache to
// NVIDIA GPUs", "1. Kernels" (a fused cache-and-expert kernel).  At one token
// the eight experts' 75.5 MB stream in about 11 us, while a chain of eight
// dependent launches costs more than that in ramps and gaps; here the weight
// stream never stops between the two projections.
//
// Phases (grid-wide waits are bounded spins on counters in the workspace; a
// cooperative launch keeps every CTA resident, so a CTA can wait on another):
//  1. router logits (decode_route.cuh): units (128-row block b, 32 experts,
//     token t) over all warps; part_b = fma chain from 0 over the block's
//     rows in order, the same fp32 order as the router kernels; every CTA also
//     zeroes its share of the step's accumulators; a grid-wide arrival.
//  2. every CTA adds the parts in block order (+ the offset), ranks the
//     scores (top-k) and groups the step's routings by expert in shared
//     memory; CTA 0 writes logits, ids and weights.
//  3. gate/up stream: the listed experts' [Wg | Wu] cut into stages of 16
//     rows, dealt as equal contiguous ranges to the CTAs (the decode stream
//     schedule); each part's sums are added to the rows' accumulators
//     gsum[p][2I] in 64-bit fixed point by integer atomics (so the sum does
//     not depend on the order the parts arrive in); after each part a release
//     on the expert's counter.
//  4. the loader goes straight on to the CTA's down stages (weights only), so
//     the DRAM stream continues while the epilogue warps wait for every
//     gate/up part of those experts and build h = silu(g) * u in bf16 in
//     shared memory, laid out as the MMA's B operand.
//  5. down MMAs into ysum[p][H] the same way; a grid-wide arrival; then every
//     CTA combines a share of the output: out[t] = sum_j w[t][j] y[pos(t, j)]
//     in fp32, j ascending, rounded to bf16.
// The last CTA to leave puts every counter back to zero.
//
// Expert-cache steps (gather mode, T*k <= S, LRU or LFU) run in the same launch
// ("Porting vllm-expert-cache to NVIDIA GPUs", "1. Kernels": a fused cache
// manager, gather and expert kernel; "Betelgeuse ... on an RTX 3060", "What it
// actually does under the hood": hits resolved in-stream, no host round trip):
//  0. before its phase-1 arrival every CTA copies the cache state (e2s, s2e,
//     prio, stamp) into shared memory; live-cache affinity reads that copy;
//  2b. after the routing every CTA runs the manage state machine on its copy
//     (deterministic, so every CTA gets the same result) and lists the step's
//     experts as hits, then misses in load order; CTA 0 writes the new state;
//  3'. CTAs 0 .. gather_ctas-1 copy the missing slabs from mapped host memory
//     into their victim slots, miss after miss, in 24 KB pieces, counting each
//     miss's finished pieces on a counter; the other CTAs run the weight
//     streams over the list, and a loader that meets a missing expert waits for
//     its counter (then a generic-to-async proxy fence) before its first
//     tensor-map copy from that slot.  The hits stream while the link copies.
// Every miss gets a victim slot the step does not need because T*k <= S, so no
// expert is loaded twice and no slot is read while it is written.
#include <algorithm>

#include "decode_route.cuh"
#include "internal.cuh"
#include "manage_core.cuh"
#include "sched.cuh"
#include "tc05.cuh"

namespace moe {

constexpr int kPThreads = 192;  // warp 0 loads, warp 1 issues MMAs, warps 2-5 epilogue
constexpr int kPWarps = kPThreads / 32;
constexpr int kPM = 128;        // output columns per MMA (M)
constexpr int kPN = 16;         // tokens per MMA (N)
constexpr int kPK = 16;         // weight rows per stage (K)
constexpr int kPBox = 64 * kPK * 2;  // one {64 columns x 16 rows} swizzle atom, 2 KB
constexpr int kPAct = 8 * kPN * 2;   // {8 rows x 16 tokens} bf16 core matrices, 256 B
constexpr int kPHStage = 2 * kPAct;  // h of one down stage, 512 B
constexpr uint32_t kPIdesc = idesc_bf16(kPM, kPN, 1, 0);
constexpr int kPMaxT = 8;
constexpr int kPMaxN = 64;      // T * k
constexpr int kPMaxE = 256;
constexpr int kPMaxStages = 4;
constexpr uint32_t kPTmemCols = 512;  // two accumulator buffers of up to 256 columns
constexpr int kPSmemMax = 232448 - 12 * 1024;  // dynamic shared memory cap (static shared memory below)

// Counters after the E per-expert gate/up counters; then, in gather mode, one counter of copied pieces per miss.
constexpr int kCtrLogits = 0, kCtrDown = 1, kCtrExit = 2, kCtrRoute = 3, kCtrCount = 4;
// Gather mode: CTAs that copy the misses (the separate gather's grid: the host link saturates well below it),
// and the piece one CTA copies at a time (eight 16-byte loads in flight per thread).
constexpr int kDGCtas = 48;
constexpr int kDGUnroll = 8;
constexpr int kDGPieceVec = kPThreads * kDGUnroll;  // 16-byte units, 24 KB

struct DecodeArgs {
  const uint16_t* x;   // bf16 [T][H]
  const uint16_t* wr;  // bf16 [H][E]
  const float* off;    // fp32 [E] or NULL
  const float* bias;   // fp32 [E] or NULL
  const int32_t* e2s;  // [E] or NULL (expert e in slot e)
  float affinity;
  int rflags;
  int T, H, E, k, I, S;
  const uint16_t* pool;
  float* lpart;   // fp32 [H/128][T][E]
  float* logits;  // fp32 [T][E]
  int32_t* ids;
  float* w;
  uint16_t* out;  // bf16 [T][H]
  unsigned long long* gsum;  // [n][2I]: the rows' gate | up sums, 64-bit fixed point (2^-32), zeroed per step
  unsigned long long* ysum;  // [n][H]: the rows' down sums, the same
  int32_t* ctr;  // E + kCtrCount (+ kPMaxN in gather mode), zero on entry and on exit
  int32_t* status;
  int stride, nst, hcap;  // ring stage stride and count; down stages the h area holds
  int ring_bytes;         // >= nst * stride and >= the router's staging (kPWarps * kRStage)
  // gather mode only: the cache state (updated in place), the host store and the copy
  int32_t* e2s_g;
  int32_t* s2e_g;
  uint32_t* prio_g;
  uint32_t* stamp_g;
  int policy;
  const uint4* host;  // mapped pinned host store, [E][slab]
  uint4* pool_w;      // the slot pool, written by the copy
  size_t slab_vec;    // 16-byte units per slab
  int64_t* stats;     // [0] += misses, [1] += 1, [2] += bytes copied, or NULL
};

// The partial sums of a step's rows meet in 64-bit fixed point with 32 fraction bits: a part v adds
// rint(v * 2^32) by an integer atomic, so the sum does not depend on the order in which parts arrive
// (and is exact for every part of magnitude 2^-8 or more, whose fp32 ulp is at least 2^-32).
constexpr float kFxScale = 4294967296.f, kFxInv = 1.f / 4294967296.f;
__device__ __forceinline__ unsigned long long to_fx(float v) { return (unsigned long long)__float2ll_rn(v * kFxScale); }
__device__ __forceinline__ float from_fx(unsigned long long s) { return __ll2float_rn((long long)s) * kFxInv; }

// TMEM accumulator columns 0..W-1 (tokens) of every tile -> the rows' fixed-point sums.
template <int W>
__device__ __forceinline__ void dec_epilogue(uint32_t taddr, unsigned long long* base, int ntiles, int N, int nb) {
  constexpr int G = W >= 32 ? 1 : 32 / W;
  for (int m0 = 0; m0 < ntiles; m0 += G) {
    float v[G][W];
#pragma unroll
    for (int gi = 0; gi < G; ++gi)
      if (m0 + gi < ntiles) tmem_ld_w<W>(taddr + (m0 + gi) * kPN, v[gi]);
    tmem_ld_wait();
#pragma unroll
    for (int gi = 0; gi < G; ++gi)
      if (m0 + gi < ntiles)
#pragma unroll
        for (int t = 0; t < W; ++t)
          if (t < nb) atomicAdd(base + (size_t)t * N + (m0 + gi) * kPM, to_fx(v[gi][t]));
  }
}

__device__ __forceinline__ void drain_tile(uint32_t taddr, unsigned long long* base, int ntiles, int N, int nb) {
  if (nb <= 1)
    dec_epilogue<1>(taddr, base, ntiles, N, nb);
  else if (nb <= 2)
    dec_epilogue<2>(taddr, base, ntiles, N, nb);
  else if (nb <= 4)
    dec_epilogue<4>(taddr, base, ntiles, N, nb);
  else
    dec_epilogue<8>(taddr, base, ntiles, N, nb);
}

// The same, out of line: the gather-mode kernel's phase loop keeps more state live, and the drain's
// accumulator registers would otherwise spill.
__device__ __noinline__ void drain_tile_call(uint32_t taddr, unsigned long long* base, int ntiles, int N, int nb) {
  drain_tile(taddr, base, ntiles, N, nb);
}

__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// One projection's stage schedule for one CTA, in phases.  Phase 0: list entries [0, nh) (every entry in
// resident mode), NSR stages each, dealt as equal contiguous ranges of L stages over the Gf streaming CTAs
// (the decode stream schedule).  Phase 1 + m (gather mode): miss m, list entry nh + m, its stages cut into
// `per` runs of L1 = ceil(NSR / Gf) stages, run r going to streaming CTA (m * per + r) % Gf: a miss streams
// on many CTAs at once as soon as its slab is in, and the runs of all misses spread evenly over the CTAs.
// Every role of a CTA walks phase after phase, gate/up before down within a phase; the down stages of a
// phase wait only for gate/up parts of the same phase, which every CTA takes before its own down stages.
static_assert(kPMaxT <= kPN, "one token batch per expert part: a part's stages are walked once");
struct DecSched {
  int NSR, nh, Gf, f;  // f: this CTA among the streaming CTAs, -1 for none
  int L, L1, per;
  __device__ __forceinline__ void init(int NSR_, int nh_, int Gf_, int f_) {
    NSR = NSR_;
    nh = nh_;
    Gf = Gf_;
    f = f_;
    L = nh > 0 ? stream_len(nh, NSR, Gf, 1 << 30) : 1;
    L1 = (NSR + Gf - 1) / Gf;
    per = (NSR + L1 - 1) / L1;
  }
  // this CTA's stage range [beg, end) of phase p (empty when beg >= end)
  __device__ __forceinline__ void range(int p, int& beg, int& end) const {
    beg = end = 0;
    if (f < 0) return;
    if (p == 0) {
      beg = f * L;
      end = min(beg + L, nh * NSR);
      return;
    }
    const int m = p - 1, r = (f - (m * per) % Gf + Gf) % Gf;
    if (r >= per) return;
    beg = (nh + m) * NSR + r * L1;
    end = min(beg + L1, (nh + m + 1) * NSR);
  }
  // the CTA parts list entry li is cut into
  __device__ __forceinline__ int parts(int li) const { return li < nh ? stream_parts(li, NSR, L) : per; }
};

template <bool kGather>
__global__ void __launch_bounds__(kPThreads, 1) decode_layer_kernel(const DecodeArgs a,
                                                                    const __grid_constant__ CUtensorMap mwg,
                                                                    const __grid_constant__ CUtensorMap mwd) {
  extern __shared__ __align__(16) unsigned char dsm_raw[];
  // 1024-byte aligned, by an offset from the shared array (so the compiler keeps shared-space accesses)
  unsigned char* ring = dsm_raw + ((1024u - (smem_u32(dsm_raw) & 1023u)) & 1023u);
  unsigned char* hsm = ring + a.ring_bytes;  // h of the down stages; the logits and scores before that
  float* slog = reinterpret_cast<float*>(hsm);
  float* ssc = slog + a.T * a.E;
  const size_t hb0 = (size_t)a.hcap * kPHStage, lb0 = (size_t)a.T * a.E * 8;
  const size_t hbytes = ((hb0 > lb0 ? hb0 : lb0) + 15) & ~size_t(15);
  uint64_t* full = reinterpret_cast<uint64_t*>(hsm + hbytes);
  uint64_t* empty = full + kPMaxStages;
  uint64_t* tfull = empty + kPMaxStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint64_t* hbar = done + 1;  // [hcap]: h of local down stage i is in place
  // gather mode: the cache state's copy (e2s [E], s2e [S], prio [S]) and the misses' slots [kPMaxN]
  int* st_e2s = reinterpret_cast<int*>(hbar + a.hcap);
  int* st_s2e = st_e2s + a.E;
  uint32_t* st_prio = reinterpret_cast<uint32_t*>(st_s2e + a.S);
  int* st_miss_s = reinterpret_cast<int*>(st_prio + a.S);
  __shared__ int s_ids[kPMaxN], s_rows[kPMaxN], s_pos[kPMaxN];
  __shared__ float s_w[kPMaxN];
  __shared__ int s_cnt[kPMaxE], s_off[kPMaxE + 1], s_act[kPMaxE], s_li[kPMaxE];
  __shared__ int tmp[33];
  __shared__ int s_nact, s_abort;
  __shared__ uint32_t s_tmem;
  __shared__ int s_nh, s_nl;  // gather mode: hits, then misses, in the list
  __shared__ uint32_t s_stamp;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, E = a.E, k = a.k, H = a.H, I = a.I, n = T * k;
  const int G = gridDim.x;
  if (tid == 0) {
    prefetch_tmap(&mwg);
    prefetch_tmap(&mwd);
    for (int s = 0; s < a.nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], 4);
    }
    mbar_init(done, 1);
    for (int i = 0; i < a.hcap; ++i) mbar_init(&hbar[i], 1);
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, kPTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;
  int32_t* gctr = a.ctr + E + kCtrCount;  // gather mode: pieces copied of miss m

  // ---- 0. gather mode: the cache state as it stands, read before this CTA's phase-1 arrival (CTA 0
  // writes the new state only once every CTA has arrived) -----------------------------------------
  if constexpr (kGather) {
    for (int e = tid; e < E; e += kPThreads) st_e2s[e] = a.e2s_g[e];
    for (int s = tid; s < a.S; s += kPThreads) {
      st_s2e[s] = a.s2e_g[s];
      st_prio[s] = a.prio_g[s];
    }
    if (tid == 0) s_stamp = *a.stamp_g;
  }

  // ---- 1. router logits: block parts -------------------------------------------------
  RouteIO rio{a.x, a.wr, a.off, a.bias, kGather ? st_e2s : a.e2s, a.affinity, a.rflags, T, H, E, k,
              a.lpart, a.logits, a.ids, a.w, &a.ctr[E + kCtrRoute], a.status};
  route_logit_parts<kPThreads>(rio, ring);
  {
    // this CTA's share of the step's fixed-point accumulators (gsum and ysum are contiguous); the
    // barrier below orders the stores before the release
    const size_t z = (size_t)n * (2 * I + H) / 2;  // 16-byte pieces
    ulonglong2* zp = reinterpret_cast<ulonglong2*>(a.gsum);
    for (size_t i = blockIdx.x * z / G + tid; i < (blockIdx.x + 1) * z / G; i += kPThreads)
      zp[i] = make_ulonglong2(0ull, 0ull);
  }
  fence_async_smem();  // the ring's staging bytes are overwritten by tensor-map copies later
  __syncthreads();
  if (tid == 0) {  // the barrier orders the CTA's stores before this (cumulative) release
    add_release(&a.ctr[E + kCtrLogits], 1);
    if (!wait_count(&a.ctr[E + kCtrLogits], G, a.status)) s_abort = 1;
  }
  __syncthreads();

  // ---- 2. logits, top-k, weights and the grouping by expert -------------------------------
  {
    const RouteSm rsm{slog, ssc, s_ids, s_w, s_cnt, s_off, s_act, s_li, s_rows, s_pos, tmp, &s_nact, abort_flag};
    route_pick_group<kPThreads>(rio, rsm);
  }

  // ---- 2b. gather mode: the manage state machine on this CTA's copy of the state ---------------
  if constexpr (kGather) {
    // work arrays in the ring (no tensor-map copy has been issued yet)
    int* mrank = reinterpret_cast<int*>(ring);
    int* hrank = mrank + E;
    int* cand = hrank + E;
    int* vict = cand + a.S;
    int* hit_t = vict + a.S;
    int* miss_t = hit_t + kPMaxN;
    const uint32_t stamp = s_stamp + 1u;
    const ManageCounts mc = manage_block(E, a.S, a.policy, false, stamp, s_cnt, st_e2s, st_s2e, st_prio, mrank,
                                         hrank, cand, vict, hit_t, miss_t, st_miss_s, nullptr, nullptr, a.status);
    // the list: hits (ascending id), then the misses in load order (ascending id); T*k <= S gives every
    // miss a slot, so together they are the routed experts
    const bool ok = mc.nh + mc.nl == s_nact && mc.nl <= kPMaxN;
    if (ok)
      for (int i = tid; i < s_nact; i += kPThreads) {
        const int e = i < mc.nh ? hit_t[i] : miss_t[i - mc.nh];
        s_act[i] = e;
        s_li[e] = i;
      }
    // a step whose wait gave up before this point leaves the state (and, its copying CTAs having given up
    // too, the pool) as it was
    if (blockIdx.x == 0 && !*abort_flag) {
      for (int e = tid; e < E; e += kPThreads) a.e2s_g[e] = st_e2s[e];
      for (int s = tid; s < a.S; s += kPThreads) {
        a.s2e_g[s] = st_s2e[s];
        a.prio_g[s] = st_prio[s];
      }
      if (tid == 0) {
        *a.stamp_g = stamp;
        if (a.stats) {
          a.stats[0] += mc.nl;
          a.stats[1] += 1;
          a.stats[2] += (int64_t)mc.nl * (int64_t)a.slab_vec * 16;
        }
      }
    }
    if (tid == 0) {
      s_nh = mc.nh;
      s_nl = ok ? mc.nl : 0;
      if (!ok) {
        set_status(a.status, MOE_DEV_BAD_SLOT);
        s_abort = 1;
      }
    }
    fence_async_smem();  // tensor-map copies overwrite the work arrays next
    __syncthreads();
  }

  // ---- 3-5. the two weight streams -----------------------------------------------------
  FfnArgs fa{};
  fa.E = E;
  fa.S = a.S;
  fa.e2s = kGather ? st_e2s : a.e2s;
  fa.list_e = s_act;
  fa.offset = s_off;
  const int n_list = s_nact;
  const int NSRg = H / kPK, NSRd = I / kPK;
  const int Ng = 2 * I;
  // gather mode with misses: CTAs 0 .. gg-1 copy them, the others stream
  const int nl = kGather ? s_nl : 0, nh = n_list - nl, nph = 1 + nl;
  const int gg = nl > 0 ? kDGCtas : 0;
  const int Gf = G - gg, fb = (int)blockIdx.x >= gg ? (int)blockIdx.x - gg : -1;
  DecSched sg, sd;
  sg.init(NSRg, nh, Gf, fb);
  sd.init(NSRd, nh, Gf, fb);
  const int wbytes_g = 2 * I * kPK * 2, wbytes_d = H * kPK * 2;
  const int gpieces = kGather ? (int)((a.slab_vec + kDGPieceVec - 1) / kDGPieceVec) : 0;
  int n_down = 0;  // this CTA's down stages: the h area holds them
  for (int p = 0; p < nph; ++p) {
    int b, e;
    sd.range(p, b, e);
    n_down += max(e - b, 0);
  }
  const bool h_ok = n_down <= a.hcap;  // the host sizes the h area for the most a CTA can get
  if (!h_ok) {
    if (tid == 0) set_status(a.status, MOE_DEV_BAD_GROUPS);
    s_abort = 1;
  }
  __syncthreads();

  // ---- 3'. gather mode: the copying CTAs, miss after miss -----------------------------------
  // Software-pipelined: the next piece's host loads are in flight while this piece is stored, fenced and
  // released, so the host link never waits on the barrier.
  if constexpr (kGather) {
    if ((int)blockIdx.x < gg && !*abort_flag) {
      const int nh = s_nh;
      const int items = s_nl * gpieces;
      // piece `it`: its source and destination, or false (a bad list entry: nothing is copied)
      auto piece = [&](int it, const uint4*& src, uint4*& dst, size_t& lim) {
        const int m = it / gpieces, c = it - m * gpieces;
        const int e = s_act[nh + m], sl = st_miss_s[m];
        if (e < 0 || e >= E || sl < 0 || sl >= a.S) {
          if (tid == 0) set_status(a.status, e < 0 || e >= E ? MOE_DEV_BAD_EXPERT : MOE_DEV_BAD_SLOT);
          return false;
        }
        src = a.host + (size_t)e * a.slab_vec + (size_t)c * kDGPieceVec;
        dst = a.pool_w + (size_t)sl * a.slab_vec + (size_t)c * kDGPieceVec;
        lim = min((size_t)kDGPieceVec, a.slab_vec - (size_t)c * kDGPieceVec);
        return true;
      };
      uint4 v[kDGUnroll], nv[kDGUnroll];
      const uint4* src = nullptr;
      uint4* dst = nullptr;
      size_t lim = 0;
      bool ok = (int)blockIdx.x < items && piece(blockIdx.x, src, dst, lim);
      if (ok)
#pragma unroll
        for (int u = 0; u < kDGUnroll; ++u) {
          const size_t j = tid + (size_t)u * kPThreads;
          if (j < lim) v[u] = ldg_stream(src + j);
        }
      for (int it = blockIdx.x; it < items; it += gg) {
        const int nx = it + gg;
        const uint4* nsrc = nullptr;
        uint4* ndst = nullptr;
        size_t nlim = 0;
        const bool nok = nx < items && piece(nx, nsrc, ndst, nlim);
        if (nok)
#pragma unroll
          for (int u = 0; u < kDGUnroll; ++u) {
            const size_t j = tid + (size_t)u * kPThreads;
            if (j < nlim) nv[u] = ldg_stream(nsrc + j);
          }
        if (ok) {
#pragma unroll
          for (int u = 0; u < kDGUnroll; ++u) {
            const size_t j = tid + (size_t)u * kPThreads;
            if (j < lim) dst[j] = v[u];
          }
          fence_async_global();  // the piece is read next by other CTAs' tensor-map copies
        }
        __syncthreads();
        if (tid == 0) add_release(&gctr[it / gpieces], 1);  // the barrier orders every thread's stores before it
#pragma unroll
        for (int u = 0; u < kDGUnroll; ++u) v[u] = nv[u];
        ok = nok;
        dst = ndst;
        lim = nlim;
      }
    }
  }

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      int last_use[kPMaxStages];
      for (int s = 0; s < kPMaxStages; ++s) last_use[s] = -1;
      auto claim = [&](int sl, uint32_t use) {
        if (use > 0 && !*abort_flag && !mbar_wait(&empty[sl], (use - 1) & 1u)) {
          *abort_flag = 1;
          set_status(a.status, MOE_DEV_TIMEOUT);
        }
        return !*abort_flag;
      };
      // gather mode: a missing expert's slot is read once all of its pieces are in (bit m: miss m seen complete)
      uint64_t seen = 0;
      auto slab_ready = [&](int e) {
        if constexpr (kGather) {
          const int m = s_li[e] - s_nh;
          if (m < 0 || m >= kPMaxN || ((seen >> m) & 1ull)) return true;
          if (*abort_flag) return false;
          if (!wait_count(&gctr[m], gpieces, a.status)) {
            *abort_flag = 1;
            return false;
          }
          fence_async_global();  // the copy's generic stores before this thread's tensor-map reads of the slot
          seen |= 1ull << m;
        }
        return true;
      };
      auto gate_up = [&](const StreamSeg& g) {
        if (!slab_ready(g.e)) return false;
        int tok[kPMaxT];
        for (int t = 0; t < g.nb; ++t) tok[t] = s_rows[g.p0 + t] / k;
        for (int s = g.s_lo; s < g.s_hi; ++s, ++it) {
          const int sl = it % a.nst;
          const uint32_t use = it / a.nst;
          if (!claim(sl, use)) return false;
          unsigned char* dst = ring + sl * a.stride;
          const int row0 = s * kPK;
          mbar_expect_tx(&full[sl], wbytes_g + g.nb * 32);
          tma_load_4d(dst, &mwg, &full[sl], 0, row0, 0, 3 * g.slot);
          tma_load_4d(dst + wbytes_g / 2, &mwg, &full[sl], 0, row0, 0, 3 * g.slot + 1);
          unsigned char* act = dst + wbytes_g;
          for (int t = 0; t < g.nb; ++t) {
            const uint16_t* xr = a.x + (size_t)tok[t] * H + row0;
            bulk_load(act + t * 16, xr, 16, &full[sl]);
            bulk_load(act + kPAct + t * 16, xr + 8, 16, &full[sl]);
          }
          last_use[sl] = (int)use;
        }
        return true;
      };
      auto down = [&](const StreamSeg& g) {
        if (!slab_ready(g.e)) return false;
        for (int s = g.s_lo; s < g.s_hi; ++s, ++it) {
          const int sl = it % a.nst;
          const uint32_t use = it / a.nst;
          if (!claim(sl, use)) return false;
          mbar_expect_tx(&full[sl], wbytes_d);
          tma_load_4d(ring + sl * a.stride, &mwd, &full[sl], 0, s * kPK, 0, 3 * g.slot + 2);
          last_use[sl] = (int)use;
        }
        return true;
      };
      bool go = true;
      for (int p = 0; p < nph && go; ++p) {
        int b, e;
        sg.range(p, b, e);
        if (b < e) stream_segments<kPN>(fa, NSRg, sg.L, b, e, [&](const StreamSeg& g) { return go = gate_up(g); });
        sd.range(p, b, e);
        if (go && b < e) stream_segments<kPN>(fa, NSRd, sd.L, b, e, [&](const StreamSeg& g) { return go = down(g); });
      }
      if (*abort_flag)  // let every copy issued land before the CTA moves on
        for (int s = 0; s < a.nst; ++s)
          if (last_use[s] >= 0) mbar_wait(&full[s], (uint32_t)last_use[s] & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      if (blockIdx.x == 0)
        for (int li = 0; li < n_list; ++li) {
          int e, slot;
          if (!stream_slot(fa, li, e, slot)) set_status(a.status, MOE_DEV_BAD_SLOT);
        }
      uint32_t it = 0, seg = 0;
      int dbase = 0;  // the phase's down stages are one contiguous range: local index = dbase + global index
      auto run = [&](const StreamSeg& g, bool down) {
        const uint32_t buf = seg & 1u, use = seg >> 1;
        if (use > 0 && !*abort_flag && !mbar_wait(&tempty[buf], (use - 1) & 1u)) {
          *abort_flag = 1;
          set_status(a.status, MOE_DEV_TIMEOUT);
        }
        tc_fence_after();
        const uint32_t d = tmem + buf * 256u;
        const int ntiles = down ? H / kPM : Ng / kPM;
        const int lbase = down ? dbase + s_li[g.e] * NSRd : 0;
        for (int s = g.s_lo; s < g.s_hi; ++s, ++it) {
          const int sl = it % a.nst;
          if (!*abort_flag && !mbar_wait(&full[sl], (it / a.nst) & 1u)) {
            *abort_flag = 1;
            set_status(a.status, MOE_DEV_TIMEOUT);
          }
          // down: this stage's h is in place (written by the epilogue warps)
          if (down && !*abort_flag && lbase + s < a.hcap && !mbar_wait(&hbar[lbase + s], 0)) {
            *abort_flag = 1;
            set_status(a.status, MOE_DEV_TIMEOUT);
          }
          tc_fence_after();
          if (!*abort_flag) {
            const uint32_t sa = smem_u32(ring + sl * a.stride);
            const uint32_t sb = down ? smem_u32(hsm + (size_t)(lbase + s) * kPHStage) : sa + wbytes_g;
            const uint64_t bdesc = smem_desc_l(sb, kPAct, 128, kLayoutNone);
            for (int m = 0; m < ntiles; ++m) {
              const uint64_t adesc = smem_desc_l(sa + m * 2 * kPBox, kPBox, 1024, kLayoutSw128);
              umma_f16(d + m * kPN, adesc, bdesc, kPIdesc, s > g.s_lo);
            }
          }
          umma_commit(&empty[sl]);
        }
        umma_commit(&tfull[buf]);
        ++seg;
        return true;
      };
      int dl = 0;  // local index of the phase's first down stage (its h stage and barrier)
      for (int p = 0; p < nph; ++p) {
        int b, e;
        sg.range(p, b, e);
        if (b < e) stream_segments<kPN>(fa, NSRg, sg.L, b, e, [&](const StreamSeg& g) { return run(g, false); });
        sd.range(p, b, e);
        if (b >= e) continue;
        dbase = dl - b;
        stream_segments<kPN>(fa, NSRd, sd.L, b, e, [&](const StreamSeg& g) { return run(g, true); });
        dl += e - b;
      }
      umma_commit(done);  // every MMA issued has finished once `done` completes
      mbar_wait(done, 0);
    }
  } else {
    // epilogue warps 2..5; TMEM lane quarter q = warp % 4 holds output columns q*32 .. q*32+31 of each tile
    const int q = warp & 3, etid = tid - 64;
    uint32_t seg = 0;
    auto drain = [&](const StreamSeg& g, bool down) {
      const uint32_t buf = seg & 1u, use = seg >> 1;
      if (!*abort_flag && !mbar_wait(&tfull[buf], use & 1u)) {
        *abort_flag = 1;
        set_status(a.status, MOE_DEV_TIMEOUT);
      }
      tc_fence_after();
      if (!*abort_flag) {
        const int N = down ? H : Ng;
        unsigned long long* base = (down ? a.ysum : a.gsum) + (size_t)g.p0 * N + q * 32 + lane;
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + buf * 256u;
        if constexpr (kGather)
          drain_tile_call(taddr, base, N / kPM, N, g.nb);
        else
          drain_tile(taddr, base, N / kPM, N, g.nb);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      ++seg;
    };
    int dl = 0;  // local index of the phase's first down stage (its h stage and barrier)
    for (int p = 0; p < nph; ++p) {
      int bg, eg, bd, ed;
      sg.range(p, bg, eg);
      sd.range(p, bd, ed);
      if (bg < eg)
        stream_segments<kPN>(fa, NSRg, sg.L, bg, eg, [&](const StreamSeg& g) {
          drain(g, false);
          // publish this part of the expert's sums (the barrier orders every epilogue thread's atomics
          // before the signalling thread's release)
          named_sync(1, 128);
          if (etid == 0) add_release(&a.ctr[s_li[g.e]], 1);
          return true;
        });
      if (bd >= ed) continue;
      // h for this phase's down stages, from the experts' gate/up sums once every part is in.  Every
      // epilogue warp walks the same segments and reaches every named barrier; only the stores depend on
      // h_ok, which is the same for the whole CTA and never changes.
      // the phase's down stages are one contiguous range: local index = dl + (global index - bd)
      const int dbase = dl - bd;
      stream_segments<kPN>(fa, NSRd, sd.L, bd, ed, [&](const StreamSeg& g) {
        const int li = s_li[g.e];
        const int Jg = sg.parts(li);
        if (etid == 0 && !wait_count(&a.ctr[li], Jg, a.status)) *abort_flag = 1;
        named_sync(1, 128);
        const int lbase = dbase + li * NSRd;
        // (stage, row, token) elements of the batch's tokens, stage-major; lane pairs take the gate sum
        // (even lane) and the up sum (odd lane) of one element.  After each round the stages it
        // completed get their padding tokens (t >= nb, zeros) and go to the tensor cores.
        const int nst_seg = g.s_hi - g.s_lo;
        const int per_st = kPK * g.nb;
        const int nel = nst_seg * per_st;
        int done_st = 0;
        auto release = [&](int st_hi) {  // uniform over the epilogue warps
          const int npad = (st_hi - done_st) * kPK * (kPN - g.nb);
          for (int v = etid; v < npad && h_ok; v += 128) {
            const int st = done_st + v / (kPK * (kPN - g.nb)), rem = v % (kPK * (kPN - g.nb));
            const int t = g.nb + rem / kPK, r = rem % kPK;
            *reinterpret_cast<uint16_t*>(hsm + (size_t)(lbase + g.s_lo + st) * kPHStage + (r >> 3) * kPAct +
                                         t * 16 + (r & 7) * 2) = 0;
          }
          fence_async_smem();
          named_sync(1, 128);
          if (etid == 0)
            for (int st = done_st; st < st_hi; ++st)
              if (lbase + g.s_lo + st < a.hcap) mbar_arrive(&hbar[lbase + g.s_lo + st]);
          done_st = st_hi;
        };
        auto store_h = [&](int el, float gsum, float usum) {
          const int st = el / per_st, rem = el - st * per_st, t = rem / kPK, r = rem - t * kPK;
          const float hv = gsum / (1.f + expf(-gsum)) * usum;
          *reinterpret_cast<uint16_t*>(hsm + (size_t)(lbase + g.s_lo + st) * kPHStage + (r >> 3) * kPAct +
                                       t * 16 + (r & 7) * 2) = f32_to_bf16(hv);
        };
        // elements (stage, row, token), four per thread a round, their gate and up sums loaded together
        for (int v0 = 0; v0 < nel; v0 += 4 * 128) {  // the same trip count in every epilogue thread
          unsigned long long gs[4], us[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int el = v0 + q4 * 128 + etid;
            gs[q4] = us[q4] = 0ull;
            if (el < nel) {
              const int st = el / per_st, rem = el - st * per_st, t = rem / kPK, r = rem - t * kPK;
              const unsigned long long* src = a.gsum + (size_t)(g.p0 + t) * Ng + (g.s_lo + st) * kPK + r;
              gs[q4] = __ldcg(src);
              us[q4] = __ldcg(src + I);
            }
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int el = v0 + q4 * 128 + etid;
            if (el < nel && h_ok) store_h(el, from_fx(gs[q4]), from_fx(us[q4]));
          }
          release(min(nel, v0 + 4 * 128) / per_st);
        }
        if (done_st < nst_seg) release(nst_seg);
        return true;
      });
      stream_segments<kPN>(fa, NSRd, sd.L, bd, ed, [&](const StreamSeg& g) {
        drain(g, true);
        return true;
      });
      dl += ed - bd;
    }
  }
  // warps 0 and 1 ran their loops on lane 0 alone: reconverge before the CTA barrier
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kPTmemCols);
  }
  if (tid == 0) {
    add_release(&a.ctr[E + kCtrDown], 1);
    wait_count(&a.ctr[E + kCtrDown], G, a.status);
  }
  __syncthreads();

  // ---- combine: out[t] = sum_j w[t][j] * y[pos(t, j)], j ascending -------------------------
  {
    // (token, column quad) items dealt round-robin over the grid; one thread per (item, pick) converts
    // its y, the thread of pick 0 adds the picks in order
    const int nc4 = H / 4, nit = T * nc4;
    const int my_items = nit > (int)blockIdx.x ? (nit - 1 - (int)blockIdx.x) / G + 1 : 0;
    float4* sy = reinterpret_cast<float4*>(ring);  // every stage has been read: the ring is free
    for (int u = tid; u < my_items * k; u += kPThreads) {
      const int m = u / k, j = u - m * k, item = (int)blockIdx.x + G * m;
      const int t = item / nc4, c4 = item - t * nc4, p = s_pos[t * k + j];
      const ulonglong2* src = reinterpret_cast<const ulonglong2*>(a.ysum + (size_t)p * H + 4 * c4);
      const ulonglong2 y01 = __ldcg(src), y23 = __ldcg(src + 1);
      sy[u] = make_float4(from_fx(y01.x), from_fx(y01.y), from_fx(y23.x), from_fx(y23.y));
    }
    __syncthreads();
    for (int m = tid; m < my_items; m += kPThreads) {
      const int item = (int)blockIdx.x + G * m, t = item / nc4, c4 = item - t * nc4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < k; ++j) {
        const float wj = s_w[t * k + j];
        const float4 yj = sy[m * k + j];
        acc.x = fmaf(wj, yj.x, acc.x);
        acc.y = fmaf(wj, yj.y, acc.y);
        acc.z = fmaf(wj, yj.z, acc.z);
        acc.w = fmaf(wj, yj.w, acc.w);
      }
      uint2 o;
      o.x = uint32_t(f32_to_bf16(acc.x)) | (uint32_t(f32_to_bf16(acc.y)) << 16);
      o.y = uint32_t(f32_to_bf16(acc.z)) | (uint32_t(f32_to_bf16(acc.w)) << 16);
      *reinterpret_cast<uint2*>(a.out + (size_t)t * H + 4 * c4) = o;
    }
  }
  // the last CTA out resets the counters: every other CTA is past its last wait
  if (tid == 0 && atomicAdd(&a.ctr[E + kCtrExit], 1) == G - 1)
    for (int i = 0; i < E + kCtrCount + (kGather ? kPMaxN : 0); ++i) a.ctr[i] = 0;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static int dec_stride(int H, int I) {
  const int s = std::max(2 * I * kPK * 2 + 2 * kPAct, H * kPK * 2);
  return (s + 1023) & ~1023;
}

bool decode_eligible(int T, int H, int E, int k, int I, int S, const void* x, const void* wr, const void* pool) {
  const int n = T * k;
  if (T < 1 || T > kPMaxT || n > kPMaxN || E > kPMaxE || E % 8 || k > kMaxK) return false;
  // accumulators of at most 16 tiles (256 TMEM columns) per projection: 2I <= 2048 and H <= 2048
  if (H % 128 || I % 128 || H > 2048 || I > 1024) return false;
  if (S < 1 || (uintptr_t)x % 16 || (uintptr_t)wr % 16 || (uintptr_t)pool % 16) return false;
  return dec_stride(H, I) * 2 + 1024 + 16 * 1024 <= kPSmemMax;
}

// Dynamic shared memory of one launch: ring | h of the down stages (the logits and scores before that) |
// barriers | gather mode: the cache state's copy.
struct DecPlan {
  int hcap = 0, nst = 0, ring_bytes = 0;
  size_t smem = 0;
};

static bool dec_plan(int T, int H, int E, int k, int I, int S, int sms, bool gather, DecPlan* p) {
  const int n = T * k, NSRd = I / kPK, lmax = std::min(n, E);
  // the most down stages a streaming CTA can get: a contiguous range of the hits' stages (stream_len with
  // every routed expert distinct) plus, in gather mode, its share of the misses' runs, which go round the
  // streaming CTAs one after another
  const int gf = sms - (gather ? kDGCtas : 0);
  if (gf < 1) return false;
  int most = (lmax * NSRd + gf - 1) / gf;
  if (gather) {
    const int L1 = (NSRd + gf - 1) / gf, per = (NSRd + L1 - 1) / L1;
    for (int nh = 0; nh <= lmax; ++nh)
      most = std::max(most, (nh * NSRd + gf - 1) / gf + ((lmax - nh) * per + gf - 1) / gf * L1);
  }
  p->hcap = most + 1;
  const size_t hbytes = (std::max((size_t)p->hcap * kPHStage, (size_t)T * E * 8) + 15) & ~size_t(15);
  const size_t state = gather ? (size_t)4 * (E + 2 * S + kPMaxN) : 0;
  const size_t fixed = 1024 + hbytes + 8 * (2 * kPMaxStages + 5 + p->hcap) + state;
  const int stride = dec_stride(H, I);
  if (fixed >= (size_t)kPSmemMax) return false;
  p->nst = (int)std::min<size_t>(kPMaxStages, (kPSmemMax - fixed) / stride);
  if (p->nst < 2) return false;
  p->ring_bytes = std::max(p->nst * stride, (kPWarps * kRStage + 1023) & ~1023);
  // gather mode: the manage call's work arrays sit in the ring before the streams start
  if (gather && (size_t)p->ring_bytes < (size_t)4 * (2 * E + 2 * S + 2 * kPMaxN)) return false;
  p->smem = fixed + (size_t)p->ring_bytes;
  return p->smem <= (size_t)kPSmemMax;
}

bool decode_gather_eligible(int T, int H, int E, int k, int I, int S, int policy, const void* x, const void* wr,
                            const void* pool, const void* host, int sms) {
  if (!decode_eligible(T, H, E, k, I, S, x, wr, pool)) return false;
  if (policy != MOE_POLICY_LRU && policy != MOE_POLICY_LFU) return false;
  // T*k <= S: every miss finds a victim among the slots the step does not need (one manage call, no deferral)
  if (T * k > S || S > kPMaxE || (uintptr_t)host % 16) return false;
  if (sms < 2 * kDGCtas) return false;  // at least as many streaming CTAs as copying ones
  DecPlan p;
  return dec_plan(T, H, E, k, I, S, sms, true, &p);
}

// the W8A8 kernel keeps the same count (it uses no per-miss counters)
size_t decode_ctr_ints(int E) { return (size_t)E + kCtrCount + kPMaxN; }

template <bool kGather>
static int launch_decode_impl(const moe_layer_args* la, float* lpart, float* logits, float* skp, size_t skp_bytes,
                              int32_t* ctr, cudaStream_t stream) {
  const int T = la->T, H = la->H, E = la->E, k = la->k, I = la->I, n = T * k;
  int dev = 0, sms = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  DecodeArgs a{};
  a.x = (const uint16_t*)la->x;
  a.wr = (const uint16_t*)la->w_router;
  a.off = la->logit_offset;
  a.bias = la->sel_bias;
  a.e2s = kGather ? nullptr : la->e2s;
  a.affinity = la->affinity;
  a.rflags = la->route_flags;
  a.T = T;
  a.H = H;
  a.E = E;
  a.k = k;
  a.I = I;
  a.S = la->S;
  a.pool = (const uint16_t*)la->pool;
  a.lpart = lpart;
  a.logits = logits;
  a.ids = la->ids;
  a.w = la->w;
  a.out = (uint16_t*)la->out;
  // the fixed-point accumulators: gsum [n][2I] then ysum [n][H]
  if (!skp || (uintptr_t)skp % 16 || skp_bytes < (size_t)n * (2 * I + H) * 8) return MOE_ERR_ALIGN;
  a.gsum = reinterpret_cast<unsigned long long*>(skp);
  a.ysum = a.gsum + (size_t)n * 2 * I;
  a.ctr = ctr;
  a.status = la->dev_status;
  a.stride = dec_stride(H, I);
  if constexpr (kGather) {
    if (!la->e2s || !la->s2e || !la->prio || !la->stamp || !la->host_slabs) return MOE_ERR_ARG;
    a.e2s_g = la->e2s;
    a.s2e_g = la->s2e;
    a.prio_g = la->prio;
    a.stamp_g = la->stamp;
    a.policy = la->policy;
    a.host = (const uint4*)la->host_slabs;
    a.pool_w = (uint4*)la->pool;
    a.slab_vec = (size_t)6 * H * I / 16;
    a.stats = la->stats;
  }
  DecPlan p;
  if (!dec_plan(T, H, E, k, I, la->S, sms, kGather, &p)) return MOE_ERR_ARG;
  a.hcap = p.hcap;
  a.nst = p.nst;
  a.ring_bytes = p.ring_bytes;
  static bool attr[64] = {};
  MOE_CUDA_TRY(ensure_smem(decode_layer_kernel<kGather>, kPSmemMax, attr));
  int occ = 0;
  MOE_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_layer_kernel<kGather>, kPThreads, p.smem));
  if (occ < 1) return MOE_ERR_ARG;
  const size_t mat = (size_t)H * I;
  CUtensorMap mwg, mwd;
  {
    const uint64_t dims[4] = {64, (uint64_t)H, (uint64_t)I / 64, 3ull * la->S};
    const uint64_t str[3] = {(uint64_t)I * 2, 128, mat * 2};
    const uint32_t box[4] = {64, kPK, (uint32_t)I / 64, 1};
    if (encode_tmap_bf16(&mwg, la->pool, 4, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B) != MOE_OK) return MOE_ERR_CUDA;
  }
  {
    const uint64_t dims[4] = {64, (uint64_t)I, (uint64_t)H / 64, 3ull * la->S};
    const uint64_t str[3] = {(uint64_t)H * 2, 128, mat * 2};
    const uint32_t box[4] = {64, kPK, (uint32_t)H / 64, 1};
    if (encode_tmap_bf16(&mwd, la->pool, 4, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B) != MOE_OK) return MOE_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, decode_layer_kernel<kGather>, a, mwg, mwd));
  return MOE_OK;
}

int launch_decode(const moe_layer_args* la, float* lpart, float* logits, float* skp, size_t skp_bytes, int32_t* ctr,
                  cudaStream_t stream) {
  return launch_decode_impl<false>(la, lpart, logits, skp, skp_bytes, ctr, stream);
}

int launch_decode_gather(const moe_layer_args* la, float* lpart, float* logits, float* skp, size_t skp_bytes,
                         int32_t* ctr, cudaStream_t stream) {
  return launch_decode_impl<true>(la, lpart, logits, skp, skp_bytes, ctr, stream);
}

}  // namespace moe
