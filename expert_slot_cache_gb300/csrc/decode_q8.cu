// One persistent kernel for a small all-resident decode step with W8A8 experts.
//
// "Porting vllm-expert-cache to NVIDIA GPUs": the measured model is
// Qwen3-30B-A3B W8A8, with the weights' scales slot-indexed like the weights
// ("1. Kernels": a fused cache-and-expert kernel); "Betelgeuse ... on an RTX
// 3060", "What it actually does under the hood": a decode pass resolved on the
// device as one graph.  Same arithmetic as the separate W8A8 kernels (exact
// int32 dot products of 8-bit codes, the same fp32 dequantisation, h
// quantised per row, the combine's fp32 fma chain in pick order), so the
// output is bit for bit theirs.
//
// One CTA per SM: sixteen consumer warps (thread c owns 4 output columns) and
// one loader warp.
//  1. router logits (decode_route.cuh); every CTA also zeroes its share of
//     the step's integer accumulators and, while the grid-wide wait runs,
//     forms the tokens' 8-bit codes (per-token scale) in shared memory.
//  2. top-k, weights, grouping by expert (decode_route.cuh).
//  3. gate/up: the listed experts' [Wg | Wu] cut into stages of 16 rows (4
//     rows per int32 quad; Wd later into stages of the same bytes), dealt
//     as contiguous ranges of equal cost (a stage costs more when its expert
//     has more rows to fold); the loader brings each stage's two 16 x I byte
//     pieces into a shared-memory ring by bulk copies; the consumers fold
//     them with dp4a into int32 sums per (row, column), add them to the
//     step's accumulator gsum[p][2I] with integer atomics (exact in any
//     order) and add the stages done to the expert's counter.
//  4. the loader goes straight on to the CTA's down stages (weights only).
//     For each of its experts the consumers wait for every gate/up part, form
//     the rows' h = silu(g) u from gsum (dequantised as the separate kernels
//     do), the rows' |h| maxima, the scale and the codes of the stages they
//     need, then fold the down stages into ysum[p][H] the same way.
//  5. a grid-wide wait; every CTA combines a share of the output:
//     out[t] = bf16(sum_j w[t][j] ((ysum * sd) * sh)), j ascending, one thread
//     per (output piece, pick) so that a piece's loads are one round trip.
// Every wait is bounded (MOE_DEV_TIMEOUT); the last CTA out puts the counters
// back to zero.
//
// Expert-cache steps (gather mode, T*k <= S, LRU or LFU) run in the same
// launch as in the bf16 kernel: the cache state copied into shared memory
// before the first grid-wide arrival, the manage state machine in every CTA
// after the routing, CTA 0 writing the new state, 48 CTAs copying the misses'
// slabs (codes and scales) host-to-slot, the other CTAs streaming in phases
// (the hits as weighted contiguous ranges, then each miss in runs over all of
// them).  A missing expert's scales are read with coherent loads once its copy
// is complete (the copy writes them during the launch).
#include <algorithm>
#include <type_traits>

#include "decode_route.cuh"
#include "fp32def.cuh"
#include "internal.cuh"
#include "manage_core.cuh"
#include "sched.cuh"

namespace moe {

constexpr int kQDConsumers = 512;                   // 16 warps; thread c owns output columns 4c .. 4c + 3
constexpr int kQDThreads = kQDConsumers + 32;       // + the loader warp
constexpr int kQDMaxT = 8;
constexpr int kQDMaxN = 64;                         // T * k
constexpr int kQDMaxE = 256;
constexpr int kQDRB = 8;                            // rows of one expert in a step (<= T)
constexpr int kQDK = 16;                            // weight rows per stage
constexpr int kQDMaxStages = 8;
constexpr int kQDMaxIQ = 256;                       // I / 4
constexpr int kQDSmemMax = 232448 - 16 * 1024;      // dynamic shared memory cap (static shared memory below)

// Counters after the E per-list-index gate/up counters.
constexpr int kQCtrLogits = 0, kQCtrDown = 1, kQCtrExit = 2, kQCtrRoute = 3, kQCtrCount = 4;

struct DecodeQ8Args {
  RouteIO r;
  int I, S;
  const unsigned char* pool;  // quantised slabs, slot-indexed
  size_t qslab;               // bytes of one slab
  int32_t* gsum;              // [n][2I]: gate | up sums of the step's rows
  int32_t* ysum;              // [n][H]: down sums
  float* sh;                  // [n]: the rows' h scales
  int32_t* ctr;               // E + kQCtrCount ints, zero on entry and on exit
  uint16_t* out;              // bf16 [T][H]
  int stride, nst;            // ring slot bytes and count
  int qd;                     // int32 quad-rows (4 weight rows) of Wd per down stage: qd * 4H <= stride
  // gather mode only: the cache state (updated in place), the host store and the copy
  int state_off;              // byte offset of the state's copy in dynamic shared memory
  int32_t* e2s_g;
  int32_t* s2e_g;
  uint32_t* prio_g;
  uint32_t* stamp_g;
  int policy;
  const uint4* host;          // mapped pinned host store, [E][slab]
  uint4* pool_w;              // the slot pool, written by the copy
  int64_t* stats;             // [0] += misses, [1] += 1, [2] += bytes copied, or NULL
};

// Gather mode: CTAs that copy the misses, and the piece one CTA copies at a time (four 16-byte loads in
// flight per thread, twice over with the software pipeline).
constexpr int kQGCtas = 48;
constexpr int kQGUnroll = 4;
constexpr int kQGPieceVec = kQDThreads * kQGUnroll;  // 16-byte units, 34 KB

__device__ __forceinline__ void q8_fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

__device__ __forceinline__ int quad_of(const int4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }

__device__ __forceinline__ uint32_t pack_codes(float a, float b, float c, float d, float s) {
  return (uint32_t)(q8_code(a, s) & 0xff) | ((uint32_t)(q8_code(b, s) & 0xff) << 8) |
         ((uint32_t)(q8_code(c, s) & 0xff) << 16) | ((uint32_t)(q8_code(d, s) & 0xff) << 24);
}

// The cost of one stage of an expert with nb rows, in units of about 0.15 us under a full-chip stream: the
// dp4a work of a stage grows with the rows (about 0.19 us per row at 16 dp4a per clock per SM), the
// bytes stay the same (about 0.45 us), so stages of up to two rows cost the same and more rows cost more.
__device__ __forceinline__ int q8d_stage_cost(int nb) { return nb <= 2 ? 3 : nb <= 4 ? 5 : 10; }

// The weighted decode stream schedule: expert li's NSR stages start at weighted positions
// NSR * wpre[li] + s * w[li]; CTA b owns the stages that start in [beg, end) = [b W / G, (b + 1) W / G),
// W = NSR * wpre[n_list].  Calls f(seg) for each expert part of the range, in list order; stops early
// when f returns false.  Every role of a CTA walks the same list.
template <class F>
__device__ __forceinline__ void q8d_segments(const FfnArgs& a, const int* wpre, int n_list, int NSR, int beg, int end,
                                             F&& f) {
  // the first expert whose stages reach past beg: the largest li with NSR * wpre[li] <= beg (binary search)
  int lo = 0, hi = n_list;  // NSR * wpre[lo] <= beg < NSR * wpre[hi] when beg is in range
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (NSR * wpre[mid] <= beg) lo = mid;
    else hi = mid;
  }
  for (int li = lo; li < n_list; ++li) {
    const int P = NSR * wpre[li];  // < 2^31: NSR <= 512, wpre <= 10 * 64
    if (P >= end) return;
    const int w = wpre[li + 1] - wpre[li];
    const int s_lo = beg > P ? (beg - P + w - 1) / w : 0;
    const int s_hi = min(NSR, (end - P + w - 1) / w);
    if (s_lo >= s_hi) continue;
    StreamSeg g;
    if (!stream_slot(a, li, g.e, g.slot)) continue;
    g.s_lo = s_lo;
    g.s_hi = s_hi;
    g.j = 0;
    g.p0 = a.offset[g.e];
    g.nb = min(kQDRB, a.offset[g.e + 1] - g.p0);
    if (!f(g)) return;
  }
}

// One phase of a CTA's stream schedule.  Phase 0: list entries [0, nh) (all of them in resident mode),
// weighted contiguous ranges over the Gf streaming CTAs (the schedule above); phase 1 + m (gather mode):
// miss m, list entry nh + m, its NSR stages cut into `per` runs of L1 = ceil(NSR / Gf), run r on streaming
// CTA (m * per + r) % Gf, so a miss streams on many CTAs as soon as its slab is in.  fb: this CTA among
// the streaming CTAs, -1 for none.
template <class F>
__device__ __forceinline__ void q8d_phase(const FfnArgs& a, const int* wpre, int nh, int NSR, int Gf, int fb, int p,
                                          F&& f) {
  if (fb < 0) return;
  if (p == 0) {
    const int W = NSR * wpre[nh];  // products with Gf stay below 2^31
    const int beg = fb * W / Gf, end = (fb + 1) * W / Gf;
    if (beg < end) q8d_segments(a, wpre, nh, NSR, beg, end, f);
    return;
  }
  const int L1 = (NSR + Gf - 1) / Gf, per = (NSR + L1 - 1) / L1;
  const int m = p - 1, r = (fb - (m * per) % Gf + Gf) % Gf;
  if (r >= per) return;
  StreamSeg g;
  if (!stream_slot(a, nh + m, g.e, g.slot)) return;
  g.s_lo = r * L1;
  g.s_hi = min(NSR, g.s_lo + L1);
  g.j = 0;
  g.p0 = a.offset[g.e];
  g.nb = min(kQDRB, a.offset[g.e + 1] - g.p0);
  f(g);
}

template <bool kGather>
__global__ void __launch_bounds__(kQDThreads, 1) decode_q8_kernel(const DecodeQ8Args a) {
  extern __shared__ __align__(16) unsigned char qd_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.r.T, E = a.r.E, k = a.r.k, H = a.r.H, I = a.I, n = T * k;
  const int G = gridDim.x;
  const size_t mat = (size_t)H * I;
  // x codes [T][H/4] int32 (a stage's four quads of a token are one 16-byte load), then the ring (the
  // router's staging and the logits before it)
  int32_t* xq = reinterpret_cast<int32_t*>(qd_raw);
  unsigned char* ring = qd_raw + (((size_t)T * H + 127) & ~size_t(127));
  __shared__ uint64_t full[kQDMaxStages], empty[kQDMaxStages];
  __shared__ int32_t hq[kQDMaxIQ * kQDRB];  // h codes of the current down segment: [quad][row]
  __shared__ int s_ids[kQDMaxN], s_rows[kQDMaxN], s_pos[kQDMaxN];
  __shared__ float s_w[kQDMaxN];
  __shared__ int s_cnt[kQDMaxE], s_off[kQDMaxE + 1], s_act[kQDMaxE], s_li[kQDMaxE], s_wpre[kQDMaxN + 1];
  __shared__ unsigned s_amax[kQDRB], s_tmax[kQDMaxT];
  __shared__ float s_sx[kQDMaxT], s_shr[kQDRB];
  __shared__ int tmp[33];
  __shared__ int s_nact, s_abort;
  __shared__ int s_nh, s_nl;  // gather mode: hits, then misses, in the list
  __shared__ uint32_t s_stamp;
  volatile int* abort_flag = &s_abort;
  int32_t* ctr = a.ctr;
  int32_t* gctr = ctr + E + kQCtrCount;  // gather mode: pieces copied of miss m
  // gather mode: the cache state's copy (e2s [E], s2e [S], prio [S]) and the misses' slots [kQDMaxN]
  int* st_e2s = reinterpret_cast<int*>(qd_raw + a.state_off);
  int* st_s2e = st_e2s + E;
  uint32_t* st_prio = reinterpret_cast<uint32_t*>(st_s2e + a.S);
  int* st_miss_s = reinterpret_cast<int*>(st_prio + a.S);
  if (tid == 0) {
    for (int s = 0; s < a.nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kQDConsumers / 32);
    }
    s_abort = 0;
    mbar_fence_init();
  }
  // ---- 0. gather mode: the cache state as it stands, read before this CTA's phase-1 arrival (CTA 0
  // writes the new state only once every CTA has arrived) -----------------------------------------
  if constexpr (kGather) {
    for (int e = tid; e < E; e += kQDThreads) st_e2s[e] = a.e2s_g[e];
    for (int s = tid; s < a.S; s += kQDThreads) {
      st_s2e[s] = a.s2e_g[s];
      st_prio[s] = a.prio_g[s];
    }
    if (tid == 0) s_stamp = *a.stamp_g;
  }
  __syncthreads();
  RouteIO rio_g = a.r;
  if constexpr (kGather) rio_g.e2s = st_e2s;  // live-cache affinity reads the state before this step's manage
  const RouteIO& rio = kGather ? rio_g : a.r;

  // ---- 1. router logits; zero the accumulators; the tokens' codes ---------------------------
  {
    // this CTA's share of the step's accumulators (the barrier below orders it before the release)
    const size_t zg = (size_t)n * 2 * I / 4, zy = (size_t)n * H / 4;  // int4 pieces
    const size_t z0 = blockIdx.x * (zg + zy) / G, z1 = (blockIdx.x + 1) * (zg + zy) / G;
    for (size_t i = z0 + tid; i < z1; i += kQDThreads) {
      int4* dst = i < zg ? reinterpret_cast<int4*>(a.gsum) + i : reinterpret_cast<int4*>(a.ysum) + (i - zg);
      *dst = make_int4(0, 0, 0, 0);
    }
  }
  if (tid < kQDMaxT) s_tmax[tid] = 0u;
  __syncthreads();
  // router unit u runs on CTA u % G, warp u / G: warps [0, busy) of this CTA have units; the others form
  // the tokens' codes meanwhile (the host keeps at least four warps free)
  const int units = (H / 128) * ((E + 31) / 32) * T;
  const int busy = min(kQDThreads / 32, max(0, (units - (int)blockIdx.x + G - 1) / G));
  if (warp < busy) {
    route_logit_parts<kQDThreads>(rio, ring);
    named_sync(3, busy * 32);
    if (tid == 0) add_release(&ctr[E + kQCtrLogits], 1);  // the barriers order the CTA's stores before it
  } else {
    if (busy == 0 && tid == 0) add_release(&ctr[E + kQCtrLogits], 1);
    // 8-element pieces of x over the free threads: the tokens' |x| maxima (atomicMax on the bit
    // patterns), the scales, then the codes (the pieces read again, from cache)
    const int ct = tid - busy * 32, nct = kQDThreads - busy * 32;
    const int npc = H / 8, np = T * npc;
    for (int pc0 = ct; pc0 < np; pc0 += 4 * nct) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int pc = pc0 + u * nct;
        if (pc < np) {
          const int t = pc / npc;
          v[u] = *reinterpret_cast<const uint4*>(a.r.x + (size_t)t * H + 8 * (pc - t * npc));
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int pc = pc0 + u * nct;
        if (pc < np) {
          const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          float m = 0.f;
#pragma unroll
          for (int b = 0; b < 4; ++b) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w4[b])), fabsf(bf16_hi(w4[b]))));
          atomicMax(&s_tmax[pc / npc], __float_as_uint(m));
        }
      }
    }
    named_sync(4, nct);
    if (ct < T) s_sx[ct] = __fdiv_rn(__uint_as_float(s_tmax[ct]), 127.f);
    named_sync(4, nct);
    for (int pc = ct; pc < np; pc += nct) {
      const int t = pc / npc;
      const uint4 v = *reinterpret_cast<const uint4*>(a.r.x + (size_t)t * H + 8 * (pc - t * npc));
      const float s = s_sx[t];
      *reinterpret_cast<int2*>(xq + (size_t)t * (H / 4) + 2 * (pc - t * npc)) =
          make_int2((int32_t)pack_codes(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y), s),
                    (int32_t)pack_codes(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w), s));
    }
  }
  if (tid == 0 && !wait_count(&ctr[E + kQCtrLogits], G, a.r.status)) s_abort = 1;
  __syncthreads();

  // ---- 2. top-k, weights, grouping --------------------------------------------------------
  {
    float* slog = reinterpret_cast<float*>(ring);
    const RouteSm rsm{slog, slog + T * E, s_ids, s_w, s_cnt, s_off, s_act, s_li, s_rows, s_pos, tmp, &s_nact,
                      abort_flag};
    route_pick_group<kQDThreads>(rio, rsm);
  }

  // ---- 2b. gather mode: the manage state machine on this CTA's copy of the state ---------------
  if constexpr (kGather) {
    __syncthreads();  // the ring's logits and scores are read: its first bytes take the work arrays
    int* mrank = reinterpret_cast<int*>(ring);
    int* hrank = mrank + E;
    int* cand = hrank + E;
    int* vict = cand + a.S;
    int* hit_t = vict + a.S;
    int* miss_t = hit_t + kQDMaxN;
    const uint32_t stamp = s_stamp + 1u;
    const ManageCounts mc = manage_block(E, a.S, a.policy, false, stamp, s_cnt, st_e2s, st_s2e, st_prio, mrank,
                                         hrank, cand, vict, hit_t, miss_t, st_miss_s, nullptr, nullptr, a.r.status);
    // the list: hits (ascending id), then the misses in load order (ascending id)
    const bool ok = mc.nh + mc.nl == s_nact && mc.nl <= kQDMaxN;
    if (ok)
      for (int i = tid; i < s_nact; i += kQDThreads) {
        const int e = i < mc.nh ? hit_t[i] : miss_t[i - mc.nh];
        s_act[i] = e;
        s_li[e] = i;
      }
    // a step whose wait gave up before this point leaves the state (and the pool) as it was
    if (blockIdx.x == 0 && !*abort_flag) {
      for (int e = tid; e < E; e += kQDThreads) a.e2s_g[e] = st_e2s[e];
      for (int s = tid; s < a.S; s += kQDThreads) {
        a.s2e_g[s] = st_s2e[s];
        a.prio_g[s] = st_prio[s];
      }
      if (tid == 0) {
        *a.stamp_g = stamp;
        if (a.stats) {
          a.stats[0] += mc.nl;
          a.stats[1] += 1;
          a.stats[2] += (int64_t)mc.nl * (int64_t)a.qslab;
        }
      }
    }
    if (tid == 0) {
      s_nh = mc.nh;
      s_nl = ok ? mc.nl : 0;
      if (!ok) {
        set_status(a.r.status, MOE_DEV_BAD_SLOT);
        s_abort = 1;
      }
    }
  }
  fence_async_smem();  // the ring's router bytes are overwritten by bulk copies next
  __syncthreads();

  // ---- 3-4. the two weight streams --------------------------------------------------------
  FfnArgs fa{};
  fa.E = E;
  fa.S = a.S;
  fa.e2s = kGather ? st_e2s : a.r.e2s;
  fa.list_e = s_act;
  fa.offset = s_off;
  const int n_list = s_nact;
  const int IQ = I / 4, NSRg = H / kQDK, NSRd = IQ / a.qd;
  // stage costs by the experts' rows; weighted ranges per CTA (the counters count stages, so parts
  // need no cap and no count)
  {
    int tot;  // n_list <= 64 < the block's threads: one scan
    const int wpre = block_exclusive_scan(tid < n_list ? q8d_stage_cost(s_cnt[s_act[tid]]) : 0, tmp, &tot);
    if (tid < n_list) s_wpre[tid] = wpre;
    if (tid == 0) s_wpre[n_list] = tot;
  }
  __syncthreads();
  // gather mode with misses: CTAs 0 .. gg-1 copy them, the others stream in phases
  const int nl = kGather ? s_nl : 0, nh = n_list - nl, nph = 1 + nl;
  const int gg = nl > 0 ? kQGCtas : 0;
  const int Gf = G - gg, fb = (int)blockIdx.x >= gg ? (int)blockIdx.x - gg : -1;
  const int wb_g = kQDK * I, wb_d = a.qd * 4 * H;  // bytes of one stage piece: Wg (or Wu), Wd
  const int Wg = NSRg * s_wpre[n_list], Wd = NSRd * s_wpre[n_list];  // resident mode: one phase
  const int bg = (int)(blockIdx.x * Wg / G), eg_end = (int)((blockIdx.x + 1) * Wg / G);
  const int bd = (int)(blockIdx.x * Wd / G), ed_end = (int)((blockIdx.x + 1) * Wd / G);
  const size_t slab_vec = a.qslab / 16;
  const int gpieces = kGather ? (int)((slab_vec + kQGPieceVec - 1) / kQGPieceVec) : 0;

  // ---- 3'. gather mode: the copying CTAs, miss after miss (the next piece's host loads in flight while
  // this piece is stored, fenced and released) ------------------------------------------------------
  if constexpr (kGather) {
    if ((int)blockIdx.x < gg && !*abort_flag) {
      const int items = nl * gpieces;
      auto piece = [&](int it, const uint4*& src, uint4*& dst, size_t& lim) {
        const int m = it / gpieces, c = it - m * gpieces;
        const int e = s_act[nh + m], sl = st_miss_s[m];
        if (e < 0 || e >= E || sl < 0 || sl >= a.S) {
          if (tid == 0) set_status(a.r.status, e < 0 || e >= E ? MOE_DEV_BAD_EXPERT : MOE_DEV_BAD_SLOT);
          return false;
        }
        src = a.host + (size_t)e * slab_vec + (size_t)c * kQGPieceVec;
        dst = a.pool_w + (size_t)sl * slab_vec + (size_t)c * kQGPieceVec;
        lim = min((size_t)kQGPieceVec, slab_vec - (size_t)c * kQGPieceVec);
        return true;
      };
      uint4 v[kQGUnroll], nv[kQGUnroll];
      const uint4* src = nullptr;
      uint4* dst = nullptr;
      size_t lim = 0;
      bool ok = (int)blockIdx.x < items && piece(blockIdx.x, src, dst, lim);
      if (ok)
#pragma unroll
        for (int u = 0; u < kQGUnroll; ++u) {
          const size_t j = tid + (size_t)u * kQDThreads;
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
          for (int u = 0; u < kQGUnroll; ++u) {
            const size_t j = tid + (size_t)u * kQDThreads;
            if (j < nlim) nv[u] = ldg_stream(nsrc + j);
          }
        if (ok) {
#pragma unroll
          for (int u = 0; u < kQGUnroll; ++u) {
            const size_t j = tid + (size_t)u * kQDThreads;
            if (j < lim) dst[j] = v[u];
          }
          q8_fence_async_global();  // the piece is read next by other CTAs' bulk copies
        }
        __syncthreads();
        if (tid == 0) add_release(&gctr[it / gpieces], 1);  // the barrier orders every thread's stores before it
#pragma unroll
        for (int u = 0; u < kQGUnroll; ++u) v[u] = nv[u];
        ok = nok;
        dst = ndst;
        lim = nlim;
      }
    }
  }

  if (warp == kQDConsumers / 32) {
    if (lane == 0) {
      uint32_t it = 0;
      int last_use[kQDMaxStages];
      for (int s = 0; s < kQDMaxStages; ++s) last_use[s] = -1;
      auto claim = [&](int sl, uint32_t use) {
        if (use > 0 && !*abort_flag && !mbar_wait(&empty[sl], (use - 1) & 1u)) {
          *abort_flag = 1;
          set_status(a.r.status, MOE_DEV_TIMEOUT);
        }
        return !*abort_flag;
      };
      // gather mode: a missing expert's slot is read once all of its pieces are in (bit m: miss m seen complete)
      uint64_t seen = 0;
      auto slab_ready = [&](int e) {
        if constexpr (kGather) {
          const int m = s_li[e] - nh;
          if (m < 0 || m >= kQDMaxN || ((seen >> m) & 1ull)) return true;
          if (*abort_flag) return false;
          if (!wait_count(&gctr[m], gpieces, a.r.status)) {
            *abort_flag = 1;
            return false;
          }
          q8_fence_async_global();  // the copy's generic stores before this thread's bulk copies of the slot
          seen |= 1ull << m;
        }
        return true;
      };
      auto gate_up = [&](const StreamSeg& g) {
        if (!slab_ready(g.e)) return false;
        const unsigned char* w = a.pool + (size_t)g.slot * a.qslab;
        for (int s = g.s_lo; s < g.s_hi; ++s, ++it) {
          const int sl = it % a.nst;
          const uint32_t use = it / a.nst;
          if (!claim(sl, use)) return false;
          unsigned char* dst = ring + sl * a.stride;
          mbar_expect_tx(&full[sl], 2 * wb_g);
          bulk_load(dst, w + (size_t)s * wb_g, wb_g, &full[sl]);
          bulk_load(dst + wb_g, w + mat + (size_t)s * wb_g, wb_g, &full[sl]);
          last_use[sl] = (int)use;
        }
        return true;
      };
      auto down = [&](const StreamSeg& g) {
        if (!slab_ready(g.e)) return false;
        const unsigned char* w = a.pool + (size_t)g.slot * a.qslab + 2 * mat;
        for (int s = g.s_lo; s < g.s_hi; ++s, ++it) {
          const int sl = it % a.nst;
          const uint32_t use = it / a.nst;
          if (!claim(sl, use)) return false;
          mbar_expect_tx(&full[sl], wb_d);
          bulk_load(ring + sl * a.stride, w + (size_t)s * wb_d, wb_d, &full[sl]);
          last_use[sl] = (int)use;
        }
        return true;
      };
      if constexpr (!kGather) {
        if (bg < eg_end) q8d_segments(fa, s_wpre, n_list, NSRg, bg, eg_end, gate_up);
        if (bd < ed_end) q8d_segments(fa, s_wpre, n_list, NSRd, bd, ed_end, down);
      } else {
        bool go = true;
        for (int p = 0; p < nph && go; ++p) {
          q8d_phase(fa, s_wpre, nh, NSRg, Gf, fb, p, [&](const StreamSeg& g) { return go = gate_up(g); });
          if (go) q8d_phase(fa, s_wpre, nh, NSRd, Gf, fb, p, [&](const StreamSeg& g) { return go = down(g); });
        }
      }
      if (*abort_flag)  // let every copy issued land before the CTA moves on
        for (int s = 0; s < a.nst; ++s)
          if (last_use[s] >= 0) mbar_wait(&full[s], (uint32_t)last_use[s] & 1u);
    }
  } else {
    const int c = tid;  // output columns 4c .. 4c + 3
    uint32_t it = 0;
    // bad slots: the schedule skips the expert; report it once
    if (blockIdx.x == 0 && c < n_list) {
      int e, slot;
      if (!stream_slot(fa, c, e, slot)) set_status(a.r.status, MOE_DEV_BAD_SLOT);
    }
    // wait for stage it's bytes; false once the CTA gave up
    auto stage_in = [&](int sl) {
      if (!*abort_flag && !mbar_wait(&full[sl], (it / a.nst) & 1u)) {
        *abort_flag = 1;
        set_status(a.r.status, MOE_DEV_TIMEOUT);
      }
      return !*abort_flag;
    };
    auto stage_out = [&](int sl) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[sl]);
    };
    auto cons_gate_up = [&](const StreamSeg& g) {
        // the stage loop for RB >= nb rows (rows past nb take token 0's codes and are not kept); RB is a
        // compile-time count, so a one-row expert costs one code load and 16 dp4a per stage
        auto stages = [&](auto rbc) {
          constexpr int RB = decltype(rbc)::value;
          const bool act = c < I / 2;  // [Wg | Wu] has 2I columns: I / 2 groups of 4
          const int off = 4 * c < I ? 16 * c : wb_g + 16 * c - 4 * I;
          int xr[RB];  // the rows' code offsets in xq
#pragma unroll
          for (int r = 0; r < RB; ++r) xr[r] = (r < g.nb ? s_rows[g.p0 + r] / k : 0) * (H / 4);
          int acc[RB][4] = {};
          for (int s = g.s_lo; s < g.s_hi; ++s, ++it) {
            const int sl = it % a.nst;
            if (stage_in(sl) && act) {
              const unsigned char* st = ring + sl * a.stride + off;
              int4 xv[RB];
#pragma unroll
              for (int r = 0; r < RB; ++r) xv[r] = *reinterpret_cast<const int4*>(xq + xr[r] + 4 * s);
#pragma unroll
              for (int qq = 0; qq < 4; ++qq) {
                const int4 w = *reinterpret_cast<const int4*>(st + qq * 4 * I);
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                  const int x = quad_of(xv[r], qq);
                  acc[r][0] = __dp4a(w.x, x, acc[r][0]);
                  acc[r][1] = __dp4a(w.y, x, acc[r][1]);
                  acc[r][2] = __dp4a(w.z, x, acc[r][2]);
                  acc[r][3] = __dp4a(w.w, x, acc[r][3]);
                }
              }
            }
            stage_out(sl);
          }
          if (act && !*abort_flag)
#pragma unroll
            for (int r = 0; r < RB; ++r)
              if (r < g.nb) {
                int32_t* dst = a.gsum + (size_t)(g.p0 + r) * 2 * I + 4 * c;
                atomicAdd(dst, acc[r][0]);
                atomicAdd(dst + 1, acc[r][1]);
                atomicAdd(dst + 2, acc[r][2]);
                atomicAdd(dst + 3, acc[r][3]);
              }
        };
        if (g.nb <= 1) stages(std::integral_constant<int, 1>{});
        else if (g.nb <= 2) stages(std::integral_constant<int, 2>{});
        else if (g.nb <= 4) stages(std::integral_constant<int, 4>{});
        else stages(std::integral_constant<int, 8>{});
        // publish this part (the barrier orders every consumer's atomics before the release)
        named_sync(1, kQDConsumers);
        if (c == 0) add_release(&ctr[s_li[g.e]], g.s_hi - g.s_lo);
        return true;
      };
    auto cons_down = [&](const StreamSeg& g) {
        const int li = s_li[g.e], nb = g.nb, nit = nb * IQ;
        // h of the segment's rows from the gate/up sums: items (row, quad), up to four per thread, two at a
        // time.  The first two items' scales do not depend on h: they are loaded before the wait for the
        // expert's parts.
        const float4* sc4 = reinterpret_cast<const float4*>(a.pool + (size_t)g.slot * a.qslab + 3 * mat);
        float4 sg4[2], su4[2];
        // gather mode: a missing expert's scales are written by this launch's copy, so they are read
        // (coherently) once the copy is complete; a hit's are in place and go the read-only path early
        const bool late = kGather && li >= nh;
        auto load_sc = [&](int u, int v) {
          const int q = v % IQ;
          if (kGather && late) {
            sg4[u] = __ldcg(sc4 + q);
            su4[u] = __ldcg(sc4 + IQ + q);
          } else {
            sg4[u] = __ldg(sc4 + q);
            su4[u] = __ldg(sc4 + IQ + q);
          }
        };
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int v = c + kQDConsumers * u;
          if (v < nit && !(kGather && late)) load_sc(u, v);
        }
        if (c == 0 && !*abort_flag && !wait_count(&ctr[li], NSRg, a.r.status)) *abort_flag = 1;
        if (kGather && late && c == 0 && !*abort_flag && !wait_count(&gctr[li - nh], gpieces, a.r.status))
          *abort_flag = 1;
        if (c < kQDRB) s_amax[c] = 0u;
        named_sync(1, kQDConsumers);
        const bool ok = !*abort_flag;
        float hv[4][4];
#pragma unroll
        for (int u0 = 0; u0 < 4; u0 += 2) {
          if (u0 > 0 || (kGather && late)) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int v = c + kQDConsumers * (u0 + u);
              if (v < nit) load_sc(u, v);
            }
          }
          int4 gi[2], ui[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {  // both items' sums in flight before the arithmetic
            const int v = c + kQDConsumers * (u0 + u);
            if (ok && v < nit) {
              const int r = v / IQ, q = v - r * IQ;
              const int32_t* gs = a.gsum + (size_t)(g.p0 + r) * 2 * I + 4 * q;
              gi[u] = __ldcg(reinterpret_cast<const int4*>(gs));
              ui[u] = __ldcg(reinterpret_cast<const int4*>(gs + I));
            }
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int v = c + kQDConsumers * (u0 + u);
            if (ok && v < nit) {
              const int r = v / IQ;
              const float s_x = s_sx[s_rows[g.p0 + r] / k];
              const int g4[4] = {gi[u].x, gi[u].y, gi[u].z, gi[u].w}, u4[4] = {ui[u].x, ui[u].y, ui[u].z, ui[u].w};
              const float sg[4] = {sg4[u].x, sg4[u].y, sg4[u].z, sg4[u].w};
              const float su[4] = {su4[u].x, su4[u].y, su4[u].z, su4[u].w};
              float hmax = 0.f;
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                const float gg = __fmul_rn(__fmul_rn(__int2float_rn(g4[b]), sg[b]), s_x);
                const float uu = __fmul_rn(__fmul_rn(__int2float_rn(u4[b]), su[b]), s_x);
                hv[u0 + u][b] = __fmul_rn(silu32_def(gg), uu);
                hmax = fmaxf(hmax, fabsf(hv[u0 + u][b]));
              }
              atomicMax(&s_amax[r], __float_as_uint(hmax));
            }
          }
        }
        named_sync(1, kQDConsumers);
        if (c < nb) {
          const float s = __fdiv_rn(__uint_as_float(s_amax[c]), 127.f);
          s_shr[c] = s;
          a.sh[g.p0 + c] = s;  // every CTA of this expert writes the same value
        }
        named_sync(1, kQDConsumers);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int v = c + kQDConsumers * u;
          if (ok && v < nit) {
            const int r = v / IQ, q = v - r * IQ;
            if (q >= a.qd * g.s_lo && q < a.qd * g.s_hi)
              hq[q * kQDRB + r] = (int32_t)pack_codes(hv[u][0], hv[u][1], hv[u][2], hv[u][3], s_shr[r]);
          }
        }
        named_sync(1, kQDConsumers);
        auto stages = [&](auto rbc) {
          constexpr int RB = decltype(rbc)::value;
          const bool act = c < H / 4;
          int acc[RB][4] = {};
          for (int s = g.s_lo; s < g.s_hi; ++s, ++it) {
            const int sl = it % a.nst;
            if (stage_in(sl) && act) {
              const unsigned char* st = ring + sl * a.stride + 16 * c;
#pragma unroll
              for (int qq = 0; qq < 4; ++qq)
                if (qq < a.qd) {
                  const int4 w = *reinterpret_cast<const int4*>(st + qq * 4 * H);
                  const int32_t* ha = hq + (a.qd * s + qq) * kQDRB;
#pragma unroll
                  for (int r = 0; r < RB; ++r) {
                    const int x = ha[r];
                    acc[r][0] = __dp4a(w.x, x, acc[r][0]);
                    acc[r][1] = __dp4a(w.y, x, acc[r][1]);
                    acc[r][2] = __dp4a(w.z, x, acc[r][2]);
                    acc[r][3] = __dp4a(w.w, x, acc[r][3]);
                  }
                }
            }
            stage_out(sl);
          }
          if (act && !*abort_flag)
#pragma unroll
            for (int r = 0; r < RB; ++r)
              if (r < nb) {
                int32_t* dst = a.ysum + (size_t)(g.p0 + r) * H + 4 * c;
                atomicAdd(dst, acc[r][0]);
                atomicAdd(dst + 1, acc[r][1]);
                atomicAdd(dst + 2, acc[r][2]);
                atomicAdd(dst + 3, acc[r][3]);
              }
        };
        if (nb <= 1) stages(std::integral_constant<int, 1>{});
        else if (nb <= 2) stages(std::integral_constant<int, 2>{});
        else if (nb <= 4) stages(std::integral_constant<int, 4>{});
        else stages(std::integral_constant<int, 8>{});
        return true;
      };
    if constexpr (!kGather) {
      if (bg < eg_end) q8d_segments(fa, s_wpre, n_list, NSRg, bg, eg_end, cons_gate_up);
      if (bd < ed_end) q8d_segments(fa, s_wpre, n_list, NSRd, bd, ed_end, cons_down);
    } else {
      q8d_phase(fa, s_wpre, nh, NSRg, Gf, fb, 0, cons_gate_up);
      q8d_phase(fa, s_wpre, nh, NSRd, Gf, fb, 0, cons_down);
#pragma unroll 1
      for (int p = 1; p < nph; ++p) {
        q8d_phase(fa, s_wpre, nh, NSRg, Gf, fb, p, cons_gate_up);
        q8d_phase(fa, s_wpre, nh, NSRd, Gf, fb, p, cons_down);
      }
    }
  }
  // ---- 5. combine: (token, column quad) items dealt round-robin over the grid, one thread per (item,
  // pick); a pick's scales are loaded before the grid-wide wait, its sums and row scale after it, and
  // the item's thread for pick 0 adds the picks in order
  const int nc4 = H / 4, nit = T * nc4;
  const int my_items = nit > (int)blockIdx.x ? (nit - 1 - (int)blockIdx.x) / G + 1 : 0;
  const bool cu = !*abort_flag && tid < my_items * k;  // the host checks my_items * k <= kQDThreads
  const int cm = cu ? tid / k : 0, cj = tid - cm * k;
  const int citem = (int)blockIdx.x + G * cm, ct = citem / nc4, cc4 = citem - ct * nc4;
  int cpos = 0, cslot = 0;
  bool chave = false;
  float4 csd = make_float4(0.f, 0.f, 0.f, 0.f);
  if (cu) {
    const int i = ct * k + cj, e = s_ids[i];
    const int slot = kGather ? st_e2s[e] : a.r.e2s ? a.r.e2s[e] : e;
    chave = slot >= 0 && slot < a.S;
    cpos = s_pos[i];
    // gather mode: after the grid-wide wait (every copy is complete by then), coherently
    if (chave && !kGather)
      csd = __ldg(reinterpret_cast<const float4*>(a.pool + (size_t)slot * a.qslab + 3 * mat) + (2 * I) / 4 + cc4);
    if constexpr (kGather) cslot = slot;
  }
  // the loader ran its loops on lane 0 alone: reconverge before the CTA barrier
  __syncwarp();
  __syncthreads();
  if (tid == 0) {
    add_release(&ctr[E + kQCtrDown], 1);
    if (!wait_count(&ctr[E + kQCtrDown], G, a.r.status)) s_abort = 1;
  }
  __syncthreads();
  if constexpr (kGather)
    if (cu && chave)
      csd = __ldcg(reinterpret_cast<const float4*>(a.pool + (size_t)cslot * a.qslab + 3 * mat) + (2 * I) / 4 + cc4);
  float4* sy = reinterpret_cast<float4*>(ring);  // every stage has landed and been read: the ring is free
  if (cu) {
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
    if (chave && !*abort_flag) {
      const int4 ys = __ldcg(reinterpret_cast<const int4*>(a.ysum + (size_t)cpos * H) + cc4);
      const float sh = __ldcg(a.sh + cpos);
      y.x = __fmul_rn(__fmul_rn(__int2float_rn(ys.x), csd.x), sh);
      y.y = __fmul_rn(__fmul_rn(__int2float_rn(ys.y), csd.y), sh);
      y.z = __fmul_rn(__fmul_rn(__int2float_rn(ys.z), csd.z), sh);
      y.w = __fmul_rn(__fmul_rn(__int2float_rn(ys.w), csd.w), sh);
    }
    sy[tid] = y;
  }
  __syncthreads();
  if (cu && cj == 0 && !*abort_flag) {
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; ++j) {
      const float wj = s_w[ct * k + j];
      const float4 y = sy[cm * k + j];
      o[0] = fmaf(wj, y.x, o[0]);
      o[1] = fmaf(wj, y.y, o[1]);
      o[2] = fmaf(wj, y.z, o[2]);
      o[3] = fmaf(wj, y.w, o[3]);
    }
    uint2 pk;
    pk.x = uint32_t(f32_to_bf16(o[0])) | (uint32_t(f32_to_bf16(o[1])) << 16);
    pk.y = uint32_t(f32_to_bf16(o[2])) | (uint32_t(f32_to_bf16(o[3])) << 16);
    *reinterpret_cast<uint2*>(a.out + (size_t)ct * H + 4 * cc4) = pk;
  }
  // the last CTA out resets the counters: every other CTA is past its last wait
  __syncthreads();
  if (tid == 0 && atomicAdd(&ctr[E + kQCtrExit], 1) == G - 1)
    for (int i = 0; i < E + kQCtrCount + (kGather ? kQDMaxN : 0); ++i) ctr[i] = 0;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static size_t qd_al(size_t v) { return (v + 255) & ~size_t(255); }

// A ring slot holds one gate/up stage (16 rows of Wg and of Wu) or, at least, one quad-row of Wd; a down
// stage takes as many whole quad-rows of Wd as fit in a slot (at most four) and divide I / 4.
static int qd_stride(int H, int I) { return std::max(2 * kQDK * I, 4 * H); }
static int qd_quads(int H, int I) {
  int q = std::min(4, qd_stride(H, I) / (4 * H));
  while ((I / 4) % q) --q;
  return q;
}

// Dynamic shared memory of one launch: x codes | ring | gather mode: the cache state's copy.
struct QdPlan {
  int nst = 0, state_off = 0;
  size_t smem = 0;
};

static bool qd_plan(int T, int H, int E, int I, int S, bool gather, QdPlan* p) {
  const size_t xq = ((size_t)T * H + 127) & ~size_t(127), fixed = xq + 128;
  const size_t state = gather ? (size_t)4 * (E + 2 * S + kQDMaxN) : 0;
  const int stride = qd_stride(H, I);
  if (fixed + state >= (size_t)kQDSmemMax) return false;
  p->nst = (int)std::min<size_t>(kQDMaxStages, (kQDSmemMax - fixed - state) / stride);
  if (p->nst < 2) return false;
  const size_t staging = (size_t)(kQDThreads / 32) * kRStage, route = (size_t)2 * T * E * 4;
  // the ring also holds the router's staging, the logits and scores, the combine's values and, in gather
  // mode, the manage call's work arrays
  size_t ring = std::max((size_t)p->nst * stride, std::max(staging, std::max(route, (size_t)16 * kQDThreads)));
  if (gather) ring = std::max(ring, (size_t)4 * (2 * E + 2 * S + 2 * kQDMaxN));
  ring = (ring + 15) & ~size_t(15);
  p->state_off = (int)(xq + ring);
  p->smem = fixed + ring + state;
  return p->smem <= (size_t)kQDSmemMax;
}

bool decode_q8_eligible(int T, int H, int E, int k, int I, int S, const void* x, const void* wr, const void* pool,
                        int sms) {
  const int n = T * k;
  if (sms < 1 || T < 1 || T > kQDMaxT || n > kQDMaxN || E > kQDMaxE || E % 8 || k > kMaxK) return false;
  // one consumer thread per 4 output columns: 2I <= 2048 and H <= 2048
  if (H % 128 || H > 4 * kQDConsumers || I % 16 || I > 2 * kQDConsumers || S < 1) return false;
  if ((uintptr_t)x % 16 || (uintptr_t)wr % 16 || (uintptr_t)pool % 16) return false;
  // at least four warps of a CTA are free of router units (they form the tokens' codes meanwhile)
  if ((H / 128) * ((E + 31) / 32) * T > (kQDThreads / 32 - 4) * sms) return false;
  // the combine gives each CTA's (item, pick) pairs one thread each
  if (((T * H / 4 + sms - 1) / sms) * k > kQDThreads) return false;
  QdPlan p;
  return qd_plan(T, H, E, I, S, false, &p);
}

bool decode_q8_gather_eligible(int T, int H, int E, int k, int I, int S, int policy, const void* x, const void* wr,
                               const void* pool, const void* host, int sms) {
  if (!decode_q8_eligible(T, H, E, k, I, S, x, wr, pool, sms)) return false;
  if (policy != MOE_POLICY_LRU && policy != MOE_POLICY_LFU) return false;
  // T*k <= S: every miss finds a victim among the slots the step does not need (one manage call)
  if (T * k > S || S > kQDMaxE || (uintptr_t)host % 16 || q8_slab_bytes_h(H, I) % 16) return false;
  if (sms < 2 * kQGCtas) return false;  // at least as many streaming CTAs as copying ones
  QdPlan p;
  return qd_plan(T, H, E, I, S, true, &p);
}

size_t decode_q8_ws_bytes(int T, int k, int H, int I) {
  const size_t n = (size_t)T * k;
  return qd_al(n * 2 * I * 4) + qd_al(n * H * 4) + qd_al(n * 4);
}

template <bool kGather>
static int launch_decode_q8_impl(const moe_layer_args* la, float* lpart, float* logits, void* ws, size_t ws_bytes,
                                 int32_t* ctr, cudaStream_t stream) {
  const int T = la->T, H = la->H, E = la->E, k = la->k, I = la->I, n = T * k;
  int dev = 0, sms = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  if (kGather ? !decode_q8_gather_eligible(T, H, E, k, I, la->S, la->policy, la->x, la->w_router, la->pool,
                                           la->host_slabs, sms)
              : !decode_q8_eligible(T, H, E, k, I, la->S, la->x, la->w_router, la->pool, sms))
    return MOE_ERR_ARG;
  if (!ws || ws_bytes < decode_q8_ws_bytes(T, k, H, I) || (uintptr_t)ws % 256) return MOE_ERR_ALIGN;
  DecodeQ8Args a{};
  a.r = RouteIO{(const uint16_t*)la->x, (const uint16_t*)la->w_router, la->logit_offset, la->sel_bias,
                kGather ? nullptr : la->e2s, la->affinity, la->route_flags, T, H, E, k, lpart, logits, la->ids,
                la->w, ctr + E + kQCtrRoute, la->dev_status};
  a.I = I;
  a.S = la->S;
  a.pool = (const unsigned char*)la->pool;
  a.qslab = q8_slab_bytes_h(H, I);
  char* b = (char*)ws;
  a.gsum = (int32_t*)b;
  b += qd_al((size_t)n * 2 * I * 4);
  a.ysum = (int32_t*)b;
  b += qd_al((size_t)n * H * 4);
  a.sh = (float*)b;
  a.ctr = ctr;
  a.out = (uint16_t*)la->out;
  a.stride = qd_stride(H, I);
  a.qd = qd_quads(H, I);
  if constexpr (kGather) {
    if (!la->e2s || !la->s2e || !la->prio || !la->stamp || !la->host_slabs) return MOE_ERR_ARG;
    a.e2s_g = la->e2s;
    a.s2e_g = la->s2e;
    a.prio_g = la->prio;
    a.stamp_g = la->stamp;
    a.policy = la->policy;
    a.host = (const uint4*)la->host_slabs;
    a.pool_w = (uint4*)la->pool;
    a.stats = la->stats;
  }
  QdPlan p;
  if (!qd_plan(T, H, E, I, la->S, kGather, &p)) return MOE_ERR_ARG;
  a.nst = p.nst;
  a.state_off = p.state_off;
  static bool attr[64] = {};
  MOE_CUDA_TRY(ensure_smem(decode_q8_kernel<kGather>, kQDSmemMax, attr));
  int occ = 0;
  MOE_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_q8_kernel<kGather>, kQDThreads, p.smem));
  if (occ < 1) return MOE_ERR_ARG;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kQDThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, decode_q8_kernel<kGather>, a));
  return MOE_OK;
}

int launch_decode_q8(const moe_layer_args* la, float* lpart, float* logits, void* ws, size_t ws_bytes, int32_t* ctr,
                     cudaStream_t stream) {
  return launch_decode_q8_impl<false>(la, lpart, logits, ws, ws_bytes, ctr, stream);
}

int launch_decode_q8_gather(const moe_layer_args* la, float* lpart, float* logits, void* ws, size_t ws_bytes,
                            int32_t* ctr, cudaStream_t stream) {
  return launch_decode_q8_impl<true>(la, lpart, logits, ws, ws_bytes, ctr, stream);
}

}  // namespace moe
