// Decode expert FFN as a balanced stream over full weight rows, on tcgen05.
//
// The expert GEMM of "Porting vllm-expert-cache to NVIDIA GPUs" ("What this
// package does": the expert GEMM runs on slot-remapped ids) for decode-sized
// groups, where it is a weight stream: every listed expert's weights are read
// once per batch of up to 16 of its tokens.
//
// Work split ("stream-K"): the listed experts' matrices are cut into stages
// of 16 consecutive input rows times all output columns.  The n_list * NSR
// stages of a pass are dealt out as contiguous, equal ranges of L stages, one
// range per CTA, so every SM streams the same number of weight bytes however
// many experts there are.  A CTA whose range covers part of an expert writes
// that part's sums, for all output columns and the batch's tokens, to
//   part[j][p][N],  j = CTA index - first CTA of the expert,
// and a reduce kernel adds the parts in j order: for gate/up it forms
// h = silu(g) * u (bf16, the down pass's operand), for down it writes y.  All
// sums run in a fixed order, so results do not depend on timing.
//
// Math: per stage and per 128 output columns, one tcgen05.mma with M = 128
// output columns (A = the stage's weights, MN-major, 128-byte swizzle as the
// tensor-map load writes it), N = 16 tokens (B = the tokens' activations for
// the stage's 16 rows, K-major, no swizzle) and K = 16, accumulating in TMEM.
// Roles: warp 0 loads (TMA), warp 1 issues the MMAs, warps 2-5 move finished
// accumulators (TMEM, double-buffered) to the parts.  Every wait is bounded.
//
// Activations, per stage and token batch: the gate/up pass copies batches of
// one or two tokens straight from x (16-byte bulk copies, one per token and 8
// rows), larger batches from x grouped by expert (two boxes of 8 rows x 16
// tokens, written by a row gather launched just before); the down pass copies
// the batch's h rows (bf16, grouped order) that the gate/up reduce wrote.
// Both passes are launched as programmatic dependents: they set up and stream
// their first weight stages before they wait (griddepcontrol.wait) for the
// kernel before them, and the gate/up pass waits only when a batch needs the
// grouped rows (and once before it exits).
#include <algorithm>

#include "internal.cuh"
#include "sched.cuh"
#include "tc05.cuh"

namespace moe {

constexpr int kDM = 128;                          // output columns per MMA (M)
constexpr int kDN = 16;                           // tokens per batch (N)
constexpr int kDK = 16;                           // weight rows per stage (K)
constexpr int kDBoxBytes = 64 * kDK * 2;          // one {64 columns x 16 rows} weight box, 2 KB
constexpr int kDActBox = 8 * kDN * 2;             // one {8 rows x 16 tokens} activation box, 256 B
constexpr int kDRing = 200 * 1024;
constexpr int kDMaxStages = 8;
constexpr int kDThreads = 192;
constexpr uint32_t kDTmemMax = 512;
constexpr int kDJcapMax = 160;
// Bytes of parts per pass (soft cap).  The buffer keeps all n rows per part index, so the cap limits the
// parts of a short expert list (the sub-batches of an expert-wave step): 64 MB lets 8 experts of a 64-token
// step spread over about 100-150 CTAs instead of 16-32 (the step 2.95 -> 2.90 ms); only the parts a list
// uses are written.
constexpr size_t kDPartBudget = size_t(64) << 20;
constexpr int kDMaxRows = 4096;
constexpr int kDDirectMax = 2;  // gate/up batches of at most this many tokens read x directly
constexpr uint32_t kDIdesc = idesc_bf16(kDM, kDN, 1, 0);

struct SkPass {
  float* part;  // [jcap][n][N]
  int N, K;     // output columns, weight rows
  int ntiles;   // N / 128
  int NSR;      // stages per expert
  int nst;      // ring stages
  int wbytes;   // weight bytes per stage
  int stride;   // stage stride in shared memory
  int G, jcap;
  uint32_t tcols;  // TMEM columns allocated: two accumulator buffers, rounded up to a power of two
};

// Accumulator columns 0..W-1 (tokens) of every tile -> parts; loads of up to
// 32 registers are issued before one wait.
template <int W>
__device__ __forceinline__ void sk_epilogue(uint32_t taddr, float* base, const SkPass& sp, int nb) {
  constexpr int G = W >= 32 ? 1 : 32 / W;
  for (int m0 = 0; m0 < sp.ntiles; m0 += G) {
    float v[G][W];
#pragma unroll
    for (int gi = 0; gi < G; ++gi)
      if (m0 + gi < sp.ntiles) tmem_ld_w<W>(taddr + (m0 + gi) * kDN, v[gi]);
    tmem_ld_wait();
#pragma unroll
    for (int gi = 0; gi < G; ++gi)
      if (m0 + gi < sp.ntiles)
#pragma unroll
        for (int t = 0; t < W; ++t)
          if (t < nb) base[(size_t)t * sp.N + (m0 + gi) * kDM] = v[gi][t];
  }
}

template <bool DOWN>
__global__ void __launch_bounds__(kDThreads, 1) ffn_sk_kernel(const FfnArgs a, const SkPass sp,
                                                              const __grid_constant__ CUtensorMap mw,
                                                              const __grid_constant__ CUtensorMap mact) {
  extern __shared__ __align__(16) unsigned char sk_raw[];
  unsigned char* ring =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(sk_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + sp.nst * sp.stride);
  uint64_t* empty = full + kDMaxStages;
  uint64_t* tfull = empty + kDMaxStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    prefetch_tmap(&mw);
    prefetch_tmap(&mact);
  }
  // the lists predate the kernel before (the row gather, or the gate/up reduce)
  const int n_list = *a.n_list;
  const int n = a.T * a.k;
  const int L = n_list > 0 ? stream_len(n_list, sp.NSR, sp.G, sp.jcap) : 1;
  const int total = n_list * sp.NSR;
  const int beg = blockIdx.x * L, end = min(beg + L, total);
  if (beg >= end) {  // uniform over the CTA: nothing allocated yet
    pdl_wait();       // still complete only after the kernel before
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < sp.nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], 4);
    }
    mbar_init(done, 1);
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, sp.tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;
  const uint32_t acc_cols = (uint32_t)sp.ntiles * kDN;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool waited = false;
      int ndef = 0, d_row[kDMaxStages], d_p0[kDMaxStages], last_use[kDMaxStages];
      for (int s = 0; s < kDMaxStages; ++s) last_use[s] = -1;
      // rows p0..p0+15 of x grouped (gate/up) or of h (down), 8 rows per box -> core matrices [k group][token][8]
      auto issue_act = [&](int sl, int row0, int p0) {
        unsigned char* dst = ring + sl * sp.stride + sp.wbytes;
        tma_load_3d(dst, &mact, &full[sl], row0, p0, 0);
        tma_load_3d(dst + kDActBox, &mact, &full[sl], row0 + 8, p0, 0);
      };
      auto flush = [&]() {
        pdl_wait();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        for (int d = 0; d < ndef; ++d) issue_act(d, d_row[d], d_p0[d]);
        ndef = 0;
        waited = true;
      };
      stream_segments<kDN>(a, sp.NSR, L, beg, end, [&](const StreamSeg& g) {
        const bool direct = !DOWN && g.nb <= kDDirectMax;
        int tok[kDDirectMax];
        if (direct)
          for (int t = 0; t < g.nb; ++t) tok[t] = a.rows[g.p0 + t] / a.k;
        if (!DOWN && !direct && !waited) flush();  // grouped rows: the row gather must be done
        for (int s = g.s_lo; s < g.s_hi; ++s, ++it) {
          const int sl = it % sp.nst;
          const uint32_t use = it / sp.nst;
          if (use > 0) {
            if (DOWN && !waited) flush();  // h copies deferred so far must go before a slot is reused
            if (!*abort_flag && !mbar_wait(&empty[sl], (use - 1) & 1u)) {
              *abort_flag = 1;
              set_status(a.status, MOE_DEV_TIMEOUT);
            }
          }
          if (*abort_flag) return false;
          unsigned char* dst = ring + sl * sp.stride;
          const int row0 = s * kDK;
          mbar_expect_tx(&full[sl], sp.wbytes + (direct ? g.nb * 32 : 2 * kDActBox));
          // weights: one 4-D box per matrix = 16 rows x all columns, as 64-column swizzle atoms 2 KB apart
          if (DOWN) {
            tma_load_4d(dst, &mw, &full[sl], 0, row0, 0, 3 * g.slot + 2);
          } else {
            tma_load_4d(dst, &mw, &full[sl], 0, row0, 0, 3 * g.slot);
            tma_load_4d(dst + sp.wbytes / 2, &mw, &full[sl], 0, row0, 0, 3 * g.slot + 1);
          }
          if (direct) {
            // x[token][row0 .. row0+15] -> core matrices [k group][token][8]: 16-byte bulk copies
            unsigned char* act = dst + sp.wbytes;
            for (int t = 0; t < g.nb; ++t) {
              const uint16_t* xr = a.x + (size_t)tok[t] * a.H + row0;
              bulk_load(act + t * 16, xr, 16, &full[sl]);
              bulk_load(act + kDActBox + t * 16, xr + 8, 16, &full[sl]);
            }
          } else if (waited) {
            issue_act(sl, row0, g.p0);
          } else {
            d_row[ndef] = row0;
            d_p0[ndef] = g.p0;
            ++ndef;
          }
          last_use[sl] = (int)use;
        }
        return true;
      });
      // every issued stage gets its activation copies, so every full barrier completes;
      // and the kernel before has completed before this one does
      if (!waited) flush();
      if (*abort_flag)
        for (int s = 0; s < sp.nst; ++s)
          if (last_use[s] >= 0) mbar_wait(&full[s], (uint32_t)last_use[s] & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int li = beg / sp.NSR; li * sp.NSR < end; ++li) {
        int e, slot;
        if (!stream_slot(a, li, e, slot)) set_status(a.status, e < 0 || e >= a.E ? MOE_DEV_BAD_EXPERT : MOE_DEV_BAD_SLOT);
      }
      uint32_t it = 0, seg = 0;
      stream_segments<kDN>(a, sp.NSR, L, beg, end, [&](const StreamSeg& g) {
        const uint32_t buf = seg & 1u, use = seg >> 1;
        if (use > 0 && !*abort_flag && !mbar_wait(&tempty[buf], (use - 1) & 1u)) {
          *abort_flag = 1;
          set_status(a.status, MOE_DEV_TIMEOUT);
        }
        tc_fence_after();
        const uint32_t d = tmem + buf * acc_cols;
        for (int s = g.s_lo; s < g.s_hi; ++s, ++it) {
          const int sl = it % sp.nst;
          if (!*abort_flag && !mbar_wait(&full[sl], (it / sp.nst) & 1u)) {
            *abort_flag = 1;
            set_status(a.status, MOE_DEV_TIMEOUT);
          }
          tc_fence_after();
          if (!*abort_flag) {
            const uint32_t sa = smem_u32(ring + sl * sp.stride);
            // B: tokens x 16 rows, K-major core matrices: 8 rows apart = 256 B, 8 tokens apart = 128 B
            const uint64_t bd = smem_desc_l(sa + sp.wbytes, kDActBox, 128, kLayoutNone);
            for (int m = 0; m < sp.ntiles; ++m) {
              // A: 128 output columns = two 64-column boxes 2 KB apart, 8-row groups 1 KB apart
              const uint64_t ad = smem_desc_l(sa + m * 2 * kDBoxBytes, kDBoxBytes, 1024, kLayoutSw128);
              umma_f16(d + m * kDN, ad, bd, kDIdesc, s > g.s_lo);
            }
          }
          umma_commit(&empty[sl]);
        }
        umma_commit(&tfull[buf]);
        ++seg;
        return true;
      });
      // all MMAs issued by this thread have finished once `done` completes
      umma_commit(done);
      mbar_wait(done, 0);
    }
  } else {
    // epilogue warps 2..5; TMEM lane quarter q = warp % 4 holds output columns q*32 .. q*32+31 of each tile
    const int q = warp & 3;
    uint32_t seg = 0;
    stream_segments<kDN>(a, sp.NSR, L, beg, end, [&](const StreamSeg& g) {
      const uint32_t buf = seg & 1u, use = seg >> 1;
      if (!*abort_flag && !mbar_wait(&tfull[buf], use & 1u)) {
        *abort_flag = 1;
        set_status(a.status, MOE_DEV_TIMEOUT);
      }
      tc_fence_after();
      if (!*abort_flag) {
        float* base = sp.part + ((size_t)g.j * n + g.p0) * sp.N + q * 32 + lane;
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + buf * acc_cols;
        if (g.nb <= 1)
          sk_epilogue<1>(taddr, base, sp, g.nb);
        else if (g.nb <= 2)
          sk_epilogue<2>(taddr, base, sp, g.nb);
        else if (g.nb <= 4)
          sk_epilogue<4>(taddr, base, sp, g.nb);
        else if (g.nb <= 8)
          sk_epilogue<8>(taddr, base, sp, g.nb);
        else
          sk_epilogue<16>(taddr, base, sp, g.nb);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      ++seg;
      return true;
    });
  }
  // warps 0 and 1 ran their loops on lane 0 alone: reconverge before the CTA barrier
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, sp.tcols);
  }
}

// Adds the parts of each listed expert's rows.  An expert with four or more
// rows: its rows are spread over the warps and a lane adds its parts in j
// order.  Fewer rows: warp w sums parts j = w, w+8, ..., then the 8 warp sums
// are added in warp order.  Either order is fixed, so results do not depend
// on timing.
//   SWIGLU: hb [n][I] bf16 = silu(sum g) * (sum u); parts hold [g | u]
//   else:   y [n][H] fp32 = sum of parts
// A block covers 128 columns (32 lanes x float4) of one listed expert's rows.
constexpr int kSkRedWarps = 8;

template <bool SWIGLU>
__global__ void __launch_bounds__(32 * kSkRedWarps) sk_reduce_kernel(const FfnArgs a, const float* __restrict__ part,
                                                                     int N, int NSR, int G, int jcap,
                                                                     float* __restrict__ y,
                                                                     uint16_t* __restrict__ hb) {
  __shared__ float4 sg[kSkRedWarps][32], su[kSkRedWarps][32];
  pdl_trigger();
  // the lists and offsets predate the pass before: read them while it finishes
  const int li = blockIdx.y;
  const int n_list = *a.n_list;
  if (li >= n_list) {
    pdl_wait();  // complete only after the pass before (ordering for later kernels)
    return;
  }
  int e, slot;
  if (!stream_slot(a, li, e, slot)) {
    pdl_wait();
    return;
  }
  const int L = stream_len(n_list, NSR, G, jcap);
  const int J = stream_parts(li, NSR, L);
  const int n = a.T * a.k;
  const int ncol = SWIGLU ? N / 2 : N;
  const int ncol4 = ncol / 4;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c4 = blockIdx.x * 32 + lane;
  const int pb = a.offset[e], pe = a.offset[e + 1];
  const size_t pstride = (size_t)n * N;
  pdl_wait();
  if (pe - pb >= 4) {
    // enough rows to go around: warp w takes rows pb + w, pb + w + 8, ...; a lane adds its quad's parts in
    // j order, eight parts' loads in flight before their adds (no barriers on this path; the branch
    // depends only on the expert's row count, so it is uniform over the block)
    if (c4 < ncol4)
      for (int p = pb + w; p < pe; p += kSkRedWarps) {
        const float* src = part + (size_t)p * N + 4 * c4;
        float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
        for (int j0 = 0; j0 < J; j0 += 8) {
          float4 tg[8], tu[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            if (j0 + jj < J) {
              tg[jj] = *reinterpret_cast<const float4*>(src + (j0 + jj) * pstride);
              if (SWIGLU) tu[jj] = *reinterpret_cast<const float4*>(src + (j0 + jj) * pstride + ncol);
            }
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            if (j0 + jj < J) {
              g.x += tg[jj].x; g.y += tg[jj].y; g.z += tg[jj].z; g.w += tg[jj].w;
              if (SWIGLU) {
                u.x += tu[jj].x; u.y += tu[jj].y; u.z += tu[jj].z; u.w += tu[jj].w;
              }
            }
        }
        if (SWIGLU) {
          const float h0 = g.x / (1.f + expf(-g.x)) * u.x, h1 = g.y / (1.f + expf(-g.y)) * u.y;
          const float h2 = g.z / (1.f + expf(-g.z)) * u.z, h3 = g.w / (1.f + expf(-g.w)) * u.w;
          uint2 wv;
          wv.x = uint32_t(f32_to_bf16(h0)) | (uint32_t(f32_to_bf16(h1)) << 16);
          wv.y = uint32_t(f32_to_bf16(h2)) | (uint32_t(f32_to_bf16(h3)) << 16);
          *reinterpret_cast<uint2*>(hb + (size_t)p * ncol + 4 * c4) = wv;
        } else {
          *reinterpret_cast<float4*>(y + (size_t)p * ncol + 4 * c4) = g;
        }
      }
    return;
  }
  // few rows: the warps split each row's parts, then warp 0 adds the eight sums
  for (int p = pb; p < pe; ++p) {
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
    if (c4 < ncol4) {
      const float* src = part + (size_t)p * N + 4 * c4;
#pragma unroll 4
      for (int jj = w; jj < J; jj += kSkRedWarps) {
        const float4 t = *reinterpret_cast<const float4*>(src + jj * pstride);
        g.x += t.x;
        g.y += t.y;
        g.z += t.z;
        g.w += t.w;
        if (SWIGLU) {
          const float4 v = *reinterpret_cast<const float4*>(src + jj * pstride + ncol);
          u.x += v.x;
          u.y += v.y;
          u.z += v.z;
          u.w += v.w;
        }
      }
    }
    sg[w][lane] = g;
    if (SWIGLU) su[w][lane] = u;
    __syncthreads();
    if (w == 0 && c4 < ncol4) {
      for (int k2 = 1; k2 < kSkRedWarps; ++k2) {
        const float4 t = sg[k2][lane];
        g.x += t.x;
        g.y += t.y;
        g.z += t.z;
        g.w += t.w;
        if (SWIGLU) {
          const float4 v = su[k2][lane];
          u.x += v.x;
          u.y += v.y;
          u.z += v.z;
          u.w += v.w;
        }
      }
      if (SWIGLU) {
        const float h0 = g.x / (1.f + expf(-g.x)) * u.x, h1 = g.y / (1.f + expf(-g.y)) * u.y;
        const float h2 = g.z / (1.f + expf(-g.z)) * u.z, h3 = g.w / (1.f + expf(-g.w)) * u.w;
        uint2 wv;
        wv.x = uint32_t(f32_to_bf16(h0)) | (uint32_t(f32_to_bf16(h1)) << 16);
        wv.y = uint32_t(f32_to_bf16(h2)) | (uint32_t(f32_to_bf16(h3)) << 16);
        *reinterpret_cast<uint2*>(hb + (size_t)p * ncol + 4 * c4) = wv;
      } else {
        *reinterpret_cast<float4*>(y + (size_t)p * ncol + 4 * c4) = g;
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static int sk_jcap(int n, int N) {
  const size_t per = (size_t)n * N * 4;
  const size_t j = per ? kDPartBudget / per : 0;
  return (int)std::max<size_t>(3, std::min<size_t>(j, kDJcapMax));
}

static size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

static size_t sk_half_bytes(int n, int H, int I) {
  const size_t g = (size_t)sk_jcap(n, 2 * I) * n * 2 * I * 4, d = (size_t)sk_jcap(n, H) * n * H * 4;
  return al256(std::max(g, d));
}

// Layout: [gate/up parts | down parts] (two equal halves), then x grouped by
// expert (bf16 [n][H]) and h (bf16 [n][I], grouped order).  A chunk smaller
// than the one the buffer was sized for gets as many parts as fit.
size_t sk_part_bytes(int n, int H, int I) {
  if (n < 1 || n > kDMaxRows) return 0;
  return 2 * sk_half_bytes(n, H, I) + al256((size_t)n * H * 2) + al256((size_t)n * I * 2);
}

struct SkCarve {
  float *gpart, *ypart;
  uint16_t *xp, *hb;
  int jg, jd;
};

static bool sk_carve(const FfnArgs& a, SkCarve* c) {
  const int n = a.T * a.k;
  const size_t act = al256((size_t)n * a.H * 2) + al256((size_t)n * a.I * 2);
  if (!a.skp || a.skp_bytes < act + 512) return false;
  const size_t half = ((a.skp_bytes - act) / 2) & ~size_t(255);
  c->gpart = a.skp;
  c->ypart = a.skp + half / 4;
  c->xp = reinterpret_cast<uint16_t*>(reinterpret_cast<char*>(a.skp) + 2 * half);
  c->hb = c->xp + al256((size_t)n * a.H * 2) / 2;
  c->jg = (int)std::min<size_t>(sk_jcap(n, 2 * a.I), half / ((size_t)n * 2 * a.I * 4));
  c->jd = (int)std::min<size_t>(sk_jcap(n, a.H), half / ((size_t)n * a.H * 4));
  return c->jg >= 2 && c->jd >= 2;
}

bool sk_part_layout(int n, int H, int I, float* skp, size_t skp_bytes, float** gpart, float** ypart, int* jg,
                    int* jd) {
  FfnArgs a{};
  a.T = n;
  a.k = 1;
  a.H = H;
  a.I = I;
  a.skp = skp;
  a.skp_bytes = skp_bytes;
  SkCarve c;
  if (!sk_carve(a, &c)) return false;
  *gpart = c.gpart;
  *ypart = c.ypart;
  *jg = c.jg;
  *jd = c.jd;
  return true;
}

static bool sk_pass(bool down, const FfnArgs& a, int G, float* part, int jcap, SkPass* out) {
  SkPass sp{};
  sp.part = part;
  sp.N = down ? a.H : 2 * a.I;
  sp.K = down ? a.I : a.H;
  if (sp.N % kDM || sp.K % kDK) return false;
  if (!down && a.I % kDM) return false;  // a tile never straddles the gate and up columns
  sp.ntiles = sp.N / kDM;
  if ((uint32_t)sp.ntiles * kDN * 2 > kDTmemMax) return false;  // two accumulator buffers in TMEM
  sp.tcols = 32;
  while (sp.tcols < (uint32_t)sp.ntiles * kDN * 2) sp.tcols *= 2;
  sp.NSR = sp.K / kDK;
  sp.wbytes = sp.N * kDK * 2;
  sp.stride = sp.wbytes + 1024;  // activation boxes, padded so every stage starts 1 KB aligned
  sp.nst = std::min(kDMaxStages, kDRing / sp.stride);
  if (sp.nst < 2) return false;
  sp.G = G;
  sp.jcap = jcap;
  *out = sp;
  return true;
}

static size_t sk_smem(const SkPass& sp) { return 1024 + (size_t)sp.nst * sp.stride + (2 * kDMaxStages + 5) * 8; }

bool sk_eligible(const FfnArgs& a) {
  const int n = a.T * a.k;
  if (!a.pool_only || a.S <= 0 || n > kDMaxRows) return false;
  if ((uintptr_t)a.x % 16 || (uintptr_t)a.pool % 16 || (uintptr_t)a.skp % 256 || (uintptr_t)a.y % 16) return false;
  SkCarve c;
  if (!sk_carve(a, &c)) return false;
  SkPass g, d;
  return sk_pass(false, a, 1, nullptr, c.jg, &g) && sk_pass(true, a, 1, nullptr, c.jd, &d);
}

template <typename K, typename... Args>
static cudaError_t sk_launch(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

int launch_ffn_sk(const FfnArgs& a, int max_list, cudaStream_t stream, Prof* prof) {
  int dev = 0, sms = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int n = a.T * a.k;
  SkCarve c;
  if (!sk_carve(a, &c)) return MOE_ERR_ARG;
  SkPass g, d;
  if (!sk_pass(false, a, sms, c.gpart, c.jg, &g) || !sk_pass(true, a, sms, c.ypart, c.jd, &d)) return MOE_ERR_ARG;
  static bool done_g[64] = {}, done_d[64] = {};
  // the limit is raised once per device, to the largest ring any shape uses
  constexpr int kSmemMax = 1024 + kDRing + (2 * kDMaxStages + 5) * 8;
  MOE_CUDA_TRY(ensure_smem(ffn_sk_kernel<false>, kSmemMax, done_g));
  MOE_CUDA_TRY(ensure_smem(ffn_sk_kernel<true>, kSmemMax, done_d));
  const size_t mat = (size_t)a.H * a.I;
  CUtensorMap mwg, mwd, mx, mh;
  // weight matrices viewed as [matrix][column atom][row][64 columns]: one box = 16 rows x all columns
  {
    const uint64_t dims[4] = {64, (uint64_t)a.H, (uint64_t)a.I / 64, 3ull * a.S};
    const uint64_t str[3] = {(uint64_t)a.I * 2, 128, mat * 2};
    const uint32_t box[4] = {64, kDK, (uint32_t)a.I / 64, 1};
    if (encode_tmap_bf16(&mwg, a.pool, 4, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B) != MOE_OK) return MOE_ERR_CUDA;
  }
  {
    const uint64_t dims[4] = {64, (uint64_t)a.I, (uint64_t)a.H / 64, 3ull * a.S};
    const uint64_t str[3] = {(uint64_t)a.H * 2, 128, mat * 2};
    const uint32_t box[4] = {64, kDK, (uint32_t)a.H / 64, 1};
    if (encode_tmap_bf16(&mwd, a.pool, 4, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B) != MOE_OK) return MOE_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {(uint64_t)a.H, (uint64_t)n, 1};
    const uint64_t str[2] = {(uint64_t)a.H * 2, (uint64_t)n * a.H * 2};
    const uint32_t box[3] = {8, kDN, 1};
    if (encode_tmap_3d_bf16(&mx, c.xp, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE) != MOE_OK) return MOE_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {(uint64_t)a.I, (uint64_t)n, 1};
    const uint64_t str[2] = {(uint64_t)a.I * 2, (uint64_t)n * a.I * 2};
    const uint32_t box[3] = {8, kDN, 1};
    if (encode_tmap_3d_bf16(&mh, c.hb, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE) != MOE_OK) return MOE_ERR_CUDA;
  }
  const dim3 rg_gu((a.I / 4 + 31) / 32, max_list);
  const dim3 rg_d((a.H / 4 + 31) / 32, max_list);
  const dim3 rb(32 * kSkRedWarps);
  if (prof) prof->begin(MOE_PROF_FFN_GATEUP, stream);
  int r = launch_gather_rows(a.x, a.rows, n, a.H, a.k, c.xp, sms, stream);
  if (r != MOE_OK) return r;
  MOE_CUDA_TRY(sk_launch(ffn_sk_kernel<false>, dim3(sms), dim3(kDThreads), sk_smem(g), stream, true, a, g, mwg, mx));
  MOE_CUDA_TRY(sk_launch(sk_reduce_kernel<true>, rg_gu, rb, 0, stream, true, a,
                         (const float*)c.gpart, g.N, g.NSR, g.G, g.jcap, (float*)nullptr, c.hb));
  if (prof) prof->end(stream);
  if (prof) prof->begin(MOE_PROF_FFN_DOWN, stream);
  MOE_CUDA_TRY(sk_launch(ffn_sk_kernel<true>, dim3(sms), dim3(kDThreads), sk_smem(d), stream, true, a, d, mwd, mh));
  MOE_CUDA_TRY(sk_launch(sk_reduce_kernel<false>, rg_d, rb, 0, stream, true, a,
                         (const float*)c.ypart, d.N, d.NSR, d.G, d.jcap, a.y, (uint16_t*)nullptr));
  if (prof) prof->end(stream);
  return MOE_OK;
}

}  // namespace moe
