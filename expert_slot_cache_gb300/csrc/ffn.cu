// Grouped SwiGLU expert FFN, weight-streaming form for decode-sized groups.
//
// "Porting vllm-expert-cache to NVIDIA GPUs", "What this package does": the
// expert GEMM runs on slot-remapped ids.  "RTX 3060 runs a 35B MoE with
// llama.cpp", chapter "Designing a fixed expert cache with zero-return for
// missing experts": one pass over the experts in VRAM, one over the experts
// still in host memory.
//
// Work is a device-side list of experts.  Each (expert, column tile) work
// item streams that tile's weight columns once, 16 bytes per load, for all
// the expert's tokens (processed in batches of <= 8).  Threads own 8 output
// columns and walk the input dimension, with the activations broadcast from
// shared memory, so a thread accumulates its outputs in registers; the
// partial sums of the 32 k-groups are reduced in a fixed order.
//   gate/up : tile = 32 columns of Wg and the same 32 of Wu; h = silu(g) * u
//   down    : tile = 64 columns of Wd; y = h Wd
#include <algorithm>

#include "internal.cuh"
#include "tma.cuh"

namespace moe {

constexpr int kFfnThreads = 256;
constexpr int kRB = 8;       // tokens per batch (max)
constexpr int kUnroll = 8;   // weight rows in flight per thread
constexpr int kKG = 32;      // k-groups per CTA
constexpr int kGUTile = 32;  // gate/up columns per tile
constexpr int kDTile = 64;   // down columns per tile

__device__ __forceinline__ void unpack8(const uint4 v, float* f) {
  f[0] = bf16_lo(v.x);
  f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y);
  f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z);
  f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w);
  f[7] = bf16_hi(v.w);
}

// Weights of expert e (slot copy when resident, else the host store); NULL
// when the slot lies outside the pool's S slots (S = 0: not checked).
__device__ __forceinline__ const uint16_t* expert_weights(const FfnArgs& a, int e) {
  const int s = a.e2s ? a.e2s[e] : e;
  if (s >= 0) return (a.S > 0 && s >= a.S) ? nullptr : a.pool + (size_t)s * a.slab_elems;
  return a.host ? a.host + (size_t)e * a.slab_elems : nullptr;
}

// Stream K rows of a [K][ldw] matrix for this thread's 8 columns (wcol = column
// base) and accumulate acc[r][q] += w[row][q] * in[r][row] over rows
// row = g + kKG * j.
template <int RB>
__device__ __forceinline__ void stream_rows(const uint16_t* __restrict__ wcol, int ldw, int K, int g,
                                            const float* __restrict__ in_s, int ld_in, float (&acc)[RB][8]) {
  constexpr int U = RB >= 8 ? kUnroll / 2 : kUnroll;
  const int nrows = K / kKG;
  for (int j0 = 0; j0 < nrows; j0 += U) {
    uint4 wv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int row = g + kKG * (j0 + u);
      if (j0 + u < nrows) wv[u] = ldg_stream(wcol + (size_t)row * ldw);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (j0 + u < nrows) {
        const int row = g + kKG * (j0 + u);
        float wf[8];
        unpack8(wv[u], wf);
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          const float xv = in_s[r * ld_in + row];
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[r][q] = fmaf(wf[q], xv, acc[r][q]);
        }
      }
    }
  }
}

// Reduce acc over the 4 k-groups of a warp (lanes differing in bits 3 and 4)
// and store the warp partial of column-thread c = lane (lanes 0..7).
template <int RB>
__device__ __forceinline__ void warp_partials(float (&acc)[RB][8], float* __restrict__ red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int r = 0; r < RB; ++r)
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float v = acc[r][q];
      v += __shfl_xor_sync(MOE_FULL_MASK, v, 8);
      v += __shfl_xor_sync(MOE_FULL_MASK, v, 16);
      acc[r][q] = v;
    }
  if (lane < 8) {
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
      for (int q = 0; q < 8; ++q) red[((warp * 8 + lane) * RB + r) * 8 + q] = acc[r][q];
  }
}

template <int RB>
__device__ __forceinline__ void gateup_batch(const FfnArgs& a, const uint16_t* __restrict__ w, int i0, int p0,
                                             int nb, float* __restrict__ xs, float* __restrict__ red) {
  const int tid = threadIdx.x, c = tid & 7, g = tid >> 3;
  const int H = a.H, I = a.I;
  for (int idx = tid; idx < RB * H; idx += kFfnThreads) {
    const int r = idx / H, h = idx - r * H;
    float v = 0.f;
    if (r < nb) {
      const int t = a.rows[p0 + r] / a.k;
      v = bf16_to_f32(a.x[(size_t)t * H + h]);
    }
    xs[idx] = v;
  }
  __syncthreads();
  float acc[RB][8];
#pragma unroll
  for (int r = 0; r < RB; ++r)
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[r][q] = 0.f;
  // c < 4: gate columns i0 + 8c; c >= 4: up columns i0 + 8(c - 4)
  const uint16_t* mat = w + (c < 4 ? 0 : (size_t)H * I);
  const uint16_t* wcol = mat + i0 + 8 * (c & 3);
  stream_rows<RB>(wcol, I, H, g, xs, H, acc);
  warp_partials<RB>(acc, red);
  __syncthreads();
  for (int o = tid; o < kGUTile * RB; o += kFfnThreads) {
    const int r = o / kGUTile, il = o - r * kGUTile;
    const int cg = il >> 3, q = il & 7;
    float gs = 0.f, us = 0.f;
#pragma unroll
    for (int wp = 0; wp < kFfnThreads / 32; ++wp) {
      gs += red[((wp * 8 + cg) * RB + r) * 8 + q];
      us += red[((wp * 8 + cg + 4) * RB + r) * 8 + q];
    }
    if (r < nb) a.hbuf[(size_t)(p0 + r) * I + i0 + il] = gs / (1.f + expf(-gs)) * us;
  }
  __syncthreads();
}

template <int RB>
__device__ __forceinline__ void down_batch(const FfnArgs& a, const uint16_t* __restrict__ w, int o0, int p0, int nb,
                                           float* __restrict__ hs, float* __restrict__ red) {
  const int tid = threadIdx.x, c = tid & 7, g = tid >> 3;
  const int H = a.H, I = a.I;
  for (int idx = tid; idx < RB * I; idx += kFfnThreads) {
    const int r = idx / I, i = idx - r * I;
    hs[idx] = r < nb ? a.hbuf[(size_t)(p0 + r) * I + i] : 0.f;
  }
  __syncthreads();
  float acc[RB][8];
#pragma unroll
  for (int r = 0; r < RB; ++r)
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[r][q] = 0.f;
  const uint16_t* wd = w + 2 * (size_t)H * I;
  stream_rows<RB>(wd + o0 + 8 * c, H, I, g, hs, I, acc);
  warp_partials<RB>(acc, red);
  __syncthreads();
  for (int o = tid; o < kDTile * RB; o += kFfnThreads) {
    const int r = o / kDTile, ol = o - r * kDTile;
    const int cg = ol >> 3, q = ol & 7;
    float s = 0.f;
#pragma unroll
    for (int wp = 0; wp < kFfnThreads / 32; ++wp) s += red[((wp * 8 + cg) * RB + r) * 8 + q];
    if (r < nb) a.y[(size_t)(p0 + r) * H + o0 + ol] = s;
  }
  __syncthreads();
}

template <bool kDown>
__global__ void __launch_bounds__(kFfnThreads, 1) ffn_kernel(const FfnArgs a) {
  extern __shared__ __align__(16) float ffn_smem[];
  float* in_s = ffn_smem;                             // [kRB][K]
  float* red = ffn_smem + kRB * (kDown ? a.I : a.H);  // [8 warps][8][kRB][8]
  const int tiles = kDown ? a.H / kDTile : a.I / kGUTile;
  const int nl = *a.n_list;
  const int items = nl * tiles;
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int li = it / tiles, tile = it - li * tiles;
    const int e = a.list_e[li];
    if (e < 0 || e >= a.E) {
      if (threadIdx.x == 0) set_status(a.status, MOE_DEV_BAD_EXPERT);
      continue;
    }
    const uint16_t* w = expert_weights(a, e);
    if (!w) {
      if (threadIdx.x == 0) set_status(a.status, MOE_DEV_BAD_SLOT);
      continue;
    }
    const int pb = a.offset[e], pe = a.offset[e + 1];
    for (int p0 = pb; p0 < pe; p0 += kRB) {
      const int nb = min(kRB, pe - p0);
      if (kDown) {
        const int o0 = tile * kDTile;
        if (nb == 1) down_batch<1>(a, w, o0, p0, nb, in_s, red);
        else if (nb == 2) down_batch<2>(a, w, o0, p0, nb, in_s, red);
        else if (nb <= 4) down_batch<4>(a, w, o0, p0, nb, in_s, red);
        else down_batch<8>(a, w, o0, p0, nb, in_s, red);
      } else {
        const int i0 = tile * kGUTile;
        if (nb == 1) gateup_batch<1>(a, w, i0, p0, nb, in_s, red);
        else if (nb == 2) gateup_batch<2>(a, w, i0, p0, nb, in_s, red);
        else if (nb <= 4) gateup_batch<4>(a, w, i0, p0, nb, in_s, red);
        else gateup_batch<8>(a, w, i0, p0, nb, in_s, red);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// TMA-staged variant (weights in the slot pool).
//
// Same work items, thread mapping, summation order and reduction as
// ffn_kernel, but the weight tiles are brought into a ring of shared-memory
// stages by one producer thread with 3-D tensor-map bulk copies
// (cp.async.bulk.tensor), so the bytes in flight no longer sit in registers.
// Warps 0-7 consume, warp 8 produces.  The pool is viewed as 3*S matrices of
// H*I bf16: gate of slot s = matrix 3s, up = 3s+1 (both [H][I]), down = 3s+2
// ([I][H]).  A stage holds kKB rows of the tile (16 KB).
// ---------------------------------------------------------------------------
constexpr int kStages = 10;
constexpr int kKB = 128;
constexpr int kStageBytes = 16384;
constexpr int kTmaConsumers = 512;             // 16 consumer warps
constexpr int kTmaKG = kTmaConsumers / 8;      // 64 k-groups of 8 column threads
constexpr int kTmaRB = 4;                      // tokens per batch
constexpr int kTmaThreads = kTmaConsumers + 32;

__device__ __forceinline__ int ffn_slot_of(const FfnArgs& a, int e) { return a.e2s ? a.e2s[e] : e; }

// Packed fp32 pairs for fma.rn.f32x2 (two independent IEEE fp32 fmas).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint64_t f2_bf16(uint32_t v) {  // bf16 pair -> fp32 pair (exact)
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(v << 16), "r"(v & 0xffff0000u));
  return r;
}
__device__ __forceinline__ void f2_fma(uint64_t& d, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 f;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
  return f;
}

// Activations of one row for RB tokens from the [K][RB] staging layout.
template <int RB>
__device__ __forceinline__ void load_row_x(const float* __restrict__ xs, int row, float (&xv)[RB]) {
  const float* p = xs + (size_t)row * RB;
  if (RB == 1) {
    xv[0] = p[0];
  } else if (RB == 2) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    xv[0] = v.x;
    xv[1] = v.y;
  } else {
#pragma unroll
    for (int r4 = 0; r4 < RB / 4; ++r4) {
      const float4 v = *reinterpret_cast<const float4*>(p + 4 * r4);
      xv[4 * r4] = v.x;
      xv[4 * r4 + 1] = v.y;
      xv[4 * r4 + 2] = v.z;
      xv[4 * r4 + 3] = v.w;
    }
  }
}

template <bool kDown, int RB>
__device__ __forceinline__ void tma_consume_batch(const FfnArgs& a, int tile, int p0, int nb, unsigned char* stages,
                                                  uint64_t* full, uint64_t* empty, float* __restrict__ in_s,
                                                  float* __restrict__ red, uint32_t& it, volatile int* abort_flag,
                                                  bool restage) {
  const int tid = threadIdx.x, c = tid & 7, g = tid >> 3, lane = tid & 31;
  const int H = a.H, I = a.I;
  const int K = kDown ? I : H;
  // Stage the batch's inputs (x rows, or h rows) as fp32 [K][RB]: thread owns
  // input index kk and writes the RB token values of it side by side.
  named_sync(1, kTmaConsumers);
  if (restage) {
    int tok[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) tok[r] = (!kDown && r < nb) ? a.rows[p0 + r] / a.k : 0;
    for (int kk = tid; kk < K; kk += kTmaConsumers) {
      float v[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        if (r < nb)
          v[r] = kDown ? a.hbuf[(size_t)(p0 + r) * I + kk] : bf16_to_f32(a.x[(size_t)tok[r] * H + kk]);
        else
          v[r] = 0.f;
      }
      float* dst = in_s + (size_t)kk * RB;
      if (RB == 1) {
        dst[0] = v[0];
      } else if (RB == 2) {
        *reinterpret_cast<float2*>(dst) = make_float2(v[0], v[1]);
      } else {
#pragma unroll
        for (int r4 = 0; r4 < RB / 4; ++r4)
          *reinterpret_cast<float4*>(dst + 4 * r4) = make_float4(v[4 * r4], v[4 * r4 + 1], v[4 * r4 + 2], v[4 * r4 + 3]);
      }
    }
    named_sync(1, kTmaConsumers);
  }
  uint64_t acc2[RB][4];  // acc2[r][p] = columns (2p, 2p+1) of token r
#pragma unroll
  for (int r = 0; r < RB; ++r)
#pragma unroll
    for (int p = 0; p < 4; ++p) acc2[r][p] = 0ull;
  // byte offset of this thread's 16 bytes within a stage row block
  const int mat_off = kDown ? 0 : (c < 4 ? 0 : kStageBytes / 2);
  const int row_bytes = kDown ? kDTile * 2 : kGUTile * 2;
  const int col_off = kDown ? 16 * c : 16 * (c & 3);
  const int nkc = K / kKB;
  for (int kc = 0; kc < nkc; ++kc, ++it) {
    const int sl = it % kStages;
    const uint32_t use = it / kStages;
    if (!*abort_flag && !mbar_wait(&full[sl], use & 1u)) {
      *abort_flag = 1;
      set_status(a.status, MOE_DEV_TIMEOUT);
    }
    const unsigned char* st = stages + sl * kStageBytes + mat_off + col_off;
#pragma unroll
    for (int j = 0; j < kKB / kTmaKG; ++j) {
      const int rl = g + kTmaKG * j;
      const uint4 wv = *reinterpret_cast<const uint4*>(st + rl * row_bytes);
      const uint64_t w2[4] = {f2_bf16(wv.x), f2_bf16(wv.y), f2_bf16(wv.z), f2_bf16(wv.w)};
      float xv[RB];
      load_row_x<RB>(in_s, kc * kKB + rl, xv);
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        const uint64_t xb = f2_pack(xv[r], xv[r]);
#pragma unroll
        for (int p = 0; p < 4; ++p) f2_fma(acc2[r][p], w2[p], xb);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[sl]);
  }
  float acc[RB][8];
#pragma unroll
  for (int r = 0; r < RB; ++r)
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 f = f2_unpack(acc2[r][p]);
      acc[r][2 * p] = f.x;
      acc[r][2 * p + 1] = f.y;
    }
  warp_partials<RB>(acc, red);
  named_sync(1, kTmaConsumers);
  if (kDown) {
    const int o0 = tile * kDTile;
    for (int o = tid; o < kDTile * RB; o += kTmaConsumers) {
      const int r = o / kDTile, ol = o - r * kDTile;
      const int cg = ol >> 3, q = ol & 7;
      float s = 0.f;
#pragma unroll
      for (int wp = 0; wp < kTmaConsumers / 32; ++wp) s += red[((wp * 8 + cg) * RB + r) * 8 + q];
      if (r < nb) a.y[(size_t)(p0 + r) * H + o0 + ol] = s;
    }
  } else {
    const int i0 = tile * kGUTile;
    for (int o = tid; o < kGUTile * RB; o += kTmaConsumers) {
      const int r = o / kGUTile, il = o - r * kGUTile;
      const int cg = il >> 3, q = il & 7;
      float gs = 0.f, us = 0.f;
#pragma unroll
      for (int wp = 0; wp < kTmaConsumers / 32; ++wp) {
        gs += red[((wp * 8 + cg) * RB + r) * 8 + q];
        us += red[((wp * 8 + cg + 4) * RB + r) * 8 + q];
      }
      if (r < nb) a.hbuf[(size_t)(p0 + r) * I + i0 + il] = gs / (1.f + expf(-gs)) * us;
    }
  }
}

template <bool kDown>
__global__ void __launch_bounds__(kTmaThreads, 1) ffn_tma_kernel(const FfnArgs a,
                                                                 const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ __align__(16) unsigned char tsm_raw[];
  // stages start on a 1024-byte boundary (the allocation carries 1 KB of slack)
  unsigned char* tsm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tsm_raw) + 1023) & ~uintptr_t(1023));
  const int K = kDown ? a.I : a.H;
  unsigned char* stages = tsm;
  float* in_s = reinterpret_cast<float*>(tsm + kStages * kStageBytes);
  float* red = in_s + kTmaRB * K;
  uint64_t* full = reinterpret_cast<uint64_t*>(red + (kTmaConsumers / 32) * 8 * kTmaRB * 8);
  uint64_t* empty = full + kStages;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kTmaConsumers / 32);
    }
    s_abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  volatile int* abort_flag = &s_abort;
  const int tiles = kDown ? a.H / kDTile : a.I / kGUTile;
  const int items = *a.n_list * tiles;
  const int nkc = K / kKB;
  // Items are expert-major and dealt round-robin: at any moment neighbouring
  // CTAs stream neighbouring column tiles of the same weight rows, which keeps
  // DRAM rows open (a contiguous range per CTA would put ~150 different
  // experts' 64-byte slices in flight at once and halves the bandwidth).
  const int beg = blockIdx.x, step = gridDim.x;

  if (warp == kTmaConsumers / 32) {
    // producer
    if (lane == 0) {
      uint32_t it = 0;
      int last_use[kStages];
      for (int s = 0; s < kStages; ++s) last_use[s] = -1;
      for (int item = beg; item < items && !*abort_flag; item += step) {
        const int li = item / tiles, tile = item - li * tiles;
        const int e = a.list_e[li];
        if (e < 0 || e >= a.E) continue;
        const int slot = ffn_slot_of(a, e);
        if (slot < 0 || slot >= a.S) continue;
        const int nbat = (a.offset[e + 1] - a.offset[e] + kTmaRB - 1) / kTmaRB;
        for (int b = 0; b < nbat; ++b) {
          for (int kc = 0; kc < nkc; ++kc, ++it) {
            const int sl = it % kStages;
            const uint32_t use = it / kStages;
            if (use > 0 && !*abort_flag && !mbar_wait(&empty[sl], (use - 1) & 1u)) {
              *abort_flag = 1;
              set_status(a.status, MOE_DEV_TIMEOUT);
            }
            if (*abort_flag) break;
            mbar_expect_tx(&full[sl], kStageBytes);
            unsigned char* dst = stages + sl * kStageBytes;
            if (kDown) {
              tma_load_3d(dst, &tmap, &full[sl], tile * kDTile, kc * kKB, 3 * slot + 2);
            } else {
              tma_load_3d(dst, &tmap, &full[sl], tile * kGUTile, kc * kKB, 3 * slot);
              tma_load_3d(dst + kStageBytes / 2, &tmap, &full[sl], tile * kGUTile, kc * kKB, 3 * slot + 1);
            }
            last_use[sl] = (int)use;
          }
        }
      }
      if (*abort_flag) {
        // let every copy this thread issued land before the CTA exits
        for (int s = 0; s < kStages; ++s)
          if (last_use[s] >= 0) mbar_wait(&full[s], (uint32_t)last_use[s] & 1u);
      }
    }
  } else {
    // consumers
    uint32_t it = 0;
    int staged_e = -1, staged_p0 = -1;
    for (int item = beg; item < items; item += step) {
      const int li = item / tiles, tile = item - li * tiles;
      const int e = a.list_e[li];
      if (e < 0 || e >= a.E) {
        if (threadIdx.x == 0) set_status(a.status, MOE_DEV_BAD_EXPERT);
        continue;
      }
      const int slot = ffn_slot_of(a, e);
      if (slot < 0 || slot >= a.S) {
        if (threadIdx.x == 0) set_status(a.status, MOE_DEV_BAD_SLOT);
        continue;
      }
      const int pb = a.offset[e], pe = a.offset[e + 1];
      for (int p0 = pb; p0 < pe; p0 += kTmaRB) {
        const int nb = min(kTmaRB, pe - p0);
        const bool restage = !(staged_e == e && staged_p0 == p0);
        staged_e = e;
        staged_p0 = p0;
        if (nb == 1)
          tma_consume_batch<kDown, 1>(a, tile, p0, nb, stages, full, empty, in_s, red, it, abort_flag, restage);
        else if (nb == 2)
          tma_consume_batch<kDown, 2>(a, tile, p0, nb, stages, full, empty, in_s, red, it, abort_flag, restage);
        else
          tma_consume_batch<kDown, 4>(a, tile, p0, nb, stages, full, empty, in_s, red, it, abort_flag, restage);
      }
    }
  }
  __syncthreads();
}

static size_t tma_smem_bytes(int K) {
  return 1024 + (size_t)kStages * kStageBytes +
         (size_t)(kTmaRB * K + (kTmaConsumers / 32) * 8 * kTmaRB * 8) * sizeof(float) + 2 * kStages * sizeof(uint64_t);
}

static size_t ffn_smem_bytes(int K) { return (size_t)(kRB * K + 8 * 8 * kRB * 8) * sizeof(float); }

int launch_ffn(const FfnArgs& a, int max_list, cudaStream_t stream, Prof* prof) {
  if (max_list <= 0) return MOE_OK;
  if (prefill_eligible(a, a.T * a.k)) return launch_prefill(a, a.T * a.k, max_list, stream, prof);
  if (sk_eligible(a)) return launch_ffn_sk(a, max_list, stream, prof);
  constexpr int kSmemCap = 160 * 1024;
  const size_t smem_gu = ffn_smem_bytes(a.H), smem_d = ffn_smem_bytes(a.I);
  if (smem_gu > (size_t)kSmemCap || smem_d > (size_t)kSmemCap) return MOE_ERR_ARG;
  static bool done_gu[64] = {}, done_d[64] = {};
  MOE_CUDA_TRY(ensure_smem(ffn_kernel<false>, kSmemCap, done_gu));
  MOE_CUDA_TRY(ensure_smem(ffn_kernel<true>, kSmemCap, done_d));
  int dev = 0, sms = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int g1 = std::min(max_list * (a.I / kGUTile), sms);
  const int g2 = std::min(max_list * (a.H / kDTile), sms);
  const bool tma = a.pool_only && a.S > 0 && a.H % kKB == 0 && a.I % kKB == 0 && tma_smem_bytes(a.H) <= 220 * 1024;
  if (tma) {
    static bool done_t1[64] = {}, done_t2[64] = {};
    MOE_CUDA_TRY(ensure_smem(ffn_tma_kernel<false>, 220 * 1024, done_t1));
    MOE_CUDA_TRY(ensure_smem(ffn_tma_kernel<true>, 220 * 1024, done_t2));
    const size_t mat = (size_t)a.H * a.I;
    CUtensorMap m_gu, m_d;
    const uint64_t d_gu[3] = {(uint64_t)a.I, (uint64_t)a.H, 3ull * a.S};
    const uint64_t s_gu[2] = {(uint64_t)a.I * 2, mat * 2};
    const uint32_t b_gu[3] = {kGUTile, kKB, 1};
    const uint64_t d_d[3] = {(uint64_t)a.H, (uint64_t)a.I, 3ull * a.S};
    const uint64_t s_d[2] = {(uint64_t)a.H * 2, mat * 2};
    const uint32_t b_d[3] = {kDTile, kKB, 1};
    int r = encode_tmap_3d_bf16(&m_gu, a.pool, d_gu, s_gu, b_gu, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (r != MOE_OK) return r;
    r = encode_tmap_3d_bf16(&m_d, a.pool, d_d, s_d, b_d, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (r != MOE_OK) return r;
    if (prof) prof->begin(MOE_PROF_FFN_GATEUP, stream);
    ffn_tma_kernel<false><<<g1, kTmaThreads, tma_smem_bytes(a.H), stream>>>(a, m_gu);
    MOE_LAUNCH_CHECK();
    if (prof) prof->end(stream);
    if (prof) prof->begin(MOE_PROF_FFN_DOWN, stream);
    ffn_tma_kernel<true><<<g2, kTmaThreads, tma_smem_bytes(a.I), stream>>>(a, m_d);
    MOE_LAUNCH_CHECK();
    if (prof) prof->end(stream);
    return MOE_OK;
  }
  if (prof) prof->begin(MOE_PROF_FFN_GATEUP, stream);
  ffn_kernel<false><<<g1, kFfnThreads, smem_gu, stream>>>(a);
  MOE_LAUNCH_CHECK();
  if (prof) prof->end(stream);
  if (prof) prof->begin(MOE_PROF_FFN_DOWN, stream);
  ffn_kernel<true><<<g2, kFfnThreads, smem_d, stream>>>(a);
  MOE_LAUNCH_CHECK();
  if (prof) prof->end(stream);
  return MOE_OK;
}

// ---------------------------------------------------------------------------
// Combine: out[t] = sum_j w[t][j] y[pos[t*k+j]] in fp32, j ascending.
// ---------------------------------------------------------------------------
constexpr int kCombThreads = 128;

// Combine over CPT columns per thread (4 from fp32 y, 8 from bf16 y: one 16-byte load per row either way),
// for k <= KM (the per-row registers are sized by KM, so k <= 8 keeps twice as many threads resident).
template <int CPT, int KM>
__global__ void __launch_bounds__(kCombThreads) combine_kernel(const float* __restrict__ y, const float* __restrict__ w,
                                                               const int32_t* __restrict__ pos,
                                                               const int32_t* __restrict__ ids,
                                                               const int32_t* __restrict__ e2s, int k, int H, int E,
                                                               int split, uint16_t* __restrict__ out,
                                                               float* __restrict__ out_res,
                                                               float* __restrict__ out_miss,
                                                               const uint16_t* __restrict__ yb) {
  pdl_trigger();
  pdl_wait();  // launched as a dependent of the FFN's last kernel: y is complete
  const int t = blockIdx.x;
  const int c = (blockIdx.y * kCombThreads + threadIdx.x) * CPT;
  if (c >= H) return;
  // all k rows first (independent loads), then the sum in j order
  uint4 raw[KM];
  float wj[KM];
  bool res[KM], have[KM];
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    have[j] = false;
    res[j] = true;
    wj[j] = 0.f;
    if (j < k) {
      const int p = pos[(size_t)t * k + j];
      if (p >= 0) {
        have[j] = true;
        wj[j] = w[(size_t)t * k + j];
        raw[j] = CPT == 8 ? *reinterpret_cast<const uint4*>(yb + (size_t)p * H + c)
                          : *reinterpret_cast<const uint4*>(y + (size_t)p * H + c);
        if (split) {
          const int e = ids[(size_t)t * k + j];
          res[j] = e >= 0 && e < E && e2s[e] >= 0;
        }
      }
    }
  }
  float acc[CPT], accm[CPT];
#pragma unroll
  for (int q = 0; q < CPT; ++q) acc[q] = accm[q] = 0.f;
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    if (j < k && have[j]) {
      float v[CPT];
      if (CPT == 8) {
        v[0] = bf16_lo(raw[j].x); v[1] = bf16_hi(raw[j].x); v[2] = bf16_lo(raw[j].y); v[3] = bf16_hi(raw[j].y);
        v[4] = bf16_lo(raw[j].z); v[5] = bf16_hi(raw[j].z); v[6] = bf16_lo(raw[j].w); v[7] = bf16_hi(raw[j].w);
      } else {
        v[0] = __uint_as_float(raw[j].x); v[1] = __uint_as_float(raw[j].y);
        v[2] = __uint_as_float(raw[j].z); v[3] = __uint_as_float(raw[j].w);
      }
#pragma unroll
      for (int q = 0; q < CPT; ++q) {
        if (res[j]) acc[q] = fmaf(wj[j], v[q], acc[q]);
        else accm[q] = fmaf(wj[j], v[q], accm[q]);
      }
    }
  }
  const size_t o = (size_t)t * H + c;
  float tot[CPT];
#pragma unroll
  for (int q = 0; q < CPT; ++q) tot[q] = split ? acc[q] + accm[q] : acc[q];
  if (split) {
#pragma unroll
    for (int q4 = 0; q4 < CPT / 4; ++q4) {
      *reinterpret_cast<float4*>(out_res + o + 4 * q4) = make_float4(acc[4 * q4], acc[4 * q4 + 1], acc[4 * q4 + 2], acc[4 * q4 + 3]);
      *reinterpret_cast<float4*>(out_miss + o + 4 * q4) =
          make_float4(accm[4 * q4], accm[4 * q4 + 1], accm[4 * q4 + 2], accm[4 * q4 + 3]);
    }
  }
  uint32_t pk[CPT / 2];
#pragma unroll
  for (int q = 0; q < CPT / 2; ++q) pk[q] = uint32_t(f32_to_bf16(tot[2 * q])) | (uint32_t(f32_to_bf16(tot[2 * q + 1])) << 16);
  if (CPT == 8) *reinterpret_cast<uint4*>(out + o) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  else *reinterpret_cast<uint2*>(out + o) = make_uint2(pk[0], pk[1]);
}

int launch_combine(const float* y, const float* w, const int32_t* pos, const int32_t* ids, const int32_t* e2s, int T,
                   int k, int H, int E, int split, void* out, float* out_res, float* out_miss, cudaStream_t stream,
                   const uint16_t* yb) {
  const bool k8 = k <= 8;
  if (yb) {
    const dim3 grid(T, (H / 8 + kCombThreads - 1) / kCombThreads);
    if (k8)
      MOE_CUDA_TRY(launch_pdl(combine_kernel<8, 8>, grid, dim3(kCombThreads), 0, stream, y, w, pos, ids, e2s, k, H, E,
                              split, (uint16_t*)out, out_res, out_miss, yb));
    else
      MOE_CUDA_TRY(launch_pdl(combine_kernel<8, kMaxK>, grid, dim3(kCombThreads), 0, stream, y, w, pos, ids, e2s, k, H,
                              E, split, (uint16_t*)out, out_res, out_miss, yb));
  } else {
    const dim3 grid(T, (H / 4 + kCombThreads - 1) / kCombThreads);
    if (k8)
      MOE_CUDA_TRY(launch_pdl(combine_kernel<4, 8>, grid, dim3(kCombThreads), 0, stream, y, w, pos, ids, e2s, k, H, E,
                              split, (uint16_t*)out, out_res, out_miss, (const uint16_t*)nullptr));
    else
      MOE_CUDA_TRY(launch_pdl(combine_kernel<4, kMaxK>, grid, dim3(kCombThreads), 0, stream, y, w, pos, ids, e2s, k, H,
                              E, split, (uint16_t*)out, out_res, out_miss, (const uint16_t*)nullptr));
  }
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe
