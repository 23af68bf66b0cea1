// Router (logits, soft-biased top-k, softmax weights) and the soft-bias table.
//
// Method: "Nudge, don't cut" (PGO-SGB), section "The method in five lines":
// experts outside the hot set get bias max(cap, ln(b / b_edge)); the top-k
// is picked by logit + bias; the weights are the router's own softmax over
// the k picked, from the unbiased logits.
#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "fp32def.cuh"
#include "perm_small.cuh"
#include "topk.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Bias table: one CTA of >= E threads (E <= 1024).  Runs once per layer.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) bias_table_kernel(const float* __restrict__ b, int E, int n_hot,
                                                          int mode, float cap, float* __restrict__ bias) {
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
      if (mode == MOE_BIAS_FLAT) {
        v = cap;
      } else if (mode == MOE_BIAS_HARD) {
        v = -INFINITY;
      } else {
        const double be = sb[e];
        v = be <= 0.0 ? cap : (float)fmax((double)cap, log(be / (double)edge));
      }
    }
    bias[e] = v;
  }
}

// ---------------------------------------------------------------------------
// Logits.  The fp32 order (the one the oracle follows): h is cut into blocks
// of 128 rows; block b gives part_b = fma chain from 0 over its rows in
// order; logit = 0 + part_0 + part_1 + ... in block order.
//
// logits_kernel: CTA = (8*CH tokens) x (32 experts), 256 threads: warp w owns
// token lanes t = w + 8c (c < CH), lane = expert.  Wr[:, e0:e0+32] and the
// CTA's x rows stream through a 4-stage cp.async ring of 128-row chunks (one
// chunk = one block), so the chains never wait on a global load.
// ---------------------------------------------------------------------------
constexpr int kRouteThreads = 256;
constexpr int kEB = 32;        // experts per CTA
constexpr int kHC = 128;       // rows of Wr per stage
constexpr int kRStages = 4;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool pred) {
  const int n = pred ? 16 : 0;  // src-size 0 zero-fills
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Packed fp32 pairs for fma.rn.f32x2 (two independent IEEE fp32 fmas).
__device__ __forceinline__ uint64_t rf2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void rf2_fma(uint64_t& d, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}
__device__ __forceinline__ float2 rf2_unpack(uint64_t v) {
  float2 f;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
  return f;
}

template <int CH>
__global__ void __launch_bounds__(kRouteThreads) logits_kernel(const uint16_t* __restrict__ x,
                                                               const uint16_t* __restrict__ wr,
                                                               const float* __restrict__ off, int T, int H, int E,
                                                               float* __restrict__ logits) {
  constexpr int TT = 8 * CH;
  constexpr int kXRow = kHC + 8;  // bf16 x row, padded against bank conflicts in the conversion
  pdl_trigger();
  // stage s: W [kHC][kEB] bf16 (8 KB) | x [TT][kXRow] bf16;  then xf [kHC][TT] fp32 (token-minor)
  constexpr int kWBytes = kHC * kEB * 2;
  constexpr int kXBytes = TT * kXRow * 2;
  constexpr int kStage = kWBytes + kXBytes;
  extern __shared__ __align__(16) unsigned char rsm[];
  float* xf = reinterpret_cast<float*>(rsm + kRStages * kStage);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * TT, e0 = blockIdx.y * kEB;
  const int nt = min(TT, T - t0);
  const int nchunk = (H + kHC - 1) / kHC;

  auto load_chunk = [&](int c, int st) {
    unsigned char* sw = rsm + st * kStage;
    unsigned char* sx = sw + kWBytes;
    const int h0 = c * kHC;
    for (int v = tid; v < kHC * 4; v += kRouteThreads) {
      const int r = v >> 2, q = v & 3;
      const bool ok = h0 + r < H && e0 + 8 * q < E;
      const uint16_t* src = ok ? wr + (size_t)(h0 + r) * E + e0 + 8 * q : wr;
      cp_async16(sw + r * 64 + q * 16, src, ok);
    }
    for (int v = tid; v < TT * (kHC / 8); v += kRouteThreads) {
      const int r = v / (kHC / 8), q = v % (kHC / 8);
      const bool ok = r < nt && h0 + 8 * q < H;
      const uint16_t* src = ok ? x + (size_t)(t0 + r) * H + h0 + 8 * q : x;
      cp_async16(sx + (r * kXRow + 8 * q) * 2, src, ok);
    }
  };

  // warp w owns tokens w*CH .. w*CH+CH-1; lane = expert
  float acc[CH];
#pragma unroll
  for (int c = 0; c < CH; ++c) acc[c] = 0.f;
#pragma unroll
  for (int c = 0; c < kRStages - 1; ++c) {
    if (c < nchunk) load_chunk(c, c);
    cp_async_commit();
  }
  for (int c = 0; c < nchunk; ++c) {
    cp_async_wait<kRStages - 2>();
    __syncthreads();
    if (c + kRStages - 1 < nchunk) load_chunk(c + kRStages - 1, (c + kRStages - 1) % kRStages);
    cp_async_commit();
    const unsigned char* sw = rsm + (c % kRStages) * kStage;
    const uint16_t* ws = reinterpret_cast<const uint16_t*>(sw);
    const uint16_t* xs = reinterpret_cast<const uint16_t*>(sw + kWBytes);
    const int hn = min(kHC, H - c * kHC);  // a multiple of 8
    // x of this chunk to fp32, token-minor, converted once for all 32 expert lanes
    for (int v = tid; v < TT * (kHC / 8); v += kRouteThreads) {
      const int r = v % TT, q = v / TT;
      const uint4 u = *reinterpret_cast<const uint4*>(xs + r * kXRow + 8 * q);
      float* d = xf + (8 * q) * TT + r;
      d[0 * TT] = bf16_lo(u.x);
      d[1 * TT] = bf16_hi(u.x);
      d[2 * TT] = bf16_lo(u.y);
      d[3 * TT] = bf16_hi(u.y);
      d[4 * TT] = bf16_lo(u.z);
      d[5 * TT] = bf16_hi(u.z);
      d[6 * TT] = bf16_lo(u.w);
      d[7 * TT] = bf16_hi(u.w);
    }
    __syncthreads();
    // this 128-row block's chains, then added to the logits in block order
    float part[CH];
    uint64_t part2[(CH + 1) / 2];
#pragma unroll
    for (int cc = 0; cc < CH; ++cc) part[cc] = 0.f;
#pragma unroll
    for (int p = 0; p < (CH + 1) / 2; ++p) part2[p] = 0ull;
    const float* xw = xf + warp * CH;
    for (int h = 0; h < hn; ++h) {
      const float wv = bf16_to_f32(ws[h * kEB + lane]);
      const float* xr = xw + h * TT;
      if (CH == 1) {
        part[0] = fmaf(xr[0], wv, part[0]);
      } else {
        const uint64_t w2 = rf2_pack(wv, wv);
#pragma unroll
        for (int p4 = 0; p4 < CH / 4 + (CH == 2 ? 1 : 0); ++p4) {
          if (CH == 2) {
            const float2 xv = *reinterpret_cast<const float2*>(xr);
            rf2_fma(part2[0], rf2_pack(xv.x, xv.y), w2);
          } else {
            const float4 xv = *reinterpret_cast<const float4*>(xr + 4 * p4);
            rf2_fma(part2[2 * p4], rf2_pack(xv.x, xv.y), w2);
            rf2_fma(part2[2 * p4 + 1], rf2_pack(xv.z, xv.w), w2);
          }
        }
      }
    }
    if (CH > 1) {
#pragma unroll
      for (int p = 0; p < CH / 2; ++p) {
        const float2 f = rf2_unpack(part2[p]);
        part[2 * p] = f.x;
        part[2 * p + 1] = f.y;
      }
    }
#pragma unroll
    for (int cc = 0; cc < CH; ++cc) acc[cc] += part[cc];
  }
  cp_async_wait<0>();
  const int e = e0 + lane;
  if (e < E) {
#pragma unroll
    for (int cc = 0; cc < CH; ++cc) {
      const int t = warp * CH + cc;
      if (t < nt) logits[(size_t)(t0 + t) * E + e] = off ? acc[cc] + off[e] : acc[cc];
    }
  }
}

// logits_block_kernel (small T): CTA = one 128-row block x 32 experts x
// 8*CH tokens; writes part[b][t][e].  topk_kernel adds the parts in order.
template <int CH>
__global__ void __launch_bounds__(kRouteThreads) logits_block_kernel(const uint16_t* __restrict__ x,
                                                                     const uint16_t* __restrict__ wr, int T, int H,
                                                                     int E, float* __restrict__ part) {
  constexpr int TT = 8 * CH;
  __shared__ __align__(16) uint16_t ws[kHC * kEB];
  __shared__ __align__(16) uint16_t xs[TT * kHC];
  pdl_trigger();  // the top-k launches meanwhile and waits for these parts
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x, e0 = blockIdx.y * kEB, t0 = blockIdx.z * TT;
  const int h0 = b * kHC;
  const int nt = min(TT, T - t0);
  const int hn = min(kHC, H - h0);
  for (int v = tid; v < kHC * 4; v += kRouteThreads) {
    const int r = v >> 2, q = v & 3;
    const bool ok = r < hn && e0 + 8 * q < E;
    cp_async16(reinterpret_cast<unsigned char*>(ws) + r * 64 + q * 16,
               ok ? wr + (size_t)(h0 + r) * E + e0 + 8 * q : wr, ok);
  }
  for (int v = tid; v < TT * (kHC / 8); v += kRouteThreads) {
    const int r = v / (kHC / 8), q = v % (kHC / 8);
    const bool ok = r < nt && 8 * q < hn;
    cp_async16(xs + r * kHC + 8 * q, ok ? x + (size_t)(t0 + r) * H + h0 + 8 * q : x, ok);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  float acc[CH];
#pragma unroll
  for (int cc = 0; cc < CH; ++cc) acc[cc] = 0.f;
  for (int hh = 0; hh < hn; hh += 8) {
    float wv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) wv[u] = bf16_to_f32(ws[(hh + u) * kEB + lane]);
#pragma unroll
    for (int cc = 0; cc < CH; ++cc) {
      const uint4 xv = *reinterpret_cast<const uint4*>(xs + (warp + 8 * cc) * kHC + hh);
      acc[cc] = fmaf(bf16_lo(xv.x), wv[0], acc[cc]);
      acc[cc] = fmaf(bf16_hi(xv.x), wv[1], acc[cc]);
      acc[cc] = fmaf(bf16_lo(xv.y), wv[2], acc[cc]);
      acc[cc] = fmaf(bf16_hi(xv.y), wv[3], acc[cc]);
      acc[cc] = fmaf(bf16_lo(xv.z), wv[4], acc[cc]);
      acc[cc] = fmaf(bf16_hi(xv.z), wv[5], acc[cc]);
      acc[cc] = fmaf(bf16_lo(xv.w), wv[6], acc[cc]);
      acc[cc] = fmaf(bf16_hi(xv.w), wv[7], acc[cc]);
    }
  }
  const int e = e0 + lane;
  if (e < E) {
#pragma unroll
    for (int cc = 0; cc < CH; ++cc) {
      const int t = warp + 8 * cc;
      if (t < nt) part[((size_t)b * T + t0 + t) * E + e] = acc[cc];
    }
  }
}

// logits_tile_kernel (large T): CTA = 64 tokens x 64 experts x one 128-row
// block, 128 threads; writes part[b][t][e].  The tile is converted to fp32
// in shared memory once (x token-minor, Wr expert-minor); thread (tx, ty)
// owns experts 4tx..4tx+3 and tokens 8ty..8ty+7, each chain an fma over the
// block's rows in order (packed fp32 pairs along the experts).  topk_kernel
// adds the parts in block order.
constexpr int kTT = 64;   // tokens per tile
constexpr int kTE = 64;   // experts per tile
constexpr int kTileThreads = 128;

__global__ void __launch_bounds__(kTileThreads) logits_tile_kernel(const uint16_t* __restrict__ x,
                                                                  const uint16_t* __restrict__ wr, int T, int H,
                                                                  int E, float* __restrict__ part) {
  extern __shared__ __align__(16) float tsm[];
  pdl_trigger();
  float* xf = tsm;               // [kHC][kTT]
  float* wf = tsm + kHC * kTT;   // [kHC][kTE]
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * kTT, e0 = blockIdx.y * kTE, b = blockIdx.z;
  const int h0 = b * kHC;
  const int hn = min(kHC, H - h0);  // a multiple of 8
  // x rows: chunk v = (token r, 8 rows q): lanes take consecutive tokens, so the
  // transposed fp32 stores of a warp hit 32 different banks
  for (int v = tid; v < kTT * (kHC / 8); v += kTileThreads) {
    const int r = v % kTT, q = v / kTT;
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (t0 + r < T && 8 * q < hn) u = *reinterpret_cast<const uint4*>(x + (size_t)(t0 + r) * H + h0 + 8 * q);
    float* d = xf + (8 * q) * kTT + r;
    d[0 * kTT] = bf16_lo(u.x);
    d[1 * kTT] = bf16_hi(u.x);
    d[2 * kTT] = bf16_lo(u.y);
    d[3 * kTT] = bf16_hi(u.y);
    d[4 * kTT] = bf16_lo(u.z);
    d[5 * kTT] = bf16_hi(u.z);
    d[6 * kTT] = bf16_lo(u.w);
    d[7 * kTT] = bf16_hi(u.w);
  }
  // Wr rows: chunk v = (row r, 8 experts q)
  for (int v = tid; v < kHC * (kTE / 8); v += kTileThreads) {
    const int r = v / (kTE / 8), q = v % (kTE / 8);
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (r < hn && e0 + 8 * q < E) u = *reinterpret_cast<const uint4*>(wr + (size_t)(h0 + r) * E + e0 + 8 * q);
    float4* d = reinterpret_cast<float4*>(wf + r * kTE + 8 * q);
    d[0] = make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
    d[1] = make_float4(bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w));
  }
  __syncthreads();
  const int tx = tid & 15, ty = tid >> 4;
  uint64_t acc[8][2];
#pragma unroll
  for (int t = 0; t < 8; ++t) acc[t][0] = acc[t][1] = 0ull;
#pragma unroll 4
  for (int h = 0; h < hn; ++h) {
    const float4 wv = *reinterpret_cast<const float4*>(wf + h * kTE + 4 * tx);
    const float4 xa = *reinterpret_cast<const float4*>(xf + h * kTT + 8 * ty);
    const float4 xb = *reinterpret_cast<const float4*>(xf + h * kTT + 8 * ty + 4);
    const uint64_t w01 = rf2_pack(wv.x, wv.y), w23 = rf2_pack(wv.z, wv.w);
    const float xs[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint64_t xx = rf2_pack(xs[t], xs[t]);
      rf2_fma(acc[t][0], w01, xx);
      rf2_fma(acc[t][1], w23, xx);
    }
  }
  const int e = e0 + 4 * tx;
  if (e < E) {  // E % 8 == 0, so all four experts are in range together
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int tt = t0 + 8 * ty + t;
      if (tt < T) {
        const float2 a01 = rf2_unpack(acc[t][0]), a23 = rf2_unpack(acc[t][1]);
        *reinterpret_cast<float4*>(part + ((size_t)b * T + tt) * E + e) = make_float4(a01.x, a01.y, a23.x, a23.y);
      }
    }
  }
}

// logits_full_kernel (many tokens): CTA = 64 tokens x 64 experts over all of
// H, 256 threads, writing the final logits (no block parts in global memory).
// Each 128-row block's bf16 tiles are copied with cp.async while the block
// before is computed (two staging buffers), converted to fp32 in shared memory
// (x token-minor, Wr expert-minor), then thread (tx, ty) runs, for experts
// 4tx..4tx+3 and tokens 4ty..4ty+3, one fma chain per logit over the block's
// rows in order from 0 (operands read four rows at a time) and adds each chain
// to the logit's running sum in block order: the same arithmetic, in the same
// order, as the block parts summed by topk_kernel.  One CTA per SM (128 of
// them at T = 4096, E = 128) with 8 warps, two per SM sub-partition.
constexpr int kFullThreads = 256;
constexpr int kFullXRow = kHC + 8;  // bf16 staging row of x, padded against bank conflicts in the conversion
constexpr int kFullStage = kTT * kFullXRow + kHC * kTE;  // bf16 elements per staging buffer

size_t logits_full_smem_bytes() {
  return (size_t)(kHC * kTT + kHC * kTE) * sizeof(float) + 2 * (size_t)kFullStage * 2;
}

__global__ void __launch_bounds__(kFullThreads) logits_full_kernel(const uint16_t* __restrict__ x,
                                                                  const uint16_t* __restrict__ wr,
                                                                  const float* __restrict__ off, int T, int H,
                                                                  int E, float* __restrict__ logits) {
  extern __shared__ __align__(16) float fsm[];
  pdl_trigger();
  float* xf = fsm;                                                           // [kHC][kTT]
  float* wf = fsm + kHC * kTT;                                               // [kHC][kTE]
  uint16_t* stg = reinterpret_cast<uint16_t*>(fsm + kHC * kTT + kHC * kTE);  // 2 x (x [kTT][kFullXRow] | Wr [kHC][kTE])
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * kTT, e0 = blockIdx.y * kTE;
  const int nblk = (H + kHC - 1) / kHC;
  auto issue = [&](int b, int st) {
    uint16_t* sx = stg + st * kFullStage;
    uint16_t* sw = sx + kTT * kFullXRow;
    const int h0 = b * kHC, hn = min(kHC, H - h0);
    for (int v = tid; v < kTT * (kHC / 8); v += kFullThreads) {
      const int r = v / (kHC / 8), q = v % (kHC / 8);
      const bool ok = t0 + r < T && 8 * q < hn;
      cp_async16(sx + r * kFullXRow + 8 * q, ok ? x + (size_t)(t0 + r) * H + h0 + 8 * q : x, ok);
    }
    for (int v = tid; v < kHC * (kTE / 8); v += kFullThreads) {
      const int r = v / (kTE / 8), q = v % (kTE / 8);
      const bool ok = r < hn && e0 + 8 * q < E;
      cp_async16(sw + r * kTE + 8 * q, ok ? wr + (size_t)(h0 + r) * E + e0 + 8 * q : wr, ok);
    }
  };
  issue(0, 0);
  cp_async_commit();
  if (nblk > 1) issue(1, 1);
  cp_async_commit();
  // warp = 8 expert quads x 4 token quads: a row's operands are one 128-byte and one 64-byte
  // shared-memory read per warp
  const int lane = tid & 31, warp = tid >> 5;
  const int tx = (lane & 7) + 8 * (warp & 1), ty = (lane >> 3) + 4 * (warp >> 1);
  float total[4][4];  // [expert 4tx + i][token 4ty + t]
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int t = 0; t < 4; ++t) total[i][t] = 0.f;
  for (int b = 0; b < nblk; ++b) {
    cp_async_wait<1>();  // block b has landed (block b + 1 may still be in flight)
    __syncthreads();     // ... for every thread's copies; and block b - 1's chains are done with xf / wf
    const uint16_t* sx = stg + (b & 1) * kFullStage;
    const uint16_t* sw = sx + kTT * kFullXRow;
    const int hn = min(kHC, H - b * kHC);  // a multiple of 8
    // x: chunk v = (token r, 8 rows q), lanes on consecutive tokens (conflict-free transposed stores)
    for (int v = tid; v < kTT * (kHC / 8); v += kFullThreads) {
      const int r = v % kTT, q = v / kTT;
      const uint4 u = *reinterpret_cast<const uint4*>(sx + r * kFullXRow + 8 * q);
      float* d = xf + (8 * q) * kTT + r;
      d[0 * kTT] = bf16_lo(u.x);
      d[1 * kTT] = bf16_hi(u.x);
      d[2 * kTT] = bf16_lo(u.y);
      d[3 * kTT] = bf16_hi(u.y);
      d[4 * kTT] = bf16_lo(u.z);
      d[5 * kTT] = bf16_hi(u.z);
      d[6 * kTT] = bf16_lo(u.w);
      d[7 * kTT] = bf16_hi(u.w);
    }
    // Wr: chunk v = (row r, 8 experts q)
    for (int v = tid; v < kHC * (kTE / 8); v += kFullThreads) {
      const int r = v / (kTE / 8), q = v % (kTE / 8);
      const uint4 u = *reinterpret_cast<const uint4*>(sw + r * kTE + 8 * q);
      float4* d = reinterpret_cast<float4*>(wf + r * kTE + 8 * q);
      d[0] = make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
      d[1] = make_float4(bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w));
    }
    __syncthreads();  // the fp32 tiles are complete, and staging buffer b & 1 is free again
    if (b + 2 < nblk) issue(b + 2, b & 1);
    cp_async_commit();
    // chains over the block: acc[i][t] = fma chain of expert 4tx + i and token 4ty + t, rows in
    // order; four rows of operands are read before their 64 fmas
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int t = 0; t < 4; ++t) acc[i][t] = 0.f;
    const float* wrow = wf + 4 * tx;
    const float* xrow = xf + 4 * ty;
#pragma unroll 1
    for (int h = 0; h < hn; h += 4) {  // hn is a multiple of 8
      float4 wv[4], xv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        wv[u] = *reinterpret_cast<const float4*>(wrow + (h + u) * kTE);
        xv[u] = *reinterpret_cast<const float4*>(xrow + (h + u) * kTT);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float w4[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w}, x4[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int t = 0; t < 4; ++t) acc[i][t] = fmaf(x4[t], w4[i], acc[i][t]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int t = 0; t < 4; ++t) total[i][t] = total[i][t] + acc[i][t];
  }
  cp_async_wait<0>();
  const int e = e0 + 4 * tx;
  if (e < E) {  // E % 8 == 0, so all four experts are in range together
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (off) o = make_float4(off[e], off[e + 1], off[e + 2], off[e + 3]);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int tt = t0 + 4 * ty + t;
      if (tt < T) {
        float4 v = make_float4(total[0][t], total[1][t], total[2][t], total[3][t]);
        if (off) v = make_float4(v.x + o.x, v.y + o.y, v.z + o.z, v.w + o.w);
        *reinterpret_cast<float4*>(logits + (size_t)tt * E + e) = v;
      }
    }
  }
}

// Top-k: one warp per token.  k rounds of a warp-wide argmax over
// score = logit + bias (ties -> lower id); the winner is marked taken.
// Weights: softmax over the k picked, from the unbiased logits.  NQ = 32-expert
// slots per lane (E <= 32 * NQ).
// ---------------------------------------------------------------------------
template <int NQ>
__global__ void __launch_bounds__(kRouteThreads) topk_kernel(float* __restrict__ logits,
                                                             const float* __restrict__ bias,
                                                             const int32_t* __restrict__ e2s, float affinity,
                                                             const float* __restrict__ part, int nb,
                                                             const float* __restrict__ off, int T, int E, int k,
                                                             int tpc, int rflags, int32_t* __restrict__ ids,
                                                             float* __restrict__ wout, const PermOut perm) {
  __shared__ float sel_l[kRouteThreads / 32][kMaxK];
  __shared__ int sel_i[kRouteThreads / 32][kMaxK];
  pdl_trigger();
  pdl_wait();  // launched as a dependent of the logits kernel: its parts / logits are complete
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tb = blockIdx.x * tpc;  // tokens tb .. tb+tpc-1, one warp each (tpc <= 8)
  if (part) {
    // finish this CTA's logits from the block parts: 0 + part_0 + part_1 + ...
    // (a value's parts are loaded, 16 at a time, before its in-order sum), then the offset
    const int nt = min(tpc, T - tb);
    const size_t bstride = (size_t)T * E;
    for (int v = threadIdx.x; v < nt * E; v += kRouteThreads) {
      const int tl = v / E, e = v - tl * E;
      const float* pp = part + (size_t)(tb + tl) * E + e;
      float l = 0.f;
      for (int b = 0; b < nb; b += 16) {
        float pv[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) pv[u] = b + u < nb ? pp[(size_t)(b + u) * bstride] : 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u)
          if (b + u < nb) l += pv[u];
      }
      logits[(size_t)(tb + tl) * E + e] = off ? l + off[e] : l;
    }
    __syncthreads();
  }
  const int t = tb + warp;
  if (warp < tpc && t < T)
    topk_token_impl<NQ>(logits, bias, e2s, affinity, E, k, rflags, t, warp, lane, sel_l, sel_i, ids, wout);
  // a CTA that routed the whole batch also groups it by expert (the ids it wrote are visible to the
  // block after the barrier)
  if (perm.count && gridDim.x == 1) {
    __syncthreads();
    permute_small_block(ids, T * k, E, perm);
  }
}

// Top-k launch (a programmatic dependent of the logits kernel) with the fewest 32-expert slots per lane
// that hold E.
static cudaError_t launch_topk(int grid, cudaStream_t s, float* logits, const float* bias, const int32_t* e2s,
                               float affinity, const float* part, int nb, const float* off, int T, int E, int k,
                               int tpc, int rflags, int32_t* ids, float* w, const PermOut& perm) {
  const dim3 g(grid), b(kRouteThreads);
  if (E <= 128)
    return launch_pdl(topk_kernel<4>, g, b, 0, s, logits, bias, e2s, affinity, part, nb, off, T, E, k, tpc, rflags,
                      ids, w, perm);
  if (E <= 256)
    return launch_pdl(topk_kernel<8>, g, b, 0, s, logits, bias, e2s, affinity, part, nb, off, T, E, k, tpc, rflags,
                      ids, w, perm);
  return launch_pdl(topk_kernel<kMaxE / 32>, g, b, 0, s, logits, bias, e2s, affinity, part, nb, off, T, E, k, tpc,
                    rflags, ids, w, perm);
}

}  // namespace moe

using namespace moe;

extern "C" int moe_bias_table_mode(const float* b, int E, int n_hot, int mode, float value, float* bias,
                                   moe_stream_t stream) {
  if (!b || !bias || E < 1 || E > kMaxE || n_hot < 1 || n_hot > E) return MOE_ERR_ARG;
  if (mode != MOE_BIAS_GRADED && mode != MOE_BIAS_FLAT && mode != MOE_BIAS_HARD) return MOE_ERR_ARG;
  const int threads = ((E + 31) / 32) * 32;
  bias_table_kernel<<<1, threads, 0, (cudaStream_t)stream>>>(b, E, n_hot, mode, value, bias);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

extern "C" int moe_bias_table(const float* b, int E, int n_hot, float cap, float* bias, moe_stream_t stream) {
  return moe_bias_table_mode(b, E, n_hot, MOE_BIAS_GRADED, cap, bias, stream);
}

extern "C" size_t moe_route_scratch_bytes(int T, int H, int E) {
  if (T < 1 || H < 1 || E < 1) return 0;
  return (size_t)((H + kHC - 1) / kHC) * T * E * sizeof(float);
}

namespace moe {

// The route entry's work; when `perm` is given and the top-k runs as one CTA over at most kSmallN
// routing slots, that CTA also groups the batch by expert into *perm and *fused is set.
int route_impl(const void* x, const void* w_router, const float* logit_offset, const float* sel_bias,
               const int32_t* e2s, float affinity, int rflags, int T, int H, int E, int k, float* logits,
               float* scratch, int32_t* ids, float* w, cudaStream_t stream, const PermOut* perm, bool* fused) {
  if (fused) *fused = false;
  const PermOut none{};
  auto pk = [&](int grid) -> PermOut {
    if (perm && fused && grid == 1 && T * k <= kSmallN) {
      *fused = true;
      return *perm;
    }
    return none;
  };
  if (!x || !w_router || !ids || !w || !logits) return MOE_ERR_ARG;
  if (rflags & ~(MOE_ROUTE_SIGMOID | MOE_ROUTE_DAMPED)) return MOE_ERR_ARG;
  if ((rflags & MOE_ROUTE_SIGMOID) && (rflags & MOE_ROUTE_DAMPED)) return MOE_ERR_ARG;
  if (T < 1 || H < 8 || H % 8 || E < 1 || E > kMaxE || E % 8 || k < 1 || k > kMaxK || k > E) return MOE_ERR_ARG;
  if ((uintptr_t)x % 16 || (uintptr_t)w_router % 16) return MOE_ERR_ALIGN;
  int sms = 0, dev = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  cudaStream_t s = (cudaStream_t)stream;
  const int eb = (E + kEB - 1) / kEB;
  const int nblk = (H + kHC - 1) / kHC;
  const uint16_t* xb = (const uint16_t*)x;
  const uint16_t* wb = (const uint16_t*)w_router;
  if (scratch && moe_route_scratch_bytes(T, H, E) > 0 && ((T + 7) / 8) * eb < sms) {
    // few tokens: every (128-row block, 32 experts, 8 tokens) is its own CTA
    const dim3 grid(nblk, eb, (T + 7) / 8);
    logits_block_kernel<1><<<grid, kRouteThreads, 0, s>>>(xb, wb, T, H, E, scratch);
    MOE_LAUNCH_CHECK();
    // tokens per CTA: 8 while that fills the SMs, else 2 (each thread then finishes about one logit)
    const int tpc = (T + 7) / 8 >= sms ? 8 : 2;
    MOE_CUDA_TRY(launch_topk((T + tpc - 1) / tpc, s, logits, sel_bias, e2s, affinity, scratch, nblk, logit_offset, T,
                             E, k, tpc, rflags, ids, w, pk((T + tpc - 1) / tpc)));
    MOE_LAUNCH_CHECK();
    return MOE_OK;
  }
  if (E % 8 == 0 && ((T + kTT - 1) / kTT) * ((E + kTE - 1) / kTE) * 2 >= sms) {
    // many tokens: (64 tokens, 64 experts) tiles over all of H, at least half as many CTAs as SMs
    const int smem = (int)logits_full_smem_bytes();
    static bool df[64] = {};
    MOE_CUDA_TRY(ensure_smem(logits_full_kernel, smem, df));
    const dim3 grid((T + kTT - 1) / kTT, (E + kTE - 1) / kTE);
    logits_full_kernel<<<grid, kFullThreads, smem, s>>>(xb, wb, logit_offset, T, H, E, logits);
    MOE_LAUNCH_CHECK();
    MOE_CUDA_TRY(launch_topk((T + 7) / 8, s, logits, sel_bias, e2s, affinity, nullptr, 0, nullptr, T, E, k, 8, rflags,
                             ids, w, pk((T + 7) / 8)));
    MOE_LAUNCH_CHECK();
    return MOE_OK;
  }
  if (scratch && moe_route_scratch_bytes(T, H, E) > 0 && E % 4 == 0) {
    // many tokens: (64 tokens, 64 experts, 128-row block) tiles, parts added in block order by the top-k
    constexpr int smem = (kHC * kTT + kHC * kTE) * (int)sizeof(float);
    static bool dt[64] = {};
    MOE_CUDA_TRY(ensure_smem(logits_tile_kernel, smem, dt));
    const dim3 grid((T + kTT - 1) / kTT, (E + kTE - 1) / kTE, nblk);
    logits_tile_kernel<<<grid, kTileThreads, smem, s>>>(xb, wb, T, H, E, scratch);
    MOE_LAUNCH_CHECK();
    // tokens per CTA: 8 while that fills the SMs, else 2 (each thread then finishes about one logit)
    const int tpc = (T + 7) / 8 >= sms ? 8 : 2;
    MOE_CUDA_TRY(launch_topk((T + tpc - 1) / tpc, s, logits, sel_bias, e2s, affinity, scratch, nblk, logit_offset, T,
                             E, k, tpc, rflags, ids, w, pk((T + tpc - 1) / tpc)));
    MOE_LAUNCH_CHECK();
    return MOE_OK;
  }
  // tokens per CTA: fewest that still give every SM a CTA, at most 64
  int ch = 8;
  while (ch > 1 && ((T + 8 * ch - 1) / (8 * ch)) * eb < sms) ch /= 2;
  const dim3 grid((T + 8 * ch - 1) / (8 * ch), eb);
  const size_t smem = (size_t)kRStages * (kHC * kEB * 2 + 8 * ch * (kHC + 8) * 2) + (size_t)kHC * 8 * ch * 4;
  static bool d1[64] = {}, d2[64] = {}, d4[64] = {}, d8[64] = {};
  switch (ch) {
    case 1:
      MOE_CUDA_TRY(ensure_smem(logits_kernel<1>, (int)smem, d1));
      logits_kernel<1><<<grid, kRouteThreads, smem, s>>>(xb, wb, logit_offset, T, H, E, logits);
      break;
    case 2:
      MOE_CUDA_TRY(ensure_smem(logits_kernel<2>, (int)smem, d2));
      logits_kernel<2><<<grid, kRouteThreads, smem, s>>>(xb, wb, logit_offset, T, H, E, logits);
      break;
    case 4:
      MOE_CUDA_TRY(ensure_smem(logits_kernel<4>, (int)smem, d4));
      logits_kernel<4><<<grid, kRouteThreads, smem, s>>>(xb, wb, logit_offset, T, H, E, logits);
      break;
    default:
      MOE_CUDA_TRY(ensure_smem(logits_kernel<8>, (int)smem, d8));
      logits_kernel<8><<<grid, kRouteThreads, smem, s>>>(xb, wb, logit_offset, T, H, E, logits);
      break;
  }
  MOE_LAUNCH_CHECK();
  MOE_CUDA_TRY(launch_topk((T + 7) / 8, s, logits, sel_bias, e2s, affinity, nullptr, 0, nullptr, T, E, k, 8, rflags,
                           ids, w, pk((T + 7) / 8)));
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe

extern "C" int moe_route_ex(const void* x, const void* w_router, const float* logit_offset, const float* sel_bias,
                            const int32_t* e2s, float affinity, int rflags, int T, int H, int E, int k,
                            float* logits, float* scratch, int32_t* ids, float* w, moe_stream_t stream) {
  return route_impl(x, w_router, logit_offset, sel_bias, e2s, affinity, rflags, T, H, E, k, logits, scratch, ids, w,
                    (cudaStream_t)stream, nullptr, nullptr);
}

extern "C" int moe_route(const void* x, const void* w_router, const float* logit_offset, const float* sel_bias,
                         const int32_t* e2s, float affinity, int T, int H, int E, int k, float* logits,
                         float* scratch, int32_t* ids, float* w, moe_stream_t stream) {
  return moe_route_ex(x, w_router, logit_offset, sel_bias, e2s, affinity, 0, T, H, E, k, logits, scratch, ids, w,
                      stream);
}
