// W8A8 experts: 8-bit weights with per-output-channel scales, 8-bit
// activations with per-row scales, exact int32 dot products.
//
// "Porting vllm-expert-cache to NVIDIA GPUs": the measured model is
// Qwen3-30B-A3B W8A8, and "weights and their scales are indexed by the same
// id, so both must be slot-indexed".  Here the scales travel inside the
// quantised slab, so manage and gather move them with the weights.
//
// Quantised slab (q8_slab_bytes = 3HI + 4(2I + H)):
//   Wg, Wu [H][I], Wd [I][H] as int8, every 4 consecutive input rows of a
//   column packed into one int32 (byte (k, n) at ((k/4)*N + n)*4 + k%4), then
//   fp32 scales sg[I], su[I], sd[H].
// Codes: symmetric, scale = amax / 127, code = rint(v / scale) clamped to
// +-127 (scale 0 gives code 0), all fp32 one operation at a time
// (fp32def.cuh), so they are reproducible bit for bit.
//
// Decode FFN: the same balanced stream as the bf16 path (sched.cuh), on CUDA
// cores: a stage is 16 input rows x all output columns (one 1-D bulk copy per
// matrix), a thread owns 4 output columns and folds 4 input rows per dp4a; a
// range's int32 sums go to parts[j][p][N]; the reduces add the parts (integer,
// exact), dequantise, form h = silu(g)*u, quantise h per row (gate/up) or write
// y (down).  The int8 tensor-core path is not used: decode is a weight stream
// and the CUDA cores keep up with it.
#include <algorithm>

#include "fp32def.cuh"
#include "internal.cuh"
#include "sched.cuh"
#include "tc05.cuh"

namespace moe {

constexpr int kQK = 16;                 // input rows per stage (4 quads)
constexpr int kQRB = 8;                 // tokens per pass over the weights
constexpr int kQActBytes = kQRB * 16;   // a batch's codes for one stage: 8 tokens x 16 rows
constexpr int kQRing = 200 * 1024;
constexpr int kQMaxStages = 8;
constexpr int kQMaxConsumers = 512;
constexpr int kQJcapMax = 160;
// Bytes of int32 parts per pass (soft cap).  Unlike the bf16 stream's, raising it to 64 MB made the W8A8
// expert-wave step slower (1.60 -> 1.76 ms at 64 tokens): short lists then fold few stages per CTA.
constexpr size_t kQPartBudget = size_t(16) << 20;
constexpr int kQMaxRows = 4096;

static size_t qal256(size_t v) { return (v + 255) & ~size_t(255); }

__host__ __device__ __forceinline__ size_t q8_slab_bytes_hd(int H, int I) {
  return (size_t)3 * H * I + (size_t)4 * (2 * I + H);
}
size_t q8_slab_bytes_h(int H, int I) { return q8_slab_bytes_hd(H, I); }

// ---------------------------------------------------------------------------
// Weight quantisation (offline, once per expert)
// ---------------------------------------------------------------------------
// grid (ceil(N/128), 3 matrices, experts); thread = one output column.
__global__ void __launch_bounds__(128) quantize_slabs_kernel(const uint16_t* __restrict__ src, int H, int I,
                                                             uint8_t* __restrict__ dst) {
  const int m = blockIdx.y;
  const int K = m < 2 ? H : I, N = m < 2 ? I : H;
  const int n = blockIdx.x * 128 + threadIdx.x;
  if (n >= N) return;
  const size_t mat = (size_t)H * I;
  const uint16_t* w = src + (size_t)blockIdx.z * 3 * mat + (size_t)m * mat;
  uint8_t* q = dst + (size_t)blockIdx.z * q8_slab_bytes_hd(H, I) + (size_t)m * mat;
  float amax = 0.f;
  for (int k = 0; k < K; ++k) amax = fmaxf(amax, fabsf(bf16_to_f32(w[(size_t)k * N + n])));
  const float s = __fdiv_rn(amax, 127.f);
  uint32_t* q4 = reinterpret_cast<uint32_t*>(q);
  for (int k = 0; k < K; k += 4) {
    uint32_t pk = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) pk |= (uint32_t)(q8_code(bf16_to_f32(w[(size_t)(k + b) * N + n]), s) & 0xff) << (8 * b);
    q4[(size_t)(k >> 2) * N + n] = pk;
  }
  float* sc = reinterpret_cast<float*>(dst + (size_t)blockIdx.z * q8_slab_bytes_hd(H, I) + 3 * mat);
  sc[(m == 0 ? 0 : m == 1 ? I : 2 * I) + n] = s;
}

// ---------------------------------------------------------------------------
// Activation codes are stored stage-major: the 16 codes of position p for
// input rows 16s .. 16s+15 are the 16 bytes at ((s * npad) + p) * 16, so one
// copy of 8 x 16 bytes brings a stage's codes for a whole token batch.
__device__ __forceinline__ size_t q8_act_word(int q, int p, int npad) {  // int32 index of quad q of position p
  return ((size_t)(q >> 2) * npad + p) * 4 + (q & 3);
}

// Activation quantisation: x rows of the grouped positions -> codes (stage-major),
// scale sx[p].  One CTA per position.
// ---------------------------------------------------------------------------
constexpr int kQRowThreads = 256;

__device__ __forceinline__ float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float r = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r = fmaxf(r, red[i]);
  return r;
}

__global__ void __launch_bounds__(kQRowThreads) q8_rows_kernel(const uint16_t* __restrict__ x,
                                                               const int32_t* __restrict__ rows, int n, int H, int k,
                                                               int npad, uint32_t* __restrict__ xq,
                                                               float* __restrict__ sx) {
  __shared__ float red[32];
  // Launched as a dependent of the permute.  Wait first, then let the stream kernel launch: it reads
  // the permute's expert list and offsets before its own wait.
  pdl_wait();
  pdl_trigger();
  const int p = blockIdx.x;
  const uint16_t* xr = x + (size_t)(rows[p] / k) * H;
  float amax = 0.f;
  for (int h = threadIdx.x; h < H; h += blockDim.x) amax = fmaxf(amax, fabsf(bf16_to_f32(xr[h])));
  amax = block_max(amax, red);
  const float s = __fdiv_rn(amax, 127.f);
  for (int q = threadIdx.x; q < H / 4; q += blockDim.x) {
    uint32_t pk = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) pk |= (uint32_t)(q8_code(bf16_to_f32(xr[4 * q + b]), s) & 0xff) << (8 * b);
    xq[q8_act_word(q, p, npad)] = pk;
  }
  if (threadIdx.x == 0) sx[p] = s;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------------------
// The stream (one pass: gate/up or down)
// ---------------------------------------------------------------------------
struct QPass {
  int32_t* part;     // [jcap][n][N]
  int32_t* vpre;     // batches before each list index (written by the pass's CTA 0 for its reduce)
  const uint32_t* act;  // stage-major codes of the pass's input rows (q8_act_word)
  int npad;
  int N, K, NSR, nst, wbytes, stride, G, jcap;
  size_t qslab;      // bytes of one quantised slab
};

__device__ __forceinline__ void q8_bulk(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  bulk_load(dst, src, bytes, bar);
}

template <bool DOWN, int RB>
__device__ __forceinline__ void q8_consume(const QPass& qp, int n, const StreamSeg& g, const unsigned char* ring,
                                           uint64_t* full, uint64_t* empty, uint32_t& it,
                                           volatile int* abort_flag, int32_t* status, int I) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int c = tid;  // output columns 4c .. 4c+3
  int acc[RB][4];
#pragma unroll
  for (int r = 0; r < RB; ++r)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[r][q] = 0;
  // byte offset of this thread's 16 bytes in quad-row 0 of a stage, and the quad-row stride
  int off, qstride;
  if (DOWN) {
    off = 16 * c;
    qstride = 4 * qp.N;
  } else {
    off = 4 * c < I ? 16 * c : kQK * I + 16 * c - 4 * I;  // Wu rows follow the stage's Wg rows
    qstride = 4 * I;
  }
  for (int s = g.s_lo; s < g.s_hi; ++s, ++it) {
    const int sl = it % qp.nst;
    if (!*abort_flag && !mbar_wait(&full[sl], (it / qp.nst) & 1u)) {
      *abort_flag = 1;
      set_status(status, MOE_DEV_TIMEOUT);
    }
    const unsigned char* st = ring + sl * qp.stride;
    const int32_t* act = reinterpret_cast<const int32_t*>(st + qp.wbytes);
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      const int4 w = *reinterpret_cast<const int4*>(st + off + qq * qstride);
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        const int xa = act[r * 4 + qq];
        acc[r][0] = __dp4a(w.x, xa, acc[r][0]);
        acc[r][1] = __dp4a(w.y, xa, acc[r][1]);
        acc[r][2] = __dp4a(w.z, xa, acc[r][2]);
        acc[r][3] = __dp4a(w.w, xa, acc[r][3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[sl]);
  }
#pragma unroll
  for (int r = 0; r < RB; ++r)
    if (r < g.nb)
      *reinterpret_cast<int4*>(qp.part + ((size_t)g.j * n + g.p0 + r) * qp.N + 4 * c) =
          make_int4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
}

template <bool DOWN>
__global__ void __launch_bounds__(kQMaxConsumers + 32, 1) ffn_q8_kernel(const FfnArgs a, const QPass qp) {
  extern __shared__ __align__(16) unsigned char q8_raw[];
  unsigned char* ring =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(q8_raw) + 127) & ~uintptr_t(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + qp.nst * qp.stride);
  uint64_t* empty = full + kQMaxStages;
  __shared__ int s_abort;
  __shared__ int s_vpre[kMaxE + 1];
  __shared__ int s_tmp[33];
  const int nc = qp.N / 4;
  const int tid = threadIdx.x;
  pdl_trigger();
  const int n_list = min(*a.n_list, kMaxE);
  const int n = a.T * a.k;
  stream_batch_prefix<kQRB>(a, n_list, s_vpre, s_tmp);
  const int nbat = s_vpre[n_list];
  if (blockIdx.x == 0)
    for (int i = tid; i <= n_list; i += blockDim.x) qp.vpre[i] = s_vpre[i];
  const int L = nbat > 0 ? stream_len(nbat, qp.NSR, qp.G, qp.jcap) : 1;
  const int total = nbat * qp.NSR;
  const int beg = blockIdx.x * L, end = min(beg + L, total);
  if (beg >= end) {
    pdl_wait();
    return;
  }
  if (tid == 0) {
    for (int s = 0; s < qp.nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nc / 32);
    }
    s_abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  volatile int* abort_flag = &s_abort;

  if (tid == nc) {
    // producer: weights stream at once; the activations (written by the kernel
    // before) only after griddepcontrol.wait
    uint32_t it = 0;
    bool waited = false;
    int ndef = 0, d_q0[kQMaxStages], d_p0[kQMaxStages], last_use[kQMaxStages];
    for (int s = 0; s < kQMaxStages; ++s) last_use[s] = -1;
    auto issue_act = [&](int sl, int q0, int p0) {
      q8_bulk(ring + sl * qp.stride + qp.wbytes, qp.act + q8_act_word(q0, p0, qp.npad), kQActBytes, &full[sl]);
    };
    auto flush = [&]() {
      pdl_wait();
      asm volatile("fence.proxy.async.global;" ::: "memory");
      for (int d = 0; d < ndef; ++d) issue_act(d, d_q0[d], d_p0[d]);
      ndef = 0;
      waited = true;
    };
    stream_segments_batched<kQRB>(a, s_vpre, n_list, qp.NSR, L, beg, end, [&](const StreamSeg& g) {
      const unsigned char* w = reinterpret_cast<const unsigned char*>(a.pool) + (size_t)g.slot * qp.qslab;
      for (int s = g.s_lo; s < g.s_hi; ++s, ++it) {
        const int sl = it % qp.nst;
        const uint32_t use = it / qp.nst;
        if (use > 0) {
          if (!waited) flush();
          if (!*abort_flag && !mbar_wait(&empty[sl], (use - 1) & 1u)) {
            *abort_flag = 1;
            set_status(a.status, MOE_DEV_TIMEOUT);
          }
        }
        if (*abort_flag) return false;
        unsigned char* dst = ring + sl * qp.stride;
        const int q0 = s * (kQK / 4);  // first quad of the stage
        mbar_expect_tx(&full[sl], qp.wbytes + kQActBytes);
        const size_t mat = (size_t)a.H * a.I;
        if (DOWN) {
          q8_bulk(dst, w + 2 * mat + (size_t)q0 * a.H * 4, qp.wbytes, &full[sl]);
        } else {
          const uint32_t mb = qp.wbytes / 2;
          q8_bulk(dst, w + (size_t)q0 * a.I * 4, mb, &full[sl]);
          q8_bulk(dst + mb, w + mat + (size_t)q0 * a.I * 4, mb, &full[sl]);
        }
        if (waited) {
          issue_act(sl, q0, g.p0);
        } else {
          d_q0[ndef] = q0;
          d_p0[ndef] = g.p0;
          ++ndef;
        }
        last_use[sl] = (int)use;
      }
      return true;
    });
    if (!waited) flush();
    if (*abort_flag)
      for (int s = 0; s < qp.nst; ++s)
        if (last_use[s] >= 0) mbar_wait(&full[s], (uint32_t)last_use[s] & 1u);
  } else if (tid < nc) {
    uint32_t it = 0;
    stream_segments_batched<kQRB>(a, s_vpre, n_list, qp.NSR, L, beg, end, [&](const StreamSeg& g) {
      if (g.nb <= 1)
        q8_consume<DOWN, 1>(qp, n, g, ring, full, empty, it, abort_flag, a.status, a.I);
      else if (g.nb <= 2)
        q8_consume<DOWN, 2>(qp, n, g, ring, full, empty, it, abort_flag, a.status, a.I);
      else if (g.nb <= 4)
        q8_consume<DOWN, 4>(qp, n, g, ring, full, empty, it, abort_flag, a.status, a.I);
      else
        q8_consume<DOWN, 8>(qp, n, g, ring, full, empty, it, abort_flag, a.status, a.I);
      return true;
    });
  }
  if (blockIdx.x == 0 && tid < n_list) {
    int e, slot;
    if (!stream_slot(a, tid, e, slot)) set_status(a.status, e < 0 || e >= a.E ? MOE_DEV_BAD_EXPERT : MOE_DEV_BAD_SLOT);
  }
  __syncwarp();
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Reduces.  Integer parts are added exactly (any order gives the same sum).
// ---------------------------------------------------------------------------
// gate/up: one CTA per listed expert; per row p: g, u (dequantised), h =
// silu(g)*u, amax over the row, codes of h into hq (quad-major), sh[p].
__global__ void __launch_bounds__(kQRowThreads) q8_reduce_gu_kernel(const FfnArgs a, const int32_t* __restrict__ part,
                                                                    const int32_t* __restrict__ vpre,
                                                                    int NSR, int G, int jcap, size_t qslab,
                                                                    const float* __restrict__ sx, int npad,
                                                                    uint32_t* __restrict__ hq,
                                                                    float* __restrict__ sh) {
  __shared__ float red[32];
  pdl_trigger();
  const int li = blockIdx.x;
  const int n_list = *a.n_list;
  int e = -1, slot = -1;
  const bool ok = li < n_list && stream_slot(a, li, e, slot);
  pdl_wait();
  if (!ok) return;
  const int nl = min(n_list, kMaxE);
  const int L = stream_len(vpre[nl], NSR, G, jcap);  // vpre: written by the pass before (completed)
  const int v0 = vpre[li];
  const int n = a.T * a.k, I = a.I, N = 2 * I;
  const size_t mat = (size_t)a.H * I;
  const float* sc = reinterpret_cast<const float*>(reinterpret_cast<const unsigned char*>(a.pool) +
                                                   (size_t)slot * qslab + 3 * mat);
  const float* sg = sc;
  const float* su = sc + I;
  const size_t pstride = (size_t)n * N;
  const int pb = a.offset[e], pe = a.offset[e + 1];
  for (int p = pb; p < pe; ++p) {
    const int J = stream_parts(v0 + (p - pb) / kQRB, NSR, L);
    const float s_x = sx[p];
    float hv[4][4];  // up to 4 quads per thread (I <= 16 * blockDim)
    float amax = 0.f;
#pragma unroll
    for (int nq = 0; nq < 4; ++nq) {
      const int q = threadIdx.x + nq * blockDim.x;
      if (q >= I / 4) break;
      // exact int32 sums, so the parts may be added in any order: eight parts' loads are issued
      // before their adds, instead of one L2 round trip per part
      int4 ag = make_int4(0, 0, 0, 0), au = ag;
      const int32_t* pp = part + (size_t)p * N + 4 * q;
      for (int j0 = 0; j0 < J; j0 += 8) {
        int4 tg[8], tu[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          tg[u] = make_int4(0, 0, 0, 0);
          tu[u] = tg[u];
          if (j0 + u < J) {
            tg[u] = *reinterpret_cast<const int4*>(pp + (size_t)(j0 + u) * pstride);
            tu[u] = *reinterpret_cast<const int4*>(pp + (size_t)(j0 + u) * pstride + I);
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          ag.x += tg[u].x; ag.y += tg[u].y; ag.z += tg[u].z; ag.w += tg[u].w;
          au.x += tu[u].x; au.y += tu[u].y; au.z += tu[u].z; au.w += tu[u].w;
        }
      }
      const int gi[4] = {ag.x, ag.y, ag.z, ag.w}, ui[4] = {au.x, au.y, au.z, au.w};
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int i = 4 * q + b;
        const float g = __fmul_rn(__fmul_rn(__int2float_rn(gi[b]), sg[i]), s_x);
        const float u = __fmul_rn(__fmul_rn(__int2float_rn(ui[b]), su[i]), s_x);
        const float h = __fmul_rn(silu32_def(g), u);
        hv[nq][b] = h;
        amax = fmaxf(amax, fabsf(h));
      }
    }
    amax = block_max(amax, red);
    const float s = __fdiv_rn(amax, 127.f);
#pragma unroll
    for (int nq = 0; nq < 4; ++nq) {
      const int q = threadIdx.x + nq * blockDim.x;
      if (q >= I / 4) break;
      uint32_t pk = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) pk |= (uint32_t)(q8_code(hv[nq][b], s) & 0xff) << (8 * b);
      hq[q8_act_word(q, p, npad)] = pk;
    }
    if (threadIdx.x == 0) sh[p] = s;
  }
}

// The same reduction with an expert's rows four at a time: 64 threads per row, each owning up to
// four quads of it (I <= 1024), with every part's loads for those quads issued before their adds
// (four parts a batch), and the row amax from the row's two warps.  An expert with a single row and
// more than four parts has that row's parts split over the four groups instead.  The path and the number of steps
// depend only on the expert's rows, so every block barrier is uniform.
constexpr int kQRowQuads = 4;   // quads per thread and row
constexpr int kQPartBatch = 4;  // parts whose loads are in flight together
__global__ void __launch_bounds__(kQRowThreads, 1) q8_reduce_gu_rows_kernel(
    const FfnArgs a, const int32_t* __restrict__ part, const int32_t* __restrict__ vpre, int NSR, int G, int jcap,
    size_t qslab, const float* __restrict__ sx, int npad, uint32_t* __restrict__ hq, float* __restrict__ sh) {
  __shared__ float red[kQRowThreads / 32];
  pdl_trigger();
  const int li = blockIdx.x;
  const int n_list = *a.n_list;
  int e = -1, slot = -1;
  const bool ok = li < n_list && stream_slot(a, li, e, slot);
  pdl_wait();
  if (!ok) return;
  const int nl = min(n_list, kMaxE);
  const int L = stream_len(vpre[nl], NSR, G, jcap);  // vpre: written by the pass before (completed)
  const int v0 = vpre[li];
  const int n = a.T * a.k, I = a.I, N = 2 * I, nq4 = I / 4;
  const size_t mat = (size_t)a.H * I;
  const float* sc = reinterpret_cast<const float*>(reinterpret_cast<const unsigned char*>(a.pool) +
                                                   (size_t)slot * qslab + 3 * mat);
  const float* sg = sc;
  const float* su = sc + I;
  const size_t pstride = (size_t)n * N;
  const int pb = a.offset[e], pe = a.offset[e + 1];
  const int grp = threadIdx.x >> 6, t64 = threadIdx.x & 63, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (pe - pb == 1 && stream_parts(v0, NSR, L) > kQPartBatch) {
    // a single row with more parts than one batch (small decode batches): all four groups work on it,
    // group g taking parts g, g+4, ...; the exact int32 sums meet in shared memory
    __shared__ int s_acc[2 * 4 * 64 * kQRowQuads];  // [g | u][column] for the row
    for (int p = pb; p < pe; ++p) {
      for (int i = threadIdx.x; i < 2 * I; i += kQRowThreads) s_acc[i] = 0;
      __syncthreads();
      const int J = stream_parts(v0 + (p - pb) / kQRB, NSR, L);
      int4 ag[kQRowQuads], au[kQRowQuads];
#pragma unroll
      for (int i = 0; i < kQRowQuads; ++i) ag[i] = au[i] = make_int4(0, 0, 0, 0);
      const int32_t* pp = part + (size_t)p * N + 4 * t64;
      for (int j0 = grp; j0 < J; j0 += 4 * kQPartBatch) {
        int4 tg[kQRowQuads][kQPartBatch], tu[kQRowQuads][kQPartBatch];
#pragma unroll
        for (int i = 0; i < kQRowQuads; ++i)
#pragma unroll
          for (int u = 0; u < kQPartBatch; ++u) {
            tg[i][u] = tu[i][u] = make_int4(0, 0, 0, 0);
            const int j = j0 + 4 * u;
            if (t64 + 64 * i < nq4 && j < J) {
              const int32_t* src = pp + (size_t)j * pstride + 256 * i;
              tg[i][u] = *reinterpret_cast<const int4*>(src);
              tu[i][u] = *reinterpret_cast<const int4*>(src + I);
            }
          }
#pragma unroll
        for (int i = 0; i < kQRowQuads; ++i)
#pragma unroll
          for (int u = 0; u < kQPartBatch; ++u) {
            ag[i].x += tg[i][u].x; ag[i].y += tg[i][u].y; ag[i].z += tg[i][u].z; ag[i].w += tg[i][u].w;
            au[i].x += tu[i][u].x; au[i].y += tu[i][u].y; au[i].z += tu[i][u].z; au[i].w += tu[i][u].w;
          }
      }
#pragma unroll
      for (int i = 0; i < kQRowQuads; ++i) {
        const int q = t64 + 64 * i;
        if (q < nq4) {
          int* dg = s_acc + 4 * q;
          int* du = s_acc + I + 4 * q;
          atomicAdd(dg, ag[i].x); atomicAdd(dg + 1, ag[i].y); atomicAdd(dg + 2, ag[i].z); atomicAdd(dg + 3, ag[i].w);
          atomicAdd(du, au[i].x); atomicAdd(du + 1, au[i].y); atomicAdd(du + 2, au[i].z); atomicAdd(du + 3, au[i].w);
        }
      }
      __syncthreads();
      // group 0 forms the row's h; its two warps give the amax
      const float s_x = sx[p];
      float hv[kQRowQuads][4];
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < kQRowQuads; ++i) {
        const int q = t64 + 64 * i;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          hv[i][b] = 0.f;
          if (grp == 0 && q < nq4) {
            const int c = 4 * q + b;
            const float g = __fmul_rn(__fmul_rn(__int2float_rn(s_acc[c]), sg[c]), s_x);
            const float u = __fmul_rn(__fmul_rn(__int2float_rn(s_acc[I + c]), su[c]), s_x);
            const float h = __fmul_rn(silu32_def(g), u);
            hv[i][b] = h;
            amax = fmaxf(amax, fabsf(h));
          }
        }
      }
      amax = warp_max(amax);
      if (lane == 0) red[w] = amax;
      __syncthreads();
      amax = fmaxf(red[0], red[1]);
      if (grp == 0) {
        const float s = __fdiv_rn(amax, 127.f);
#pragma unroll
        for (int i = 0; i < kQRowQuads; ++i) {
          const int q = t64 + 64 * i;
          if (q < nq4) {
            uint32_t pk = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) pk |= (uint32_t)(q8_code(hv[i][b], s) & 0xff) << (8 * b);
            hq[q8_act_word(q, p, npad)] = pk;
          }
        }
        if (t64 == 0) sh[p] = s;
      }
      __syncthreads();  // s_acc and red are reused by the next row
    }
    return;
  }
  for (int p0 = pb; p0 < pe; p0 += kQRowThreads / 64) {
    const int p = p0 + grp;
    const bool row = p < pe;
    float hv[kQRowQuads][4];
    float amax = 0.f;
    if (row) {
      const int J = stream_parts(v0 + (p - pb) / kQRB, NSR, L);
      const float s_x = sx[p];
      int4 ag[kQRowQuads], au[kQRowQuads];
#pragma unroll
      for (int i = 0; i < kQRowQuads; ++i) ag[i] = au[i] = make_int4(0, 0, 0, 0);
      const int32_t* pp = part + (size_t)p * N + 4 * t64;
      for (int j0 = 0; j0 < J; j0 += kQPartBatch) {
        int4 tg[kQRowQuads][kQPartBatch], tu[kQRowQuads][kQPartBatch];
#pragma unroll
        for (int i = 0; i < kQRowQuads; ++i)
#pragma unroll
          for (int u = 0; u < kQPartBatch; ++u) {
            tg[i][u] = tu[i][u] = make_int4(0, 0, 0, 0);
            if (t64 + 64 * i < nq4 && j0 + u < J) {
              const int32_t* src = pp + (size_t)(j0 + u) * pstride + 256 * i;
              tg[i][u] = *reinterpret_cast<const int4*>(src);
              tu[i][u] = *reinterpret_cast<const int4*>(src + I);
            }
          }
#pragma unroll
        for (int i = 0; i < kQRowQuads; ++i)
#pragma unroll
          for (int u = 0; u < kQPartBatch; ++u) {
            ag[i].x += tg[i][u].x; ag[i].y += tg[i][u].y; ag[i].z += tg[i][u].z; ag[i].w += tg[i][u].w;
            au[i].x += tu[i][u].x; au[i].y += tu[i][u].y; au[i].z += tu[i][u].z; au[i].w += tu[i][u].w;
          }
      }
#pragma unroll
      for (int i = 0; i < kQRowQuads; ++i) {
        const int q = t64 + 64 * i;
        const int gi[4] = {ag[i].x, ag[i].y, ag[i].z, ag[i].w}, ui[4] = {au[i].x, au[i].y, au[i].z, au[i].w};
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          hv[i][b] = 0.f;
          if (q < nq4) {
            const int c = 4 * q + b;
            const float g = __fmul_rn(__fmul_rn(__int2float_rn(gi[b]), sg[c]), s_x);
            const float u = __fmul_rn(__fmul_rn(__int2float_rn(ui[b]), su[c]), s_x);
            const float h = __fmul_rn(silu32_def(g), u);
            hv[i][b] = h;
            amax = fmaxf(amax, fabsf(h));
          }
        }
      }
    }
    // the row's amax: its two warps' maxima (every thread reaches both barriers)
    amax = warp_max(amax);
    if (lane == 0) red[w] = amax;
    __syncthreads();
    amax = fmaxf(red[2 * grp], red[2 * grp + 1]);
    __syncthreads();  // red is reused by the next rows
    if (row) {
      const float s = __fdiv_rn(amax, 127.f);
#pragma unroll
      for (int i = 0; i < kQRowQuads; ++i) {
        const int q = t64 + 64 * i;
        if (q < nq4) {
          uint32_t pk = 0;
#pragma unroll
          for (int b = 0; b < 4; ++b) pk |= (uint32_t)(q8_code(hv[i][b], s) & 0xff) << (8 * b);
          hq[q8_act_word(q, p, npad)] = pk;
        }
      }
      if (t64 == 0) sh[p] = s;
    }
  }
}

// down: y[p][n] = (float(sum of parts) * sd[n]) * sh[p]; block = 128 columns of one listed expert.  The
// block's branch (rows or parts over the warps) depends only on the expert's row count, so it is uniform.
__global__ void __launch_bounds__(256) q8_reduce_d_kernel(const FfnArgs a, const int32_t* __restrict__ part,
                                                          const int32_t* __restrict__ vpre, int NSR,
                                                          int G, int jcap, size_t qslab,
                                                          const float* __restrict__ sh, float* __restrict__ y) {
  __shared__ int4 sp[8][32];
  pdl_trigger();
  const int li = blockIdx.y;
  const int n_list = *a.n_list;
  int e = -1, slot = -1;
  const bool ok = li < n_list && stream_slot(a, li, e, slot);
  pdl_wait();
  if (!ok) return;
  const int nl = min(n_list, kMaxE);
  const int L = stream_len(vpre[nl], NSR, G, jcap);
  const int v0 = vpre[li];
  const int n = a.T * a.k, H = a.H;
  const float* sd = reinterpret_cast<const float*>(reinterpret_cast<const unsigned char*>(a.pool) +
                                                   (size_t)slot * qslab + (size_t)3 * H * a.I + (size_t)8 * a.I);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c4 = blockIdx.x * 32 + lane;
  const size_t pstride = (size_t)n * H;
  const int pb = a.offset[e], pe = a.offset[e + 1];
  if (pe - pb >= 4) {
    // enough rows to go around: warp w takes rows pb + w, pb + w + 8, ...; a lane adds every part of its
    // quad, eight parts' loads in flight before their adds (no barriers on this path)
    if (4 * c4 < H)
      for (int p = pb + w; p < pe; p += 8) {
        const int J = stream_parts(v0 + (p - pb) / kQRB, NSR, L);
        const int32_t* src = part + (size_t)p * H + 4 * c4;
        int4 acc = make_int4(0, 0, 0, 0);
        for (int j0 = 0; j0 < J; j0 += 8) {
          int4 t[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            t[u] = j0 + u < J ? *reinterpret_cast<const int4*>(src + (size_t)(j0 + u) * pstride) : make_int4(0, 0, 0, 0);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            acc.x += t[u].x; acc.y += t[u].y; acc.z += t[u].z; acc.w += t[u].w;
          }
        }
        const float s = sh[p];
        const int ai[4] = {acc.x, acc.y, acc.z, acc.w};
        float o[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) o[b] = __fmul_rn(__fmul_rn(__int2float_rn(ai[b]), sd[4 * c4 + b]), s);
        *reinterpret_cast<float4*>(y + (size_t)p * H + 4 * c4) = make_float4(o[0], o[1], o[2], o[3]);
      }
    return;
  }
  // few rows: the warps split each row's parts, then warp 0 adds the eight sums
  for (int p = pb; p < pe; ++p) {
    const int J = stream_parts(v0 + (p - pb) / kQRB, NSR, L);
    int4 acc = make_int4(0, 0, 0, 0);
    if (4 * c4 < H)
      for (int jj = w; jj < J; jj += 8) {
        const int4 t = *reinterpret_cast<const int4*>(part + jj * pstride + (size_t)p * H + 4 * c4);
        acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
      }
    sp[w][lane] = acc;
    __syncthreads();
    if (w == 0 && 4 * c4 < H) {
      for (int k2 = 1; k2 < 8; ++k2) {
        const int4 t = sp[k2][lane];
        acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
      }
      const float s = sh[p];
      const int ai[4] = {acc.x, acc.y, acc.z, acc.w};
      float o[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) o[b] = __fmul_rn(__fmul_rn(__int2float_rn(ai[b]), sd[4 * c4 + b]), s);
      *reinterpret_cast<float4*>(y + (size_t)p * H + 4 * c4) = make_float4(o[0], o[1], o[2], o[3]);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static int q_jcap(int n, int N) {
  const size_t per = (size_t)n * N * 4;
  const size_t j = per ? kQPartBudget / per : 0;
  return (int)std::max<size_t>(3, std::min<size_t>(j, kQJcapMax));
}

static int q_npad(int n) { return n + kQRB; }  // a batch copy may run RB positions past the last one

// Layout: [gate/up parts | down parts] (equal halves, int32), xq [H/4][npad],
// hq [I/4][npad] (int32 quads), sx [n], sh [n] (fp32).
size_t q8_ws_bytes(int n, int H, int I) {
  if (n < 1 || n > kQMaxRows) return 0;
  const size_t half = qal256(std::max((size_t)q_jcap(n, 2 * I) * n * 2 * I * 4, (size_t)q_jcap(n, H) * n * H * 4));
  const int np = q_npad(n);
  return 2 * half + qal256((size_t)H * np) + qal256((size_t)I * np) + 2 * qal256((size_t)4 * n) +
         2 * qal256((size_t)4 * (kMaxE + 1));
}

struct QCarve {
  int32_t *gpart, *ypart;
  uint32_t *xq, *hq;
  float *sx, *sh;
  int32_t *vpre_g, *vpre_d;
  int jg, jd, npad;
};

static bool q_carve(const FfnArgs& a, void* base, size_t bytes, QCarve* c) {
  const int n = a.T * a.k;
  const int np = q_npad(n);
  const size_t act = qal256((size_t)a.H * np) + qal256((size_t)a.I * np) + 2 * qal256((size_t)4 * n) +
                     2 * qal256((size_t)4 * (kMaxE + 1));
  if (!base || bytes < act + 512) return false;
  const size_t half = ((bytes - act) / 2) & ~size_t(255);
  char* b = reinterpret_cast<char*>(base);
  c->gpart = reinterpret_cast<int32_t*>(b);
  c->ypart = reinterpret_cast<int32_t*>(b + half);
  char* q = b + 2 * half;
  c->xq = reinterpret_cast<uint32_t*>(q);
  q += qal256((size_t)a.H * np);
  c->hq = reinterpret_cast<uint32_t*>(q);
  q += qal256((size_t)a.I * np);
  c->sx = reinterpret_cast<float*>(q);
  q += qal256((size_t)4 * n);
  c->sh = reinterpret_cast<float*>(q);
  q += qal256((size_t)4 * n);
  c->vpre_g = reinterpret_cast<int32_t*>(q);
  q += qal256((size_t)4 * (kMaxE + 1));
  c->vpre_d = reinterpret_cast<int32_t*>(q);
  c->npad = np;
  c->jg = (int)std::min<size_t>(q_jcap(n, 2 * a.I), half / ((size_t)n * 2 * a.I * 4));
  c->jd = (int)std::min<size_t>(q_jcap(n, a.H), half / ((size_t)n * a.H * 4));
  return c->jg >= 2 && c->jd >= 2;
}

static bool q_pass(bool down, const FfnArgs& a, int G, int32_t* part, int32_t* vpre, const uint32_t* act, int npad,
                   int jcap, QPass* out) {
  QPass qp{};
  qp.part = part;
  qp.vpre = vpre;
  qp.act = act;
  qp.npad = npad;
  qp.N = down ? a.H : 2 * a.I;
  qp.K = down ? a.I : a.H;
  if (qp.N % 128 || qp.K % kQK || qp.N / 4 > kQMaxConsumers) return false;
  qp.NSR = qp.K / kQK;
  qp.wbytes = kQK * qp.N;  // 16 rows x N int8
  qp.stride = qp.wbytes + 128;
  qp.nst = std::min(kQMaxStages, kQRing / qp.stride);
  if (qp.nst < 2) return false;
  qp.G = G;
  qp.jcap = jcap;
  qp.qslab = q8_slab_bytes_h(a.H, a.I);
  *out = qp;
  return jcap >= 2;
}

static size_t q_smem(const QPass& qp) { return 128 + (size_t)qp.nst * qp.stride + 2 * kQMaxStages * 8; }

template <typename K, typename... Args>
static cudaError_t q_launch(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, Args... args) {
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

int launch_ffn_q8(const FfnArgs& a, void* ws, size_t ws_bytes, int max_list, cudaStream_t stream, Prof* prof) {
  if (max_list <= 0) return MOE_OK;
  const int n = a.T * a.k;
  if (n > kQMaxRows || !a.pool_only || a.S <= 0 || a.H % 16 || a.I % 16 || a.I / 4 > 4 * kQRowThreads)
    return MOE_ERR_ARG;
  if ((uintptr_t)a.pool % 16 || (uintptr_t)a.y % 16 || (uintptr_t)ws % 256) return MOE_ERR_ALIGN;
  int dev = 0, sms = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  QCarve c;
  if (!q_carve(a, ws, ws_bytes, &c)) return MOE_ERR_ALIGN;
  QPass g, d;
  if (!q_pass(false, a, sms, c.gpart, c.vpre_g, c.xq, c.npad, c.jg, &g) ||
      !q_pass(true, a, sms, c.ypart, c.vpre_d, c.hq, c.npad, c.jd, &d))
    return MOE_ERR_ARG;
  static bool done_g[64] = {}, done_d[64] = {};
  constexpr int kSmemMax = 128 + kQRing + 2 * kQMaxStages * 8;
  MOE_CUDA_TRY(ensure_smem(ffn_q8_kernel<false>, kSmemMax, done_g));
  MOE_CUDA_TRY(ensure_smem(ffn_q8_kernel<true>, kSmemMax, done_d));
  if (prof) prof->begin(MOE_PROF_FFN_GATEUP, stream);
  MOE_CUDA_TRY(launch_pdl(q8_rows_kernel, dim3(n), dim3(kQRowThreads), 0, stream, a.x, a.rows, n, a.H, a.k, c.npad,
                          c.xq, c.sx));
  MOE_CUDA_TRY(q_launch(ffn_q8_kernel<false>, dim3(sms), dim3(g.N / 4 + 32), q_smem(g), stream, true, a, g));
  // an expert's rows four at a time when a row fits 64 threads x 4 quads (I <= 1024)
  const bool rows4 = a.I / 4 <= 64 * kQRowQuads;
  MOE_CUDA_TRY(q_launch(rows4 ? q8_reduce_gu_rows_kernel : q8_reduce_gu_kernel, dim3(max_list), dim3(kQRowThreads),
                        0, stream, true, a, (const int32_t*)c.gpart, (const int32_t*)c.vpre_g, g.NSR, g.G, g.jcap,
                        g.qslab, (const float*)c.sx, c.npad, c.hq, c.sh));
  if (prof) prof->end(stream);
  if (prof) prof->begin(MOE_PROF_FFN_DOWN, stream);
  MOE_CUDA_TRY(q_launch(ffn_q8_kernel<true>, dim3(sms), dim3(d.N / 4 + 32), q_smem(d), stream, true, a, d));
  MOE_CUDA_TRY(q_launch(q8_reduce_d_kernel, dim3((a.H / 4 + 31) / 32, max_list), dim3(256), 0, stream, true, a,
                        (const int32_t*)c.ypart, (const int32_t*)c.vpre_d, d.NSR, d.G, d.jcap, d.qslab,
                        (const float*)c.sh, a.y));
  if (prof) prof->end(stream);
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_q8_slab_bytes(int H, int I) {
  if (H < 1 || I < 1) return 0;
  return q8_slab_bytes_h(H, I);
}

extern "C" int moe_quantize_slabs(const void* src, int n_experts, int H, int I, void* dst, moe_stream_t stream) {
  if (!src || !dst || n_experts < 1 || H < 16 || I < 16 || H % 16 || I % 16) return MOE_ERR_ARG;
  if ((uintptr_t)src % 16 || (uintptr_t)dst % 16) return MOE_ERR_ALIGN;
  const int nmax = std::max(H, I);
  const dim3 grid((nmax + 127) / 128, 3, n_experts);
  quantize_slabs_kernel<<<grid, 128, 0, (cudaStream_t)stream>>>((const uint16_t*)src, H, I, (uint8_t*)dst);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

extern "C" size_t moe_ffn_q8_workspace_bytes(int T, int H, int k, int I) {
  if (T < 1 || H < 1 || k < 1 || I < 1) return 0;
  return q8_ws_bytes(T * k, H, I);
}

extern "C" int moe_expert_ffn_q8(const void* x, int T, int H, int I, int k, int E, const int32_t* offset,
                                 const int32_t* rows, const int32_t* list_e, const int32_t* n_list, int max_list,
                                 const void* pool_q, int S, const int32_t* e2s, float* y, void* workspace,
                                 size_t workspace_bytes, int32_t* dev_status, moe_stream_t stream) {
  if (!x || !offset || !rows || !list_e || !n_list || !pool_q || !y || !workspace) return MOE_ERR_ARG;
  if (T < 1 || k < 1 || E < k || H < 16 || I < 16 || max_list < 0 || S < 1 || (!e2s && S < E)) return MOE_ERR_ARG;
  FfnArgs a{(const uint16_t*)x, T, H, I, k, E, offset, rows, list_e, n_list, (const uint16_t*)pool_q, e2s,
            nullptr, 0, nullptr, y, dev_status, S, 1};
  return launch_ffn_q8(a, workspace, workspace_bytes, std::min(max_list, E), (cudaStream_t)stream, nullptr);
}
