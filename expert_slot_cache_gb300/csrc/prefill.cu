// Grouped SwiGLU expert FFN for prefill-sized groups on the tcgen05 tensor cores.
//
// "Porting vllm-expert-cache to NVIDIA GPUs", "What this package does": the
// expert GEMM runs on the grouped, slot-remapped ids.  When the groups are
// large (prefill), the two GEMMs are dense contractions and run here:
//   GEMM 1: [g | u] = Xp_e Wg_e | Xp_e Wu_e, epilogue h = silu(g) * u (bf16)
//   GEMM 2: y = h_e Wd_e (fp32)
// Xp is the routed rows of x in grouped order (copied once by
// gather_rows_kernel).  Tiles are M = 128 grouped rows x N = 256 columns:
// in GEMM 1 the 256 columns are 128 gate columns followed by the same 128 up
// columns, so one MMA per K step feeds both and the epilogue pairs them.
//
// One CTA per SM, persistent over the tiles of all experts (expert-major,
// then row tile, then column tile, so an expert's weights stay hot in L2):
//   warp 0: TMA producer (one thread), 4-stage ring of 48 KB stages
//   warp 1: TMEM allocation + MMA issue (one thread)
//   warps 2-5: epilogue, TMEM -> registers -> global
// Shared-memory operands use the 128-byte swizzle written by the tensor-map
// loads: activations K-major (rows of 64 bf16 = 128 B), weights MN-major
// (stored input-major: 64 output columns = 128 B per K row, 8 K rows per
// 1 KB swizzle atom, 64-column atoms 8 KB apart).  Accumulators are fp32 in
// TMEM, two 256-column buffers so the epilogue of one tile overlaps the MMAs
// of the next.
#include "internal.cuh"
#include "tc05.cuh"

namespace moe {

constexpr int kPM = 128;
constexpr int kPN = 256;
constexpr int kPK = 64;
constexpr int kPStages = 4;
constexpr int kPAbytes = kPM * kPK * 2;            // 16 KB
constexpr int kPBbytes = kPN * kPK * 2;            // 32 KB
constexpr int kPStageBytes = kPAbytes + kPBbytes;  // 48 KB
constexpr int kPThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr int kPrefillMinRows = 4096;
// per epilogue warp: a 32 x 33 fp32 transpose buffer (padded: conflict-free)
constexpr int kEpiBuf = 32 * 33;

// Instruction descriptor: D fp32, A and B bf16, A K-major, B MN-major, N = 256, M = 128.
constexpr uint32_t kIdesc = idesc_bf16(kPM, kPN, 0, 1);

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return smem_desc_l(saddr, lbo, sbo, kLayoutSw128);
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  umma_f16(d_tmem, adesc, bdesc, kIdesc, accumulate);
}

struct PrefillArgs {
  int H, I, E, n;
  const int32_t* offset;  // [E+1] grouped row offsets
  const int32_t* list_e;  // experts to process
  const int32_t* n_list;  // device count
  const int32_t* e2s;     // NULL = expert e in slot e
  int S;
  uint16_t* hb;  // bf16 [n][I]: GEMM 1 output
  float* y;      // fp32 [n][H]: GEMM 2 output (when yb == NULL)
  int32_t* status;
  uint16_t* yb;  // bf16 [n][H]: GEMM 2 output, or NULL
};

// Locate tile t: expert list index (by prefix search), row tile, column tile.
__device__ __forceinline__ void find_tile(const int* pre, int nl, int t, int nt, int& li, int& m, int& ct) {
  int lo = 0, hi = nl;  // pre[lo] <= t < pre[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= t) lo = mid;
    else hi = mid;
  }
  li = lo;
  const int local = t - pre[lo];
  m = local / nt;
  ct = local - m * nt;
}

template <int kMode>
__global__ void __launch_bounds__(kPThreads, 1) prefill_gemm_kernel(const PrefillArgs a,
                                                                    const __grid_constant__ CUtensorMap mapA,
                                                                    const __grid_constant__ CUtensorMap mapB) {
  extern __shared__ __align__(16) unsigned char psm_raw[];
  unsigned char* psm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(psm_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(psm + kPStages * kPStageBytes);
  uint64_t* empty = full + kPStages;
  uint64_t* tfull = empty + kPStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  float* epi = reinterpret_cast<float*>(full + 16);  // after the 16 barrier words: [4 warps][32][33]
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_pre[kMaxE + 1];
  __shared__ int s_total;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = kMode == 0 ? a.I / 128 : a.H / kPN;  // column tiles per row tile
  const int K = kMode == 0 ? a.H : a.I;
  const int nkb = K / kPK;
  const int nl = *a.n_list;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], 4);
    }
    mbar_init(done, 1);
    s_abort = 0;
    int acc = 0;
    for (int li = 0; li < nl; ++li) {
      s_pre[li] = acc;
      const int e = a.list_e[li];
      const int rows = (e >= 0 && e < a.E) ? a.offset[e + 1] - a.offset[e] : 0;
      acc += ((rows + kPM - 1) / kPM) * NT;
    }
    s_pre[nl] = acc;
    s_total = acc;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int total = s_total;
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      int last_use[kPStages];
      for (int s = 0; s < kPStages; ++s) last_use[s] = -1;
      for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
        int li, m, ct;
        find_tile(s_pre, nl, t, NT, li, m, ct);
        const int e = a.list_e[li];
        const int slot = a.e2s ? a.e2s[e] : e;
        const int row0 = a.offset[e] + m * kPM;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kPStages;
          const uint32_t use = it / kPStages;
          if (use > 0 && !*abort_flag && !mbar_wait(&empty[s], (use - 1) & 1u)) {
            *abort_flag = 1;
            set_status(a.status, MOE_DEV_TIMEOUT);
          }
          if (*abort_flag) break;
          unsigned char* st = psm + s * kPStageBytes;
          mbar_expect_tx(&full[s], kPStageBytes);
          tma_load_3d(st, &mapA, &full[s], kb * kPK, row0, 0);
          unsigned char* sb = st + kPAbytes;
          // weights: one 4-D box per matrix = 64 K-rows x all of the tile's 64-column swizzle atoms (8 KB apart)
          if (kMode == 0) {
            const int a0 = ct * 2;  // 128 gate columns, then the same 128 up columns
            tma_load_4d(sb, &mapB, &full[s], 0, kb * kPK, a0, 3 * slot);
            tma_load_4d(sb + 16384, &mapB, &full[s], 0, kb * kPK, a0, 3 * slot + 1);
          } else {
            tma_load_4d(sb, &mapB, &full[s], 0, kb * kPK, ct * (kPN / 64), 3 * slot + 2);
          }
          last_use[s] = (int)use;
        }
      }
      if (*abort_flag)
        for (int s = 0; s < kPStages; ++s)
          if (last_use[s] >= 0) mbar_wait(&full[s], (uint32_t)last_use[s] & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, tc = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
        const uint32_t acc = tc & 1u, ause = tc >> 1;
        if (ause > 0 && !*abort_flag && !mbar_wait(&tempty[acc], (ause - 1) & 1u)) {
          *abort_flag = 1;
          set_status(a.status, MOE_DEV_TIMEOUT);
        }
        tc_fence_after();
        const uint32_t d = tmem + acc * kPN;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kPStages;
          if (!*abort_flag && !mbar_wait(&full[s], (it / kPStages) & 1u)) {
            *abort_flag = 1;
            set_status(a.status, MOE_DEV_TIMEOUT);
          }
          tc_fence_after();
          if (!*abort_flag) {
            const uint32_t sa = smem_u32(psm + s * kPStageBytes);
            const uint64_t ad = smem_desc(sa, 16, 1024);
            const uint64_t bd = smem_desc(sa + kPAbytes, 8192, 1024);
#pragma unroll
            for (int kk = 0; kk < kPK / 16; ++kk)
              umma_bf16(d, ad + (uint64_t)((kk * 32) >> 4), bd + (uint64_t)((kk * 2048) >> 4), (kb | kk) != 0);
          }
          umma_commit(&empty[s]);
        }
        umma_commit(&tfull[acc]);
      }
      // all MMAs issued by this thread have finished once `done` completes
      umma_commit(done);
      mbar_wait(done, 0);
    }
  } else {
    // epilogue warps 2..5; TMEM lane quarter = warp % 4
    const int q = warp & 3;
    uint32_t tc = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
      int li, m, ct;
      find_tile(s_pre, nl, t, NT, li, m, ct);
      const int e = a.list_e[li];
      const int ne = a.offset[e + 1] - a.offset[e];
      const uint32_t acc = tc & 1u, ause = tc >> 1;
      if (!*abort_flag && !mbar_wait(&tfull[acc], ause & 1u)) {
        *abort_flag = 1;
        set_status(a.status, MOE_DEV_TIMEOUT);
      }
      tc_fence_after();
      // rows of this warp: m*128 + q*32 + r (r = 0..31); thread `lane` holds row q*32 + lane
      const int rbase = m * kPM + q * 32;
      const int nvalid = *abort_flag ? 0 : max(0, min(32, ne - rbase));
      const size_t p0 = (size_t)a.offset[e] + rbase;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + acc * kPN;
      float* buf = epi + (warp & 3) * kEpiBuf;
      if (kMode == 0) {
        const int n0 = ct * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float g[32], u[32];
          tmem_ld32(taddr + 32 * c, g);
          tmem_ld32(taddr + 128 + 32 * c, u);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) buf[lane * 33 + j] = g[j] / (1.f + expf(-g[j])) * u[j];
          __syncwarp();
          // two rows per instruction: lanes 0-15 row r, 16-31 row r+1, 2 columns each (64 B per row)
          const int half = lane >> 4, col = 2 * (lane & 15);
#pragma unroll 4
          for (int r = 0; r < 32; r += 2) {
            const int rr = r + half;
            if (rr < nvalid) {
              const uint32_t w = uint32_t(f32_to_bf16(buf[rr * 33 + col])) |
                                 (uint32_t(f32_to_bf16(buf[rr * 33 + col + 1])) << 16);
              *reinterpret_cast<uint32_t*>(a.hb + (p0 + rr) * a.I + n0 + 32 * c + col) = w;
            }
          }
          __syncwarp();
        }
      } else {
        const int o0 = ct * kPN;
#pragma unroll 1
        for (int c = 0; c < kPN / 32; ++c) {
          float v[32];
          tmem_ld32(taddr + 32 * c, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) buf[lane * 33 + j] = v[j];
          __syncwarp();
          if (a.yb) {
            // bf16: two rows per instruction, 2 columns per lane (64 B per row)
            const int half = lane >> 4, col = 2 * (lane & 15);
#pragma unroll 4
            for (int r = 0; r < 32; r += 2) {
              const int rr = r + half;
              if (rr < nvalid) {
                const uint32_t wv = uint32_t(f32_to_bf16(buf[rr * 33 + col])) |
                                    (uint32_t(f32_to_bf16(buf[rr * 33 + col + 1])) << 16);
                *reinterpret_cast<uint32_t*>(a.yb + (p0 + rr) * a.H + o0 + 32 * c + col) = wv;
              }
            }
          } else {
            // one row per instruction: 32 lanes x 4 B = 128 contiguous bytes
#pragma unroll 4
            for (int r = 0; r < 32; ++r)
              if (r < nvalid) a.y[(p0 + r) * a.H + o0 + 32 * c + lane] = buf[r * 33 + lane];
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }
  // warps 0 and 1 ran their loops on lane 0 alone: reconverge before the CTA barrier
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Xp[p] = x[rows[p] / k] for the n grouped rows (16-byte copies).
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ rows, int n, int H, int k,
                                                          uint16_t* __restrict__ xp) {
  pdl_trigger();
  const int H8 = H / 8;
  for (int p = blockIdx.x; p < n; p += gridDim.x) {
    const int t = rows[p] / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)p * H);
    for (int v = threadIdx.x; v < H8; v += blockDim.x) dst[v] = src[v];
  }
}

int launch_gather_rows(const uint16_t* x, const int32_t* rows, int n, int H, int k, uint16_t* xp, int sms,
                       cudaStream_t stream) {
  gather_rows_kernel<<<std::min(n, sms * 8), 256, 0, stream>>>(x, rows, n, H, k, xp);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

static size_t prefill_smem_bytes() {
  return 1024 + (size_t)kPStages * kPStageBytes + 16 * sizeof(uint64_t) + 4 * kEpiBuf * sizeof(float);
}

bool prefill_eligible(const FfnArgs& a, int n) {
  return a.pool_only && a.S > 0 && a.xp && a.hb && n >= kPrefillMinRows && a.H % kPN == 0 && a.I % 128 == 0 &&
         a.E <= kMaxE;
}

size_t prefill_extra_bytes(int n, int H, int I) {
  if (n < kPrefillMinRows) return 0;
  return (size_t)n * H * 2 + (size_t)n * I * 2 + 512;
}

int launch_prefill(const FfnArgs& a, int n, int max_list, cudaStream_t stream, Prof* prof) {
  static bool done0[64] = {}, done1[64] = {};
  MOE_CUDA_TRY(ensure_smem(prefill_gemm_kernel<0>, (int)prefill_smem_bytes(), done0));
  MOE_CUDA_TRY(ensure_smem(prefill_gemm_kernel<1>, (int)prefill_smem_bytes(), done1));
  int dev = 0, sms = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const size_t mat = (size_t)a.H * a.I;
  CUtensorMap mx, mh, mgu, md;
  {
    const uint64_t d[3] = {(uint64_t)a.H, (uint64_t)n, 1};
    const uint64_t s[2] = {(uint64_t)a.H * 2, (uint64_t)n * a.H * 2};
    const uint32_t b[3] = {kPK, kPM, 1};
    if (encode_tmap_3d_bf16(&mx, a.xp, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B) != MOE_OK) return MOE_ERR_CUDA;
  }
  {
    const uint64_t d[3] = {(uint64_t)a.I, (uint64_t)n, 1};
    const uint64_t s[2] = {(uint64_t)a.I * 2, (uint64_t)n * a.I * 2};
    const uint32_t b[3] = {kPK, kPM, 1};
    if (encode_tmap_3d_bf16(&mh, a.hb, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B) != MOE_OK) return MOE_ERR_CUDA;
  }
  // weight matrices viewed as [matrix][64-column atom][K row][64 columns]
  {
    const uint64_t d[4] = {64, (uint64_t)a.H, (uint64_t)a.I / 64, 3ull * a.S};
    const uint64_t s[3] = {(uint64_t)a.I * 2, 128, mat * 2};
    const uint32_t b[4] = {64, kPK, 2, 1};
    if (encode_tmap_bf16(&mgu, a.pool, 4, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B) != MOE_OK) return MOE_ERR_CUDA;
  }
  {
    const uint64_t d[4] = {64, (uint64_t)a.I, (uint64_t)a.H / 64, 3ull * a.S};
    const uint64_t s[3] = {(uint64_t)a.H * 2, 128, mat * 2};
    const uint32_t b[4] = {64, kPK, kPN / 64, 1};
    if (encode_tmap_bf16(&md, a.pool, 4, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B) != MOE_OK) return MOE_ERR_CUDA;
  }
  PrefillArgs p{a.H, a.I, a.E, n, a.offset, a.list_e, a.n_list, a.e2s, a.S, a.hb, a.y, a.status, a.yb};
  (void)max_list;
  if (prof) prof->begin(MOE_PROF_FFN_ROWS, stream);
  gather_rows_kernel<<<std::min(n, sms * 8), 256, 0, stream>>>(a.x, a.rows, n, a.H, a.k, a.xp);
  MOE_LAUNCH_CHECK();
  if (prof) prof->end(stream);
  if (prof) prof->begin(MOE_PROF_FFN_GATEUP, stream);
  prefill_gemm_kernel<0><<<sms, kPThreads, prefill_smem_bytes(), stream>>>(p, mx, mgu);
  MOE_LAUNCH_CHECK();
  if (prof) prof->end(stream);
  if (prof) prof->begin(MOE_PROF_FFN_DOWN, stream);
  prefill_gemm_kernel<1><<<sms, kPThreads, prefill_smem_bytes(), stream>>>(p, mh, md);
  MOE_LAUNCH_CHECK();
  if (prof) prof->end(stream);
  return MOE_OK;
}

}  // namespace moe
