// Grouped SwiGLU expert FFN for prefill-sized groups on the tcgen05 tensor cores.
//
// "Porting vllm-expert-cache to NVIDIA GPUs", "What this package does": the
// expert GEMM runs on the grouped, slot-remapped ids.  When the groups are
// large (prefill), the two GEMMs are dense contractions and run here:
//   GEMM 1: [g | u] = Xp_e Wg_e | Xp_e Wu_e, epilogue h = silu(g) * u (bf16)
//   GEMM 2: y = h_e Wd_e (bf16, or fp32)
// Xp is the routed rows of x in grouped order (copied once by
// gather_rows_kernel).
//
// The products are computed transposed, D^T = W^T X^T, by CTA pairs (a
// cluster of two on neighbouring SMs): the pair's MMA has M = 256 weight
// features (128 in each CTA's shared memory and TMEM) and N = up to 256 of
// one expert's grouped rows, rounded up to a multiple of 32, half of them in
// each CTA's shared memory.  Each CTA thus loads 64 KB of operands per 128-deep
// K step for a 128 x 256 x 128 share of the work, two thirds of what a lone
// CTA needs for the same tile.  Groups are ragged (a skewed router gives
// 0 .. thousands of rows per expert), and rows on the N side pad a group only
// to the next 32 rows instead of the next 128 or 256.  In GEMM 1 a CTA's 128
// features are 64 gate columns followed by the same 64 up columns, so one
// MMA per K step feeds both and the epilogue pairs them.
//
// Persistent clusters over the tiles of all experts (expert-major, then
// token tile, then feature tile, so a token tile stays hot in L2 while the
// clusters walk the expert's weights); per CTA:
//   warp 0: TMA producer (one thread), 3-stage ring of 64 KB stages; the
//           loads of both CTAs complete on rank 0's barrier
//   warp 1: TMEM allocation (both CTAs) + pair MMA issue (rank 0, one thread)
//   warps 2-5: epilogue, TMEM -> registers -> shared (transpose) -> global
// Shared-memory operands use the 128-byte swizzle written by the tensor-map
// loads: weights MN-major (stored input-major: 64 output columns = 128 B per
// K row, 8 K rows per 1 KB swizzle group, 64-column atoms 16 KB apart),
// grouped rows K-major (rows of 64 bf16 = 128 B, the two 64-deep K halves of
// a stage 16 KB apart).  One thread issues the MMAs, and a tcgen05.mma costs
// it tens of cycles to issue, so a stage is 128 deep: the barrier wait, fence
// and commit per stage are spread over eight MMAs.  Accumulators are fp32 in TMEM, two
// 256-column buffers so the epilogue of one tile overlaps the MMAs of the
// next.
#include "internal.cuh"
#include "tc05.cuh"

namespace moe {

constexpr int kPM = 128;     // weight features per CTA (the pair's MMA M is 256)
constexpr int kPT = 256;     // grouped rows per tile, at most (MMA N)
constexpr int kPTBox = 128;  // grouped rows per CTA and tile, at most (one tensor-map box)
constexpr int kPK = 128;    // K depth of a ring stage: eight 16-deep MMAs per barrier wait and commit
constexpr int kPStages = 3;
constexpr int kPAbytes = kPM * kPK * 2;            // 32 KB of weights: two 64-feature atoms, 16 KB apart
constexpr int kPBbytes = kPTBox * kPK * 2;         // 32 KB of rows: two 64-deep K halves, 16 KB apart
constexpr int kPStageBytes = kPAbytes + kPBbytes;  // 64 KB
constexpr int kPThreads = 192;
constexpr uint32_t kTmemCols = 2 * kPT;
constexpr int kPBarWords = 32;  // mbarriers: full / empty per stage, two accumulators, done
constexpr int kPrefillMinRows = 4096;
// per epilogue warp: a staging tile of 32 rows x 32 features (fp32 at most) and a 16 x 32 fp32
// gate/up exchange buffer
constexpr int kEpiStageBytes = 32 * 32 * 4;
constexpr int kEpiXFloats = 16 * 32;

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return smem_desc_l(saddr, lbo, sbo, kLayoutSw128);
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

// Locate tile t: expert list index (by prefix search), token tile, feature tile.
__device__ __forceinline__ void find_tile(const int* pre, int nl, int t, int nf, int& li, int& m, int& ft) {
  int lo = 0, hi = nl;  // pre[lo] <= t < pre[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= t) lo = mid;
    else hi = mid;
  }
  li = lo;
  const int local = t - pre[lo];
  m = local / nf;
  ft = local - m * nf;
}

template <int kMode>
__global__ void __launch_bounds__(kPThreads, 1) prefill_gemm_kernel(const PrefillArgs a,
                                                                    const __grid_constant__ CUtensorMap mapX,
                                                                    const __grid_constant__ CUtensorMap mapW) {
  extern __shared__ __align__(16) unsigned char psm_raw[];
  unsigned char* psm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(psm_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(psm + kPStages * kPStageBytes);
  uint64_t* empty = full + kPStages;
  uint64_t* tfull = empty + kPStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  // after the barrier words: per epilogue warp a 4 KB staging tile and a 2 KB exchange buffer
  unsigned char* epi_stage = reinterpret_cast<unsigned char*>(full + kPBarWords);
  float* epi_x = reinterpret_cast<float*>(epi_stage + 4 * kEpiStageBytes);
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_pre[kMaxE + 1];
  __shared__ int s_total;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int cl = (int)cluster_index(), ncl = (int)cluster_count();
  const int NF = kMode == 0 ? a.I / (2 * 64) : a.H / (2 * kPM);  // pair feature tiles per token tile
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
      mbar_init(&tempty[s], 8);  // the epilogue warps of both CTAs
    }
    mbar_init(done, 1);
    s_abort = 0;
    int acc = 0;
    for (int li = 0; li < nl; ++li) {
      s_pre[li] = acc;
      const int e = a.list_e[li];
      const int rows = (e >= 0 && e < a.E) ? a.offset[e + 1] - a.offset[e] : 0;
      acc += ((rows + kPT - 1) / kPT) * NF;
    }
    s_pre[nl] = acc;
    s_total = acc;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&s_tmem, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated on both
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int total = s_total;
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t s = 0, use = 0;  // ring position: stage, and how often it has been filled before
      int last_use[kPStages];
      for (int i = 0; i < kPStages; ++i) last_use[i] = -1;
      bool dead = false;
      for (int t = cl; t < total && !dead; t += ncl) {
        int li, m, ft;
        find_tile(s_pre, nl, t, NF, li, m, ft);
        const int e = a.list_e[li];
        const int slot = a.e2s ? a.e2s[e] : e;
        const int row0 = a.offset[e] + m * kPT;
        const int ntok = min(kPT, a.offset[e + 1] - row0);
        const int rrow = row0 + (int)rank * (((ntok + 31) & ~31) >> 1);  // this CTA's half of the N rows
        const int watom = kMode == 0 ? 2 * ft + (int)rank : 4 * ft + 2 * (int)rank;
        for (int kb = 0; kb < nkb; ++kb) {
          if (use > 0 && !mbar_try_wait(&empty[s], (use - 1) & 1u) && !mbar_wait(&empty[s], (use - 1) & 1u)) {
            dead = true;
            *abort_flag = 1;
            set_status(a.status, MOE_DEV_TIMEOUT);
            break;
          }
          unsigned char* st = psm + s * kPStageBytes;
          // rank 0's barrier counts the bytes of both CTAs
          if (rank == 0) mbar_expect_tx(&full[s], 2 * kPStageBytes);
          const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
          // weights: 128 K rows x this CTA's 128 features (two 64-column swizzle atoms, 16 KB apart)
          if (kMode == 0) {
            tma_load_4d_pair(st, &mapW, fb, 0, kb * kPK, watom, 3 * slot);              // 64 gate columns
            tma_load_4d_pair(st + 16384, &mapW, fb, 0, kb * kPK, watom, 3 * slot + 1);  // the same 64 up columns
          } else {
            tma_load_4d_pair(st, &mapW, fb, 0, kb * kPK, watom, 3 * slot + 2);
          }
          // grouped rows: this CTA's half of the tile, 128 rows x 64 K per box, the stage's two K halves
          tma_load_3d_pair(st + kPAbytes, &mapX, fb, kb * kPK, rrow, 0);
          tma_load_3d_pair(st + kPAbytes + 16384, &mapX, fb, kb * kPK + 64, rrow, 0);
          last_use[s] = (int)use;
          if (++s == kPStages) {
            s = 0;
            ++use;
          }
        }
      }
      // after any timeout, rank 0 lets every load of both CTAs land before the CTAs can exit
      if ((dead || *abort_flag) && rank == 0)
        for (int i = 0; i < kPStages; ++i)
          if (last_use[i] >= 0) mbar_wait(&full[i], (uint32_t)last_use[i] & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // one thread issues every pair MMA; the loop keeps per-K-block work to a barrier test, a fence,
      // four MMAs and a commit (stage index and phase advance incrementally, descriptors are a base
      // plus the stage offset)
      const uint32_t sbase = smem_u32(psm);
      const uint64_t ad0 = smem_desc(sbase, 16384, 1024);            // weights, MN-major
      const uint64_t bd0 = smem_desc(sbase + kPAbytes, 16, 1024);    // grouped rows, K-major
      constexpr uint32_t kStageDesc = kPStageBytes >> 4;             // stage stride in descriptor units
      uint32_t s = 0, ph = 0, tc = 0;
      bool dead = false;
      for (int t = cl; t < total; t += ncl, ++tc) {
        int li, m, ft;
        find_tile(s_pre, nl, t, NF, li, m, ft);
        const int e = a.list_e[li];
        const int ntok = min(kPT, a.offset[e + 1] - a.offset[e] - m * kPT);
        // D^T = W^T X^T: M = 256 features (A MN-major, 128 per CTA), N = the tile's rows rounded up
        // to 32 (B K-major, half per CTA)
        const uint32_t idesc = idesc_bf16(2 * kPM, (ntok + 31) & ~31, 1, 0);
        const uint32_t acc = tc & 1u, ause = tc >> 1;
        if (ause > 0 && !dead && !mbar_wait(&tempty[acc], (ause - 1) & 1u)) {
          dead = true;
          *abort_flag = 1;
          set_status(a.status, MOE_DEV_TIMEOUT);
        }
        tc_fence_after();
        const uint32_t d = tmem + acc * kPT;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!dead && !mbar_try_wait(&full[s], ph) && !mbar_wait(&full[s], ph)) {
            dead = true;
            *abort_flag = 1;
            set_status(a.status, MOE_DEV_TIMEOUT);
          }
          tc_fence_after();
          if (!dead) {
            const uint64_t so = (uint64_t)(s * kStageDesc);
            // K 0..63 from the first K half of the rows, K 64..127 from the second (16 KB further)
            umma_f16_pair_k64(d, ad0 + so, bd0 + so, idesc, kb != 0, 2048 >> 4, 32 >> 4);
            umma_f16_pair_k64(d, ad0 + so + 4 * (2048 >> 4), bd0 + so + (16384 >> 4), idesc, 1, 2048 >> 4, 32 >> 4);
          }
          umma_commit_pair(&empty[s]);  // frees stage s in both CTAs
          if (++s == kPStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        umma_commit_pair(&tfull[acc]);
      }
      // `done` completes in both CTAs once every pair MMA has finished
      umma_commit_pair(done);
    }
    if (lane == 0) mbar_wait(done, 0);
  } else {
    // epilogue warps 2..5; TMEM lane quarter q = warp % 4 holds features 32q .. 32q+31 of this CTA's
    // 128, one grouped row per TMEM column (all N rows of the tile, in both CTAs).  A chunk is 32
    // rows: TMEM -> registers, transposed through shared memory into rows of 32 features, then
    // stored as 16-byte pieces of the output rows.
    const int q = warp & 3;
    unsigned char* stage = epi_stage + q * kEpiStageBytes;  // this warp's [32 rows][32 features]
    const uint32_t tempty_c0 = mapa_shared(smem_u32(&tempty[0]), 0);
    const uint32_t tempty_c1 = mapa_shared(smem_u32(&tempty[1]), 0);
    uint32_t tc = 0;
    for (int t = cl; t < total; t += ncl, ++tc) {
      int li, m, ft;
      find_tile(s_pre, nl, t, NF, li, m, ft);
      const int e = a.list_e[li];
      const int ntok = min(kPT, a.offset[e + 1] - a.offset[e] - m * kPT);
      const size_t p0 = (size_t)a.offset[e] + m * kPT;
      const uint32_t acc = tc & 1u, ause = tc >> 1;
      if (!*abort_flag && !mbar_wait(&tfull[acc], ause & 1u)) {
        *abort_flag = 1;
        set_status(a.status, MOE_DEV_TIMEOUT);
      }
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + acc * kPT;
      // the chunk count depends on the tile alone, so both warps of a pair take the same barriers
      const int nch = (ntok + 31) >> 5;
      if (kMode == 0) {
        // pair p = q & 1: warp q = p holds the gate values of features f0 + lane, warp q = p + 2 the
        // same features' up values.  Each hands the other the half it does not compute (gate warp:
        // rows 16..31 of the chunk, up warp: rows 0..15) and computes h for its own 16 rows.
        const int p = q & 1, role = q >> 1;
        float* xmine = epi_x + q * kEpiXFloats;
        const float* xother = epi_x + (q ^ 2) * kEpiXFloats;
        uint16_t* st16 = reinterpret_cast<uint16_t*>(stage);
        const int f0 = ft * 128 + 64 * (int)rank + 32 * p;
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
          float v[32];
          tmem_ld32(taddr + 32 * c, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) xmine[j * 32 + lane] = v[role == 0 ? 16 + j : j];
          named_sync(1 + p, 64);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float o = xother[j * 32 + lane];
            const float g = role == 0 ? v[j] : o, u = role == 0 ? o : v[16 + j];
            st16[j * 32 + lane] = f32_to_bf16(__fdividef(g, 1.f + __expf(-g)) * u);
          }
          __syncwarp();
          // 16 rows x 64 B: two 16-byte pieces per lane
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int idx = i * 32 + lane, r = idx >> 2, seg = idx & 3;
            const int tok = 32 * c + 16 * role + r;
            const uint4 val = *reinterpret_cast<const uint4*>(st16 + r * 32 + seg * 8);
            if (tok < ntok && !*abort_flag)
              *reinterpret_cast<uint4*>(a.hb + (p0 + tok) * a.I + f0 + seg * 8) = val;
          }
          named_sync(1 + p, 64);  // both warps are done with the exchange and staging buffers
        }
      } else {
        const int o0 = ft * 2 * kPM + kPM * (int)rank + 32 * q;
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
          float v[32];
          tmem_ld32(taddr + 32 * c, v);
          tmem_ld_wait();
          const bool store = !*abort_flag;
          if (a.yb) {
            uint16_t* st16 = reinterpret_cast<uint16_t*>(stage);
#pragma unroll
            for (int j = 0; j < 32; ++j) st16[j * 32 + lane] = f32_to_bf16(v[j]);
            __syncwarp();
            // 32 rows x 64 B: four 16-byte pieces per lane
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int idx = i * 32 + lane, r = idx >> 2, seg = idx & 3;
              const int tok = 32 * c + r;
              const uint4 val = *reinterpret_cast<const uint4*>(st16 + r * 32 + seg * 8);
              if (store && tok < ntok) *reinterpret_cast<uint4*>(a.yb + (p0 + tok) * a.H + o0 + seg * 8) = val;
            }
          } else {
            float* st32 = reinterpret_cast<float*>(stage);
#pragma unroll
            for (int j = 0; j < 32; ++j) st32[j * 32 + lane] = v[j];
            __syncwarp();
            // 32 rows x 128 B: eight 16-byte pieces per lane
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int idx = i * 32 + lane, r = idx >> 3, seg = idx & 7;
              const int tok = 32 * c + r;
              const uint4 val = *reinterpret_cast<const uint4*>(st32 + r * 32 + seg * 4);
              if (store && tok < ntok) *reinterpret_cast<uint4*>(a.y + (p0 + tok) * a.H + o0 + seg * 4) = val;
            }
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? tempty_c1 : tempty_c0);  // rank 0's accumulator barrier
    }
  }
  // warps 0 and 1 ran their loops on lane 0 alone: reconverge before the cluster barrier, which also
  // keeps each CTA's shared memory alive while its peer may still signal it
  __syncwarp();
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Xp[p] = x[rows[p] / k] for the n grouped rows (16-byte copies).
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ rows, int n, int H, int k,
                                                          uint16_t* __restrict__ xp) {
  // Launched as a dependent of the permute (stream path).  Wait first, then let the stream kernel
  // launch: it reads the permute's expert list and offsets before its own wait, so the permute must
  // have completed by the time it can start.
  pdl_wait();
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
  MOE_CUDA_TRY(launch_pdl(gather_rows_kernel, dim3(std::min(n, sms * 8)), dim3(256), 0, stream, x, rows, n, H, k, xp));
  return MOE_OK;
}

static size_t prefill_smem_bytes() {
  return 1024 + (size_t)kPStages * kPStageBytes + kPBarWords * sizeof(uint64_t) + 4 * kEpiStageBytes +
         4 * kEpiXFloats * sizeof(float);
}

bool prefill_eligible(const FfnArgs& a, int n) {
  return a.pool_only && a.S > 0 && a.xp && a.hb && n >= kPrefillMinRows && a.H % (2 * kPM) == 0 && a.I % 128 == 0 && a.H % kPK == 0 && a.I % kPK == 0 &&
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
    const uint32_t b[3] = {64, kPTBox, 1};  // 64 K = one 128-byte swizzle row
    if (encode_tmap_3d_bf16(&mx, a.xp, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B) != MOE_OK) return MOE_ERR_CUDA;
  }
  {
    const uint64_t d[3] = {(uint64_t)a.I, (uint64_t)n, 1};
    const uint64_t s[2] = {(uint64_t)a.I * 2, (uint64_t)n * a.I * 2};
    const uint32_t b[3] = {64, kPTBox, 1};
    if (encode_tmap_3d_bf16(&mh, a.hb, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B) != MOE_OK) return MOE_ERR_CUDA;
  }
  // weight matrices viewed as [matrix][64-column atom][K row][64 columns]
  {
    const uint64_t d[4] = {64, (uint64_t)a.H, (uint64_t)a.I / 64, 3ull * a.S};
    const uint64_t s[3] = {(uint64_t)a.I * 2, 128, mat * 2};
    const uint32_t b[4] = {64, kPK, 1, 1};  // one 64-column atom: the gate or the up half of a tile
    if (encode_tmap_bf16(&mgu, a.pool, 4, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B) != MOE_OK) return MOE_ERR_CUDA;
  }
  {
    const uint64_t d[4] = {64, (uint64_t)a.I, (uint64_t)a.H / 64, 3ull * a.S};
    const uint64_t s[3] = {(uint64_t)a.H * 2, 128, mat * 2};
    const uint32_t b[4] = {64, kPK, kPM / 64, 1};
    if (encode_tmap_bf16(&md, a.pool, 4, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B) != MOE_OK) return MOE_ERR_CUDA;
  }
  PrefillArgs p{a.H, a.I, a.E, n, a.offset, a.list_e, a.n_list, a.e2s, a.S, a.hb, a.y, a.status, a.yb};
  (void)max_list;
  // persistent CTA pairs: as many clusters of two as fit at once (one CTA per SM)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = prefill_smem_bytes();
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int ncl_cached[64] = {};
  const int di = dev < 64 ? dev : 63;
  if (ncl_cached[di] == 0) {
    cfg.gridDim = dim3((unsigned)(sms & ~1));
    int ncl = 0;
    MOE_CUDA_TRY(cudaOccupancyMaxActiveClusters(&ncl, (void*)prefill_gemm_kernel<0>, &cfg));
    if (ncl < 1) return MOE_ERR_CUDA;
    ncl_cached[di] = ncl;
  }
  cfg.gridDim = dim3((unsigned)(2 * ncl_cached[di]));
  if (prof) prof->begin(MOE_PROF_FFN_ROWS, stream);
  gather_rows_kernel<<<std::min(n, sms * 8), 256, 0, stream>>>(a.x, a.rows, n, a.H, a.k, a.xp);
  MOE_LAUNCH_CHECK();
  if (prof) prof->end(stream);
  if (prof) prof->begin(MOE_PROF_FFN_GATEUP, stream);
  MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, prefill_gemm_kernel<0>, p, mx, mgu));
  if (prof) prof->end(stream);
  if (prof) prof->begin(MOE_PROF_FFN_DOWN, stream);
  MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, prefill_gemm_kernel<1>, p, mh, md));
  if (prof) prof->end(stream);
  return MOE_OK;
}

}  // namespace moe
