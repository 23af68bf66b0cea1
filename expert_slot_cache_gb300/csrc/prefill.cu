// Grouped SwiGLU expert FFN for prefill-sized groups on the tcgen05 tensor cores.
//
// "Porting vllm-expert-cache to NVIDIA GPUs", "What this package does": the
// expert GEMM runs on the grouped, slot-remapped ids.  When the groups are
// large (prefill), the two GEMMs are dense contractions and run here:
//   GEMM 1: g = Xp_e Wg_e, u = Xp_e Wu_e, epilogue h = silu(g) * u (bf16)
//   GEMM 2: y = h_e Wd_e (bf16, or fp32)
// Xp is the routed rows of x in grouped order (copied once by
// gather_rows_kernel).
//
// The products are computed transposed, D^T = W^T X^T, by CTA pairs (a
// cluster of two on neighbouring SMs): the pair's MMA has M = 256 weight
// features (128 in each CTA's shared memory and TMEM) and N = up to 256 of
// one expert's grouped rows, rounded up to a multiple of 32, half of them in
// each CTA's shared memory.
//
// What sets the pace is how fast the operands reach shared memory (about
// 40 B per clock per SM from L2 on this part), not the MMAs, so the tiles
// are shaped to move few bytes per MMA cycle:
//   - GEMM 1 keeps two accumulators per tile: a CTA's 128 gate features and
//     the same 128 up features.  The grouped rows of a stage then feed 256
//     h features per CTA pair instead of 128, and the epilogue finds g and u
//     of one feature in the same TMEM lane.  The two accumulators fill TMEM
//     (2 x 256 columns), so the epilogue of a tile does not overlap the MMAs
//     of the next; it is short next to the 2048-deep main loop.
//   - GEMM 2 (K = I, a short main loop) keeps one accumulator per tile and
//     double-buffers it, so its epilogue overlaps the next tile.
//   - A ragged tile loads only its rows (rounded up to 16 per CTA): tensor
//     maps with boxes of 128, 64, 32 and 16 rows.
//
// Persistent clusters over the tiles of all experts (expert-major, then
// token tile, then feature tile, so a token tile stays hot in L2 while the
// clusters walk the expert's weights); per CTA:
//   warp 0: TMA producer (one thread); the loads of both CTAs complete on
//           rank 0's barrier
//   warp 1: TMEM allocation (both CTAs) + pair MMA issue (rank 0, one thread)
//   warps 2-5: epilogue, TMEM -> registers -> shared (transpose) -> global
// Shared-memory operands use the 128-byte swizzle written by the tensor-map
// loads: weights MN-major (stored input-major: 64 output columns = 128 B per
// K row, 8 K rows per 1 KB swizzle group, 64-column atoms one K depth
// apart), grouped rows K-major (rows of 64 bf16 = 128 B).  One thread issues
// the MMAs, and a tcgen05.mma costs it tens of cycles to issue, so each ring
// stage carries eight MMAs per barrier wait and commit.
#include "internal.cuh"
#include "tc05.cuh"

namespace moe {

constexpr int kPM = 128;     // weight features per CTA (the pair's MMA M is 256)
constexpr int kPT = 256;     // grouped rows per tile, at most (MMA N)
constexpr int kPTBox = 128;  // grouped rows per CTA and tile, at most
constexpr uint32_t kTmemCols = 512;
constexpr int kPBarWords = 32;  // mbarriers: full / empty per stage, two accumulators, done
constexpr int kPrefillMinRows = 4096;
constexpr int kMaxTT = 2048;    // token tiles per launch

// Ring geometry.  GEMM 1: a 64-deep stage holds 128 gate and the same 128 up features (2 x 16 KB)
// and up to 128 rows (16 KB).  GEMM 2: a 128-deep stage holds 128 features (32 KB) and up to 128
// rows in two 64-deep halves (32 KB).  GEMM 1 drains its tile with eight epilogue warps (two per
// TMEM lane quarter, alternate 32-row chunks), as that drain is not overlapped with the next
// tile's MMAs; GEMM 2 with four.
template <int kMode>
struct PGeo {
  static constexpr int K = kMode == 0 ? 64 : 128;        // K depth of a stage
  static constexpr int Stages = kMode == 0 ? 4 : 3;
  static constexpr int ABytes = (kMode == 0 ? 2 : 1) * kPM * K * 2;
  static constexpr int StageBytes = ABytes + kPTBox * K * 2;
  static constexpr int Acc = kMode == 0 ? 1 : 2;         // accumulator buffers
  static constexpr uint32_t AtomBytes = 64 * K * 2;      // one 64-feature column atom of a stage
  static constexpr int EpiWarps = kMode == 0 ? 8 : 4;
  static constexpr int Threads = 64 + 32 * EpiWarps;
  static constexpr int EpiBytes = kMode == 0 ? 32 * 32 * 2 : 32 * 32 * 4;  // staging per epilogue warp
};

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

// Tensor maps of the grouped-row operand (Xp for GEMM 1, h for GEMM 2): the
// same [n][K] matrix with boxes of 128, 64, 32 and 16 rows x 64 K.
struct RowMaps {
  CUtensorMap m[4];
};

// Load r rows (a multiple of 16, at most 128) from row `row`, K columns kc .. kc+63, into dst:
// 128 rows in one box, fewer as 64 + 32 + 16 (rows of 128 B, so every piece starts on a 1 KB
// swizzle group).
__device__ __forceinline__ void load_rows(unsigned char* dst, const RowMaps& mx, uint32_t cbar, int kc, int row,
                                          int r) {
  if (r == kPTBox) {
    tma_load_3d_pair(dst, &mx.m[0], cbar, kc, row, 0);
    return;
  }
  int d = 0;
  if (r & 64) {
    tma_load_3d_pair(dst, &mx.m[1], cbar, kc, row, 0);
    d = 64;
  }
  if (r & 32) {
    tma_load_3d_pair(dst + d * 128, &mx.m[2], cbar, kc, row + d, 0);
    d += 32;
  }
  if (r & 16) tma_load_3d_pair(dst + d * 128, &mx.m[3], cbar, kc, row + d, 0);
}

// Tile t of the launch: token tile tt[t / nf] (expert list index and 256-row tile), feature tile
// t % nf.
__device__ __forceinline__ void tile_of(const int* tt, int t, int nf, int& li, int& m, int& ft) {
  const int i = t / nf;
  ft = t - i * nf;
  const int p = tt[i];
  li = p & (kMaxE - 1);
  m = p >> 10;
}
static_assert(kMaxE == 1024, "token-tile entries pack the list index in 10 bits");

template <int kMode>
__global__ void __launch_bounds__(PGeo<kMode>::Threads, 1) prefill_gemm_kernel(const PrefillArgs a,
                                                                    const __grid_constant__ RowMaps mapX,
                                                                    const __grid_constant__ CUtensorMap mapW) {
  using G = PGeo<kMode>;
  extern __shared__ __align__(16) unsigned char psm_raw[];
  unsigned char* psm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(psm_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(psm + G::Stages * G::StageBytes);
  uint64_t* empty = full + G::Stages;
  uint64_t* tfull = empty + G::Stages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  unsigned char* epi_stage = reinterpret_cast<unsigned char*>(full + kPBarWords);  // G::EpiBytes per epilogue warp
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_tt[kMaxTT];  // token tiles: (256-row tile << 10) | expert list index
  __shared__ int s_ntt;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int cl = (int)cluster_index(), ncl = (int)cluster_count();
  const int NF = kMode == 0 ? a.I / (2 * kPM) : a.H / (2 * kPM);  // pair feature tiles per token tile
  const int K = kMode == 0 ? a.H : a.I;
  const int nkb = K / G::K;
  const int nl = min(*a.n_list, kMaxE);

  // Token-tile list, built by all threads: each expert's row count, an exclusive scan of the tile
  // counts by warp 0, then each expert's entries.  The ring is not in use yet, so its first bytes
  // hold the per-expert counts.
  int* s_cnt = reinterpret_cast<int*>(psm);
  int* s_pre = s_cnt + kMaxE;
  for (int li = threadIdx.x; li < nl; li += G::Threads) {
    const int e = a.list_e[li];
    const int rows = (e >= 0 && e < a.E) ? a.offset[e + 1] - a.offset[e] : 0;
    s_cnt[li] = rows > 0 ? (rows + kPT - 1) / kPT : 0;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < G::Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], 2 * G::EpiWarps);  // the epilogue warps of both CTAs
    }
    mbar_init(done, 1);
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&s_tmem, kTmemCols);
    tmem_relinquish_pair();
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < nl; base += 32) {
      const int li = base + lane;
      const int c = li < nl ? s_cnt[li] : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(MOE_FULL_MASK, incl, o);
        if (lane >= o) incl += v;
      }
      if (li < nl) s_pre[li] = carry + incl - c;
      carry += __shfl_sync(MOE_FULL_MASK, incl, 31);
    }
    if (lane == 0) {
      s_ntt = carry;
      if (carry > kMaxTT) set_status(a.status, MOE_DEV_BAD_GROUPS);  // the host sized the table for n rows
    }
  }
  __syncthreads();
  const int ntt = s_ntt <= kMaxTT ? s_ntt : 0;
  for (int li = threadIdx.x; li < nl; li += G::Threads)
    for (int m = 0, p = s_pre[li]; m < s_cnt[li] && p + m < ntt; ++m) s_tt[p + m] = (m << 10) | li;
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated on both, tile list complete
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int total = ntt * NF;
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t s = 0, use = 0;  // ring position: stage, and how often it has been filled before
      int last_use[G::Stages];
      for (int i = 0; i < G::Stages; ++i) last_use[i] = -1;
      bool dead = false;
      for (int t = cl; t < total && !dead; t += ncl) {
        int li, m, ft;
        tile_of(s_tt, t, NF, li, m, ft);
        const int e = a.list_e[li];
        const int slot = a.e2s ? a.e2s[e] : e;
        const int row0 = a.offset[e] + m * kPT;
        const int ntok = min(kPT, a.offset[e + 1] - row0);
        const int r = ((ntok + 31) & ~31) >> 1;  // rows per CTA: half the MMA's N
        const int rrow = row0 + (int)rank * r;    // this CTA's half of the tile's rows
        const int watom = 4 * ft + 2 * (int)rank;  // this CTA's first 64-feature column atom
        const uint32_t bytes = 2u * (uint32_t)(G::ABytes + (G::K / 64) * r * 128);  // both CTAs
        for (int kb = 0; kb < nkb; ++kb) {
          if (use > 0 && !mbar_try_wait(&empty[s], (use - 1) & 1u) && !mbar_wait(&empty[s], (use - 1) & 1u)) {
            dead = true;
            *abort_flag = 1;
            set_status(a.status, MOE_DEV_TIMEOUT);
            break;
          }
          unsigned char* st = psm + s * G::StageBytes;
          // rank 0's barrier counts the bytes of both CTAs
          if (rank == 0) mbar_expect_tx(&full[s], bytes);
          const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
          if (kMode == 0) {
            // 64 K rows x this CTA's 128 gate features, then the same 128 up features
            tma_load_4d_pair(st, &mapW, fb, 0, kb * G::K, watom, 3 * slot);
            tma_load_4d_pair(st + 16384, &mapW, fb, 0, kb * G::K, watom, 3 * slot + 1);
            load_rows(st + G::ABytes, mapX, fb, kb * G::K, rrow, r);
          } else {
            // 128 K rows x this CTA's 128 features; the rows' two 64-deep K halves 16 KB apart
            tma_load_4d_pair(st, &mapW, fb, 0, kb * G::K, watom, 3 * slot + 2);
            load_rows(st + G::ABytes, mapX, fb, kb * G::K, rrow, r);
            load_rows(st + G::ABytes + 16384, mapX, fb, kb * G::K + 64, rrow, r);
          }
          last_use[s] = (int)use;
          if (++s == G::Stages) {
            s = 0;
            ++use;
          }
        }
      }
      // after any timeout, rank 0 lets every load of both CTAs land before the CTAs can exit
      if ((dead || *abort_flag) && rank == 0)
        for (int i = 0; i < G::Stages; ++i)
          if (last_use[i] >= 0) mbar_wait(&full[i], (uint32_t)last_use[i] & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // one thread issues every pair MMA; the loop keeps per-stage work to a barrier test, a fence,
      // eight MMAs and a commit (stage index and phase advance incrementally, descriptors are a base
      // plus the stage offset)
      const uint32_t sbase = smem_u32(psm);
      const uint64_t ad0 = smem_desc(sbase, G::AtomBytes, 1024);        // weights, MN-major
      const uint64_t bd0 = smem_desc(sbase + G::ABytes, 16, 1024);      // grouped rows, K-major
      constexpr uint32_t kStageDesc = G::StageBytes >> 4;               // stage stride in descriptor units
      constexpr uint32_t kAStep = 2048 >> 4, kBStep = 32 >> 4;         // one 16-deep K step
      uint32_t s = 0, ph = 0, tc = 0;
      bool dead = false;
      for (int t = cl; t < total; t += ncl, ++tc) {
        int li, m, ft;
        tile_of(s_tt, t, NF, li, m, ft);
        const int e = a.list_e[li];
        const int ntok = min(kPT, a.offset[e + 1] - a.offset[e] - m * kPT);
        // D^T = W^T X^T: M = 256 features (A MN-major, 128 per CTA), N = the tile's rows rounded up
        // to 32 (B K-major, half per CTA)
        const uint32_t idesc = idesc_bf16(2 * kPM, (ntok + 31) & ~31, 1, 0);
        const uint32_t acc = tc % G::Acc, ause = tc / G::Acc;
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
            if (kMode == 0) {
              // gate accumulator in columns 0..255, up accumulator in 256..511
              umma_f16_pair_k64(d, ad0 + so, bd0 + so, idesc, kb != 0, kAStep, kBStep);
              umma_f16_pair_k64(d + kPT, ad0 + so + (16384 >> 4), bd0 + so, idesc, kb != 0, kAStep, kBStep);
            } else {
              // K 0..63 from the first K half of the rows, K 64..127 from the second (16 KB further)
              umma_f16_pair_k64(d, ad0 + so, bd0 + so, idesc, kb != 0, kAStep, kBStep);
              umma_f16_pair_k64(d, ad0 + so + 4 * kAStep, bd0 + so + (16384 >> 4), idesc, 1, kAStep, kBStep);
            }
          }
          umma_commit_pair(&empty[s]);  // frees stage s in both CTAs
          if (++s == G::Stages) {
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
    const int q = warp & 3, half = (warp - 2) >> 2;  // lane quarter; which alternate chunks (GEMM 1)
    unsigned char* stage = epi_stage + (warp - 2) * G::EpiBytes;  // this warp's [32 rows][32 features]
    const uint32_t tempty_c0 = mapa_shared(smem_u32(&tempty[0]), 0);
    const uint32_t tempty_c1 = mapa_shared(smem_u32(&tempty[1]), 0);
    const int f0 = kPM * (int)rank + 32 * q;  // this warp's first feature within the pair's 256
    uint32_t tc = 0;
    for (int t = cl; t < total; t += ncl, ++tc) {
      int li, m, ft;
      tile_of(s_tt, t, NF, li, m, ft);
      const int e = a.list_e[li];
      const int ntok = min(kPT, a.offset[e + 1] - a.offset[e] - m * kPT);
      const size_t p0 = (size_t)a.offset[e] + m * kPT;
      const uint32_t acc = tc % G::Acc, ause = tc / G::Acc;
      if (!*abort_flag && !mbar_wait(&tfull[acc], ause & 1u)) {
        *abort_flag = 1;
        set_status(a.status, MOE_DEV_TIMEOUT);
      }
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + acc * kPT;
      const int nch = (ntok + 31) >> 5;
      const int col0 = ft * 2 * kPM + f0;  // output column of lane 0's feature
      if (kMode == 0) {
        // lane = feature: its gate values in accumulator 0, its up values in accumulator 1
        uint16_t* st16 = reinterpret_cast<uint16_t*>(stage);
#pragma unroll 1
        for (int c = half; c < nch; c += 2) {
          float g[32], u[32];
          tmem_ld32(taddr + 32 * c, g);
          tmem_ld32(taddr + kPT + 32 * c, u);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) st16[j * 32 + lane] = f32_to_bf16(__fdividef(g[j], 1.f + __expf(-g[j])) * u[j]);
          __syncwarp();
          const bool store = !*abort_flag;
          // 32 rows x 64 B: four 16-byte pieces per lane
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int idx = i * 32 + lane, r = idx >> 2, seg = idx & 3;
            const int tok = 32 * c + r;
            const uint4 val = *reinterpret_cast<const uint4*>(st16 + r * 32 + seg * 8);
            if (store && tok < ntok) *reinterpret_cast<uint4*>(a.hb + (p0 + tok) * a.I + col0 + seg * 8) = val;
          }
          __syncwarp();
        }
      } else {
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
              if (store && tok < ntok) *reinterpret_cast<uint4*>(a.yb + (p0 + tok) * a.H + col0 + seg * 8) = val;
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
              if (store && tok < ntok) *reinterpret_cast<uint4*>(a.y + (p0 + tok) * a.H + col0 + seg * 4) = val;
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

template <int kMode>
static size_t prefill_smem_bytes() {
  using G = PGeo<kMode>;
  return 1024 + (size_t)G::Stages * G::StageBytes + kPBarWords * sizeof(uint64_t) + (size_t)G::EpiWarps * G::EpiBytes;
}

bool prefill_eligible(const FfnArgs& a, int n) {
  // features in whole pair tiles (256 h features in GEMM 1, 256 outputs in GEMM 2), K in whole
  // stages, and a token-tile list that fits the kernel's table
  return a.pool_only && a.S > 0 && a.xp && a.hb && n >= kPrefillMinRows && a.H % (2 * kPM) == 0 &&
         a.I % (2 * kPM) == 0 && a.E <= kMaxE && (int64_t)n / kPT + a.E <= kMaxTT;
}

size_t prefill_extra_bytes(int n, int H, int I) {
  if (n < kPrefillMinRows) return 0;
  return (size_t)n * H * 2 + (size_t)n * I * 2 + 512;
}

// The four row maps (boxes of 128, 64, 32, 16 rows x 64 K) of a bf16 [n][K] matrix.
static int encode_row_maps(RowMaps* rm, const void* base, int n, int K) {
  const uint64_t d[3] = {(uint64_t)K, (uint64_t)n, 1};
  const uint64_t s[2] = {(uint64_t)K * 2, (uint64_t)n * K * 2};
  for (int i = 0; i < 4; ++i) {
    const uint32_t b[3] = {64, (uint32_t)(kPTBox >> i), 1};  // 64 K = one 128-byte swizzle row
    if (encode_tmap_3d_bf16(&rm->m[i], base, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B) != MOE_OK) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int launch_prefill(const FfnArgs& a, int n, int max_list, cudaStream_t stream, Prof* prof) {
  static bool done0[64] = {}, done1[64] = {};
  MOE_CUDA_TRY(ensure_smem(prefill_gemm_kernel<0>, (int)prefill_smem_bytes<0>(), done0));
  MOE_CUDA_TRY(ensure_smem(prefill_gemm_kernel<1>, (int)prefill_smem_bytes<1>(), done1));
  int dev = 0, sms = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const size_t mat = (size_t)a.H * a.I;
  RowMaps mx, mh;
  CUtensorMap mgu, md;
  if (encode_row_maps(&mx, a.xp, n, a.H) != MOE_OK) return MOE_ERR_CUDA;
  if (encode_row_maps(&mh, a.hb, n, a.I) != MOE_OK) return MOE_ERR_CUDA;
  // weight matrices viewed as [matrix][64-column atom][K row][64 columns]; a box is one stage's
  // K rows x two atoms (this CTA's 128 features)
  {
    const uint64_t d[4] = {64, (uint64_t)a.H, (uint64_t)a.I / 64, 3ull * a.S};
    const uint64_t s[3] = {(uint64_t)a.I * 2, 128, mat * 2};
    const uint32_t b[4] = {64, (uint32_t)PGeo<0>::K, kPM / 64, 1};
    if (encode_tmap_bf16(&mgu, a.pool, 4, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B) != MOE_OK) return MOE_ERR_CUDA;
  }
  {
    const uint64_t d[4] = {64, (uint64_t)a.I, (uint64_t)a.H / 64, 3ull * a.S};
    const uint64_t s[3] = {(uint64_t)a.H * 2, 128, mat * 2};
    const uint32_t b[4] = {64, (uint32_t)PGeo<1>::K, kPM / 64, 1};
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
  cfg.blockDim = dim3(PGeo<0>::Threads);
  cfg.dynamicSmemBytes = prefill_smem_bytes<0>();
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
  cfg.dynamicSmemBytes = prefill_smem_bytes<1>();
  cfg.blockDim = dim3(PGeo<1>::Threads);
  MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, prefill_gemm_kernel<1>, p, mh, md));
  if (prof) prof->end(stream);
  return MOE_OK;
}

}  // namespace moe
