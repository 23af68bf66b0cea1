// C ABI entry points that compose the kernels: the expert FFN, the combine and
// the whole layer forward (route, then per chunk permute, manage, gather on
// the side stream overlapped with the hit experts' FFN, the missed experts'
// FFN, combine).
#include <algorithm>
#include <mutex>

#include "internal.cuh"

namespace moe {

static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// A later wave's loads go in up to kMaxSub sub-batches: the side stream gathers them back to back
// while the main stream runs each sub-batch's FFN once its gather has landed.
constexpr int kMaxSub = kMaxSubBatches;

// Sub-batch boundaries of a later wave's loads (at most wmax), in eighths 1 : 3 : 3 : 1.  A small first
// sub-batch, since the FFN of the experts it evicts keeps the host link idle until it ends; a small last
// one, since its FFN follows the last gather.  (Measured on the T = 64, 64-slot step, graph replay:
// quarters 3.007 ms, 1 : 3 : 3 : 1 2.998 ms, 1 : 7 : 7 : 1 3.05 ms, 1 : 15 : 15 : 1 3.2 ms; gathers of
// many experts at once ran slower per expert.)
static SubBatches sub_batches(int wmax) {
  SubBatches sb;
  if (wmax < 4) {
    sb.n = wmax > 0 ? 1 : 0;
    sb.off[1] = wmax;
    return sb;
  }
  const int edge = std::max(1, (wmax + 4) / 8), mid = edge + (wmax - 2 * edge + 1) / 2;
  sb.n = 4;
  sb.off[0] = 0;
  sb.off[1] = edge;
  sb.off[2] = mid;
  sb.off[3] = wmax - edge;
  sb.off[4] = wmax;
  return sb;
}

// Workspace layout of the layer forward, for chunks of up to n = C*k routing slots.
struct LayerWs {
  int32_t* ctr;  // arrival counters of the persistent decode kernel (zero between calls)
  int32_t* sub_n;  // per-sub-batch counts of a later wave's loads
  int32_t *count, *offset, *rows, *pos, *act_e, *n_act, *miss_e, *miss_s, *n_miss, *hit_e, *n_hit, *def_e, *n_def;
  int32_t *wl_e, *wl_s, *n_wl, *ev_e, *kept_e, *n_kept;  // later waves: loads, evicted experts, kept experts
  float *hbuf, *y, *logits, *route;
  uint16_t *xp, *hb;
  int32_t* perm;
  float* skp;
  size_t skp_bytes;
  size_t bytes;
};

// n = routing slots per chunk, T = tokens of the whole step (router logits).
static LayerWs carve(void* base, int n, int H, int E, int I, int T) {
  LayerWs w{};
  size_t off = 0;
  char* b = (char*)base;
  auto take = [&](size_t bytes) {
    char* p = b ? b + off : nullptr;
    off += align256(bytes);
    return p;
  };
  const int lmax = std::min(n, E);
  w.ctr = (int32_t*)take(4 * decode_ctr_ints(E));  // first, so its place does not depend on n
  w.sub_n = (int32_t*)take(4 * kMaxSub);
  w.count = (int32_t*)take(4 * (size_t)E);
  w.offset = (int32_t*)take(4 * (size_t)(E + 1));
  w.rows = (int32_t*)take(4 * (size_t)n);
  w.pos = (int32_t*)take(4 * (size_t)n);
  w.act_e = (int32_t*)take(4 * (size_t)E);
  w.n_act = (int32_t*)take(4);
  w.miss_e = (int32_t*)take(4 * (size_t)lmax);
  w.miss_s = (int32_t*)take(4 * (size_t)lmax);
  w.n_miss = (int32_t*)take(4);
  w.hit_e = (int32_t*)take(4 * (size_t)lmax);
  w.n_hit = (int32_t*)take(4);
  w.def_e = (int32_t*)take(4 * (size_t)lmax);
  w.n_def = (int32_t*)take(4);
  w.wl_e = (int32_t*)take(4 * (size_t)lmax);
  w.wl_s = (int32_t*)take(4 * (size_t)lmax);
  w.n_wl = (int32_t*)take(4);
  w.ev_e = (int32_t*)take(4 * (size_t)lmax);
  w.kept_e = (int32_t*)take(4 * (size_t)lmax);
  w.n_kept = (int32_t*)take(4);
  w.hbuf = (float*)take(4 * (size_t)n * I);
  w.y = (float*)take(4 * (size_t)n * H);
  w.logits = (float*)take(4 * (size_t)T * E);
  w.route = (float*)take(moe_route_scratch_bytes(T, H, E) + 4);
  w.perm = (int32_t*)take(moe_permute_scratch_bytes(n, E) + 4);
  if (prefill_extra_bytes(n, H, I) > 0) {
    w.xp = (uint16_t*)take(2 * (size_t)n * H);
    w.hb = (uint16_t*)take(2 * (size_t)n * I);
  }
  w.skp_bytes = std::max(sk_part_bytes(n, H, I), q8_ws_bytes(n, H, I));  // bf16 stream or W8A8 buffers
  if (w.skp_bytes) w.skp = (float*)take(w.skp_bytes);
  w.bytes = off;
  return w;
}

static int chunk_tokens(int T, int k, int S, int E, int mode, int policy, int schedule) {
  if (mode != MOE_MODE_GATHER || policy == MOE_POLICY_STATIC || schedule == MOE_SCHED_WAVES) return T;
  if (S >= E || T * k <= S) return T;
  return S / k;
}

// Manage calls after the first one in the expert-wave schedule: the deferred
// experts (at most min(n, E) - S of them) in batches of S.
static int later_waves(int n, int E, int S) {
  const int most = std::min(n, E) - S;
  return most > 0 ? (most + S - 1) / S : 0;
}

// Cached events per device for the fork/join with the side stream (one per sub-batch of a wave's gather).
struct DevEvents {
  cudaEvent_t fork = nullptr, join = nullptr, sub[kMaxSub] = {};
};
static DevEvents g_events[64];
static std::mutex g_events_mu;

static int get_events(DevEvents** out) {
  int dev = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_events_mu);
  DevEvents& d = g_events[dev];
  if (!d.fork) {
    MOE_CUDA_TRY(cudaEventCreateWithFlags(&d.fork, cudaEventDisableTiming));
    MOE_CUDA_TRY(cudaEventCreateWithFlags(&d.join, cudaEventDisableTiming));
    for (int b = 0; b < kMaxSub; ++b) MOE_CUDA_TRY(cudaEventCreateWithFlags(&d.sub[b], cudaEventDisableTiming));
  }
  *out = &d;
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" const char* moe_status_str(int s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_CAPACITY: return "step needs more slots than the pool holds";
    case MOE_ERR_ALIGN: return "slab size or pointer not a 16-byte multiple (or workspace too small)";
    case MOE_ERR_NOT_DEVICE_ACCESSIBLE: return "host store is not addressable by the device";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_STATUS: return "a kernel reported an invalid item";
    case MOE_ERR_SCRATCH_LIMIT: return "request exceeds the fixed scratch of the allocation-free entry point";
    default: return "unknown status";
  }
}

extern "C" size_t moe_ffn_workspace_bytes(int T, int H, int k, int I) {
  if (T < 1 || H < 1 || k < 1 || I < 1) return 0;
  const size_t n = (size_t)T * k;
  size_t b = align256(4 * n * I);
  if (prefill_extra_bytes((int)n, H, I) > 0) b += align256(2 * n * H) + align256(2 * n * I);
  const size_t skb = sk_part_bytes((int)n, H, I);
  if (skb) b += 256 + skb;  // 256: the parts start on a 256-byte boundary of a 16-byte aligned workspace
  return b;
}

extern "C" int moe_expert_ffn(const void* x, int T, int H, int I, int k, int E, const int32_t* offset,
                              const int32_t* rows, const int32_t* list_e, const int32_t* n_list, int max_list,
                              const void* pool, int S, const int32_t* e2s, const void* host_slabs, float* y,
                              void* workspace, size_t workspace_bytes, int32_t* dev_status, moe_stream_t stream) {
  if (!x || !offset || !rows || !list_e || !n_list || !pool || !y || !workspace) return MOE_ERR_ARG;
  if (!shape_ok(T, H, I, k, E) || max_list < 0 || S < 1 || (!e2s && S < E)) return MOE_ERR_ARG;
  if ((uintptr_t)pool % 16 || (uintptr_t)y % 16 || (uintptr_t)workspace % 16 || (uintptr_t)x % 16)
    return MOE_ERR_ALIGN;
  const size_t n = (size_t)T * k;
  if (workspace_bytes < align256(4 * n * I)) return MOE_ERR_ALIGN;
  if (host_slabs) {
    if ((uintptr_t)host_slabs % 16) return MOE_ERR_ALIGN;
    const int acc = check_host_accessible(host_slabs);
    if (acc != MOE_OK) return acc;
  }
  FfnArgs a{(const uint16_t*)x, T, H, I, k, E, offset, rows, list_e, n_list, (const uint16_t*)pool, e2s,
            (const uint16_t*)host_slabs, (size_t)3 * H * I, (float*)workspace, y, dev_status, S,
            host_slabs == nullptr, nullptr, nullptr, nullptr, nullptr, 0};
  if (workspace_bytes >= moe_ffn_workspace_bytes(T, H, k, I)) {
    char* b = (char*)workspace + align256(4 * n * I);
    if (prefill_extra_bytes((int)n, H, I) > 0) {
      a.xp = (uint16_t*)b;
      a.hb = (uint16_t*)(b + align256(2 * n * H));
      b += align256(2 * n * H) + align256(2 * n * I);
    }
    a.skp_bytes = sk_part_bytes((int)n, H, I);
    if (a.skp_bytes) a.skp = (float*)(((uintptr_t)b + 255) & ~uintptr_t(255));
  }
  return launch_ffn(a, std::min(max_list, E), (cudaStream_t)stream);
}

extern "C" int moe_combine(const float* y, const float* w, const int32_t* pos, const int32_t* ids, const int32_t* e2s,
                           int T, int k, int H, int E, int split, void* out, float* out_res, float* out_miss,
                           moe_stream_t stream) {
  if (!y || !w || !pos || !out || T < 1 || k < 1 || k > kMaxK || H < 4 || H % 4 || E < 1) return MOE_ERR_ARG;
  if (split && (!ids || !e2s || !out_res || !out_miss)) return MOE_ERR_ARG;
  if ((uintptr_t)y % 16 || (uintptr_t)out % 8) return MOE_ERR_ALIGN;
  if (split && ((uintptr_t)out_res % 16 || (uintptr_t)out_miss % 16)) return MOE_ERR_ALIGN;
  return launch_combine(y, w, pos, ids, e2s, T, k, H, E, split, out, out_res, out_miss, (cudaStream_t)stream);
}

extern "C" size_t moe_layer_workspace_bytes(int T, int H, int E, int k, int I, int S) {
  if (T < 1 || k < 1 || E < 1 || S < 1) return 0;
  // Worst case over modes: the largest chunk is all T tokens.
  return carve(nullptr, T * k, H, E, I, T).bytes;
}

extern "C" size_t moe_workspace_bytes(int T, int H, int I, int E, int k) {
  return moe_layer_workspace_bytes(T, H, E, k, I, E);
}

extern "C" int moe_layer_forward(const moe_layer_args* a, moe_stream_t main_s, moe_stream_t side_s) {
  if (!a) return MOE_ERR_ARG;
  const int T = a->T, H = a->H, E = a->E, k = a->k, I = a->I, S = a->S;
  if (!shape_ok(T, H, I, k, E) || S < 1) return MOE_ERR_ARG;
  if (!a->x || !a->w_router || !a->pool || !a->ids || !a->w || !a->out || !a->workspace) return MOE_ERR_ARG;
  const int mode = a->mode, policy = a->policy;
  if (mode < MOE_MODE_RESIDENT || mode > MOE_MODE_ZERO_RETURN) return MOE_ERR_ARG;
  if (mode == MOE_MODE_GATHER && policy != MOE_POLICY_LRU && policy != MOE_POLICY_LFU) return MOE_ERR_ARG;
  if (mode == MOE_MODE_ZERO_RETURN && policy != MOE_POLICY_STATIC) return MOE_ERR_ARG;
  if (mode != MOE_MODE_RESIDENT) {
    if (!a->e2s || !a->s2e || !a->prio || !a->stamp || !a->host_slabs) return MOE_ERR_ARG;
    if ((uintptr_t)a->host_slabs % 16) return MOE_ERR_ALIGN;
    const int acc = check_host_accessible(a->host_slabs);
    if (acc != MOE_OK) return acc;
  } else if (!a->e2s && S < E) {
    return MOE_ERR_ARG;
  }
  if (mode == MOE_MODE_ZERO_RETURN && (!a->out_res || !a->out_miss)) return MOE_ERR_ARG;
  if (a->quant != 0 && a->quant != 1) return MOE_ERR_ARG;
  if (a->quant && (mode == MOE_MODE_ZERO_RETURN || H % 16 || I % 16)) return MOE_ERR_ARG;
  if (a->schedule != MOE_SCHED_CHUNKS && a->schedule != MOE_SCHED_WAVES) return MOE_ERR_ARG;
  if (a->decode_kernels != 0 && a->decode_kernels != 1) return MOE_ERR_ARG;
  if (a->route_flags & ~(MOE_ROUTE_SIGMOID | MOE_ROUTE_DAMPED)) return MOE_ERR_ARG;
  if ((a->route_flags & MOE_ROUTE_SIGMOID) && (a->route_flags & MOE_ROUTE_DAMPED)) return MOE_ERR_ARG;
  const bool waves = mode == MOE_MODE_GATHER && a->schedule == MOE_SCHED_WAVES;
  if (mode == MOE_MODE_GATHER && !waves && S < E && S < k) return MOE_ERR_CAPACITY;
  if ((uintptr_t)a->pool % 16 || (uintptr_t)a->workspace % 256 || (uintptr_t)a->x % 16 || (uintptr_t)a->out % 8)
    return MOE_ERR_ALIGN;

  const int C = chunk_tokens(T, k, S, E, mode, policy, a->schedule);
  LayerWs ws = carve(a->workspace, C * k, H, E, I, T);
  if (a->workspace_bytes < ws.bytes) return MOE_ERR_ALIGN;

  cudaStream_t ms = (cudaStream_t)main_s;
  cudaStream_t ss = (cudaStream_t)side_s;
  const bool two = ss != nullptr && ss != ms;
  DevEvents* ev = nullptr;
  if (two) {
    const int r = get_events(&ev);
    if (r != MOE_OK) return r;
  }
  int64_t* stats = a->stats;
  Prof prof;
  prof.p = a->prof;
  if (prof.p) prof.p->used = 0;
  const size_t slab_bytes = a->quant ? q8_slab_bytes_h(H, I) : (size_t)6 * H * I;
  if (mode == MOE_MODE_GATHER && !a->window_counts && a->decode_kernels == 0 && C >= T && ws.skp) {
    // a small expert-cache step: manage, gather and the whole layer in one persistent launch
    int dev = 0, sms = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const bool bf = !a->quant && decode_gather_eligible(T, H, E, k, I, S, policy, a->x, a->w_router, a->pool,
                                                        a->host_slabs, sms);
    const bool q8 = a->quant && decode_q8_gather_eligible(T, H, E, k, I, S, policy, a->x, a->w_router, a->pool,
                                                          a->host_slabs, sms);
    if (bf || q8) {
      prof.begin(MOE_PROF_DECODE, ms);
      const int rd = bf ? launch_decode_gather(a, ws.route, ws.logits, ws.skp, ws.skp_bytes, ws.ctr, ms)
                        : launch_decode_q8_gather(a, ws.route, ws.logits, ws.skp, ws.skp_bytes, ws.ctr, ms);
      prof.end(ms);
      return rd;
    }
  }
  if (mode == MOE_MODE_RESIDENT && !a->window_counts && a->decode_kernels == 0 && H % 8 == 0 && ws.skp) {
    // a small all-resident step: the whole layer in one persistent launch
    int dev = 0, sms = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const bool bf = !a->quant && decode_eligible(T, H, E, k, I, S, a->x, a->w_router, a->pool);
    const bool q8 = a->quant && decode_q8_eligible(T, H, E, k, I, S, a->x, a->w_router, a->pool, sms);
    if (bf || q8) {
      prof.begin(MOE_PROF_DECODE, ms);
      const int rd = bf ? launch_decode(a, ws.route, ws.logits, ws.skp, ws.skp_bytes, ws.ctr, ms)
                        : launch_decode_q8(a, ws.route, ws.logits, ws.skp, ws.skp_bytes, ws.ctr, ms);
      prof.end(ms);
      return rd;
    }
  }
  prof.begin(MOE_PROF_ROUTE, ms);
  // a one-chunk step: the top-k CTA may group the batch by expert itself (then no permute launch)
  const PermOut perm0{ws.count, ws.offset, ws.rows, ws.pos, ws.act_e, ws.n_act, a->dev_status};
  bool grouped = false;
  int r = route_impl(a->x, a->w_router, a->logit_offset, a->sel_bias, a->affinity != 0.f ? a->e2s : nullptr,
                     a->affinity, a->route_flags, T, H, E, k, ws.logits,
                     moe_route_scratch_bytes(T, H, E) ? ws.route : nullptr, a->ids, a->w, ms,
                     C >= T ? &perm0 : nullptr, &grouped);
  if (r != MOE_OK) return r;
  prof.end(ms);

  for (int t0 = 0; t0 < T; t0 += C) {
    const int tc = std::min(C, T - t0);
    const int n = tc * k;
    const int lmax = std::min(n, E);
    const int32_t* ids_c = a->ids + (size_t)t0 * k;
    prof.begin(MOE_PROF_PERMUTE, ms);
    if (!(grouped && t0 == 0)) {
      r = launch_permute(ids_c, n, E, ws.count, ws.offset, ws.rows, ws.pos, ws.act_e, ws.n_act, a->dev_status, ws.perm,
                         ms);
      if (r != MOE_OK) return r;
    }
    prof.end(ms);
    if (a->window_counts && (r = launch_window_add(ws.count, E, a->window_counts, ms)) != MOE_OK) return r;
    FfnArgs f{(const uint16_t*)a->x + (size_t)t0 * H, tc, H, I, k, E, ws.offset, ws.rows, nullptr, nullptr,
              (const uint16_t*)a->pool, a->e2s, (const uint16_t*)a->host_slabs, (size_t)3 * H * I, ws.hbuf, ws.y,
              a->dev_status, S, 1, ws.xp, ws.hb, nullptr, ws.skp, ws.skp_bytes};
    // tensor-core path: y travels as bf16 through the same buffer (half the bytes)
    const bool y_bf16 = !a->quant && mode != MOE_MODE_ZERO_RETURN && prefill_eligible(f, n);
    // the FFN of one expert list: bf16 slabs (stream / prefill / CUDA-core paths) or W8A8 slabs
    auto ffn = [&](const FfnArgs& fa, cudaStream_t st) {
      return a->quant ? launch_ffn_q8(fa, ws.skp, ws.skp_bytes, lmax, st, &prof) : launch_ffn(fa, lmax, st, &prof);
    };
    if (y_bf16) f.yb = (uint16_t*)ws.y;
    if (mode == MOE_MODE_RESIDENT) {
      f.list_e = ws.act_e;
      f.n_list = ws.n_act;
      f.host = nullptr;
      if ((r = ffn(f, ms)) != MOE_OK) return r;
    } else {
      prof.begin(MOE_PROF_MANAGE, ms);
      ManageWave w0;  // expert waves: the misses that find no free slot are deferred
      w0.def_e = ws.def_e;
      w0.n_def = ws.n_def;
      r = launch_manage(ids_c, n, E, S, policy, a->e2s, a->s2e, a->prio, a->stamp, ws.miss_e, ws.miss_s, ws.n_miss,
                        ws.hit_e, ws.n_hit, nullptr, stats, a->dev_status, ms, waves ? &w0 : nullptr);
      if (r != MOE_OK) return r;
      prof.end(ms);
      FfnArgs fh = f, fm = f;
      fm.pool_only = mode == MOE_MODE_GATHER;  // zero-return reads the missing experts from host memory
      fh.list_e = ws.hit_e;
      fh.n_list = ws.n_hit;
      fm.list_e = ws.miss_e;
      fm.n_list = ws.n_miss;
      if (two) {
        MOE_CUDA_TRY(cudaEventRecord(ev->fork, ms));
        MOE_CUDA_TRY(cudaStreamWaitEvent(ss, ev->fork, 0));
      }
      cudaStream_t side = two ? ss : ms;
      if (mode == MOE_MODE_GATHER) {
        const int nw = waves ? later_waves(n, E, S) : 0;
        const int wmax = std::min(S, lmax);
        const SubBatches sb = sub_batches(wmax);
        const int n_sub = sb.n;
        auto sub_len = [&](int b) { return sb.off[b + 1] - sb.off[b]; };
        // the FFN of a device-side list (slots from e2s, or from `ls` for experts already evicted)
        auto ffn_list = [&](const int32_t* le, const int32_t* ls, const int32_t* nl, int maxl) -> int {
          FfnArgs fb = fm;
          fb.list_e = le;
          fb.list_s = ls;
          fb.n_list = nl;
          return a->quant ? launch_ffn_q8(fb, ws.skp, ws.skp_bytes, maxl, ms, &prof) : launch_ffn(fb, maxl, ms, &prof);
        };
        auto gather_list = [&](const int32_t* le, const int32_t* ls, const int32_t* nl, int maxl) -> int {
          prof.begin(MOE_PROF_GATHER, side);
          const int rg = launch_gather(a->host_slabs, a->pool, slab_bytes, E, S, le, ls, nl, maxl, stats,
                                       a->dev_status, side);
          prof.end(side);
          return rg;
        };
        auto manage_wave = [&](int wv, const ManageKeep* keep) -> int {
          ManageWave bw;
          bw.n_dev = ws.n_def;
          bw.n_off = (wv - 1) * S;
          bw.sub_n = ws.sub_n;
          bw.sub = sb;
          if (keep) bw.keep = *keep;
          prof.begin(MOE_PROF_MANAGE, ms);
          const int rm = launch_manage(ws.def_e, wmax, E, S, policy, a->e2s, a->s2e, a->prio, a->stamp, ws.wl_e,
                                       ws.wl_s, ws.n_wl, nullptr, nullptr, nullptr, stats, a->dev_status, ms, &bw);
          prof.end(ms);
          return rm;
        };
        // a later wave: the next S deferred experts evict slots whose experts this step has computed
        // already; the side stream gathers its sub-batches back to back, the main stream runs each
        // sub-batch's FFN once its gather has landed
        auto later_wave = [&](int wv) -> int {
          int rw = manage_wave(wv, nullptr);
          if (rw != MOE_OK) return rw;
          if (two) {
            MOE_CUDA_TRY(cudaEventRecord(ev->fork, ms));
            MOE_CUDA_TRY(cudaStreamWaitEvent(ss, ev->fork, 0));
          }
          for (int b = 0; b < n_sub; ++b) {
            // the sub-batch's slots are its own (one manage call gave every load a different victim)
            if ((rw = gather_list(ws.wl_e + sb.off[b], ws.wl_s + sb.off[b], ws.sub_n + b, sub_len(b))) != MOE_OK)
              return rw;
            if (two) {
              MOE_CUDA_TRY(cudaEventRecord(ev->join, ss));
              MOE_CUDA_TRY(cudaStreamWaitEvent(ms, ev->join, 0));
            }
            if ((rw = ffn_list(ws.wl_e + sb.off[b], nullptr, ws.sub_n + b, sub_len(b))) != MOE_OK) return rw;
          }
          return MOE_OK;
        };
        // With a later wave and the decode stream FFN, wave 1's manage call runs before any FFN of the
        // step: the experts it evicts (hits or wave 0's loads) are computed first, sub-batch by
        // sub-batch, reading their old slots, and each sub-batch's gather follows them at once; the
        // experts that stay in place are computed while wave 1's gather runs.  The calls, and so the
        // cache state, are those of the plain order.
        const bool ahead = nw >= 1 && two && (a->quant || sk_eligible(fm));
        if (ahead) {
          // wave 0's loads go to slots the step does not need: their gather starts beside wave 1's manage
          // call (which decides, on the main stream, which slots wave 1 overwrites later)
          MOE_CUDA_TRY(cudaEventRecord(ev->fork, ms));
          MOE_CUDA_TRY(cudaStreamWaitEvent(ss, ev->fork, 0));
          if ((r = gather_list(ws.miss_e, ws.miss_s, ws.n_miss, lmax)) != MOE_OK) return r;
          MOE_CUDA_TRY(cudaEventRecord(ev->join, ss));
          const ManageKeep keep{ws.ev_e, ws.hit_e, ws.n_hit, ws.miss_e, ws.n_miss, ws.kept_e, ws.n_kept};
          if ((r = manage_wave(1, &keep)) != MOE_OK) return r;
          MOE_CUDA_TRY(cudaStreamWaitEvent(ms, ev->join, 0));  // wave 0's loads are in their slots
          for (int b = 0; b < n_sub; ++b) {
            if ((r = ffn_list(ws.ev_e + sb.off[b], ws.wl_s + sb.off[b], ws.sub_n + b, sub_len(b))) != MOE_OK)
              return r;
            MOE_CUDA_TRY(cudaEventRecord(ev->fork, ms));
            MOE_CUDA_TRY(cudaStreamWaitEvent(ss, ev->fork, 0));
            if ((r = gather_list(ws.wl_e + sb.off[b], ws.wl_s + sb.off[b], ws.sub_n + b, sub_len(b))) != MOE_OK)
              return r;
            MOE_CUDA_TRY(cudaEventRecord(ev->sub[b], ss));
          }
          if ((r = ffn_list(ws.kept_e, nullptr, ws.n_kept, lmax)) != MOE_OK) return r;
          for (int b = 0; b < n_sub; ++b) {
            MOE_CUDA_TRY(cudaStreamWaitEvent(ms, ev->sub[b], 0));
            if ((r = ffn_list(ws.wl_e + sb.off[b], nullptr, ws.sub_n + b, sub_len(b))) != MOE_OK) return r;
          }
          for (int wv = 2; wv <= nw; ++wv)
            if ((r = later_wave(wv)) != MOE_OK) return r;
        } else {
          // side: gather the misses; main: the hit experts' FFN meanwhile; then the misses.
          if ((r = gather_list(ws.miss_e, ws.miss_s, ws.n_miss, lmax)) != MOE_OK) return r;
          if (two) MOE_CUDA_TRY(cudaEventRecord(ev->join, ss));
          if ((r = ffn(fh, ms)) != MOE_OK) return r;
          if (two) MOE_CUDA_TRY(cudaStreamWaitEvent(ms, ev->join, 0));
          if ((r = ffn(fm, ms)) != MOE_OK) return r;
          for (int wv = 1; wv <= nw; ++wv)
            if ((r = later_wave(wv)) != MOE_OK) return r;
        }
      } else {
        // zero-return: resident experts from the pool on main, missing ones
        // straight from the host store on the side stream; then one add.
        if ((r = ffn(fm, side)) != MOE_OK) return r;
        if (two) MOE_CUDA_TRY(cudaEventRecord(ev->join, ss));
        if ((r = ffn(fh, ms)) != MOE_OK) return r;
        if (two) MOE_CUDA_TRY(cudaStreamWaitEvent(ms, ev->join, 0));
      }
    }
    const int split = mode == MOE_MODE_ZERO_RETURN;
    prof.begin(MOE_PROF_COMBINE, ms);
    r = launch_combine(ws.y, a->w + (size_t)t0 * k, ws.pos, ids_c, a->e2s, tc, k, H, E, split,
                       (uint16_t*)a->out + (size_t)t0 * H, split ? a->out_res + (size_t)t0 * H : nullptr,
                       split ? a->out_miss + (size_t)t0 * H : nullptr, ms, y_bf16 ? (const uint16_t*)ws.y : nullptr);
    if (r != MOE_OK) return r;
    prof.end(ms);
  }
  return MOE_OK;
}
