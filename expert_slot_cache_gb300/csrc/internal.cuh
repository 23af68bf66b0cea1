// Internal launchers shared by the translation units of the library.
#pragma once

#include "common.cuh"
#include "perm_small.cuh"

namespace moe {

struct FfnArgs {
  const uint16_t* x;      // device bf16 [T][H]
  int T, H, I, k, E;
  const int32_t* offset;  // [E+1]
  const int32_t* rows;    // [T*k]
  const int32_t* list_e;  // experts to process
  const int32_t* n_list;  // device count
  const uint16_t* pool;   // slot pool
  const int32_t* e2s;     // NULL = expert e in slot e
  const uint16_t* host;   // host store (zero-return second pass) or NULL
  size_t slab_elems;
  float* hbuf;            // [T*k][I]
  float* y;               // [T*k][H]
  int32_t* status;
  int S;                  // slots in pool (0 = unknown)
  int pool_only;          // every listed expert is in the pool (e2s[e] >= 0 or e2s == NULL)
  uint16_t* xp;           // bf16 [T*k][H] grouped copy of x (tensor-core path), or NULL
  uint16_t* hb;           // bf16 [T*k][I] h for the tensor-core path, or NULL
  uint16_t* yb;           // tensor-core path: write y as bf16 [T*k][H] here instead of fp32 y (or NULL)
  float* skp;             // partial sums of the decode stream path (sk_part_bytes), or NULL
  size_t skp_bytes;
  const int32_t* list_s;  // slot of each listed expert (stream paths), or NULL: the slot comes from e2s
};

// Records (start, end) event pairs around kernel launches when tracing is on.
// Inside a stream capture the records become graph nodes (external records),
// so a replayed graph still timestamps every launch.
struct Prof {
  moe_prof* p = nullptr;
  int cur = -1;
  static void record(void* ev, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(s, &cs);
    if (cs == cudaStreamCaptureStatusActive)
      cudaEventRecordWithFlags((cudaEvent_t)ev, s, cudaEventRecordExternal);
    else
      cudaEventRecord((cudaEvent_t)ev, s);
  }
  void begin(int tag, cudaStream_t s) {
    cur = -1;
    if (!p || !p->events || p->used + 2 > p->capacity) return;
    cur = p->used;
    record(p->events[cur], s);
    if (p->tags) p->tags[cur / 2] = tag;
  }
  void end(cudaStream_t s) {
    if (cur < 0) return;
    record(p->events[cur + 1], s);
    p->used = cur + 2;
    cur = -1;
  }
};

// Shapes every FFN entry point accepts (H % 64, I % 32, 1 <= k <= kMaxK, k <= E <= kMaxE).
inline bool shape_ok(int T, int H, int I, int k, int E) {
  return T >= 1 && H >= 64 && H % 64 == 0 && I >= 32 && I % 32 == 0 && k >= 1 && k <= kMaxK && E >= k &&
         E <= kMaxE;
}

int launch_ffn(const FfnArgs& a, int max_list, cudaStream_t stream, Prof* prof = nullptr);
bool prefill_eligible(const FfnArgs& a, int n);
int launch_gather_rows(const uint16_t* x, const int32_t* rows, int n, int H, int k, uint16_t* xp, int sms,
                       cudaStream_t stream);
size_t sk_part_bytes(int n, int H, int I);
// Gate/up parts [jg][n][2I] and down parts [jd][n][H] (fp32) inside a buffer of sk_part_bytes(n, H, I).
bool sk_part_layout(int n, int H, int I, float* skp, size_t skp_bytes, float** gpart, float** ypart, int* jg,
                    int* jd);
size_t q8_slab_bytes_h(int H, int I);
size_t q8_ws_bytes(int n, int H, int I);
int launch_ffn_q8(const FfnArgs& a, void* ws, size_t ws_bytes, int max_list, cudaStream_t stream, Prof* prof);
bool sk_eligible(const FfnArgs& a);
int launch_ffn_sk(const FfnArgs& a, int max_list, cudaStream_t stream, Prof* prof);
size_t prefill_extra_bytes(int n, int H, int I);
int launch_prefill(const FfnArgs& a, int n, int max_list, cudaStream_t stream, Prof* prof);
int launch_combine(const float* y, const float* w, const int32_t* pos, const int32_t* ids, const int32_t* e2s, int T,
                   int k, int H, int E, int split, void* out, float* out_res, float* out_miss, cudaStream_t stream,
                   const uint16_t* yb = nullptr);
// What a later wave's manage call reports for scheduling the FFN around its evictions:
//   ev_e[r]        the expert the r-th load evicted from its slot (-1: the slot was empty)
//   kept_e/n_kept  the experts of the lists in0 (n_in0) and in1 (n_in1) that the call did not evict,
//                  ascending: with the step's hits and first loads as the lists, the experts that
//                  stay in place
struct ManageKeep {
  int32_t* ev_e = nullptr;
  const int32_t *in0 = nullptr, *n_in0 = nullptr, *in1 = nullptr, *n_in1 = nullptr;
  int32_t *kept_e = nullptr, *n_kept = nullptr;
};

// Expert-wave options of one manage call: wave 0 defers the misses that find no
// victim (def_e, n_def); a later wave manages ids[n_off .. n_off + m) with
// m = clamp(*n_dev - n_off, 0, n) read on the device (no call when m = 0).
// Sub-batches of a wave's loads (list positions [off[b], off[b+1]) for b < n).
constexpr int kMaxSubBatches = 4;
struct SubBatches {
  int off[kMaxSubBatches + 1] = {};
  int n = 0;
};
struct ManageWave {
  int32_t* def_e = nullptr;
  int32_t* n_def = nullptr;
  const int32_t* n_dev = nullptr;
  int n_off = 0;
  int32_t* sub_n = nullptr;  // sub_n[b] = clamp(n_miss - sub.off[b], 0, sub.off[b+1] - sub.off[b]) for b < sub.n
  SubBatches sub;
  ManageKeep keep;
};
int launch_manage(const int32_t* ids, int n, int E, int S, int policy, int32_t* e2s, int32_t* s2e, uint32_t* prio,
                  uint32_t* stamp, int32_t* miss_e, int32_t* miss_s, int32_t* n_miss, int32_t* hit_e,
                  int32_t* n_hit, int32_t* sid, int64_t* stats, int32_t* dev_status, cudaStream_t stream,
                  const ManageWave* wave = nullptr);
int launch_gather(const void* host_slabs, void* pool, size_t slab_bytes, int E, int S, const int32_t* miss_e,
                  const int32_t* miss_s, const int32_t* n_miss, int max_miss, int64_t* stats, int32_t* dev_status,
                  cudaStream_t stream);
int check_host_accessible(const void* p);
int launch_window_add(const int32_t* count, int E, int32_t* counts, cudaStream_t stream);
// The persistent decode kernel (all-resident small batches, one cooperative launch).
bool decode_eligible(int T, int H, int E, int k, int I, int S, const void* x, const void* wr, const void* pool);
size_t decode_ctr_ints(int E);
int launch_decode(const moe_layer_args* la, float* lpart, float* logits, float* skp, size_t skp_bytes, int32_t* ctr,
                  cudaStream_t stream);
// The same kernel for a small expert-cache step (GATHER, T*k <= S, LRU / LFU): manage, the gather of the
// misses and the weight streams in the one launch; the cache state is updated in place.
bool decode_gather_eligible(int T, int H, int E, int k, int I, int S, int policy, const void* x, const void* wr,
                            const void* pool, const void* host, int sms);
int launch_decode_gather(const moe_layer_args* la, float* lpart, float* logits, float* skp, size_t skp_bytes,
                         int32_t* ctr, cudaStream_t stream);
// Its W8A8 counterpart (decode_q8.cu): CUDA-core weight streams; the step's integer sums meet in
// accumulators of T*k*(2I + H) int32 (+ T*k row scales) at the start of `ws`.
bool decode_q8_eligible(int T, int H, int E, int k, int I, int S, const void* x, const void* wr, const void* pool,
                        int sms);
size_t decode_q8_ws_bytes(int T, int k, int H, int I);
int launch_decode_q8(const moe_layer_args* la, float* lpart, float* logits, void* ws, size_t ws_bytes, int32_t* ctr,
                     cudaStream_t stream);
// Its expert-cache step (GATHER, T*k <= S, LRU / LFU): manage, the copy of the misses (codes and scales)
// and the streams in the one launch.
bool decode_q8_gather_eligible(int T, int H, int E, int k, int I, int S, int policy, const void* x, const void* wr,
                               const void* pool, const void* host, int sms);
int launch_decode_q8_gather(const moe_layer_args* la, float* lpart, float* logits, void* ws, size_t ws_bytes,
                            int32_t* ctr, cudaStream_t stream);
int route_impl(const void* x, const void* w_router, const float* logit_offset, const float* sel_bias,
               const int32_t* e2s, float affinity, int rflags, int T, int H, int E, int k, float* logits,
               float* scratch, int32_t* ids, float* w, cudaStream_t stream, const PermOut* perm, bool* fused);
int launch_permute(const int32_t* ids, int n, int E, int32_t* count, int32_t* offset, int32_t* rows, int32_t* pos,
                   int32_t* act_e, int32_t* n_act, int32_t* dev_status, int32_t* scratch, cudaStream_t s);

}  // namespace moe
