// moe_expert_ffn_noalloc: the grouped expert FFN without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run
// the FFN: code that runs inside a host callback or a signal-restricted
// worker where CUDA allocation calls are not allowed, plug-ins that must not
// touch the host process's memory pool, or runtimes whose allocator is
// frozen after start-up.  This entry point takes the FFN's intermediate
// activations h from a fixed array compiled into the library instead of a
// workspace argument, and calls no allocating routine.  Inputs and outputs
// are still the caller's.
#include <mutex>

#include "internal.cuh"

namespace moe {

// h = silu(x Wg) * (x Wu) for up to this many (routing slot, column) pairs.
constexpr size_t kNoAllocScratchFloats = size_t(MOE_FFN_NOALLOC_MAX_H);

// One copy per GPU that loads the library, held until the process exits.
static __device__ __align__(256) float g_ffn_scratch[kNoAllocScratchFloats];

// Device address of g_ffn_scratch, looked up once per device.  In host code
// the name g_ffn_scratch is only a host-side stand-in, never a device
// address, so it is never passed to a kernel directly.
static float* g_scratch_addr[64] = {};
static std::mutex g_scratch_mu;

static int scratch_address(float** out) {
  int dev = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_ffn_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" int moe_expert_ffn_noalloc(const void* x, int T, int H, int I, int k, int E, const int32_t* offset,
                                      const int32_t* rows, const int32_t* list_e, const int32_t* n_list,
                                      int max_list, const void* pool, int S, const int32_t* e2s,
                                      const void* host_slabs, float* y, int32_t* dev_status, moe_stream_t stream) {
  // the argument checks of moe_expert_ffn, minus the workspace
  if (!x || !offset || !rows || !list_e || !n_list || !pool || !y) return MOE_ERR_ARG;
  if (!shape_ok(T, H, I, k, E) || max_list < 0 || S < 1 || (!e2s && S < E)) return MOE_ERR_ARG;
  if ((uintptr_t)pool % 16 || (uintptr_t)y % 16 || (uintptr_t)x % 16) return MOE_ERR_ALIGN;
  if ((size_t)T * (size_t)k * (size_t)I > kNoAllocScratchFloats) return MOE_ERR_SCRATCH_LIMIT;
  if (host_slabs) {
    if ((uintptr_t)host_slabs % 16) return MOE_ERR_ALIGN;
    const int acc = check_host_accessible(host_slabs);
    if (acc != MOE_OK) return acc;
  }
  float* h = nullptr;
  const int r = scratch_address(&h);
  if (r != MOE_OK) return r;
  // Nothing in the scratch has to start at zero: every h row the down
  // projection reads is written earlier in the same call, on the same stream.
  // Without a host store every listed expert is in the pool, so the weight
  // tiles can be streamed by tensor-map copies; slots are checked against S.
  FfnArgs a{(const uint16_t*)x, T, H, I, k, E, offset, rows, list_e, n_list, (const uint16_t*)pool, e2s,
            (const uint16_t*)host_slabs, (size_t)3 * H * I, h, y, dev_status, S, host_slabs == nullptr};
  return launch_ffn(a, max_list < E ? max_list : E, (cudaStream_t)stream);
}
