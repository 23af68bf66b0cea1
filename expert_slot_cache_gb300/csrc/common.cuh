// Device helpers shared by the slot-cache kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moeslot.h"

#define MOE_FULL_MASK 0xffffffffu

namespace moe {

constexpr int kMaxE = 1024;
constexpr int kMaxK = 16;

// bf16 bit pattern -> fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t v) { return __uint_as_float(uint32_t(v) << 16); }

// fp32 -> bf16, round to nearest even.
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ void set_status(int32_t* st, int code) {
  if (st) *(volatile int32_t*)st = code;  // last writer wins; any nonzero value flags the call
}

// 16-byte read-only load through the non-coherent path, no L1 allocation.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Block-wide exclusive scan of one int per thread (blockDim.x multiple of 32,
// <= 1024).  `tmp` holds >= 33 ints of shared memory.  Returns the exclusive
// prefix; *total receives the block sum.  All threads must call it.
__device__ __forceinline__ int block_exclusive_scan(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int o = __shfl_up_sync(MOE_FULL_MASK, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? tmp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int o = __shfl_up_sync(MOE_FULL_MASK, wi, d);
      if (lane >= d) wi += o;
    }
    if (lane < nw) tmp[lane] = wi - w;
    if (lane == 31) tmp[32] = wi;
  }
  __syncthreads();
  int res = tmp[warp] + incl - v;
  *total = tmp[32];
  __syncthreads();
  return res;
}

// Programmatic dependent launch: let the next kernel in the stream start /
// wait until the previous kernel has completed and its writes are visible.
// A kernel launched as a programmatic dependent (launch_pdl) waits before it
// reads the previous kernel's output and before it exits, so completion stays
// ordered along the stream; in a kernel launched plainly the wait is a no-op.
// A kernel that triggers before its own wait lets its dependent start before
// the kernel before it has completed: it may do so only when that dependent
// reads nothing of earlier kernels before its own wait.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kernel` as a programmatic dependent of the kernel before it in `s`.
template <typename K, typename... Args>
inline cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Raise a kernel's dynamic shared memory limit once per device.
template <typename F>
inline cudaError_t ensure_smem(F* func, int bytes, bool* done /* [64] per device */) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

}  // namespace moe

// Host-side launch helpers
#define MOE_CUDA_TRY(expr)                      \
  do {                                          \
    cudaError_t _e = (expr);                    \
    if (_e != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

#define MOE_LAUNCH_CHECK() MOE_CUDA_TRY(cudaGetLastError())
