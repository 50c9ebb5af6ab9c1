// Device helpers shared by the library's kernels.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <stdlib.h>
#include <atomic>
#include <utility>
#include "internal.h"

namespace s1 {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum for blockDim.x a multiple of 32 (<= 1024). `red` holds 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = (lane < nw) ? red[lane] : 0.f;
  return warp_sum(t);
}

__device__ __forceinline__ float bf2f(bf16 x) { return __bfloat162float(x); }
__device__ __forceinline__ bf16 f2bf(float x) { return __float2bfloat16_rn(x); }
__device__ __forceinline__ float h2f(f16 x) { return __half2float(x); }
__device__ __forceinline__ f16 f2h(float x) { return __float2half_rn(x); }

__device__ __forceinline__ float silu_f(float g) { return g / (1.f + __expf(-g)); }

// Programmatic dependent launch: lets the next kernel in the stream (launched with the
// programmatic-serialisation attribute) start its independent prologue now; it still waits
// for this grid's completion before it touches data this grid produces.
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Waits until the preceding grid in the stream has completed and its writes are visible (a
// no-op for kernels launched without the attribute).
__device__ __forceinline__ void wait_prerequisites() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Returns a CUDA error from the enclosing launcher.
#define CK_RET(x)                               \
  do {                                          \
    cudaError_t e_ = (x);                       \
    if (e_ != cudaSuccess) return e_;           \
  } while (0)

// Models being profiled (their per-launch CUDA events must not absorb an early-launched kernel's
// wait for its predecessor, so programmatic dependent launch is off while any model profiles).
inline std::atomic<int>& pdl_suppressed() {
  static std::atomic<int> n{0};
  return n;
}
// Programmatic dependent launch is on unless S1_PDL=0 (a measurement override) or a model
// is being profiled.
inline bool pdl_enabled() {
  static const bool on = !(getenv("S1_PDL") && getenv("S1_PDL")[0] == '0');
  return on && pdl_suppressed().load(std::memory_order_relaxed) == 0;
}

// Launch with the programmatic-serialisation attribute: the kernel may start while its
// predecessor in the stream finishes. Every kernel launched this way calls wait_prerequisites()
// before its first access to data an earlier kernel wrote, in every CTA and before any early
// return, so the completion of any kernel still implies the completion of all earlier ones.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace s1
