// Shared device helpers for the semmoe kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "semmoe.h"

namespace semmoe {

// ---------------------------------------------------------------------------
// element types
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// silu(z) = z / (1 + exp(-z)), fp32.
__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch.  The kernels of the layer follow one another
// on a stream; each launched as a dependent may start -- and run its setup
// (barriers, tensor memory, tensor-map prefetches: nothing in global memory) --
// once every CTA of the kernel before it has run pdl_trigger, and it waits in
// pdl_wait until that kernel has completed and its writes are visible.  So each
// kernel calls pdl_trigger at its start and, when it can be launched as a
// dependent (launch_kernel), pdl_wait before its first global load or store (a kernel that waits
// completes only after the kernel before it, so the guarantee chains).  Both
// are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Read and clear one translation unit's device error word.
template <typename Sym>
inline int take_error_word(const Sym& sym, cudaStream_t s, int* bits) {
  int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, sym, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess) return -1;
  if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
  if (v) {
    int z = 0;
    if (cudaMemcpyToSymbolAsync(sym, &z, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess) return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
  }
  *bits |= v;
  return 0;
}

// ---------------------------------------------------------------------------
// host helpers
// ---------------------------------------------------------------------------
__host__ __device__ inline constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Raise `kernel`'s dynamic shared-memory limit to `bytes` once per device;
// `done` is a per-call-site bit mask of devices already set.
template <typename K>
inline cudaError_t ensure_smem_limit(K kernel, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_relaxed);
  return e;
}
inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Launch `kern` on `s` with an optional cluster size; dependent = true makes it
// a programmatic dependent of the kernel before it on `s`
// (cudaLaunchAttributeProgrammaticStreamSerialization; see pdl_wait).  Its CTAs
// may then occupy SMs while they wait, so only the layer's chain of steps on the
// caller's stream launches this way, not work beside it on another stream.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 unsigned cluster, bool dependent, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (dependent) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Streaming multiprocessors of the current device.
inline int sm_count() {
  int dev = 0, n = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

}  // namespace semmoe
