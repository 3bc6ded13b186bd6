// Shared device helpers for the semmoe kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

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

// Streaming multiprocessors of the current device.
inline int sm_count() {
  int dev = 0, n = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

}  // namespace semmoe
