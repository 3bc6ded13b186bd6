// Un-permute + gate-weighted combine: the single-device form of the
// Shuffled-Allgather, which brings the expert results back to the original
// token order (Semantic Parallelism (de) §2 B, (ja) §2.2 B):
//   out[t] = y_shared[t] + sum_{j<k_t} w[t,j] * y_perm[pair_to_sorted[t*k_max+j]]
// summed in that order in fp32.
#include "common.cuh"
#include "internal.h"

namespace semmoe {
namespace {

__device__ int g_err;
__device__ __forceinline__ void flag(int bit) { atomicOr(&g_err, bit); }

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void load(const float* p, float* v) {
    float4 a = *reinterpret_cast<const float4*>(p);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  }
  __device__ static void store(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
  __device__ static void unpack(const uint4& a, float* v) {
    v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
    v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
  }
};
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const __nv_bfloat16* p, float* v) { unpack(*reinterpret_cast<const uint4*>(p), v); }
  __device__ static void unpack(const uint4& a, float* v) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&a);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x; v[2 * i + 1] = f.y;
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float* v) {
    uint4 a;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&a);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = a;
  }
};

// One warp per (token, column pass): a pass covers 32 lanes x CH 16-byte
// chunks of the row.  The token's (sorted row, gate) pairs sit in lanes
// 0..k_max-1 and are broadcast with shuffles; the rows are fetched JB slots at
// a time with every load of a batch issued before the first add (padding slots
// load nothing and leave the sum untouched), so each lane keeps JB * CH
// 16-byte loads in flight.  CH = 2, JB = 3 at four CTAs per SM measured best of
// the forms tried (CH x JB x CTAs per SM: 2x2x4, 1x4x4, 1x6x4, 2x3x4, 1x8x3,
// 2x4x3, 4x4x2): 67% / 89% / 86% of the HBM copy bandwidth on the DeepSeek /
// Qwen3 / MoE-Prism shapes.  The sum runs y_shared first, then the slots in
// order, with fmaf.
template <typename T, int CH, int JB>
__global__ void __launch_bounds__(kThreads, 4)
combine_kernel(const T* __restrict__ y_perm, const int32_t* __restrict__ pair_to_sorted,
               const float* __restrict__ topk_w, const T* __restrict__ y_shared, int T_, int H, int k_max,
               int P, T* __restrict__ out) {
  using V = Vec16<T>;
  pdl_trigger();
  pdl_wait();  // y_perm (the grouped FFN before it)
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int kk = k_max < 32 ? k_max : 32;
  const int pass_elems = 32 * V::N * CH;
  const int n_pass = (H + pass_elems - 1) / pass_elems;
  const long long units = (long long)T_ * n_pass;
  for (long long u = (long long)blockIdx.x * kWarps + warp; u < units; u += (long long)gridDim.x * kWarps) {
    const int t = (int)(u / n_pass);
    const int base = (int)(u - (long long)t * n_pass) * pass_elems;
    const int32_t* q_row = pair_to_sorted + (size_t)t * k_max;
    const float* w_row = topk_w + (size_t)t * k_max;
    int q_l = -1;
    float w_l = 0.f;
    if (lane < kk) {
      q_l = q_row[lane];
      w_l = w_row[lane];
      if (q_l >= P) { flag(SEMMOE_DEVERR_PAIRS); q_l = -1; }
    }
    float acc[CH][V::N];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int col = base + (c * 32 + lane) * V::N;
      if (y_shared != nullptr && col < H) {
        V::load(y_shared + (size_t)t * H + col, acc[c]);
      } else {
#pragma unroll
        for (int i = 0; i < V::N; ++i) acc[c][i] = 0.f;
      }
    }
    for (int j0 = 0; j0 < kk; j0 += JB) {
      uint4 raw[JB][CH];
      float wj[JB];
      bool ok[JB];
#pragma unroll
      for (int b = 0; b < JB; ++b) {
        const int q = __shfl_sync(0xffffffffu, q_l, (j0 + b) & 31);
        wj[b] = __shfl_sync(0xffffffffu, w_l, (j0 + b) & 31);
        ok[b] = j0 + b < kk && q >= 0;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int col = base + (c * 32 + lane) * V::N;
          raw[b][c] = (ok[b] && col < H) ? *reinterpret_cast<const uint4*>(y_perm + (size_t)q * H + col)
                                          : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int b = 0; b < JB; ++b) {
        if (!ok[b]) continue;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          float v[V::N];
          V::unpack(raw[b][c], v);
#pragma unroll
          for (int i = 0; i < V::N; ++i) acc[c][i] = fmaf(wj[b], v[i], acc[c][i]);
        }
      }
    }
    for (int j = 32; j < k_max; ++j) {  // budgets above 32 experts: read the slot directly
      const int q = q_row[j];
      if (q < 0) continue;
      if (q >= P) { flag(SEMMOE_DEVERR_PAIRS); continue; }
      const float w = w_row[j];
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int col = base + (c * 32 + lane) * V::N;
        if (col < H) {
          float v[V::N];
          V::load(y_perm + (size_t)q * H + col, v);
#pragma unroll
          for (int i = 0; i < V::N; ++i) acc[c][i] = fmaf(w, v[i], acc[c][i]);
        }
      }
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int col = base + (c * 32 + lane) * V::N;
      if (col < H) V::store(out + (size_t)t * H + col, acc[c]);
    }
  }
}

// out[t] = y_shared[t] + acc[t] in bf16 (y_shared may be null): the last step of
// the combine folded into GEMM2.  Eight elements per thread.
__global__ void __launch_bounds__(kThreads)
combine_finish_kernel(const float4* __restrict__ acc, const uint4* __restrict__ y_shared, long long n8,
                      uint4* __restrict__ out) {
  pdl_trigger();
  pdl_wait();  // acc (the grouped FFN before it)
  for (long long i = blockIdx.x * (long long)kThreads + threadIdx.x; i < n8; i += (long long)gridDim.x * kThreads) {
    const float4 a = acc[2 * i], b = acc[2 * i + 1];
    float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    if (y_shared != nullptr) {
      float sv[8];
      Vec16<__nv_bfloat16>::unpack(y_shared[i], sv);
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = sv[k] + v[k];
    }
    uint4 o;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
    out[i] = o;
  }
}

}  // namespace

cudaError_t launch_combine_finish(const float* acc, const void* y_shared, int T, int H, void* out, cudaStream_t s) {
  const long long n8 = (long long)T * H / 8;
  if (n8 == 0) return cudaSuccess;
  long long blocks = (n8 + kThreads - 1) / kThreads;
  const long long cap = 8LL * sm_count();
  if (blocks > cap) blocks = cap;
  cudaError_t e = launch_kernel(combine_finish_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, s, 1, true,
                                reinterpret_cast<const float4*>(acc), static_cast<const uint4*>(y_shared), n8,
                                static_cast<uint4*>(out));
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaGetLastError();
}

int combine_take_errors(cudaStream_t s, int* bits) { return take_error_word(g_err, s, bits); }

cudaError_t launch_combine(const void* y_perm, const int32_t* pair_to_sorted, const float* topk_w,
                           const void* y_shared, int dtype, int T, int H, int k_max, int P, void* out,
                           cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  constexpr int kCH = 2, kJB = 3;
  const int vec = dtype == SEMMOE_BF16 ? 8 : 4;
  const long long units = (long long)T * ((H + 32 * vec * kCH - 1) / (32 * vec * kCH));
  long long blocks = (units + kWarps - 1) / kWarps;
  const long long cap = 8LL * sm_count();
  if (blocks > cap) blocks = cap;
  cudaError_t e;
  if (dtype == SEMMOE_BF16)
    e = launch_kernel(combine_kernel<__nv_bfloat16, kCH, kJB>, dim3((unsigned)blocks), dim3(kThreads), 0, s, 1, true,
                      static_cast<const __nv_bfloat16*>(y_perm), pair_to_sorted, topk_w,
                      static_cast<const __nv_bfloat16*>(y_shared), T, H, k_max, P, static_cast<__nv_bfloat16*>(out));
  else
    e = launch_kernel(combine_kernel<float, kCH, kJB>, dim3((unsigned)blocks), dim3(kThreads), 0, s, 1, true,
                      static_cast<const float*>(y_perm), pair_to_sorted, topk_w, static_cast<const float*>(y_shared),
                      T, H, k_max, P, static_cast<float*>(out));
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace semmoe
