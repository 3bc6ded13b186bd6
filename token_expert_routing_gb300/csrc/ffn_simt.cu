// Grouped SwiGLU expert FFN on CUDA cores (fp32 accumulation).
//
// The experts' computation (Semantic Parallelism (ko) §1; an expert is a set
// of intermediate neurons, MoE-Prism (ko) §2 A), as a SwiGLU FFN per expert
// over that expert's contiguous block of sorted rows:
//   GEMM1 + SwiGLU: h = silu(x W1_e^T) * (x W3_e^T)   (w13_e = [W1_e; W3_e])
//   GEMM2:          y = h W2_e^T
// This file is the fp32 path (and the reference-speed path for bf16); the bf16
// tensor-core path lives in ffn_tc.cu.
#include "common.cuh"
#include "internal.h"
#include "ffn_common.cuh"

namespace semmoe {
namespace {

__device__ int g_err;

constexpr int BM = 64, BN = 64, BK = 16, kThreads = 256;

// C[rows of group g, n] = epilogue(sum_k A[row, k] * W_e[n, k]) for the group's
// expert e; with GLU, W_e's rows n (gate) and n + glu_off (up) are both used.
template <typename T, bool GLU>
__global__ void __launch_bounds__(kThreads)
ffn_simt_kernel(const T* __restrict__ A, const int32_t* __restrict__ offsets,
                const int32_t* __restrict__ phys_to_expert, int n_groups, int P, const T* __restrict__ W,
                long long w_stride, int N, int K, int glu_off, int E, const int32_t* __restrict__ gather,
                int gather_div, int gather_rows, T* __restrict__ C) {
  __shared__ float As[BK][BM];
  __shared__ float Bg[BK][BN];
  __shared__ float Bu[GLU ? BK : 1][GLU ? BN : 1];
  __shared__ int scan[kThreads];
  __shared__ GroupTile gt_s;
  __shared__ int src_row[BM];  // A row of each tile row (sorted row, or gathered x row)

  const GroupTile gt =
      group_tile_block(offsets, phys_to_expert, n_groups, P, E, BM, blockIdx.x, scan, &gt_s, &g_err);
  if (gt.group < 0) return;
  const int row0 = gt.row0, rows = gt.rows, e = gt.expert;
  const int n0 = blockIdx.y * BN;
  const T* We = W + (long long)e * w_stride;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  for (int m = threadIdx.x; m < BM; m += kThreads) {
    int r = row0 + m;
    if (gather != nullptr) {
      r = 0;
      if (m < rows) {
        const int p = gather[row0 + m];
        r = p >= 0 ? p / gather_div : -1;
        if (r < 0 || r >= gather_rows) {
          atomicOr(&g_err, SEMMOE_DEVERR_PAIRS);
          r = 0;
        }
      }
    }
    src_row[m] = r;
  }
  __syncthreads();

  float acc[4][4] = {}, accu[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int i = threadIdx.x; i < BM * BK; i += kThreads) {
      int m = i / BK, k = i % BK;
      As[k][m] = (m < rows && k0 + k < K) ? to_f32(A[(long long)src_row[m] * K + k0 + k]) : 0.f;
    }
    for (int i = threadIdx.x; i < BN * BK; i += kThreads) {
      int n = i / BK, k = i % BK;
      bool ok = n0 + n < N && k0 + k < K;
      Bg[k][n] = ok ? to_f32(We[(long long)(n0 + n) * K + k0 + k]) : 0.f;
      if (GLU) Bu[k][n] = ok ? to_f32(We[(long long)(glu_off + n0 + n) * K + k0 + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      float a[4], b[4], u[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[k][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b[j] = Bg[k][tx + 16 * j];
        if (GLU) u[j] = Bu[k][tx + 16 * j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          if (GLU) accu[i][j] = fmaf(a[i], u[j], accu[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int m = ty + 16 * i;
    if (m >= rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int n = n0 + tx + 16 * j;
      if (n >= N) continue;
      float v = GLU ? silu_f32(acc[i][j]) * accu[i][j] : acc[i][j];
      C[(long long)(row0 + m) * N + n] = from_f32<T>(v);
    }
  }
}

template <typename T>
cudaError_t run_simt(const void* x, const int32_t* offsets, const int32_t* p2e, const void* w13, const void* w2,
                     int P, int E, int H, int I, void* y, void* ws, const int32_t* gather, int gather_div, int T_x,
                     cudaStream_t s) {
  const int n_groups = offsets ? E : 1;
  const int max_mtiles = (P + BM - 1) / BM + n_groups;
  T* h = static_cast<T*>(ws);
  dim3 g1(max_mtiles, (I + BN - 1) / BN);
  ffn_simt_kernel<T, true><<<g1, kThreads, 0, s>>>(static_cast<const T*>(x), offsets, p2e, n_groups, P,
                                                   static_cast<const T*>(w13), 2LL * I * H, I, H, I, E, gather,
                                                   gather_div, T_x, h);
  count_launches(1);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  dim3 g2(max_mtiles, (H + BN - 1) / BN);
  ffn_simt_kernel<T, false><<<g2, kThreads, 0, s>>>(h, offsets, p2e, n_groups, P, static_cast<const T*>(w2),
                                                    (long long)H * I, H, I, 0, E, nullptr, 1, 0,
                                                    static_cast<T*>(y));
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

int ffn_simt_take_errors(cudaStream_t s, int* bits) { return take_error_word(g_err, s, bits); }

cudaError_t launch_ffn_simt(const void* x, const int32_t* offsets, const int32_t* p2e, const void* w13,
                            const void* w2, int dtype, int P, int E, int H, int I, void* y, void* ws,
                            const int32_t* gather, int gather_div, int T_x, cudaStream_t s) {
  if (P == 0) return cudaSuccess;
  if (dtype == SEMMOE_BF16)
    return run_simt<__nv_bfloat16>(x, offsets, p2e, w13, w2, P, E, H, I, y, ws, gather, gather_div, T_x, s);
  return run_simt<float>(x, offsets, p2e, w13, w2, P, E, H, I, y, ws, gather, gather_div, T_x, s);
}

}  // namespace semmoe
