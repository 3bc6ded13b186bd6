// Grouped-FFN dispatch: bf16 runs on the tensor cores (ffn_tc.cu); fp32 runs
// on CUDA cores (ffn_simt.cu).  The kernel depends only on the dtype and, for
// the tensor-core forms, on the shapes, unless the caller pins a form
// (semmoe_grouped_ffn_form, for tests that compare the forms bit for bit).
#include "common.cuh"
#include "internal.h"

namespace semmoe {

cudaError_t launch_ffn_simt(const void* x, const int32_t* offsets, const int32_t* p2e, const void* w13,
                            const void* w2, int dtype, int P, int E, int H, int I, void* y, void* ws,
                            const int32_t* gather, int gather_div, int T_x, cudaStream_t s);
cudaError_t launch_ffn_tc(const void* x, const int32_t* offsets, const int32_t* p2e, const void* w13,
                          const void* w2, int P, int E, int H, int I, void* y, void* ws, const int32_t* gather,
                          int gather_div, int T_x, int form1, int form2, cudaStream_t s,
                          const int32_t* sorted_to_pair = nullptr, const float* topk_w = nullptr, int k_max = 1,
                          int T_acc = 0, float* acc = nullptr, int fused_stall = 0, bool dependent = true);
int ffn_simt_take_errors(cudaStream_t s, int* bits);
int ffn_tc_take_errors(cudaStream_t s, int* bits);

int ffn_take_errors(cudaStream_t s, int* bits) {
  if (ffn_simt_take_errors(s, bits)) return -1;
  return ffn_tc_take_errors(s, bits);
}

// Workspace: the SwiGLU activation h [P, I] in the activation type.
size_t ffn_ws_bytes(int P, int I, int dtype) {
  const size_t es = dtype == SEMMOE_BF16 ? 2 : 4;
  // h [P, I], then one readiness counter per m-tile for the one-launch form
  // (at most ceil(P / 128) + 256 m-tiles: one partial tile per group)
  return align_up((size_t)(P > 0 ? P : 1) * I * es, 256) + ffn_ready_bytes(P);
}

cudaError_t launch_ffn(const void* x, const int32_t* offsets, const int32_t* p2e, const void* w13,
                       const void* w2, int dtype, int P, int E, int H, int I, void* y, void* ws,
                       const int32_t* gather, int gather_div, int T_x, cudaStream_t s, int form1, int form2,
                       bool dependent) {
  if (dtype == SEMMOE_BF16 && form1 != SEMMOE_FORM_CUDA_CORE)
    return launch_ffn_tc(x, offsets, p2e, w13, w2, P, E, H, I, y, ws, gather, gather_div, T_x, form1, form2, s,
                         nullptr, nullptr, 1, 0, nullptr, 0, dependent);
  return launch_ffn_simt(x, offsets, p2e, w13, w2, dtype, P, E, H, I, y, ws, gather, gather_div, T_x, s);
}

cudaError_t launch_ffn_combine(const void* x, bool gathered, const int32_t* sorted_to_pair, int k_max, int T,
                               const int32_t* offsets, const int32_t* p2e, const void* w13, const void* w2,
                               const float* topk_w, int P, int E, int H, int I, float* acc, void* ws,
                               cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(acc, 0, (size_t)T * H * sizeof(float), s);
  if (e != cudaSuccess || P == 0) return e;
  return launch_ffn_tc(x, offsets, p2e, w13, w2, P, E, H, I, nullptr, ws, gathered ? sorted_to_pair : nullptr, k_max,
                       T, SEMMOE_FORM_DEFAULT, SEMMOE_FORM_DEFAULT, s, sorted_to_pair, topk_w, k_max, T, acc);
}

// One group of P rows through the one-launch FFN with GEMM2's readiness waits
// made unreachable: every GEMM2 tile's wait runs out after its bound, sets the
// timeout bit and stops its CTA (bf16 only; the failure-path self-test).
cudaError_t launch_selftest_fused_ready_wait(const void* x, const void* w13, const void* w2, int P, int H, int I,
                                             void* y, void* ws, cudaStream_t s) {
  return launch_ffn_tc(x, nullptr, nullptr, w13, w2, P, 1, H, I, y, ws, nullptr, 1, 0, SEMMOE_FORM_FUSED,
                       SEMMOE_FORM_FUSED, s, nullptr, nullptr, 1, 0, nullptr, 1);
}

}  // namespace semmoe
