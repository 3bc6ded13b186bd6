// Grouped-FFN dispatch: fp32 runs on CUDA cores (ffn_simt.cu); bf16 runs on
// the tensor cores (ffn_tc.cu).
#include "common.cuh"
#include "internal.h"

namespace semmoe {

cudaError_t launch_ffn_simt(const void* x, const int32_t* offsets, const int32_t* p2e, const void* w13,
                            const void* w2, int dtype, int P, int E, int H, int I, void* y, void* ws,
                            cudaStream_t s);
int ffn_simt_take_errors(cudaStream_t s, int* bits);

int ffn_take_errors(cudaStream_t s, int* bits) { return ffn_simt_take_errors(s, bits); }

// Workspace: the SwiGLU activation h [P, I] in the activation type.
size_t ffn_ws_bytes(int P, int I, int dtype) {
  const size_t es = dtype == SEMMOE_BF16 ? 2 : 4;
  return align_up((size_t)(P > 0 ? P : 1) * I * es, 256);
}

cudaError_t launch_ffn(const void* x, const int32_t* offsets, const int32_t* p2e, const void* w13,
                       const void* w2, int dtype, int P, int E, int H, int I, void* y, void* ws,
                       cudaStream_t s) {
  return launch_ffn_simt(x, offsets, p2e, w13, w2, dtype, P, E, H, I, y, ws, s);
}

}  // namespace semmoe
