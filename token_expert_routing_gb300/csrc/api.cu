// C ABI of the semmoe library: host-side argument validation, error
// reporting, and the launch of each step's kernels.  See include/semmoe.h.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <string>

#include "common.cuh"
#include "internal.h"

namespace {

thread_local std::string g_msg;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_msg = buf;
  return code;
}

int cuda_status(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return SEMMOE_OK;
  return fail(SEMMOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool valid_dtype(int d) { return d == SEMMOE_F32 || d == SEMMOE_BF16; }
// Router weights may also come as the split of an fp32 weight, for bf16
// activations with 16-byte rows (the tensor-core router).
bool valid_router_dtype(int w, int x, int H) {
  return valid_dtype(w) || (w == SEMMOE_F32_SPLIT && x == SEMMOE_BF16 && H % 8 == 0);
}
size_t elem_size(int d) { return d == SEMMOE_BF16 ? 2 : 4; }

// The kernels are built for sm_103a only.
int require_sm103(const char* fn) {
  int dev = 0, major = 0, minor = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) return cuda_status(e, fn);
  if (major != 10 || minor != 3)
    return fail(SEMMOE_ERR_UNSUPPORTED, "%s: built for sm_103a, device is sm_%d%d", fn, major, minor);
  return SEMMOE_OK;
}

#define REQUIRE(cond, ...)                                              \
  do {                                                                  \
    if (!(cond)) return fail(SEMMOE_ERR_INVALID_ARG, __VA_ARGS__);      \
  } while (0)

#define CHECK_DEVICE(fn)                   \
  do {                                     \
    int _rc = require_sm103(fn);           \
    if (_rc != SEMMOE_OK) return _rc;      \
  } while (0)

std::atomic<unsigned long long> g_launches{0};

}  // namespace

void semmoe::count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

using namespace semmoe;

extern "C" {

const char* semmoe_last_error(void) { return g_msg.c_str(); }

int semmoe_version(void) { return 100; }

unsigned long long semmoe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int semmoe_check_errors(void* stream, int* bits) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_status(e, "semmoe_check_errors");
  int b = 0;
  if (route_take_errors(s, &b) || permute_take_errors(s, &b) || ffn_take_errors(s, &b) ||
      combine_take_errors(s, &b) || schedule_take_errors(s, &b) || selftest_take_errors(s, &b))
    return cuda_status(cudaGetLastError(), "semmoe_check_errors: reading the device error word");
  if (bits != nullptr) *bits = b;
  if (b & SEMMOE_DEVERR_TIMEOUT) return fail(SEMMOE_ERR_DEVICE_TIMEOUT, "a bounded in-kernel wait ran out (bits 0x%x)", b);
  if (b) return fail(SEMMOE_ERR_DEVICE_CHECK, "kernels saw invalid data (device error bits 0x%x)", b);
  return SEMMOE_OK;
}

size_t semmoe_route_workspace_size(int T, int H, int E, int x_dtype, int w_dtype) {
  if (T < 0 || H < 1 || E < 1 || !valid_dtype(x_dtype) || !valid_router_dtype(w_dtype, x_dtype, H)) return 0;
  const size_t b = route_ws_bytes(T, H, E, x_dtype, w_dtype);
  return b > 0 ? b : 256;
}

size_t semmoe_pair_counts_size(int T, int E) {
  if (T < 0 || E < 1) return 0;
  return pair_counts_bytes(T, E);
}

int semmoe_pair_counts_stride(int T) { return T < 0 ? 0 : pair_counts_stride(T); }

int semmoe_route(const void* x, int x_dtype, const void* w_router, int w_dtype, const float* logits_in,
                 float* logits_out, const int32_t* k_per_token, int k_uniform, int T, int H, int E, int k_max,
                 int32_t* topk_idx, float* topk_w, int32_t* pair_counts, void* ws, size_t ws_bytes, void* stream) {
  REQUIRE(T >= 0, "semmoe_route: T = %d < 0", T);
  REQUIRE(E >= 1 && E <= 256, "semmoe_route: E = %d outside [1, 256]", E);
  REQUIRE(k_max >= 1 && k_max <= E, "semmoe_route: k_max = %d outside [1, E = %d]", k_max, E);
  REQUIRE((long long)T * (k_max > E ? k_max : E) < (1LL << 31), "semmoe_route: T * E too large");
  REQUIRE(k_per_token != nullptr || (k_uniform >= 1 && k_uniform <= k_max),
          "semmoe_route: k_uniform = %d outside [1, k_max = %d]", k_uniform, k_max);
  if (T == 0) return SEMMOE_OK;
  REQUIRE(topk_idx != nullptr && topk_w != nullptr, "semmoe_route: null output pointer");
  if (logits_in == nullptr) {
    REQUIRE(x != nullptr && w_router != nullptr, "semmoe_route: null x or w_router without logits_in");
    REQUIRE(valid_dtype(x_dtype) && valid_router_dtype(w_dtype, x_dtype, H), "semmoe_route: bad dtype (%d, %d)",
            x_dtype, w_dtype);
    REQUIRE(H >= 1, "semmoe_route: H = %d < 1", H);
    REQUIRE(aligned(x, 16) && aligned(w_router, 16), "semmoe_route: x and w_router must be 16-byte aligned");
    const size_t need = route_ws_bytes(T, H, E, x_dtype, w_dtype);
    REQUIRE(need == 0 || (ws != nullptr && aligned(ws, 256) && ws_bytes >= need),
            "semmoe_route: workspace null, not 256-byte aligned or below %zu bytes", need);
  } else {
    REQUIRE(aligned(logits_in, 4), "semmoe_route: misaligned logits_in");
  }
  REQUIRE(aligned(topk_idx, 4) && aligned(topk_w, 4) && aligned(logits_out, 4) && aligned(k_per_token, 4) &&
              aligned(pair_counts, 16),
          "semmoe_route: misaligned output or k_per_token");
  CHECK_DEVICE("semmoe_route");
  return cuda_status(launch_route(x, x_dtype, w_router, w_dtype, logits_in, logits_out, k_per_token, k_uniform, T,
                                  H, E, k_max, topk_idx, topk_w, pair_counts, ws, static_cast<cudaStream_t>(stream)),
                     "semmoe_route");
}

size_t semmoe_route_split_size(int H, int E) {
  if (H < 8 || H % 8 != 0 || E < 1 || E > 256) return 0;
  return route_split_size(H, E);
}

int semmoe_route_split_weight(const float* w, int H, int E, void* split, void* stream) {
  REQUIRE(H >= 8 && H % 8 == 0, "semmoe_route_split_weight: H = %d must be a positive multiple of 8", H);
  REQUIRE(E >= 1 && E <= 256, "semmoe_route_split_weight: E = %d outside [1, 256]", E);
  REQUIRE(w != nullptr && split != nullptr, "semmoe_route_split_weight: null pointer");
  REQUIRE(aligned(w, 4) && aligned(split, 256), "semmoe_route_split_weight: misaligned pointer");
  CHECK_DEVICE("semmoe_route_split_weight");
  return cuda_status(launch_route_split(w, H, E, split, static_cast<cudaStream_t>(stream)),
                     "semmoe_route_split_weight");
}

size_t semmoe_route_hier_workspace_size(int T, int H, int Ep, int x_dtype, int w_dtype) {
  if (T < 0 || H < 1 || Ep < 1 || !valid_dtype(x_dtype) || !valid_router_dtype(w_dtype, x_dtype, H)) return 0;
  const size_t b = route_hier_ws_bytes(T, H, Ep, x_dtype, w_dtype);
  return b > 0 ? b : 256;
}

int semmoe_route_hier(const void* x, int x_dtype, const void* w_parent, int w_dtype, const float* logits_in,
                      float* logits_out, const float* sub_logw, int N, const int32_t* k_per_token, int k_uniform,
                      int T, int H, int Ep, int k_max, int32_t* topk_idx, float* topk_w, int32_t* pair_counts,
                      void* ws, size_t ws_bytes, void* stream) {
  REQUIRE(T >= 0, "semmoe_route_hier: T = %d < 0", T);
  REQUIRE(N >= 1 && Ep >= 1 && (long long)Ep * N <= 256, "semmoe_route_hier: Ep * N = %lld outside [1, 256]",
          (long long)Ep * N);
  const int E = Ep * N;
  REQUIRE(k_max >= 1 && k_max <= E, "semmoe_route_hier: k_max = %d outside [1, Ep*N = %d]", k_max, E);
  REQUIRE((long long)T * E < (1LL << 31), "semmoe_route_hier: T * Ep * N too large");
  REQUIRE(k_per_token != nullptr || (k_uniform >= 1 && k_uniform <= k_max),
          "semmoe_route_hier: k_uniform = %d outside [1, k_max = %d]", k_uniform, k_max);
  if (T == 0) return SEMMOE_OK;
  REQUIRE(topk_idx != nullptr && topk_w != nullptr && sub_logw != nullptr, "semmoe_route_hier: null pointer");
  if (logits_in == nullptr) {
    REQUIRE(x != nullptr && w_parent != nullptr, "semmoe_route_hier: null x or w_parent without logits_in");
    REQUIRE(valid_dtype(x_dtype) && valid_router_dtype(w_dtype, x_dtype, H), "semmoe_route_hier: bad dtype (%d, %d)",
            x_dtype, w_dtype);
    REQUIRE(H >= 1, "semmoe_route_hier: H = %d < 1", H);
    REQUIRE(aligned(x, 16) && aligned(w_parent, 16), "semmoe_route_hier: x and w_parent must be 16-byte aligned");
    const size_t need = route_hier_ws_bytes(T, H, Ep, x_dtype, w_dtype);
    REQUIRE(need == 0 || (ws != nullptr && aligned(ws, 256) && ws_bytes >= need),
            "semmoe_route_hier: workspace null, not 256-byte aligned or below %zu bytes", need);
  } else {
    REQUIRE(aligned(logits_in, 4), "semmoe_route_hier: misaligned logits_in");
  }
  REQUIRE(aligned(topk_idx, 4) && aligned(topk_w, 4) && aligned(logits_out, 4) && aligned(k_per_token, 4) &&
              aligned(sub_logw, 4) && aligned(pair_counts, 16),
          "semmoe_route_hier: misaligned pointer");
  CHECK_DEVICE("semmoe_route_hier");
  return cuda_status(launch_route_hier(x, x_dtype, w_parent, w_dtype, logits_in, logits_out, sub_logw, N,
                                       k_per_token, k_uniform, T, H, Ep, k_max, topk_idx, topk_w, pair_counts, ws,
                                       static_cast<cudaStream_t>(stream)),
                     "semmoe_route_hier");
}

int semmoe_affinity_lookup(const int32_t* token_ids, const int32_t* lut, int V, int R, int T, int32_t* pred_rank,
                           void* stream) {
  REQUIRE(T >= 0 && V >= 1 && R >= 1, "semmoe_affinity_lookup: bad sizes T=%d V=%d R=%d", T, V, R);
  if (T == 0) return SEMMOE_OK;
  REQUIRE(token_ids && lut && pred_rank, "semmoe_affinity_lookup: null pointer");
  REQUIRE(aligned(token_ids, 4) && aligned(lut, 4) && aligned(pred_rank, 4), "semmoe_affinity_lookup: misaligned");
  CHECK_DEVICE("semmoe_affinity_lookup");
  return cuda_status(launch_affinity_lookup(token_ids, lut, V, R, T, pred_rank, static_cast<cudaStream_t>(stream)),
                     "semmoe_affinity_lookup");
}

int semmoe_remote_count(const int32_t* topk_idx, const int32_t* pred_rank, const int32_t* expert_rank, int T,
                        int k_max, int E, int R, int32_t* counts, int32_t* remote, void* stream) {
  REQUIRE(T >= 0 && k_max >= 1 && E >= 1 && E <= 256, "semmoe_remote_count: bad sizes T=%d k_max=%d E=%d", T, k_max,
          E);
  REQUIRE(R >= 1 && R <= 64, "semmoe_remote_count: R = %d outside [1, 64]", R);
  REQUIRE(counts && remote && expert_rank, "semmoe_remote_count: null pointer");
  REQUIRE(T == 0 || (topk_idx && pred_rank), "semmoe_remote_count: null topk_idx or pred_rank");
  REQUIRE((long long)T * k_max < (1LL << 31), "semmoe_remote_count: T * k_max too large");
  CHECK_DEVICE("semmoe_remote_count");
  return cuda_status(launch_remote_count(topk_idx, pred_rank, expert_rank, T, k_max, E, R, counts, remote,
                                         static_cast<cudaStream_t>(stream)),
                     "semmoe_remote_count");
}

size_t semmoe_permute_workspace_size(int T, int k_max, int E) {
  if (T < 0 || k_max < 1 || E < 1) return 0;
  return permute_ws_bytes(T, k_max, E);
}

int semmoe_permute(const int32_t* topk_idx, const int32_t* expert_rank, const void* x, int dtype, int T, int H,
                   int E, int R, int k_max, int P, int32_t* expert_offsets, int32_t* rank_offsets,
                   int32_t* phys_to_expert, int32_t* expert_counts, int32_t* sorted_to_pair,
                   int32_t* pair_to_sorted, void* x_perm, const int32_t* pair_counts, void* ws, size_t ws_bytes,
                   void* stream) {
  REQUIRE(T >= 0, "semmoe_permute: T = %d < 0", T);
  REQUIRE(E >= 1 && E <= 256, "semmoe_permute: E = %d outside [1, 256]", E);
  REQUIRE(R >= 1 && R <= E, "semmoe_permute: R = %d outside [1, E]", R);
  REQUIRE(k_max >= 1 && k_max <= E, "semmoe_permute: k_max = %d outside [1, E]", k_max);
  REQUIRE((long long)T * k_max < (1LL << 31), "semmoe_permute: T * k_max too large");
  REQUIRE(P >= 0 && (long long)P <= (long long)T * k_max, "semmoe_permute: P = %d outside [0, T*k_max]", P);
  REQUIRE(expert_rank && expert_offsets && rank_offsets && phys_to_expert && expert_counts,
          "semmoe_permute: null table pointer");
  REQUIRE(T == 0 || (topk_idx && pair_to_sorted), "semmoe_permute: null topk_idx or pair_to_sorted");
  REQUIRE(P == 0 || sorted_to_pair, "semmoe_permute: null sorted_to_pair");
  REQUIRE((x == nullptr) == (x_perm == nullptr), "semmoe_permute: x and x_perm must both be set or both NULL");
  if (x != nullptr) {
    REQUIRE(valid_dtype(dtype), "semmoe_permute: bad dtype %d", dtype);
    REQUIRE(H >= 1 && (H * elem_size(dtype)) % 16 == 0, "semmoe_permute: H * elem size must be a multiple of 16");
    REQUIRE(aligned(x, 16) && aligned(x_perm, 16), "semmoe_permute: x / x_perm not 16-byte aligned");
  }
  REQUIRE(ws != nullptr && aligned(ws, 256), "semmoe_permute: workspace null or not 256-byte aligned");
  REQUIRE(ws_bytes >= permute_ws_bytes(T, k_max, E), "semmoe_permute: workspace %zu < %zu bytes", ws_bytes,
          permute_ws_bytes(T, k_max, E));
  REQUIRE(aligned(pair_counts, 16), "semmoe_permute: pair_counts not 16-byte aligned");
  CHECK_DEVICE("semmoe_permute");
  return cuda_status(launch_permute(topk_idx, expert_rank, x, dtype, T, H, E, R, k_max, P, expert_offsets,
                                    rank_offsets, phys_to_expert, expert_counts, sorted_to_pair, pair_to_sorted,
                                    x_perm, pair_counts, ws, static_cast<cudaStream_t>(stream)),
                     "semmoe_permute");
}

int semmoe_permute_noalloc(const int32_t* topk_idx, const int32_t* expert_rank, const void* x, int dtype, int T,
                           int H, int E, int R, int k_max, int P, int32_t* expert_offsets, int32_t* rank_offsets,
                           int32_t* phys_to_expert, int32_t* expert_counts, int32_t* sorted_to_pair,
                           int32_t* pair_to_sorted, void* x_perm, void* stream) {
  REQUIRE(T >= 0, "semmoe_permute_noalloc: T = %d < 0", T);
  REQUIRE(E >= 1 && E <= 256, "semmoe_permute_noalloc: E = %d outside [1, 256]", E);
  REQUIRE(R >= 1 && R <= E, "semmoe_permute_noalloc: R = %d outside [1, E]", R);
  REQUIRE(k_max >= 1 && k_max <= E, "semmoe_permute_noalloc: k_max = %d outside [1, E]", k_max);
  REQUIRE((long long)T * k_max < (1LL << 31), "semmoe_permute_noalloc: T * k_max too large");
  REQUIRE(permute_ws_bytes(T, k_max, E) <= permute_noalloc_max_scratch(),
          "semmoe_permute_noalloc: T=%d, k_max=%d, E=%d need %zu bytes of scratch; the built-in scratch holds "
          "%zu bytes (use semmoe_permute with a caller workspace)",
          T, k_max, E, permute_ws_bytes(T, k_max, E), permute_noalloc_max_scratch());
  REQUIRE(P >= 0 && (long long)P <= (long long)T * k_max, "semmoe_permute_noalloc: P = %d outside [0, T*k_max]", P);
  REQUIRE(expert_rank && expert_offsets && rank_offsets && phys_to_expert && expert_counts,
          "semmoe_permute_noalloc: null table pointer");
  REQUIRE(T == 0 || (topk_idx && pair_to_sorted), "semmoe_permute_noalloc: null topk_idx or pair_to_sorted");
  REQUIRE(P == 0 || sorted_to_pair, "semmoe_permute_noalloc: null sorted_to_pair");
  REQUIRE((x == nullptr) == (x_perm == nullptr),
          "semmoe_permute_noalloc: x and x_perm must both be set or both NULL");
  if (x != nullptr) {
    REQUIRE(valid_dtype(dtype), "semmoe_permute_noalloc: bad dtype %d", dtype);
    REQUIRE(H >= 1 && (H * elem_size(dtype)) % 16 == 0,
            "semmoe_permute_noalloc: H * elem size must be a multiple of 16");
    REQUIRE(aligned(x, 16) && aligned(x_perm, 16), "semmoe_permute_noalloc: x / x_perm not 16-byte aligned");
  }
  CHECK_DEVICE("semmoe_permute_noalloc");
  return cuda_status(launch_permute_noalloc(topk_idx, expert_rank, x, dtype, T, H, E, R, k_max, P, expert_offsets,
                                            rank_offsets, phys_to_expert, expert_counts, sorted_to_pair,
                                            pair_to_sorted, x_perm, static_cast<cudaStream_t>(stream)),
                     "semmoe_permute_noalloc");
}

size_t semmoe_grouped_ffn_workspace_size(int P, int I, int dtype) {
  if (P < 0 || I < 1 || !valid_dtype(dtype)) return 0;
  return ffn_ws_bytes(P, I, dtype);
}

static int check_ffn_args(const char* fn, const void* x, const void* w13, const void* w2, int dtype, int P, int H,
                          int I, const void* y, const void* ws, size_t ws_bytes) {
  REQUIRE(valid_dtype(dtype), "%s: bad dtype %d", fn, dtype);
  REQUIRE(P >= 0 && H >= 8 && I >= 8 && H % 8 == 0 && I % 8 == 0, "%s: need P >= 0 and H, I multiples of 8 (P=%d H=%d I=%d)",
          fn, P, H, I);
  REQUIRE((long long)P * (H > I ? H : I) < (1LL << 40), "%s: P too large", fn);
  REQUIRE(w13 && w2 && (P == 0 || (x && y)), "%s: null pointer", fn);  // no rows: x and y may be empty
  REQUIRE(aligned(x, 16) && aligned(w13, 16) && aligned(w2, 16) && aligned(y, 16), "%s: pointers must be 16-byte aligned",
          fn);
  REQUIRE(ws != nullptr && aligned(ws, 256), "%s: workspace null or not 256-byte aligned", fn);
  REQUIRE(ws_bytes >= ffn_ws_bytes(P, I, dtype), "%s: workspace %zu < %zu bytes", fn, ws_bytes,
          ffn_ws_bytes(P, I, dtype));
  return SEMMOE_OK;
}

int semmoe_grouped_ffn(const void* x_perm, const int32_t* expert_offsets, const int32_t* phys_to_expert,
                       const void* w13, const void* w2, int dtype, int P, int E, int H, int I, void* y_perm,
                       void* ws, size_t ws_bytes, void* stream) {
  REQUIRE(E >= 1 && E <= 256, "semmoe_grouped_ffn: E = %d outside [1, 256]", E);
  REQUIRE(expert_offsets && phys_to_expert, "semmoe_grouped_ffn: null offsets");
  int rc = check_ffn_args("semmoe_grouped_ffn", x_perm, w13, w2, dtype, P, H, I, y_perm, ws, ws_bytes);
  if (rc != SEMMOE_OK) return rc;
  if (P == 0) return SEMMOE_OK;
  CHECK_DEVICE("semmoe_grouped_ffn");
  return cuda_status(launch_ffn(x_perm, expert_offsets, phys_to_expert, w13, w2, dtype, P, E, H, I, y_perm, ws,
                                nullptr, 1, 0, static_cast<cudaStream_t>(stream)),
                     "semmoe_grouped_ffn");
}

int semmoe_grouped_ffn_gather(const void* x, const int32_t* sorted_to_pair, int k_max, int T,
                              const int32_t* expert_offsets, const int32_t* phys_to_expert, const void* w13,
                              const void* w2, int dtype, int P, int E, int H, int I, void* y_perm, void* ws,
                              size_t ws_bytes, void* stream) {
  REQUIRE(E >= 1 && E <= 256, "semmoe_grouped_ffn_gather: E = %d outside [1, 256]", E);
  REQUIRE(T >= 0 && k_max >= 1 && (long long)T * k_max < (1LL << 31),
          "semmoe_grouped_ffn_gather: bad sizes T=%d k_max=%d", T, k_max);
  REQUIRE(P <= (long long)T * k_max, "semmoe_grouped_ffn_gather: P = %d > T * k_max", P);
  REQUIRE(expert_offsets && phys_to_expert, "semmoe_grouped_ffn_gather: null offsets");
  REQUIRE(P == 0 || sorted_to_pair, "semmoe_grouped_ffn_gather: null sorted_to_pair");
  int rc = check_ffn_args("semmoe_grouped_ffn_gather", x, w13, w2, dtype, P, H, I, y_perm, ws, ws_bytes);
  if (rc != SEMMOE_OK) return rc;
  if (P == 0) return SEMMOE_OK;
  CHECK_DEVICE("semmoe_grouped_ffn_gather");
  return cuda_status(launch_ffn(x, expert_offsets, phys_to_expert, w13, w2, dtype, P, E, H, I, y_perm, ws,
                                sorted_to_pair, k_max, T, static_cast<cudaStream_t>(stream)),
                     "semmoe_grouped_ffn_gather");
}

int semmoe_grouped_ffn_form(const void* x, const int32_t* sorted_to_pair, int k_max, int T,
                            const int32_t* expert_offsets, const int32_t* phys_to_expert, const void* w13,
                            const void* w2, int dtype, int P, int E, int H, int I, void* y_perm, void* ws,
                            size_t ws_bytes, int form1, int form2, void* stream) {
  const char* fn = "semmoe_grouped_ffn_form";
  REQUIRE(E >= 1 && E <= 256, "%s: E = %d outside [1, 256]", fn, E);
  REQUIRE(expert_offsets && phys_to_expert, "%s: null offsets", fn);
  const bool gathered = sorted_to_pair != nullptr;
  if (gathered) {
    REQUIRE(T >= 0 && k_max >= 1 && (long long)T * k_max < (1LL << 31), "%s: bad sizes T=%d k_max=%d", fn, T, k_max);
    REQUIRE(P <= (long long)T * k_max, "%s: P = %d > T * k_max", fn, P);
  }
  const bool cc1 = form1 == SEMMOE_FORM_CUDA_CORE, cc2 = form2 == SEMMOE_FORM_CUDA_CORE;
  const bool fu1 = form1 == SEMMOE_FORM_FUSED, fu2 = form2 == SEMMOE_FORM_FUSED;
  REQUIRE(form1 >= SEMMOE_FORM_DEFAULT && form1 <= SEMMOE_FORM_FUSED && form2 >= SEMMOE_FORM_DEFAULT &&
              form2 <= SEMMOE_FORM_FUSED && cc1 == cc2 && fu1 == fu2,
          "%s: bad form pair (%d, %d)", fn, form1, form2);
  REQUIRE(!fu1 || !gathered, "%s: SEMMOE_FORM_FUSED reads x_perm (no gathered rows)", fn);
  REQUIRE(form2 != SEMMOE_FORM_SINGLE_TMA_GATHER && (form1 != SEMMOE_FORM_SINGLE_TMA_GATHER || gathered),
          "%s: SEMMOE_FORM_SINGLE_TMA_GATHER applies to a GEMM1 with gathered rows only", fn);
  REQUIRE(dtype != SEMMOE_F32 || ((form1 == SEMMOE_FORM_DEFAULT || cc1) && (form2 == SEMMOE_FORM_DEFAULT || cc2)),
          "%s: fp32 runs on CUDA cores only (form SEMMOE_FORM_DEFAULT or SEMMOE_FORM_CUDA_CORE)", fn);
  int rc = check_ffn_args(fn, x, w13, w2, dtype, P, H, I, y_perm, ws, ws_bytes);
  if (rc != SEMMOE_OK) return rc;
  if (P == 0) return SEMMOE_OK;
  CHECK_DEVICE(fn);
  return cuda_status(launch_ffn(x, expert_offsets, phys_to_expert, w13, w2, dtype, P, E, H, I, y_perm, ws,
                                sorted_to_pair, gathered ? k_max : 1, gathered ? T : 0,
                                static_cast<cudaStream_t>(stream), form1, form2),
                     fn);
}

int semmoe_grouped_ffn_combine(const void* x, int x_rows_are_tokens, const int32_t* sorted_to_pair, int k_max, int T,
                               const int32_t* expert_offsets, const int32_t* phys_to_expert, const void* w13,
                               const void* w2, const float* topk_w, int dtype, int P, int E, int H, int I, float* acc,
                               void* ws, size_t ws_bytes, void* stream) {
  const char* fn = "semmoe_grouped_ffn_combine";
  REQUIRE(E >= 1 && E <= 256, "%s: E = %d outside [1, 256]", fn, E);
  REQUIRE(T >= 0 && k_max >= 1 && (long long)T * k_max < (1LL << 31), "%s: bad sizes T=%d k_max=%d", fn, T, k_max);
  REQUIRE(P >= 0 && P <= (long long)T * k_max, "%s: P = %d outside [0, T * k_max]", fn, P);
  REQUIRE(H >= 8 && I >= 8 && H % 8 == 0 && I % 8 == 0, "%s: need H, I multiples of 8 (H=%d I=%d)", fn, H, I);
  if (dtype != SEMMOE_BF16) return fail(SEMMOE_ERR_UNSUPPORTED, "%s: bf16 activations and experts only", fn);
  if (T == 0) return SEMMOE_OK;
  REQUIRE(expert_offsets && phys_to_expert && w13 && w2 && topk_w && acc, "%s: null pointer", fn);
  REQUIRE(P == 0 || (x && sorted_to_pair), "%s: null x or sorted_to_pair", fn);
  REQUIRE(aligned(x, 16) && aligned(w13, 16) && aligned(w2, 16) && aligned(acc, 16) && aligned(topk_w, 4),
          "%s: misaligned pointer", fn);
  REQUIRE(ws != nullptr && aligned(ws, 256) && ws_bytes >= ffn_ws_bytes(P, I, dtype),
          "%s: workspace null, not 256-byte aligned or below %zu bytes", fn, ffn_ws_bytes(P, I, dtype));
  CHECK_DEVICE(fn);
  return cuda_status(launch_ffn_combine(x, x_rows_are_tokens != 0, sorted_to_pair, k_max, T, expert_offsets,
                                        phys_to_expert, w13, w2, topk_w, P, E, H, I, acc, ws,
                                        static_cast<cudaStream_t>(stream)),
                     fn);
}

int semmoe_combine_finish(const float* acc, const void* y_shared, int dtype, int T, int H, void* out, void* stream) {
  const char* fn = "semmoe_combine_finish";
  REQUIRE(T >= 0 && H >= 8 && H % 8 == 0, "%s: bad sizes T=%d H=%d", fn, T, H);
  if (dtype != SEMMOE_BF16) return fail(SEMMOE_ERR_UNSUPPORTED, "%s: bf16 output only", fn);
  if (T == 0) return SEMMOE_OK;
  REQUIRE(acc && out, "%s: null pointer", fn);
  REQUIRE(aligned(acc, 16) && aligned(y_shared, 16) && aligned(out, 16), "%s: misaligned pointer", fn);
  CHECK_DEVICE(fn);
  return cuda_status(launch_combine_finish(acc, y_shared, T, H, out, static_cast<cudaStream_t>(stream)), fn);
}

size_t semmoe_shared_ffn_workspace_size(int T, int I_s, int dtype) {
  if (T < 0 || I_s < 1 || !valid_dtype(dtype)) return 0;
  return ffn_ws_bytes(T, I_s, dtype);
}

int semmoe_shared_ffn(const void* x, const void* ws13, const void* ws2, int dtype, int T, int H, int I_s,
                      void* y_shared, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_ffn_args("semmoe_shared_ffn", x, ws13, ws2, dtype, T, H, I_s, y_shared, ws, ws_bytes);
  if (rc != SEMMOE_OK) return rc;
  if (T == 0) return SEMMOE_OK;
  CHECK_DEVICE("semmoe_shared_ffn");
  // not as programmatic dependents: it runs beside the layer's steps on another
  // stream, where CTAs waiting for their turn would hold SMs those steps could use
  return cuda_status(launch_ffn(x, nullptr, nullptr, ws13, ws2, dtype, T, 1, H, I_s, y_shared, ws, nullptr, 1, 0,
                                static_cast<cudaStream_t>(stream), SEMMOE_FORM_DEFAULT, SEMMOE_FORM_DEFAULT, false),
                     "semmoe_shared_ffn");
}

int semmoe_combine(const void* y_perm, const int32_t* pair_to_sorted, const float* topk_w, const void* y_shared,
                   int dtype, int T, int H, int k_max, int P, void* out, void* stream) {
  REQUIRE(valid_dtype(dtype), "semmoe_combine: bad dtype %d", dtype);
  REQUIRE(T >= 0 && k_max >= 1 && P >= 0, "semmoe_combine: bad sizes T=%d k_max=%d P=%d", T, k_max, P);
  REQUIRE(H >= 1 && (H * elem_size(dtype)) % 16 == 0, "semmoe_combine: H * elem size must be a multiple of 16");
  REQUIRE((long long)T * k_max < (1LL << 31), "semmoe_combine: T * k_max too large");
  if (T == 0) return SEMMOE_OK;
  REQUIRE(pair_to_sorted && topk_w && out, "semmoe_combine: null pointer");
  REQUIRE(P == 0 || y_perm, "semmoe_combine: null y_perm");
  REQUIRE(aligned(y_perm, 16) && aligned(y_shared, 16) && aligned(out, 16), "semmoe_combine: pointers must be 16-byte aligned");
  CHECK_DEVICE("semmoe_combine");
  return cuda_status(launch_combine(y_perm, pair_to_sorted, topk_w, y_shared, dtype, T, H, k_max, P, out,
                                    static_cast<cudaStream_t>(stream)),
                     "semmoe_combine");
}

int semmoe_dp_schedule(const int32_t* pred_rank, const int32_t* req_offsets, int T, int n_req, int R, int32_t* hist,
                       int32_t* req_rank, int32_t* req_order, int32_t* rank_req_offsets, int32_t* req_tok_start,
                       int32_t* tok_order, int32_t* tok_rank, int32_t* rank_tok_offsets, void* stream) {
  REQUIRE(T >= 0 && n_req >= 0, "semmoe_dp_schedule: bad sizes T=%d n_req=%d", T, n_req);
  REQUIRE(R >= 1 && R <= 64, "semmoe_dp_schedule: R = %d outside [1, 64]", R);
  REQUIRE(n_req >= 1 || T == 0, "semmoe_dp_schedule: %d tokens but no request", T);
  REQUIRE((long long)n_req * R < (1LL << 31), "semmoe_dp_schedule: n_req * R too large");
  REQUIRE(req_offsets && rank_req_offsets && rank_tok_offsets, "semmoe_dp_schedule: null pointer");
  REQUIRE(n_req == 0 || (hist && req_rank && req_order && req_tok_start), "semmoe_dp_schedule: null request output");
  REQUIRE(T == 0 || (pred_rank && tok_order && tok_rank), "semmoe_dp_schedule: null token array");
  CHECK_DEVICE("semmoe_dp_schedule");
  return cuda_status(launch_dp_schedule(pred_rank, req_offsets, T, n_req, R, hist, req_rank, req_order,
                                        rank_req_offsets, req_tok_start, tok_order, tok_rank, rank_tok_offsets,
                                        static_cast<cudaStream_t>(stream)),
                     "semmoe_dp_schedule");
}

int semmoe_transition_lookup(const int32_t* topk_idx, const int32_t* k_per_token, int k_uniform, const float* trans,
                             int T, int k_max, int E, int R, int32_t* pred_next, void* stream) {
  REQUIRE(T >= 0 && k_max >= 1 && E >= 1, "semmoe_transition_lookup: bad sizes T=%d k_max=%d E=%d", T, k_max, E);
  REQUIRE(R >= 1 && R <= 64, "semmoe_transition_lookup: R = %d outside [1, 64]", R);
  REQUIRE((long long)T * k_max < (1LL << 31) && (long long)E * R < (1LL << 31),
          "semmoe_transition_lookup: T * k_max or E * R too large");
  REQUIRE(k_per_token != nullptr || (k_uniform >= 1 && k_uniform <= k_max),
          "semmoe_transition_lookup: k_uniform = %d outside [1, k_max = %d]", k_uniform, k_max);
  if (T == 0) return SEMMOE_OK;
  REQUIRE(topk_idx && trans && pred_next, "semmoe_transition_lookup: null pointer");
  REQUIRE(aligned(trans, 4) && aligned(topk_idx, 4) && aligned(pred_next, 4) && aligned(k_per_token, 4),
          "semmoe_transition_lookup: misaligned pointer");
  CHECK_DEVICE("semmoe_transition_lookup");
  return cuda_status(launch_transition_lookup(topk_idx, k_per_token, k_uniform, trans, T, k_max, E, R, pred_next,
                                              static_cast<cudaStream_t>(stream)),
                     "semmoe_transition_lookup");
}

int semmoe_selftest_bounded_wait(void* stream) {
  CHECK_DEVICE("semmoe_selftest_bounded_wait");
  return cuda_status(launch_selftest_bounded_wait(static_cast<cudaStream_t>(stream)), "semmoe_selftest_bounded_wait");
}

int semmoe_selftest_fused_ready_wait(const void* x_perm, const void* w13, const void* w2, int P, int H, int I,
                                     void* y_perm, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_ffn_args("semmoe_selftest_fused_ready_wait", x_perm, w13, w2, SEMMOE_BF16, P, H, I, y_perm, ws,
                          ws_bytes);
  if (rc != SEMMOE_OK) return rc;
  REQUIRE(P > 0 && P <= 4096, "semmoe_selftest_fused_ready_wait: need 0 < P <= 4096 (P=%d)", P);
  CHECK_DEVICE("semmoe_selftest_fused_ready_wait");
  return cuda_status(launch_selftest_fused_ready_wait(x_perm, w13, w2, P, H, I, y_perm, ws,
                                                      static_cast<cudaStream_t>(stream)),
                     "semmoe_selftest_fused_ready_wait");
}

}  // extern "C"
