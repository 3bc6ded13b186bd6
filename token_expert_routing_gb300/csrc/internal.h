// Launchers behind the C ABI (host code; arguments already validated).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "semmoe.h"

namespace semmoe {

// Adds n to the library-wide count of kernel launches (see semmoe_kernel_launches).
void count_launches(int n);

// Each translation unit keeps its own device error word; these read and clear it.
int route_take_errors(cudaStream_t s, int* bits);
int permute_take_errors(cudaStream_t s, int* bits);
int ffn_take_errors(cudaStream_t s, int* bits);
int combine_take_errors(cudaStream_t s, int* bits);
int schedule_take_errors(cudaStream_t s, int* bits);
int selftest_take_errors(cudaStream_t s, int* bits);
cudaError_t launch_selftest_bounded_wait(cudaStream_t s);
cudaError_t launch_selftest_fused_ready_wait(const void* x, const void* w13, const void* w2, int P, int H, int I,
                                             void* y, void* ws, cudaStream_t s);

size_t route_ws_bytes(int T, int H, int E, int x_dtype, int w_dtype);
// Tensor-core router (route_tc.cu): fp32 logits of bf16 activations.
int route_tc_take_errors(cudaStream_t s, int* bits);
size_t route_tc_split_bytes(int H, int E, int w_dtype);
size_t route_split_size(int H, int E);
cudaError_t launch_route_split(const float* w, int H, int E, void* split, cudaStream_t s);
int route_tc_k_slices(int T, int H, int E, int w_dtype);
cudaError_t launch_route_logits_tc(const void* x, const void* w, int w_dtype, int T, int H, int E, float* partials,
                                   int ks, void* split, cudaStream_t s);
// The router GEMM and the top-k in one tensor-core kernel (route_tc.cu), for
// routers whose experts fit one MMA (route_topk_tc_ok); writes the count table
// (counts, row stride count_stride) in full when counts is not null.
bool route_topk_tc_ok(int E, int k_max, int w_dtype);
cudaError_t launch_route_topk_tc(const void* x, const void* w, int w_dtype, int T, int H, int E, int k_max,
                                 float* logits_out, const int32_t* kpt, int k_uniform, int32_t* topk_idx,
                                 float* topk_w, int32_t* counts, int count_stride, void* split, cudaStream_t s);
// The same for fewer token tiles than SMs: a cluster of CS CTAs per tile, each
// contracting a slice of H, reduced through distributed shared memory.
// route_topk_cl_slices gives CS (0: not applicable).
int route_topk_cl_slices(int T, int H, int E, int k_max, int w_dtype);
cudaError_t launch_route_topk_cl(const void* x, const void* w, int w_dtype, int T, int H, int E, int k_max, int CS,
                                 float* logits_out, const int32_t* kpt, int k_uniform, int32_t* topk_idx,
                                 float* topk_w, int32_t* counts, int count_stride, void* split, cudaStream_t s);
// pair_counts (nullable): zeroed here, then the live picks are counted into it
// (layout of pair_counts_bytes).
cudaError_t launch_route(const void* x, int x_dtype, const void* w, int w_dtype,
                         const float* logits_in, float* logits_out, const int32_t* k_per_token,
                         int k_uniform, int T, int H, int E, int k_max, int32_t* topk_idx,
                         float* topk_w, int32_t* pair_counts, void* ws, cudaStream_t s);

// MoE-Prism hierarchical gating over Ep parents x N sub-experts.
size_t route_hier_ws_bytes(int T, int H, int Ep, int x_dtype, int w_dtype);
cudaError_t launch_route_hier(const void* x, int x_dtype, const void* w, int w_dtype, const float* logits_in,
                              float* logits_out, const float* sub_logw, int N, const int32_t* kpt, int k_uniform,
                              int T, int H, int Ep, int k_max, int32_t* topk_idx, float* topk_w,
                              int32_t* pair_counts, void* ws, cudaStream_t s);

cudaError_t launch_affinity_lookup(const int32_t* token_ids, const int32_t* lut, int V, int R,
                                   int T, int32_t* pred, cudaStream_t s);

cudaError_t launch_remote_count(const int32_t* topk_idx, const int32_t* pred,
                                const int32_t* expert_rank, int T, int k_max, int E, int R,
                                int32_t* counts, int32_t* remote, cudaStream_t s);

size_t permute_ws_bytes(int T, int k_max, int E);
// The pair count table [E][pair_counts_stride(T)] of 128-token chunks
// (SEMMOE_PAIR_COUNT_CHUNK) that the router can write for the permute.
size_t pair_counts_bytes(int T, int E);
int pair_counts_stride(int T);
cudaError_t launch_permute(const int32_t* topk_idx, const int32_t* expert_rank, const void* x,
                           int dtype, int T, int H, int E, int R, int k_max, int P,
                           int32_t* expert_offsets, int32_t* rank_offsets,
                           int32_t* phys_to_expert, int32_t* expert_counts,
                           int32_t* sorted_to_pair, int32_t* pair_to_sorted, void* x_perm,
                           const int32_t* pair_counts, void* ws, cudaStream_t s);

// semmoe_permute with its scratch in a static device array (no allocation).
size_t permute_noalloc_max_scratch();
cudaError_t launch_permute_noalloc(const int32_t* topk_idx, const int32_t* expert_rank, const void* x,
                                   int dtype, int T, int H, int E, int R, int k_max, int P,
                                   int32_t* expert_offsets, int32_t* rank_offsets, int32_t* phys_to_expert,
                                   int32_t* expert_counts, int32_t* sorted_to_pair, int32_t* pair_to_sorted,
                                   void* x_perm, cudaStream_t s);

size_t ffn_ws_bytes(int P, int I, int dtype);
// Readiness counters of the one-launch grouped FFN (one int per m-tile), after h in its workspace.
inline size_t ffn_ready_bytes(int P) { return align_up((size_t)((P > 0 ? P : 1) + 127) / 128 * 4 + 257 * 4, 256); }
// offsets == nullptr: one group of rows [0, P) using expert 0 of w13/w2.
// gather != nullptr: x is [T_x, H] unpermuted and GEMM1's sorted row q reads x
// row gather[q] / gather_div; otherwise x holds the P sorted rows.
// form1 / form2: SEMMOE_FORM_* of GEMM1 / GEMM2 (SEMMOE_FORM_DEFAULT: chosen from
// the shapes; SEMMOE_FORM_CUDA_CORE in form1 runs both GEMMs on CUDA cores).
// dependent: the tensor-core kernels launch as programmatic dependents of the
// kernel before them on s (the layer's own chain; false beside it).
cudaError_t launch_ffn(const void* x, const int32_t* offsets, const int32_t* phys_to_expert,
                       const void* w13, const void* w2, int dtype, int P, int E, int H, int I,
                       void* y, void* ws, const int32_t* gather, int gather_div, int T_x, cudaStream_t s,
                       int form1 = SEMMOE_FORM_DEFAULT, int form2 = SEMMOE_FORM_DEFAULT, bool dependent = true);

// The combine folded into GEMM2 (bf16): acc [T, H] fp32 zeroed, then the grouped
// FFN whose GEMM2 adds its gate-weighted rows into acc; launch_combine_finish
// then writes out = y_shared + acc.
cudaError_t launch_ffn_combine(const void* x, bool gathered, const int32_t* sorted_to_pair, int k_max, int T,
                               const int32_t* offsets, const int32_t* p2e, const void* w13, const void* w2,
                               const float* topk_w, int P, int E, int H, int I, float* acc, void* ws,
                               cudaStream_t s);
cudaError_t launch_combine_finish(const float* acc, const void* y_shared, int T, int H, void* out, cudaStream_t s);

cudaError_t launch_combine(const void* y_perm, const int32_t* pair_to_sorted, const float* topk_w,
                           const void* y_shared, int dtype, int T, int H, int k_max, int P,
                           void* out, cudaStream_t s);

cudaError_t launch_dp_schedule(const int32_t* pred, const int32_t* off, int T, int n_req, int R, int32_t* hist,
                               int32_t* req_rank, int32_t* req_order, int32_t* rank_req_offsets,
                               int32_t* req_tok_start, int32_t* tok_order, int32_t* tok_rank,
                               int32_t* rank_tok_offsets, cudaStream_t s);

cudaError_t launch_transition_lookup(const int32_t* topk_idx, const int32_t* kpt, int ku, const float* trans, int T,
                                     int k_max, int E, int R, int32_t* pred_next, cudaStream_t s);

}  // namespace semmoe
