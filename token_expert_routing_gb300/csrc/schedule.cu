// Table-driven scheduling around the layer.
//
// dp_schedule: the online inter-request scheduling of Attention-DP (Semantic
// Parallelism (ko) §2.2 item 2, (de) §2 B, (ja) §2.2 B.1).  Each request's
// tokens vote with their predicted rank; the request goes to the rank with the
// most votes (ties to the lowest rank) and the requests are regrouped stably by
// rank, so each rank's batch is its requests' tokens laid end to end.
//
// transition_lookup: the next layer's device predicted from the experts a
// token chose in this layer (Semantic Parallelism (ko) §2.1, (de) §2 A, (ja)
// §2.3): score[r] = sum over the token's live slots of trans[e][r], argmax r.
#include "common.cuh"
#include "internal.h"

namespace semmoe {
namespace {

__device__ int g_err;  // SEMMOE_DEVERR_* bits seen by this file's kernels

__device__ __forceinline__ void flag(int bit) { atomicOr(&g_err, bit); }

constexpr int kMaxR = 64;
constexpr int kHistThreads = 128;  // 4 warps
constexpr int kOrderThreads = 1024;
constexpr int kOrderWarps = kOrderThreads / 32;

// Token range [lo, hi) of request i, clamped into [0, T] and to lo <= hi so that
// invalid offsets can never index outside the token arrays.  Every kernel here
// derives a request's range with this one function.
__device__ __forceinline__ void req_range(const int32_t* __restrict__ off, int i, int T, int& lo, int& hi) {
  lo = min(max(off[i], 0), T);
  hi = min(max(off[i + 1], lo), T);
}

// Warp argmax over a histogram row h[0..R) held in shared memory: the largest
// count, the lowest rank among equal counts.  Valid in every lane.
__device__ __forceinline__ int warp_argmax_row(const int* h, int R, int lane) {
  int v = lane < R ? h[lane] : -1, i = lane;
  if (lane + 32 < R && h[lane + 32] > v) { v = h[lane + 32]; i = lane + 32; }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const int ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
  }
  return i;
}

// One group of WPR warps per request (4 / WPR requests per 128-thread block):
// the rank histogram of the request's tokens, its argmax, and the request's
// rank written to each of its tokens.  WPR = 4 suits long requests, WPR = 1
// many short ones.
template <int WPR>
__global__ void __launch_bounds__(kHistThreads)
dp_hist_kernel(const int32_t* __restrict__ pred, const int32_t* __restrict__ off, int n_req, int T, int R,
               int32_t* __restrict__ hist, int32_t* __restrict__ req_rank, int32_t* __restrict__ tok_rank) {
  constexpr int G = 4 / WPR;
  __shared__ int h[G][kMaxR];
  __shared__ int best_s[G];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = warp / WPR, wg = warp % WPR;
  const int gt = wg * 32 + lane;  // thread index within the group
  for (long long base = (long long)blockIdx.x * G; base < n_req; base += (long long)gridDim.x * G) {
    const long long r = base + g;
    const bool live = r < n_req;
    for (int q = gt; q < R; q += WPR * 32) h[g][q] = 0;
    if (WPR > 1) __syncthreads(); else __syncwarp();
    int lo = 0, hi = 0;
    if (live) {
      const int ri = (int)r;
      const int a = off[ri], b = off[ri + 1];
      if (a < 0 || b < a || b > T || (ri == 0 && a != 0) || (ri == n_req - 1 && b != T)) {
        if (gt == 0) flag(SEMMOE_DEVERR_OFFSETS);
      }
      req_range(off, ri, T, lo, hi);
      for (int t0 = lo + wg * 32; t0 < hi; t0 += WPR * 32) {
        const int t = t0 + lane;
        int q = -1;
        if (t < hi) {
          q = pred[t];
          if (q < 0 || q >= R) { flag(SEMMOE_DEVERR_RANK); q = 0; }
        }
        const unsigned peers = __match_any_sync(0xffffffffu, q);
        if (q >= 0 && (peers & lanemask_lt()) == 0) atomicAdd(&h[g][q], __popc(peers));
      }
    }
    if (WPR > 1) __syncthreads(); else __syncwarp();
    if (wg == 0) {
      const int best = warp_argmax_row(h[g], R, lane);
      if (live) {
        for (int q = lane; q < R; q += 32) hist[r * R + q] = h[g][q];
        if (lane == 0) req_rank[r] = best;
      }
      if (lane == 0) best_s[g] = best;
    }
    if (WPR > 1) __syncthreads(); else __syncwarp();
    if (live) {
      const int best = best_s[g];
      for (int t = lo + gt; t < hi; t += WPR * 32) tok_rank[t] = best;
    }
    if (WPR > 1) __syncthreads(); else __syncwarp();
  }
}

// One CTA: the stable counting sort of the requests by rank, and where each
// request's first token lands in the scheduled token order.  Pass 1 counts
// requests and tokens per rank; pass 2 walks the requests in id order, 1024 at
// a time, giving each its position among the earlier requests of its rank
// (in-warp rank from __match_any_sync, then the per-rank totals of the
// earlier warps of the chunk, then the earlier chunks).
__global__ void __launch_bounds__(kOrderThreads)
dp_order_kernel(const int32_t* __restrict__ off, const int32_t* __restrict__ req_rank, int n_req, int T, int R,
                int32_t* __restrict__ req_order, int32_t* __restrict__ rank_req_offsets,
                int32_t* __restrict__ req_tok_start, int32_t* __restrict__ rank_tok_offsets) {
  __shared__ int cnt[kMaxR + 1], tsum[kMaxR + 1];
  __shared__ int run_c[kMaxR], run_t[kMaxR];
  __shared__ int wc[kOrderWarps][kMaxR + 1], wt[kOrderWarps][kMaxR + 1];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Request i's rank (clamped into [0, R)) and token count.
  auto load = [&](int i, int& q, int& len) {
    q = req_rank[i];
    if (q < 0 || q >= R) { flag(SEMMOE_DEVERR_RANK); q = 0; }
    int lo, hi;
    req_range(off, i, T, lo, hi);
    len = hi - lo;
  };

  for (int q = tid; q <= R; q += kOrderThreads) { cnt[q] = 0; tsum[q] = 0; }
  __syncthreads();
  for (int i = tid; i < n_req; i += kOrderThreads) {
    int q, len;
    load(i, q, len);
    atomicAdd(&cnt[q], 1);
    atomicAdd(&tsum[q], len);
  }
  __syncthreads();
  if (tid == 0) {
    int c = 0, s = 0;
    for (int q = 0; q < R; ++q) {
      rank_req_offsets[q] = c;
      rank_tok_offsets[q] = s;
      run_c[q] = c;
      run_t[q] = s;
      c += cnt[q];
      s += tsum[q];
    }
    rank_req_offsets[R] = c;
    rank_tok_offsets[R] = s;
  }
  __syncthreads();

  for (int c0 = 0; c0 < n_req; c0 += kOrderThreads) {
    const int i = c0 + tid;
    int q = R, len = 0;  // lanes past the end use the spare bucket R
    if (i < n_req) load(i, q, len);
    const unsigned peers = __match_any_sync(0xffffffffu, q);
    const unsigned below = peers & lanemask_lt();
    const int pc = __popc(below);
    int pl = 0;  // tokens of the earlier requests of this rank in the warp
#pragma unroll
    for (int src = 0; src < 32; ++src) {
      const int v = __shfl_sync(0xffffffffu, len, src);
      if ((below >> src) & 1u) pl += v;
    }
    for (int j = tid; j < kOrderWarps * (kMaxR + 1); j += kOrderThreads) {
      (&wc[0][0])[j] = 0;
      (&wt[0][0])[j] = 0;
    }
    __syncthreads();
    if ((peers >> lane) == 1u) {  // highest lane of its group: the warp's totals for q
      wc[warp][q] = pc + 1;
      wt[warp][q] = pl + len;
    }
    __syncthreads();
    if (tid < R) {
      int c = run_c[tid], s = run_t[tid];
      for (int w = 0; w < kOrderWarps; ++w) {
        const int a = wc[w][tid], b = wt[w][tid];
        wc[w][tid] = c;
        wt[w][tid] = s;
        c += a;
        s += b;
      }
      run_c[tid] = c;
      run_t[tid] = s;
    }
    __syncthreads();
    if (i < n_req) {
      const int pos = wc[warp][q] + pc;
      if (pos >= 0 && pos < n_req) req_order[pos] = i;
      else flag(SEMMOE_DEVERR_PAIRS);
      req_tok_start[i] = wt[warp][q] + pl;
    }
    __syncthreads();
  }
}

// The scheduled token order: request r's tokens, in order, from req_tok_start[r].
template <int WPR>
__global__ void __launch_bounds__(kHistThreads)
dp_scatter_kernel(const int32_t* __restrict__ off, const int32_t* __restrict__ req_tok_start, int n_req, int T,
                  int32_t* __restrict__ tok_order) {
  constexpr int G = 4 / WPR;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = warp / WPR, gt = (warp % WPR) * 32 + lane;
  for (long long r = (long long)blockIdx.x * G + g; r < n_req; r += (long long)gridDim.x * G) {
    int lo, hi;
    req_range(off, (int)r, T, lo, hi);
    const long long d0 = (long long)req_tok_start[r] - lo;
    for (int t = lo + gt; t < hi; t += WPR * 32) {
      const long long d = d0 + t;
      if (d >= 0 && d < T) tok_order[d] = t;
      else flag(SEMMOE_DEVERR_OFFSETS);
    }
  }
}

// One warp per token; lane l accumulates ranks l and l + 32.
constexpr int kTransThreads = 256;

__global__ void __launch_bounds__(kTransThreads)
transition_kernel(const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ kpt, int ku,
                  const float* __restrict__ trans, int T, int k_max, int E, int R, int32_t* __restrict__ pred_next) {
  const int lane = threadIdx.x & 31;
  const int wpb = kTransThreads / 32;
  for (long long t = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += (long long)gridDim.x * wpb) {
    int k = kpt ? kpt[t] : ku;
    if (k < 1 || k > k_max) {
      if (lane == 0) flag(SEMMOE_DEVERR_K);
      k = min(max(k, 0), k_max);
    }
    const int32_t* slots = topk_idx + t * k_max;
    float s0 = 0.0f, s1 = 0.0f;
    for (int j0 = 0; j0 < k; j0 += 32) {
      const int mine = j0 + lane < k ? slots[j0 + lane] : -1;
      const int n = min(32, k - j0);
      for (int j = 0; j < n; ++j) {
        const int e = __shfl_sync(0xffffffffu, mine, j);
        if (e < 0) continue;
        if (e >= E) {
          if (lane == 0) flag(SEMMOE_DEVERR_EXPERT);
          continue;
        }
        const float* row = trans + (size_t)e * R;
        if (lane < R) s0 = __fadd_rn(s0, row[lane]);
        if (lane + 32 < R) s1 = __fadd_rn(s1, row[lane + 32]);
      }
    }
    float v = lane < R ? s0 : -INFINITY;
    int i = lane;
    if (lane + 32 < R && s1 > v) { v = s1; i = lane + 32; }
    if ((lane < R && !isfinite(s0)) || (lane + 32 < R && !isfinite(s1))) flag(SEMMOE_DEVERR_NONFINITE);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, i, o);
      if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
    }
    if (lane == 0) pred_next[t] = i;
  }
}

int grid_for(long long units, int per_block) {
  long long b = (units + per_block - 1) / per_block;
  const long long cap = 8LL * sm_count();
  return (int)(b < 1 ? 1 : (b > cap ? cap : b));
}

}  // namespace

int schedule_take_errors(cudaStream_t s, int* bits) { return take_error_word(g_err, s, bits); }

cudaError_t launch_dp_schedule(const int32_t* pred, const int32_t* off, int T, int n_req, int R, int32_t* hist,
                               int32_t* req_rank, int32_t* req_order, int32_t* rank_req_offsets,
                               int32_t* req_tok_start, int32_t* tok_order, int32_t* tok_rank,
                               int32_t* rank_tok_offsets, cudaStream_t s) {
  // Long requests get a whole 4-warp block each; short ones one warp each.
  const bool wide = n_req > 0 && (long long)T >= 128LL * n_req;
  if (n_req > 0) {
    if (wide)
      dp_hist_kernel<4><<<grid_for(n_req, 1), kHistThreads, 0, s>>>(pred, off, n_req, T, R, hist, req_rank, tok_rank);
    else
      dp_hist_kernel<1><<<grid_for(n_req, 4), kHistThreads, 0, s>>>(pred, off, n_req, T, R, hist, req_rank, tok_rank);
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  dp_order_kernel<<<1, kOrderThreads, 0, s>>>(off, req_rank, n_req, T, R, req_order, rank_req_offsets, req_tok_start,
                                              rank_tok_offsets);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || n_req == 0) return e;
  if (wide)
    dp_scatter_kernel<4><<<grid_for(n_req, 1), kHistThreads, 0, s>>>(off, req_tok_start, n_req, T, tok_order);
  else
    dp_scatter_kernel<1><<<grid_for(n_req, 4), kHistThreads, 0, s>>>(off, req_tok_start, n_req, T, tok_order);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_transition_lookup(const int32_t* topk_idx, const int32_t* kpt, int ku, const float* trans, int T,
                                     int k_max, int E, int R, int32_t* pred_next, cudaStream_t s) {
  transition_kernel<<<grid_for(T, kTransThreads / 32), kTransThreads, 0, s>>>(topk_idx, kpt, ku, trans, T, k_max, E,
                                                                              R, pred_next);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace semmoe
