// Router GEMM + fp32 softmax + per-token top-k; token-id affinity lookup;
// per-(source rank, destination rank) activation counts.
//
// Router: the gate that scores experts per token (Semantic Parallelism (ko)
// §1, MoE-Prism (ko) §1) with a per-request budget k (MoE-Prism (ko) §2 B).
// Lookup table: Semantic Parallelism (ja) §2.3.  Local activation rate:
// Semantic Parallelism (ko) §3-§4.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace semmoe {
namespace {

__device__ int g_err;  // SEMMOE_DEVERR_* bits seen by this file's kernels

__device__ __forceinline__ void flag(int bit) { atomicOr(&g_err, bit); }

// Optional count table of the picks for the permute: counts[e * stride + c] =
// live pairs of expert e among the tokens of 128-token chunk c (zeroed before
// the kernel; one atomic add per pick).
struct PairCounts {
  int32_t* p = nullptr;
  int stride = 0;
};
__device__ __forceinline__ void count_pick(const PairCounts& pc, int e, int t) {
  if (pc.p != nullptr) atomicAdd(pc.p + (size_t)e * pc.stride + t / SEMMOE_PAIR_COUNT_CHUNK, 1);
}

constexpr int kRouteThreads = 256;
constexpr int kRouteTok = 32;   // tokens per block
constexpr int kRouteEC = 64;    // experts per GEMM chunk
constexpr int kRouteHK = 32;    // hidden elements per k step
constexpr int kRouteMaxE = 256;
constexpr int kWarps = kRouteThreads / 32;

// Shared-memory layout of route_kernel (floats unless noted):
//   lg   [kRouteTok][Epad]        logits of the block's tokens
//   xs   [kRouteTok][kRouteHK+1]  x tile (fp32)
//   ws   [kRouteEC][kRouteHK+1]   router-weight tile (fp32)
//   sel_v[kWarps][k_max], sel_e[kWarps][k_max] (int)
__host__ __device__ inline size_t route_smem_bytes(int E, int k_max) {
  int Epad = (E + 31) / 32 * 32;
  return sizeof(float) * ((size_t)kRouteTok * Epad + (size_t)(kRouteTok + kRouteEC) * (kRouteHK + 1)) +
         (size_t)kWarps * k_max * (sizeof(float) + sizeof(int));
}

// Token t's budget k_t, clamped into [1, k_max] (and flagged) when out of range.
__device__ __forceinline__ int warp_budget(const int32_t* __restrict__ k_per_token, int k_uniform, int k_max,
                                           int t) {
  int kt = k_per_token != nullptr ? k_per_token[t] : k_uniform;
  if (kt < 1 || kt > k_max) {
    if ((threadIdx.x & 31) == 0) flag(SEMMOE_DEVERR_K);
    kt = kt < 1 ? 1 : k_max;
  }
  return kt;
}

// One warp loads a token's E logits into v (lane holds e = lane + 32 i): the
// sum of `ks` partial rows slice_stride floats apart, added in slice order
// (each batch of slices loaded before any is added, so the loads are in flight
// together), copied to logits_out when that is set.  Entries past E and
// non-finite logits (flagged) become -inf.
template <int NPER>
__device__ __forceinline__ void warp_load_logits(const float* row, int ks, size_t slice_stride, float* logits_out,
                                                 int E, float (&v)[NPER]) {
  const int lane = threadIdx.x % 32;
  constexpr int SB = NPER <= 2 ? 8 : (NPER == 4 ? 4 : 2);
#pragma unroll
  for (int i = 0; i < NPER; ++i) v[i] = 0.f;
  for (int k0 = 0; k0 < ks; k0 += SB) {
    float part[NPER][SB];
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
      const int e = lane + 32 * i;
#pragma unroll
      for (int u = 0; u < SB; ++u)
        part[i][u] = (e < E && k0 + u < ks) ? row[(size_t)(k0 + u) * slice_stride + e] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
#pragma unroll
      for (int u = 0; u < SB; ++u) {
        if (k0 + u < ks) v[i] = (k0 + u == 0) ? part[i][u] : v[i] + part[i][u];
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      if (logits_out != nullptr) logits_out[e] = v[i];
      if (!isfinite(v[i])) {
        flag(SEMMOE_DEVERR_NONFINITE);
        v[i] = -INFINITY;
      }
    } else {
      v[i] = -INFINITY;
    }
  }
}

// k_t rounds of a warp argmax over (score descending, index ascending) of the
// n scores in v.  Lane 0 writes the j-th pick to my_v[j] / my_e[j] (-1 when
// fewer than k_t scores are left, flagged).  Each score becomes an
// order-preserving 32-bit key (-0.0 counted as +0.0; key 0 marks padding,
// below every float including -inf).  Two forms with the same picks: rescanning
// the lane's keys every round (cheaper for 2-4 scores per lane), or sorting them
// once (13% faster than rescanning at 8 per lane, E = 256, k <= 24; 3-6% slower
// at 2-4).  In the sorted form the winning lane's next key comes from shared
// memory instead of shifting its registers: 16.2 against 17.5 us per top-k of
// 8192 tokens at E = 256, k <= 24 (CUDA graph of 20 calls).

// Few scores per lane (NPER <= 4): each round rescans the lane's keys -- two
// warp reductions (the largest key, then the lowest index holding it), and the
// picked score's key becomes 0 (taken).
template <int NPER>
__device__ __forceinline__ void warp_select_rescan(const float (&v)[NPER], int n, int kt, float* my_v, int* my_e) {
  const int lane = threadIdx.x % 32;
  uint32_t key[NPER];
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
    const uint32_t b = __float_as_uint(__fadd_rn(v[i], 0.0f));  // -0.0 -> +0.0
    key[i] = lane + 32 * i < n ? ((b & 0x80000000u) ? ~b : (b | 0x80000000u)) : 0u;
  }
  for (int j = 0; j < kt; ++j) {
    uint32_t m = key[0];
#pragma unroll
    for (int i = 1; i < NPER; ++i) m = max(m, key[i]);
    m = __reduce_max_sync(0xffffffffu, m);
    int be = -1;
    if (m != 0u) {
      uint32_t mine = 0xffffffffu;  // this lane's lowest index whose key is m
#pragma unroll
      for (int i = NPER - 1; i >= 0; --i)
        if (key[i] == m) mine = (uint32_t)(lane + 32 * i);
      be = (int)__reduce_min_sync(0xffffffffu, mine);
#pragma unroll
      for (int i = 0; i < NPER; ++i)
        if (be == lane + 32 * i) key[i] = 0u;
    } else if (lane == 0) {
      flag(SEMMOE_DEVERR_NONFINITE);  // fewer than kt scores
    }
    if (lane == 0) {
      my_v[j] = be >= 0 ? __uint_as_float((m & 0x80000000u) ? (m ^ 0x80000000u) : ~m) : -INFINITY;
      my_e[j] = be;
    }
  }
  __syncwarp();
}

// Many scores per lane (NPER >= 8): each score's key is packed with its inverted
// index into a 64-bit word that orders (score descending, index ascending).
// Each lane sorts its NPER words once and keeps the first in a register (its
// head) and the rest, then a 0, in `lists` (shared memory, [NPER][32] words
// for the warp, entry i of lane l at i * 32 + l).  A round is two warp
// reductions over the heads (the largest key, then the lowest index holding
// it); the winning lane loads its next word as its new head.  A head with the
// round's key is its lane's lowest index with that key, so the lowest index
// among heads is the lowest overall.
template <int NPER>
__device__ __forceinline__ void warp_select_sorted(const float (&v)[NPER], int n, int kt, float* my_v, int* my_e,
                                                   unsigned long long* lists) {
  const int lane = threadIdx.x % 32;
  unsigned long long c[NPER];
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
    const uint32_t b = __float_as_uint(__fadd_rn(v[i], 0.0f));  // -0.0 -> +0.0
    const uint32_t key = lane + 32 * i < n ? ((b & 0x80000000u) ? ~b : (b | 0x80000000u)) : 0u;
    c[i] = key == 0u ? 0ull : ((unsigned long long)key << 32) | (uint32_t)~(uint32_t)(lane + 32 * i);
  }
#pragma unroll
  for (int i = 1; i < NPER; ++i)  // insertion network: c[0] >= c[1] >= ...
#pragma unroll
    for (int j = i; j > 0; --j) {
      const unsigned long long a = c[j - 1], d = c[j];
      c[j - 1] = a > d ? a : d;
      c[j] = a > d ? d : a;
    }
#pragma unroll
  for (int i = 1; i < NPER; ++i) lists[(i - 1) * 32 + lane] = c[i];
  lists[(NPER - 1) * 32 + lane] = 0ull;  // a lane can win NPER times, then its head is 0
  unsigned long long head = c[0];
  int pos = 0;
  for (int j = 0; j < kt; ++j) {
    const uint32_t hk = (uint32_t)(head >> 32);
    const uint32_t m = __reduce_max_sync(0xffffffffu, hk);
    int be = -1;
    if (m != 0u) {
      const uint32_t mine = hk == m ? ~(uint32_t)head : 0xffffffffu;  // the head's index
      be = (int)__reduce_min_sync(0xffffffffu, mine);
      if (mine == (uint32_t)be) head = lists[(pos++) * 32 + lane];  // this lane's head is the pick
    } else if (lane == 0) {
      flag(SEMMOE_DEVERR_NONFINITE);  // fewer than kt scores
    }
    if (lane == 0) {
      my_v[j] = be >= 0 ? __uint_as_float((m & 0x80000000u) ? (m ^ 0x80000000u) : ~m) : -INFINITY;
      my_e[j] = be;
    }
  }
  __syncwarp();
}

// lists: the warp's [NPER][32] words of shared memory when NPER >= 8 (else unused)
template <int NPER>
__device__ __forceinline__ void warp_select(const float (&v)[NPER], int n, int kt, float* my_v, int* my_e,
                                            unsigned long long* lists) {
  if constexpr (NPER >= 8) warp_select_sorted<NPER>(v, n, kt, my_v, my_e, lists);
  else warp_select_rescan<NPER>(v, n, kt, my_v, my_e);
}

// Words of selection lists per warp (warp_select) for NPER scores per lane.
__host__ __device__ constexpr int sel_list_words(int nper) { return nper >= 8 ? 32 * nper : 1; }

// One warp routes token t: its logits (see warp_load_logits), k_t picks (see
// warp_select), then the gates, the softmax of the selected logits
// renormalised over the selection (fp32).  my_v / my_e: k_max floats / ints of
// scratch for this warp; lists: its selection lists (warp_select).
template <int NPER>  // logits held per lane: E <= 32 * NPER
__device__ void warp_topk(const float* row, int ks, size_t slice_stride, float* logits_out, int E, int t,
                          const int32_t* __restrict__ k_per_token, int k_uniform, int k_max, float* my_v, int* my_e,
                          unsigned long long* lists, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                          const PairCounts& pc) {
  const int lane = threadIdx.x % 32;
  const int kt = warp_budget(k_per_token, k_uniform, k_max, t);
  float v[NPER];
  warp_load_logits<NPER>(row, ks, slice_stride, logits_out, E, v);
  warp_select<NPER>(v, E, kt, my_v, my_e, lists);
  const float m = my_v[0];
  float den = 0.f;
  for (int j = lane; j < kt; j += 32) den += my_e[j] >= 0 ? expf(my_v[j] - m) : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  for (int j = lane; j < k_max; j += 32) {
    int e = -1;
    float g = 0.f;
    if (j < kt && my_e[j] >= 0) {
      e = my_e[j];
      g = expf(my_v[j] - m) / den;
      count_pick(pc, e, t);
    }
    topk_idx[(size_t)t * k_max + j] = e;
    topk_w[(size_t)t * k_max + j] = g;
  }
  __syncwarp();
}

template <typename TX, typename TW>
__global__ void __launch_bounds__(kRouteThreads)
route_kernel(const TX* __restrict__ x, const TW* __restrict__ w, const float* __restrict__ logits_in,
             float* __restrict__ logits_out, const int32_t* __restrict__ k_per_token, int k_uniform,
             int T, int H, int E, int k_max, int32_t* __restrict__ topk_idx,
             float* __restrict__ topk_w, PairCounts pc) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  pdl_trigger();  // the permute after it may start its setup
  const int Epad = (E + 31) / 32 * 32;
  float* lg = reinterpret_cast<float*>(smem_raw);
  float* xs = lg + kRouteTok * Epad;
  float* wsm = xs + kRouteTok * (kRouteHK + 1);
  float* sel_v = wsm + kRouteEC * (kRouteHK + 1);
  int* sel_e = reinterpret_cast<int*>(sel_v + kWarps * k_max);

  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * kRouteTok;

  if (logits_in != nullptr) {
    for (int i = tid; i < kRouteTok * Epad; i += kRouteThreads) {
      int tl = i / Epad, e = i % Epad;
      int t = t0 + tl;
      lg[i] = (t < T && e < E) ? logits_in[(size_t)t * E + e] : -INFINITY;
    }
  } else {
    // logits[t, e] = sum_h x[t, h] * w[e, h]; thread = 2 tokens x 4 experts.
    const int ty = tid / 16, tx = tid % 16;
    for (int ec0 = 0; ec0 < E; ec0 += kRouteEC) {
      float acc[2][4] = {};
      for (int k0 = 0; k0 < H; k0 += kRouteHK) {
        for (int i = tid; i < kRouteTok * kRouteHK; i += kRouteThreads) {
          int r = i / kRouteHK, k = i % kRouteHK;
          int t = t0 + r, h = k0 + k;
          xs[r * (kRouteHK + 1) + k] = (t < T && h < H) ? to_f32(x[(size_t)t * H + h]) : 0.f;
        }
        for (int i = tid; i < kRouteEC * kRouteHK; i += kRouteThreads) {
          int r = i / kRouteHK, k = i % kRouteHK;
          int e = ec0 + r, h = k0 + k;
          wsm[r * (kRouteHK + 1) + k] = (e < E && h < H) ? to_f32(w[(size_t)e * H + h]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < kRouteHK; ++k) {
          float a0 = xs[(ty * 2 + 0) * (kRouteHK + 1) + k];
          float a1 = xs[(ty * 2 + 1) * (kRouteHK + 1) + k];
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            float bv = wsm[(tx + 16 * b) * (kRouteHK + 1) + k];
            acc[0][b] = fmaf(a0, bv, acc[0][b]);
            acc[1][b] = fmaf(a1, bv, acc[1][b]);
          }
        }
        __syncthreads();
      }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          int tl = ty * 2 + a, e = ec0 + tx + 16 * b;
          if (e < Epad) lg[tl * Epad + e] = (e < E) ? acc[a][b] : -INFINITY;
          if (logits_out != nullptr && e < E && t0 + tl < T)
            logits_out[(size_t)(t0 + tl) * E + e] = acc[a][b];
        }
    }
  }
  __syncthreads();

  // Top-k_t per token, one warp per token.
  __shared__ unsigned long long sel_lists[kWarps * sel_list_words(kRouteMaxE / 32)];
  const int warp = tid / 32;
  for (int tl = warp; tl < kRouteTok; tl += kWarps) {
    const int t = t0 + tl;
    if (t >= T) break;
    warp_topk<kRouteMaxE / 32>(lg + tl * Epad, 1, 0, nullptr, E, t, k_per_token, k_uniform, k_max,
                               sel_v + warp * k_max, sel_e + warp * k_max,
                               sel_lists + warp * sel_list_words(kRouteMaxE / 32), topk_idx, topk_w, pc);
  }
}

// Top-k of precomputed fp32 logits [T,E] (the sum of ks partial [T,E] slices):
// one warp per token, 8 tokens per CTA,
// so every token's (latency-bound) selection runs concurrently with the others.
constexpr int kTopkWarps = 8;

template <int NPER>
__global__ void __launch_bounds__(kTopkWarps * 32)
topk_kernel(const float* __restrict__ logits, int ks, float* __restrict__ logits_out,
            const int32_t* __restrict__ k_per_token, int k_uniform, int T, int E, int k_max,
            int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, PairCounts pc) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ unsigned long long sel_lists[kTopkWarps * sel_list_words(NPER)];
  float* sel_v = reinterpret_cast<float*>(smem_raw);
  int* sel_e = reinterpret_cast<int*>(sel_v + kTopkWarps * k_max);
  const int warp = threadIdx.x / 32;
  const int t = blockIdx.x * kTopkWarps + warp;
  if (t >= T) return;
  warp_topk<NPER>(logits + (size_t)t * E, ks, (size_t)T * E, logits_out != nullptr ? logits_out + (size_t)t * E : nullptr,
            E, t, k_per_token, k_uniform, k_max, sel_v + warp * k_max, sel_e + warp * k_max,
            sel_lists + warp * sel_list_words(NPER), topk_idx, topk_w, pc);
}

// MoE-Prism's training-free hierarchical gating, one warp per token: the
// parent logits (summed over K slices) go to shared memory; sub-expert s of
// parent s / N scores l[s / N] + sub_logw[s] (fp32); the k_t best scores are
// picked as in warp_select; each pick carries its parent's softmax weight
// renormalised over the distinct parents picked.
template <int NPER>  // sub-experts (and parents) held per lane: Ep * N <= 32 * NPER
__global__ void __launch_bounds__(kTopkWarps * 32)
hier_topk_kernel(const float* __restrict__ logits, int ks, float* __restrict__ logits_out,
                 const float* __restrict__ sub_logw, int N, const int32_t* __restrict__ k_per_token, int k_uniform,
                 int T, int Ep, int k_max, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                 PairCounts pc) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ unsigned long long sel_lists[kTopkWarps * sel_list_words(NPER)];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  float* base = reinterpret_cast<float*>(smem_raw);
  float* lg = base + warp * Ep;
  float* sel_v = base + kTopkWarps * Ep + warp * k_max;
  int* sel_e = reinterpret_cast<int*>(base + kTopkWarps * (Ep + k_max)) + warp * k_max;
  const int t = blockIdx.x * kTopkWarps + warp;
  if (t >= T) return;
  const int E = Ep * N;
  const int kt = warp_budget(k_per_token, k_uniform, k_max, t);
  {
    float v[NPER];
    warp_load_logits<NPER>(logits + (size_t)t * Ep, ks, (size_t)T * Ep,
                           logits_out != nullptr ? logits_out + (size_t)t * Ep : nullptr, Ep, v);
#pragma unroll
    for (int i = 0; i < NPER; ++i)
      if (lane + 32 * i < Ep) lg[lane + 32 * i] = v[i];
  }
  __syncwarp();
  float sc[NPER];
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
    const int sx = lane + 32 * i;
    sc[i] = -INFINITY;
    if (sx < E) {
      const float v = __fadd_rn(lg[sx / N], sub_logw[sx]);
      if (isfinite(v)) sc[i] = v;
      else flag(SEMMOE_DEVERR_NONFINITE);
    }
  }
  warp_select<NPER>(sc, E, kt, sel_v, sel_e, sel_lists + warp * sel_list_words(NPER));
  float m = -INFINITY;
  for (int j = lane; j < kt; j += 32)
    if (sel_e[j] >= 0) m = fmaxf(m, lg[sel_e[j] / N]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float den = 0.f;
  for (int j = lane; j < kt; j += 32) {
    const int sx = sel_e[j];
    if (sx < 0) continue;
    const int pe = sx / N;
    bool first = true;  // the parent's first pick counts once in the denominator
    for (int i = 0; i < j && first; ++i) first = !(sel_e[i] >= 0 && sel_e[i] / N == pe);
    if (first) den += expf(lg[pe] - m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  for (int j = lane; j < k_max; j += 32) {
    int sx = -1;
    float g = 0.f;
    if (j < kt && sel_e[j] >= 0) {
      sx = sel_e[j];
      g = expf(lg[sx / N] - m) / den;
      count_pick(pc, sx, t);
    }
    topk_idx[(size_t)t * k_max + j] = sx;
    topk_w[(size_t)t * k_max + j] = g;
  }
}

__global__ void affinity_lookup_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ lut,
                                       int V, int R, int T, int32_t* __restrict__ pred) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
    int id = ids[t];
    int r = 0;
    if (id < 0 || id >= V) {
      flag(SEMMOE_DEVERR_TOKEN_ID);
    } else {
      r = lut[id];
      if (r < 0 || r >= R) {
        flag(SEMMOE_DEVERR_LUT);
        r = 0;
      }
    }
    pred[t] = r;
  }
}

constexpr int kMaxR = 64;

// Activations per (source rank, destination rank), one pair per thread per
// pass: equal (src, dst) keys of a warp are merged with __match_any_sync before
// the shared-memory add, and each CTA adds its non-zero counts -- and its
// off-diagonal row sums, the remote activations -- to the zeroed outputs.
constexpr int kCountThreads = 256;

__global__ void __launch_bounds__(kCountThreads)
remote_count_kernel(const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ pred,
                    const int32_t* __restrict__ expert_rank, int T, int k_max, int E, int R,
                    int32_t* __restrict__ counts, int32_t* __restrict__ remote) {
  __shared__ int c[kMaxR * kMaxR];
  __shared__ int rank_s[kRouteMaxE];
  for (int i = threadIdx.x; i < R * R; i += kCountThreads) c[i] = 0;
  for (int e = threadIdx.x; e < E; e += kCountThreads) rank_s[e] = expert_rank[e];
  __syncthreads();
  const long long n = (long long)T * k_max;
  const long long stride = (long long)gridDim.x * kCountThreads;
  const long long first = (long long)blockIdx.x * kCountThreads;
  for (long long p0 = first; p0 < n; p0 += stride) {  // uniform trip count within a warp
    const long long p = p0 + threadIdx.x;
    int key = -1;
    if (p < n) {
      const int e = topk_idx[p];
      if (e >= E) {
        flag(SEMMOE_DEVERR_EXPERT);
      } else if (e >= 0) {
        const int src = pred[p / k_max];
        const int dst = rank_s[e];
        if (src < 0 || src >= R || dst < 0 || dst >= R) flag(SEMMOE_DEVERR_LUT);
        else key = src * R + dst;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && (peers & lanemask_lt()) == 0) atomicAdd(&c[key], __popc(peers));
  }
  __syncthreads();
  for (int i = threadIdx.x; i < R * R; i += kCountThreads)
    if (c[i]) atomicAdd(&counts[i], c[i]);
  if (threadIdx.x < R) {
    int sum = 0;
    for (int d = 0; d < R; ++d) sum += d != (int)threadIdx.x ? c[threadIdx.x * R + d] : 0;
    if (sum) atomicAdd(&remote[threadIdx.x], sum);
  }
}

template <typename TX, typename TW>
cudaError_t launch_route_t(const void* x, const void* w, const float* li, float* lo, const int32_t* kpt,
                           int ku, int T, int H, int E, int k_max, int32_t* idx, float* wt,
                           cudaStream_t s, PairCounts pc = PairCounts()) {
  size_t sm = route_smem_bytes(E, k_max);
  auto kern = route_kernel<TX, TW>;
  {  // raise the limit once to the largest layout (E = k_max = 256; with the 16 KB of
     // static selection lists, layouts above 32 KB need it)
    static std::atomic<unsigned long long> smem_set{0};
    cudaError_t e = ensure_smem_limit(kern, (int)route_smem_bytes(kRouteMaxE, kRouteMaxE), smem_set);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((T + kRouteTok - 1) / kRouteTok);
  kern<<<grid, kRouteThreads, sm, s>>>(static_cast<const TX*>(x), static_cast<const TW*>(w), li, lo, kpt,
                                       ku, T, H, E, k_max, idx, wt, pc);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

int route_take_errors(cudaStream_t s, int* bits) {
  if (take_error_word(g_err, s, bits)) return -1;
  return route_tc_take_errors(s, bits);
}

// bf16 activations with 16-byte rows take the tensor-core router; the rest the
// CUDA-core kernel that fuses the GEMM with the top-k.
static bool route_on_tensor_cores(int x_dtype, int H) { return x_dtype == SEMMOE_BF16 && H % 8 == 0; }

// Workspace: [fp32 partial logits ks x T x E][three-part bf16 split of an fp32 router weight].
static size_t route_partials_bytes(int T, int H, int E, int w_dtype) {
  return align_up((size_t)route_tc_k_slices(T, H, E, w_dtype) * (T > 0 ? T : 1) * E * sizeof(float), 256);
}

size_t route_ws_bytes(int T, int H, int E, int x_dtype, int w_dtype) {
  if (!route_on_tensor_cores(x_dtype, H)) return 0;
  return route_partials_bytes(T, H, E, w_dtype) + route_tc_split_bytes(H, E, w_dtype);
}

// Tensor-core logits into the workspace: fp32 partial sums over *ks K slices,
// laid out [ks][T][E].
static cudaError_t route_partials_tc(const void* x, const void* w, int w_dtype, int T, int H, int E, void* ws,
                                     const float** partials, int* ks, cudaStream_t s) {
  unsigned char* w8 = static_cast<unsigned char*>(ws);
  float* p = reinterpret_cast<float*>(w8);
  void* split = w8 + route_partials_bytes(T, H, E, w_dtype);
  int k = route_tc_k_slices(T, H, E, w_dtype);
  cudaError_t e = launch_route_logits_tc(x, w, w_dtype, T, H, E, p, k, split, s);
  if (e != cudaSuccess) return e;
  const int kb_all = (H + 63) / 64, per = (kb_all + k - 1) / k;
  *ks = (kb_all + per - 1) / per;  // the slices the launcher actually used
  *partials = p;
  return cudaSuccess;
}

// The count table for the permute, zeroed on the stream (the top-k kernels add to it).
static cudaError_t pair_counts_begin(int32_t* counts, int T, int E, PairCounts* pc, cudaStream_t s) {
  if (counts == nullptr) return cudaSuccess;
  pc->p = counts;
  pc->stride = pair_counts_stride(T);
  return cudaMemsetAsync(counts, 0, pair_counts_bytes(T, E), s);
}

cudaError_t launch_route(const void* x, int x_dtype, const void* w, int w_dtype, const float* logits_in,
                         float* logits_out, const int32_t* kpt, int k_uniform, int T, int H, int E, int k_max,
                         int32_t* topk_idx, float* topk_w, int32_t* pair_counts, void* ws, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  // The one-kernel router needs at least half the SMs' worth of 128-token tiles
  // (it has no K slices: at the DeepSeek shape, 32 tiles, 22.8 us against 17 us
  // for the split-K GEMM and a top-k kernel); below that its cluster form splits
  // H over 2-8 CTAs per tile (route stage 18.6 against 20.6 us there, 14.5
  // against 16.7 us at 64 tokens); the split-K path stays for the rest.
  if (logits_in == nullptr && route_on_tensor_cores(x_dtype, H)) {
    void* split = static_cast<unsigned char*>(ws) + route_partials_bytes(T, H, E, w_dtype);
    const int cstride = pair_counts != nullptr ? pair_counts_stride(T) : 0;
    if (route_topk_tc_ok(E, k_max, w_dtype) && 2LL * ((T + 127) / 128) >= sm_count())
      return launch_route_topk_tc(x, w, w_dtype, T, H, E, k_max, logits_out, kpt, k_uniform, topk_idx, topk_w,
                                  pair_counts, cstride, split, s);
    // fewer tiles (slices of H), or several passes of experts: a cluster of CTAs per tile
    const int ks = route_topk_cl_slices(T, H, E, k_max, w_dtype);
    if (ks >= 1)
      return launch_route_topk_cl(x, w, w_dtype, T, H, E, k_max, ks, logits_out, kpt, k_uniform, topk_idx, topk_w,
                                  pair_counts, cstride, split, s);
  }
  PairCounts pc;
  cudaError_t ec = pair_counts_begin(pair_counts, T, E, &pc, s);
  if (ec != cudaSuccess) return ec;
  int ks = 1;
  if (logits_in == nullptr && route_on_tensor_cores(x_dtype, H)) {
    cudaError_t e = route_partials_tc(x, w, w_dtype, T, H, E, ws, &logits_in, &ks, s);
    if (e != cudaSuccess) return e;
  } else if (logits_in != nullptr && logits_out == logits_in) {
    logits_out = nullptr;
  }
  if (logits_in != nullptr) {  // top-k of the (summed) logits; x and w unused here
    const size_t sm = (size_t)kTopkWarps * k_max * (sizeof(float) + sizeof(int));
    const dim3 grid((T + kTopkWarps - 1) / kTopkWarps), block(kTopkWarps * 32);
    if (E <= 32)
      topk_kernel<1><<<grid, block, sm, s>>>(logits_in, ks, logits_out, kpt, k_uniform, T, E, k_max, topk_idx, topk_w,
                                               pc);
    else if (E <= 64)
      topk_kernel<2><<<grid, block, sm, s>>>(logits_in, ks, logits_out, kpt, k_uniform, T, E, k_max, topk_idx, topk_w,
                                               pc);
    else if (E <= 128)
      topk_kernel<4><<<grid, block, sm, s>>>(logits_in, ks, logits_out, kpt, k_uniform, T, E, k_max, topk_idx, topk_w,
                                               pc);
    else
      topk_kernel<8><<<grid, block, sm, s>>>(logits_in, ks, logits_out, kpt, k_uniform, T, E, k_max, topk_idx, topk_w,
                                               pc);
    count_launches(1);
    return cudaGetLastError();
  }
  if (x_dtype == SEMMOE_BF16 && w_dtype == SEMMOE_F32)
    return launch_route_t<__nv_bfloat16, float>(x, w, nullptr, logits_out, kpt, k_uniform, T, H, E, k_max,
                                                topk_idx, topk_w, s, pc);
  if (x_dtype == SEMMOE_BF16 && w_dtype == SEMMOE_BF16)
    return launch_route_t<__nv_bfloat16, __nv_bfloat16>(x, w, nullptr, logits_out, kpt, k_uniform, T, H, E,
                                                        k_max, topk_idx, topk_w, s, pc);
  if (x_dtype == SEMMOE_F32 && w_dtype == SEMMOE_F32)
    return launch_route_t<float, float>(x, w, nullptr, logits_out, kpt, k_uniform, T, H, E, k_max, topk_idx,
                                        topk_w, s, pc);
  return launch_route_t<float, __nv_bfloat16>(x, w, nullptr, logits_out, kpt, k_uniform, T, H, E, k_max,
                                              topk_idx, topk_w, s, pc);
}

size_t route_hier_ws_bytes(int T, int H, int Ep, int x_dtype, int w_dtype) {
  if (route_on_tensor_cores(x_dtype, H)) return route_ws_bytes(T, H, Ep, x_dtype, w_dtype);
  // CUDA-core logits [T][Ep] plus the (unused) one-expert picks of that kernel
  const size_t t = T > 0 ? T : 1;
  return align_up(t * Ep * sizeof(float), 256) + 2 * align_up(t * sizeof(float), 256);
}

cudaError_t launch_route_hier(const void* x, int x_dtype, const void* w, int w_dtype, const float* logits_in,
                              float* logits_out, const float* sub_logw, int N, const int32_t* kpt, int k_uniform,
                              int T, int H, int Ep, int k_max, int32_t* topk_idx, float* topk_w,
                              int32_t* pair_counts, void* ws, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  int ks = 1;
  if (logits_in == nullptr) {
    if (route_on_tensor_cores(x_dtype, H)) {
      cudaError_t e = route_partials_tc(x, w, w_dtype, T, H, Ep, ws, &logits_in, &ks, s);
      if (e != cudaSuccess) return e;
    } else {
      unsigned char* w8 = static_cast<unsigned char*>(ws);
      float* lg = reinterpret_cast<float*>(w8);
      unsigned char* rest = w8 + align_up((size_t)T * Ep * sizeof(float), 256);
      int32_t* idx1 = reinterpret_cast<int32_t*>(rest);
      float* w1 = reinterpret_cast<float*>(rest + align_up((size_t)T * sizeof(float), 256));
      cudaError_t e;
      if (x_dtype == SEMMOE_BF16 && w_dtype == SEMMOE_F32)
        e = launch_route_t<__nv_bfloat16, float>(x, w, nullptr, lg, nullptr, 1, T, H, Ep, 1, idx1, w1, s);
      else if (x_dtype == SEMMOE_BF16)
        e = launch_route_t<__nv_bfloat16, __nv_bfloat16>(x, w, nullptr, lg, nullptr, 1, T, H, Ep, 1, idx1, w1, s);
      else if (w_dtype == SEMMOE_F32)
        e = launch_route_t<float, float>(x, w, nullptr, lg, nullptr, 1, T, H, Ep, 1, idx1, w1, s);
      else
        e = launch_route_t<float, __nv_bfloat16>(x, w, nullptr, lg, nullptr, 1, T, H, Ep, 1, idx1, w1, s);
      if (e != cudaSuccess) return e;
      logits_in = lg;
    }
  } else if (logits_out == logits_in) {
    logits_out = nullptr;
  }
  const int E = Ep * N;
  PairCounts pc;
  cudaError_t ec = pair_counts_begin(pair_counts, T, E, &pc, s);
  if (ec != cudaSuccess) return ec;
  const size_t sm = (size_t)kTopkWarps * (Ep + 2 * k_max) * sizeof(float);
  const dim3 grid((T + kTopkWarps - 1) / kTopkWarps), block(kTopkWarps * 32);
  if (E <= 32)
    hier_topk_kernel<1><<<grid, block, sm, s>>>(logits_in, ks, logits_out, sub_logw, N, kpt, k_uniform, T, Ep,
                                                k_max, topk_idx, topk_w, pc);
  else if (E <= 64)
    hier_topk_kernel<2><<<grid, block, sm, s>>>(logits_in, ks, logits_out, sub_logw, N, kpt, k_uniform, T, Ep,
                                                k_max, topk_idx, topk_w, pc);
  else if (E <= 128)
    hier_topk_kernel<4><<<grid, block, sm, s>>>(logits_in, ks, logits_out, sub_logw, N, kpt, k_uniform, T, Ep,
                                                k_max, topk_idx, topk_w, pc);
  else
    hier_topk_kernel<8><<<grid, block, sm, s>>>(logits_in, ks, logits_out, sub_logw, N, kpt, k_uniform, T, Ep,
                                                k_max, topk_idx, topk_w, pc);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_affinity_lookup(const int32_t* ids, const int32_t* lut, int V, int R, int T, int32_t* pred,
                                   cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  int blocks = (T + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  affinity_lookup_kernel<<<blocks, 256, 0, s>>>(ids, lut, V, R, T, pred);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_remote_count(const int32_t* topk_idx, const int32_t* pred, const int32_t* expert_rank, int T,
                                int k_max, int E, int R, int32_t* counts, int32_t* remote, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * R * R, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(remote, 0, sizeof(int32_t) * R, s);
  if (e != cudaSuccess) return e;
  const long long n = (long long)T * k_max;
  if (n == 0) return cudaSuccess;
  long long blocks = (n + kCountThreads - 1) / kCountThreads;
  const long long cap = 4LL * sm_count();
  if (blocks > cap) blocks = cap;
  remote_count_kernel<<<(int)blocks, kCountThreads, 0, s>>>(topk_idx, pred, expert_rank, T, k_max, E, R, counts,
                                                            remote);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace semmoe
