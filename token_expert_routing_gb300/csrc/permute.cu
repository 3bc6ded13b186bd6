// Stable counting sort of the (token, expert) pairs by (destination rank,
// expert) and the row gather that follows it: the single-device form of the
// Shuffled-Reduce-Scatter token shuffle (Semantic Parallelism (ko) §2.2,
// (de) §2 B, (ja) §2.2 B).  The rank-major expert order is the physical
// layout that (ja) §2.2 A obtains by shuffling the gate matrix's columns.
//
// Three passes over the pair ids, none waiting on another CTA:
//   1. perm_hist:    each CTA counts its chunk of pairs per physical bucket
//   2. perm_scan:    one CTA turns the [chunk][bucket] counts into bucket
//                    offsets and per-chunk starting positions
//   3. perm_scatter: each CTA ranks its pairs stably within its chunk (warp
//                    match + per-warp bucket counts) and writes both maps
// then perm_gather copies x rows into sorted order (one warp per row,
// 16-byte vectors).
#include <mutex>

#include "common.cuh"
#include "internal.h"

// Scratch of semmoe_permute_noalloc: the per-chunk bucket counts live in this
// file-scope device array instead of a caller workspace.  Every GPU that loads
// the library holds it until the process exits.
static constexpr size_t kNoAllocScratchBytes = 1u << 20;  // 1 MiB
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

namespace semmoe {
namespace {

__device__ int g_err;
__device__ __forceinline__ void flag(int bit) { atomicOr(&g_err, bit); }

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRounds = 8;
constexpr int kChunk = kThreads * kRounds;  // pairs per CTA
constexpr int kMaxE = 256;

inline int n_chunks(long long n_pairs) { return (int)((n_pairs + kChunk - 1) / kChunk); }

// phys_s[e] = position of expert e in the (expert_rank[e], e) order.
__device__ void physical_positions(const int32_t* __restrict__ expert_rank, int E, int R, int* rank_s,
                                   int* phys_s) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int r = expert_rank[e];
    if (r < 0 || r >= R) {
      flag(SEMMOE_DEVERR_LUT);
      r = r < 0 ? 0 : R - 1;
    }
    rank_s[e] = r;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int re = rank_s[e], pos = 0;
    for (int f = 0; f < E; ++f) {
      int rf = rank_s[f];
      pos += (rf < re) || (rf == re && f < e);
    }
    phys_s[e] = pos;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads)
perm_hist_kernel(const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ expert_rank,
                 long long n_pairs, int E, int R, int32_t* __restrict__ hist) {
  __shared__ int rank_s[kMaxE], phys_s[kMaxE], h[kMaxE];
  physical_positions(expert_rank, E, R, rank_s, phys_s);
  for (int b = threadIdx.x; b < E; b += kThreads) h[b] = 0;
  __syncthreads();
  const long long base = (long long)blockIdx.x * kChunk;
  for (int i = threadIdx.x; i < kChunk; i += kThreads) {
    long long p = base + i;
    if (p >= n_pairs) break;
    int e = topk_idx[p];
    if (e < 0) continue;
    if (e >= E) { flag(SEMMOE_DEVERR_EXPERT); continue; }
    atomicAdd(&h[phys_s[e]], 1);
  }
  __syncthreads();
  for (int b = threadIdx.x; b < E; b += kThreads) hist[(size_t)blockIdx.x * E + b] = h[b];
}

// One CTA: column-wise exclusive scan of hist (in place -> per-chunk start
// offsets), bucket offsets, and the small per-expert / per-rank tables.
__global__ void __launch_bounds__(kThreads)
perm_scan_kernel(int32_t* __restrict__ hist, int nchunks, const int32_t* __restrict__ expert_rank, int E,
                 int R, int P, int32_t* __restrict__ expert_offsets, int32_t* __restrict__ rank_offsets,
                 int32_t* __restrict__ phys_to_expert, int32_t* __restrict__ expert_counts) {
  __shared__ int rank_s[kMaxE], phys_s[kMaxE], total[kMaxE], excl[kMaxE + 1];
  physical_positions(expert_rank, E, R, rank_s, phys_s);
  const int b = threadIdx.x;
  if (b < E) {
    int run = 0;
    for (int c = 0; c < nchunks; ++c) {
      int v = hist[(size_t)c * E + b];
      hist[(size_t)c * E + b] = run;
      run += v;
    }
    total[b] = run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {  // E <= 256 buckets: a serial scan is cheapest here
    int s = 0;
    for (int i = 0; i < E; ++i) { excl[i] = s; s += total[i]; }
    excl[E] = s;
    if (s != P) flag(SEMMOE_DEVERR_PAIRS);
  }
  __syncthreads();
  if (b < E) {
    const int off = excl[b];
    for (int c = 0; c < nchunks; ++c) hist[(size_t)c * E + b] += off;
    expert_offsets[b] = off;
  }
  if (b == 0) expert_offsets[E] = excl[E];
  for (int e = threadIdx.x; e < E; e += kThreads) {
    phys_to_expert[phys_s[e]] = e;
    expert_counts[e] = total[phys_s[e]];
  }
  for (int r = threadIdx.x; r <= R; r += kThreads) {
    int nb = 0;  // buckets of ranks below r
    for (int e = 0; e < E; ++e) nb += rank_s[e] < r;
    rank_offsets[r] = excl[nb];
  }
}

__global__ void __launch_bounds__(kThreads)
perm_scatter_kernel(const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ expert_rank,
                    long long n_pairs, int E, int R, int P, const int32_t* __restrict__ chunk_off,
                    int32_t* __restrict__ sorted_to_pair, int32_t* __restrict__ pair_to_sorted) {
  __shared__ int rank_s[kMaxE], phys_s[kMaxE], run[kMaxE];
  __shared__ int wcnt[kWarps][kMaxE];
  physical_positions(expert_rank, E, R, rank_s, phys_s);
  for (int i = threadIdx.x; i < E; i += kThreads) {
    run[i] = chunk_off[(size_t)blockIdx.x * E + i];
    for (int w = 0; w < kWarps; ++w) wcnt[w][i] = 0;
  }
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const long long base = (long long)blockIdx.x * kChunk;
  for (int r = 0; r < kRounds; ++r) {
    const long long p = base + (long long)r * kThreads + threadIdx.x;
    int key = E;  // E = "no bucket" (padding slot or past the end)
    if (p < n_pairs) {
      int e = topk_idx[p];
      if (e >= E) flag(SEMMOE_DEVERR_EXPERT);
      else if (e >= 0) key = phys_s[e];
    }
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int rank_in_warp = __popc(peers & lanemask_lt());
    if (key < E && rank_in_warp == 0) wcnt[warp][key] = __popc(peers);
    __syncthreads();
    if (p < n_pairs) {
      int pos = -1;
      if (key < E) {
        pos = run[key] + rank_in_warp;
        for (int w = 0; w < warp; ++w) pos += wcnt[w][key];
        if (pos >= P) { flag(SEMMOE_DEVERR_PAIRS); pos = -1; }
        else sorted_to_pair[pos] = (int32_t)p;
      }
      pair_to_sorted[p] = pos;
    }
    __syncthreads();
    for (int b = threadIdx.x; b < E; b += kThreads) {
      int s = 0;
      for (int w = 0; w < kWarps; ++w) { s += wcnt[w][b]; wcnt[w][b] = 0; }
      run[b] += s;
    }
    __syncthreads();
  }
}

// x_perm[q, :] = x[sorted_to_pair[q] / k_max, :], one warp per sorted row.
__global__ void __launch_bounds__(kThreads)
perm_gather_kernel(const unsigned char* __restrict__ x, const int32_t* __restrict__ sorted_to_pair, int P,
                   int T, int k_max, int row_bytes, unsigned char* __restrict__ x_perm) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int q = blockIdx.x * kWarps + warp; q < P; q += gridDim.x * kWarps) {
    const int p = sorted_to_pair[q];
    const int t = p / k_max;
    uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)q * row_bytes);
    if (p < 0 || t >= T) {
      if (lane == 0) flag(SEMMOE_DEVERR_PAIRS);
      for (int off = lane; off < row_bytes / 16; off += 32) dst[off] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * row_bytes);
    for (int off = lane; off < row_bytes / 16; off += 32) dst[off] = src[off];
  }
}

int sm_count() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

}  // namespace

int permute_take_errors(cudaStream_t s, int* bits) { return take_error_word(g_err, s, bits); }

size_t permute_ws_bytes(int T, int k_max, int E) {
  long long n = (long long)T * k_max;
  int nc = n_chunks(n > 0 ? n : 1);
  return align_up((size_t)nc * E * sizeof(int32_t), 256);
}

cudaError_t launch_permute(const int32_t* topk_idx, const int32_t* expert_rank, const void* x, int dtype, int T,
                           int H, int E, int R, int k_max, int P, int32_t* expert_offsets,
                           int32_t* rank_offsets, int32_t* phys_to_expert, int32_t* expert_counts,
                           int32_t* sorted_to_pair, int32_t* pair_to_sorted, void* x_perm, void* ws,
                           cudaStream_t s) {
  const long long n_pairs = (long long)T * k_max;
  const int nc = n_chunks(n_pairs > 0 ? n_pairs : 1);
  int32_t* hist = static_cast<int32_t*>(ws);
  if (n_pairs > 0) {
    perm_hist_kernel<<<nc, kThreads, 0, s>>>(topk_idx, expert_rank, n_pairs, E, R, hist);
    count_launches(1);
  } else {
    cudaError_t e = cudaMemsetAsync(hist, 0, sizeof(int32_t) * E, s);
    if (e != cudaSuccess) return e;
  }
  perm_scan_kernel<<<1, kThreads, 0, s>>>(hist, n_pairs > 0 ? nc : 1, expert_rank, E, R, P, expert_offsets,
                                          rank_offsets, phys_to_expert, expert_counts);
  count_launches(1);
  if (n_pairs > 0) {
    perm_scatter_kernel<<<nc, kThreads, 0, s>>>(topk_idx, expert_rank, n_pairs, E, R, P, hist, sorted_to_pair,
                                                pair_to_sorted);
    count_launches(1);
  }
  if (x != nullptr && x_perm != nullptr && P > 0) {
    const int row_bytes = H * (dtype == SEMMOE_BF16 ? 2 : 4);
    int blocks = (P + kWarps - 1) / kWarps;
    const int cap = sm_count() * 16;
    if (blocks > cap) blocks = cap;
    perm_gather_kernel<<<blocks, kThreads, 0, s>>>(static_cast<const unsigned char*>(x), sorted_to_pair, P, T,
                                                   k_max, row_bytes, static_cast<unsigned char*>(x_perm));
    count_launches(1);
  }
  return cudaGetLastError();
}

size_t permute_noalloc_max_scratch() { return kNoAllocScratchBytes; }

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
static cudaError_t noalloc_scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

cudaError_t launch_permute_noalloc(const int32_t* topk_idx, const int32_t* expert_rank, const void* x, int dtype,
                                   int T, int H, int E, int R, int k_max, int P, int32_t* expert_offsets,
                                   int32_t* rank_offsets, int32_t* phys_to_expert, int32_t* expert_counts,
                                   int32_t* sorted_to_pair, int32_t* pair_to_sorted, void* x_perm, cudaStream_t s) {
  void* scratch = nullptr;
  cudaError_t e = noalloc_scratch_address(&scratch);
  if (e != cudaSuccess) return e;
  // The kernels overwrite every scratch entry they later read (the zero-pair
  // case clears its one row), so stale contents of an earlier call never leak.
  return launch_permute(topk_idx, expert_rank, x, dtype, T, H, E, R, k_max, P, expert_offsets, rank_offsets,
                        phys_to_expert, expert_counts, sorted_to_pair, pair_to_sorted, x_perm, scratch, s);
}

}  // namespace semmoe
