// Stable counting sort of the (token, expert) pairs by (destination rank,
// expert) and the row gather that follows it: the single-device form of the
// Shuffled-Reduce-Scatter token shuffle (Semantic Parallelism (ko) §2.2,
// (de) §2 B, (ja) §2.2 B).  The rank-major expert order is the physical
// layout that (ja) §2.2 A obtains by shuffling the gate matrix's columns.
//
// Two passes over the pair ids, neither waiting on another CTA:
//   1. perm_hist:    each CTA counts its chunk of pairs per physical bucket
//   2. perm_scatter: each CTA scans the [chunk][bucket] counts for its own
//                    starting positions, ranks its pairs stably within the
//                    chunk (warp match + per-warp bucket counts) and writes
//                    both maps; CTA 0 writes the bucket and rank tables
// then perm_copy writes each x row to its tokens' sorted rows (one warp per
// token, 16-byte vectors).
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

// Scratch of semmoe_permute_noalloc: the per-chunk bucket counts live in this
// file-scope device array instead of a caller workspace.  Every GPU that loads
// the library holds it until the process exits.
// The permute splits the pairs into at most 96 chunks, so it needs at most
// 96 * E * 4 bytes of scratch: 96 KiB covers every E up to the 256 it accepts.
static constexpr size_t kNoAllocScratchBytes = 96u * 256u * 4u;  // 96 KiB
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

namespace semmoe {
namespace {

__device__ int g_err;
__device__ __forceinline__ void flag(int bit) { atomicOr(&g_err, bit); }

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxE = 256;
constexpr int kTargetChunks = 96;  // enough CTAs to cover the GPU, few enough to scan cheaply
constexpr int kPre = 8;            // pair ids loaded ahead per thread (rounds of a chunk)
static_assert(kTargetChunks * kMaxE * 4 <= kNoAllocScratchBytes, "no-alloc scratch too small");

// Pairs per CTA: a multiple of kThreads (one "round" each) giving about
// kTargetChunks chunks.
inline int rounds_per_chunk(long long n_pairs) {
  const long long r = (n_pairs + (long long)kTargetChunks * kThreads - 1) / ((long long)kTargetChunks * kThreads);
  return r < 1 ? 1 : (int)r;
}
inline int n_chunks(long long n_pairs) {
  const long long chunk = (long long)rounds_per_chunk(n_pairs) * kThreads;
  return (int)((n_pairs + chunk - 1) / chunk);
}

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
#pragma unroll 16
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
                 long long n_pairs, int rounds, int E, int R, int32_t* __restrict__ hist) {
  __shared__ int rank_s[kMaxE], phys_s[kMaxE], h[kMaxE];
  physical_positions(expert_rank, E, R, rank_s, phys_s);
  for (int b = threadIdx.x; b < E; b += kThreads) h[b] = 0;
  __syncthreads();
  const int chunk = rounds * kThreads;
  const long long base = (long long)blockIdx.x * chunk;
  for (int i0 = 0; i0 < chunk; i0 += kPre * kThreads) {  // kPre loads in flight per thread
    int ev[kPre];
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      const int i = i0 + u * kThreads + threadIdx.x;
      ev[u] = (i < chunk && base + i < n_pairs) ? topk_idx[base + i] : -1;
    }
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      const int e = ev[u];
      if (e < 0) continue;
      if (e >= E) { flag(SEMMOE_DEVERR_EXPERT); continue; }
      atomicAdd(&h[phys_s[e]], 1);
    }
  }
  __syncthreads();
  for (int b = threadIdx.x; b < E; b += kThreads) hist[(size_t)blockIdx.x * E + b] = h[b];
}

// Each CTA ranks the pairs of its chunk.  Its starting position in every bucket
// is derived from the per-chunk histograms of pass 1: it sums, per bucket, the
// counts of all chunks (totals) and of the chunks before its own, and scans the
// totals over buckets.  CTA 0 also writes the bucket / rank tables.  Nothing
// waits on another CTA: every CTA recomputes the (small) scan for itself.
__global__ void __launch_bounds__(kThreads)
perm_scatter_kernel(const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ expert_rank,
                    long long n_pairs, int rounds, int nchunks, int E, int R, int P,
                    const int32_t* __restrict__ hist,
                    int32_t* __restrict__ expert_offsets, int32_t* __restrict__ rank_offsets,
                    int32_t* __restrict__ phys_to_expert, int32_t* __restrict__ expert_counts,
                    int32_t* __restrict__ sorted_to_pair, int32_t* __restrict__ pair_to_sorted) {
  __shared__ int rank_s[kMaxE], phys_s[kMaxE], run[kMaxE], total[kMaxE], scan[kThreads];
  __shared__ int wcnt[kWarps][kMaxE];
  __shared__ int part_before[kThreads], part_tot[kThreads];
  physical_positions(expert_rank, E, R, rank_s, phys_s);
  const int tid = threadIdx.x;
  // G threads per bucket (G = kThreads / E) each sum every G-th chunk's count,
  // eight loads in flight at a time; the G partial sums are added below.
  const int G = kThreads / E;
  if (tid < G * E) {
    const int b = tid % E, g = tid / E;
    int before = 0, tot = 0;
    constexpr int B = 8;
    for (int c0 = g; c0 < nchunks; c0 += B * G) {
      int v[B];
#pragma unroll
      for (int u = 0; u < B; ++u) {
        const int c = c0 + u * G;
        v[u] = c < nchunks ? hist[(size_t)c * E + b] : 0;
      }
#pragma unroll
      for (int u = 0; u < B; ++u) {
        before += c0 + u * G < (int)blockIdx.x ? v[u] : 0;
        tot += v[u];
      }
    }
    part_before[tid] = before;
    part_tot[tid] = tot;
  }
  __syncthreads();
  if (tid < E) {
    int before = 0, tot = 0;
    for (int g = 0; g < G; ++g) {
      before += part_before[g * E + tid];
      tot += part_tot[g * E + tid];
    }
    total[tid] = tot;
    run[tid] = before;
    for (int w = 0; w < kWarps; ++w) wcnt[w][tid] = 0;
  }
  __syncthreads();
  scan[tid] = tid < E ? total[tid] : 0;
  __syncthreads();
  for (int d = 1; d < kThreads; d <<= 1) {  // inclusive scan of the bucket totals
    const int v = tid >= d ? scan[tid - d] : 0;
    __syncthreads();
    scan[tid] += v;
    __syncthreads();
  }
  const int sum = scan[kThreads - 1];
  if (tid < E) run[tid] += scan[tid] - total[tid];  // bucket start + rows of earlier chunks
  if (blockIdx.x == 0) {
    if (tid < E) {
      expert_offsets[tid] = scan[tid] - total[tid];
      phys_to_expert[phys_s[tid]] = tid;
      expert_counts[tid] = total[phys_s[tid]];
    }
    if (tid == 0) {
      expert_offsets[E] = sum;
      if (sum != P) flag(SEMMOE_DEVERR_PAIRS);
    }
    for (int r = tid; r <= R; r += kThreads) {  // R + 1 entries (R may be 256)
      int nb = 0;  // buckets of ranks below r
      for (int e = 0; e < E; ++e) nb += rank_s[e] < r;
      rank_offsets[r] = nb == 0 ? 0 : scan[nb - 1];
    }
  }
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  (void)lane;
  const long long base = (long long)blockIdx.x * rounds * kThreads;
  int ev[kPre];  // the pair ids of rounds r0 .. r0 + kPre - 1, loaded together
  for (int r = 0; r < rounds; ++r) {
    if (base + (long long)r * kThreads >= n_pairs) break;  // uniform across the CTA
    if (r % kPre == 0) {
#pragma unroll
      for (int u = 0; u < kPre; ++u) {
        const long long pu = base + (long long)(r + u) * kThreads + threadIdx.x;
        ev[u] = (r + u < rounds && pu < n_pairs) ? topk_idx[pu] : -1;
      }
    }
    const long long p = base + (long long)r * kThreads + threadIdx.x;
    int key = E;  // E = "no bucket" (padding slot or past the end)
    if (p < n_pairs) {
      int e = 0;
#pragma unroll
      for (int u = 0; u < kPre; ++u)
        if (u == r % kPre) e = ev[u];  // register select, no local-memory indexing
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
      int s2 = 0;
      for (int w = 0; w < kWarps; ++w) { s2 += wcnt[w][b]; wcnt[w][b] = 0; }
      run[b] += s2;
    }
    __syncthreads();
  }
}

// x_perm[pair_to_sorted[t * k_max + j], :] = x[t, :] for every live slot j of
// token t: one warp per token reads its row once, in segments of up to 4 KB
// held in registers, and writes each segment to the token's k_t sorted rows.
// (Walking the sorted rows instead re-reads each x row k_t times, far apart
// in time, and the row writes push those reads out of L2.)
constexpr int kSegVec = 8;  // 16-byte vectors per lane per segment: 32 x 8 x 16 B = 4 KB

__global__ void __launch_bounds__(kThreads)
perm_copy_kernel(const unsigned char* __restrict__ x, const int32_t* __restrict__ pair_to_sorted, int T, int k_max,
                 int P, int row_bytes, unsigned char* __restrict__ x_perm) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n16 = row_bytes / 16;
  const int kk = k_max < 32 ? k_max : 32;
  for (int t = blockIdx.x * kWarps + warp; t < T; t += gridDim.x * kWarps) {
    const int32_t* slots = pair_to_sorted + (size_t)t * k_max;
    int q_l = -1;
    if (lane < kk) {
      q_l = slots[lane];
      if (q_l >= P) { flag(SEMMOE_DEVERR_PAIRS); q_l = -1; }
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * row_bytes);
    for (int seg = 0; seg < n16; seg += 32 * kSegVec) {
      uint4 v[kSegVec];
#pragma unroll
      for (int u = 0; u < kSegVec; ++u) {
        const int c = seg + u * 32 + lane;
        if (c < n16) v[u] = src[c];
      }
      for (int j = 0; j < kk; ++j) {
        const int q = __shfl_sync(0xffffffffu, q_l, j);
        if (q < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)q * row_bytes);
#pragma unroll
        for (int u = 0; u < kSegVec; ++u) {
          const int c = seg + u * 32 + lane;
          if (c < n16) dst[c] = v[u];
        }
      }
      for (int j = 32; j < k_max; ++j) {  // budgets above 32 experts: read the slot directly
        const int q = slots[j];
        if (q < 0) continue;
        if (q >= P) { if (lane == 0) flag(SEMMOE_DEVERR_PAIRS); continue; }
        uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)q * row_bytes);
#pragma unroll
        for (int u = 0; u < kSegVec; ++u) {
          const int c = seg + u * 32 + lane;
          if (c < n16) dst[c] = v[u];
        }
      }
    }
  }
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
    perm_hist_kernel<<<nc, kThreads, 0, s>>>(topk_idx, expert_rank, n_pairs, rounds_per_chunk(n_pairs), E, R,
                                             hist);
    count_launches(1);
  }
  perm_scatter_kernel<<<n_pairs > 0 ? nc : 1, kThreads, 0, s>>>(
      topk_idx, expert_rank, n_pairs, rounds_per_chunk(n_pairs), n_pairs > 0 ? nc : 0, E, R, P, hist,
      expert_offsets, rank_offsets,
      phys_to_expert, expert_counts, sorted_to_pair, pair_to_sorted);
  count_launches(1);
  if (x != nullptr && x_perm != nullptr && P > 0) {
    const int row_bytes = H * (dtype == SEMMOE_BF16 ? 2 : 4);
    int blocks = (T + kWarps - 1) / kWarps;
    const int cap = sm_count() * 16;
    if (blocks > cap) blocks = cap;
    perm_copy_kernel<<<blocks, kThreads, 0, s>>>(static_cast<const unsigned char*>(x), pair_to_sorted, T, k_max, P,
                                                 row_bytes, static_cast<unsigned char*>(x_perm));
    count_launches(1);
  }
  return cudaGetLastError();
}

size_t permute_noalloc_max_scratch() { return kNoAllocScratchBytes; }

// Device address of g_noalloc_scratch in the current CUDA context.  In host
// code the array's name is only a host-side stand-in, so the address is looked
// up with cudaGetSymbolAddress, with the context current, and cached.  The
// cache is keyed on the context's unique ID (cuCtxGetId), not on the device
// number: after cudaDeviceReset, or in another context on the same device, the
// library's module is loaded again and the array has another address, while a
// context's ID is never reused within the process.
// The two driver calls, fetched through the runtime (the library links no
// driver library, so it still loads on hosts without one).
template <typename F>
static F driver_fn(const char* name, int version) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(p);
}

static cudaError_t noalloc_scratch_address(void** out) {
  using CtxGetCurrent = CUresult (*)(CUcontext*);
  using CtxGetId = CUresult (*)(CUcontext, unsigned long long*);
  static const CtxGetCurrent ctx_get_current = driver_fn<CtxGetCurrent>("cuCtxGetCurrent", 4000);
  static const CtxGetId ctx_get_id = driver_fn<CtxGetId>("cuCtxGetId", 12000);
  if (ctx_get_current == nullptr || ctx_get_id == nullptr) return cudaErrorNotSupported;
  struct Entry {
    unsigned long long ctx_id;
    void* addr;
  };
  constexpr int kSlots = 16;
  static std::mutex mu;
  static Entry cache[kSlots] = {};
  static int next_slot = 0;
  CUcontext ctx = nullptr;
  if (ctx_get_current(&ctx) != CUDA_SUCCESS) return cudaErrorInitializationError;
  if (ctx == nullptr) {  // the runtime has not made a context current on this thread yet: let it
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorInitializationError;
  }
  unsigned long long id = 0;
  if (ctx_get_id(ctx, &id) != CUDA_SUCCESS) return cudaErrorInitializationError;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& en : cache)
    if (en.addr != nullptr && en.ctx_id == id) {
      *out = en.addr;
      return cudaSuccess;
    }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  cache[next_slot] = Entry{id, p};  // oldest entry replaced once all slots are used
  next_slot = (next_slot + 1) % kSlots;
  *out = p;
  return cudaSuccess;
}

cudaError_t launch_permute_noalloc(const int32_t* topk_idx, const int32_t* expert_rank, const void* x, int dtype,
                                   int T, int H, int E, int R, int k_max, int P, int32_t* expert_offsets,
                                   int32_t* rank_offsets, int32_t* phys_to_expert, int32_t* expert_counts,
                                   int32_t* sorted_to_pair, int32_t* pair_to_sorted, void* x_perm, cudaStream_t s) {
  void* scratch = nullptr;
  cudaError_t e = noalloc_scratch_address(&scratch);
  if (e != cudaSuccess) return e;
  // The kernels write every scratch entry before they read it, so stale contents of an
  // earlier call never leak into this one.
  return launch_permute(topk_idx, expert_rank, x, dtype, T, H, E, R, k_max, P, expert_offsets, rank_offsets,
                        phys_to_expert, expert_counts, sorted_to_pair, pair_to_sorted, x_perm, scratch, s);
}

}  // namespace semmoe
