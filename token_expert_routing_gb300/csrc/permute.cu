// Stable counting sort of the (token, expert) pairs by (destination rank,
// expert) and the row gather that follows it: the single-device form of the
// Shuffled-Reduce-Scatter token shuffle (Semantic Parallelism (ko) §2.2,
// (de) §2 B, (ja) §2.2 B).  The rank-major expert order is the physical
// layout that (ja) §2.2 A obtains by shuffling the gate matrix's columns.
//
// The sort starts from a count table, counts[e][c] = live pairs of expert e
// among the tokens of chunk c: the router writes it as it picks the experts
// (128-token chunks, semmoe_route's pair_counts), or, when the caller has none,
// perm_count_kernel makes it (one CTA per chunk).  perm_rank_copy_kernel then
// does the rest: each CTA derives its first row in every bucket from the table,
// ranks its own tokens' pairs stably (warp match + per-warp bucket counts),
// writes both maps, and copies its tokens' x rows to their sorted rows (bulk
// copies through shared memory) -- or, for copies of 256 MB and more,
// perm_copy_kernel does the copy as a kernel of its own (one warp per token,
// 16-byte vectors, more warps per SM).
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

// Scratch of semmoe_permute_noalloc: the count table lives in this file-scope
// device array instead of a caller workspace.  Every GPU that loads the library
// holds it until the process exits.  The table the permute makes itself has at
// most 96 chunks, so it needs at most 96 * E * 4 bytes of scratch: 96 KiB
// covers every E up to the 256 it accepts.
static constexpr size_t kNoAllocScratchBytes = 96u * 256u * 4u;  // 96 KiB
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

namespace semmoe {
namespace {

__device__ int g_err;
__device__ __forceinline__ void flag(int bit) { atomicOr(&g_err, bit); }

constexpr int kMaxE = 256;
constexpr int kHistThreads = 256;
constexpr int kThreads = 512;               // the ranking + copy kernel
constexpr int kWarps = kThreads / 32;
constexpr int kPre = 8;                     // loads in flight per thread in the counting loops
constexpr int kMaxInternalChunks = 96;      // chunks of the count table the permute makes itself
static_assert(kMaxInternalChunks * kMaxE * 4 <= kNoAllocScratchBytes, "no-alloc scratch too small");

// Row stride of a [E][chunks] count table: chunks rounded up to a multiple of 4,
// so that each expert's row starts 16-byte aligned.
inline int padded_chunks(int nc) { return (nc + 3) / 4 * 4; }

// Tokens per chunk of the count table the permute makes itself (when the caller
// passes none): SEMMOE_PAIR_COUNT_CHUNK, or more so that there are at most 96
// chunks (the table then fits the no-alloc scratch for every E <= 256).
inline int internal_chunk_tokens(int T) {
  const int c = (T + kMaxInternalChunks - 1) / kMaxInternalChunks;
  return c > SEMMOE_PAIR_COUNT_CHUNK ? c : SEMMOE_PAIR_COUNT_CHUNK;
}

// Count table of the pairs: counts[e * ncp + c] = live pairs of expert e among
// the tokens [c * chunk, (c + 1) * chunk).  One CTA per chunk; every entry of its
// column is written (no zeroing needed).
__global__ void __launch_bounds__(kHistThreads)
perm_count_kernel(const int32_t* __restrict__ topk_idx, int T, int k_max, int E, int chunk, int ncp,
                  int32_t* __restrict__ counts) {
  pdl_trigger();
  pdl_wait();  // topk_idx (the router before it)
  __shared__ int h[kMaxE];
  for (int e = threadIdx.x; e < E; e += kHistThreads) h[e] = 0;
  __syncthreads();
  const long long p0 = (long long)blockIdx.x * chunk * k_max;
  const long long p1 = min((long long)T, (long long)(blockIdx.x + 1) * chunk) * k_max;
  for (long long i0 = p0; i0 < p1; i0 += (long long)kPre * kHistThreads) {
    int ev[kPre];
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      const long long i = i0 + (long long)u * kHistThreads + threadIdx.x;
      ev[u] = i < p1 ? topk_idx[i] : -1;
    }
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      const int e = ev[u];
      if (e < 0) continue;
      if (e >= E) { flag(SEMMOE_DEVERR_EXPERT); continue; }
      atomicAdd(&h[e], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kHistThreads) counts[(size_t)e * ncp + blockIdx.x] = h[e];
}

// Row gather inside the ranking kernel: each warp owns a 4 KB shared-memory
// slot.  For each of its tokens, lane 0 bulk-loads the row (a segment of up to
// 4 KB at a time) into the slot and bulk-stores it to the token's k_t sorted
// rows, so the row is read from HBM once and moves by the copy engine.
constexpr int kSlotBytes = 4096;

// One warp writes token t's activation row x[t] to its live slots' sorted rows
// pair_to_sorted[t * k_max + j]: the row is read once, in segments of up to
// 4 KB held in registers, and each segment is written to the k_t rows.
// (Walking the sorted rows instead re-reads each x row k_t times, far apart in
// time, and the row writes push those reads out of L2.)
constexpr int kSegVec = 8;  // 16-byte vectors per lane per segment: 32 x 8 x 16 B = 4 KB

__device__ __forceinline__ void copy_token_row(const unsigned char* __restrict__ x, const int32_t* slots, int t,
                                               int k_max, int P, int row_bytes, unsigned char* __restrict__ x_perm) {
  const int lane = threadIdx.x % 32;
  const int n16 = row_bytes / 16;
  const int kk = k_max < 32 ? k_max : 32;
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


// The row gather as a kernel of its own (large copies): one warp per token,
// 256-thread CTAs, up to 16 per SM.
__global__ void __launch_bounds__(kHistThreads)
perm_copy_kernel(const unsigned char* __restrict__ x, const int32_t* __restrict__ pair_to_sorted, int T, int k_max,
                 int P, int row_bytes, unsigned char* __restrict__ x_perm) {
  pdl_trigger();
  pdl_wait();  // pair_to_sorted (the ranking kernel before it)
  const int warp = threadIdx.x / 32;
  for (int t = blockIdx.x * 8 + warp; t < T; t += gridDim.x * 8)
    copy_token_row(x, pair_to_sorted + (size_t)t * k_max, t, k_max, P, row_bytes, x_perm);
}

// The stable counting sort and the row gather in one pass.  CTA b takes the
// tokens [t0, t1) = [b * tpc, (b + 1) * tpc) and
//  1. derives, per expert, the rows of all tokens (totals) and of the tokens
//     before t0 from the count table: whole chunks before t0's chunk from the
//     table, the part of t0's own chunk before t0 by counting those pairs;
//  2. scans the totals in physical order (bucket starts; CTA 0 writes the
//     bucket and rank tables), so its first row in bucket b is
//     start[b] + (rows of b before t0);
//  3. ranks its own pairs in pair order, a round of kThreads pairs at a time
//     (warp match + per-warp bucket counts), and writes both maps;
//  4. copies each of its tokens' x rows to the token's sorted rows (bulk
//     copies through a shared-memory slot per warp; every wait bounded).
// No CTA waits on another: each recomputes the (small) prefix for itself.
__global__ void __launch_bounds__(kThreads)
perm_rank_copy_kernel(const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ expert_rank,
                      const int32_t* __restrict__ counts, int nc, int ncp, int chunk, int T, int k_max, int E, int R,
                      int P, int tpc, int32_t* __restrict__ expert_offsets, int32_t* __restrict__ rank_offsets,
                      int32_t* __restrict__ phys_to_expert, int32_t* __restrict__ expert_counts,
                      int32_t* __restrict__ sorted_to_pair, int32_t* pair_to_sorted,
                      const unsigned char* __restrict__ x, int row_bytes, unsigned char* __restrict__ x_perm) {
  __shared__ int rank_s[kMaxE], phys_s[kMaxE], run[kMaxE], total[kMaxE], sub[kMaxE], bef_s[kMaxE], scan[kMaxE];
  __shared__ int part_tot[kThreads], part_bef[kThreads];
  __shared__ int wcnt[kWarps][kMaxE];
  __shared__ uint64_t cbar[kWarps];   // per-warp slot barrier of the row copies
  __shared__ int abort_s;
  extern __shared__ __align__(128) unsigned char slots_smem[];  // kWarps x kSlotBytes (copy only)
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  pdl_trigger();
  if (tid == 0) {
    for (int w = 0; w < kWarps; ++w) tc::mbar_init(&cbar[w], 1);
    abort_s = 0;
    tc::mbar_init_fence();
  }
  const int t0 = min(T, (int)blockIdx.x * tpc), t1 = min(T, t0 + tpc);
  const int c0 = t0 / chunk;  // the chunk holding t0
  for (int i = tid; i < E; i += kThreads) sub[i] = 0;
  for (int i = tid; i < kWarps * kMaxE; i += kThreads) (&wcnt[0][0])[i] = 0;
  __syncthreads();
  pdl_wait();  // topk_idx and the count table (the router before it)

  // Every load that depends on nothing computed here is issued first, so that
  // their latencies overlap: the first row each warp copies (the row does not
  // depend on the ranking, only its destinations do), this thread's share of
  // the count table, the pairs of t0's chunk before t0, and the CTA's own pairs
  // of the first ranking round.
  const bool copy = x != nullptr && P > 0;
  unsigned char* slot = slots_smem + (size_t)warp * kSlotBytes;
  uint64_t* bar = &cbar[warp];
  if (copy && lane == 0 && t0 + warp < t1) {
    const uint32_t bytes = (uint32_t)(row_bytes < kSlotBytes ? row_bytes : kSlotBytes);
    tc::mbar_expect_tx(bar, bytes);
    tc::bulk_load_1d(slot, x + (size_t)(t0 + warp) * row_bytes, bytes, bar);
  }
  const int G = kThreads / E;  // threads per expert for the table (>= 2: E <= 256)
  const int ge = tid % E, gg = tid / E;
  const int4* crow = reinterpret_cast<const int4*>(counts + (size_t)ge * ncp);
  constexpr int kCv = 4;  // table vectors per thread per batch
  int4 cv[kCv];  // first batch of this thread's table vectors: vector gg + u * G of expert ge
#pragma unroll
  for (int u = 0; u < kCv; ++u) {
    const int vi = gg + u * G;
    cv[u] = (tid < G * E && vi * 4 < nc) ? crow[vi] : make_int4(0, 0, 0, 0);
  }
  const long long sp0 = (long long)c0 * chunk * k_max, sp1 = (long long)t0 * k_max;
  int sv[kPre];  // first batch of the pairs before t0 in its chunk
#pragma unroll
  for (int u = 0; u < kPre; ++u) {
    const long long i = sp0 + (long long)u * kThreads + tid;
    sv[u] = i < sp1 ? topk_idx[i] : -1;
  }
  const long long pb = (long long)t0 * k_max, pe = (long long)t1 * k_max;
  const int e_first = pb + tid < pe ? topk_idx[pb + tid] : -1;  // first ranking round

  // Physical position of each expert: M threads per expert split the E compares.
  {
    int M = kThreads / E;
    M = M >= 32 ? 32 : (M >= 16 ? 16 : (M >= 8 ? 8 : (M >= 4 ? 4 : 2)));
    for (int e = tid; e < E; e += kThreads) {
      int r = expert_rank[e];
      if (r < 0 || r >= R) {
        flag(SEMMOE_DEVERR_LUT);
        r = r < 0 ? 0 : R - 1;
      }
      rank_s[e] = r;
    }
    __syncthreads();
    const int e = tid / M, m = tid % M;  // M divides 32: the M threads of an expert share a warp
    int pos = 0;
    if (e < E) {
      const int re = rank_s[e];
      for (int f = m; f < E; f += M) {
        const int rf = rank_s[f];
        pos += (rf < re) || (rf == re && f < e);
      }
    }
#pragma unroll
    for (int d = 1; d < 32; d <<= 1)
      if (d < M) pos += __shfl_xor_sync(0xffffffffu, pos, d);
    if (e < E && m == 0) phys_s[e] = pos;
  }

  // 1a. the table: totals and the chunks before c0, per expert
  {
    int tot = 0, bef = 0;
    auto add = [&](const int4& v, int c) {
      const int a4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (c + i < nc) {
          tot += a4[i];
          if (c + i < c0) bef += a4[i];
        }
    };
#pragma unroll
    for (int u = 0; u < kCv; ++u) add(cv[u], (gg + u * G) * 4);
    if (tid < G * E)
      for (int v0 = gg + kCv * G; v0 * 4 < nc; v0 += kCv * G) {  // tables of more than 4 G vectors
#pragma unroll
        for (int u = 0; u < kCv; ++u) {
          const int vi = v0 + u * G;
          cv[u] = vi * 4 < nc ? crow[vi] : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kCv; ++u) add(cv[u], (v0 + u * G) * 4);
      }
    if (tid < G * E) {
      part_tot[tid] = tot;
      part_bef[tid] = bef;
    }
  }
  // 1b. pairs of t0's chunk before t0
#pragma unroll
  for (int u = 0; u < kPre; ++u)
    if (sv[u] >= 0 && sv[u] < E) atomicAdd(&sub[sv[u]], 1);
  for (long long i0 = sp0 + (long long)kPre * kThreads; i0 < sp1; i0 += (long long)kPre * kThreads) {
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      const long long i = i0 + (long long)u * kThreads + tid;
      sv[u] = i < sp1 ? topk_idx[i] : -1;
    }
#pragma unroll
    for (int u = 0; u < kPre; ++u)
      if (sv[u] >= 0 && sv[u] < E) atomicAdd(&sub[sv[u]], 1);
  }
  __syncthreads();
  if (tid < E) {
    int tot = 0, bef = 0;
    for (int g = 0; g < G; ++g) {
      tot += part_tot[g * E + tid];
      bef += part_bef[g * E + tid];
    }
    total[phys_s[tid]] = tot;               // indexed by physical bucket from here on
    bef_s[tid] = bef + sub[tid];            // rows of expert tid before t0
  }
  __syncthreads();
  // 2. inclusive scan of the bucket totals: a shuffle scan per warp of 32
  //    buckets, then the warps' sums (E <= 256: at most 8 warps)
  {
    int v = tid < E ? total[tid] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, v, d);
      if (lane >= d) v += o;
    }
    if (lane == 31 && warp < kMaxE / 32) part_tot[warp] = v;  // (part_tot is free again)
    __syncthreads();
    if (tid < E) {
      for (int w = 0; w < warp; ++w) v += part_tot[w];
      scan[tid] = v;
    }
    __syncthreads();
  }
  const int sum = E > 0 ? scan[E - 1] : 0;
  if (tid < E) run[phys_s[tid]] = scan[phys_s[tid]] - total[phys_s[tid]] + bef_s[tid];
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

  // 3. stable ranking of the pairs [t0 * k_max, t1 * k_max), kThreads per round
  for (long long base = pb; base < pe; base += kThreads) {
    const long long p = base + tid;
    int key = E;  // E = "no bucket" (padding slot or past the end)
    if (p < pe) {
      const int e = base == pb ? e_first : topk_idx[p];
      if (e >= E) flag(SEMMOE_DEVERR_EXPERT);
      else if (e >= 0) key = phys_s[e];
    }
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int rank_in_warp = __popc(peers & lanemask_lt());
    if (key < E && rank_in_warp == 0) wcnt[warp][key] = __popc(peers);
    __syncthreads();
    if (p < pe) {
      int pos = -1;
      if (key < E) {
        pos = run[key] + rank_in_warp;
        for (int w = 0; w < warp; ++w) pos += wcnt[w][key];
        if (pos < 0 || pos >= P) { flag(SEMMOE_DEVERR_PAIRS); pos = -1; }
        else sorted_to_pair[pos] = (int32_t)p;
      }
      pair_to_sorted[p] = pos;
    }
    __syncthreads();
    for (int b = tid; b < E; b += kThreads) {
      int s2 = 0;
      for (int w = 0; w < kWarps; ++w) { s2 += wcnt[w][b]; wcnt[w][b] = 0; }
      run[b] += s2;
    }
    __syncthreads();
  }

  // 4. the rows (this CTA's own pair_to_sorted entries, written above)
  if (copy) {
    volatile int* abort_flag = &abort_s;
    const int kk = k_max < 32 ? k_max : 32;
    uint32_t phase = 0;
    bool used = false, ok = true, loaded = true;  // the first segment was loaded at the start
    for (int t = t0 + warp; ok && t < t1; t += kWarps) {
      const int32_t* slots = pair_to_sorted + (size_t)t * k_max;
      int q_l = -1;
      if (lane < kk) {
        q_l = slots[lane];
        if (q_l >= P) { flag(SEMMOE_DEVERR_PAIRS); q_l = -1; }
      }
      for (int off = 0; ok && off < row_bytes; off += kSlotBytes) {
        const uint32_t bytes = (uint32_t)(row_bytes - off < kSlotBytes ? row_bytes - off : kSlotBytes);
        int good = 1;
        if (lane == 0) {
          if (!loaded) {
            if (used) tc::bulk_wait_read<0>();  // the slot's previous stores have read it
            tc::mbar_expect_tx(bar, bytes);
            tc::bulk_load_1d(slot, x + (size_t)t * row_bytes + off, bytes, bar);
          }
          loaded = false;
          good = tc::mbar_wait(bar, phase, abort_flag, &g_err);
          if (!good) tc::mbar_drain(bar, phase, &g_err);  // bounded: no load may land after the CTA exits
          phase ^= 1;
          used = true;
        }
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) { ok = false; break; }
        for (int j = 0; j < kk; ++j) {
          const int q = __shfl_sync(0xffffffffu, q_l, j);
          if (lane == 0 && q >= 0) tc::bulk_store_1d(x_perm + (size_t)q * row_bytes + off, slot, bytes);
        }
        if (lane == 0) {
          for (int j = 32; j < k_max; ++j) {  // budgets above 32 experts: read the slot directly
            const int q = slots[j];
            if (q < 0) continue;
            if (q >= P) { flag(SEMMOE_DEVERR_PAIRS); continue; }
            tc::bulk_store_1d(x_perm + (size_t)q * row_bytes + off, slot, bytes);
          }
          tc::bulk_commit();
        }
      }
    }
    if (lane == 0) tc::bulk_wait_all();  // every store done before the CTA exits
  }
}

}  // namespace

int permute_take_errors(cudaStream_t s, int* bits) { return take_error_word(g_err, s, bits); }

// Scratch of the permute: the count table it makes itself when the caller
// passes none.
size_t permute_ws_bytes(int T, int k_max, int E) {
  (void)k_max;
  const int chunk = internal_chunk_tokens(T > 0 ? T : 1);
  const int nc = (T + chunk - 1) / chunk;
  return align_up((size_t)E * padded_chunks(nc > 0 ? nc : 1) * sizeof(int32_t), 256);
}

size_t pair_counts_bytes(int T, int E) {
  const int nc = (T + SEMMOE_PAIR_COUNT_CHUNK - 1) / SEMMOE_PAIR_COUNT_CHUNK;
  return (size_t)E * padded_chunks(nc > 0 ? nc : 1) * sizeof(int32_t);
}

int pair_counts_stride(int T) {
  return padded_chunks((T + SEMMOE_PAIR_COUNT_CHUNK - 1) / SEMMOE_PAIR_COUNT_CHUNK);
}

cudaError_t launch_permute(const int32_t* topk_idx, const int32_t* expert_rank, const void* x, int dtype, int T,
                           int H, int E, int R, int k_max, int P, int32_t* expert_offsets,
                           int32_t* rank_offsets, int32_t* phys_to_expert, int32_t* expert_counts,
                           int32_t* sorted_to_pair, int32_t* pair_to_sorted, void* x_perm,
                           const int32_t* pair_counts, void* ws, cudaStream_t s) {
  // The count table: the caller's (128-token chunks, from the router) while it
  // has at most 1024 chunks, else one made here (at most 96 chunks).
  int chunk = SEMMOE_PAIR_COUNT_CHUNK;
  int nc = (T + chunk - 1) / chunk;
  const int32_t* counts = pair_counts;
  if (counts == nullptr || nc > 1024) {
    chunk = internal_chunk_tokens(T > 0 ? T : 1);
    nc = (T + chunk - 1) / chunk;
    int32_t* own = static_cast<int32_t*>(ws);
    if (nc > 0) {
      cudaError_t e = launch_kernel(perm_count_kernel, dim3(nc), dim3(kHistThreads), 0, s, 1, true, topk_idx, T,
                                    k_max, E, chunk, padded_chunks(nc), own);
      if (e != cudaSuccess) return e;
      count_launches(1);
    }
    counts = own;
  }
  // tokens per CTA: about two CTAs per SM
  const int target = 2 * sm_count();
  int tpc = (T + target - 1) / target;
  if (tpc < 1) tpc = 1;
  const int grid = T > 0 ? (T + tpc - 1) / tpc : 1;
  const int row_bytes = H * (dtype == SEMMOE_BF16 ? 2 : 4);
  // Where the rows are copied: inside the ranking kernel for copies under
  // 256 MB, by a copy kernel of its own (more warps per SM) above that.
  // Measured per call with L2 flushed: DeepSeek prefill (101 MB) 29.3 us inside
  // against 35.5 us separate; Qwen3 (537 MB) 119.4 against 114.3; MoE-Prism
  // (604 MB) 136.8 against 128.7.
  const bool any_copy = x != nullptr && x_perm != nullptr && P > 0;
  const bool separate = any_copy && (long long)P * row_bytes >= (256LL << 20);
  const bool copy = any_copy && !separate;
  const size_t dyn = copy ? (size_t)kWarps * kSlotBytes : 0;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = ensure_smem_limit(perm_rank_copy_kernel, (int)(kWarps * kSlotBytes), smem_set);
  if (e != cudaSuccess) return e;
  e = launch_kernel(perm_rank_copy_kernel, dim3(grid), dim3(kThreads), dyn, s, 1, true, topk_idx, expert_rank,
                    counts, nc, padded_chunks(nc), chunk, T, k_max, E, R, P, tpc, expert_offsets, rank_offsets,
                    phys_to_expert, expert_counts, sorted_to_pair, pair_to_sorted,
                    copy ? static_cast<const unsigned char*>(x) : static_cast<const unsigned char*>(nullptr),
                    row_bytes, static_cast<unsigned char*>(x_perm));
  if (e != cudaSuccess) return e;
  count_launches(1);
  if (separate) {
    int blocks = (T + 7) / 8;
    const int cap = sm_count() * 16;
    if (blocks > cap) blocks = cap;
    e = launch_kernel(perm_copy_kernel, dim3(blocks), dim3(kHistThreads), 0, s, 1, true,
                      static_cast<const unsigned char*>(x), static_cast<const int32_t*>(pair_to_sorted), T, k_max, P,
                      row_bytes, static_cast<unsigned char*>(x_perm));
    if (e != cudaSuccess) return e;
    count_launches(1);
  }
  return cudaGetLastError();
}

size_t permute_noalloc_max_scratch() { return kNoAllocScratchBytes; }

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

// Device address of g_noalloc_scratch in the current CUDA context.  In host
// code the array's name is only a host-side stand-in, so the address is looked
// up with cudaGetSymbolAddress, with the context current, and cached.  The
// cache is keyed on the context's unique ID (cuCtxGetId), not on the device
// number: after cudaDeviceReset, or in another context on the same device, the
// library's module is loaded again and the array has another address, while a
// context's ID is never reused within the process.
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
  // The count kernel writes every table entry the ranking kernel adds up before
  // that kernel runs, so stale contents of an earlier call never leak into this one.
  return launch_permute(topk_idx, expert_rank, x, dtype, T, H, E, R, k_max, P, expert_offsets, rank_offsets,
                        phys_to_expert, expert_counts, sorted_to_pair, pair_to_sorted, x_perm, nullptr, scratch, s);
}

}  // namespace semmoe
