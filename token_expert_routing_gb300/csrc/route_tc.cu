// Router GEMM on the tensor cores: logits[t, e] = sum_h x[t,h] * Wr[e,h] for
// bf16 activations, with fp32 accumulation in TMEM.
//
// The router ("gate") scores experts per token (Semantic Parallelism (ko) §1,
// MoE-Prism (ko) §1).  With a bf16 router weight the GEMM is one bf16 MMA.  An
// fp32 router weight is split exactly into three bf16 parts, Wr = hi + mid + lo
// (hi = bf16(Wr), mid = bf16(Wr - hi), lo = bf16(Wr - hi - mid)); x is bf16, so
// each product x*part is exact in fp32, and the three partial sums are kept in
// separate accumulator columns and added in fp32 in the epilogue:
//   logit = (x.hi + x.mid) + x.lo.
// The stacked parts form one B operand of 3*EC rows, so one MMA (N = 3*EC)
// computes all three.
//
// One CTA per (128-token tile, pass of EC experts); warp 0 issues TMA, warp 1
// allocates TMEM and issues the MMAs, warps 2..5 read the accumulator and write
// fp32 logits.  The operand ring has as many stages (up to 8) as fit 200 KB, so
// a CTA keeps as many loads in flight as the tile size allows: the GEMM is
// small and the ring depth is what hides HBM latency.  Waits are bounded as in
// the grouped-FFN kernel.
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace semmoe {
namespace {

using namespace tc;

__device__ int g_err;

constexpr int BM = 128, BK = 64, UK = 16, THREADS = 192;
constexpr int MAX_STAGES = 8;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
// Operand ring per CTA: 200 KB when the grid fits one CTA per SM, 100 KB (two
// CTAs per SM, each one's epilogue beside the other's loads) when it is larger.
__host__ __device__ constexpr size_t stage_budget(int cps) { return cps == 1 ? 200 * 1024 : 100 * 1024; }
constexpr uint32_t TMEM_COLS = 256;
constexpr int kMaxKSlices = 8;

struct Shared {
  uint64_t full[MAX_STAGES], empty[MAX_STAGES], tfull, done;
  uint32_t tmem_base;
  int abort_flag;
};

__host__ __device__ constexpr size_t smem_bytes(int cps) { return 1024 + stage_budget(cps) + sizeof(Shared); }

// Experts per pass: S * EC <= 256 columns, EC a multiple of 16.
inline int experts_per_pass(int E, int S) {
  const int e16 = (E + 15) / 16 * 16;
  const int cap = S == 3 ? 64 : 256;
  return e16 < cap ? e16 : cap;
}

// out rows ((p * 3 + s) * EC + j): part s of expert e = p*EC + j (zero for e >= E).
__global__ void split_router_kernel(const float* __restrict__ w, int E, int H, int EC, int n_pass,
                                    __nv_bfloat16* __restrict__ out) {
  const long long total = (long long)n_pass * 3 * EC * H;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int h = (int)(i % H);
    const long long row = i / H;
    const int j = (int)(row % EC), part = (int)((row / EC) % 3), p = (int)(row / (3LL * EC));
    const int e = p * EC + j;
    float v = 0.f;
    if (e < E) {
      const float x = w[(size_t)e * H + h];
      const __nv_bfloat16 hi = __float2bfloat16_rn(x);
      const float r1 = x - __bfloat162float(hi);
      const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
      const float r2 = r1 - __bfloat162float(mid);
      v = part == 0 ? __bfloat162float(hi) : part == 1 ? __bfloat162float(mid) : r2;
    }
    out[i] = __float2bfloat16_rn(v);
  }
}

template <int S, int CPS>  // CPS: resident CTAs per SM the ring is sized for
__global__ void __launch_bounds__(THREADS, CPS)
route_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w, int T, int H,
                int E, int EC, int stages, int kb_per_slice, float* __restrict__ partials) {
  pdl_trigger();  // the kernel after it may start its setup
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* ring = smem_raw + pad;  // stage s: A tile then B tile, stage_bytes apart
  Shared& sh = *reinterpret_cast<Shared*>(ring + stage_budget(CPS));
  volatile int* abort_flag = &sh.abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int NB = S * EC;
  const uint32_t b_bytes = (uint32_t)NB * BK * 2;
  const uint32_t stage_bytes = A_BYTES + b_bytes;  // a multiple of 1024 (NB % 16 == 0)
  const int t0 = blockIdx.x * BM, pass = blockIdx.y, slice = blockIdx.z;
  const int kb_all = (H + BK - 1) / BK;
  const int kb0 = slice * kb_per_slice;
  const int kb_n = kb_all - kb0 < kb_per_slice ? kb_all - kb0 : kb_per_slice;  // >= 1 by construction
  float* logits = partials + (size_t)slice * T * E;  // this K slice's partial sums

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    mbar_init(&sh.tfull, 1);
    mbar_init(&sh.done, 1);
    sh.abort_flag = 0;
    mbar_init_fence();
    prefetch_map(&map_x);
    prefetch_map(&map_w);
  }
  if (warp == 1) tmem_alloc(&sh.tmem_base, TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      int it = 0;
      for (int kb = 0; kb < kb_n; ++kb) {
        const int s = kb % stages;
        const uint32_t ph = (kb / stages) & 1;
        if (!mbar_wait(&sh.empty[s], ph ^ 1, abort_flag, &g_err)) break;
        unsigned char* st = ring + (size_t)s * stage_bytes;
        mbar_expect_tx(&sh.full[s], stage_bytes);
        tma_load_2d(st, &map_x, &sh.full[s], (kb0 + kb) * BK, t0);
        tma_load_2d(st + A_BYTES, &map_w, &sh.full[s], (kb0 + kb) * BK, pass * NB);
        ++it;
      }
      if (*abort_flag)
        for (int j = it > stages ? it - stages : 0; j < it; ++j)
          mbar_drain(&sh.full[j % stages], (j / stages) & 1, &g_err);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      const uint32_t idesc = idesc_bf16_f32(BM, NB);
      bool ok = true;
      for (int kb = 0; kb < kb_n; ++kb) {
        const int s = kb % stages;
        const uint32_t ph = (kb / stages) & 1;
        if (!mbar_wait(&sh.full[s], ph, abort_flag, &g_err)) { ok = false; break; }
        fence_after();
        const uint32_t sa = smem_u32(ring + (size_t)s * stage_bytes), sb = sa + A_BYTES;
#pragma unroll
        for (int k = 0; k < BK / UK; ++k)
          mma_bf16(tmem, sw128_desc(sa + k * UK * 2), sw128_desc(sb + k * UK * 2), idesc, (kb | k) != 0);
        commit(&sh.empty[s]);
      }
      if (ok) commit(&sh.tfull);
      commit(&sh.done);
      mbar_drain(&sh.done, 0, &g_err);
    }
  } else {  // epilogue: thread = one token row of the accumulator
    const int q = warp & 3;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(&sh.tfull, 0, abort_flag, &g_err);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      fence_after();
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
      // The warp's 32 rows x 16 columns pass through 2 KB of the operand ring
      // (every MMA has read it once tfull has fired): lane l stores its row's
      // four 16-byte pieces at piece p ^ ((l >> 1) & 3) of its 64-byte row, then
      // each store instruction writes two rows' 64-byte segments.
      float* stg = reinterpret_cast<float*>(ring) + q * 32 * 16;
      const int sw = (lane >> 1) & 3;
      for (int c = 0; c < EC; c += 16) {
        uint32_t v0[16], v1[16], v2[16];
        tmem_ld16(trow + c, v0);
        if (S == 3) {
          tmem_ld16(trow + EC + c, v1);
          tmem_ld16(trow + 2 * EC + c, v2);
        }
        tmem_ld_wait();
        float l[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          l[i] = __uint_as_float(v0[i]);
          if (S == 3) l[i] = (l[i] + __uint_as_float(v1[i])) + __uint_as_float(v2[i]);
        }
#pragma unroll
        for (int p = 0; p < 4; ++p)
          *reinterpret_cast<float4*>(stg + lane * 16 + ((p ^ sw) << 2)) =
              make_float4(l[4 * p], l[4 * p + 1], l[4 * p + 2], l[4 * p + 3]);
        __syncwarp();
        const int col = lane & 15, e = pass * EC + c + col;
#pragma unroll 4
        for (int rr = 0; rr < 32; rr += 2) {
          const int row = rr + (lane >> 4), t = t0 + q * 32 + row;
          const float val = stg[row * 16 + ((((col >> 2) ^ ((row >> 1) & 3))) << 2) + (col & 3)];
          if (t < T && e < E) logits[(size_t)t * E + e] = val;
        }
        __syncwarp();
      }
    }
  }

  fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}


// ---------------------------------------------------------------------------
// Router GEMM and top-k in one kernel (E16 * S <= 256 accumulator columns,
// k_max <= KM): one CTA per 128-token tile reads the whole contraction over H
// (no K slices, no logits in memory).  The epilogue has G groups of four warps;
// a thread of group g owns one token row of the accumulator and the g-th of G
// contiguous column ranges: it adds the weight parts' columns into logits and
// keeps the KM best as (key, index) in a sorted register list.  Groups 1..G-1
// leave their lists in shared memory; group 0 merges them in column order
// (so equal scores keep the lower expert first) and writes the k_t picks,
// their gates and the tile's pair counts.  (With one group the selection ran
// about 10K dependent instructions per warp and set the kernel's time.)  The
// k-blocks are visited from a per-tile starting block (tile index mod the
// block count), so the tiles do not all read the same weight lines at once.
// ---------------------------------------------------------------------------

// Order-preserving 32-bit key of an fp32 score: larger key = larger score; -0.0
// counts as +0.0; 0 is below every float (an empty list slot).
__device__ __forceinline__ uint32_t score_key(float v) {
  const uint32_t b = __float_as_uint(__fadd_rn(v, 0.0f));
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// Insert (key, e) into keys/ids, sorted by key descending; entries scanned in
// increasing e, so among equal keys the earlier (lower) index stays ahead.
template <int KM>
__device__ __forceinline__ void list_insert(uint32_t (&keys)[KM], int (&ids)[KM], uint32_t key, int e) {
  if (!(key > keys[KM - 1])) return;
  bool placed = false;
#pragma unroll
  for (int i = KM - 1; i > 0; --i) {
    const bool up = key > keys[i - 1];
    const uint32_t nk = placed ? keys[i] : (up ? keys[i - 1] : key);
    const int ne = placed ? ids[i] : (up ? ids[i - 1] : e);
    keys[i] = nk;
    ids[i] = ne;
    placed = placed || !up;
  }
  if (!placed) {
    keys[0] = key;
    ids[0] = e;
  }
}

template <int S, int KM, int CPS, int G>
__global__ void __launch_bounds__(64 + 128 * G, CPS)
route_topk_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w, int T,
                     int H, int E, int E16, int stages, float* __restrict__ logits_out,
                     const int32_t* __restrict__ k_per_token, int k_uniform, int k_max,
                     int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ counts,
                     int count_stride) {
  pdl_trigger();  // the kernel after it may start its setup
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* ring = smem_raw + pad;
  Shared& sh = *reinterpret_cast<Shared*>(ring + stage_budget(CPS));
  __shared__ int hist[256];
  volatile int* abort_flag = &sh.abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int NB = S * E16;
  const uint32_t b_bytes = (uint32_t)NB * BK * 2;
  const uint32_t stage_bytes = A_BYTES + b_bytes;
  const int t0 = blockIdx.x * BM;
  const int kb_all = (H + BK - 1) / BK;
  const int kb_first = (int)(blockIdx.x % (unsigned)kb_all);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    mbar_init(&sh.tfull, 1);
    mbar_init(&sh.done, 1);
    sh.abort_flag = 0;
    mbar_init_fence();
    prefetch_map(&map_x);
    prefetch_map(&map_w);
  }
  for (int e = threadIdx.x; e < 256; e += blockDim.x) hist[e] = 0;
  if (warp == 1) tmem_alloc(&sh.tmem_base, TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      int it = 0;
      for (int i = 0; i < kb_all; ++i) {
        const int kb = kb_first + i < kb_all ? kb_first + i : kb_first + i - kb_all;
        const int s = i % stages;
        const uint32_t ph = (i / stages) & 1;
        if (!mbar_wait(&sh.empty[s], ph ^ 1, abort_flag, &g_err)) break;
        unsigned char* st = ring + (size_t)s * stage_bytes;
        mbar_expect_tx(&sh.full[s], stage_bytes);
        tma_load_2d(st, &map_x, &sh.full[s], kb * BK, t0);
        tma_load_2d(st + A_BYTES, &map_w, &sh.full[s], kb * BK, 0);
        ++it;
      }
      if (*abort_flag)
        for (int j = it > stages ? it - stages : 0; j < it; ++j)
          mbar_drain(&sh.full[j % stages], (j / stages) & 1, &g_err);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      const uint32_t idesc = idesc_bf16_f32(BM, NB);
      bool ok = true;
      for (int i = 0; i < kb_all; ++i) {
        const int s = i % stages;
        const uint32_t ph = (i / stages) & 1;
        if (!mbar_wait(&sh.full[s], ph, abort_flag, &g_err)) { ok = false; break; }
        fence_after();
        const uint32_t sa = smem_u32(ring + (size_t)s * stage_bytes), sb = sa + A_BYTES;
#pragma unroll
        for (int k = 0; k < BK / UK; ++k)
          mma_bf16(tmem, sw128_desc(sa + k * UK * 2), sw128_desc(sb + k * UK * 2), idesc, (i | k) != 0);
        commit(&sh.empty[s]);
      }
      if (ok) commit(&sh.tfull);
      commit(&sh.done);
      mbar_drain(&sh.done, 0, &g_err);
    }
  } else {  // epilogue: thread = token row t of the tile, column range g
    const int q = warp & 3;            // TMEM lane quarter of this warp
    const int g = (warp - 2) / 4;      // column group
    const int r = q * 32 + lane;       // tile row
    const int t = t0 + r;
    const int nch = E16 / 16;
    const int c_lo = (g * nch / G) * 16, c_hi = ((g + 1) * nch / G) * 16;
    // groups 1..G-1 hand their lists over in the (by then idle) operand ring
    uint32_t* mkeys = reinterpret_cast<uint32_t*>(ring);
    int* mids = reinterpret_cast<int*>(ring + (size_t)(G > 1 ? G - 1 : 1) * BM * KM * 4);
    uint32_t keys[KM];
    int ids[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      keys[j] = 0u;
      ids[j] = -1;
    }
    bool nonfinite = false;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(&sh.tfull, 0, abort_flag, &g_err);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      fence_after();
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
      for (int c = c_lo; c < c_hi; c += 16) {
        uint32_t v0[16], v1[16], v2[16];
        tmem_ld16(trow + c, v0);
        if (S == 3) {
          tmem_ld16(trow + E16 + c, v1);
          tmem_ld16(trow + 2 * E16 + c, v2);
        }
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int e = c + i;
          if (e < E) {
            float l = __uint_as_float(v0[i]);
            if (S == 3) l = (l + __uint_as_float(v1[i])) + __uint_as_float(v2[i]);
            if (logits_out != nullptr && t < T) logits_out[(size_t)t * E + e] = l;
            if (!isfinite(l)) {
              nonfinite = true;
              l = -INFINITY;
            }
            list_insert<KM>(keys, ids, score_key(l), e);
          }
        }
      }
      if (G > 1 && g > 0) {
#pragma unroll
        for (int j = 0; j < KM; ++j) {
          mkeys[((size_t)(g - 1) * BM + r) * KM + j] = keys[j];
          mids[((size_t)(g - 1) * BM + r) * KM + j] = ids[j];
        }
      }
    }
    if (nonfinite && t < T) atomicOr(&g_err, SEMMOE_DEVERR_NONFINITE);
    if (G > 1) asm volatile("bar.sync 1, %0;" ::"r"(128 * G) : "memory");
    if (g == 0) {
      if (ok) {
        for (int h = 1; h < G; ++h) {  // later column ranges: equal keys stay behind
          for (int j = 0; j < KM; ++j) {
            const uint32_t k2 = mkeys[((size_t)(h - 1) * BM + r) * KM + j];
            if (!(k2 > keys[KM - 1])) break;  // the rest of that sorted list is no better
            list_insert<KM>(keys, ids, k2, mids[((size_t)(h - 1) * BM + r) * KM + j]);
          }
        }
      }
      if (ok && t < T) {
        int kt = k_per_token != nullptr ? k_per_token[t] : k_uniform;
        if (kt < 1 || kt > k_max) {
          atomicOr(&g_err, SEMMOE_DEVERR_K);
          kt = kt < 1 ? 1 : k_max;
        }
        const float m = key_score(keys[0]);
        float den = 0.f;
#pragma unroll
        for (int j = 0; j < KM; ++j)
          if (j < kt && ids[j] >= 0) den += expf(key_score(keys[j]) - m);
#pragma unroll
        for (int j = 0; j < KM; ++j) {
          if (j < k_max) {
            int e = -1;
            float gw = 0.f;
            if (j < kt) {
              if (ids[j] >= 0) {
                e = ids[j];
                gw = expf(key_score(keys[j]) - m) / den;
                atomicAdd(&hist[e], 1);
              } else {
                atomicOr(&g_err, SEMMOE_DEVERR_NONFINITE);  // fewer than k_t scores
              }
            }
            topk_idx[(size_t)t * k_max + j] = e;
            topk_w[(size_t)t * k_max + j] = gw;
          }
        }
      }
      // the tile's pair counts (the tile is chunk blockIdx.x of the count table)
      asm volatile("bar.sync 2, 128;" ::: "memory");
      if (counts != nullptr) {
        const int et = threadIdx.x - 64;  // group 0 is threads 64 .. 191
        for (int e = et; e < E; e += 128) counts[(size_t)e * count_stride + blockIdx.x] = hist[e];
        if (blockIdx.x == 0) {  // entries past the last chunk are 0
          const int nchunk = (int)gridDim.x, padn = count_stride - nchunk;
          for (int i = et; i < E * padn; i += 128) counts[(size_t)(i / padn) * count_stride + nchunk + i % padn] = 0;
        }
      }
    }
  }

  fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Router GEMM and top-k in one launch for fewer token tiles than SMs: a
// cluster of CS = passes x KS CTAs per 128-token tile, CTA r contracting the
// (r % KS)-th of KS slices of H for the experts of pass r / KS (EC of them)
// into its own TMEM accumulator (the host runs one pass: CS = KS).  Each CTA
// leaves its partial logits (the weight parts already added, as in
// route_tc_kernel) in its shared memory; after a cluster barrier each CTA
// pushes to CTA q, by one bulk copy into q's shared memory, its partials of
// the rows [q * 128 / CS, (q + 1) * 128 / CS) that q selects.  CTA q adds an
// expert's KS slices in slice order (a fixed order: the logits do not depend on
// timing) and selects with one warp per row as the top-k kernel does: k_t
// rounds of a warp argmax over order-preserving keys (ties to the lower
// expert), then the gates and the picks.  The CTAs add their pick histograms
// into CTA 0's (shared-memory atomics across the cluster), which writes the
// tile's column of the count table.  No logits in memory, no second launch;
// every cluster barrier is reached by every thread on every path.  One CTA per
// SM (the host keeps tiles x CS <= SMs).  Measured on the way (64 tokens,
// %globaltimer stamps): loads of the other CTAs' shared memory, thread by
// thread, took 9-25 us where the pushed copies take ~0.7 us; sorted lists per
// thread merged across a row's threads are one long dependent chain per row.
// ---------------------------------------------------------------------------
constexpr int kClThreads = 64 + 4 * 128;  // producer, MMA, 16 epilogue / selection warps

template <int S, int NPER>  // NPER experts per lane in the selection: E <= 32 * NPER
__global__ void __launch_bounds__(kClThreads, 1)
route_topk_cl_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w, int T,
                     int H, int E, int EC, int KS, int CS, int stages, int kb_slice, float* __restrict__ logits_out,
                     const int32_t* __restrict__ k_per_token, int k_uniform, int k_max,
                     int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ counts,
                     int count_stride) {
  pdl_trigger();  // the kernel after it may start its setup
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* ring = smem_raw + pad;
  Shared& sh = *reinterpret_cast<Shared*>(ring + stage_budget(1));
  __shared__ int hist[256];
  __shared__ uint64_t recv_bar;  // the other CTAs' partial rows for this CTA's rows have landed
  volatile int* abort_flag = &sh.abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int NB = S * EC;
  const uint32_t b_bytes = (uint32_t)NB * BK * 2;
  const uint32_t stage_bytes = A_BYTES + b_bytes;
  const int rank = (int)cluster_ctarank();
  const int pass = rank / KS, slice = rank % KS;  // this CTA: experts [pass * EC, +EC), k-block slice
  const int tile = blockIdx.x / CS;
  const int t0 = tile * BM;
  const int kb_all = (H + BK - 1) / BK;
  const int kb0 = slice * kb_slice;
  const int kb_n = kb_all - kb0 < kb_slice ? kb_all - kb0 : kb_slice;  // >= 1 by the host's choice of CS
  const int kb_first = tile % kb_n;  // tiles start at different k-blocks of their slice
  // after the MMAs, in the operand ring: this CTA's partial logits [128][EC + 4]
  // fp32, then what the others send of theirs for this CTA's rows: recv[q] =
  // CTA q's rows [rank * rpc, (rank + 1) * rpc)
  const int pstride = EC + 4;
  const int rpc = BM / CS;
  float* part = reinterpret_cast<float*>(ring);
  float* recv = part + (size_t)BM * pstride;
  const uint32_t slice_bytes = (uint32_t)(rpc * pstride * 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    mbar_init(&sh.tfull, 1);
    mbar_init(&sh.done, 1);
    mbar_init(&recv_bar, 1);
    mbar_expect_tx(&recv_bar, (uint32_t)(CS - 1) * slice_bytes);  // the one arrival; the copies' bytes follow
    sh.abort_flag = 0;
    mbar_init_fence();
    prefetch_map(&map_x);
    prefetch_map(&map_w);
  }
  for (int e = threadIdx.x; e < 256; e += blockDim.x) hist[e] = 0;
  if (warp == 1) tmem_alloc(&sh.tmem_base, TMEM_COLS);
  fence_before();
  __syncthreads();  // (the other CTAs see the receive barrier once past the cluster barrier before the copies)
  fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    if (lane == 0) {  // TMA producer: this CTA's k-blocks
      int it = 0;
      for (int i = 0; i < kb_n; ++i) {
        const int kb = kb0 + (kb_first + i < kb_n ? kb_first + i : kb_first + i - kb_n);
        const int s = i % stages;
        const uint32_t ph = (i / stages) & 1;
        if (!mbar_wait(&sh.empty[s], ph ^ 1, abort_flag, &g_err)) break;
        unsigned char* st = ring + (size_t)s * stage_bytes;
        mbar_expect_tx(&sh.full[s], stage_bytes);
        tma_load_2d(st, &map_x, &sh.full[s], kb * BK, t0);
        tma_load_2d(st + A_BYTES, &map_w, &sh.full[s], kb * BK, pass * NB);
        ++it;
      }
      if (*abort_flag)
        for (int j = it > stages ? it - stages : 0; j < it; ++j)
          mbar_drain(&sh.full[j % stages], (j / stages) & 1, &g_err);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      const uint32_t idesc = idesc_bf16_f32(BM, NB);
      bool ok = true;
      for (int i = 0; i < kb_n; ++i) {
        const int s = i % stages;
        const uint32_t ph = (i / stages) & 1;
        if (!mbar_wait(&sh.full[s], ph, abort_flag, &g_err)) { ok = false; break; }
        fence_after();
        const uint32_t sa = smem_u32(ring + (size_t)s * stage_bytes), sb = sa + A_BYTES;
#pragma unroll
        for (int k = 0; k < BK / UK; ++k)
          mma_bf16(tmem, sw128_desc(sa + k * UK * 2), sw128_desc(sb + k * UK * 2), idesc, (i | k) != 0);
        commit(&sh.empty[s]);
      }
      if (ok) commit(&sh.tfull);
      commit(&sh.done);
      mbar_drain(&sh.done, 0, &g_err);
    }
  } else {  // 16 epilogue warps: the rows of their TMEM lane quarter, a quarter of the columns, into `part`
    const int q = warp & 3, r = q * 32 + lane, g = (warp - 2) / 4;
    const int nch = EC / 16, c_lo = (g * nch / 4) * 16, c_hi = ((g + 1) * nch / 4) * 16;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(&sh.tfull, 0, abort_flag, &g_err);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      fence_after();
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
      for (int c = c_lo; c < c_hi; c += 16) {
        uint32_t v0[16], v1[16], v2[16];
        tmem_ld16(trow + c, v0);
        if (S == 3) {
          tmem_ld16(trow + EC + c, v1);
          tmem_ld16(trow + 2 * EC + c, v2);
        }
        tmem_ld_wait();
        float l[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          l[i] = __uint_as_float(v0[i]);
          if (S == 3) l[i] = (l[i] + __uint_as_float(v1[i])) + __uint_as_float(v2[i]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)  // row stride EC + 4 words: the 16-byte stores of 8 lanes hit 8 bank groups
          *reinterpret_cast<float4*>(part + (size_t)r * pstride + c + 4 * j) =
              make_float4(l[4 * j], l[4 * j + 1], l[4 * j + 2], l[4 * j + 3]);
      }
    }
    fence_async_smem();  // the rows are read by bulk copies next
  }
  fence_before();
  cluster_sync_all();  // every CTA is done with its operand ring, where the copies land
  // push: the rows of CTA q go to q (even after an abort, so that every receive completes)
  if (threadIdx.x == 64)
    for (int q = 0; q < CS; ++q)
      if (q != rank)
        bulk_copy_to_peer(mapa_rank(recv + (size_t)rank * rpc * pstride, (uint32_t)q),
                          part + (size_t)q * rpc * pstride, slice_bytes, mapa_rank(&recv_bar, (uint32_t)q));

  // selection: CTA `rank` takes rows [rank * rpc, (rank + 1) * rpc); one warp
  // per row (16 warps: a row's chain of rounds is latency, so rows run side by
  // side), lane l holding experts l + 32 i, each the sum of its pass's KS
  // slices in slice order; k_t rounds of a warp argmax (the largest key, then
  // the lowest expert holding it, which is taken out)
  if (warp >= 2) {
    const bool got = mbar_wait(&recv_bar, 0, abort_flag, &g_err);  // every lane: acquire the copies
    for (int row = rank * rpc + (warp - 2); got && row < (rank + 1) * rpc; row += kClThreads / 32 - 2) {
      const int t = t0 + row;
      int kt = 0;  // loaded first: its latency overlaps the sums
      if (t < T) kt = k_per_token != nullptr ? k_per_token[t] : k_uniform;
      float l[NPER];
#pragma unroll
      for (int i = 0; i < NPER; ++i) {
        const int e = lane + 32 * i;
        const int pe = e / EC, c = e - pe * EC;  // the expert's pass and column in it
        l[i] = 0.f;
        if (e < E)
          for (int sk = 0; sk < KS; ++sk) {  // slice order
            const int qc = pe * KS + sk;
            const float* src = qc == rank ? part + (size_t)row * pstride
                                          : recv + ((size_t)qc * rpc + (row - rank * rpc)) * pstride;
            l[i] = sk == 0 ? src[c] : l[i] + src[c];
          }
      }
      bool nonfinite = false;
      uint32_t key[NPER];
#pragma unroll
      for (int i = 0; i < NPER; ++i) {
        const int e = lane + 32 * i;
        key[i] = 0u;
        if (e < E) {
          if (logits_out != nullptr && t < T) logits_out[(size_t)t * E + e] = l[i];
          float lv = l[i];
          if (!isfinite(lv)) {
            nonfinite = true;
            lv = -INFINITY;
          }
          key[i] = score_key(lv);
        }
      }
      if (t < T) {
        if (kt < 1 || kt > k_max) {
          if (lane == 0) atomicOr(&g_err, SEMMOE_DEVERR_K);
          kt = kt < 1 ? 1 : k_max;
        }
        uint32_t pk = 0u;  // lane j: the j-th pick (key, expert)
        int pe = -1;
        for (int j = 0; j < kt; ++j) {
          uint32_t mk = key[0];
#pragma unroll
          for (int i = 1; i < NPER; ++i) mk = max(mk, key[i]);
          const uint32_t m = __reduce_max_sync(0xffffffffu, mk);
          int be = -1;
          if (m != 0u) {
            uint32_t mine = 0xffffffffu;
#pragma unroll
            for (int i = NPER - 1; i >= 0; --i)
              if (key[i] == m) mine = (uint32_t)(lane + 32 * i);
            be = (int)__reduce_min_sync(0xffffffffu, mine);
#pragma unroll
            for (int i = 0; i < NPER; ++i)
              if (be == lane + 32 * i) key[i] = 0u;
          }
          if (lane == j) {
            pk = m;
            pe = be;
          }
        }
        const float mx = key_score(__shfl_sync(0xffffffffu, pk, 0));
        float ex = lane < kt && pe >= 0 ? expf(key_score(pk) - mx) : 0.f;
        float den = ex;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
        if (lane < k_max) {
          int e = -1;
          float gw = 0.f;
          if (lane < kt) {
            if (pe >= 0) {
              e = pe;
              gw = ex / den;
              atomicAdd(&hist[e], 1);
            } else {
              atomicOr(&g_err, SEMMOE_DEVERR_NONFINITE);  // fewer than k_t scores
            }
          }
          topk_idx[(size_t)t * k_max + lane] = e;
          topk_w[(size_t)t * k_max + lane] = gw;
        }
        if (nonfinite) atomicOr(&g_err, SEMMOE_DEVERR_NONFINITE);
      }
    }
  }
  __syncthreads();
  if (rank != 0 && counts != nullptr)  // this CTA's picks into CTA 0's histogram
    for (int e = threadIdx.x; e < E; e += kClThreads)
      if (hist[e] != 0) red_cluster_add_u32(mapa_rank(&hist[e], 0u), (uint32_t)hist[e]);
  cluster_sync_all();  // every copy has landed, every pick is in CTA 0's histogram; then nobody
                       // touches another CTA's shared memory
  if (rank == 0 && counts != nullptr) {  // the tile's column of the count table
    for (int e = threadIdx.x; e < E; e += kClThreads) counts[(size_t)e * count_stride + tile] = hist[e];
    if (tile == 0) {  // entries past the last chunk are 0
      const int nchunk = (int)gridDim.x / CS, padn = count_stride - nchunk;
      for (int j = threadIdx.x; j < E * padn; j += kClThreads)
        counts[(size_t)(j / padn) * count_stride + nchunk + j % padn] = 0;
    }
  }
  if (warp == 1) {
    __syncwarp();
    fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Epilogue column groups: four with one CTA per SM and k_max <= 16 (the lists'
// registers allow it), else fewer.
template <int S, int KM, int CPS>
static cudaError_t launch_topk_k(int grid, const CUtensorMap& mx, const CUtensorMap& mw, int T, int H, int E, int E16,
                                 int stages, float* logits_out, const int32_t* kpt, int k_uniform, int k_max,
                                 int32_t* topk_idx, float* topk_w, int32_t* counts, int count_stride, cudaStream_t s) {
  constexpr int G = CPS == 1 ? (KM <= 16 ? 4 : 2) : 1;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = ensure_smem_limit(route_topk_tc_kernel<S, KM, CPS, G>, (int)smem_bytes(CPS), smem_set);
  if (e != cudaSuccess) return e;
  route_topk_tc_kernel<S, KM, CPS, G><<<grid, 64 + 128 * G, smem_bytes(CPS), s>>>(
      mx, mw, T, H, E, E16, stages, logits_out, kpt, k_uniform, k_max, topk_idx, topk_w, counts, count_stride);
  return cudaSuccess;
}

template <int S, int KM>
static cudaError_t launch_topk_km(int grid, int cps, const CUtensorMap& mx, const CUtensorMap& mw, int T, int H, int E,
                                  int E16, int stages, float* lo, const int32_t* kpt, int ku, int k_max, int32_t* idx,
                                  float* w, int32_t* counts, int cs, cudaStream_t s) {
  if (cps == 1) return launch_topk_k<S, KM, 1>(grid, mx, mw, T, H, E, E16, stages, lo, kpt, ku, k_max, idx, w, counts, cs, s);
  return launch_topk_k<S, KM, 2>(grid, mx, mw, T, H, E, E16, stages, lo, kpt, ku, k_max, idx, w, counts, cs, s);
}

}  // namespace

int route_tc_take_errors(cudaStream_t s, int* bits) { return take_error_word(g_err, s, bits); }

// Workspace of the tensor-core router: the three-part split of an fp32 weight
// (none when the caller passes the split already made).
size_t route_tc_split_bytes(int H, int E, int w_dtype) {
  if (w_dtype != SEMMOE_F32) return 0;
  return route_split_size(H, E);
}

size_t route_split_size(int H, int E) {
  const int EC = experts_per_pass(E, 3), n_pass = (E + EC - 1) / EC;
  return align_up((size_t)n_pass * 3 * EC * H * 2, 256);
}

// K slices of the router GEMM: enough (token tile, pass, slice) CTAs to fill
// the GPU once, with at least 4 k-blocks of H per slice.
int route_tc_k_slices(int T, int H, int E, int w_dtype) {
  const int S = w_dtype == SEMMOE_BF16 ? 1 : 3;
  const int EC = experts_per_pass(E, S), n_pass = (E + EC - 1) / EC;
  const long long ctas = (long long)((T + BM - 1) / BM) * n_pass;
  const int kb_all = (H + BK - 1) / BK;
  int ks = (int)(sm_count() / (ctas > 0 ? ctas : 1));
  if (ks > kb_all / 4) ks = kb_all / 4;
  if (ks > kMaxKSlices) ks = kMaxKSlices;
  return ks < 1 ? 1 : ks;
}

cudaError_t launch_route_split(const float* w, int H, int E, void* split, cudaStream_t s) {
  const int EC = experts_per_pass(E, 3), n_pass = (E + EC - 1) / EC;
  const long long total = (long long)n_pass * 3 * EC * H;
  long long blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  split_router_kernel<<<(int)blocks, 256, 0, s>>>(w, E, H, EC, n_pass, static_cast<__nv_bfloat16*>(split));
  count_launches(1);
  return cudaGetLastError();
}

template <int S, int CPS>
static cudaError_t launch_k(dim3 grid, const CUtensorMap& mx, const CUtensorMap& mw, int T, int H, int E, int EC,
                            int stages, int kb_per_slice, float* partials, cudaStream_t s) {
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = ensure_smem_limit(route_tc_kernel<S, CPS>, (int)smem_bytes(CPS), smem_set);
  if (e != cudaSuccess) return e;
  route_tc_kernel<S, CPS><<<grid, THREADS, smem_bytes(CPS), s>>>(mx, mw, T, H, E, EC, stages, kb_per_slice,
                                                                 partials);
  return cudaSuccess;
}

// x [T,H] bf16 (H % 8 == 0); w [E,H] fp32 or bf16, or the split of an fp32
// weight (SEMMOE_F32_SPLIT); partials [ks][T][E] fp32 out (ks =
// route_tc_k_slices(); the logits are their sum in slice order); split:
// workspace of route_tc_split_bytes() (fp32 weight only).
cudaError_t launch_route_logits_tc(const void* x, const void* w, int w_dtype, int T, int H, int E, float* partials,
                                   int ks, void* split, cudaStream_t s) {
  const int S = w_dtype == SEMMOE_BF16 ? 1 : 3;
  const int EC = experts_per_pass(E, S), n_pass = (E + EC - 1) / EC;
  const int kb_all = (H + BK - 1) / BK;
  const int kb_per_slice = (kb_all + ks - 1) / ks;
  ks = (kb_all + kb_per_slice - 1) / kb_per_slice;  // every slice non-empty
  const void* wb = w;
  int w_rows = E;
  if (S == 3) {
    if (w_dtype == SEMMOE_F32) {
      cudaError_t e = launch_route_split(static_cast<const float*>(w), H, E, split, s);
      if (e != cudaSuccess) return e;
      wb = split;
    }
    w_rows = n_pass * 3 * EC;
  }
  CUtensorMap mx, mw;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t str[1] = {(cuuint64_t)H * 2};
    const cuuint32_t box[2] = {BK, BM};
    if (!make_map_bf16(&mx, x, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)w_rows};
    const cuuint64_t str[1] = {(cuuint64_t)H * 2};
    const cuuint32_t box[2] = {BK, (cuuint32_t)(S * EC)};
    if (!make_map_bf16(&mw, wb, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  const size_t stage_bytes = A_BYTES + (size_t)S * EC * BK * 2;
  dim3 grid((T + BM - 1) / BM, n_pass, ks);
  const int cps = (long long)grid.x * grid.y * grid.z > sm_count() ? 2 : 1;
  int stages = (int)(stage_budget(cps) / stage_bytes);
  if (stages > MAX_STAGES) stages = MAX_STAGES;
  cudaError_t e;
  if (S == 3 && cps == 1) e = launch_k<3, 1>(grid, mx, mw, T, H, E, EC, stages, kb_per_slice, partials, s);
  else if (S == 3) e = launch_k<3, 2>(grid, mx, mw, T, H, E, EC, stages, kb_per_slice, partials, s);
  else if (cps == 1) e = launch_k<1, 1>(grid, mx, mw, T, H, E, EC, stages, kb_per_slice, partials, s);
  else e = launch_k<1, 2>(grid, mx, mw, T, H, E, EC, stages, kb_per_slice, partials, s);
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaGetLastError();
}

// The one-kernel router applies when every expert's accumulator columns fit one
// MMA (S parts x E rounded up to 16 <= 256; an fp32 weight's split holds up to 64
// experts in one pass) and k_max <= 32.
bool route_topk_tc_ok(int E, int k_max, int w_dtype) {
  const int S = w_dtype == SEMMOE_BF16 ? 1 : 3;
  const int E16 = (E + 15) / 16 * 16;
  if (S == 3 && E16 > 64) return false;
  return S * E16 <= 256 && k_max <= 32;
}

cudaError_t launch_route_topk_tc(const void* x, const void* w, int w_dtype, int T, int H, int E, int k_max,
                                 float* logits_out, const int32_t* kpt, int k_uniform, int32_t* topk_idx,
                                 float* topk_w, int32_t* counts, int count_stride, void* split, cudaStream_t s) {
  const int S = w_dtype == SEMMOE_BF16 ? 1 : 3;
  const int E16 = (E + 15) / 16 * 16;
  const void* wb = w;
  int w_rows = E;
  if (S == 3) {
    if (w_dtype == SEMMOE_F32) {  // one pass: the split's EC is E16 when E16 <= 64
      cudaError_t e = launch_route_split(static_cast<const float*>(w), H, E, split, s);
      if (e != cudaSuccess) return e;
      wb = split;
    }
    w_rows = 3 * E16;
  }
  CUtensorMap mx, mw;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t str[1] = {(cuuint64_t)H * 2};
    const cuuint32_t box[2] = {BK, BM};
    if (!make_map_bf16(&mx, x, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)w_rows};
    const cuuint64_t str[1] = {(cuuint64_t)H * 2};
    const cuuint32_t box[2] = {BK, (cuuint32_t)(S * E16)};
    if (!make_map_bf16(&mw, wb, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  const int grid = (T + BM - 1) / BM;
  const int cps = grid > sm_count() ? 2 : 1;
  const size_t stage_bytes = A_BYTES + (size_t)S * E16 * BK * 2;
  int stages = (int)(stage_budget(cps) / stage_bytes);
  if (stages > MAX_STAGES) stages = MAX_STAGES;
  cudaError_t e;
  const int km = k_max <= 8 ? 8 : (k_max <= 16 ? 16 : 32);
  if (S == 1 && km == 8) e = launch_topk_km<1, 8>(grid, cps, mx, mw, T, H, E, E16, stages, logits_out, kpt, k_uniform, k_max, topk_idx, topk_w, counts, count_stride, s);
  else if (S == 1 && km == 16) e = launch_topk_km<1, 16>(grid, cps, mx, mw, T, H, E, E16, stages, logits_out, kpt, k_uniform, k_max, topk_idx, topk_w, counts, count_stride, s);
  else if (S == 1) e = launch_topk_km<1, 32>(grid, cps, mx, mw, T, H, E, E16, stages, logits_out, kpt, k_uniform, k_max, topk_idx, topk_w, counts, count_stride, s);
  else if (km == 8) e = launch_topk_km<3, 8>(grid, cps, mx, mw, T, H, E, E16, stages, logits_out, kpt, k_uniform, k_max, topk_idx, topk_w, counts, count_stride, s);
  else if (km == 16) e = launch_topk_km<3, 16>(grid, cps, mx, mw, T, H, E, E16, stages, logits_out, kpt, k_uniform, k_max, topk_idx, topk_w, counts, count_stride, s);
  else e = launch_topk_km<3, 32>(grid, cps, mx, mw, T, H, E, E16, stages, logits_out, kpt, k_uniform, k_max, topk_idx, topk_w, counts, count_stride, s);
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaGetLastError();
}

// K slices of the cluster router; 0 when it does not apply (the one-kernel
// router or the split-K path takes the call): the largest KS in {2, 4, 8} with
// one CTA per SM for every (tile, slice) and at least 2 k-blocks per slice, for
// routers whose experts fit one pass (a bf16 weight, or an fp32 one with
// E <= 64).  The kernel also takes several passes of experts as further CTAs of
// the cluster, but with the whole of H per CTA that measured slower than the
// split-K path for an fp32 weight over 128 or 256 experts (T = 1024 .. 8192:
// 25-60 against 16-41 us per call), so it is not used for them.  The partial and
// received logits (2 x 128 rows of EC + 4 fp32) must fit the 200 KB operand
// ring: EC <= 192.
int route_topk_cl_slices(int T, int H, int E, int k_max, int w_dtype) {
  if (k_max > 32) return 0;
  const int S = w_dtype == SEMMOE_BF16 ? 1 : 3;
  const int EC = experts_per_pass(E, S), n_pass = (E + EC - 1) / EC;
  if (EC > 192 || n_pass > 1) return 0;
  const long long tiles = (T + BM - 1) / BM;
  const int kb_all = (H + BK - 1) / BK;
  int ks = 0;
  for (int c = 2; c <= 8; c *= 2)
    if (tiles * c <= sm_count() && kb_all >= 2 * c) ks = c;
  return ks;
}

cudaError_t launch_route_topk_cl(const void* x, const void* w, int w_dtype, int T, int H, int E, int k_max, int KS,
                                 float* logits_out, const int32_t* kpt, int k_uniform, int32_t* topk_idx,
                                 float* topk_w, int32_t* counts, int count_stride, void* split, cudaStream_t s) {
  const int S = w_dtype == SEMMOE_BF16 ? 1 : 3;
  const int E16 = (E + 15) / 16 * 16;
  const int EC = experts_per_pass(E, S), n_pass = (E + EC - 1) / EC, CS = n_pass * KS;
  const void* wb = w;
  int w_rows = E;
  if (S == 3) {
    if (w_dtype == SEMMOE_F32) {
      cudaError_t e = launch_route_split(static_cast<const float*>(w), H, E, split, s);
      if (e != cudaSuccess) return e;
      wb = split;
    }
    w_rows = n_pass * 3 * EC;  // [pass][part][EC][H]
  }
  CUtensorMap mx, mw;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t str[1] = {(cuuint64_t)H * 2};
    const cuuint32_t box[2] = {BK, BM};
    if (!make_map_bf16(&mx, x, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)w_rows};
    const cuuint64_t str[1] = {(cuuint64_t)H * 2};
    const cuuint32_t box[2] = {BK, (cuuint32_t)(S * EC)};
    if (!make_map_bf16(&mw, wb, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  const int kb_all = (H + BK - 1) / BK, kb_slice = (kb_all + KS - 1) / KS;
  if (CS < 2 || CS > 8 || (KS - 1) * kb_slice >= kb_all) return cudaErrorInvalidValue;  // every slice holds k-blocks
  const size_t stage_bytes = A_BYTES + (size_t)S * EC * BK * 2;
  int stages = (int)(stage_budget(1) / stage_bytes);
  if (stages > MAX_STAGES) stages = MAX_STAGES;
  using K = void (*)(CUtensorMap, CUtensorMap, int, int, int, int, int, int, int, int, float*, const int32_t*, int,
                     int, int32_t*, float*, int32_t*, int);
  // experts per lane in the selection (E <= 32 NPER)
  const int np = E16 <= 32 ? 1 : (E16 <= 64 ? 2 : (E16 <= 128 ? 4 : 8));
  const int ki = (S == 1 ? 0 : 4) + (np == 1 ? 0 : (np == 2 ? 1 : (np == 4 ? 2 : 3)));
  static const K kerns[8] = {route_topk_cl_kernel<1, 1>, route_topk_cl_kernel<1, 2>, route_topk_cl_kernel<1, 4>,
                             route_topk_cl_kernel<1, 8>, route_topk_cl_kernel<3, 1>, route_topk_cl_kernel<3, 2>,
                             route_topk_cl_kernel<3, 4>, route_topk_cl_kernel<3, 8>};
  const K kern = kerns[ki];
  static std::atomic<unsigned long long> smem_set[8];
  cudaError_t e = ensure_smem_limit(kern, (int)smem_bytes(1), smem_set[ki]);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(((T + BM - 1) / BM) * CS));
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = smem_bytes(1);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, mx, mw, T, H, E, EC, KS, CS, stages, kb_slice, logits_out, kpt, k_uniform,
                         k_max, topk_idx, topk_w, counts, count_stride);
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace semmoe
