// Grouped SwiGLU expert FFN on the 5th-generation tensor cores (bf16 in,
// fp32 accumulation): tcgen05.mma with accumulators in tensor memory (TMEM),
// operands staged in shared memory by TMA.
//
// The experts' computation (Semantic Parallelism (ko) §1; MoE-Prism (ko) §2 A)
// over each expert's contiguous block of sorted rows:
//   GEMM1 (GLU):   h = silu(x W1_e^T) * (x W3_e^T)     -> bf16
//   GEMM2 (PLAIN): y = h W2_e^T                        -> bf16
//
// One persistent CTA per SM walks the (m-tile, n-tile) list of all groups.
// Warp roles (192 threads):
//   warp 0      TMA producer: A tile [128 x 64] + B tile [256 x 64] per stage
//   warp 1      allocates TMEM; one thread issues tcgen05.mma (M128 N256 K16)
//   warps 2..5  epilogue: tcgen05.ld the accumulator, SwiGLU / convert, stage
//               32 x 64 bf16 blocks in shared memory and write them with TMA
//               stores (a warp whose rows cross its group's end stores directly)
//   warps 6..13 (GEMM1 gathering x rows, single-CTA form only): the A rows,
//               fetched with 16-byte loads and stored in the swizzled layout;
//               warp 0 then loads only the weight tile
// Pipelines: a 4-stage smem ring (full/empty mbarriers) and a 2-deep TMEM
// accumulator ring (tfull/tempty), so the epilogue of tile i overlaps the MMAs
// of tile i+1.  GEMM1's B tile is 128 gate rows + the 128 matching up rows, so
// accumulator columns [0,128) hold x W1^T and [128,256) hold x W3^T for the
// same 128 h-columns.
//
// Forms of the same computation (all bit-identical):
//  * independent CTAs (above): M128 x N256 per SM;
//  * 2-SM pairs (ffn_pair_kernel, the default for I >= 512): a cluster of two
//    CTAs runs tcgen05.mma.cta_group::2 with M = 256, each SM staging its own
//    A rows and half of the weight tile, a third less shared-memory traffic per
//    SM; pairs cover two m-tiles of one expert, so groups with an odd m-tile
//    count leave one half idle, which costs more than it saves on short
//    (I < 512) tiles;
//  * both GEMMs in one launch of independent CTAs (ffn_fused_kernel, the
//    default where both GEMMs would run as independent CTAs): GEMM2 tiles
//    start while GEMM1 tiles of other m-tiles still run, so the grid's last
//    partial wave and the launch boundary between the GEMMs are paid once.
//
// Every wait is bounded (%globaltimer and a poll count); a wait that runs out sets the timeout
// bit of the device error word and an abort flag, after which every role
// stops, in-flight TMA loads and MMAs are drained (again with a bound), and
// TMEM is freed before the CTA exits.
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace semmoe {
namespace {

using namespace tc;

__device__ int g_err;

constexpr int BM = 128;                 // tile rows = MMA M
constexpr int BN = 256;                 // MMA N
constexpr int BK = 64;                  // K per stage: one 128-byte swizzle row of bf16
constexpr int UK = 16;                  // K per tcgen05.mma, kind::f16
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;    // 16 KB
constexpr int B_BYTES = BN * BK * 2;    // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t ACC_COLS = 256;      // fp32 accumulator columns per buffer
constexpr uint32_t TMEM_COLS = 512;     // two buffers: all of TMEM
constexpr int MAX_GROUPS = 256;

struct Shared {
  uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], done;
  uint32_t tmem_base;
  int abort_flag;
  int armed, producer_done;  // gathering warps: stage positions the producer armed, and its exit
  int total_mtiles;
  int off[MAX_GROUPS + 1];
  int pe[MAX_GROUPS];
  int tp[MAX_GROUPS + 1];
};

// Output staging of the epilogue: per epilogue warp one 4 KB buffer (two boxes of
// 32 rows x 32 bf16 columns), written back by TMA stores.
constexpr int OUT_STAGE_BYTES = 4 * 2 * 2048;

constexpr size_t kSmemBytes = 1024 + (size_t)STAGES * STAGE_BYTES + OUT_STAGE_BYTES + sizeof(Shared);

constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN);

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// silu(g) * u on raw fp32 accumulator words
__device__ __forceinline__ float swiglu(uint32_t gw, uint32_t uw) {
  const float g = __uint_as_float(gw), u = __uint_as_float(uw);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Epilogue output of one 64-column chunk of an epilogue warp's 32 tile rows
// (lane = row; w = the row's 64 bf16 values, packed in pairs).  A warp whose 32
// rows all hold data stages the chunk in shared memory as two 32 x 32 boxes
// (64-byte rows, 64-byte swizzle: 16-byte piece v of row r sits at piece
// v ^ ((r >> 1) & 3)) and writes them with TMA stores; the warp at a group's end
// (some rows past it) writes its valid rows directly, so no store reaches another
// group's rows.  Columns past N are clipped by the store / skipped.
struct ChunkOut {
  const CUtensorMap* map;  // [rows, N] bf16, box {32 columns, 32 rows}, 64-byte swizzle
  unsigned char* stage;    // this warp's 4 KB staging buffer
  uint32_t n;              // chunks stored through the buffer so far
};

__device__ __forceinline__ void emit_chunk(ChunkOut& co, const uint32_t (&w)[32], bool full, bool row_ok,
                                           __nv_bfloat16* orow, int col0, int N, int wrow0, int lane) {
  if (col0 >= N) return;
  if (full) {
    if (co.n > 0 && lane == 0) bulk_wait_read<0>();  // the previous chunk's stores have read the buffer
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int v = 0; v < 4; ++v)
        *reinterpret_cast<uint4*>(co.stage + h * 2048 + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4)) =
            make_uint4(w[16 * h + 4 * v], w[16 * h + 4 * v + 1], w[16 * h + 4 * v + 2], w[16 * h + 4 * v + 3]);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(co.map, co.stage, col0, wrow0);
      if (col0 + 32 < N) tma_store_2d(co.map, co.stage + 2048, col0 + 32, wrow0);
      bulk_commit();
    }
    ++co.n;
  } else if (row_ok) {
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const int col = col0 + 8 * v;
      if (col + 8 <= N)
        *reinterpret_cast<uint4*>(orow + col) = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
    }
  }
}

// GEMM2 adding its rows into the token-order output instead of storing y_perm
// (the combine folded into the epilogue): sorted row q is pair p =
// pairs[q] of token p / div, weighted by gates[p], and added into acc [T, N]
// fp32.  Each epilogue warp transposes its 32 rows x 32 columns through its
// staging buffer (16-byte piece v of row r at piece v ^ (r & 7)) so that
// eight lanes cover one row's 128 bytes: the adds are float4 atomics, four
// rows per instruction.  Scattered per-row atomics measured half the rate.
struct Scatter {
  const int32_t* pairs = nullptr;  // sorted_to_pair [P]
  const float* gates = nullptr;    // topk_w [T * div], by pair id
  int div = 1;                     // k_max
  int T = 0;
  float* acc = nullptr;            // [T, N] fp32, zeroed before GEMM2
};

// The token (or -1) and gate of sorted row q.
__device__ __forceinline__ void scatter_row(const Scatter& sc, int q, bool row_ok, int& t, float& g) {
  t = -1;
  g = 0.f;
  if (!row_ok) return;
  const int p = sc.pairs[q];
  const int tt = p >= 0 ? p / sc.div : -1;
  if (tt < 0 || tt >= sc.T) {
    atomicOr(&g_err, SEMMOE_DEVERR_PAIRS);
    return;
  }
  t = tt;
  g = sc.gates[p];
}

// Half a 64-column chunk (32 accumulator words of the thread's row) weighted by
// g and added into acc rows of the warp's 32 tokens.
__device__ __forceinline__ void scatter_half(const Scatter& sc, unsigned char* stage, const uint32_t (&y)[32], int t,
                                             float g, int col0, int N, int lane) {
#pragma unroll
  for (int v = 0; v < 8; ++v)
    *reinterpret_cast<float4*>(stage + lane * 128 + ((v ^ (lane & 7)) << 4)) =
        make_float4(g * __uint_as_float(y[4 * v]), g * __uint_as_float(y[4 * v + 1]),
                    g * __uint_as_float(y[4 * v + 2]), g * __uint_as_float(y[4 * v + 3]));
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int rr = i * 4 + (lane >> 3), v = lane & 7;
    const float4 val = *reinterpret_cast<const float4*>(stage + rr * 128 + ((v ^ (rr & 7)) << 4));
    const int tr = __shfl_sync(0xffffffffu, t, rr);
    const int col = col0 + 4 * v;
    if (tr >= 0 && col < N) atomicAdd(reinterpret_cast<float4*>(sc.acc + (size_t)tr * N + col), val);
  }
  __syncwarp();
}

// Tile unit mu (CL consecutive m-tiles of one group: CL = 1 for independent
// CTAs, 2 for a 2-SM pair, one m-tile per CTA) -> this CTA's (first row, valid
// rows, expert).  A CTA whose m-tile
// lies past its group's end gets rows = 0 (it still takes part in the loads).
template <int CL, typename SH>
__device__ __forceinline__ void decode_mtile(const SH& sh, int G, int mu, int rank, int& row0, int& rows, int& e) {
  int lo = 0, hi = G - 1;  // largest g with tp[g] <= mu
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sh.tp[mid] <= mu) lo = mid;
    else hi = mid - 1;
  }
  row0 = sh.off[lo] + ((mu - sh.tp[lo]) * CL + rank) * BM;
  const int left = sh.off[lo + 1] - row0;
  rows = left <= 0 ? 0 : (left < BM ? left : BM);
  if (left <= 0) row0 = sh.off[lo + 1];
  e = sh.pe[lo];
}

// Row gather of the A operand (GEMM1 reading x directly instead of x_perm):
// lane l of the producer warp fetches tile rows 4l .. 4l+3; sorted row q reads
// x row gather[q] / gather_div (the token of pair q).  Rows past P, and bad pair
// ids (flagged), read row 0: their results are never stored.
__device__ __forceinline__ void gather_sources(const int32_t* __restrict__ gather, int gather_div, int gather_rows,
                                               int P, int row0, int lane, int (&src)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int q = row0 + 4 * lane + i;
    int r = 0;
    if (q < P) {
      const int p = gather[q];
      r = p >= 0 ? p / gather_div : -1;
      if (r < 0 || r >= gather_rows) {
        atomicOr(&g_err, SEMMOE_DEVERR_PAIRS);
        r = 0;
      }
    }
    src[i] = r;
  }
}

// GW > 0: GW more warps gather the A rows (x row gather[q] / gather_div) with
// 16-byte loads into registers and shared-memory stores in the swizzled layout,
// each lane then fencing for the async proxy and arriving on the stage barrier.
// Each warp keeps the loads of GATHER_DEPTH k-blocks in flight.  Routed FFN,
// single-CTA form: one warp issuing TMA four-row gathers 855 / 2148 / 1350 us
// (DeepSeek / Qwen3 / MoE-Prism shapes); 8 warps 2 deep 543 / 1388 / 814; 3 deep
// 451 / 1129 / 686; 4 deep 426 / 1060 / 650; 5 deep 414 / 1032 / 635; 6 and 7
// deep spill registers and lose (460 / 1152 / 700 at 6).  Tiled loads of a
// permuted copy take 346-354 / 789-832 / 554-570 us in the default forms.
constexpr int GATHER_WARPS = 8;
constexpr int GATHER_DEPTH = 5;
constexpr int RPL = 4;  // 16-byte pieces per lane per k-block: 8 warps x 32 lanes x 4 = 128 rows x 128 B
template <bool GLU, int GW = 0, bool SC = false>
__global__ void __launch_bounds__(THREADS + 32 * GW, 1)
ffn_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
              const __grid_constant__ CUtensorMap map_out,
              const int32_t* __restrict__ offsets, const int32_t* __restrict__ phys_to_expert, int G, int P,
              int E, int N, int K, int n_tiles, const int32_t* __restrict__ gather, int gather_div, int gather_rows,
              __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ gx, Scatter sc) {
  pdl_trigger();  // the kernel after it may start its setup
  static_assert(GW == 0 || GW * 32 * RPL * 16 == BM * BK * 2, "gather warps cover one A stage");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* stage_a = smem_raw + pad;                 // STAGES x [128 x 64] bf16
  unsigned char* stage_b = stage_a + STAGES * A_BYTES;     // STAGES x [256 x 64] bf16
  unsigned char* out_stage = stage_a + STAGES * STAGE_BYTES;  // OUT_STAGE_BYTES, 1024-aligned
  Shared& sh = *reinterpret_cast<Shared*>(out_stage + OUT_STAGE_BYTES);
  volatile int* abort_flag = &sh.abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh.full[s], 1 + 32 * GW);
      mbar_init(&sh.empty[s], 1);  // released by the MMA's commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh.tfull[a], 1);
      mbar_init(&sh.tempty[a], 128);
    }
    mbar_init(&sh.done, 1);
    sh.abort_flag = 0;
    sh.armed = 0;
    sh.producer_done = 0;
    mbar_init_fence();
    prefetch_map(&map_a);
    prefetch_map(&map_b);
    prefetch_map(&map_out);
  }
  if (warp == 1) {  // whole warp: allocate all 512 TMEM columns
    tmem_alloc(&sh.tmem_base, TMEM_COLS);
  }
  pdl_wait();  // the rows and group offsets the kernels before it wrote
  for (int g = threadIdx.x; g <= G; g += blockDim.x) sh.off[g] = offsets ? offsets[g] : (g == 0 ? 0 : P);
  for (int g = threadIdx.x; g < G; g += blockDim.x) sh.pe[g] = phys_to_expert ? phys_to_expert[g] : 0;
  __syncthreads();

  if (warp == 0) {  // exclusive prefix of m-tiles per group, 8 groups per lane
    int cnt[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int g = lane * 8 + i;
      int c = 0;
      if (g < G) {
        const int lo = sh.off[g], hi = sh.off[g + 1], e = sh.pe[g];
        if (lo < 0 || hi < lo || hi > P) atomicOr(&g_err, SEMMOE_DEVERR_PAIRS);
        else if (e < 0 || e >= E) atomicOr(&g_err, SEMMOE_DEVERR_EXPERT);
        else c = (hi - lo + BM - 1) / BM;
      }
      cnt[i] = c;
      sum += c;
    }
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int g = lane * 8 + i;
      if (g < G) sh.tp[g] = run;
      run += cnt[i];
    }
    if (lane == 31) {
      sh.tp[G] = incl;
      sh.total_mtiles = incl;
    }
  }
  fence_before();
  __syncthreads();
  fence_after();

  const uint32_t tmem = sh.tmem_base;
  const int total = sh.total_mtiles * n_tiles;  // tile units: (m-tile, n-tile)
  const int kb_n = (K + BK - 1) / BK;
  const int unit0 = blockIdx.x, units = gridDim.x;

  if (warp == 0) {
    // ---------------- TMA producer (warp 0; lane 0 unless A rows are gathered) ----------------
    uint32_t it = 0;
    const int32_t* tg = GW > 0 ? nullptr : gather;  // TMA row gathers only without gathering warps
    if (tg != nullptr || lane == 0)  // without row gathers lane 0 alone: 1% faster than the warp
    for (int tile = unit0; tile < total; tile += units) {
      if (*abort_flag) break;
      const int mt = tile / n_tiles, nt = tile % n_tiles;
      int row0, rows, e;
      decode_mtile<1>(sh, G, mt, 0, row0, rows, e);
      int src[4] = {0, 0, 0, 0};
      if (tg != nullptr) gather_sources(tg, gather_div, gather_rows, P, row0, lane, src);
      bool ok = true;
      for (int kb = 0; kb < kb_n; ++kb) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        int good = 1;
        if (lane == 0) good = mbar_wait(&sh.empty[s], ph ^ 1, abort_flag, &g_err);
        if (tg != nullptr ? !__shfl_sync(0xffffffffu, good, 0) : !good) { ok = false; break; }
        if (GW > 0) {
          mbar_expect_tx(&sh.full[s], B_BYTES);
        } else if (tg != nullptr) {
          if (lane == 0) mbar_expect_tx(&sh.full[s], STAGE_BYTES);
          tma_gather4(stage_a + s * A_BYTES + lane * 4 * (BK * 2), &map_a, &sh.full[s], kb * BK, src[0], src[1],
                      src[2], src[3]);
        } else if (lane == 0) {
          mbar_expect_tx(&sh.full[s], STAGE_BYTES);
          tma_load_2d(stage_a + s * A_BYTES, &map_a, &sh.full[s], kb * BK, row0);
        }
        if (lane == 0) {
          unsigned char* b = stage_b + s * B_BYTES;
          if (GLU) {
            tma_load_4d(b, &map_b, &sh.full[s], kb * BK, nt * 128, 0, e);
            tma_load_4d(b + B_BYTES / 2, &map_b, &sh.full[s], kb * BK, nt * 128, 1, e);
          } else {
            tma_load_3d(b, &map_b, &sh.full[s], kb * BK, nt * BN, e);
          }
        }
        ++it;
      }
      if (!ok) break;
    }
    if (lane == 0) {  // positions armed: how far gathering warps arrive, and what is drained, on an abort
      *reinterpret_cast<volatile int*>(&sh.armed) = (int)it;
      __threadfence_block();
      *reinterpret_cast<volatile int*>(&sh.producer_done) = 1;
    }
    if (lane == 0 && *abort_flag) {  // no TMA write may still be landing when the CTA exits
      for (uint32_t j = it > (uint32_t)STAGES ? it - STAGES : 0; j < it; ++j)
        mbar_drain(&sh.full[j % STAGES], (j / STAGES) & 1, &g_err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      uint32_t it = 0, acc_it = 0;
      for (int tile = unit0; tile < total; tile += units) {
        if (*abort_flag) break;
        const uint32_t a = acc_it & 1, aph = (acc_it >> 1) & 1;
        if (!mbar_wait(&sh.tempty[a], aph ^ 1, abort_flag, &g_err)) break;
        fence_after();
        const uint32_t d = tmem + a * ACC_COLS;
        bool ok = true;
        for (int kb = 0; kb < kb_n; ++kb) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&sh.full[s], ph, abort_flag, &g_err)) { ok = false; break; }
          fence_after();
          const uint32_t sa = smem_u32(stage_a + s * A_BYTES), sb = smem_u32(stage_b + s * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / UK; ++k)
            mma_bf16(d, sw128_desc(sa + k * UK * 2), sw128_desc(sb + k * UK * 2), kIdesc, (kb | k) != 0);
          commit(&sh.empty[s]);  // frees the stage once these MMAs have read it
          ++it;
        }
        if (!ok) break;
        commit(&sh.tfull[a]);    // accumulator ready for the epilogue
        ++acc_it;
      }
      commit(&sh.done);          // every MMA issued above has completed ...
      mbar_drain(&sh.done, 0, &g_err);      // ... before TMEM can be released
    }
  } else if (warp < 6) {
    // ---------------- epilogue (warps 2..5) ----------------
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;      // tile row held by this thread
    uint32_t acc_it = 0;
    ChunkOut co{&map_out, out_stage + q * 4096, 0};
    for (int tile = unit0; tile < total; tile += units) {
      const int mt = tile / n_tiles, nt = tile % n_tiles;
      int row0, rows, e;
      decode_mtile<1>(sh, G, mt, 0, row0, rows, e);
      const uint32_t a = acc_it & 1, aph = (acc_it >> 1) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&sh.tfull[a], aph, abort_flag, &g_err);
      ok = __shfl_sync(0xffffffffu, ok, 0);  // keep the warp converged for tcgen05.ld
      if (!ok) break;
      fence_after();
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + a * ACC_COLS;
      const bool row_ok = r < rows;
      __nv_bfloat16* orow = out + (size_t)(row0 + (row_ok ? r : 0)) * N;
      const bool full = q * 32 + 32 <= rows;  // all 32 rows of this warp lie in the group
      if (GLU) {  // accumulator columns [0, 128) gate, [128, 256) up; 128 output columns
#pragma unroll 1
        for (int c = 0; c < 128; c += 64) {
          uint32_t g0[32], g1[32], u0[32], u1[32], w[32];
          tmem_ld32(t_row + c, g0);
          tmem_ld32(t_row + c + 32, g1);
          tmem_ld32(t_row + 128 + c, u0);
          tmem_ld32(t_row + 128 + c + 32, u1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            w[i] = pack_bf16x2(swiglu(g0[2 * i], u0[2 * i]), swiglu(g0[2 * i + 1], u0[2 * i + 1]));
            w[16 + i] = pack_bf16x2(swiglu(g1[2 * i], u1[2 * i]), swiglu(g1[2 * i + 1], u1[2 * i + 1]));
          }
          emit_chunk(co, w, full, row_ok, orow, nt * 128 + c, N, row0 + q * 32, lane);
        }
      } else if (SC) {  // rows weighted and added into the token-order output
        int st;
        float sg;
        scatter_row(sc, row0 + (row_ok ? r : 0), row_ok, st, sg);
#pragma unroll 1
        for (int c = 0; c < BN; c += 64) {
          if (nt * BN + c >= N) break;
          uint32_t y0[32], y1[32];
          tmem_ld32(t_row + c, y0);
          tmem_ld32(t_row + c + 32, y1);
          tmem_ld_wait();
          scatter_half(sc, co.stage, y0, st, sg, nt * BN + c, N, lane);
          scatter_half(sc, co.stage, y1, st, sg, nt * BN + c + 32, N, lane);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN; c += 64) {
          uint32_t y0[32], y1[32], w[32];
          tmem_ld32(t_row + c, y0);
          tmem_ld32(t_row + c + 32, y1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            w[i] = pack_bf16x2(__uint_as_float(y0[2 * i]), __uint_as_float(y0[2 * i + 1]));
            w[16 + i] = pack_bf16x2(__uint_as_float(y1[2 * i]), __uint_as_float(y1[2 * i + 1]));
          }
          emit_chunk(co, w, full, row_ok, orow, nt * BN + c, N, row0 + q * 32, lane);
        }
      }
      fence_before();
      mbar_arrive(&sh.tempty[a]);
      ++acc_it;
    }
    if (lane == 0) bulk_wait_all();  // this warp's output stores are complete
  } else if (GW > 0) {
    // ---------------- row-gathering warps (6 .. 5 + GW) ----------------
    // Lane l copies 16-byte piece l & 7 of rows gw * (128 / GW) + 4 j + (l >> 3), j < RPL,
    // into the layout a 128-byte-swizzled TMA load of the [128 x 64] box writes
    // (piece c of row r at piece c ^ (r & 7)).  The loads of the next
    // GATHER_DEPTH - 1 k-blocks are in flight (registers v, a ring indexed by the
    // k-block count) while this one waits for its stage.
    const int gw = warp - 6, c = lane & 7;
    const __nv_bfloat16* cur[RPL];
    auto sources = [&](int t, const __nv_bfloat16* (&p)[RPL]) {
      int row0, rows, e;
      decode_mtile<1>(sh, G, t / n_tiles, 0, row0, rows, e);
#pragma unroll
      for (int j = 0; j < RPL; ++j) {
        const int q = row0 + gw * (BM / GW) + 4 * j + (lane >> 3);
        int r = 0;
        if (q < P) {
          const int pid = gather[q];
          r = pid >= 0 ? pid / gather_div : -1;
          if (r < 0 || r >= gather_rows) {
            atomicOr(&g_err, SEMMOE_DEVERR_PAIRS);
            r = 0;
          }
        }
        p[j] = gx + (size_t)r * K;
      }
    };
    auto fetch = [&](const __nv_bfloat16* const (&p)[RPL], int kb, uint4 (&v)[RPL]) {
      const int col = kb * BK + c * 8;
#pragma unroll
      for (int j = 0; j < RPL; ++j)
        v[j] = col < K ? __ldg(reinterpret_cast<const uint4*>(p[j] + col)) : make_uint4(0, 0, 0, 0);
    };
    constexpr int D = GATHER_DEPTH;  // k-blocks of loads in flight per warp
    uint4 v[D][RPL];
    const int my_tiles = unit0 < total ? (total - unit0 + units - 1) / units : 0;
    const int npos = my_tiles * kb_n;
    int ltile = unit0, lkb = 0;  // position of the next k-block to load
    auto load_next = [&](uint4 (&dst)[RPL]) {
      if (lkb == 0) sources(ltile, cur);
      fetch(cur, lkb, dst);
      if (++lkb == kb_n) {
        lkb = 0;
        ltile += units;
      }
    };
#pragma unroll
    for (int u = 0; u < D - 1; ++u)
      if (u < npos) load_next(v[u]);
    bool ok = true;
    int stop = npos;  // the first position this warp did not fill (on abort)
    for (int base = 0; ok && base < npos; base += D) {
#pragma unroll
      for (int u = 0; u < D; ++u) {
        const int it = base + u;
        if (it >= npos) break;
        if (it + D - 1 < npos) load_next(v[(u + D - 1) % D]);
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!mbar_wait(&sh.empty[s], ph ^ 1, abort_flag, &g_err)) {
          ok = false;
          stop = it;
          break;
        }
        unsigned char* a = stage_a + s * A_BYTES;
#pragma unroll
        for (int j = 0; j < RPL; ++j) {
          const int r = gw * (BM / GW) + 4 * j + (lane >> 3);
          *reinterpret_cast<uint4*>(a + r * 128 + ((c ^ (r & 7)) << 4)) = v[u][j];
        }
        fence_async_smem();
        mbar_arrive(&sh.full[s]);
      }
    }
    if (!ok) {
      // Abort: the producer armed its positions up to sh.armed with the weight
      // tile's bytes; arriving (once per lane) on those this warp did not fill
      // lets each complete when its weight tile lands, so the producer's drain
      // sees the copies end instead of running to its bound.  Every position
      // before `stop` was filled, and the producer is at most STAGES positions
      // ahead, so each of these barriers is in the phase of that position.
      volatile int* done_flag = &sh.producer_done;
      const uint64_t t_start = globaltimer_ns();
      for (uint32_t polls = 0; *done_flag == 0; ++polls)
        if (globaltimer_ns() - t_start > kWaitNs || polls > kWaitPolls) break;
      if (*done_flag != 0) {
        const int armed = *reinterpret_cast<volatile int*>(&sh.armed);
        for (int q2 = stop; q2 < armed; ++q2) mbar_arrive(&sh.full[q2 % STAGES]);
      }
    }
  }

  fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {  // also an abort raised after the producer left its loop
    const int armed = sh.armed;
    for (int j = armed > STAGES ? armed - STAGES : 0; j < armed; ++j)
      mbar_drain(&sh.full[j % STAGES], (j / STAGES) & 1, &g_err);
  }
  if (warp == 1) {
    __syncwarp();
    fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Both GEMMs in one persistent launch (independent CTAs).  The tiles are
// numbered GEMM1 first (m-tile major), then GEMM2, and each CTA's producer
// claims the next number from a global counter whenever it starts a tile, so a
// CTA whose last GEMM1 tile ends early goes on with GEMM2 tiles while others
// finish GEMM1, instead of idling until the last GEMM1 CTA ends.  A GEMM2 tile
// reads the h rows of one m-tile, written by that m-tile's nt1 GEMM1 tiles:
// each of the four epilogue warps of a GEMM1 tile, once its h stores have
// completed, adds 1 to ready[m-tile] (release), and the producer of a GEMM2
// tile waits, bounded, until ready[m-tile] = 4 nt1 (acquire) before loading the
// rows.  A tile is claimed only by a CTA that is running, GEMM1 tiles wait for
// nothing, and every GEMM1 tile is numbered before every GEMM2 tile, so each
// GEMM1 tile a GEMM2 tile waits for belongs to a running CTA that finishes it:
// no CTA has to be resident for another to progress (a kernel on another stream
// may hold SMs meanwhile).
// ---------------------------------------------------------------------------
// Upper bound on the m-tiles of P rows in G groups: the size of the ready counters.
__host__ __device__ __forceinline__ int mtiles_max_of(int P, int G) { return (P + BM - 1) / BM + G; }

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Orders this thread's async-proxy (TMA) global accesses with its generic ones.
__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

__global__ void __launch_bounds__(THREADS, 1)
ffn_fused_kernel(const __grid_constant__ CUtensorMap map_a1, const __grid_constant__ CUtensorMap map_b1,
                 const __grid_constant__ CUtensorMap map_o1, const __grid_constant__ CUtensorMap map_a2,
                 const __grid_constant__ CUtensorMap map_b2, const __grid_constant__ CUtensorMap map_o2,
                 const int32_t* __restrict__ offsets, const int32_t* __restrict__ phys_to_expert, int G, int P,
                 int E, int H, int I, int nt1, int nt2, __nv_bfloat16* __restrict__ h, __nv_bfloat16* __restrict__ y,
                 int* __restrict__ ready, int ready_extra) {
  pdl_trigger();  // the kernel after it may start its setup
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* stage_a = smem_raw + pad;
  unsigned char* stage_b = stage_a + STAGES * A_BYTES;
  unsigned char* out_stage = stage_a + STAGES * STAGE_BYTES;
  Shared& sh = *reinterpret_cast<Shared*>(out_stage + OUT_STAGE_BYTES);
  // tiles are claimed one at a time from a counter (next, after the ready
  // counters); the producer passes each to the MMA and the epilogue through a
  // ring (the producer runs at most STAGES tiles ahead of the MMA and that at
  // most 2 ahead of the epilogue, so 16 slots are never overtaken)
  constexpr int kRing = 16;
  __shared__ int tile_ring[kRing];
  __shared__ uint64_t tile_bar[kRing];
  volatile int* abort_flag = &sh.abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh.tfull[a], 1);
      mbar_init(&sh.tempty[a], 128);
    }
    mbar_init(&sh.done, 1);
    for (int i = 0; i < kRing; ++i) mbar_init(&tile_bar[i], 1);
    sh.abort_flag = 0;
    sh.armed = 0;
    mbar_init_fence();
    prefetch_map(&map_a1);
    prefetch_map(&map_b1);
    prefetch_map(&map_o1);
    prefetch_map(&map_a2);
    prefetch_map(&map_b2);
    prefetch_map(&map_o2);
  }
  if (warp == 1) tmem_alloc(&sh.tmem_base, TMEM_COLS);
  pdl_wait();  // the rows and group offsets the kernels before it wrote
  for (int g = threadIdx.x; g <= G; g += blockDim.x) sh.off[g] = offsets ? offsets[g] : (g == 0 ? 0 : P);
  for (int g = threadIdx.x; g < G; g += blockDim.x) sh.pe[g] = phys_to_expert ? phys_to_expert[g] : 0;
  __syncthreads();
  if (warp == 0) {  // exclusive prefix of m-tiles per group, 8 groups per lane
    int cnt[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int g = lane * 8 + i;
      int c = 0;
      if (g < G) {
        const int lo = sh.off[g], hi = sh.off[g + 1], e = sh.pe[g];
        if (lo < 0 || hi < lo || hi > P) atomicOr(&g_err, SEMMOE_DEVERR_PAIRS);
        else if (e < 0 || e >= E) atomicOr(&g_err, SEMMOE_DEVERR_EXPERT);
        else c = (hi - lo + BM - 1) / BM;
      }
      cnt[i] = c;
      sum += c;
    }
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int g = lane * 8 + i;
      if (g < G) sh.tp[g] = run;
      run += cnt[i];
    }
    if (lane == 31) {
      sh.tp[G] = incl;
      sh.total_mtiles = incl;
    }
  }
  fence_before();
  __syncthreads();
  fence_after();

  const uint32_t tmem = sh.tmem_base;
  const int mtiles = sh.total_mtiles;
  const int total1 = mtiles * nt1, total = total1 + mtiles * nt2;
  int* next = ready + (mtiles_max_of(P, G));  // the tile counter
  // tile u: GEMM1 (m-tile, n-tile) for u < total1, else GEMM2
  auto tile_of = [&](int u, bool& g2, int& mt, int& nt) {
    g2 = u >= total1;
    const int v = g2 ? u - total1 : u, nn = g2 ? nt2 : nt1;
    mt = v / nn;
    nt = v - mt * nn;
  };

  if (warp == 0) {
    if (lane == 0) {  // TMA producer: claims tiles, hands each to the MMA and the epilogue
      uint32_t it = 0;
      for (int k = 0;; ++k) {
        const int u = *abort_flag ? total : atomicAdd(next, 1);
        tile_ring[k % kRing] = u;  // total or more: no more tiles
        mbar_arrive(&tile_bar[k % kRing]);
        if (u >= total) break;
        bool g2;
        int mt, nt, row0, rows, e;
        tile_of(u, g2, mt, nt);
        decode_mtile<1>(sh, G, mt, 0, row0, rows, e);
        if (g2) {  // the m-tile's h rows: all its GEMM1 tiles published (4 epilogue warps each)
          const uint64_t t_start = globaltimer_ns();
          bool ok = true;
          for (uint32_t polls = 0; ld_acquire_gpu(ready + mt) < 4 * nt1 + ready_extra; ++polls) {
            if (*abort_flag) { ok = false; break; }
            if (globaltimer_ns() - t_start > kWaitNs || polls > kWaitPolls) {
              atomicOr(&g_err, SEMMOE_DEVERR_TIMEOUT);
              *abort_flag = 1;
              ok = false;
              break;
            }
          }
          if (!ok) break;
          fence_async_global();  // the TMA loads below come after the acquire
        }
        const int kb_n = ((g2 ? I : H) + BK - 1) / BK;
        bool ok = true;
        for (int kb = 0; kb < kb_n; ++kb) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&sh.empty[s], ph ^ 1, abort_flag, &g_err)) { ok = false; break; }
          mbar_expect_tx(&sh.full[s], STAGE_BYTES);
          unsigned char* b = stage_b + s * B_BYTES;
          if (g2) {
            tma_load_2d(stage_a + s * A_BYTES, &map_a2, &sh.full[s], kb * BK, row0);
            tma_load_3d(b, &map_b2, &sh.full[s], kb * BK, nt * BN, e);
          } else {
            tma_load_2d(stage_a + s * A_BYTES, &map_a1, &sh.full[s], kb * BK, row0);
            tma_load_4d(b, &map_b1, &sh.full[s], kb * BK, nt * 128, 0, e);
            tma_load_4d(b + B_BYTES / 2, &map_b1, &sh.full[s], kb * BK, nt * 128, 1, e);
          }
          ++it;
        }
        if (!ok) break;
      }
      *reinterpret_cast<volatile int*>(&sh.armed) = (int)it;  // for the drain after an abort
      if (*abort_flag)  // no TMA write may still be landing when the CTA exits
        for (uint32_t j = it > (uint32_t)STAGES ? it - STAGES : 0; j < it; ++j)
          mbar_drain(&sh.full[j % STAGES], (j / STAGES) & 1, &g_err);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      uint32_t it = 0, acc_it = 0;
      for (int tk = 0;; ++tk) {
        if (!mbar_wait(&tile_bar[tk % kRing], (uint32_t)(tk / kRing) & 1, abort_flag, &g_err)) break;
        const int u = tile_ring[tk % kRing];
        const uint32_t a = acc_it & 1, aph = (acc_it >> 1) & 1;
        if (!mbar_wait(&sh.tempty[a], aph ^ 1, abort_flag, &g_err)) break;
        if (u >= total) {  // tell the epilogue: a completion of the next accumulator phase with no tile
          mbar_arrive(&sh.tfull[a]);
          break;
        }
        bool g2;
        int mt, nt;
        tile_of(u, g2, mt, nt);
        const int kb_n = ((g2 ? I : H) + BK - 1) / BK;
        fence_after();
        const uint32_t d = tmem + a * ACC_COLS;
        bool ok = true;
        for (int kb = 0; kb < kb_n; ++kb) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&sh.full[s], ph, abort_flag, &g_err)) { ok = false; break; }
          fence_after();
          const uint32_t sa = smem_u32(stage_a + s * A_BYTES), sb = smem_u32(stage_b + s * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / UK; ++k)
            mma_bf16(d, sw128_desc(sa + k * UK * 2), sw128_desc(sb + k * UK * 2), kIdesc, (kb | k) != 0);
          commit(&sh.empty[s]);
          ++it;
        }
        if (!ok) break;
        commit(&sh.tfull[a]);
        ++acc_it;
      }
      commit(&sh.done);
      mbar_drain(&sh.done, 0, &g_err);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int q = warp & 3, r = q * 32 + lane;
    uint32_t acc_it = 0;
    ChunkOut co{&map_o1, out_stage + q * 4096, 0};
    for (int k = 0;; ++k) {
      const uint32_t a = acc_it & 1, aph = (acc_it >> 1) & 1;
      int ok = 1, u = 0;
      if (lane == 0) {
        ok = mbar_wait(&tile_bar[k % kRing], (uint32_t)(k / kRing) & 1, abort_flag, &g_err) &&
             mbar_wait(&sh.tfull[a], aph, abort_flag, &g_err);
        if (ok) u = tile_ring[k % kRing];
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      u = __shfl_sync(0xffffffffu, u, 0);
      if (!ok || u >= total) break;
      bool g2;
      int mt, nt, row0, rows, e;
      tile_of(u, g2, mt, nt);
      decode_mtile<1>(sh, G, mt, 0, row0, rows, e);
      fence_after();
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + a * ACC_COLS;
      const bool row_ok = r < rows;
      const bool full = q * 32 + 32 <= rows;  // all 32 rows of this warp lie in the group
      co.map = g2 ? &map_o2 : &map_o1;
      if (!g2) {  // GEMM1: accumulator columns [0, 128) gate, [128, 256) up; 128 h columns
        __nv_bfloat16* orow = h + (size_t)(row0 + (row_ok ? r : 0)) * I;
#pragma unroll 1
        for (int c = 0; c < 128; c += 64) {
          uint32_t g0[32], g1[32], u0[32], u1[32], w[32];
          tmem_ld32(t_row + c, g0);
          tmem_ld32(t_row + c + 32, g1);
          tmem_ld32(t_row + 128 + c, u0);
          tmem_ld32(t_row + 128 + c + 32, u1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            w[i] = pack_bf16x2(swiglu(g0[2 * i], u0[2 * i]), swiglu(g0[2 * i + 1], u0[2 * i + 1]));
            w[16 + i] = pack_bf16x2(swiglu(g1[2 * i], u1[2 * i]), swiglu(g1[2 * i + 1], u1[2 * i + 1]));
          }
          emit_chunk(co, w, full, row_ok, orow, nt * 128 + c, I, row0 + q * 32, lane);
        }
      } else {  // GEMM2: 256 y columns
        __nv_bfloat16* orow = y + (size_t)(row0 + (row_ok ? r : 0)) * H;
#pragma unroll 1
        for (int c = 0; c < BN; c += 64) {
          uint32_t y0[32], y1[32], w[32];
          tmem_ld32(t_row + c, y0);
          tmem_ld32(t_row + c + 32, y1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            w[i] = pack_bf16x2(__uint_as_float(y0[2 * i]), __uint_as_float(y0[2 * i + 1]));
            w[16 + i] = pack_bf16x2(__uint_as_float(y1[2 * i]), __uint_as_float(y1[2 * i + 1]));
          }
          emit_chunk(co, w, full, row_ok, orow, nt * BN + c, H, row0 + q * 32, lane);
        }
      }
      fence_before();
      mbar_arrive(&sh.tempty[a]);  // the MMA may reuse the accumulator while this warp publishes
      ++acc_it;
      if (!g2) {  // this warp's h rows of the m-tile, written (TMA stores and direct stores) and visible
        if (lane == 0) {
          bulk_wait_all();       // its TMA stores have completed
          fence_async_global();  // ... and are ordered before the release below
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          atomicAdd(ready + mt, 1);
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // this warp's output stores are complete
  }

  fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {  // also an abort raised after the producer left its loop
    const int armed = sh.armed;
    for (int j = armed > STAGES ? armed - STAGES : 0; j < armed; ++j)
      mbar_drain(&sh.full[j % STAGES], (j / STAGES) & 1, &g_err);
  }
  if (warp == 1) {
    __syncwarp();
    fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Zeroes the one-launch FFN's readiness and tile counters; waits for the
// kernel before it so that the FFN after it, waiting for this one, also
// finds that kernel's writes (see pdl_wait).
__global__ void __launch_bounds__(256) zero_counters_kernel(int* __restrict__ p, int n) {
  pdl_trigger();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = 0;
  pdl_wait();
}

cudaError_t launch_fused(const CUtensorMap& ma1, const CUtensorMap& mb1, const CUtensorMap& mo1,
                         const CUtensorMap& ma2, const CUtensorMap& mb2, const CUtensorMap& mo2, const int32_t* offsets,
                         const int32_t* p2e, int G, int P, int E, int H, int I, __nv_bfloat16* h, __nv_bfloat16* y,
                         int* ready, cudaStream_t s, int ready_extra, bool dependent) {
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = ensure_smem_limit(ffn_fused_kernel, (int)kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  const int nt1 = (I + 127) / 128, nt2 = (H + BN - 1) / BN;
  const long long mtiles_max = mtiles_max_of(P, G);
  const int n_counters = (int)(mtiles_max + 1);  // + the tile counter
  e = launch_kernel(zero_counters_kernel, dim3((n_counters + 255) / 256), dim3(256), 0, s, 1, dependent, ready,
                    n_counters);
  if (e != cudaSuccess) return e;
  count_launches(1);
  const long long max_units = mtiles_max * (nt1 + nt2);
  int grid = sm_count();  // one CTA per SM (shared memory)
  if (max_units < grid) grid = (int)max_units;
  e = launch_kernel(ffn_fused_kernel, dim3(grid), dim3(THREADS), kSmemBytes, s, 1, dependent, ma1, mb1, mo1, ma2, mb2,
                    mo2, offsets, p2e, G, P, E, H, I, nt1, nt2, h, y, ready, ready_extra);
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// 2-SM variant: clusters of two CTAs on two SMs run
// tcgen05.mma.cta_group::2 with M = 256.  Each CTA stages its own 128 A rows and
// half of the 256-row weight tile (CTA 0 the gate / first half, CTA 1 the up /
// second half); the pair's even CTA issues the MMAs, and each CTA's TMEM holds
// the accumulator rows of its own A rows.  Per SM and k-block that is 32 KB of
// TMA writes and 32 KB of MMA operand reads instead of 48 + 48 KB.
// ---------------------------------------------------------------------------
constexpr int P_STAGES = 6;
constexpr int P_B_BYTES = 128 * BK * 2;             // half of the 256-row weight tile
constexpr int P_STAGE_BYTES = A_BYTES + P_B_BYTES;  // 32 KB

struct PairShared {
  uint64_t full[P_STAGES], empty[P_STAGES], tfull[2], tempty[2], done;
  uint32_t tmem_base;
  int abort_flag;
  int total_mtiles;
  int off[MAX_GROUPS + 1];
  int pe[MAX_GROUPS];
  int tp[MAX_GROUPS + 1];
};

constexpr size_t kPairSmemBytes = 1024 + (size_t)P_STAGES * P_STAGE_BYTES + OUT_STAGE_BYTES + sizeof(PairShared);
constexpr uint32_t kIdescPair = idesc_bf16_f32(2 * BM, BN);

template <bool GLU, int NBUF, bool SC = false>
__global__ void __launch_bounds__(THREADS, 1)
ffn_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                const __grid_constant__ CUtensorMap map_out,
                const int32_t* __restrict__ offsets, const int32_t* __restrict__ phys_to_expert, int G, int P,
                int E, int N, int K, int n_tiles, const int32_t* __restrict__ gather, int gather_div, int gather_rows,
                __nv_bfloat16* __restrict__ out, Scatter sc) {
  pdl_trigger();  // the kernel after it may start its setup
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* ring = smem_raw + pad;  // stage s: A [128 x 64] then B half [128 x 64]
  unsigned char* out_stage = ring + P_STAGES * P_STAGE_BYTES;  // OUT_STAGE_BYTES, 1024-aligned
  PairShared& sh = *reinterpret_cast<PairShared*>(out_stage + OUT_STAGE_BYTES);
  volatile int* abort_flag = &sh.abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int rank = (int)cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(&sh.full[s], 1);   // the leader's arrive.expect_tx; both CTAs' bytes
      mbar_init(&sh.empty[s], 1);  // the pair MMA's commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh.tfull[a], 1);
      mbar_init(&sh.tempty[a], 2 * 128);  // both CTAs' epilogue threads (leader's copy is used)
    }
    mbar_init(&sh.done, 1);
    sh.abort_flag = 0;
    mbar_init_fence();
    prefetch_map(&map_a);
    prefetch_map(&map_b);
    prefetch_map(&map_out);
  }
  if (warp == 1) tmem_alloc_pair(&sh.tmem_base, NBUF * ACC_COLS);
  pdl_wait();  // the rows and group offsets the kernels before it wrote
  for (int g = threadIdx.x; g <= G; g += THREADS) sh.off[g] = offsets ? offsets[g] : (g == 0 ? 0 : P);
  for (int g = threadIdx.x; g < G; g += THREADS) sh.pe[g] = phys_to_expert ? phys_to_expert[g] : 0;
  __syncthreads();
  if (warp == 0) {  // exclusive prefix of m-tile pairs per group, 8 groups per lane
    int cnt[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int g = lane * 8 + i;
      int c = 0;
      if (g < G) {
        const int lo = sh.off[g], hi = sh.off[g + 1], e = sh.pe[g];
        if (lo < 0 || hi < lo || hi > P) atomicOr(&g_err, SEMMOE_DEVERR_PAIRS);
        else if (e < 0 || e >= E) atomicOr(&g_err, SEMMOE_DEVERR_EXPERT);
        else c = ((hi - lo + BM - 1) / BM + 1) / 2;
      }
      cnt[i] = c;
      sum += c;
    }
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int g = lane * 8 + i;
      if (g < G) sh.tp[g] = run;
      run += cnt[i];
    }
    if (lane == 31) {
      sh.tp[G] = incl;
      sh.total_mtiles = incl;
    }
  }
  fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers and TMEM exist before anything crosses the pair
  fence_after();

  const uint32_t tmem = sh.tmem_base;
  const int total = sh.total_mtiles * n_tiles;
  const int kb_n = (K + BK - 1) / BK;
  const int unit0 = blockIdx.x / 2, units = gridDim.x / 2;

  if (warp == 0) {  // TMA producer (both CTAs): own A rows + own half of B, counted on the leader's barrier
    uint32_t it = 0;
    int s = 0;          // stage of k-block `it` ...
    uint32_t ph = 0;    // ... and the parity of its use
    const uint32_t fb0 = mapa_rank(&sh.full[0], 0);  // the leader's barriers, 8 bytes apart
    if (gather != nullptr || lane == 0)  // without row gathers lane 0 alone: 1% faster than the warp
    for (int tile = unit0; tile < total; tile += units) {
      if (*abort_flag) break;
      const int mt = tile / n_tiles, nt = tile % n_tiles;
      int row0, rows, e;
      decode_mtile<2>(sh, G, mt, rank, row0, rows, e);
      int src[4] = {0, 0, 0, 0};
      if (gather != nullptr) gather_sources(gather, gather_div, gather_rows, P, row0, lane, src);
      bool ok = true;
      for (int kb = 0; kb < kb_n; ++kb) {
        int good = 1;
        if (lane == 0) good = mbar_wait(&sh.empty[s], ph ^ 1, abort_flag, &g_err);
        if (gather != nullptr ? !__shfl_sync(0xffffffffu, good, 0) : !good) { ok = false; break; }
        if (lane == 0 && leader) mbar_expect_tx(&sh.full[s], 2 * P_STAGE_BYTES);
        const uint32_t fb = fb0 + 8u * s;
        unsigned char* st = ring + (size_t)s * P_STAGE_BYTES;
        if (gather != nullptr)
          tma_gather4_pair(st + lane * 4 * (BK * 2), &map_a, fb, kb * BK, src[0], src[1], src[2], src[3]);
        else if (lane == 0)
          tma_load_2d_pair(st, &map_a, fb, kb * BK, row0);
        if (lane == 0) {
          if (GLU) tma_load_4d_pair(st + A_BYTES, &map_b, fb, kb * BK, nt * 128, rank, e);
          else tma_load_3d_pair(st + A_BYTES, &map_b, fb, kb * BK, nt * BN + rank * 128, e);
        }
        ++it;
        if (++s == P_STAGES) {
          s = 0;
          ph ^= 1;
        }
      }
      if (!ok) break;
    }
    if (lane == 0 && *abort_flag && leader) {
      for (uint32_t j = it > (uint32_t)P_STAGES ? it - P_STAGES : 0; j < it; ++j)
        mbar_drain(&sh.full[j % P_STAGES], (j / P_STAGES) & 1, &g_err);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {  // MMA issuer: the pair's even CTA only
      uint32_t acc_it = 0, ph = 0;
      int s = 0;
      for (int tile = unit0; tile < total; tile += units) {
        if (*abort_flag) break;
        const uint32_t a = acc_it % NBUF, aph = (acc_it / NBUF) & 1;
        if (!mbar_wait(&sh.tempty[a], aph ^ 1, abort_flag, &g_err)) break;
        fence_after();
        const uint32_t d = tmem + a * ACC_COLS;
        bool ok = true;
        for (int kb = 0; kb < kb_n; ++kb) {
          if (!mbar_wait(&sh.full[s], ph, abort_flag, &g_err)) { ok = false; break; }
          fence_after();
          const uint32_t sa = smem_u32(ring + (size_t)s * P_STAGE_BYTES), sb = sa + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / UK; ++k)
            mma_bf16_pair(d, sw128_desc(sa + k * UK * 2), sw128_desc(sb + k * UK * 2), kIdescPair, (kb | k) != 0);
          commit_pair_mc(&sh.empty[s], 0x3);  // both CTAs may refill this stage
          if (++s == P_STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        commit_pair_mc(&sh.tfull[a], 0x3);    // both CTAs' accumulator rows are ready
        ++acc_it;
      }
      commit_pair_mc(&sh.done, 0x1);
      mbar_drain(&sh.done, 0, &g_err);
    }
  } else {  // epilogue (both CTAs): this CTA's 128 rows of the 256-row tile
    const int q = warp & 3, r = q * 32 + lane;
    uint32_t acc_it = 0;
    ChunkOut co{&map_out, out_stage + q * 4096, 0};
    for (int tile = unit0; tile < total; tile += units) {
      const int mt = tile / n_tiles, nt = tile % n_tiles;
      int row0, rows, e;
      decode_mtile<2>(sh, G, mt, rank, row0, rows, e);
      const uint32_t a = acc_it % NBUF, aph = (acc_it / NBUF) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&sh.tfull[a], aph, abort_flag, &g_err);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      fence_after();
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + a * ACC_COLS;
      const bool row_ok = r < rows;
      __nv_bfloat16* orow = out + (size_t)(row0 + (row_ok ? r : 0)) * N;
      const bool full = q * 32 + 32 <= rows;  // all 32 rows of this warp lie in the group
      if (GLU) {  // accumulator columns [0, 128) gate, [128, 256) up; 128 output columns
#pragma unroll 1
        for (int c = 0; c < 128; c += 64) {
          uint32_t g0[32], g1[32], u0[32], u1[32], w[32];
          tmem_ld32(t_row + c, g0);
          tmem_ld32(t_row + c + 32, g1);
          tmem_ld32(t_row + 128 + c, u0);
          tmem_ld32(t_row + 128 + c + 32, u1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            w[i] = pack_bf16x2(swiglu(g0[2 * i], u0[2 * i]), swiglu(g0[2 * i + 1], u0[2 * i + 1]));
            w[16 + i] = pack_bf16x2(swiglu(g1[2 * i], u1[2 * i]), swiglu(g1[2 * i + 1], u1[2 * i + 1]));
          }
          emit_chunk(co, w, full, row_ok, orow, nt * 128 + c, N, row0 + q * 32, lane);
        }
      } else if (SC) {  // rows weighted and added into the token-order output
        int st;
        float sg;
        scatter_row(sc, row0 + (row_ok ? r : 0), row_ok, st, sg);
#pragma unroll 1
        for (int c = 0; c < BN; c += 64) {
          if (nt * BN + c >= N) break;
          uint32_t y0[32], y1[32];
          tmem_ld32(t_row + c, y0);
          tmem_ld32(t_row + c + 32, y1);
          tmem_ld_wait();
          scatter_half(sc, co.stage, y0, st, sg, nt * BN + c, N, lane);
          scatter_half(sc, co.stage, y1, st, sg, nt * BN + c + 32, N, lane);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN; c += 64) {
          uint32_t y0[32], y1[32], w[32];
          tmem_ld32(t_row + c, y0);
          tmem_ld32(t_row + c + 32, y1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            w[i] = pack_bf16x2(__uint_as_float(y0[2 * i]), __uint_as_float(y0[2 * i + 1]));
            w[16 + i] = pack_bf16x2(__uint_as_float(y1[2 * i]), __uint_as_float(y1[2 * i + 1]));
          }
          emit_chunk(co, w, full, row_ok, orow, nt * BN + c, N, row0 + q * 32, lane);
        }
      }
      fence_before();
      mbar_arrive_cluster(mapa_rank(&sh.tempty[a], 0));  // the leader's MMA may reuse this buffer
      ++acc_it;
    }
    if (lane == 0) bulk_wait_all();  // this warp's output stores are complete
  }

  fence_before();
  __syncthreads();
  cluster_sync_all();  // nothing crosses the pair any more
  if (warp == 1) {
    __syncwarp();
    fence_after();
    tmem_dealloc_pair(tmem, NBUF * ACC_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// gather != nullptr: the A operand's sorted row q is x row gather[q] / gather_div
// (ma then maps x with one-row boxes).
struct Gather {
  const int32_t* rows = nullptr;
  int div = 1, n = 0;
  const __nv_bfloat16* x = nullptr;
};

template <bool GLU, int GW = 0, bool SC = false>
cudaError_t launch_one(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo, const int32_t* offsets,
                       const int32_t* p2e,
                       int G, int P, int E, int N, int K, int n_tiles, Gather ga, __nv_bfloat16* out,
                       cudaStream_t s, bool dependent, Scatter sc = Scatter()) {
  auto kern = ffn_tc_kernel<GLU, GW, SC>;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = ensure_smem_limit(kern, (int)kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  const long long max_units = ((long long)(P + BM - 1) / BM + G) * n_tiles;  // >= tile units of any grouping
  int grid = sm_count();
  if (max_units < grid) grid = (int)max_units;
  e = launch_kernel(kern, dim3(grid), dim3(THREADS + 32 * GW), kSmemBytes, s, 1, dependent, ma, mb, mo, offsets, p2e,
                    G, P, E, N, K, n_tiles, ga.rows, ga.div, ga.n, out, ga.x, sc);
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaGetLastError();
}

template <bool GLU, int NBUF, bool SC = false>
cudaError_t launch_pair(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo, const int32_t* offsets,
                        const int32_t* p2e,
                        int G, int P, int E, int N, int K, int n_tiles, Gather ga, __nv_bfloat16* out,
                        cudaStream_t s, bool dependent, Scatter sc = Scatter()) {
  auto kern = ffn_pair_kernel<GLU, NBUF, SC>;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = ensure_smem_limit(kern, (int)kPairSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  const long long max_units = ((long long)(P + BM - 1) / BM + G) * n_tiles;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = kPairSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(sm_count() / 2 * 2);
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  long long units = clusters;
  if (max_units < units) units = max_units;
  e = launch_kernel(kern, dim3((unsigned)(units * 2)), dim3(THREADS), kPairSmemBytes, s, 2, dependent, ma, mb, mo,
                    offsets, p2e, G, P, E, N, K, n_tiles, ga.rows, ga.div, ga.n, out, sc);
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

int ffn_tc_take_errors(cudaStream_t s, int* bits) { return take_error_word(g_err, s, bits); }

// Grouped-GEMM form of one GEMM (SEMMOE_FORM_*).  The default picks, from the
// shapes alone: GEMM1 (K = H) in 2-SM pairs when the groups average at least
// 512 rows (P >= 512 G), GEMM2 (K = I) when I >= 512 and they average at least
// 256 (P >= 256 G), independent CTAs otherwise (measured per GEMM on the
// DeepSeek, Qwen3 and MoE-Prism shapes).  A pair covers two m-tiles of one
// group, so short groups leave half of it idle.  A GEMM1 that gathers its rows
// runs in the single-CTA form, where gathering warps feed it (2.1x faster than
// TMA row gathers from the producer warp at the DeepSeek shape; gathering warps
// in the 2-SM form measured twice as slow as in the single-CTA form).
static int resolve_form(int form, bool glu, int I, int P, int G, bool gathered) {
  if (form != SEMMOE_FORM_DEFAULT) return form;
  if (glu) return !gathered && (long long)P >= 4LL * BM * G ? SEMMOE_FORM_PAIR : SEMMOE_FORM_SINGLE;
  return (I >= 512 && (long long)P >= 2LL * BM * G) ? SEMMOE_FORM_PAIR : SEMMOE_FORM_SINGLE;
}

// One GEMM of the FFN in a resolved form.
template <bool GLU>
static cudaError_t launch_gemm(int form, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo,
                               const int32_t* offsets, const int32_t* p2e, int G, int P, int E, int N, int K,
                               int n_tiles, Gather ga, __nv_bfloat16* out, cudaStream_t s, bool dep,
                               const Scatter* sc = nullptr) {
  if constexpr (!GLU) {
    if (sc != nullptr) {  // GEMM2 adding its rows into the token-order output
      if (form == SEMMOE_FORM_PAIR1)
        return launch_pair<false, 1, true>(ma, mb, mo, offsets, p2e, G, P, E, N, K, n_tiles, ga, out, s, dep, *sc);
      if (form == SEMMOE_FORM_PAIR)
        return launch_pair<false, 2, true>(ma, mb, mo, offsets, p2e, G, P, E, N, K, n_tiles, ga, out, s, dep, *sc);
      return launch_one<false, 0, true>(ma, mb, mo, offsets, p2e, G, P, E, N, K, n_tiles, ga, out, s, dep, *sc);
    }
  }
  switch (form) {
    case SEMMOE_FORM_PAIR1:
      return launch_pair<GLU, 1>(ma, mb, mo, offsets, p2e, G, P, E, N, K, n_tiles, ga, out, s, dep);
    case SEMMOE_FORM_PAIR:
      return launch_pair<GLU, 2>(ma, mb, mo, offsets, p2e, G, P, E, N, K, n_tiles, ga, out, s, dep);
    case SEMMOE_FORM_SINGLE_TMA_GATHER:  // gathered rows by TMA four-row gathers from the producer warp
      return launch_one<GLU>(ma, mb, mo, offsets, p2e, G, P, E, N, K, n_tiles, ga, out, s, dep);
    default:
      if constexpr (GLU) {
        if (ga.rows != nullptr)  // gathered rows: gathering warps
          return launch_one<GLU, GATHER_WARPS>(ma, mb, mo, offsets, p2e, G, P, E, N, K, n_tiles, ga, out, s, dep);
      }
      return launch_one<GLU>(ma, mb, mo, offsets, p2e, G, P, E, N, K, n_tiles, ga, out, s, dep);
  }
}

// gather_rows != nullptr: x is the unpermuted [T_x, H] activation and sorted row
// q of GEMM1 reads x row gather_rows[q] / gather_div.
// acc != nullptr: GEMM2 adds each row, weighted by topk_w[sorted_to_pair[q]],
// into acc [T_acc, H] fp32 (row of token sorted_to_pair[q] / k_max) instead of
// writing y.
// fused_stall != 0 (failure-path self-test only): both GEMMs in one launch,
// with every GEMM2 tile waiting for one readiness count more than its m-tile's
// GEMM1 tiles ever publish, so each of those waits runs out.
// dependent: every launch is a programmatic dependent of the kernel before it
// on s (launch_kernel); false for work that runs beside the layer's chain.
cudaError_t launch_ffn_tc(const void* x, const int32_t* offsets, const int32_t* p2e, const void* w13,
                          const void* w2, int P, int E, int H, int I, void* y, void* ws, const int32_t* gather_rows,
                          int gather_div, int T_x, int form1, int form2, cudaStream_t s, const int32_t* sorted_to_pair,
                          const float* topk_w, int k_max, int T_acc, float* acc, int fused_stall, bool dependent) {
  if (P == 0) return cudaSuccess;
  const int G = offsets ? E : 1;
  int mode1 = resolve_form(form1, true, I, P, G, gather_rows != nullptr);
  int mode2 = resolve_form(form2, false, I, P, G, false);
  // where both GEMMs run in independent CTAs by default (groups of few rows), one
  // launch for both: routed FFN, decode T = 64 / 256 / 512, 171 / 175 / 179 us
  // against 180 / 184 / 189 us (GEMM1's last wave no longer idles half the SMs)
  if (form1 == SEMMOE_FORM_DEFAULT && form2 == SEMMOE_FORM_DEFAULT && gather_rows == nullptr && acc == nullptr &&
      mode1 == SEMMOE_FORM_SINGLE && mode2 == SEMMOE_FORM_SINGLE)
    mode1 = mode2 = SEMMOE_FORM_FUSED;
  if (fused_stall) mode1 = mode2 = SEMMOE_FORM_FUSED;
  const bool fused = mode1 == SEMMOE_FORM_FUSED && gather_rows == nullptr && acc == nullptr;
  // GEMM2's weight box: 256 rows for independent CTAs, 128 for a pair CTA's half of the tile
  const int CL = (mode2 == SEMMOE_FORM_SINGLE || fused) ? 1 : 2;
  const cuuint64_t es = 2;
  CUtensorMap ma1, mb1, ma2, mb2;
  Gather ga;
  if (gather_rows != nullptr) {  // x rows fetched by row gathers: one-row boxes
    ga.rows = gather_rows;
    ga.div = gather_div;
    ga.n = T_x;
    ga.x = static_cast<const __nv_bfloat16*>(x);
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)T_x};
    const cuuint64_t str[1] = {(cuuint64_t)H * es};
    const cuuint32_t box[2] = {BK, 1};
    if (!make_map_bf16(&ma1, x, 2, dims, str, box)) return cudaErrorInvalidValue;
  } else {
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)P};
    const cuuint64_t str[1] = {(cuuint64_t)H * es};
    const cuuint32_t box[2] = {BK, BM};
    if (!make_map_bf16(&ma1, x, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[4] = {(cuuint64_t)H, (cuuint64_t)I, 2, (cuuint64_t)E};
    const cuuint64_t str[3] = {(cuuint64_t)H * es, (cuuint64_t)I * H * es, (cuuint64_t)2 * I * H * es};
    const cuuint32_t box[4] = {BK, 128, 1, 1};
    if (!make_map_bf16(&mb1, w13, 4, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)I, (cuuint64_t)P};
    const cuuint64_t str[1] = {(cuuint64_t)I * es};
    const cuuint32_t box[2] = {BK, BM};
    if (!make_map_bf16(&ma2, ws, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)I, (cuuint64_t)H, (cuuint64_t)E};
    const cuuint64_t str[2] = {(cuuint64_t)I * es, (cuuint64_t)H * I * es};
    const cuuint32_t box[3] = {BK, (cuuint32_t)(BN / CL), 1};  // a pair CTA loads half of the tile
    if (!make_map_bf16(&mb2, w2, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  // outputs h [P, I] and y [P, H], written by the epilogue's TMA stores in
  // boxes of 32 rows x 32 columns (64-byte rows, 64-byte swizzle)
  CUtensorMap mo1, mo2;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)I, (cuuint64_t)P};
    const cuuint64_t str[1] = {(cuuint64_t)I * es};
    const cuuint32_t box[2] = {32, 32};
    if (!make_map_bf16(&mo1, ws, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return cudaErrorInvalidValue;
  }
  if (acc == nullptr) {
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)P};
    const cuuint64_t str[1] = {(cuuint64_t)H * es};
    const cuuint32_t box[2] = {32, 32};
    if (!make_map_bf16(&mo2, y, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return cudaErrorInvalidValue;
  } else {
    mo2 = mo1;  // no y: GEMM2 adds into acc (the map is not used)
  }
  Scatter sc;
  sc.pairs = sorted_to_pair;
  sc.gates = topk_w;
  sc.div = k_max;
  sc.T = T_acc;
  sc.acc = acc;
  __nv_bfloat16* h = static_cast<__nv_bfloat16*>(ws);
  __nv_bfloat16* yb = static_cast<__nv_bfloat16*>(y);
  if (fused) {
    int* ready = reinterpret_cast<int*>(static_cast<unsigned char*>(ws) + align_up((size_t)P * I * 2, 256));
    return launch_fused(ma1, mb1, mo1, ma2, mb2, mo2, offsets, p2e, G, P, E, H, I, h, yb, ready, s, fused_stall ? 1 : 0,
                        dependent);
  }
  cudaError_t e = launch_gemm<true>(mode1, ma1, mb1, mo1, offsets, p2e, G, P, E, I, H, (I + 127) / 128, ga, h, s,
                                    dependent);
  if (e != cudaSuccess) return e;
  return launch_gemm<false>(mode2, ma2, mb2, mo2, offsets, p2e, G, P, E, H, I, (H + BN - 1) / BN, Gather(), yb, s,
                            dependent, acc != nullptr ? &sc : nullptr);
}

}  // namespace semmoe
