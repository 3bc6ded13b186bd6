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
// fp32 logits.  When every expert fits one pass and k_max <= 16, the epilogue
// also does the top-k and the gates (one token per thread), so the logits never
// go through memory.  Waits are bounded as in the grouped-FFN kernel.
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace semmoe {
namespace {

using namespace tc;

__device__ int g_err;

constexpr int BM = 128, BK = 64, UK = 16, STAGES = 4, THREADS = 192;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int MAX_NB = 256;                     // MMA N limit
constexpr int B_BYTES_MAX = MAX_NB * BK * 2;    // 32 KB
constexpr uint32_t TMEM_COLS = 256;

struct Shared {
  uint64_t full[STAGES], empty[STAGES], tfull, done;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t kSmemBytes = 1024 + (size_t)STAGES * (A_BYTES + B_BYTES_MAX) + sizeof(Shared);

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

// Outputs of the fused top-k (every field unused unless TOPK).
struct TopkOut {
  const int32_t* k_per_token;  // nullable: k_uniform then
  int k_uniform, k_max;
  int32_t* topk_idx;
  float* topk_w;
};

constexpr int KREG = 16;  // largest k_max the fused top-k keeps in registers

template <int S, bool TOPK>
__global__ void __launch_bounds__(THREADS, 1)
route_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w, int T, int H,
                int E, int EC, float* __restrict__ logits, TopkOut tk) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* stage_a = smem_raw + pad;
  unsigned char* stage_b = stage_a + STAGES * A_BYTES;
  Shared& sh = *reinterpret_cast<Shared*>(stage_b + STAGES * B_BYTES_MAX);
  volatile int* abort_flag = &sh.abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int NB = S * EC;
  const uint32_t b_bytes = (uint32_t)NB * BK * 2;
  const int t0 = blockIdx.x * BM, pass = blockIdx.y;
  const int kb_n = (H + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
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
        const int s = kb % STAGES;
        const uint32_t ph = (kb / STAGES) & 1;
        if (!mbar_wait(&sh.empty[s], ph ^ 1, abort_flag, &g_err)) break;
        mbar_expect_tx(&sh.full[s], A_BYTES + b_bytes);
        tma_load_2d(stage_a + s * A_BYTES, &map_x, &sh.full[s], kb * BK, t0);
        tma_load_2d(stage_b + s * B_BYTES_MAX, &map_w, &sh.full[s], kb * BK, pass * NB);
        ++it;
      }
      if (*abort_flag)
        for (int j = it > STAGES ? it - STAGES : 0; j < it; ++j)
          mbar_drain(&sh.full[j % STAGES], (j / STAGES) & 1, &g_err);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      const uint32_t idesc = idesc_bf16_f32(BM, NB);
      bool ok = true;
      for (int kb = 0; kb < kb_n; ++kb) {
        const int s = kb % STAGES;
        const uint32_t ph = (kb / STAGES) & 1;
        if (!mbar_wait(&sh.full[s], ph, abort_flag, &g_err)) { ok = false; break; }
        fence_after();
        const uint32_t sa = smem_u32(stage_a + s * A_BYTES), sb = smem_u32(stage_b + s * B_BYTES_MAX);
#pragma unroll
        for (int k = 0; k < BK / UK; ++k)
          mma_bf16(tmem, sw128_desc(sa + k * UK * 2), sw128_desc(sb + k * UK * 2), idesc, (kb | k) != 0);
        commit(&sh.empty[s]);
      }
      if (ok) commit(&sh.tfull);
      commit(&sh.done);
      mbar_drain(&sh.done, 0, &g_err);
    }
  } else {  // epilogue: one token row per thread
    const int q = warp & 3, r = q * 32 + lane, t = t0 + r;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(&sh.tfull, 0, abort_flag, &g_err);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      fence_after();
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
      float* lrow = logits != nullptr ? logits + (size_t)(t < T ? t : 0) * E : nullptr;
      // Fused top-k (single pass, experts in ascending order): a register list
      // sorted by logit descending; a new logit enters only if strictly larger
      // than the last entry and bubbles past strictly smaller ones, so equal
      // logits keep the lower expert index first.
      float bv[TOPK ? KREG : 1];
      int be[TOPK ? KREG : 1];
#pragma unroll
      for (int i = 0; i < (TOPK ? KREG : 1); ++i) { bv[i] = -INFINITY; be[i] = -1; }
      for (int c = 0; c < EC; c += 16) {
        uint32_t v0[16], v1[16], v2[16];
        tmem_ld16(trow + c, v0);
        if (S == 3) {
          tmem_ld16(trow + EC + c, v1);
          tmem_ld16(trow + 2 * EC + c, v2);
        }
        tmem_ld_wait();
        if (t < T) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int e = pass * EC + c + i;
            if (e < E) {
              float l = __uint_as_float(v0[i]);
              if (S == 3) l = (l + __uint_as_float(v1[i])) + __uint_as_float(v2[i]);
              if (lrow != nullptr) lrow[e] = l;
              if (TOPK) {
                if (!isfinite(l)) {
                  atomicOr(&g_err, SEMMOE_DEVERR_NONFINITE);
                  l = -INFINITY;
                }
                if (l > bv[KREG - 1]) {
                  bv[KREG - 1] = l;
                  be[KREG - 1] = e;
#pragma unroll
                  for (int j = KREG - 1; j > 0; --j) {
                    if (bv[j] > bv[j - 1]) {
                      const float tv = bv[j]; bv[j] = bv[j - 1]; bv[j - 1] = tv;
                      const int te = be[j]; be[j] = be[j - 1]; be[j - 1] = te;
                    }
                  }
                }
              }
            }
          }
        }
      }
      if (TOPK && t < T) {
        int kt = tk.k_per_token != nullptr ? tk.k_per_token[t] : tk.k_uniform;
        if (kt < 1 || kt > tk.k_max) {
          atomicOr(&g_err, SEMMOE_DEVERR_K);
          kt = kt < 1 ? 1 : tk.k_max;
        }
        // gates: softmax over the selected logits, renormalised (fp32)
        const float m = bv[0];
        float den = 0.f;
#pragma unroll
        for (int j = 0; j < KREG; ++j)
          if (j < kt && be[j] >= 0) den += expf(bv[j] - m);
        int32_t* irow = tk.topk_idx + (size_t)t * tk.k_max;
        float* wrow = tk.topk_w + (size_t)t * tk.k_max;
#pragma unroll
        for (int j = 0; j < KREG; ++j) {
          if (j < tk.k_max) {
            const bool live = j < kt && be[j] >= 0;
            if (j < kt && be[j] < 0) atomicOr(&g_err, SEMMOE_DEVERR_NONFINITE);
            irow[j] = live ? be[j] : -1;
            wrow[j] = live ? expf(bv[j] - m) / den : 0.f;
          }
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

}  // namespace

int route_tc_take_errors(cudaStream_t s, int* bits) { return take_error_word(g_err, s, bits); }

// Workspace of the tensor-core router: the three-part split of an fp32 weight.
size_t route_tc_split_bytes(int H, int E, int w_dtype) {
  if (w_dtype != SEMMOE_F32) return 0;
  const int EC = experts_per_pass(E, 3), n_pass = (E + EC - 1) / EC;
  return align_up((size_t)n_pass * 3 * EC * H * 2, 256);
}

// Whether the top-k can run in the router kernel's epilogue: every expert in
// one pass and k_max within the register list.
bool route_tc_fuses_topk(int E, int k_max, int w_dtype) {
  const int S = w_dtype == SEMMOE_F32 ? 3 : 1;
  return E <= experts_per_pass(E, S) && k_max <= KREG;
}

// x [T,H] bf16 (H % 8 == 0); w [E,H] fp32 or bf16; split: workspace of
// route_tc_split_bytes() (fp32 weight only).  Writes logits [T,E] (nullable
// when topk_idx is set) and, when topk_idx != nullptr (only if
// route_tc_fuses_topk), the top-k indices and gates.
cudaError_t launch_route_logits_tc(const void* x, const void* w, int w_dtype, int T, int H, int E, float* logits,
                                   void* split, const int32_t* k_per_token, int k_uniform, int k_max,
                                   int32_t* topk_idx, float* topk_w, cudaStream_t s) {
  const int S = w_dtype == SEMMOE_F32 ? 3 : 1;
  const int EC = experts_per_pass(E, S), n_pass = (E + EC - 1) / EC;
  const void* wb = w;
  int w_rows = E;
  if (S == 3) {
    const long long total = (long long)n_pass * 3 * EC * H;
    long long blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    split_router_kernel<<<(int)blocks, 256, 0, s>>>(static_cast<const float*>(w), E, H, EC, n_pass,
                                                    static_cast<__nv_bfloat16*>(split));
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    wb = split;
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
  const TopkOut tk{k_per_token, k_uniform, k_max, topk_idx, topk_w};
  const bool topk = topk_idx != nullptr;
  dim3 grid((T + BM - 1) / BM, n_pass);
  cudaError_t e;
#define SEMMOE_ROUTE_TC_LAUNCH(S_, K_)                                                   \
  do {                                                                                   \
    static std::atomic<unsigned long long> smem_set{0};                                  \
    e = ensure_smem_limit(route_tc_kernel<S_, K_>, (int)kSmemBytes, smem_set);           \
    if (e != cudaSuccess) return e;                                                      \
    route_tc_kernel<S_, K_><<<grid, THREADS, kSmemBytes, s>>>(mx, mw, T, H, E, EC, logits, tk); \
  } while (0)
  if (S == 3 && topk) SEMMOE_ROUTE_TC_LAUNCH(3, true);
  else if (S == 3) SEMMOE_ROUTE_TC_LAUNCH(3, false);
  else if (topk) SEMMOE_ROUTE_TC_LAUNCH(1, true);
  else SEMMOE_ROUTE_TC_LAUNCH(1, false);
#undef SEMMOE_ROUTE_TC_LAUNCH
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace semmoe
