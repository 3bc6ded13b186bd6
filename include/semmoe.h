/*
 * semmoe.h -- C ABI of the affinity-aware MoE layer forward on one GPU.
 *
 * The layer follows two systems described in
 *   [SP]  "Semantic Parallelism: Redefining Efficient MoE Inference via
 *          Model-Data Co-Scheduling" (Sem-MoE; summaries in Korean (ko),
 *          German (de) and Japanese (ja)), and
 *   [MP]  "MoE-Prism: Disentangling Monolithic Experts for Elastic MoE
 *          Services via Model-System Co-Designs" (Korean summary).
 * One forward is six steps, each one call below, all asynchronous on one
 * CUDA stream:
 *   semmoe_route            router GEMM, fp32 softmax, per-token top-k
 *   semmoe_route_hier       the same over sub-experts, by hierarchical gating
 *   semmoe_affinity_lookup  token id -> predicted logical rank
 *   semmoe_remote_count     activations per (source rank, destination rank)
 *   semmoe_permute          stable sort of (token, expert) pairs by
 *                           (destination rank, expert) + row gather
 *   semmoe_grouped_ffn      per-expert SwiGLU FFN over the sorted rows
 *   semmoe_grouped_ffn_gather  the same, reading x through the permutation
 *   semmoe_shared_ffn       dense SwiGLU of the shared experts (optional)
 *   semmoe_combine          un-permute and gate-weighted sum
 * and, around the layer:
 *   semmoe_dp_schedule      requests placed on data-parallel ranks by affinity
 *   semmoe_transition_lookup next layer's rank predicted from this layer's experts
 *
 * Conventions (every call):
 *  - Pointers marked [device] are CUDA device pointers owned by the caller;
 *    the library never allocates, frees or retains them.  Pointers marked
 *    [host] are ordinary host memory.
 *  - Arrays are dense and row-major; the last dimension is contiguous.
 *    Activation/weight pointers must be 16-byte aligned; workspaces 256-byte.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls only
 *    enqueue work; none synchronises the host except semmoe_check_errors.
 *  - dtype: SEMMOE_F32 (fp32 activations and expert weights) or SEMMOE_BF16
 *    (bf16 storage, fp32 accumulation).
 *  - Return value: SEMMOE_OK or an error code.  Arguments are validated on
 *    the host before anything is enqueued; on error nothing is enqueued and
 *    semmoe_last_error() (thread-local) describes the problem.
 *  - Data errors that only the device can see (an expert index >= E, a token
 *    id >= V, a table value >= R, k_t outside [1, k_max], more pairs than P,
 *    a non-finite logit) never fault: the offending element is skipped or
 *    clamped, a bit is set in a device error word, and the next
 *    semmoe_check_errors() reports SEMMOE_ERR_DEVICE_CHECK.
 *
 * Notation: T tokens, H hidden, E experts, I expert intermediate, R logical
 * ranks, k_t the per-token budget (k of the token's request), k_max its
 * maximum, pair id p = t*k_max + j for slot j < k_t, P = sum_t k_t.
 */
#ifndef SEMMOE_H
#define SEMMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  SEMMOE_OK = 0,
  SEMMOE_ERR_INVALID_ARG = 1,    /* bad pointer, size, alignment or workspace */
  SEMMOE_ERR_UNSUPPORTED = 2,    /* shape/dtype outside the supported set, or not sm_103 */
  SEMMOE_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed */
  SEMMOE_ERR_DEVICE_CHECK = 4,   /* a kernel saw invalid data (see the device error word) */
  SEMMOE_ERR_DEVICE_TIMEOUT = 5  /* a bounded wait inside a kernel ran out */
};

enum { SEMMOE_F32 = 0, SEMMOE_BF16 = 1 };
/* Router-weight type only: an fp32 router weight already split into three
 * bf16 parts by semmoe_route_split_weight() (bf16 activations, H % 8 == 0). */
enum { SEMMOE_F32_SPLIT = 2 };

/* Tokens per chunk of the pair count table (semmoe_pair_counts_size). */
enum { SEMMOE_PAIR_COUNT_CHUNK = 128 };

/* Device error word bits reported through semmoe_check_errors(). */
enum {
  SEMMOE_DEVERR_EXPERT = 1,      /* expert index outside [0, E) */
  SEMMOE_DEVERR_TOKEN_ID = 2,    /* token id outside [0, V) */
  SEMMOE_DEVERR_LUT = 4,         /* table value outside [0, R) */
  SEMMOE_DEVERR_K = 8,           /* k_t outside [1, k_max] */
  SEMMOE_DEVERR_PAIRS = 16,      /* more live pairs than the P passed in, or a bad pair index */
  SEMMOE_DEVERR_TIMEOUT = 32,    /* a bounded in-kernel wait gave up */
  SEMMOE_DEVERR_NONFINITE = 64,  /* a non-finite router logit or transition score */
  SEMMOE_DEVERR_OFFSETS = 128,   /* request offsets not non-decreasing from 0 to T */
  SEMMOE_DEVERR_RANK = 256       /* a predicted or request rank outside [0, R) */
};

/* Message of the last failing call on this host thread ("" if none). */
const char* semmoe_last_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int semmoe_version(void);

/* Number of kernels this library has launched in this process (all devices,
 * all threads), counted on the host at each launch.  Not a device query. */
unsigned long long semmoe_kernel_launches(void);

/*
 * Synchronise `stream`, then read and clear the device error words of the
 * current device.  Returns SEMMOE_OK, SEMMOE_ERR_DEVICE_CHECK,
 * SEMMOE_ERR_DEVICE_TIMEOUT or SEMMOE_ERR_CUDA.  If `bits` is not NULL
 * [host], the OR of the SEMMOE_DEVERR_* bits seen is stored there.
 */
int semmoe_check_errors(void* stream, int* bits);

/*
 * semmoe_route -- router GEMM, fp32 softmax and per-token top-k.
 *
 * The router ("gate") scores every expert for every token and activates a
 * few ([SP] ko §1; [MP] §1); [MP] §1, §2 B and §5 let each request run with
 * its own routing budget k in one batch, so k is given per token.
 *
 *   logits[t,e] = sum_h x[t,h] * w_router[e,h]                 (fp32 accumulation)
 *   experts are ordered by logit, descending; equal logits keep the lower
 *   index first (-0.0 equals +0.0); slot j < k_t holds the j-th of that order
 *   gates: w[t,j] = exp(l_j - m) / sum_{i<k_t} exp(l_i - m),  m = max selected
 *   (the fp32 softmax renormalised over the selected experts)
 *
 * x          [device] [T,H], x_dtype (SEMMOE_F32 or SEMMOE_BF16), 16-byte aligned
 * w_router   [device] [E,H], w_dtype (SEMMOE_F32 or SEMMOE_BF16), 16-byte aligned
 * logits_in  [device] [T,E] fp32 or NULL.  If set, x and w_router are not
 *            read (may be NULL) and these logits are routed as given.
 * logits_out [device] [T,E] fp32 or NULL: receives the logits used.
 * k_per_token[device] [T] int32 in [1,k_max], or NULL to use k_uniform.
 * k_uniform  budget of every token when k_per_token is NULL (1..k_max).
 * topk_idx   [device] [T,k_max] int32 out: slot j < k_t = expert, else -1.
 * topk_w     [device] [T,k_max] fp32 out: gates, 0 in padding slots.
 * pair_counts[device] NULL, or semmoe_pair_counts_size(T, E) bytes (16-byte
 *            aligned) out: the count table of the picks, for semmoe_permute
 *            (which then skips its own counting pass).  Layout [E][S] int32,
 *            S = semmoe_pair_counts_stride(T): entry [e][c] = live pairs of
 *            expert e among the tokens [128c, 128c + 128); entries c >= the
 *            number of chunks are 0.  Zeroed and filled by this call.
 * ws         [device] workspace of semmoe_route_workspace_size() bytes (may be
 *            NULL when that size is 256, i.e. the CUDA-core path).
 * Limits: 1 <= k_max <= E <= 256; T >= 0 (T = 0 enqueues nothing).
 *
 * bf16 activations (H % 8 == 0) run the GEMM on the tensor cores; an fp32
 * router weight is then split exactly into three bf16 parts (hi + mid + lo)
 * whose products with the bf16 activations are exact, summed in fp32.  fp32
 * activations run a CUDA-core fp32 GEMM fused with the top-k.
 */
size_t semmoe_route_workspace_size(int T, int H, int E, int x_dtype, int w_dtype);
int semmoe_route(const void* x, int x_dtype, const void* w_router, int w_dtype,
                 const float* logits_in, float* logits_out,
                 const int32_t* k_per_token, int k_uniform,
                 int T, int H, int E, int k_max,
                 int32_t* topk_idx, float* topk_w, int32_t* pair_counts,
                 void* ws, size_t ws_bytes, void* stream);

/* Bytes and row stride (entries) of the pair count table of T tokens and E
 * experts: E rows of semmoe_pair_counts_stride(T) int32 entries, one per
 * 128-token chunk, rounded up to a multiple of 4. */
size_t semmoe_pair_counts_size(int T, int E);
int semmoe_pair_counts_stride(int T);

/*
 * semmoe_route_split_weight -- the form of an fp32 router weight that the
 * tensor-core router multiplies: each value split exactly into three bf16
 * parts (hi + mid + lo), stacked per pass of experts.  semmoe_route and
 * semmoe_route_hier do this split on every call for w_dtype = SEMMOE_F32; a
 * caller whose router weight does not change passes the split once made, with
 * w_dtype = SEMMOE_F32_SPLIT, and saves that work.  Same results, bit for bit.
 *
 * w      [device] [E,H] fp32;  split [device] semmoe_route_split_size(H, E)
 *        bytes out (256-byte aligned).  Limits: H % 8 == 0, 1 <= E <= 256.
 */
size_t semmoe_route_split_size(int H, int E);
int semmoe_route_split_weight(const float* w, int H, int E, void* split, void* stream);

/*
 * semmoe_route_hier -- MoE-Prism's training-free hierarchical gating over
 * sub-experts ([MP] §2 A: each of Ep parent experts is split into N
 * sub-experts, disjoint sets of its intermediate neurons; the routing is
 * rebuilt without training from co-activation statistics).
 *
 * The parent router gives l[t,e] = x[t] . Wp[e] (fp32, as semmoe_route).
 * Sub-expert s = e*N + i scores  score[t,s] = l[t,e] + sub_logw[s]  (fp32 add;
 * sub_logw = log of the sub-expert's profiled co-activation weight, so the
 * order is that of p_e * a[e,i]).  The k_t best scores are taken, ties to the
 * lower s, slot j holding the j-th; the gate of a taken sub-expert of parent e
 * is p_e renormalised over the distinct parents taken:
 *   w = exp(l_e - m) / sum_{e' in parents taken} exp(l_e' - m),  m = their max logit.
 * A parent's sub-experts all carry its gate (their outputs add up to the
 * parent's output), so taking every sub-expert of the top-m parents gives
 * back the parent router's renormalised top-m.
 *
 * x, x_dtype, w_parent [Ep,H], w_dtype, logits_in / logits_out [T,Ep],
 * k_per_token / k_uniform, T, H: as semmoe_route with E = Ep.
 * sub_logw  [device] [Ep*N] fp32, finite
 * topk_idx  [device] [T,k_max] int32 out: sub-expert ids (-1 = padding)
 * topk_w    [device] [T,k_max] fp32 out (0 = padding)
 * pair_counts [device] NULL or the count table of the picks, as semmoe_route
 *           with E = Ep*N sub-experts
 * ws        [device] workspace of semmoe_route_hier_workspace_size() bytes
 * Limits: 1 <= N, 1 <= Ep*N <= 256, 1 <= k_max <= Ep*N.
 */
size_t semmoe_route_hier_workspace_size(int T, int H, int Ep, int x_dtype, int w_dtype);
int semmoe_route_hier(const void* x, int x_dtype, const void* w_parent, int w_dtype, const float* logits_in,
                      float* logits_out, const float* sub_logw, int N, const int32_t* k_per_token, int k_uniform,
                      int T, int H, int Ep, int k_max, int32_t* topk_idx, float* topk_w,
                      int32_t* pair_counts, void* ws, size_t ws_bytes, void* stream);

/*
 * semmoe_affinity_lookup -- predicted logical rank of each token from its id.
 *
 * [SP] ja §2.3: a lightweight table, built offline from the token-expert
 * affinity ([SP] de §2 A), maps a token to its expert group and device:
 *   pred_rank[t] = lut[token_ids[t]].
 *
 * token_ids [device] [T] int32 in [0,V);  lut [device] [V] int32 in [0,R)
 * pred_rank [device] [T] int32 out (an out-of-range id or value gives 0 and
 *           sets a device error bit).
 */
int semmoe_affinity_lookup(const int32_t* token_ids, const int32_t* lut, int V, int R,
                           int T, int32_t* pred_rank, void* stream);

/*
 * semmoe_remote_count -- activations by (predicted source rank, destination
 * rank); the remote ones per source rank.
 *
 * A pair (t, j) is a local activation when its expert is hosted on the
 * token's own rank, remote otherwise; [SP] ko §3-§4 and de §4 measure the
 * local activation rate.  counts[src][dst] += 1 for every live pair with
 * src = pred_rank[t], dst = expert_rank[topk_idx[t,j]];
 * remote[src] = sum_{dst != src} counts[src][dst];  LAR = trace(counts) / P.
 * counts is also the send-count table of an expert-parallel all-to-all.
 *
 * topk_idx    [device] [T,k_max] int32 (-1 = padding slot, skipped)
 * pred_rank   [device] [T] int32;  expert_rank [device] [E] int32 in [0,R)
 * counts      [device] [R,R] int32 out (overwritten);  remote [device] [R] int32 out
 * Limits: 1 <= R <= 64, 1 <= E <= 256.
 */
int semmoe_remote_count(const int32_t* topk_idx, const int32_t* pred_rank,
                        const int32_t* expert_rank, int T, int k_max, int E, int R,
                        int32_t* counts, int32_t* remote, void* stream);

/*
 * semmoe_permute -- the single-device form of the Shuffled-Reduce-Scatter
 * token shuffle: tokens go to the rank hosting their target experts
 * ([SP] ko §2.2, de §2 B, ja §2.2 B).  Experts are laid out rank-major, the
 * physical order that [SP] ja §2.2 A obtains by shuffling gate columns:
 * phys(e) = position of e when experts are sorted by (expert_rank[e], e).
 * Pairs are sorted stably by phys(topk_idx[p]) (ties keep increasing p), and
 * each sorted row receives its token's activation row.
 *
 * topk_idx       [device] [T,k_max] int32 (-1 = padding slot)
 * expert_rank    [device] [E] int32 in [0,R)
 * x              [device] [T,H] dtype, or NULL to skip the row gather
 * P              number of live pairs (sum_t k_t), known to the caller
 * expert_offsets [device] [E+1] int32 out: row range of physical bucket b
 * rank_offsets   [device] [R+1] int32 out: row range of rank r
 * phys_to_expert [device] [E]   int32 out: expert in physical bucket b
 * expert_counts  [device] [E]   int32 out: pairs per expert (logical order)
 * sorted_to_pair [device] [P]   int32 out: pair id of sorted row q
 * pair_to_sorted [device] [T*k_max] int32 out: sorted row of pair p, -1 for padding
 * x_perm         [device] [P,H] dtype out (x_perm[q] = x[sorted_to_pair[q] / k_max]),
 *                or NULL when x is NULL
 * pair_counts    [device] NULL, or the count table that semmoe_route /
 *                semmoe_route_hier wrote for these same topk_idx: the permute
 *                then starts from it instead of counting the pairs itself (one
 *                kernel instead of two).  A table that does not match topk_idx
 *                gives wrong maps (rows past P are dropped and flagged
 *                SEMMOE_DEVERR_PAIRS, never written out of bounds).  Used while
 *                T <= 131072 (1024 chunks); larger batches count for themselves.
 * ws, ws_bytes   [device] workspace of at least semmoe_permute_workspace_size()
 * Limits: 1 <= E <= 256, 1 <= R <= E, 1 <= k_max <= E.
 *
 * Kernels: each CTA takes a run of tokens, derives its first row in every
 * bucket from the count table, ranks its own pairs stably, writes both maps
 * and copies its tokens' rows (copies of 256 MB and more run as a second
 * kernel) -- no CTA waiting on another.
 */
size_t semmoe_permute_workspace_size(int T, int k_max, int E);
int semmoe_permute(const int32_t* topk_idx, const int32_t* expert_rank,
                   const void* x, int dtype, int T, int H, int E, int R, int k_max, int P,
                   int32_t* expert_offsets, int32_t* rank_offsets, int32_t* phys_to_expert,
                   int32_t* expert_counts, int32_t* sorted_to_pair, int32_t* pair_to_sorted,
                   void* x_perm, const int32_t* pair_counts, void* ws, size_t ws_bytes, void* stream);

/*
 * semmoe_permute_noalloc -- semmoe_permute for callers that cannot allocate
 * device memory.  The pages have no counterpart of this call: it exists for
 * callers that own no allocator, such as a plugin inside a host engine that
 * manages every byte of device memory itself and gives the plugin no
 * allocation hook, or a latency-critical serving loop that forbids cudaMalloc
 * after start-up because it can synchronise the whole device.
 *
 * Same arguments, outputs and errors as semmoe_permute, minus the workspace
 * and the count table (it always counts for itself): the scratch (that count
 * table: at most 96 chunks * E * 4 bytes) lives
 * in a static 96 KiB device array compiled into the library, which every GPU
 * that loads the library holds until the process exits.  That covers every
 * E <= 256; sizes beyond it (E > 256, T*k_max >= 2^31) are rejected with
 * SEMMOE_ERR_INVALID_ARG before anything runs.  The call makes no cudaMalloc,
 * cudaFree or other allocating call.
 *
 * The first call in each CUDA context (normally: on each device) looks up the
 * array's device address with that context current and caches it under the
 * context's unique ID, so a context made after cudaDeviceReset looks it up
 * afresh; make that first call before any stream capture.  All calls share the one array and it keeps the last call's
 * contents (the kernels overwrite whatever they read), so two calls that
 * overlap on the GPU -- on different streams, or from different threads --
 * race on it; order them on one stream.
 */
int semmoe_permute_noalloc(const int32_t* topk_idx, const int32_t* expert_rank,
                           const void* x, int dtype, int T, int H, int E, int R, int k_max, int P,
                           int32_t* expert_offsets, int32_t* rank_offsets, int32_t* phys_to_expert,
                           int32_t* expert_counts, int32_t* sorted_to_pair, int32_t* pair_to_sorted,
                           void* x_perm, void* stream);

/*
 * semmoe_grouped_ffn -- SwiGLU expert FFN over the sorted rows.
 *
 * The activated experts' computation ([SP] ko §1; [MP] §2 A: an expert is a
 * set of intermediate neurons).  Rows [expert_offsets[b], expert_offsets[b+1])
 * belong to expert e = phys_to_expert[b]:
 *   h = silu(x W1_e^T) * (x W3_e^T),  silu(z) = z / (1 + exp(-z)),  h stored in dtype
 *   y = h W2_e^T, stored in dtype
 *
 * x_perm  [device] [P,H] dtype
 * w13     [device] [E,2I,H] dtype: rows 0..I-1 = W1_e (gate), I..2I-1 = W3_e (up)
 * w2      [device] [E,H,I] dtype
 * y_perm  [device] [P,H] dtype out
 * ws      [device] workspace of at least semmoe_grouped_ffn_workspace_size()
 * Limits: H % 8 == 0 and I % 8 == 0 (16-byte rows for bf16 tensor-core tiles).
 * Device checks: offsets that decrease or leave [0, P] set
 * SEMMOE_DEVERR_PAIRS, an expert id outside [0, E) SEMMOE_DEVERR_EXPERT; such
 * a group is skipped (its rows of y_perm keep what they held).  P == 0 needs
 * no activation buffers.
 */
size_t semmoe_grouped_ffn_workspace_size(int P, int I, int dtype);
int semmoe_grouped_ffn(const void* x_perm, const int32_t* expert_offsets,
                       const int32_t* phys_to_expert, const void* w13, const void* w2,
                       int dtype, int P, int E, int H, int I,
                       void* y_perm, void* ws, size_t ws_bytes, void* stream);

/*
 * semmoe_grouped_ffn_gather -- semmoe_grouped_ffn reading the expert inputs
 * straight from the unpermuted activations: sorted row q of GEMM1 is
 * x[sorted_to_pair[q] / k_max] (the row semmoe_permute would have gathered into
 * x_perm[q]), fetched into GEMM1's staged tiles by gathering warps (TMA row
 * gathers in the 2-SM form), so the permute can run on index tables only
 * (x = x_perm = NULL) and no x_perm is written or read back.  Each row is
 * fetched once per 128 columns of h, so this pays off for narrow experts only
 * (measured faster for I = 352, slower for I = 768 and 1408).  The
 * on-device shuffle fused into the expert GEMM ([SP] ko §2.2, de §2 B).
 * Results are bit-identical to semmoe_permute + semmoe_grouped_ffn.
 *
 * x              [device] [T,H] dtype (16-byte aligned)
 * sorted_to_pair [device] [P] int32, from semmoe_permute (a bad pair id reads
 *                row 0 and sets SEMMOE_DEVERR_PAIRS)
 * other arguments, workspace and limits as semmoe_grouped_ffn.
 */
int semmoe_grouped_ffn_gather(const void* x, const int32_t* sorted_to_pair, int k_max, int T,
                              const int32_t* expert_offsets, const int32_t* phys_to_expert, const void* w13,
                              const void* w2, int dtype, int P, int E, int H, int I, void* y_perm, void* ws,
                              size_t ws_bytes, void* stream);

/*
 * semmoe_grouped_ffn_form -- semmoe_grouped_ffn (sorted_to_pair == NULL) or
 * semmoe_grouped_ffn_gather (sorted_to_pair set) with the kernel form of each
 * GEMM pinned by the caller instead of chosen from the shapes.  The pages have
 * no counterpart: it exists so that tests can run every form of the same
 * computation and check that they agree bit for bit.  The two production
 * calls above are this call with SEMMOE_FORM_DEFAULT for both GEMMs.
 *
 * form1 (GEMM1 + SwiGLU) and form2 (GEMM2), one of
 *   SEMMOE_FORM_DEFAULT            chosen from P, E, I and dtype (what the
 *                                  production calls run)
 *   SEMMOE_FORM_SINGLE             one CTA per SM, M128 x N256 tiles (GEMM1
 *                                  with gathered rows: gathering warps)
 *   SEMMOE_FORM_PAIR1              2-SM pairs (tcgen05 cta_group::2, M256 x
 *                                  N256), one accumulator buffer
 *   SEMMOE_FORM_PAIR               2-SM pairs, two accumulator buffers
 *   SEMMOE_FORM_SINGLE_TMA_GATHER  GEMM1 with gathered rows only: one CTA per
 *                                  SM, rows fetched by TMA four-row gathers
 *   SEMMOE_FORM_CUDA_CORE          both GEMMs on CUDA cores (form1 and form2
 *                                  both this value)
 *   SEMMOE_FORM_FUSED              both GEMMs in one persistent launch of
 *                                  independent CTAs, GEMM2's tiles of an m-tile
 *                                  starting once GEMM1's tiles of it are stored
 *                                  (form1 and form2 both this value; rows read
 *                                  from x_perm, not gathered)
 * bf16 accepts all of them; fp32 only SEMMOE_FORM_DEFAULT or
 * SEMMOE_FORM_CUDA_CORE (it always runs on CUDA cores).  Any other combination
 * returns SEMMOE_ERR_INVALID_ARG.  Arguments, workspace, limits and device
 * checks as semmoe_grouped_ffn / semmoe_grouped_ffn_gather (x is x_perm when
 * sorted_to_pair is NULL; k_max and T are then ignored).
 */
enum {
  SEMMOE_FORM_DEFAULT = 0,
  SEMMOE_FORM_SINGLE = 1,
  SEMMOE_FORM_PAIR1 = 2,
  SEMMOE_FORM_PAIR = 3,
  SEMMOE_FORM_SINGLE_TMA_GATHER = 4,
  SEMMOE_FORM_CUDA_CORE = 5,
  SEMMOE_FORM_FUSED = 6
};
int semmoe_grouped_ffn_form(const void* x, const int32_t* sorted_to_pair, int k_max, int T,
                            const int32_t* expert_offsets, const int32_t* phys_to_expert, const void* w13,
                            const void* w2, int dtype, int P, int E, int H, int I, void* y_perm, void* ws,
                            size_t ws_bytes, int form1, int form2, void* stream);

/*
 * semmoe_grouped_ffn_combine -- semmoe_grouped_ffn with the combine folded
 * into GEMM2: the on-device Shuffled-Allgather ([SP] de §2 B, ja §2.2 B)
 * returning each expert row to its token's position as GEMM2 produces it, so
 * no y_perm is written or read back.  The expert rows add into their token's
 * row the way MoE-Prism's sub-expert outputs add into their parent's ([MP]
 * §2 A).  semmoe_combine_finish then adds the shared experts and rounds:
 *
 *   acc[t] = sum_{j<k_t} topk_w[t,j] * y_j   (fp32; y_j = GEMM2 row of pair t*k_max+j)
 *   out[t] = y_shared[t] + acc[t]            (semmoe_combine_finish, rounded to bf16)
 *
 * This call zeroes acc, runs GEMM1 and then GEMM2, whose epilogue multiplies
 * each fp32 row by its gate and adds it into acc (float4 atomic adds).
 * Differences from semmoe_grouped_ffn + semmoe_combine: y is not rounded to
 * bf16 before the weighted sum, and the sum's order depends on scheduling, so
 * results are not bit-reproducible from run to run (they stay within the bf16
 * tolerance of the layer's definition).
 *
 * x              [device] x_perm [P,H] (x_rows_are_tokens = 0), or the token rows
 *                x [T,H] gathered through sorted_to_pair (x_rows_are_tokens = 1,
 *                as semmoe_grouped_ffn_gather)
 * sorted_to_pair [device] [P] int32 (from semmoe_permute); a pair naming no
 *                token sets SEMMOE_DEVERR_PAIRS and its row is dropped
 * topk_w         [device] [T,k_max] fp32 gates, indexed by pair id
 * acc            [device] [T,H] fp32 out (16-byte aligned)
 * ws             [device] workspace of semmoe_grouped_ffn_workspace_size(P, I, dtype)
 * dtype must be SEMMOE_BF16 (tensor cores), else SEMMOE_ERR_UNSUPPORTED.
 * Other arguments, limits and device checks as semmoe_grouped_ffn.
 */
int semmoe_grouped_ffn_combine(const void* x, int x_rows_are_tokens, const int32_t* sorted_to_pair, int k_max,
                               int T, const int32_t* expert_offsets, const int32_t* phys_to_expert,
                               const void* w13, const void* w2, const float* topk_w, int dtype, int P, int E,
                               int H, int I, float* acc, void* ws, size_t ws_bytes, void* stream);

/*
 * semmoe_combine_finish -- out = y_shared + acc, rounded to dtype (bf16 only):
 * the last step after semmoe_grouped_ffn_combine.
 * acc [device] [T,H] fp32; y_shared [device] [T,H] or NULL; out [device] [T,H].
 * H % 8 == 0; pointers 16-byte aligned.
 */
int semmoe_combine_finish(const float* acc, const void* y_shared, int dtype, int T, int H, void* out, void* stream);

/*
 * semmoe_shared_ffn -- the shared experts (applied to every token with gate 1,
 * their weights concatenated along the intermediate dimension I_s):
 *   y_shared = (silu(x Ws1^T) * (x Ws3^T)) Ws2^T.
 * x [device] [T,H]; ws13 [device] [2*I_s,H]; ws2 [device] [H,I_s];
 * y_shared [device] [T,H] out; ws workspace of semmoe_shared_ffn_workspace_size().
 */
size_t semmoe_shared_ffn_workspace_size(int T, int I_s, int dtype);
int semmoe_shared_ffn(const void* x, const void* ws13, const void* ws2, int dtype,
                      int T, int H, int I_s, void* y_shared, void* ws, size_t ws_bytes,
                      void* stream);

/*
 * semmoe_combine -- the single-device form of the Shuffled-Allgather: expert
 * results return to the original token order ([SP] de §2 B, ja §2.2 B) and
 * are mixed by the gates:
 *   out[t] = y_shared[t] + sum_{j<k_t} topk_w[t,j] * y_perm[pair_to_sorted[t*k_max+j]]
 * summed in that order in fp32, stored in dtype.
 *
 * y_perm [device] [P,H]; pair_to_sorted [device] [T*k_max] (-1 = padding, skipped);
 * topk_w [device] [T,k_max] fp32; y_shared [device] [T,H] or NULL;
 * out [device] [T,H] dtype out.
 */
int semmoe_combine(const void* y_perm, const int32_t* pair_to_sorted, const float* topk_w,
                   const void* y_shared, int dtype, int T, int H, int k_max, int P,
                   void* out, void* stream);

/*
 * semmoe_dp_schedule -- online inter-request scheduling of Attention-DP: a
 * request is batched onto the data-parallel rank its tokens have the most
 * affinity with ([SP] ko §2.2 item 2, de §2 B, ja §2.2 B.1).
 *
 * Request r owns tokens [req_offsets[r], req_offsets[r+1]).  Its affinity to
 * rank q is hist[r][q] = #{t in r : pred_rank[t] = q}; req_rank[r] = the q
 * with the largest count, the lowest q among equal counts (an empty request
 * goes to rank 0).  Requests are then ordered stably by req_rank, and rank q's
 * batch is its requests' tokens laid end to end in that order.
 *
 * pred_rank        [device] [T] int32 in [0,R) (e.g. from semmoe_affinity_lookup)
 * req_offsets      [device] [n_req+1] int32, non-decreasing, 0 .. T
 * hist             [device] [n_req,R] int32 out
 * req_rank         [device] [n_req] int32 out
 * req_order        [device] [n_req] int32 out: request ids in scheduled order
 * rank_req_offsets [device] [R+1] int32 out: req_order range of rank q
 * req_tok_start    [device] [n_req] int32 out: first slot of request r in tok_order
 * tok_order        [device] [T] int32 out: token ids in scheduled order
 * tok_rank         [device] [T] int32 out: req_rank of the token's request (the
 *                  source rank to pass to semmoe_remote_count)
 * rank_tok_offsets [device] [R+1] int32 out: tok_order range of rank q
 * Limits: 1 <= R <= 64; n_req >= 1 unless T == 0.  Offsets that are not
 * non-decreasing from 0 to T set SEMMOE_DEVERR_OFFSETS (the ranges are clamped
 * into [0,T] and writes past T are dropped); a pred_rank outside [0,R) counts
 * as rank 0 and sets SEMMOE_DEVERR_RANK.
 */
int semmoe_dp_schedule(const int32_t* pred_rank, const int32_t* req_offsets, int T, int n_req, int R,
                       int32_t* hist, int32_t* req_rank, int32_t* req_order, int32_t* rank_req_offsets,
                       int32_t* req_tok_start, int32_t* tok_order, int32_t* tok_rank,
                       int32_t* rank_tok_offsets, void* stream);

/*
 * semmoe_transition_lookup -- the rank a token is expected to need in the next
 * layer, from the experts it chose in this one: the Markovian inter-layer
 * dependency of [SP] ko §2.1 / de §2 A, held as a table from experts to devices
 * ([SP] ja §2.3).
 *   score[t][q] = sum_{j < k_t, topk_idx[t,j] >= 0} trans[topk_idx[t,j]][q],
 * added in slot order in fp32; pred_next[t] = argmax_q score, lowest q on ties.
 *
 * topk_idx    [device] [T,k_max] int32 (-1 = padding slot, skipped)
 * k_per_token [device] [T] int32 or NULL to use k_uniform for every token
 * trans       [device] [E,R] fp32 transition weights (finite)
 * pred_next   [device] [T] int32 out
 * Limits: 1 <= R <= 64, E >= 1, 1 <= k_max.  Bad experts set
 * SEMMOE_DEVERR_EXPERT (slot skipped), k_t outside [1,k_max] SEMMOE_DEVERR_K
 * (clamped), a non-finite score SEMMOE_DEVERR_NONFINITE.
 */
int semmoe_transition_lookup(const int32_t* topk_idx, const int32_t* k_per_token, int k_uniform,
                             const float* trans, int T, int k_max, int E, int R, int32_t* pred_next,
                             void* stream);

/*
 * semmoe_selftest_bounded_wait -- exercises the failure path of the kernels'
 * waits (not part of the layer; the pages have no counterpart).  It launches
 * one CTA whose mbarrier wait can never complete; like every wait in the
 * tensor-core kernels, it gives up after its 2 s bound and sets
 * SEMMOE_DEVERR_TIMEOUT, so the next semmoe_check_errors() on the stream
 * returns SEMMOE_ERR_DEVICE_TIMEOUT and the CUDA context stays usable.
 */
int semmoe_selftest_bounded_wait(void* stream);

/*
 * semmoe_selftest_fused_ready_wait -- exercises the failure path of the
 * one-launch grouped FFN (SEMMOE_FORM_FUSED), whose GEMM2 tiles wait on
 * counters that GEMM1's epilogue raises (not part of the layer; the pages have
 * no counterpart).  It runs one group of P bf16 rows (0 < P <= 4096; x_perm
 * [P, H], w13 [1, 2I, H], w2 [1, H, I], y_perm [P, H], workspace as
 * semmoe_grouped_ffn_workspace_size(P, I, SEMMOE_BF16)) with every GEMM2 tile
 * waiting for one count more than its GEMM1 tiles publish.  Each such wait gives
 * up after its 2 s bound, sets SEMMOE_DEVERR_TIMEOUT and stops its CTA (in-flight
 * copies drained, tensor memory freed), so the next semmoe_check_errors() on
 * the stream returns SEMMOE_ERR_DEVICE_TIMEOUT and the CUDA context stays
 * usable; y_perm is left unspecified.  Argument errors as semmoe_grouped_ffn.
 */
int semmoe_selftest_fused_ready_wait(const void* x_perm, const void* w13, const void* w2, int P, int H, int I,
                                     void* y_perm, void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SEMMOE_H */
