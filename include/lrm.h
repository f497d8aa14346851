/*
 * lrm.h - C ABI of the GB300 (sm_103a) library for LRMoE's demand-side
 * backward recalibration of one MoE layer's FC2 (down) projection.
 *
 * Source: "LRMoE: Demand-Side Load Re-Calibration for Efficient MoE Training
 * on Memory-Constrained Nodes" (Hu et al.), sec. 3.1-3.4, Alg. 1, Fig. 4,
 * appendix 7.1-7.2; routing statistics from "Expert Parallel Math Deep"
 * (sections on routing as an expectation over a batch, the load-balancing
 * auxiliary loss, and capacity / drop rate).
 *
 * The path, in call order on one stream, with no host synchronisation:
 *   lrm_route_stats -> lrm_score -> lrm_select -> lrm_compact
 *                   -> lrm_grouped_dgrad -> lrm_grouped_wgrad
 *
 * Notation: T tokens, E experts, k experts per token, h model width (rows of
 * W_e, length of g_t), I expert intermediate width (columns of W_e, length of
 * phi_u).  A routed pair u = (t, e) has index u = t*k + j, where j is its
 * routing slot.  N = T*k.
 *
 * Conventions shared by every call:
 *  - Every tensor argument is a device pointer to caller-owned, row-major,
 *    contiguous memory, unless a parameter says "host".  The library never
 *    allocates, frees or reads device data on the host in these calls; the
 *    context owns only a small device status word.
 *  - bf16 tensors are passed as uint16_t bit patterns (IEEE bfloat16).
 *  - Base pointers of bf16 tensors must be 16-byte aligned, h and I must be
 *    multiples of 8; otherwise LRM_ERR_ALIGN.  Index and fp32 tensors must be
 *    4-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *    call is asynchronous: a returned LRM_OK means the work was enqueued.
 *  - Argument errors (null pointers, bad sizes, alignment) return
 *    synchronously and enqueue nothing.  Data errors found on the device
 *    (an expert id outside [0,E) or repeated within a token, a quota outside
 *    [0, n_e], a ragged total above max_rows, a device wait that ran out of
 *    time) set a bit (1u << code) in the context's device status word; the
 *    kernel skips the offending writes and exits normally.  Read and clear
 *    that word with lrm_get_device_status.  No call traps or hangs the GPU.
 *  - Ragged totals (sum of quotas, per-expert row counts) stay on the device;
 *    the caller passes max_rows, an upper bound used to size buffers.
 *  - Because no call but lrm_get_device_status synchronises with the host, a
 *    sequence of calls can be captured into a CUDA graph.  The first call of
 *    each kind on a device also sets up its kernels (function attributes,
 *    occupancy queries) on the host; make one call of each kind before
 *    capturing, so that the capture holds the launches only.
 */
#ifndef LRM_H
#define LRM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LRM_ABI_VERSION 1

/* Entry points keep default symbol visibility when the library is built
 * with -fvisibility=hidden. */
#if defined(__GNUC__)
#define LRM_API __attribute__((visibility("default")))
#else
#define LRM_API
#endif

typedef enum lrm_status {
  LRM_OK = 0,
  LRM_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, bad rational */
  LRM_ERR_SHAPE = 2,       /* sizes beyond the supported limits; on the device: ragged total > max_rows */
  LRM_ERR_ALIGN = 3,       /* misaligned pointer, h or I not a multiple of 8 */
  LRM_ERR_WORKSPACE = 4,   /* workspace missing or smaller than lrm_workspace_size */
  LRM_ERR_INDEX = 5,       /* device: expert id outside [0,E) or repeated within a token */
  LRM_ERR_QUOTA = 6,       /* device: quota Q_e < 0 or Q_e > n_e (clamped into range) */
  LRM_ERR_TIMEOUT = 7,     /* device: a bounded wait gave up */
  LRM_ERR_ARCH = 8,        /* the device is not sm_103 / the library was not built for it */
  LRM_ERR_CUDA = 9         /* a CUDA runtime or driver call failed */
} lrm_status;

/* Operations that take a workspace, for lrm_workspace_size. */
typedef enum lrm_op {
  LRM_OP_ROUTE_STATS = 0,
  LRM_OP_SELECT = 1,
  LRM_OP_ZERO_DROPPED = 2,
  LRM_OP_COMBINE = 3
} lrm_op;

/* Layer sizes.  Limits: 1 <= E <= 1024, 1 <= k <= 32, k <= E, N = T*k < 2^31,
 * h and I multiples of 8 in [8, 65536]. */
typedef struct lrm_dims {
  int32_t T, E, k, h, I;
} lrm_dims;

/* Routing summary written on the device by lrm_route_stats. */
typedef struct lrm_route_summary {
  int32_t N;           /* routed pairs T*k */
  int32_t C;           /* capacity floor(CF * N / E) */
  int32_t slots;       /* E * C, the padded slots of a fixed-shape layout */
  int32_t dropped;     /* sum_e max(0, n_e - C) */
  int32_t retained;    /* sum_e Q_e */
  int32_t max_count;   /* max_e n_e */
  int32_t min_count;   /* min_e n_e */
  int32_t nonempty;    /* experts with n_e > 0 */
  float aux_unscaled;  /* E * sum_e f_e P_e (multiply by the loss coefficient) */
  float drop_rate;     /* dropped / N */
  float util;          /* (N - dropped) / (E * C) */
  float rho_real;      /* retained / N */
  float max_over_mean; /* max_e n_e / (N / E), the straggler factor */
  float sum_P;         /* sum_e P_e (1 up to rounding) */
} lrm_route_summary;

typedef struct lrm_ctx lrm_ctx;

/* Create a context on `device` (the caller's current device is left as it
 * was).  Allocates the 4-byte device status word; fails with LRM_ERR_ARCH if
 * the device is not compute capability 10.3.  *out owns the context. */
LRM_API lrm_status lrm_create(int device, lrm_ctx** out);
/* Destroy a context created by lrm_create (NULL is accepted). */
LRM_API lrm_status lrm_destroy(lrm_ctx* ctx);
/* Static, human-readable name of a status code. */
LRM_API const char* lrm_status_string(lrm_status s);
/* LRM_ABI_VERSION of the built library. */
LRM_API int32_t lrm_abi_version(void);
/* Number of SMs of the context's device (host value). */
LRM_API lrm_status lrm_sm_count(const lrm_ctx* ctx, int32_t* out);

/* Bytes of device workspace `op` needs for `dims` (0 is possible). */
LRM_API lrm_status lrm_workspace_size(const lrm_ctx* ctx, lrm_op op, lrm_dims dims, size_t* bytes);

/*
 * Step 1 - routing statistics and retention quotas.
 * "Expert Parallel Math Deep": P_e = (1/T) sum_t softmax(logits_t)_e over all
 * E experts, f_e = n_e / N, aux = E sum f_e P_e, C = CF N / E,
 * dropped = sum max(0, n_e - C).  LRMoE sec. 3.1 / Alg. 1: routed
 * counts n_e and quotas K_e (here Q_e) with 0 <= Q_e <= n_e; the quota rule is
 * Q_e = ceil(rho * min(n_e, C)); CF = cf_num/cf_den and rho = rho_num/rho_den
 * are exact rationals (C is the floor).
 *   logits     [T, E] fp32      router logits
 *   expert_idx [T, k] int32     routed expert of pair u = t*k + j
 *   counts     [E]    int32 out n_e
 *   offsets    [E+1]  int32 out exclusive prefix sum of counts
 *   bucket     [N]    int32 out pair ids grouped by expert, ascending u within an expert
 *   P, f       [E]    fp32  out importance and load
 *   quota      [E]    int32 out Q_e
 *   summary    [1]    device lrm_route_summary out
 *   ws, ws_bytes      workspace of at least lrm_workspace_size(LRM_OP_ROUTE_STATS)
 * Requires cf_num, cf_den, rho_den > 0, 0 <= rho_num <= rho_den.
 */
LRM_API lrm_status lrm_route_stats(lrm_ctx* ctx, const float* logits, const int32_t* expert_idx, lrm_dims dims,
                           int32_t cf_num, int32_t cf_den, int32_t rho_num, int32_t rho_den,
                           int32_t* counts, int32_t* offsets, int32_t* bucket, float* P, float* f,
                           int32_t* quota, lrm_route_summary* summary, void* ws, size_t ws_bytes,
                           void* stream);

/*
 * Host queries of the capacity and quota rule of lrm_route_stats, computed
 * by the same code the kernels use (no context, no device work, no
 * allocation; callable without a GPU):
 *   lrm_capacity  *C = floor(CF * N / E), N = T*k ("Expert Parallel Math
 *                 Deep", capacity section: capacity is CF times the mean
 *                 load per expert).
 *   lrm_max_rows  *max_rows = an upper bound of sum_e Q_e over every routing
 *                 of the layer, Q_e = ceil(rho * min(n_e, C)) (LRMoE sec. 3.1:
 *                 quotas with 0 <= Q_e <= n_e): the smallest of N,
 *                 E * ceil(rho * C) and floor((rho_num N + E (rho_den - 1)) /
 *                 rho_den).  It sizes sel_ids and the compacted buffers.
 * CF = cf_num / cf_den and rho = rho_num / rho_den as for lrm_route_stats.
 * Errors: LRM_ERR_INVALID_ARG (null output, bad rational), the dims checks
 * of every call, LRM_ERR_SHAPE if E * C does not fit in int32.
 */
LRM_API lrm_status lrm_capacity(lrm_dims dims, int32_t cf_num, int32_t cf_den, int32_t* C);
LRM_API lrm_status lrm_max_rows(lrm_dims dims, int32_t cf_num, int32_t cf_den, int32_t rho_num, int32_t rho_den,
                                int32_t* max_rows);

/*
 * Step 2 - the Load Recalibration Metric (LRMoE sec. 3.2 Prop. 3.1 eq. (3);
 * Alg. 1): score[u] = alpha[u]^2 * ||g_t||^2 * ||phi_u||^2, the
 * squared Frobenius norm of the rank-one gradient contribution
 * (alpha_u g_t) phi_u^T, in fp32.
 *   g     [T, h]    bf16  gradient at the expert output, before alpha
 *   phi   [N, I]    bf16  saved FC2 input of pair u (row u)
 *   alpha [N]       fp32  gate weight of pair u
 *   score [N]       fp32  out
 */
LRM_API lrm_status lrm_score(lrm_ctx* ctx, const uint16_t* g, const uint16_t* phi, const float* alpha,
                     lrm_dims dims, float* score, void* stream);

/*
 * Step 2 with the selection metrics of LRMoE's ablation (sec. 4.7, Table 2),
 * for comparing selection rules on the same pairs:
 *   LRM_METRIC_LRM       the Load Recalibration Metric (same as lrm_score)
 *   LRM_METRIC_GRAD_L2SQ score[u] = ||g_t||^2 (gradient only)
 *   LRM_METRIC_GRAD_L1   score[u] = sum_i |g_t,i| (gradient only; the
 *                        ablation's "|g|" read as an L1 sum)
 *   LRM_METRIC_RANDOM    score[u] = top 24 bits of the (u+1)-th output of the
 *                        SplitMix64 generator (Steele, Lea and Flood, OOPSLA
 *                        2014) started from state `seed`, times 2^-24
 * phi and alpha are read only by LRM_METRIC_LRM, g by every metric but
 * LRM_METRIC_RANDOM (unused pointers may be NULL).  fp32 accumulation as in
 * lrm_score.  An unknown metric returns LRM_ERR_INVALID_ARG.
 */
typedef enum lrm_metric {
  LRM_METRIC_LRM = 0,
  LRM_METRIC_GRAD_L2SQ = 1,
  LRM_METRIC_GRAD_L1 = 2,
  LRM_METRIC_RANDOM = 3
} lrm_metric;
LRM_API lrm_status lrm_score_metric(lrm_ctx* ctx, int32_t metric, const uint16_t* g, const uint16_t* phi,
                            const float* alpha, lrm_dims dims, uint64_t seed, float* score, void* stream);

/*
 * Step 3 - per-expert TopK within the quota (LRMoE sec. 3.2, Alg. 1,
 * appendix 7.2 Prop. 7.1): for every expert e keep the quota[e] pairs of
 * bucket[offsets[e] .. offsets[e+1]) with the largest score; equal scores go
 * to the lower pair index.  Retained ids are written expert-major, ascending
 * u within an expert.
 *   score, offsets, bucket   as produced by lrm_score / lrm_route_stats
 *   quota       [E]   int32  Q_e (from lrm_route_stats or the caller; out-of-range
 *                            values are clamped into [0, n_e] and flagged LRM_ERR_QUOTA)
 *   sel_offsets [E+1] int32 out exclusive prefix sum of the (clamped) quotas
 *   sel_ids     [max_rows] int32 out retained pair ids
 *   max_rows    host int, capacity of sel_ids; a larger total is flagged LRM_ERR_SHAPE
 * Scores must be finite and >= 0 (the metric's range).
 */
LRM_API lrm_status lrm_select(lrm_ctx* ctx, const float* score, const int32_t* offsets, const int32_t* bucket,
                      const int32_t* quota, lrm_dims dims, int32_t max_rows, int32_t* sel_offsets,
                      int32_t* sel_ids, void* ws, size_t ws_bytes, void* stream);

/*
 * Step 4 - physical compaction (LRMoE sec. 3.1, 3.3, 3.4, Fig. 4; weighted
 * cotangent of appendix eq. (5)): for row r < sel_offsets[E], u = sel_ids[r],
 * t = u / k:
 *   delta_c[r] = bf16_rne(fp32(alpha[u] * g[t]))   [max_rows, h] bf16 out
 *   phi_c[r]   = phi[u]                            [max_rows, I] bf16 out
 *   alpha_c[r] = alpha[u]                          [max_rows] fp32 out (may be NULL)
 * Rows at or beyond sel_offsets[E] are left untouched.
 */
LRM_API lrm_status lrm_compact(lrm_ctx* ctx, const uint16_t* g, const uint16_t* phi, const float* alpha,
                       const int32_t* sel_offsets, const int32_t* sel_ids, lrm_dims dims, int32_t max_rows,
                       uint16_t* delta_c, uint16_t* phi_c, float* alpha_c, void* stream);

/*
 * Step 5a - grouped FC2 input gradient, variable M, no padding (LRMoE
 * sec. 3.3: the retained count is the row dimension of the input-gradient
 * product; appendix eq. (6)):  for every expert e and row r of its segment
 * [sel_offsets[e], sel_offsets[e+1]):
 *   dphi_c[r, :] = delta_c[r, :] . W_e          (fp32 accumulation, bf16 out)
 *   delta_c [max_rows, h] bf16, W [E, h, I] bf16, dphi_c [max_rows, I] bf16 out.
 * tcgen05 tensor cores with TMA-fed shared-memory tiles.
 */
LRM_API lrm_status lrm_grouped_dgrad(lrm_ctx* ctx, const uint16_t* delta_c, const uint16_t* W,
                             const int32_t* sel_offsets, lrm_dims dims, int32_t max_rows,
                             uint16_t* dphi_c, void* stream);

/*
 * The inverse mapping (LRMoE sec. 1 and 3.3; Alg. 1, ScatterWithZeros;
 * sec. 3.4: kept rows return to their pairs' slots, dropped pairs' slots are
 * zero-filled for the next dense layer), in two calls:
 *
 * lrm_grouped_dgrad_scatter: step 5a with the rows written through the
 * selection: the input-gradient row of retained pair u = sel_ids[r] goes to
 * row u of dphi_rows [N, I] bf16 (the pair-major layout of phi) instead of row
 * r of the compacted output.  The values are those of lrm_grouped_dgrad bit
 * for bit.  Rows of pairs that were not retained are not written.  A sel_ids
 * entry outside [0, N) sets LRM_ERR_INDEX and its row is skipped.
 *
 * lrm_zero_dropped_rows: writes zeros to every row u of rows [N, I] bf16 whose
 * pair is not among sel_ids[0 .. sel_offsets[E]) (clamped to max_rows).  ws:
 * an N-bit map (lrm_workspace_size with LRM_OP_ZERO_DROPPED), cleared on the
 * stream by the call.  The two calls write disjoint rows, in either order.
 */
LRM_API lrm_status lrm_grouped_dgrad_scatter(lrm_ctx* ctx, const uint16_t* delta_c, const uint16_t* W,
                                     const int32_t* sel_offsets, const int32_t* sel_ids, lrm_dims dims,
                                     int32_t max_rows, uint16_t* dphi_rows, void* stream);
LRM_API lrm_status lrm_zero_dropped_rows(lrm_ctx* ctx, const int32_t* sel_offsets, const int32_t* sel_ids,
                                 lrm_dims dims, int32_t max_rows, uint16_t* rows, void* ws, size_t ws_bytes,
                                 void* stream);

/*
 * FC1 side of the expert backward on the retained pairs (LRMoE sec. 3.4: the
 * compacted row count sizes all four expert-backward GEMMs).
 * The activation is read as SwiGLU: FC1 gives [a | b] (gate, up; width 2I)
 * per pair and phi = silu(a) * b, silu(a) = a / (1 + exp(-a)).  The FC1 GEMMs
 * are lrm_grouped_dgrad / lrm_grouped_wgrad with the dimensions relabelled:
 *   compacted FC1 inputs:   lrm_compact(g = x [T, h], phi = ab [N, 2I], alpha = 1,
 *                           dims with I -> 2I) gives Xc and ABc;
 *   FC1 input gradient:     lrm_grouped_dgrad(delta_c = dh1, W = W1 [E, 2I, h],
 *                           dims with h -> 2I, I -> h) gives dXc [rows, h];
 *   FC1 weight gradient:    lrm_grouped_wgrad(delta_c = dh1, phi_c = Xc,
 *                           dims with h -> 2I, I -> h) gives dW1 [E, 2I, h].
 *
 * lrm_swiglu_backward: dh1[r] = [dphi_c[r] * b * silu'(a) | dphi_c[r] * silu(a)]
 * for the compacted rows r < sel_offsets[E] (clamped to max_rows), [a | b] =
 * ab_c[r]; fp32 math, bf16 (round to nearest even) out.
 *   dphi_c [rows, I] bf16, ab_c [rows, 2I] bf16, dh1 [rows, 2I] bf16
 *
 * lrm_combine_rows: the input gradient of every token: out[t] = bf16(sum of
 * rows[r] over the retained pairs u = sel_ids[r] of token t = u div k), zeros
 * for tokens without a retained pair (the inverse mapping followed by the MoE
 * combine over the token's k experts).  rows [max_rows, width] bf16 (the
 * compacted order), out [T, width] bf16, width a multiple of 8.  ws: N int32
 * (lrm_workspace_size with LRM_OP_COMBINE).
 */
LRM_API lrm_status lrm_swiglu_backward(lrm_ctx* ctx, const uint16_t* dphi_c, const uint16_t* ab_c,
                               const int32_t* sel_offsets, lrm_dims dims, int32_t max_rows, uint16_t* dh1,
                               void* stream);
LRM_API lrm_status lrm_combine_rows(lrm_ctx* ctx, const uint16_t* rows, const int32_t* sel_offsets,
                            const int32_t* sel_ids, lrm_dims dims, int32_t max_rows, int32_t width, uint16_t* out,
                            void* ws, size_t ws_bytes, void* stream);

/*
 * Step 5b - grouped FC2 weight gradient, variable K, no padding (LRMoE
 * sec. 3.3: the retained count is the reduction dimension of the
 * weight-gradient product; eq. (1), (8), (9)):
 *   dW[e] (=|+=) delta_c[seg e]^T . phi_c[seg e]     [E, h, I] fp32 out
 * accumulate = 0 overwrites (experts with no retained row get exact zeros),
 * accumulate = 1 adds into dW.
 */
LRM_API lrm_status lrm_grouped_wgrad(lrm_ctx* ctx, const uint16_t* delta_c, const uint16_t* phi_c,
                             const int32_t* sel_offsets, lrm_dims dims, int32_t max_rows, int32_t accumulate,
                             float* dW, void* stream);

/*
 * Step 5b with a bf16 weight gradient: the same products accumulated in fp32
 * in TMEM, each dW element rounded once to bf16 (nearest even) when it is
 * stored.  The pages train in BF16 (LRMoE sec. 4.1), and TopoEP sec. 3.2
 * counts the gradient of BF16 mixed-precision training as BF16 next to an
 * FP32 master copy, so this is the dtype such a step hands to the optimizer;
 * it halves the dW bytes that bound lrm_grouped_wgrad.  dW [E, h, I] bf16 bits,
 * 16-byte aligned.  accumulate = 1 adds the fp32 products to the stored bf16
 * values and rounds the sum.  Errors as for lrm_grouped_wgrad.
 */
LRM_API lrm_status lrm_grouped_wgrad_bf16(lrm_ctx* ctx, const uint16_t* delta_c, const uint16_t* phi_c,
                                  const int32_t* sel_offsets, lrm_dims dims, int32_t max_rows, int32_t accumulate,
                                  uint16_t* dW, void* stream);

/*
 * Comparator (measurement only) - the zero-masked fixed-shape layout of
 * LRMoE sec. 3.4: expert e owns C slots; its retained rows fill the first
 * Q_e slots and the rest are zero.
 *   delta_pad [E*C, h] bf16 out, phi_pad [E*C, I] bf16 out,
 *   pad_offsets [E+1] int32 out = {0, C, 2C, ...}.
 * Running lrm_grouped_dgrad / lrm_grouped_wgrad with pad_offsets and
 * max_rows = E*C gives the same gradients on capacity-padded tensors.
 * A quota above C is flagged LRM_ERR_SHAPE and its extra rows dropped.
 */
LRM_API lrm_status lrm_compact_padded(lrm_ctx* ctx, const uint16_t* delta_c, const uint16_t* phi_c,
                              const int32_t* sel_offsets, lrm_dims dims, int32_t C, uint16_t* delta_pad,
                              uint16_t* phi_pad, int32_t* pad_offsets, void* stream);

/*
 * lrm_route_stats without a caller-provided workspace: the same three kernels
 * and the same outputs, but the scratch they need lives in a fixed array
 * inside this library (LRM_ROUTE_STATS_SCRATCH_BYTES of device memory, held
 * on every GPU that loads the library until the process exits).
 *
 * It is meant for callers that hold only the tensors they pass in and cannot
 * obtain extra device memory: for example a host framework whose memory pool
 * owns the GPU's memory and forbids outside allocation, or code that must not
 * allocate once it is running.  The call itself allocates nothing: no
 * cudaMalloc, cudaFree or allocating library routine.
 *
 * - The scratch holds two E x B tables of 4-byte entries, one column per
 *   block of floor(1024 / k) tokens (B = ceil(T / floor(1024 / k)), about
 *   8 * E * T * k / 1024 bytes); sizes that do not fit in
 *   LRM_ROUTE_STATS_SCRATCH_BYTES (4 MiB: for example E = 128 with up to
 *   about 4 million routed pairs) return LRM_ERR_SHAPE before any device
 *   work.  Every entry is written before it is read, so nothing in the
 *   scratch has to start at zero and stale contents of an earlier call are
 *   harmless.
 * - Every call looks up the array's device address with the device current
 *   (host-side, no device work), so a call after a reset of the device
 *   (cudaDeviceReset) finds the array the module was loaded with again.
 * - All calls share the one array, so calls that may overlap on the GPU
 *   (different streams without ordering between them) race; serialise them.
 * The paper has no counterpart of this entry point.
 */
#define LRM_ROUTE_STATS_SCRATCH_BYTES (4u << 20)
LRM_API lrm_status lrm_route_stats_noalloc(lrm_ctx* ctx, const float* logits, const int32_t* expert_idx,
                                           lrm_dims dims, int32_t cf_num, int32_t cf_den, int32_t rho_num,
                                           int32_t rho_den, int32_t* counts, int32_t* offsets, int32_t* bucket,
                                           float* P, float* f, int32_t* quota, lrm_route_summary* summary,
                                           void* stream);

/* Synchronise `stream`, return the device status word in *flags (bit
 * (1u << code) for every lrm_status code raised on the device since the last
 * read) and clear it. */
LRM_API lrm_status lrm_get_device_status(lrm_ctx* ctx, void* stream, uint32_t* flags);

/* Time limit, in nanoseconds, of every device-side wait of the grouped GEMM
 * kernels (default 2e9).  A wait that runs out sets LRM_ERR_TIMEOUT and the
 * kernel winds down and returns. */
LRM_API lrm_status lrm_set_wait_budget(lrm_ctx* ctx, uint64_t ns);

/* Failure-detection self test: launch one block that waits, with the same
 * bounded wait the GEMM kernels use, on a barrier nothing will ever complete,
 * for at most budget_ns; it must give up, set LRM_ERR_TIMEOUT and return. */
LRM_API lrm_status lrm_selftest_wait_timeout(lrm_ctx* ctx, uint64_t budget_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LRM_H */
