/*
 * moe.h — C ABI of the GB300 (sm_103a) fused Mixture-of-Experts feed-forward layer.
 *
 * The layer (page "Mixture-of-Experts Kernels: Routing, Permutation, and Grouped GEMM",
 * §1-§2 and §11): a router scores E experts per token and keeps k; an align step turns
 * the chosen ids into a block-aligned indirection table; two grouped GEMMs run every
 * expert's SwiGLU on exactly the rows routed to it; a combine sums the k weighted slots:
 *
 *   x[T,H] --router--> logits[T,E] --top-k--> topk_ids[T,k], topk_w[T,k]
 *   --align--> sorted_ids[max_padded], expert_ids[max_padded/block_m], num_post_padded
 *   --GEMM1 (gather x[sorted_ids/k], W13[e]) + silu(h[:, :I]) * h[:, I:]--> act[max_padded, I]
 *   --GEMM2 (act, W2[e]) * topk_w[r]--> y[T*k, H] at flat row r = t*k + j
 *   --combine--> out[t] = sum_j y[t*k + j]
 *
 * Conventions for every entry point:
 *  - Tensors are DEVICE pointers, contiguous and row-major, in nn.Linear [E, N, K] layout:
 *    x[T,H], Wg[E,H], W13[E,2I,H] (rows 0..I-1 = gate projection W1, rows I..2I-1 = up
 *    projection W3), W2[E,H,I], y[T*k,H], out[T,H]. x's dtype (cfg->dtype) is the dtype of
 *    Wg, act, y and out, and of W13 and W2 unless cfg->weight_format selects FP8 weights.
 *    logits, topk_w, the biases and the weight scales are always fp32; ids int32.
 *  - bf16 tensors must start on a 16-byte boundary and H, I must be multiples of 8
 *    (tensor-memory-access copies move 16-byte units).
 *  - The CALLER owns every buffer, workspaces included. The library never allocates or
 *    frees device memory, never synchronises the stream and never reads device data on
 *    the host: every call only enqueues kernels on `stream`, so a sequence of calls can be
 *    captured in a CUDA graph. (moe_device_status is the one diagnostic exception.)
 *  - Host-side argument checks return MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *    MOE_ERR_WORKSPACE before anything is enqueued; a failed launch returns MOE_ERR_CUDA.
 *  - Faults found on the device (an expert id outside [0, E), a pipeline wait that ran
 *    out of time) never trap: the kernel skips the bad item or returns early and records
 *    a code in a device status word, read with moe_device_status().
 *  - Ties in top-k go to the lower expert (or group) id. Rows inside one expert's run of
 *    sorted_ids are in ascending flat row r. Padding rows and the unused tail of
 *    sorted_ids hold the sentinel T*k; unused tail entries of expert_ids hold -1.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 9

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* a null pointer, a size out of range, misaligned memory */
  MOE_ERR_UNSUPPORTED = 2,  /* valid arguments the library does not handle (e.g. E > 512) */
  MOE_ERR_WORKSPACE = 3,    /* workspace pointer null or smaller than required */
  MOE_ERR_CUDA = 4          /* a CUDA runtime/driver call or a kernel launch failed */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;

typedef enum {
  /* softmax over the E logits (after the optional logit_bias), keep the k largest;
   * renormalize=1 divides the k kept probabilities by their sum, which equals a softmax
   * over the k largest logits (the gpt-oss "softmax over top-k" form). Page §3 route(). */
  MOE_ROUTE_SOFTMAX = 0,
  /* DeepSeek-V3 rule (page §4): s = sigmoid(logit); c = s + select_bias chooses, s weighs;
   * groups of E/n_group consecutive experts scored by the sum of their two largest c; the
   * topk_group best groups stay eligible; top-k of c inside them; w = scale * s / sum(s)
   * (renormalize=1) or scale * s (renormalize=0). */
  MOE_ROUTE_SIGMOID_GROUPED = 1
} moe_route_mode_t;

/* Storage of the expert weights W13 and W2 (page §8: an FP8 expert holds one byte per
 * weight; §9: the FP8 weight variants of the fused kernel; §10: FP8 scale handling).
 * The router weight Wg always has cfg->dtype. */
typedef enum {
  MOE_WEIGHTS_NATIVE = 0, /* W13, W2 in cfg->dtype */
  /* W13, W2 hold FP8 E4M3 (OCP "FN": bias 7, max 448, no infinities) bytes, same shapes;
   * the weight used is code * scale of the code's 128 x 128 block (fp32 scales):
   *   W13: w13_scale[E', 2, ceil(I/128), ceil(H/128)] - grid 0 covers the gate rows
   *        0..I-1, grid 1 the up rows I..2I-1 (row blocks start at row 0 and row I);
   *   W2 : w2_scale[E', ceil(H/128), ceil(I/128)].
   * E' = E + n_shared. Needs dtype MOE_BF16 and H, I multiples of 16. The tensor cores
   * see bf16(code * scale): exact when the scale is a power of two. */
  MOE_WEIGHTS_FP8_E4M3_B128 = 1
} moe_weight_format_t;

typedef struct moe_config {
  int T;                    /* tokens, >= 1 */
  int H;                    /* hidden size (multiple of 8) */
  int I;                    /* expert intermediate size (multiple of 8) */
  int E;                    /* routed experts, 1..512 */
  int k;                    /* experts per token, 1..min(E, 32) */
  moe_dtype_t dtype;        /* MOE_BF16 (tensor-core path) or MOE_F32 (FFMA path) */
  moe_route_mode_t mode;
  int renormalize;          /* 1: weights of the k kept experts sum to 1 (times scale) */
  float scale;              /* routed scaling factor applied to the weights (1.0; 2.5 DSv3) */
  int n_group;              /* mode 1: expert groups (E % n_group == 0, n_group <= 32) */
  int topk_group;           /* mode 1: groups kept (topk_group * E / n_group >= k) */
  const float* logit_bias;  /* mode 0: device fp32 [E] added to the logits, or NULL */
  const float* select_bias; /* mode 1: device fp32 [E] selection-only bias, or NULL */
  /* Expert parallelism (page §10, "Try this"): device int32 [E] or NULL. Expert e's weights
   * sit in slot expert_map[e] of W13/W2 (0 <= slot < E); -1 marks an expert held by another
   * device: its tiles are skipped and its slots add nothing to out. Routing stays global. */
  const int32_t* expert_map;
  /* Shared experts (page §1: DeepSeek-V3 / Kimi K2 "+1 shared"): n_shared >= 0 SwiGLU experts
   * applied to every token with weight 1, outside the router and its scale. Their weights
   * follow the routed experts: W13/W2 hold E + n_shared experts. The router writes them as
   * slots k..k+n_shared-1 of every token (ids E..E+n_shared-1); align, the grouped GEMMs and
   * the combine then see k + n_shared slots and E + n_shared experts (expert_map, if given,
   * has E + n_shared entries). */
  int n_shared;
  moe_weight_format_t weight_format; /* MOE_WEIGHTS_NATIVE (0) unless FP8 weights */
  const float* w13_scale;            /* device fp32 block scales of W13 (FP8 only) */
  const float* w2_scale;             /* device fp32 block scales of W2 (FP8 only) */
} moe_config_t;

/* Byte offsets of the intermediates inside a moe_forward workspace (256-byte aligned). */
typedef struct moe_ws_layout {
  size_t logits;           /* fp32 [T, E] */
  size_t topk_ids;         /* int32 [T, k] */
  size_t topk_w;           /* fp32 [T, k] */
  size_t sorted_ids;       /* int32 [max_padded] */
  size_t expert_ids;       /* int32 [max_padded / block_m] */
  size_t num_post_padded;  /* int32 [1] */
  size_t counts;           /* int32 [E] */
  size_t align_scratch;    /* moe_align workspace */
  size_t act;              /* dtype [max_padded, I] */
  size_t xs;               /* bf16 [max_padded, H]: routed token rows in padded order */
  size_t y;                /* dtype [T*k, H] */
  size_t gemm_scratch;     /* FP8 weights, batches of > 128 tokens with >= 256 routed rows per
                              expert (shared experts counted): bf16 copies of one grouped GEMM's
                              weights, E x 2I x H x 2 bytes (see moe_forward); else empty */
  size_t total;            /* bytes required */
  int block_m;
  int max_padded;
} moe_ws_layout_t;

/* ABI version of the loaded library (MOE_ABI_VERSION). */
int moe_abi_version(void);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status_t s);

/* Tile height (BLOCK_M) the grouped GEMMs use for this configuration: 128 for bf16
 * (one tensor-core M tile), 16 for fp32. Host arithmetic only. Returns 0 on bad args. */
int moe_block_m(const moe_config_t* cfg);

/* 1 when the grouped GEMMs of this configuration run as the small-batch kernels (bf16
 * layers of at most 2 tokens, or at most 24 with FP8 expert weights; see
 * moe_expert_gemm1), 0 otherwise or on bad args. Host arithmetic only. */
int moe_small_batch(const moe_config_t* cfg);

/* Which kernels run the grouped GEMMs of a configuration (with block_m = moe_block_m(cfg)):
 * the same predicates the GEMM entry points dispatch on. Host arithmetic only. */
typedef enum {
  MOE_GEMM_INVALID = 0,      /* bad configuration */
  MOE_GEMM_SIMT = 1,         /* fp32 layers: CUDA-core tiles */
  MOE_GEMM_SMALL_BATCH = 2,  /* bf16 <= 2 tokens (FP8 weights <= 24): CUDA-core GEMVs */
  MOE_GEMM_DECODE_TC = 3,    /* other bf16 batches of <= 128 tokens: decode tensor-core GEMMs */
  MOE_GEMM_PAIR_TC = 4       /* larger bf16 batches: CTA-pair tensor-core GEMMs */
} moe_gemm_kernel_t;
moe_gemm_kernel_t moe_gemm_kernel(const moe_config_t* cfg);

/* Worst-case padded length T*k + min(E, T*k)*(block_m-1) (page §5: every expert that can
 * hold a row pads at most block_m-1 slots). Host arithmetic only; 0 on bad args. */
size_t moe_max_padded_rows(int T, int k, int E, int block_m);

/* Scratch bytes moe_align needs for (T, k, E, block_m); 0 is a valid answer. */
moe_status_t moe_align_workspace_size(int T, int k, int E, int block_m, size_t* bytes);

/* Workspace layout / size of moe_forward for cfg (host arithmetic only). */
moe_status_t moe_workspace_layout(const moe_config_t* cfg, moe_ws_layout_t* layout);
moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes);

/* The router GEMM alone (page §3: logits = x @ w_gate.T, the scores every router starts
 * from): logits[T, E] fp32 = x @ Wg^T accumulated in fp32, without the logit_bias (the
 * top-k adds it). Same kernels as the first half of moe_route. */
moe_status_t moe_route_logits(const moe_config_t* cfg, const void* x, const void* Wg,
                              float* logits, cudaStream_t stream);

/* Router (page §3 route(), §4 route_grouped()): logits = x @ Wg^T (+ logit_bias in mode 0)
 * accumulated in fp32, then top-k per cfg->mode. Writes logits[T,E] (fp32, required),
 * topk_ids[T,k+n_shared] (routed slots in descending selection key, then the shared
 * experts E..E+n_shared-1) and topk_w[T,k+n_shared] fp32 (shared slots: 1). */
moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* Wg, float* logits,
                       int32_t* topk_ids, float* topk_w, cudaStream_t stream);

/* Align (page §5): histogram of the T*k flat rows over E experts, pad every count to a
 * multiple of block_m, exclusive scan, stable scatter. Writes sorted_ids[max_padded],
 * expert_ids[max_padded/block_m], num_post_padded[1] (the padded total, on the device)
 * and, if non-NULL, counts[E]. ws/ws_bytes: scratch of moe_align_workspace_size bytes
 * (may be NULL when that size is 0). Ids outside [0, E) are skipped and flagged. */
moe_status_t moe_align(const int32_t* topk_ids, int T, int k, int E, int block_m,
                       int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_padded,
                       int32_t* counts, void* ws, size_t ws_bytes, cudaStream_t stream);

/* moe_align without a workspace argument. The pages have no counterpart: this exists for
 * callers that cannot give the library any device memory besides their inputs and outputs
 * (an application or server whose device memory is owned by its own pool, or a path where
 * cudaMalloc, which can synchronise the device, is not acceptable). Same arguments, results
 * and checks as moe_align, but the per-chunk histograms live in a fixed 256 KiB array inside
 * the library (held by every GPU that loads it until the process exits), so it never
 * allocates. Limit: ceil(T*k / 1024) * E <= 65536 (e.g. T*k <= 524288 at E = 128); larger
 * problems return MOE_ERR_UNSUPPORTED without launching anything. The first call on a device
 * looks up the array's device address (make it before any stream capture) and keeps it for
 * the life of the process: after cudaDeviceReset, or any teardown of the device's primary
 * context, the library's module reloads and that address is stale, so this entry point must
 * not be called on that device again in the same process. All calls on a
 * device share the array and it keeps the last call's contents (nothing in it needs to start
 * at zero: every call overwrites the part it reads); calls that overlap on the GPU race. */
moe_status_t moe_align_noalloc(const int32_t* topk_ids, int T, int k, int E, int block_m,
                               int32_t* sorted_ids, int32_t* expert_ids,
                               int32_t* num_post_padded, int32_t* counts, cudaStream_t stream);

/* Expert parallelism, applied to an align table: every tile label e >= 0 of
 * expert_ids[0..num_tiles) becomes expert_map[e] (-1: not on this device, skipped by the
 * GEMMs). Map entries outside [-1, E) become -1 and set device status 1. */
moe_status_t moe_apply_expert_map(int32_t* expert_ids, int num_tiles, const int32_t* expert_map,
                                  int E, cudaStream_t stream);

/* GEMM1 + SwiGLU (page §6 with the gate/up halves fused in one epilogue): for every
 * padded position p < num_post_padded whose row r = sorted_ids[p] < T*k,
 *   act[p, :] = silu(x[r / k] @ W1[e]^T) * (x[r / k] @ W3[e]^T),  e = expert_ids[p / block_m].
 * act is [max_padded, I] in padded order; rows of padding positions are not written.
 * block_m must be a multiple of moe_block_m(cfg). bf16: the routed token rows are first
 * gathered into padded order in ws (moe_expert_gemm1_workspace_size bytes, 256-byte
 * aligned), then multiplied on the tensor cores; fp32 gathers inside the GEMM.
 *
 * Decode batches (bf16 activations, at most 128 tokens, not small): both grouped GEMMs run
 * on the tensor cores with the expert weights as the 128-row MMA operand and each tile's
 * token rows, up to its last real one, as the other; one work item is (tile, 128 output
 * columns), one CTA per SM streams the weights. FP8 weights are turned into bf16 (code times
 * block scale) in shared memory on the way. Results agree with the larger-batch kernels to
 * within rounding (the same products, summed in another order), bit for bit from run to run.
 *
 * Small batches (moe_small_batch(cfg) = 1: bf16 layers of at most 2 tokens, 24 with FP8
 * weights): a tile then holds a few
 * real rows, and both grouped GEMMs run on CUDA cores as one pass over the active experts'
 * weights, fp32 products of the same operands summed in another order than the tensor-core
 * kernels' (the results agree to within rounding, not bit for bit). FP8 weights: each
 * 16-code partial sum is scaled by its block scale. No workspace is touched and the bf16
 * moe_expert_gemm1 reads the token rows in place (no gather). */
moe_status_t moe_expert_gemm1_workspace_size(const moe_config_t* cfg, int block_m,
                                             size_t* bytes);
moe_status_t moe_expert_gemm1(const moe_config_t* cfg, const void* x, const void* W13,
                              const int32_t* sorted_ids, const int32_t* expert_ids,
                              const int32_t* num_post_padded, int block_m, void* act,
                              void* ws, size_t ws_bytes, cudaStream_t stream);

/* The two halves of the bf16 moe_expert_gemm1, for callers that keep the routed rows:
 * moe_gather_rows writes xs[p, :] = x[sorted_ids[p] / k, :] for every p < num_post_padded
 * with sorted_ids[p] < T*k (padding rows untouched; xs is [max_padded, H] of dtype, 16-byte
 * aligned); moe_expert_gemm1_gathered runs GEMM1 + SwiGLU on those rows (bf16 only, else
 * MOE_ERR_UNSUPPORTED) with ws of moe_expert_gemm1_gathered_workspace_size bytes (0 with the
 * current kernels, ws may then be NULL; callers that size ws through this query stay correct
 * if a kernel needs scratch). Page §2 lists both
 * feeds, a permuted copy and an in-GEMM gather; this pair is the permuted-copy feed with the
 * permutation taken from sorted_ids. */
moe_status_t moe_gather_rows(const void* x, const int32_t* sorted_ids,
                             const int32_t* num_post_padded, int T, int k, int H,
                             moe_dtype_t dtype, void* xs, cudaStream_t stream);
moe_status_t moe_expert_gemm1_gathered_workspace_size(const moe_config_t* cfg, int block_m,
                                                      size_t* bytes);
moe_status_t moe_expert_gemm1_gathered(const moe_config_t* cfg, const void* xs,
                                       const void* W13, const int32_t* sorted_ids,
                                       const int32_t* expert_ids,
                                       const int32_t* num_post_padded, int block_m, void* act,
                                       void* ws, size_t ws_bytes, cudaStream_t stream);

/* FP8 E4M3 expert weights (cfg->weight_format MOE_WEIGHTS_FP8_E4M3_B128) as bf16 weights:
 * out[e, r, c] = code[e, r, c] * its 128 x 128 block scale, rounded to bf16 as the grouped
 * GEMMs' in-kernel conversion rounds it (exact for power-of-two scales), for every expert slot
 * e < E + n_shared. matrix 1: codes are W13 [E+n_shared, 2I, H] with cfg->w13_scale; matrix
 * 2: W2 [E+n_shared, H, I] with cfg->w2_scale. counts (optional, E+n_shared entries, e.g.
 * moe_align's): experts whose count is 0 are skipped (out left untouched). codes and out
 * 16-byte aligned; out holds (E+n_shared) x 2I x H (matrix 1) or x H x I (matrix 2) bf16.
 * moe_forward does this at prefill, with out in its workspace's gemm_scratch, and runs the
 * bf16 grouped GEMMs on it; a caller of the separate entry points can do the same (a
 * configuration without the scales then describes the bf16 weights). The pages give FP8
 * weights as a storage format (§8 intensity with 1-byte weights); the conversion is this
 * library's. */
moe_status_t moe_dequant_fp8_weights(const moe_config_t* cfg, int matrix, const void* codes,
                                     const int32_t* counts, void* out, cudaStream_t stream);

/* GEMM2 with the router weight (page §6): for every padded position p with r < T*k,
 *   y[r, :] = topk_w[r] * (act[p] @ W2[e]^T).  Each row r < T*k is written exactly once;
 * padding rows are never written. ws: moe_expert_gemm2_workspace_size bytes, 256-byte
 * aligned (0 with the current kernels, ws may then be NULL). */
moe_status_t moe_expert_gemm2_workspace_size(const moe_config_t* cfg, int block_m,
                                             size_t* bytes);
moe_status_t moe_expert_gemm2(const moe_config_t* cfg, const void* act, const void* W2,
                              const int32_t* sorted_ids, const int32_t* expert_ids,
                              const int32_t* num_post_padded, int block_m,
                              const float* topk_w, void* y, void* ws, size_t ws_bytes,
                              cudaStream_t stream);

/* Both expert GEMMs: GEMM1 into ws (act, then GEMM1's scratch: the gathered rows of bf16),
 * then GEMM2 into y[T*k, H]. ws: moe_grouped_swiglu_workspace_size bytes, 256-byte
 * aligned. */
moe_status_t moe_grouped_swiglu_workspace_size(const moe_config_t* cfg, int block_m,
                                               size_t* bytes);
moe_status_t moe_grouped_swiglu(const moe_config_t* cfg, const void* x, const void* W13,
                                const void* W2, const int32_t* sorted_ids,
                                const int32_t* expert_ids, const int32_t* num_post_padded,
                                int block_m, const float* topk_w, void* y, void* ws,
                                size_t ws_bytes, cudaStream_t stream);

/* Combine (page §6, the sum over k): out[t, :] = sum_{j=0..k-1} y[t*k + j, :] in fp32,
 * slots added in order j = 0, 1, ..., stored in dtype. */
moe_status_t moe_combine(const void* y, int T, int k, int H, moe_dtype_t dtype, void* out,
                         cudaStream_t stream);

/* Combine with expert parallelism: as moe_combine, but slot j of token t is skipped when
 * expert_map[topk_ids[t, j]] < 0 (its expert is on another device and its y row is not
 * written here). topk_ids [T, k] int32, expert_map [E] int32, both on the device. A slot
 * whose id lies outside [0, E) is skipped too (its y row was never written: the align step
 * drops such ids) and sets device status 1. */
moe_status_t moe_combine_local(const void* y, const int32_t* topk_ids, const int32_t* expert_map,
                               int E, int T, int k, int H, moe_dtype_t dtype, void* out,
                               cudaStream_t stream);

/* Fixed-capacity ("masked") expert layout for decode without an align step (page §7:
 * "fixed-capacity masked layouts that keep shapes static for CUDA Graphs"; §9: DeepGEMM's
 * masked layout, a capacity per expert plus a valid-row count). Tokens arrive bucketed:
 * x_masked[E, C, H] (cfg->dtype) with counts[e] valid rows (device int32 [E], 0..C) in
 * expert e's bucket; for i < counts[e]:
 *   y_masked[e, i, :] = row_w[e, i] * W2[e] (silu(W1[e] x) * (W3[e] x)),   x = x_masked[e, i]
 * (row_w: device fp32 [E, C], or NULL for weight 1). Rows past a count are never written.
 * C must be a multiple of moe_block_m(cfg); cfg->T, k and the router fields are ignored.
 * bf16 with C = 128 (one tile per expert, the decode case) runs the decode tensor-core
 * GEMMs, which stream each active expert's weights once; larger C the CTA-pair GEMMs.
 * moe_masked_table builds the equivalent sorted_ids / expert_ids / num_post_padded (the
 * identity on valid rows, tiles past a count labelled -1) for callers of the GEMM entries. */
moe_status_t moe_masked_table(const int32_t* counts, int E, int capacity, int block_m,
                              int32_t* sorted_ids, int32_t* expert_ids,
                              int32_t* num_post_padded, cudaStream_t stream);
moe_status_t moe_masked_workspace_size(const moe_config_t* cfg, int capacity, size_t* bytes);
moe_status_t moe_masked_forward(const moe_config_t* cfg, const void* x_masked,
                                const int32_t* counts, int capacity, const float* row_w,
                                const void* W13, const void* W2, void* y_masked, void* ws,
                                size_t ws_bytes, cudaStream_t stream);

/* The whole layer: route -> align (-> expert map) -> GEMM1+SwiGLU -> GEMM2 -> combine, all
 * enqueued on `stream` with no host round-trip. ws must hold moe_workspace_size(cfg) bytes, 256-byte
 * aligned; its intermediates sit at moe_workspace_layout(cfg) offsets. Decode batches (at most
 * 8 tokens and 32 routed slots) take top-k and the table (expert map applied) from one small
 * CTA. With FP8 weights and a large batch (the layout's gemm_scratch is not empty), each
 * grouped GEMM's weights are first written as bf16 (code times block scale, rounded as the
 * GEMMs' in-kernel conversion rounds it) into gemm_scratch, skipping experts no row reached
 * unless an expert map is set, and the bf16 GEMM runs on them. The results are those of the
 * separate entry points, bit for bit. */
moe_status_t moe_forward(const moe_config_t* cfg, const void* x, const void* Wg,
                         const void* W13, const void* W2, void* out, void* ws,
                         size_t ws_bytes, cudaStream_t stream);

/* Diagnostic self-test of the failure path: enqueues one CTA whose pipeline waits nothing
 * will satisfy (it also holds tensor memory). After the 2 s pipeline-wait limit the waits
 * give up, the CTA frees its tensor memory and returns, and the device status word reads 2
 * (a pipeline wait ran out of time): a stalled pipeline ends with a status, not a hang, and
 * the context stays usable. Takes about 2 s of device time. */
moe_status_t moe_selftest_wait_timeout(cudaStream_t stream);

/* Diagnostic (synchronises the current device): returns the device status word (0 = no
 * fault seen; 1 = an expert id outside [0, E); 2 = a wait ran out of time; 3 = the
 * two CTAs of a tensor-core pair were given different tensor-memory columns) and
 * clears it when reset != 0. Not for use inside stream capture. */
int moe_device_status(int reset);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
