/*
 * moe_prefill.h -- C ABI of the GB300 (sm_103a) routed-MoE NVFP4 (W4A16) prefill library.
 *
 * One chunk of prefill rows runs: top-k routing -> stable expert sort -> one grouped W4A16
 * gate/up GEMM over all experts (activations gathered in the kernel through
 * sorted_token_ids) -> clamped SwiGLU -> one grouped down GEMM -> routing-weighted combine
 * back to token order.  The operations follow the web pages "Module forward_prefill_gemm"
 * (module docs and source of spark_model::layers::glm5next_mlp::forward_prefill_gemm) and
 * the two "glm5next_mlp/forward.rs" pages (spark_model, older; metrale_model_arch, newer).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers marked "device" are CUDA device pointers; "host" pointers are CPU memory.
 * - BF16 tensors are passed as uint16_t bit patterns.  All matrices are row-major.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Every
 *   compute call is asynchronous on that stream, launches kernels only, allocates nothing
 *   and never synchronises or copies device -> host.
 * - The caller owns every buffer.  The only calls that allocate are
 *   moe_expert_table_create (once, at load) and moe_expert_table_destroy (frees it).
 * - Every call returns a moe_status.  Host-side argument checks run before any launch; a
 *   call that returns an error has launched nothing.  Problems only the GPU can see (an
 *   expert id out of range, inconsistent offsets, a pipeline wait that timed out) set a
 *   sticky device error word that moe_get_device_error() reads and clears.  Nothing aborts
 *   the process, nothing traps the GPU.
 */
#ifndef MOE_PREFILL_H
#define MOE_PREFILL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status codes */
typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,        /* NULL where a buffer is required, negative size, ...  */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* a shape outside what the kernels support (see calls) */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3,
  MOE_ERR_CUDA = 4,               /* a CUDA runtime call failed (launch, copy, attribute) */
  MOE_ERR_DEVICE = 5,             /* moe_get_device_error: a device-side check fired      */
  MOE_ERR_NOT_BUILT_FOR_DEVICE = 6,/* the current GPU is not sm_103 / sm_100 family       */
  MOE_ERR_SCRATCH_LIMIT = 7       /* needs more than the fixed static scratch of
                                     moe_sort_by_expert_noalloc (MOE_SORT_NOALLOC_MAX_INTS) */
} moe_status;

/* device error codes (value of *code from moe_get_device_error) */
#define MOE_DEVERR_NONE 0
#define MOE_DEVERR_BAD_EXPERT_ID 1   /* an id outside [-1, E) reached the sort; treated as -1 */
#define MOE_DEVERR_BAD_OFFSETS 2     /* expert_offsets not monotone or past R; GEMM skipped  */
#define MOE_DEVERR_TIMEOUT 3         /* a pipeline wait in a GEMM kernel exceeded its limit  */
#define MOE_DEVERR_NAN_LOGIT 4       /* a NaN routing logit; it is ranked below every number */
#define MOE_DEVERR_BAD_GATHER 5      /* a gather index outside [0, a_rows); row 0 was read */
#define MOE_DEVERR_SMALL_ROWS 6      /* an expert has more rows than the small-row products take */

/* output element type of the grouped GEMM */
#define MOE_DTYPE_BF16 0
#define MOE_DTYPE_F32 1

/* ---------------------------------------------------------------- NVFP4 expert tables */
/*
 * One projection (gate/up, or down) of all experts, indexed by GLOBAL expert id.
 * Per expert e ("Module forward_prefill_gemm", table "Layout compatibility"):
 *   packed[e]  device, uint8 [N, K/2]: row n, byte k/2 holds logical k; even k is the low
 *              nibble, odd k the high nibble; each nibble is an E2M1 code.
 *   scales[e]  device, uint8 [N, K/16]: E4M3 block scale of (n, k) at [n, k/16].
 *   scale2[e]  FP32 per-expert scale.
 * The dequantised weight is bf16( fp32( fp32(E2M1[nibble] * e4m3) * scale2 ) ), i.e. the
 * value the pages' grouped kernel stages ("What is NOT bit-identical", item 2).
 * packed[e] == NULL marks an absent (remote, expert-parallel) expert: its rows are never
 * read; the GEMMs write zeros to its output rows, which is what the pages' zeroed
 * routed-output buffer left there.
 *
 * Requirements: 1 <= E <= 512, N % 8 == 0, 8 <= N, K % 256 == 0, K >= 256; every non-NULL
 * packed[e] and scales[e] 16-byte aligned.  The weights are NOT copied: the table refers to
 * the caller's buffers, which must outlive it.
 *
 * packed, scales: host arrays of E device pointers.  scale2: host array of E floats.
 * On success *out receives an opaque table (device memory for the per-expert TMA
 * descriptors, pointers and scale2 values, allocated here, once).
 */
typedef struct moe_expert_table moe_expert_table;

int moe_expert_table_create(const void* const* packed, const void* const* scales, const float* scale2,
                            int E, int N, int K, moe_expert_table** out);
/* Frees a table (synchronises the device first). NULL is accepted. */
int moe_expert_table_destroy(moe_expert_table* table);
/* Reads back E, N, K of a table (host only). */
int moe_expert_table_shape(const moe_expert_table* table, int* E, int* N, int* K);

/* ---------------------------------------------------------------- routing */
/*
 * Router logits: logits[t, e] = sum_h x[t, h] * w_router[e, h], BF16 inputs, FP32
 * accumulation and output ("glm5next_mlp/forward.rs", forward_moe: the router writes
 * [rows, num_experts] F32 logits).
 *   x        device BF16 [T, H]
 *   w_router device BF16 [E, H]
 *   logits   device FP32 [T, E] (output)
 * Requirements: T >= 1, 1 <= E <= 1024, H % 8 == 0, x and w_router 16-byte aligned.
 */
int moe_router_logits(const uint16_t* x, const uint16_t* w_router, int T, int H, int E, float* logits,
                      void* stream);

/*
 * Top-k routing, one launch for all rows ("glm5next_mlp/forward.rs", forward_moe: one
 * glm5next_router_topk launch with router_bias, routed_scale and renormalize):
 *   key[t, e] = logits[t, e] (+ bias[e], FP32 add, when bias != NULL; bias only selects);
 *   ids[t, :] = the k experts of largest key, in descending key order, ties to the lower id;
 *   wts[t, s] = softmax of the k selected (unbiased) logits * routed_scale when renormalize,
 *               else the full-E softmax value * routed_scale.
 *   logits device FP32 [T, E]; bias device FP32 [E] or NULL;
 *   ids    device int32 [T, k] (output); wts device FP32 [T, k] (output).
 * Requirements: T >= 1, 1 <= E <= 1024, 1 <= k <= min(E, 32).
 * A NaN logit ranks below every number and sets MOE_DEVERR_NAN_LOGIT.
 */
int moe_route_topk(const float* logits, const float* bias, int T, int E, int k, int renormalize,
                   float routed_scale, int32_t* ids, float* wts, void* stream);

/* ---------------------------------------------------------------- expert sort */
/*
 * Stable counting sort of the R = T*k routed slots by expert id ("glm5next_mlp/forward.rs"
 * (metrale), Glm5NextMlpWorkspace fields sorted_token_ids, sorted_expert_ids,
 * expert_offsets, token_to_perm).  Slot i = t*k + s with id e goes to sorted row
 *   p = expert_offsets[e] + (number of earlier slots i' < i with the same id);
 *   sorted_token_ids[p] = t (the original token), sorted_expert_ids[p] = e,
 *   token_to_perm[i] = p, expert_offsets[0] = 0, expert_offsets[E] = number of valid slots.
 * A slot with id -1 (the pages' "slot unfilled" sentinel) goes to a tail after
 * expert_offsets[E] (sorted_expert_ids = -1) and gets token_to_perm = -1.  An id outside
 * [-1, E) is treated as -1 and sets MOE_DEVERR_BAD_EXPERT_ID.
 *   ids              device int32 [T, k]
 *   sorted_token_ids device int32 [T*k] (output)
 *   sorted_expert_ids device int32 [T*k] (output)
 *   expert_offsets   device int32 [E+1] (output)
 *   token_to_perm    device int32 [T*k] (output)
 *   ws, ws_bytes     device scratch of at least moe_sort_workspace_bytes(T, k, E) bytes
 * Requirements: T >= 1, 1 <= k <= 32, 1 <= E <= 1024, T*k < 2^31.
 */
size_t moe_sort_workspace_bytes(int T, int k, int E);
int moe_sort_by_expert(const int32_t* ids, int T, int k, int E, int32_t* sorted_token_ids,
                       int32_t* sorted_expert_ids, int32_t* expert_offsets, int32_t* token_to_perm, void* ws,
                       size_t ws_bytes, void* stream);

/*
 * moe_sort_by_expert without a caller workspace and without allocating.  The pages describe
 * no such call: it exists for callers that cannot hand the library scratch memory and must
 * not allocate any -- e.g. a serving loop that froze its memory pool after warm-up, code
 * running inside an allocator's own callback, or any place where cudaMalloc/cudaFree would be
 * wrong because they can synchronise the device or fail under memory pressure.
 *
 * Same arguments, outputs, requirements and device errors as moe_sort_by_expert, minus
 * ws/ws_bytes.  The scratch (the per-segment expert histogram, (E+1)*ceil(T*k/2048) int32) is
 * a fixed array of MOE_SORT_NOALLOC_MAX_INTS int32 (256 KiB) in the library's own device
 * memory, one per device, reserved when the library's device code loads; no call allocates.
 *   - Limit: (E+1) * ceil(T*k / 2048) <= MOE_SORT_NOALLOC_MAX_INTS (e.g. E = 160: T*k up to
 *     about 833k slots; E = 512: about 261k).  A larger problem returns MOE_ERR_SCRATCH_LIMIT
 *     before anything is launched; use moe_sort_by_expert with a workspace instead.
 *   - Nothing in the scratch has to start at zero: every count is written before it is read
 *     in the same call.
 *   - Calls that can overlap in time on one device race on the shared scratch: two streams,
 *     or two host threads, each with a call in flight.  Calls issued in order on one stream
 *     are safe.
 *   - The first call on each device looks the scratch's address up (cudaGetSymbolAddress);
 *     make that first call before any stream capture that includes this call.
 */
#define MOE_SORT_NOALLOC_MAX_INTS 65536
int moe_sort_by_expert_noalloc(const int32_t* ids, int T, int k, int E, int32_t* sorted_token_ids,
                               int32_t* sorted_expert_ids, int32_t* expert_offsets, int32_t* token_to_perm,
                               void* stream);

/* ---------------------------------------------------------------- grouped W4A16 GEMM */
/*
 * One launch for all experts ("Module forward_prefill_gemm", "What this replaces"):
 *   C[p, n] = sum_k A[g(p), k] * Wdq_e[n, k]   for every sorted row p in
 *   [expert_offsets[e], expert_offsets[e+1]), n < N,
 * where g(p) = gather_ids[p] (the in-kernel A gather through sorted_token_ids) or p when
 * gather_ids is NULL, and Wdq_e is expert e's dequantised BF16 weight (see the table).
 * BF16 operands, FP32 accumulation; C is BF16 (rounded to nearest even) or FP32.
 * Rows of absent experts (packed NULL) are written as zeros; rows past expert_offsets[E]
 * are not touched.
 *   A            device BF16 [a_rows, lda], K = W->K columns used, lda >= K
 *   gather_ids   device int32 [R] or NULL; every value must be in [0, a_rows)
 *   W            expert table (E, N, K)
 *   expert_offsets device int32 [E+1], non-decreasing, expert_offsets[E] <= R
 *   C            device [R, ldc] of c_dtype (output), ldc >= N
 * Requirements: lda % 8 == 0, ldc % 8 == 0, A and C 16-byte aligned, R >= 1.
 * The kernel reads expert_offsets on the device: no host round trip, graph-capturable.
 * Kernels: up to ~128 rows per expert (or with gather_ids) single-CTA tiles whose thread-block
 * clusters share activation tiles through cluster-multicast TMA loads; above that, and for
 * contiguous rows with N % 256 == 0 and K % 256 == 0, CTA pairs (tcgen05 cta_group::2).  A run on
 * more than one GPU uses moe_prefill_forward with MOE_FWD_NO_MULTICAST instead.
 */
int moe_w4a16_grouped_gemm(const uint16_t* A, int a_rows, int lda, const int32_t* gather_ids,
                           const moe_expert_table* W, const int32_t* expert_offsets, int R, void* C, int ldc,
                           int c_dtype, void* stream);

/*
 * The gate/up GEMM with the clamped SwiGLU fused into its epilogue ("glm5next_mlp/forward.rs"
 * (metrale), swiglu_rows, applied to the gate/up product of the grouped-prefill arm):
 *   act[p, j] = silu(min(g, L)) * clamp(u, -L, L),  g = C[p, j], u = C[p, I + j], j < I,
 * with C the moe_w4a16_grouped_gemm product over a gate/up table of N = 2I rows (rows 0..I-1
 * gate, I..2I-1 up).  g and u are the FP32 accumulators rounded to BF16 (nearest even), the
 * values the pages' BF16 gate and up buffers hold ("glm5next_mlp/forward.rs" (spark),
 * forward_dense: a_gate, a_up); silu(z) = z / (1 + e^-z) in FP32; act is rounded to BF16.  The
 * N x R product never goes to memory.  Rows of absent experts are written as zeros.
 *   act          device BF16 [R, ld_act] (output), ld_act >= I, ld_act % 8 == 0
 * Other arguments as moe_w4a16_grouped_gemm.  Requires W->N = 2I with I % 128 == 0.
 */
int moe_w4a16_grouped_gemm_swiglu(const uint16_t* A, int a_rows, int lda, const int32_t* gather_ids,
                                  const moe_expert_table* W, const int32_t* expert_offsets, int R, uint16_t* act,
                                  int ld_act, float limit, void* stream);

/*
 * Dequantise one expert's NVFP4 weight to a dense BF16 matrix with the grouped GEMM's own
 * device routine (for inspection and tests; the GEMMs never materialise this matrix):
 *   out[n, k] = bf16( fp32( fp32(E2M1[nibble(n, k)] * e4m3(scales[n, k/16])) * scale2 ) ).
 *   packed device uint8 [N, K/2]; scales device uint8 [N, K/16]; out device BF16 [N, K].
 * Requirements: N >= 1, K % 64 == 0, packed and out 16-byte aligned, scales 4-byte aligned.
 */
int moe_dequant_nvfp4(const void* packed, const void* scales, float scale2, int N, int K, uint16_t* out,
                      void* stream);

/* ---------------------------------------------------------------- activation and combine */
/*
 * Clamped SwiGLU ("glm5next_mlp/forward.rs", swiglu / swiglu_rows):
 *   out[r, j] = silu(min(gate[r, j], L)) * clamp(up[r, j], -L, L),  silu(z) = z / (1 + e^-z),
 * FP32 math, BF16 in and out.  gate/up/out are device BF16 with row strides ld_in/ld_out
 * (elements); the fused gate/up GEMM output [R, 2I] is used as gate = G, up = G + I.
 * Requirements: rows >= 0, width >= 1, width % 8 == 0, ld_in % 8 == 0, ld_out % 8 == 0,
 * 16-byte aligned pointers.
 */
int moe_swiglu_clamp(const uint16_t* gate, const uint16_t* up, int64_t rows, int64_t width, int64_t ld_in,
                     uint16_t* out, int64_t ld_out, float limit, void* stream);

/*
 * Routing-weighted combine back to token order ("glm5next_mlp/forward.rs" (metrale),
 * forward_moe: glm5next_moe_combine_indexed):
 *   out[t, h] = sum_{s<k} wts[t, s] * Y[token_to_perm[t, s], h]  (+ shared_out[t, h]),
 * FP32 accumulation in slot order, BF16 output.  A slot with token_to_perm = -1 adds zero.
 *   Y device BF16 [*, H] expert-sorted; token_to_perm device int32 [T, k];
 *   wts device FP32 [T, k]; shared_out device BF16 [T, H] or NULL; out device BF16 [T, H].
 * Requirements: T >= 1, 1 <= k <= 32, H % 8 == 0, 16-byte aligned BF16 pointers.
 */
int moe_combine_indexed(const uint16_t* Y, const int32_t* token_to_perm, const float* wts,
                        const uint16_t* shared_out, int T, int k, int H, uint16_t* out, void* stream);

/* ---------------------------------------------------------------- small-row products */
/*
 * The grouped W4A16 products for chunks with at most 8 rows per expert (decode-like): the same
 * C[p, n] = sum_k A[g(p), k] * W_e[n, k] as moe_w4a16_grouped_gemm, computed without tensor
 * cores with the dequantised weights kept in FP32 (E2M1 * E4M3 exact, scale2 applied to the
 * FP32 sums), the arithmetic of the pages' decode GEMV ("Module forward_prefill_gemm",
 * "What is NOT bit-identical", item 2); C is BF16.  _swiglu: a gate/up table of N = 2I rows
 * gives act[p, j] = silu(min(g, L)) * clamp(u, -L, L) from the FP32 gate and up sums.
 * Arguments as moe_w4a16_grouped_gemm(_swiglu) (C BF16 only).  An expert with more than 8 rows
 * sets MOE_DEVERR_SMALL_ROWS and its rows are not written; expert_offsets outside [0, R] set
 * MOE_DEVERR_BAD_OFFSETS.  Requires lda % 8 == 0 and A 16-byte aligned.
 * Measured on GB300 at GLM shapes (hidden 5120, intermediate 1536, 160 experts, top-8), whole
 * forward: 0.155 / 0.204 / 0.287 / 0.462 ms at T = 1 / 2 / 4 / 8 rows against 0.116 / 0.173 /
 * 0.233 / 0.379 ms with the tensor-core GEMMs: the numerics option, not the fast path.
 */
int moe_w4a16_grouped_gemv(const uint16_t* A, int a_rows, int lda, const int32_t* gather_ids,
                           const moe_expert_table* W, const int32_t* expert_offsets, int R, uint16_t* C, int ldc,
                           void* stream);
int moe_w4a16_grouped_gemv_swiglu(const uint16_t* A, int a_rows, int lda, const int32_t* gather_ids,
                                  const moe_expert_table* W, const int32_t* expert_offsets, int R, uint16_t* act,
                                  int ld_act, float limit, void* stream);

/* ---------------------------------------------------------------- shared expert */
/*
 * The shared expert over every row ("glm5next_mlp/forward.rs" (spark), forward_dense): a
 * dense SwiGLU MLP with BF16 weights,
 *   gate = x W_gate^T, up = x W_up^T (BF16 out), act = silu(min(gate, L)) * clamp(up, -L, L)
 *   (BF16), shared_out = act W_down^T (BF16),
 * FP32 accumulation.  Its output joins the routed sum in moe_prefill_forward's combine.
 * Three launches of this library's kernels: one dense tensor-core GEMM for gate and up (written
 * as gate | up into the workspace), the SwiGLU, and one dense tensor-core GEMM for down.
 *   x          device BF16 [T, H]
 *   w_gate, w_up device BF16 [I, H];  w_down device BF16 [H, I]
 *   ws, ws_bytes device workspace of at least moe_shared_expert_workspace_bytes(T, H, I) bytes,
 *              256-byte aligned: gate | up [T, 2I] BF16 at offset 0, then act [T, I] BF16 at the
 *              next multiple of 256 bytes (nothing is allocated per call)
 *   shared_out device BF16 [T, H] (output)
 * Requirements: T >= 1, H and I multiples of 8, buffers 16-byte aligned, 0 < limit.
 */
size_t moe_shared_expert_workspace_bytes(int T, int H, int I);
int moe_shared_expert_forward(const uint16_t* x, int T, int H, int I, const uint16_t* w_gate, const uint16_t* w_up,
                              const uint16_t* w_down, float limit, void* ws, size_t ws_bytes, uint16_t* shared_out,
                              void* stream);

/* ---------------------------------------------------------------- fused forward */
typedef struct {
  int hidden;             /* H */
  int moe_intermediate;   /* I (gate/up table has N = 2I: rows 0..I-1 gate, I..2I-1 up) */
  int num_experts;        /* E */
  int top_k;              /* k */
  float swiglu_limit;     /* L, e.g. 7.0 */
  int renormalize;        /* 1: renormalise the top-k weights */
  float routed_scale;     /* multiplier of the routing weights, e.g. 1.0 */
  int flags;              /* 0, or MOE_FWD_SEPARATE_SWIGLU | MOE_FWD_SMALL_ROWS | MOE_FWD_NO_MULTICAST */
} moe_prefill_config;

/* moe_prefill_config.flags: run the SwiGLU as its own kernel on a materialised G [R, 2I]
 * (BF16) instead of in the gate/up GEMM's epilogue (the default); for inspection and tests. */
#define MOE_FWD_SEPARATE_SWIGLU 1
/* moe_prefill_config.flags: chunks of at most 8 rows take the small-row products
 * (moe_w4a16_grouped_gemv*: FP32 dequantised weights, the numerics of the pages' decode GEMV)
 * instead of the tensor-core GEMMs (faster on this GPU: see the small-row products' header). */
#define MOE_FWD_SMALL_ROWS 2
/* moe_prefill_config.flags: no cluster-multicast TMA loads (the single-CTA GEMM's activation
 * tiles are then loaded by each CTA itself).  For runs on more than one GPU (expert parallelism,
 * "Module forward_prefill_gemm", "Layout compatibility": remote experts as NULL table entries,
 * the caller all-reducing out), where this library keeps multicast out; results are identical. */
#define MOE_FWD_NO_MULTICAST 4

/* Workspace bytes for moe_prefill_forward with up to max_rows rows (0 on a bad config). */
size_t moe_workspace_bytes(const moe_prefill_config* cfg, int max_rows);

/* Number of stage events moe_prefill_forward records when stage_events != NULL. */
#define MOE_FWD_NUM_EVENTS 8

/*
 * The whole routed-MoE prefill site for T rows ("glm5next_mlp/forward.rs" (metrale),
 * forward_moe, grouped-prefill arm): router logits (when w_router != NULL) -> top-k ->
 * expert sort -> grouped gate/up GEMM with the A gather -> SwiGLU -> grouped down GEMM ->
 * indexed combine.  No host round trip (the pages read expert_offsets back once; here the
 * GEMMs schedule their tiles from expert_offsets on the device), so the call can be captured
 * in a CUDA graph.
 *   x          BF16 [T, H], device memory or host memory the device can read (page-locked, or
 *              any host memory where the device has pageable memory access): a host x is staged
 *              into the workspace's x_stage by the router kernel as it reads it (without a router,
 *              by a staging kernel), and the expert GEMMs read the staged rows; when the CTA-pair
 *              gate/up GEMM takes its rows in expert order (more than 128 rows per expert) and
 *              there is no router, the kernel that stores those rows reads each host row once
 *              and x_stage stays unused
 *   w_router   device BF16 [E, H] or NULL
 *   logits_in  FP32 [T, E] or NULL (exactly one of w_router / logits_in); device memory or host
 *              memory the device can read (the top-k reads it in place)
 *   router_bias device FP32 [E] or NULL (selection only)
 *   w_gate_up  table with E = cfg E, N = 2I, K = H;  w_down: E, N = H, K = I
 *   ws, ws_bytes device workspace >= moe_workspace_bytes(cfg, T), 256-byte aligned (G takes
 *              space only with MOE_FWD_SEPARATE_SWIGLU).  Its
 *              contents after the call: logits, ids, wts, the sort arrays, G, act, Y, at the
 *              offsets moe_workspace_layout reports.
 *   out        BF16 [T, H] in memory the device can store to: device memory, or host memory
 *              as for x (the combine then writes the result straight to the host; no copy
 *              follows).  An x, logits_in or out the device cannot reach: MOE_ERR_INVALID_ARG.
 *   shared_out device BF16 [T, H] or NULL: the shared expert's output, added in the combine
 *              (moe_shared_expert_forward)
 *   shared_ready NULL, or a cudaEvent_t (as void*) the stream waits for right before the
 *              combine: shared_out may then be produced on another stream, concurrently with
 *              the routed steps
 *   stage_events NULL, or a host array of MOE_FWD_NUM_EVENTS cudaEvent_t (as void*) recorded
 *              on `stream` before the first stage and after each of the 7 stages (router,
 *              top-k, sort count, sort scatter, gate/up GEMM, SwiGLU, down GEMM, combine
 *              -> events 0..7 bracket them; with a router and E <= 64 the router GEMM and
 *              the top-k run as one launch (event 2 = event 1; the logits, ids and weights
 *              equal those of moe_router_logits + moe_route_topk), a skipped router records event 1 = event
 *              0, and with the fused SwiGLU (the default) event 5 = event 4).
 * The SwiGLU runs in the gate/up GEMM's epilogue (moe_w4a16_grouped_gemm_swiglu) unless
 * cfg->flags has MOE_FWD_SEPARATE_SWIGLU; then G is written to the workspace first.  With the
 * fused SwiGLU the down GEMM overlaps the gate/up GEMM's last tiles: it starts on an expert once
 * the gate/up GEMM has published that expert's activation rows through the workspace's `ready`
 * counters, and takes its tiles dynamically (bounded waits; a gate/up launch that fails to
 * publish makes the down launch record MOE_DEVERR_TIMEOUT after 2 s instead of hanging).  With
 * MOE_FWD_SMALL_ROWS, chunks of T <= 8 rows take the small-row products (FP32 dequantised
 * weights, as the pages' decode GEMV) instead of the tensor-core GEMMs.
 */
int moe_prefill_forward(const moe_prefill_config* cfg, const uint16_t* x, int T, const uint16_t* w_router,
                        const float* logits_in, const float* router_bias, const moe_expert_table* w_gate_up,
                        const moe_expert_table* w_down, void* ws, size_t ws_bytes, uint16_t* out,
                        const uint16_t* shared_out, void* shared_ready, void* const* stage_events, void* stream);

/* Byte offsets of the workspace buffers moe_prefill_forward fills (for tests/inspection).
 * `ready`: INT32 [2E + 1]: [0, E) per-expert counters through which the down GEMM starts on an
 * expert as soon as the gate/up GEMM has stored its activation rows, [E] the down GEMM's dynamic
 * tile counter, [E + 1, 2E + 1) the per-expert counts of token rows the CTA-pair gate/up GEMM
 * has stored in expert order (all cleared by the sort on every call).  `x_stage`: BF16 [T, H],
 * the device copy of an x passed in host memory (unused when x is device memory, and on the
 * host-x CTA-pair path above).  `x_sorted`: BF16 [T * top_k, H], the token rows in expert order
 * (row p = x[sorted_token_ids[p]], for the rows of experts present in w_gate_up) that the CTA-pair
 * gate/up GEMM stores and reads (unused with the single-CTA kernel, which gathers inside the
 * GEMM). */
typedef struct {
  size_t logits, ids, wts, sorted_token_ids, sorted_expert_ids, expert_offsets, token_to_perm, sort_scratch, ready,
      G, act, Y, x_stage, x_sorted, total;
} moe_workspace_layout_t;
int moe_workspace_layout(const moe_prefill_config* cfg, int max_rows, moe_workspace_layout_t* layout);

/* ---------------------------------------------------------------- debug controls */
/*
 * Test and debug settings of the whole process (no counterpart on the pages).  They change
 * which code runs or how long it waits, never what it computes; both are process-global and
 * take effect for the launches issued after the call.
 *
 * moe_debug_set_gemm_kernel: which grouped GEMM kernel the GEMM entry points and the forward
 * launch.  MOE_GEMM_KERNEL_AUTO (the default) takes the CTA-pair kernel where it is faster
 * (experts averaging more than 128 sorted rows) and its shapes allow it (N % 256 == 0; with the
 * fused SwiGLU I % 128 == 0; A rows contiguous -- in the forward the pair kernel stores the gate/up
 * GEMM's gathered rows in expert order itself), and the single-CTA kernel otherwise; SINGLE always takes the
 * single-CTA kernel; PAIR takes the pair kernel for every shape it allows and makes the entry
 * points return MOE_ERR_UNSUPPORTED_SHAPE for the others.  Returns MOE_ERR_INVALID_ARG for
 * another value.
 *
 * moe_debug_set_wait_limit_ns: the bound of every pipeline wait of the CTA-pair kernel
 * (default and maximum 2 s; 0 restores the default).  After the bound a waiting kernel records
 * MOE_DEVERR_TIMEOUT, drains its copies and MMAs and returns.  Returns the previous bound.
 */
#define MOE_GEMM_KERNEL_AUTO 0
#define MOE_GEMM_KERNEL_SINGLE 1
#define MOE_GEMM_KERNEL_PAIR 2
int moe_debug_set_gemm_kernel(int which);
unsigned long long moe_debug_set_wait_limit_ns(unsigned long long ns);

/*
 * moe_debug_grouped_gemm_after: moe_w4a16_grouped_gemm as the consumer side of the forward's GEMM
 * overlap: expert e's A rows are read only once ready[e] >= rows_e * ready_need * 4 (the count a
 * producer GEMM's epilogue warps publish as they store those rows; ready device int32 [E]).  For
 * the failure-path tests: counters that never reach the count make the wait run out, and the
 * kernel returns with MOE_DEVERR_TIMEOUT after the wait bound.  Other arguments as
 * moe_w4a16_grouped_gemm; MOE_ERR_INVALID_ARG for a NULL ready or ready_need < 1.
 */
int moe_debug_grouped_gemm_after(const uint16_t* A, int a_rows, int lda, const int32_t* gather_ids,
                                 const moe_expert_table* W, const int32_t* expert_offsets, int R, void* C, int ldc,
                                 int c_dtype, const int32_t* ready, int ready_need, void* stream);

/* ---------------------------------------------------------------- errors */
/*
 * Synchronises `stream`, returns the sticky device error word of the current device in
 * *code (MOE_DEVERR_*) and clears it.  Returns MOE_ERR_DEVICE when *code != 0.
 * For tests and debugging: it blocks the host.
 */
int moe_get_device_error(void* stream, int* code);

/* Human-readable name of a moe_status. */
const char* moe_status_string(int status);

/* Library version string. */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_PREFILL_H */
