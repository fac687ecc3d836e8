// internal.h -- declarations shared between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_prefill.h"

namespace moe {

// Arguments of the grouped W4A16 GEMM kernel (the activation tensor map is passed separately as
// a __grid_constant__ parameter).
struct GemmArgs {
  const CUtensorMap* wmaps;   // device [E][2]: packed [N, K/2] map, scales [N, K/16] map (128-row boxes)
  const CUtensorMap* wmaps64; // device [E][2]: the same maps with 64-row boxes (CTA-pair kernel)
  const void* A;              // activations (BF16, row stride lda elements); the pair kernel reads them directly
  int lda;
  uint64_t wait_ns;           // bound of every pipeline wait of the CTA-pair kernel
  const void* const* packed;  // device [E]: packed pointers (NULL = absent expert)
  const float* scale2;        // device [E]
  const int32_t* gather;      // device [R] or NULL (identity)
  const int32_t* offsets;     // device [E+1]
  void* C;
  int E, N, K, R, a_rows, ldc, c_dtype;
  int* err;                   // device error word
  // fused SwiGLU epilogue: 0 = plain GEMM (C is [R, N]); otherwise N = 2 * swiglu_half, the
  // CTA pairs gate block j (weight rows j*128..) with up block j (rows swiglu_half + j*128..)
  // and C is the BF16 activation [R, swiglu_half]
  int swiglu_half;
  float limit;
  // Overlap of the two GEMMs of one forward (all NULL = off).  Producer: after its stores of a
  // tile each of the 4 epilogue warps adds the tile's row count to ready_out[expert]; after
  // zero-filling rows of an absent expert each adds their count times ready_need.  Consumer:
  // expert e's A rows are loaded only once ready_in[e] >= rows_e * ready_need * 4 (ready_need =
  // the producer's CTA tiles covering one row); its clusters take tiles dynamically from
  // *tile_counter (zero at launch), so the CTAs that start early, on SMs the producer has left,
  // take more tiles; it waits for the previous grid only at its end.
  int* ready_out;
  const int* ready_in;
  int ready_need;
  int* tile_counter;
  // widest thread-block cluster the single-CTA kernel may take (1: no multicast activation loads)
  int max_cluster;
  // Rows in expert order stored by the CTA-pair kernel itself (row_src NULL: A holds them
  // already).  Its epilogue warps store A[p, :] = row_src[row_ids[p], :] (row stride row_src_ld)
  // for the sorted rows p of present experts while they have no accumulator to drain, and add 1
  // to rows_ready[e] (zero at launch) per stored row of expert e; the B producer loads expert e's
  // rows once rows_ready[e] reaches its row count.  A token id outside [0, row_src_rows) records
  // MOE_DEVERR_BAD_GATHER and stores token row 0.
  const uint16_t* row_src;
  int row_src_rows, row_src_ld;
  const int32_t* row_ids;
  int* rows_ready;
};

// Host: encode a tiled tensor map through the driver entry point (no libcuda link needed).
int encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, void* base, const cuuint64_t* dims,
                const cuuint64_t* strides_bytes, const cuuint32_t* box, const cuuint32_t* elem_strides,
                CUtensorMapSwizzle swizzle);
int device_sm_count();
int* device_error_word();  // device address of the current device's error word

int grouped_gemm_launch(const GemmArgs& args, const void* A, int a_rows, int lda, cudaStream_t stream);
// The CTA-pair kernel (pair_gemm.cu): N a multiple of 256 (gate/up with the fused SwiGLU: N = 2I,
// I a multiple of 128), K a multiple of 256, 64-row weight maps present.
bool pair_gemm_supported(const GemmArgs& args);
bool pair_gemm_shape_ok(int N, int K, int E, int swiglu_half);
// whether the automatic choice takes the pair kernel for R sorted rows over E experts
bool pair_gemm_preferred(int R, int E);
// epilogue warpgroups of the pair kernel config the launch takes (each of their warps publishes
// a tile's rows to the forward's GEMM overlap)
int pair_gemm_epilogue_groups(const GemmArgs& args);
// x in host memory, read by the device's own loads: stage_rows copies x [T, H] into dst;
// scatter_rows stores each token row to its k sorted positions xs[token_to_perm[t, s]] (rows of
// unused slots, position -1, are not written); k <= 32
int stage_rows_launch(const uint16_t* x, int T, int H, uint16_t* dst, cudaStream_t st);
int scatter_rows_launch(const uint16_t* x, int T, int H, const int32_t* token_to_perm, int k, int R, uint16_t* xs,
                        cudaStream_t st);
int pair_gemm_launch(const GemmArgs& args, cudaStream_t stream);
// Bound of the pipeline waits of the GEMM kernels (2 s; a debug entry point may lower it).
uint64_t gemm_wait_limit_ns();

// Launch with programmatic stream serialization (the kernel calls griddep_wait() before it reads
// what earlier work in the stream wrote).
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ... with thread-block clusters of cluster_x CTAs along x (grid.x a multiple of cluster_x)
template <typename... KArgs, typename... Args>
int launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster_x,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// small-row products (small_rows.cu): at most 8 rows per expert, FP32 weights, BF16 out
struct SmallRowsArgs {
  const uint16_t* A;
  int lda, a_rows;
  const int32_t* gather;      // [R] or NULL (identity)
  const void* const* packed;  // device [E]
  const void* const* scales;  // device [E]
  const float* scale2;        // device [E]
  const int32_t* offsets;     // [E+1]
  int E, N, K, R;
  int swiglu_half;            // 0: C = A W^T [R, N]; I: gate/up pair -> SwiGLU act [R, I]
  float limit;
  uint16_t* C;
  int ldc;
  int* err;
};
int small_rows_launch(const SmallRowsArgs& a, cudaStream_t st);

// Dense BF16 GEMM on the tensor cores (dense_gemm.cu): for each weight segment s < nseg,
// C[t, col[s] + n] = sum_k B[t, k] W[s][n, k] (t < T, n < rows[s], k < K), FP32 accumulation, BF16
// out.  B [T, K] with row stride ldb, W[s] [rows[s], K] with row stride ldw[s], C row stride ldc
// (elements); K, strides, rows and col multiples of 8, pointers 16-byte aligned.
struct DenseGemm {
  const uint16_t* B;
  int T, K, ldb;
  int nseg;
  const uint16_t* W[2];
  int rows[2], ldw[2], col[2];
  uint16_t* C;
  int ldc;
};
int dense_gemm_launch(const DenseGemm& d, cudaStream_t stream);
// token-tile width the launch takes for T tokens over weight_tiles tiles of 128 weight rows
int dense_gemm_token_tile(int T, int weight_tiles, int nsm);

// shared expert (shared_expert.cu): workspace = gate|up [T, 2I] BF16 and act [T, I] BF16, each
// 256-byte aligned; returns the total bytes
size_t shared_expert_ws_layout(int T, int I, size_t* off_gu, size_t* off_act);
int shared_expert_launch(const uint16_t* x, int T, int H, int I, const uint16_t* w_gate, const uint16_t* w_up,
                         const uint16_t* w_down, float limit, void* ws, uint16_t* shared_out, cudaStream_t st);

// SIMT kernels (small_kernels.cu)
// Router logits (tensor-core MMAs, h split over a cluster of up to 8 CTAs per 16 rows).  x_copy:
// NULL, or a device BF16 [T, H] buffer that receives x as the kernel reads it (x in host memory).
int router_logits_launch(const uint16_t* x, const uint16_t* w, int T, int H, int E, float* logits, cudaStream_t st,
                         uint16_t* x_copy = nullptr);
// router logits + top-k in one launch (same results as router_logits_launch + route_topk_launch)
// when E <= 64; MOE_ERR_UNSUPPORTED_SHAPE otherwise
constexpr int kRouterTopkMaxE = 64;
int router_topk_launch(const uint16_t* x, const uint16_t* w, int T, int H, int E, const float* bias, int k,
                       int renormalize, float scale, float* logits, int32_t* ids, float* wts, int* err,
                       cudaStream_t st, uint16_t* x_copy = nullptr);
int route_topk_launch(const float* logits, const float* bias, int T, int E, int k, int renormalize, float scale,
                      int32_t* ids, float* wts, int* err, cudaStream_t st);
int sort_segments(int R, int E);
size_t sort_scratch_bytes(int R, int E);
// The stable sort: one block when R <= 2048 (cnt unused), else histogram + scatter kernels over
// segments of 2048 slots with the per-segment counts in cnt (sort_scratch_bytes).
// zero: NULL, or an INT32 array of zero_n elements the sort clears (the forward's overlap counters)
int sort_launch(const int32_t* ids, int R, int k, int E, int32_t* cnt, int32_t* sorted_token_ids,
                int32_t* sorted_expert_ids, int32_t* expert_offsets, int32_t* token_to_perm, int* err,
                cudaStream_t st, int32_t* zero = nullptr, int zero_n = 0);
int swiglu_launch(const uint16_t* gate, const uint16_t* up, int64_t rows, int64_t width, int64_t ld_in, uint16_t* out,
                  int64_t ld_out, float limit, cudaStream_t st);
int combine_launch(const uint16_t* Y, const int32_t* perm, const float* wts, const uint16_t* shared_out, int T, int k,
                   int H, uint16_t* out, cudaStream_t st);
int dequant_launch(const uint8_t* packed, const uint8_t* scales, float scale2, int N, int K, uint16_t* out,
                   cudaStream_t st);

}  // namespace moe
