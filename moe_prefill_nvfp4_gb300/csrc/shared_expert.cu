// shared_expert.cu -- the shared expert: a dense BF16 SwiGLU MLP over every row of the chunk
// ("glm5next_mlp/forward.rs" (spark), forward_dense):
//   gate = x W_gate^T, up = x W_up^T      plain BF16 GEMMs (cuBLAS, FP32 accumulation, BF16 out)
//   act  = silu(min(gate, L)) * clamp(up, -L, L)   the SwiGLU kernel of small_kernels.cu
//   shared_out = act W_down^T             plain BF16 GEMM (cuBLAS)
// Its output joins the routed sum in the combine ("glm5next_mlp/forward.rs" (metrale),
// forward_moe).  The three products are ordinary dense GEMMs with no dequantisation, gather or
// fused epilogue, so they go to the library.

#include <cublas_v2.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kMaxDev = 64;
std::mutex g_blas_mu;
cublasHandle_t g_blas[kMaxDev] = {nullptr};

// Row-major C[M, N] = A[M, K] * B[N, K]^T, all BF16, FP32 accumulation: the column-major
// product C^T = B * A^T, B read transposed.
int gemm_bf16_nt(cublasHandle_t h, const uint16_t* A, int lda, const uint16_t* B, int ldb, uint16_t* C, int ldc,
                 int M, int N, int K) {
  const float one = 1.0f, zero = 0.0f;
  const cublasStatus_t s = cublasGemmEx(h, CUBLAS_OP_T, CUBLAS_OP_N, N, M, K, &one, B, CUDA_R_16BF, ldb, A, CUDA_R_16BF,
                                        lda, &zero, C, CUDA_R_16BF, ldc, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
  return s == CUBLAS_STATUS_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t shared_expert_ws_layout(int T, int I, size_t* off_gu, size_t* off_act, size_t* off_blas) {
  size_t o = 0;
  *off_gu = o;
  o = align256(o + (size_t)T * 2 * I * 2);
  *off_act = o;
  o = align256(o + (size_t)T * I * 2);
  *off_blas = o;
  return o + kSharedExpertBlasWorkspace;
}

int shared_expert_launch(const uint16_t* x, int T, int H, int I, const uint16_t* w_gate, const uint16_t* w_up,
                         const uint16_t* w_down, float limit, void* ws, uint16_t* shared_out, cudaStream_t st) {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDev) return MOE_ERR_CUDA;
  size_t o_gu, o_act, o_blas;
  shared_expert_ws_layout(T, I, &o_gu, &o_act, &o_blas);
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint16_t* gu = reinterpret_cast<uint16_t*>(base + o_gu);  // [T, 2I]: gate | up
  uint16_t* act = reinterpret_cast<uint16_t*>(base + o_act);
  // one handle per device; its stream and workspace are set per call, under the lock, so
  // concurrent callers cannot interleave their settings with the enqueued GEMMs
  std::lock_guard<std::mutex> lk(g_blas_mu);
  if (g_blas[d] == nullptr && cublasCreate(&g_blas[d]) != CUBLAS_STATUS_SUCCESS) {
    g_blas[d] = nullptr;
    return MOE_ERR_CUDA;
  }
  cublasHandle_t h = g_blas[d];
  if (cublasSetStream(h, st) != CUBLAS_STATUS_SUCCESS) return MOE_ERR_CUDA;
  if (cublasSetWorkspace(h, base + o_blas, kSharedExpertBlasWorkspace) != CUBLAS_STATUS_SUCCESS) return MOE_ERR_CUDA;
  int rc = gemm_bf16_nt(h, x, H, w_gate, H, gu, 2 * I, T, I, H);
  if (rc == MOE_OK) rc = gemm_bf16_nt(h, x, H, w_up, H, gu + I, 2 * I, T, I, H);
  if (rc == MOE_OK) rc = swiglu_launch(gu, gu + I, T, I, 2 * I, act, I, limit, st);
  if (rc == MOE_OK) rc = gemm_bf16_nt(h, act, I, w_down, I, shared_out, H, T, H, I);
  return rc;
}

}  // namespace moe
