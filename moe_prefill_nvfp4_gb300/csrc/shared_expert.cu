// shared_expert.cu -- the shared expert: a dense BF16 SwiGLU MLP over every row of the chunk
// ("glm5next_mlp/forward.rs" (spark), forward_dense):
//   gate = x W_gate^T, up = x W_up^T      one dense tensor-core launch (dense_gemm.cu) writing
//                                         gate | up into one [T, 2I] BF16 buffer
//   act  = silu(min(gate, L)) * clamp(up, -L, L)   the SwiGLU kernel of small_kernels.cu
//   shared_out = act W_down^T             a second dense tensor-core launch
// FP32 accumulation, BF16 at every stage boundary.  Its output joins the routed sum in the
// combine ("glm5next_mlp/forward.rs" (metrale), forward_moe).

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t shared_expert_ws_layout(int T, int I, size_t* off_gu, size_t* off_act) {
  size_t o = 0;
  *off_gu = o;
  o = align256(o + (size_t)T * 2 * I * 2);
  *off_act = o;
  return align256(o + (size_t)T * I * 2);
}

int shared_expert_launch(const uint16_t* x, int T, int H, int I, const uint16_t* w_gate, const uint16_t* w_up,
                         const uint16_t* w_down, float limit, void* ws, uint16_t* shared_out, cudaStream_t st) {
  size_t o_gu, o_act;
  shared_expert_ws_layout(T, I, &o_gu, &o_act);
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint16_t* gu = reinterpret_cast<uint16_t*>(base + o_gu);  // [T, 2I]: gate | up
  uint16_t* act = reinterpret_cast<uint16_t*>(base + o_act);
  DenseGemm g = {};
  g.B = x;
  g.T = T;
  g.K = H;
  g.ldb = H;
  g.nseg = 2;
  g.W[0] = w_gate;
  g.W[1] = w_up;
  g.rows[0] = g.rows[1] = I;
  g.ldw[0] = g.ldw[1] = H;
  g.col[0] = 0;
  g.col[1] = I;
  g.C = gu;
  g.ldc = 2 * I;
  int rc = dense_gemm_launch(g, st);
  if (rc == MOE_OK) rc = swiglu_launch(gu, gu + I, T, I, 2 * I, act, I, limit, st);
  if (rc != MOE_OK) return rc;
  DenseGemm d = {};
  d.B = act;
  d.T = T;
  d.K = I;
  d.ldb = I;
  d.nseg = 1;
  d.W[0] = w_down;
  d.rows[0] = H;
  d.ldw[0] = I;
  d.col[0] = 0;
  d.C = shared_out;
  d.ldc = H;
  return dense_gemm_launch(d, st);
}

}  // namespace moe
