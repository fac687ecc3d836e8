// small_rows.cu -- the grouped W4A16 products for chunks with at most 8 rows per expert (decode-
// like prefill chunks), without tensor cores: every weight element is used by so few rows that
// staging a dequantised BF16 tile for a 16-column MMA costs more than it saves.  Each warp
// streams one output row of an expert's packed weights (8-byte loads, lane-interleaved 16-k
// chunks, coalesced) and its E4M3 block scales, turns each 16-element chunk into exact FP32
// products E2M1 * E4M3, and accumulates FP32 FMAs with the expert's (<= 8) activation rows;
// scale2 multiplies the sums.  This is the arithmetic of the pages' decode GEMV, whose weights
// stay FP32 into the FMA ("Module forward_prefill_gemm", "What is NOT bit-identical", item 2)
// -- not BF16-rounded as in the tensor-core path.  The gate/up kernel holds the gate row j and
// the up row I + j of the same expert and applies the clamped SwiGLU to the two sums.

#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int SR_WARPS = 8;   // warps per block
constexpr int SR_MAXM = 8;    // rows of one expert held in registers
constexpr int SR_ROWS = 2;    // weight rows per warp (gate/up: one gate row and its up row)

// 32 consecutive weights of one row: 16 packed bytes (low nibble = even k) and the two f16
// block scales (low and high half of scale_h) -> exact FP32 products E2M1 * E4M3.
MOE_DEV void dequant32_f32(uint4 pk, uint32_t scale_h, float (&w)[32]) {
  const uint32_t words[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t h[4];
    e2m1x8_to_f16x2(words[j], h);
    const uint32_t sc = j < 2 ? scale_h : scale_h >> 16;  // 16 weights per block scale
#pragma unroll
    for (int q = 0; q < 4; ++q) f16x2_times_f16(h[q], sc, w[8 * j + 2 * q], w[8 * j + 2 * q + 1]);
  }
}

// acc[mm] += sum_i w[i] * x[rows[mm], 32 c + i] for the expert's M rows (the activation rows are
// few and L1-resident, so they are re-read for every weight row instead of held in registers)
template <int M>
MOE_DEV void fma_rows(const uint16_t* __restrict__ x, int lda, const int (&rows)[SR_MAXM], int c,
                      const float (&w)[32], float (&acc)[M]) {
#pragma unroll
  for (int mm = 0; mm < M; ++mm) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)rows[mm] * lda + c * 32);
    float a = acc[mm];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = __ldg(xr + q);
      const uint32_t xa[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a = fmaf(w[8 * q + 2 * i], bf16_lo(xa[i]), a);
        a = fmaf(w[8 * q + 2 * i + 1], bf16_hi(xa[i]), a);
      }
    }
    acc[mm] = a;
  }
}

MOE_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The expert's rows [p0, p0 + m): lane i < m returns the A row of row i (gathered or identity),
// checked against a_rows.
MOE_DEV int expert_row_of_lane(const int32_t* gather, int p0, int m, int a_rows, int* err) {
  const int lane = threadIdx.x & 31;
  int src = 0;
  if (lane < m) {
    src = gather ? gather[p0 + lane] : p0 + lane;
    if ((unsigned)src >= (unsigned)a_rows) {
      set_error(err, MOE_DEVERR_BAD_GATHER);
      src = 0;
    }
  }
  return src;
}

// One work item: this warp's weight rows of expert e (gate row and up row of column n0 with
// SWIGLU, else rows n0 .. n0 + SR_ROWS - 1) times the expert's M activation rows.
template <bool SWIGLU, int M>
MOE_DEV void small_rows_item(const uint16_t* __restrict__ x, int lda, const int (&rows)[SR_MAXM], const void* packed,
                             const void* scales, float s2, int p0, int n0, int n_out, int half, int K, float L,
                             uint16_t* __restrict__ C, int ldc) {
  constexpr int NR = SR_ROWS;                    // weight rows held per warp
  constexpr int NOUT = SWIGLU ? 1 : SR_ROWS;     // output columns per warp
  const int lane = threadIdx.x & 31;
  const uint8_t* pw[NR];
  const uint8_t* sw[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const int o = min(n0 + (SWIGLU ? 0 : r), n_out - 1);
    const int row = SWIGLU && r == 1 ? half + o : o;
    pw[r] = static_cast<const uint8_t*>(packed) + (size_t)row * (K / 2);
    sw[r] = static_cast<const uint8_t*>(scales) + (size_t)row * (K / 16);
  }
  float acc[NR][M];
#pragma unroll
  for (int r = 0; r < NR; ++r)
#pragma unroll
    for (int mm = 0; mm < M; ++mm) acc[r][mm] = 0.f;
  for (int c = lane; c < K / 32; c += 32) {
    uint4 pk[NR];
    uint16_t sc2[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {  // every row's loads first: NR requests in flight per lane
      pk[r] = __ldg(reinterpret_cast<const uint4*>(pw[r] + c * 16));
      sc2[r] = __ldg(reinterpret_cast<const uint16_t*>(sw[r] + c * 2));
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      uint32_t sh, unused;
      e4m3x4_to_f16x2(sc2[r], sh, unused);
      float w[32];
      dequant32_f32(pk[r], sh, w);
      fma_rows<M>(x, lda, rows, c, w, acc[r]);
    }
  }
#pragma unroll
  for (int mm = 0; mm < M; ++mm) {
#pragma unroll
    for (int o = 0; o < NOUT; ++o) {
      float v;
      if (SWIGLU) {
        v = swiglu_clamped(warp_sum(acc[0][mm]) * s2, warp_sum(acc[1][mm]) * s2, L);
      } else {
        v = warp_sum(acc[o][mm]) * s2;
      }
      if (lane == mm && n0 + o < n_out) C[(size_t)(p0 + mm) * ldc + n0 + o] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
  }
}

// Persistent kernel: work item = (expert e, SR_ROWS output rows of one warp); warps walk the
// items with a grid stride, skipping experts without rows.  SWIGLU: the warp's output rows are
// activation columns j, each built from gate row j and up row half + j.
template <bool SWIGLU>
__global__ void __launch_bounds__(SR_WARPS * 32, 2)
    small_rows_kernel(const uint16_t* __restrict__ x, int lda, int a_rows, const int32_t* __restrict__ gather,
                      const void* const* __restrict__ packed, const void* const* __restrict__ scales,
                      const float* __restrict__ scale2, const int32_t* __restrict__ offsets, int E, int n_out,
                      int half, int K, float L, uint16_t* __restrict__ C, int ldc, int R, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int NOUT = SWIGLU ? 1 : SR_ROWS;  // output columns per warp
  const int lane = threadIdx.x & 31;
  const int groups = (n_out + NOUT - 1) / NOUT;
  const long long items = (long long)E * groups;
  const long long nwarps = (long long)gridDim.x * SR_WARPS;
  for (long long it = blockIdx.x * SR_WARPS + (threadIdx.x >> 5); it < items; it += nwarps) {
    const int e = (int)(it / groups);
    const int n0 = (int)(it - (long long)e * groups) * NOUT;
    const int p0 = offsets[e];
    const int m = offsets[e + 1] - p0;
    if (m <= 0) continue;
    if (p0 < 0 || p0 + m > R) {
      if (lane == 0 && n0 == 0) set_error(err, MOE_DEVERR_BAD_OFFSETS);
      continue;
    }
    if (m > SR_MAXM) {
      if (lane == 0 && n0 == 0) set_error(err, MOE_DEVERR_SMALL_ROWS);
      continue;
    }
    if (packed[e] == nullptr) {  // absent expert: its rows are zero
      for (int o = 0; o < NOUT; ++o)
        if (lane < m && n0 + o < n_out) C[(size_t)(p0 + lane) * ldc + n0 + o] = 0;
      continue;
    }
    const int src = expert_row_of_lane(gather, p0, m, a_rows, err);
    // at most 4 rows in registers: an expert with 5..8 rows is done in two batches
    for (int b0 = 0; b0 < m; b0 += 4) {
      const int mb = min(4, m - b0);
      int rsub[SR_MAXM];
#pragma unroll
      for (int i = 0; i < SR_MAXM; ++i) rsub[i] = __shfl_sync(0xffffffffu, src, min(b0 + i, 31));
      switch (mb) {
        case 1: small_rows_item<SWIGLU, 1>(x, lda, rsub, packed[e], scales[e], scale2[e], p0 + b0, n0, n_out, half, K, L, C, ldc); break;
        case 2: small_rows_item<SWIGLU, 2>(x, lda, rsub, packed[e], scales[e], scale2[e], p0 + b0, n0, n_out, half, K, L, C, ldc); break;
        case 3: small_rows_item<SWIGLU, 3>(x, lda, rsub, packed[e], scales[e], scale2[e], p0 + b0, n0, n_out, half, K, L, C, ldc); break;
        default: small_rows_item<SWIGLU, 4>(x, lda, rsub, packed[e], scales[e], scale2[e], p0 + b0, n0, n_out, half, K, L, C, ldc); break;
      }
    }
  }
}

int small_rows_launch(const SmallRowsArgs& a, cudaStream_t st) {
  const int nsm = device_sm_count();
  if (nsm <= 0) return MOE_ERR_CUDA;
  const dim3 grid(nsm * 2), block(SR_WARPS * 32);  // two resident blocks per SM
  if (a.swiglu_half)
    return launch_pdl(small_rows_kernel<true>, grid, block, 0, st, a.A, a.lda, a.a_rows, a.gather, a.packed, a.scales,
                      a.scale2, a.offsets, a.E, a.swiglu_half, a.swiglu_half, a.K, a.limit, a.C, a.ldc, a.R, a.err);
  return launch_pdl(small_rows_kernel<false>, grid, block, 0, st, a.A, a.lda, a.a_rows, a.gather, a.packed, a.scales,
                    a.scale2, a.offsets, a.E, a.N, 0, a.K, 0.f, a.C, a.ldc, a.R, a.err);
}

}  // namespace moe
