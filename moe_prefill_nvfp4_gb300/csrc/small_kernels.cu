// small_kernels.cu -- the bandwidth/latency-bound steps around the two grouped GEMMs:
// router logits, top-k routing, the stable expert sort, the clamped SwiGLU, the indexed
// combine, and a standalone NVFP4 -> BF16 dequantisation (same device routine as the GEMM).
//
// Each is one launch over all rows (the pages measured per-row launches of top-k and combine
// as pure launch overhead: "glm5next_mlp/forward.rs", forward_moe comments), with 16-byte
// vector loads/stores on the row-major BF16 tensors, the router's dense contraction on the
// tensor cores (warp-level MMAs), and warp-level primitives (reductions, ballot, shuffles) for
// selection, counting and the per-expert prefix.

#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

// ------------------------------------------------------------------------------------------------
// router logits: logits[t, e] = sum_h x[t, h] * w[e, h]  (BF16 in, FP32 accumulate and out)
//
// A cluster of `cl` CTAs owns a 16-token x 64-expert tile and its 8 * cl warps split h into
// 32-element super-steps (warp gw of the cluster takes super-steps gw, gw + 8 cl, ...).  Per
// super-step a warp runs two BF16 tensor-core MMAs (m16n8k16, FP32 accumulate) on each of the
// tile's eight 8-expert column groups.  The order of k inside an MMA is free as long as x and w
// use the same one: lane (g, q) loads one 16-byte vector (8 consecutive h) of token rows g and
// g + 8 and of expert row g of each column group; its elements 0-3 are that lane's k pairs
// {2q, 2q+1} and {2q+8, 2q+9} of the first MMA, elements 4-7 those of the second.  The partial
// tiles are added over the CTA's warps (through shared memory, in warp order) and over the
// cluster's CTAs: CTA r owns rows r * 16/cl .. of the tile, every CTA sends its partial of those
// rows into CTA r's shared memory, and CTA r adds them in rank order.  The summation order
// depends on H alone, so the standalone router and the fused router + top-k give the same bits.

constexpr int RT_TOK = 16, RT_EXP = 64, RT_WARPS = 8;

// Split of h over the cluster: as wide as 8 CTAs while every warp still gets a super-step.
static int router_cluster(int H) {
  const int ns = (H + 31) / 32;
  int cl = 8;
  while (cl > 1 && cl * RT_WARPS > ns) cl >>= 1;
  return cl;
}

// D += A * B for one m16n8k16 tile: A row-major 16 x 16 BF16 (a0: row g, k 2q..2q+1; a1: row
// g + 8; a2, a3: the same at k + 8), B 16 x 8 BF16 (b0: k 2q..2q+1 of column g; b1: k + 8),
// D 16 x 8 FP32 (d0, d1: row g, columns 2q, 2q + 1; d2, d3: row g + 8).
MOE_DEV void mma_bf16_m16n8k16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                               uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

struct RouterSmem {
  float red[RT_WARPS][RT_TOK][RT_EXP];  // each warp's partial tile
  float part[RT_TOK * RT_EXP];          // [sender rank][owned row][expert]: partials of this CTA's rows
  float rows[RT_TOK][RT_EXP];           // this CTA's finished rows (the top-k's input)
};

// The logits of the rows CTA `rank` owns (tile rows rank * 16/cl ..), left in s.rows[0 .. 16/cl)
// and written to `logits`.  Every thread of every CTA of the cluster calls it.  x_copy (NULL, or
// device BF16 [T, H]): the first 64-expert tile's clusters store every x vector they load there
// (each vector of x is loaded by exactly one lane of them), staging an x held in host memory.
MOE_DEV void router_cluster_tile(const uint16_t* __restrict__ x, const uint16_t* __restrict__ w, int T, int H, int E,
                                 int t0, int e0, int cl, int rank, RouterSmem& s, float* __restrict__ logits,
                                 uint16_t* __restrict__ x_copy) {
  // this CTA has started: the matching wait below precedes the first store into another CTA
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  float acc[RT_EXP / 8][4];
#pragma unroll
  for (int j = 0; j < RT_EXP / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  const int ns = (H + 31) / 32;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  for (int st = rank * RT_WARPS + warp; st < ns; st += cl * RT_WARPS) {
    const int h = st * 32 + q * 8;
    const bool hv = h < H;  // H % 8 == 0: a vector is wholly inside or wholly outside
    const uint4 xa = (hv && t0 + g < T) ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + g) * H + h)) : zero;
    const uint4 xb =
        (hv && t0 + g + 8 < T) ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + g + 8) * H + h)) : zero;
    uint4 wv[RT_EXP / 8];
#pragma unroll
    for (int j = 0; j < RT_EXP / 8; ++j)
      wv[j] = (hv && e0 + 8 * j + g < E) ? __ldg(reinterpret_cast<const uint4*>(w + (size_t)(e0 + 8 * j + g) * H + h))
                                         : zero;
    if (x_copy != nullptr && e0 == 0 && hv) {
      if (t0 + g < T) *reinterpret_cast<uint4*>(x_copy + (size_t)(t0 + g) * H + h) = xa;
      if (t0 + g + 8 < T) *reinterpret_cast<uint4*>(x_copy + (size_t)(t0 + g + 8) * H + h) = xb;
    }
#pragma unroll
    for (int j = 0; j < RT_EXP / 8; ++j) {
      mma_bf16_m16n8k16(acc[j], xa.x, xb.x, xa.y, xb.y, wv[j].x, wv[j].y);
      mma_bf16_m16n8k16(acc[j], xa.z, xb.z, xa.w, xb.w, wv[j].z, wv[j].w);
    }
  }
#pragma unroll
  for (int j = 0; j < RT_EXP / 8; ++j) {
    *reinterpret_cast<float2*>(&s.red[warp][g][8 * j + 2 * q]) = make_float2(acc[j][0], acc[j][1]);
    *reinterpret_cast<float2*>(&s.red[warp][g + 8][8 * j + 2 * q]) = make_float2(acc[j][2], acc[j][3]);
  }
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every CTA of the cluster has started
  const int rows = RT_TOK / cl;
  for (int i = threadIdx.x; i < RT_TOK * RT_EXP; i += RT_WARPS * 32) {
    const int row = i / RT_EXP, col = i % RT_EXP;
    float v = s.red[0][row][col];
#pragma unroll
    for (int ww = 1; ww < RT_WARPS; ++ww) v += s.red[ww][row][col];
    st_shared_cluster_f32(smem_u32(&s.part[(rank * rows + row % rows) * RT_EXP + col]), row / rows, v);
  }
  cluster_sync_all();  // every CTA's partials of the rows it owns are in its shared memory
  for (int i = threadIdx.x; i < rows * RT_EXP; i += RT_WARPS * 32) {
    const int lr = i / RT_EXP, col = i % RT_EXP;
    float v = s.part[lr * RT_EXP + col];
    for (int r = 1; r < cl; ++r) v += s.part[(r * rows + lr) * RT_EXP + col];
    s.rows[lr][col] = v;
    const int t = t0 + rank * rows + lr, e = e0 + col;
    if (t < T && e < E) logits[(size_t)t * E + e] = v;
  }
}

// ------------------------------------------------------------------------------------------------
// top-k routing: one warp per row; lane l holds logits of experts l, l+32, ... in registers.

constexpr int TOPK_WARPS = 8;

// Order-preserving code of a selection key: a larger key gets a larger code, +0 and -0 the same
// one, and every key (-inf included) a code above 0, which marks "no candidate".
MOE_DEV uint32_t key_code(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp routes one row: top-k of (logit + bias) with ties to the lower expert index, weights
// from the unbiased logits (softmax over the k picks, or over all experts).  `lrow` may point to
// global or shared memory.  Shared by the standalone top-k kernel and the fused router + top-k
// kernel.
template <int NPL>
MOE_DEV void topk_row(const float* lrow, const float* __restrict__ bias, int E, int k, int renormalize,
                      float routed_scale, int32_t* __restrict__ ids_row, float* __restrict__ wts_row, int* err) {
  const int lane = threadIdx.x & 31;
  float val[NPL], key[NPL];
  bool nan_seen = false;
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = lane + 32 * j;
    val[j] = e < E ? lrow[e] : -INFINITY;
    key[j] = e < E ? (bias ? val[j] + bias[e] : val[j]) : -INFINITY;
    if (e < E && (isnan(val[j]) || isnan(key[j]))) {
      nan_seen = true;
      key[j] = -INFINITY;
    }
  }
  if (__any_sync(0xffffffffu, nan_seen) && lane == 0) set_error(err, MOE_DEVERR_NAN_LOGIT);
  // selection s: the largest remaining key, ties to the lower expert.  A lane's candidate is its
  // best remaining code (strict >: the lower j, i.e. the lower expert, on ties); the warp takes
  // the largest code, then the lowest expert among the lanes holding it.
  uint32_t code[NPL];
#pragma unroll
  for (int j = 0; j < NPL; ++j) code[j] = lane + 32 * j < E ? key_code(key[j]) : 0u;
  int my_id = -1;
  for (int s = 0; s < k; ++s) {
    uint32_t bc = 0u, be = 0x7fffffffu;
#pragma unroll
    for (int j = 0; j < NPL; ++j)
      if (code[j] > bc) {
        bc = code[j];
        be = lane + 32 * j;
      }
    const uint32_t mc = __reduce_max_sync(0xffffffffu, bc);
    const int pick = (int)__reduce_min_sync(0xffffffffu, bc == mc ? be : 0x7fffffffu);
#pragma unroll
    for (int j = 0; j < NPL; ++j)
      if (pick == lane + 32 * j) code[j] = 0u;
    if (lane == s) my_id = pick;
  }
  // routing weights from the unbiased logits
  const bool mine = lane < k;
  const float l = mine ? lrow[my_id] : -INFINITY;
  float w;
  if (renormalize) {
    float m = l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float ex = mine ? expf(l - m) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    w = ex / sum;
  } else {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < NPL; ++j) m = fmaxf(m, val[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < NPL; ++j)
      if (lane + 32 * j < E) sum += expf(val[j] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    w = mine ? expf(l - m) / sum : 0.f;
  }
  if (mine) {
    ids_row[lane] = my_id;
    wts_row[lane] = w * routed_scale;
  }
}

template <int NPL>
__global__ void __launch_bounds__(TOPK_WARPS * 32)
    route_topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E, int k,
                      int renormalize, float routed_scale, int32_t* __restrict__ ids, float* __restrict__ wts,
                      int* err) {
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int row = blockIdx.x * TOPK_WARPS + warp;
  if (row >= T) return;
  topk_row<NPL>(logits + (size_t)row * E, bias, E, k, renormalize, routed_scale, ids + (size_t)row * k,
                wts + (size_t)row * k, err);
}

int route_topk_launch(const float* logits, const float* bias, int T, int E, int k, int renormalize, float scale,
                      int32_t* ids, float* wts, int* err, cudaStream_t st) {
  const int grid = (T + TOPK_WARPS - 1) / TOPK_WARPS;
  const int npl = (E + 31) / 32;
#define MOE_TOPK_CASE(N)                                                                                  \
  launch_pdl(route_topk_kernel<N>, dim3(grid), dim3(TOPK_WARPS * 32), 0, st, logits, bias, T, E, k, renormalize, \
             scale, ids, wts, err)
  if (npl <= 1) return MOE_TOPK_CASE(1);
  if (npl <= 2) return MOE_TOPK_CASE(2);
  if (npl <= 4) return MOE_TOPK_CASE(4);
  if (npl <= 8) return MOE_TOPK_CASE(8);
  if (npl <= 16) return MOE_TOPK_CASE(16);
  return MOE_TOPK_CASE(32);
#undef MOE_TOPK_CASE
}

// ------------------------------------------------------------------------------------------------
// router kernels.  TOPK = false: the standalone router (any E, 64-expert tiles along grid z).
// TOPK = true: router logits + top-k in one launch (the forward's routing when it owns the router
// GEMM and E <= 64): after the cluster reduction each CTA routes the rows it owns, one warp per
// row, with the standalone top-k routine.  Same bits as the two separate launches, one launch and
// one HBM round trip of the logits fewer.

template <bool TOPK, int NPL>
__global__ void __launch_bounds__(RT_WARPS * 32)
    router_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ w, int T, int H, int E,
                  const float* __restrict__ bias, int k, int renormalize, float routed_scale,
                  float* __restrict__ logits, int32_t* __restrict__ ids, float* __restrict__ wts, int* err,
                  uint16_t* __restrict__ x_copy) {
  __shared__ __align__(16) RouterSmem s;
  griddep_wait();
  griddep_launch_dependents();
  const int cl = gridDim.x, rank = blockIdx.x;  // the cluster spans grid x
  const int t0 = blockIdx.y * RT_TOK, e0 = blockIdx.z * RT_EXP;
  router_cluster_tile(x, w, T, H, E, t0, e0, cl, rank, s, logits, x_copy);
  if constexpr (TOPK) {
    __syncthreads();
    const int rows = RT_TOK / cl;
    for (int lr = threadIdx.x >> 5; lr < rows; lr += RT_WARPS) {
      const int t = t0 + rank * rows + lr;
      if (t < T)
        topk_row<NPL>(s.rows[lr], bias, E, k, renormalize, routed_scale, ids + (size_t)t * k, wts + (size_t)t * k,
                      err);
    }
  }
}

int router_logits_launch(const uint16_t* x, const uint16_t* w, int T, int H, int E, float* logits, cudaStream_t st,
                         uint16_t* x_copy) {
  const int cl = router_cluster(H);
  const dim3 grid(cl, (T + RT_TOK - 1) / RT_TOK, (E + RT_EXP - 1) / RT_EXP);
  return launch_pdl_cluster(router_kernel<false, 1>, grid, dim3(RT_WARPS * 32), 0, st, cl, x, w, T, H, E, nullptr, 0,
                            0, 0.f, logits, nullptr, nullptr, nullptr, x_copy);
}

int router_topk_launch(const uint16_t* x, const uint16_t* w, int T, int H, int E, const float* bias, int k,
                       int renormalize, float scale, float* logits, int32_t* ids, float* wts, int* err,
                       cudaStream_t st, uint16_t* x_copy) {
  if (E > kRouterTopkMaxE) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int cl = router_cluster(H);
  const dim3 grid(cl, (T + RT_TOK - 1) / RT_TOK, 1);
  if (E <= 32)
    return launch_pdl_cluster(router_kernel<true, 1>, grid, dim3(RT_WARPS * 32), 0, st, cl, x, w, T, H, E, bias, k,
                              renormalize, scale, logits, ids, wts, err, x_copy);
  return launch_pdl_cluster(router_kernel<true, 2>, grid, dim3(RT_WARPS * 32), 0, st, cl, x, w, T, H, E, bias, k,
                            renormalize, scale, logits, ids, wts, err, x_copy);
}

// ------------------------------------------------------------------------------------------------
// stable expert sort.  The R slots are cut into segments of SORT_SEG; bucket b is expert b, or
// the tail b = E for -1 / invalid ids.
//   hist:    one block per segment counts its slots per bucket in shared memory -> cnt[b*S + seg]
//   scatter: one block per segment; the sorted position of a slot is
//              (slots of all buckets < b) + (slots of bucket b in earlier segments)
//              + (slots of bucket b earlier in this segment),
//            the last term from the lanes with the same bucket (ballots over the bucket's bits)
//            inside 32-slot chunks plus per-warp running counts, which keeps flat slot order (a
//            stable sort).  Block 0 writes expert_offsets.

constexpr int SORT_SEG = 2048;
constexpr int SORT_THREADS = 256;
constexpr int SORT_WARPS = SORT_THREADS / 32;
constexpr int SORT_PER_WARP = SORT_SEG / SORT_WARPS;

int sort_segments(int R, int E) {
  (void)E;
  return std::max(1, (R + SORT_SEG - 1) / SORT_SEG);
}

size_t sort_scratch_bytes(int R, int E) { return (size_t)(E + 1) * sort_segments(R, E) * sizeof(int32_t); }

MOE_DEV int bucket_of(int id, int E) { return (id >= 0 && id < E) ? id : E; }

// Lanes of the warp whose key equals this lane's (0 <= key < 2^nbits): the AND over the key's
// bits of the ballot of that bit (or of its complement where the bit is clear).  nbits
// independent ballots take the place of a warp match, which is slow.
MOE_DEV uint32_t same_key_lanes(int key, int nbits) {
  uint32_t m = 0xffffffffu;
  for (int i = 0; i < nbits; ++i) {
    const bool bit = (key >> i) & 1;
    const uint32_t bal = __ballot_sync(0xffffffffu, bit);
    m &= bit ? bal : ~bal;
  }
  return m;
}

__global__ void __launch_bounds__(SORT_THREADS)
    sort_hist_kernel(const int32_t* __restrict__ ids, int R, int E, int S, int32_t* __restrict__ cnt, int* err) {
  extern __shared__ int s_hist[];
  griddep_wait();
  griddep_launch_dependents();
  const int seg = blockIdx.x;
  for (int b = threadIdx.x; b <= E; b += SORT_THREADS) s_hist[b] = 0;
  __syncthreads();
  const int lo = seg * SORT_SEG, hi = min(R, lo + SORT_SEG);
  bool bad = false;
  for (int i = lo + threadIdx.x; i < hi; i += SORT_THREADS) {
    const int id = ids[i];
    if (id < -1 || id >= E) bad = true;
    atomicAdd(&s_hist[bucket_of(id, E)], 1);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) set_error(err, MOE_DEVERR_BAD_EXPERT_ID);
  for (int b = threadIdx.x; b <= E; b += SORT_THREADS) cnt[b * S + seg] = s_hist[b];
}

__global__ void __launch_bounds__(SORT_THREADS)
    sort_scatter_kernel(const int32_t* __restrict__ ids, int R, int k, int E, int S, const int32_t* __restrict__ cnt,
                        int32_t* __restrict__ sorted_token_ids, int32_t* __restrict__ sorted_expert_ids,
                        int32_t* __restrict__ expert_offsets, int32_t* __restrict__ token_to_perm,
                        int32_t* __restrict__ zero, int zero_n) {
  extern __shared__ int s_mem[];
  griddep_wait();
  griddep_launch_dependents();
  const int NB = E + 1;
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < zero_n; i += SORT_THREADS) zero[i] = 0;
  int* s_base = s_mem;                                              // [NB]
  int16_t* s_wcnt = reinterpret_cast<int16_t*>(s_base + NB);        // [SORT_WARPS][NB]
  int16_t* s_lpos = s_wcnt + SORT_WARPS * NB;                       // [SORT_SEG]
  int16_t* s_bkt = s_lpos + SORT_SEG;                               // [SORT_SEG]
  const int seg = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // this lane's slots, loaded first so their latency overlaps the bucket prefix below
  const int lo = seg * SORT_SEG, hi = min(R, lo + SORT_SEG);
  int bk[SORT_PER_WARP / 32];
#pragma unroll
  for (int c = 0; c < SORT_PER_WARP / 32; ++c) {
    const int i = lo + warp * SORT_PER_WARP + c * 32 + lane;
    bk[c] = i < hi ? bucket_of(ids[i], E) : -1;
  }

  // (1) total slots per bucket over all segments
  for (int b = tid; b < NB; b += SORT_THREADS) {
    int tot = 0;
    for (int s = 0; s < S; ++s) tot += cnt[b * S + s];
    s_base[b] = tot;
  }
  __syncthreads();
  // exclusive prefix of the totals over buckets (warp 0: each lane a contiguous run)
  if (warp == 0) {
    const int per = (NB + 31) / 32;
    const int b0 = min(NB, lane * per), b1 = min(NB, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b) sum += s_base[b];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int b = b0; b < b1; ++b) {
      const int t = s_base[b];
      s_base[b] = run;
      if (seg == 0) expert_offsets[b] = run;  // b == E: number of valid slots
      run += t;
    }
  }
  __syncthreads();
  // ... plus this bucket's slots in the earlier segments
  for (int b = tid; b < NB; b += SORT_THREADS) {
    int own = 0;
    for (int s = 0; s < seg; ++s) own += cnt[b * S + s];
    s_base[b] += own;
  }
  for (int i = tid; i < SORT_WARPS * NB; i += SORT_THREADS) s_wcnt[i] = 0;
  __syncthreads();

  // (2) stable ranks inside the segment
  const uint32_t lt = (1u << lane) - 1u;
  const int nbits = 32 - __clz(E + 1);  // keys b + 1 lie in [0, E + 1]
  int16_t* wc = s_wcnt + warp * NB;
#pragma unroll
  for (int c = 0; c < SORT_PER_WARP; c += 32) {
    const int li = warp * SORT_PER_WARP + c + lane;  // slot index inside the segment
    const int b = bk[c / 32];
    const uint32_t peers = same_key_lanes(b + 1, nbits);  // b = -1 (no slot) -> key 0
    int local = 0;
    if (b >= 0) local = wc[b] + __popc(peers & lt);
    __syncwarp();
    if (b >= 0 && (__ffs(peers) - 1) == lane) wc[b] = (int16_t)(wc[b] + __popc(peers));
    __syncwarp();
    s_lpos[li] = (int16_t)local;
    s_bkt[li] = (int16_t)b;
  }
  __syncthreads();
  // (3) per bucket, exclusive prefix over the warps
  for (int b = tid; b < NB; b += SORT_THREADS) {
    int run = 0;
    for (int w = 0; w < SORT_WARPS; ++w) {
      const int t = s_wcnt[w * NB + b];
      s_wcnt[w * NB + b] = (int16_t)run;
      run += t;
    }
  }
  __syncthreads();
  // (4) write
  for (int li = tid; li < SORT_SEG; li += SORT_THREADS) {
    const int i = lo + li;
    if (i >= hi) break;
    const int b = s_bkt[li];
    const int w = li / SORT_PER_WARP;
    const int p = s_base[b] + s_wcnt[w * NB + b] + s_lpos[li];
    sorted_token_ids[p] = i / k;
    sorted_expert_ids[p] = b < E ? b : -1;
    token_to_perm[i] = b < E ? p : -1;
  }
}

// R <= SORT_SEG: one block does the whole sort (histogram, bucket prefix, stable ranks and the
// writes) with the counts in shared memory: no scratch, one launch.
__global__ void __launch_bounds__(SORT_THREADS)
    sort_single_kernel(const int32_t* __restrict__ ids, int R, int k, int E, int32_t* __restrict__ sorted_token_ids,
                       int32_t* __restrict__ sorted_expert_ids, int32_t* __restrict__ expert_offsets,
                       int32_t* __restrict__ token_to_perm, int32_t* __restrict__ zero, int zero_n, int* err) {
  extern __shared__ int s_mem[];
  griddep_wait();
  griddep_launch_dependents();
  const int NB = E + 1;
  for (int i = threadIdx.x; i < zero_n; i += SORT_THREADS) zero[i] = 0;
  int* s_base = s_mem;                                              // [NB]
  int16_t* s_wcnt = reinterpret_cast<int16_t*>(s_base + NB);        // [SORT_WARPS][NB]
  int16_t* s_lpos = s_wcnt + SORT_WARPS * NB;                       // [SORT_SEG]
  int16_t* s_bkt = s_lpos + SORT_SEG;                               // [SORT_SEG]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int bk[SORT_PER_WARP / 32];
  bool bad = false;
#pragma unroll
  for (int c = 0; c < SORT_PER_WARP / 32; ++c) {
    const int i = warp * SORT_PER_WARP + c * 32 + lane;
    const int id = i < R ? ids[i] : -1;
    if (i < R && (id < -1 || id >= E)) bad = true;
    bk[c] = i < R ? bucket_of(id, E) : -1;
  }
  for (int i = tid; i < SORT_WARPS * NB; i += SORT_THREADS) s_wcnt[i] = 0;
  if (__syncthreads_or(bad) && tid == 0) set_error(err, MOE_DEVERR_BAD_EXPERT_ID);
  // stable ranks inside each warp's run of slots, per-warp bucket counts
  const uint32_t lt = (1u << lane) - 1u;
  const int nbits = 32 - __clz(E + 1);  // keys b + 1 lie in [0, E + 1]
  int16_t* wc = s_wcnt + warp * NB;
#pragma unroll
  for (int c = 0; c < SORT_PER_WARP / 32; ++c) {
    const int li = warp * SORT_PER_WARP + c * 32 + lane;
    const int b = bk[c];
    const uint32_t peers = same_key_lanes(b + 1, nbits);  // b = -1 (no slot) -> key 0
    int local = 0;
    if (b >= 0) local = wc[b] + __popc(peers & lt);
    __syncwarp();
    if (b >= 0 && (__ffs(peers) - 1) == lane) wc[b] = (int16_t)(wc[b] + __popc(peers));
    __syncwarp();
    s_lpos[li] = (int16_t)local;
    s_bkt[li] = (int16_t)b;
  }
  __syncthreads();
  // per bucket: exclusive prefix over the warps, and the bucket total
  for (int b = tid; b < NB; b += SORT_THREADS) {
    int run = 0;
    for (int w = 0; w < SORT_WARPS; ++w) {
      const int t = s_wcnt[w * NB + b];
      s_wcnt[w * NB + b] = (int16_t)run;
      run += t;
    }
    s_base[b] = run;
  }
  __syncthreads();
  // exclusive prefix of the totals over buckets (warp 0: each lane a contiguous run)
  if (warp == 0) {
    const int per = (NB + 31) / 32;
    const int b0 = min(NB, lane * per), b1 = min(NB, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b) sum += s_base[b];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int b = b0; b < b1; ++b) {
      const int t = s_base[b];
      s_base[b] = run;
      expert_offsets[b] = run;  // b == E: number of valid slots
      run += t;
    }
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < SORT_SEG / SORT_THREADS; ++c) {
    const int i = tid + c * SORT_THREADS;
    if (i < R) {
      const int b = s_bkt[i];
      const int p = s_base[b] + s_wcnt[(i / SORT_PER_WARP) * NB + b] + s_lpos[i];
      sorted_token_ids[p] = i / k;
      sorted_expert_ids[p] = b < E ? b : -1;
      token_to_perm[i] = b < E ? p : -1;
    }
  }
}

static size_t scatter_smem(int E) {
  const int NB = E + 1;
  return (size_t)NB * 4 + (size_t)SORT_WARPS * NB * 2 + (size_t)SORT_SEG * 2 * 2;
}

int sort_launch(const int32_t* ids, int R, int k, int E, int32_t* cnt, int32_t* sorted_token_ids,
                int32_t* sorted_expert_ids, int32_t* expert_offsets, int32_t* token_to_perm, int* err,
                cudaStream_t st, int32_t* zero, int zero_n) {
  if (zero == nullptr) zero_n = 0;
  if (R <= SORT_SEG)
    return launch_pdl(sort_single_kernel, dim3(1), dim3(SORT_THREADS), scatter_smem(E), st, ids, R, k, E,
                      sorted_token_ids, sorted_expert_ids, expert_offsets, token_to_perm, zero, zero_n, err);
  const int S = sort_segments(R, E);
  const int rc = launch_pdl(sort_hist_kernel, dim3(S), dim3(SORT_THREADS), (E + 1) * sizeof(int), st, ids, R, E, S,
                            cnt, err);
  if (rc != MOE_OK) return rc;
  return launch_pdl(sort_scatter_kernel, dim3(S), dim3(SORT_THREADS), scatter_smem(E), st, ids, R, k, E, S, cnt,
                    sorted_token_ids, sorted_expert_ids, expert_offsets, token_to_perm, zero, zero_n);
}

// ------------------------------------------------------------------------------------------------
// clamped SwiGLU: out = silu(min(g, L)) * clamp(u, -L, L), 8 elements per thread

__global__ void swiglu_kernel(const uint16_t* __restrict__ gate, const uint16_t* __restrict__ up, int64_t rows,
                              int64_t width, int64_t ld_in, uint16_t* __restrict__ out, int64_t ld_out, float L) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t vpr = width / 8;
  const int64_t total = rows * vpr;
  for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < total; v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = v / vpr, c = (v - r * vpr) * 8;
    const uint4 g = *reinterpret_cast<const uint4*>(gate + r * ld_in + c);
    const uint4 u = *reinterpret_cast<const uint4*>(up + r * ld_in + c);
    const uint32_t ga[4] = {g.x, g.y, g.z, g.w}, ua[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = pack_bf16x2(swiglu_clamped(bf16_lo(ga[i]), bf16_lo(ua[i]), L),
                         swiglu_clamped(bf16_hi(ga[i]), bf16_hi(ua[i]), L));
    *reinterpret_cast<uint4*>(out + r * ld_out + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

int swiglu_launch(const uint16_t* gate, const uint16_t* up, int64_t rows, int64_t width, int64_t ld_in, uint16_t* out,
                  int64_t ld_out, float limit, cudaStream_t st) {
  const int64_t total = rows * (width / 8);
  if (total == 0) return MOE_OK;
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>((total + threads - 1) / threads, (int64_t)device_sm_count() * 16);
  return launch_pdl(swiglu_kernel, dim3((unsigned)blocks), dim3(threads), 0, st, gate, up, rows, width, ld_in, out,
                    ld_out, limit);
}

// ------------------------------------------------------------------------------------------------
// indexed combine: out[t] = sum_s wts[t, s] * Y[token_to_perm[t, s]] (+ shared_out[t]), slot order
//
// One thread per (token, 8-column vector).  The slots are taken 8 at a time with all 8 row loads
// issued before the FP32 accumulation, which stays in slot order (deterministic).

constexpr int CMB_THREADS = 256;
constexpr int CMB_BATCH = 8;

__global__ void __launch_bounds__(CMB_THREADS)
    combine_kernel(const uint16_t* __restrict__ Y, const int32_t* __restrict__ perm, const float* __restrict__ wts,
                   const uint16_t* __restrict__ shared_out, int T, int k, int H, uint16_t* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const int nvec = H / 8;
  const int64_t g = (int64_t)blockIdx.x * CMB_THREADS + threadIdx.x;
  if (g >= (int64_t)T * nvec) return;
  const int t = (int)(g / nvec), v = (int)(g - (int64_t)t * nvec);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int s0 = 0; s0 < k; s0 += CMB_BATCH) {
    uint4 y[CMB_BATCH];
    float w[CMB_BATCH];
#pragma unroll
    for (int j = 0; j < CMB_BATCH; ++j) {
      const int s = s0 + j;
      const int p = s < k ? __ldg(perm + (size_t)t * k + s) : -1;
      w[j] = s < k ? __ldg(wts + (size_t)t * k + s) : 0.f;
      y[j] = p >= 0 ? __ldg(reinterpret_cast<const uint4*>(Y + (size_t)p * H) + v) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < CMB_BATCH; ++j) {
      if (s0 + j >= k) break;
      const uint32_t ya[4] = {y[j].x, y[j].y, y[j].z, y[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(w[j], bf16_lo(ya[i]), acc[2 * i]);
        acc[2 * i + 1] = fmaf(w[j], bf16_hi(ya[i]), acc[2 * i + 1]);
      }
    }
  }
  if (shared_out) {
    const uint4 y = __ldg(reinterpret_cast<const uint4*>(shared_out + (size_t)t * H) + v);
    const uint32_t ya[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] += bf16_lo(ya[i]);
      acc[2 * i + 1] += bf16_hi(ya[i]);
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
  reinterpret_cast<uint4*>(out + (size_t)t * H)[v] = make_uint4(o[0], o[1], o[2], o[3]);
}

int combine_launch(const uint16_t* Y, const int32_t* perm, const float* wts, const uint16_t* shared_out, int T, int k,
                   int H, uint16_t* out, cudaStream_t st) {
  const int64_t total = (int64_t)T * (H / 8);
  return launch_pdl(combine_kernel, dim3((unsigned)((total + CMB_THREADS - 1) / CMB_THREADS)), dim3(CMB_THREADS), 0, st,
                    Y, perm, wts, shared_out, T, k, H, out);
}

// ------------------------------------------------------------------------------------------------
// x in host memory: the device reads it over the CPU-GPU link with its own loads (each thread
// four 16-byte loads in flight), which for tens of MB measured faster than a copy-engine copy.
//   stage_rows: x [T, H] -> dst [T, H] (the workspace's x_stage), any T, H % 8 == 0.
//   scatter_rows: each token row read once and stored to its k sorted positions
//     xs[token_to_perm[t, s]] (the CTA-pair gate/up GEMM's rows in expert order); slots whose
//     position is -1 (unused) store nothing.  One warp per token.

constexpr int STAGE_THREADS = 256;

__global__ void __launch_bounds__(STAGE_THREADS)
    stage_rows_kernel(const uint4* __restrict__ src, int64_t n, uint4* __restrict__ dst) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t stride = (int64_t)gridDim.x * STAGE_THREADS;
  int64_t i = blockIdx.x * (int64_t)STAGE_THREADS + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n; i += stride) dst[i] = src[i];
}

int stage_rows_launch(const uint16_t* x, int T, int H, uint16_t* dst, cudaStream_t st) {
  const int64_t n = (int64_t)T * H / 8;
  if (n == 0) return MOE_OK;
  const int nsm = device_sm_count();
  const int64_t blocks = std::min<int64_t>((n + STAGE_THREADS - 1) / STAGE_THREADS, (int64_t)(nsm > 0 ? nsm : 148) * 8);
  return launch_pdl(stage_rows_kernel, dim3((unsigned)blocks), dim3(STAGE_THREADS), 0, st,
                    reinterpret_cast<const uint4*>(x), n, reinterpret_cast<uint4*>(dst));
}

constexpr int SCATTER_THREADS = 256;
constexpr int SCATTER_WARPS = SCATTER_THREADS / 32;

__global__ void __launch_bounds__(SCATTER_THREADS)
    scatter_rows_kernel(const uint16_t* __restrict__ x, int T, int H, const int32_t* __restrict__ t2p, int k, int R,
                        uint16_t* __restrict__ xs) {
  griddep_wait();
  griddep_launch_dependents();
  const int nvec = H / 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = blockIdx.x * SCATTER_WARPS + warp; t < T; t += gridDim.x * SCATTER_WARPS) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    int pos[32];  // k <= 32
    for (int s = 0; s < k; ++s) {
      const int p = __ldg(t2p + (size_t)t * k + s);
      pos[s] = (p >= 0 && p < R) ? p : -1;
    }
    for (int v0 = 0; v0 < nvec; v0 += 128) {
      uint4 val[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int v = v0 + lane + 32 * j;
        if (v < nvec) val[j] = src[v];
      }
      for (int s = 0; s < k; ++s) {
        if (pos[s] < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)pos[s] * H);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int v = v0 + lane + 32 * j;
          if (v < nvec) dst[v] = val[j];
        }
      }
    }
  }
}

int scatter_rows_launch(const uint16_t* x, int T, int H, const int32_t* token_to_perm, int k, int R, uint16_t* xs,
                        cudaStream_t st) {
  if (T == 0) return MOE_OK;
  if (k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int nsm = device_sm_count();
  const int need = (T + SCATTER_WARPS - 1) / SCATTER_WARPS;
  const int grid = std::max(1, std::min(need, (nsm > 0 ? nsm : 148) * 8));
  return launch_pdl(scatter_rows_kernel, dim3(grid), dim3(SCATTER_THREADS), 0, st, x, T, H, token_to_perm, k, R, xs);
}

// ------------------------------------------------------------------------------------------------
// standalone dequantisation: one thread per (row, 64-k chunk), the GEMM's dequant64 routine

__global__ void dequant_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales, float s2, int N,
                               int K, uint16_t* __restrict__ out) {
  const int chunks = K / 64;
  const int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (idx >= (int64_t)N * chunks) return;
  const int n = (int)(idx / chunks), c = (int)(idx - (int64_t)n * chunks);
  const uint4* src = reinterpret_cast<const uint4*>(packed + (size_t)n * (K / 2) + c * 32);
  const uint4 p0 = src[0], p1 = src[1];
  const uint32_t sc = *reinterpret_cast<const uint32_t*>(scales + (size_t)n * (K / 16) + c * 4);
  const uint32_t w[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
  uint32_t o[32];
  dequant64(w, sc, s2, o);
  uint4* dst = reinterpret_cast<uint4*>(out + (size_t)n * K + c * 64);
#pragma unroll
  for (int i = 0; i < 8; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
}

int dequant_launch(const uint8_t* packed, const uint8_t* scales, float scale2, int N, int K, uint16_t* out,
                   cudaStream_t st) {
  const int64_t total = (int64_t)N * (K / 64);
  const int threads = 128;
  dequant_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, st>>>(packed, scales, scale2, N, K, out);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
