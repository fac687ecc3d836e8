// dense_gemm.cu -- dense BF16 GEMM on the 5th-generation tensor cores (tcgen05, sm_103a) for the
// shared expert's three products ("glm5next_mlp/forward.rs" (spark), forward_dense: gate and up
// GEMMs, SwiGLU, down GEMM, all BF16 with FP32 accumulation).
//
//     C[t, col_s + n] = sum_k B[t, k] * W_s[n, k]      (BF16 out, FP32 accumulation)
//
// for up to two weight segments W_s ([rows_s, K], row-major BF16) sharing the activations B
// ([T, K], row-major BF16): the gate and up projections run as one launch writing the two halves
// of one [T, 2I] buffer.  As in the grouped kernels the weight rows are the MMA's M operand (128
// per tile, TMEM lanes) and the token rows its N operand (BN per tile); both operands are staged
// by TMA in the canonical 128-byte-swizzled K-major layout and read by the MMA from shared memory
// (kind::f16, cta_group::1, M = 128, N = BN), the accumulator double-buffered in TMEM so that a
// tile's epilogue overlaps the next tile's MMAs.  Out-of-range rows and k (a tail token tile, a
// weight segment that is not a multiple of 128 rows, K not a multiple of 64) are zero-filled by
// the TMA and never stored.
//
// Warp roles (6 warps): 0 TMA producer, 1 MMA issuer (one thread) and TMEM owner, 2-5 epilogue
// (warp w reads TMEM lanes 32 (w % 4) ..).  Persistent: CTA b takes tiles b, b + grid, ...; tile g
// is (token tile g / NT, weight tile g % NT), weight tiles fastest so CTAs running together share
// the token rows in L2.  Every pipeline wait is bounded (MOE_DEVERR_TIMEOUT, then the CTA drains
// its copies and MMAs, frees TMEM and returns).

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace dg {

constexpr int BM = 128;                // weight rows per tile
constexpr int BK = 64;                 // k per stage: one 128-byte swizzle row
constexpr int A_STAGE = BM * BK * 2;   // 16 KB

template <int BN_>
struct Cfg {
  static constexpr int BN = BN_;
  static constexpr int B_STAGE = BN * BK * 2;
  static constexpr int STAGE = A_STAGE + B_STAGE;
  static constexpr int NS = std::min(8, (192 * 1024) / STAGE);
  static constexpr int TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;  // two accumulators
  static constexpr int THREADS = 6 * 32;
  static constexpr int EPI_WARP_BYTES = 32 * 32 * 2;  // 32 tokens x 32 BF16 outputs
  static constexpr int OFF_EPI = NS * STAGE;
  static constexpr int OFF_BAR = OFF_EPI + 4 * EPI_WARP_BYTES;
  // barriers: full[NS] empty[NS] d_full[2] d_empty[2] drain
  static constexpr int NBAR = 2 * NS + 5;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int SMEM_ALLOC = BYTES + 1024;
  static_assert(BN % 16 == 0 && BN >= 32 && BN <= 256, "MMA N");
  static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0 && TMEM_COLS <= 512, "TMEM allocation");
  static_assert(STAGE % 1024 == 0 && A_STAGE % 1024 == 0, "swizzle atom alignment");
  // more than half of the shared memory: no second CTA of a TMEM-allocating kernel shares the SM
  static_assert(SMEM_ALLOC > 232448 / 2 && SMEM_ALLOC <= 232448, "shared memory");
};

struct Args {
  int T, K;
  int nseg;
  int rows[2];  // weight rows of each segment
  int col[2];   // output column of each segment's row 0
  int nt0, nt;  // weight tiles of segment 0, of both
  int total;    // tiles
  uint16_t* C;
  int ldc;
  int* err;
  uint64_t wait_ns;
};

MOE_DEV bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err, uint64_t limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit) {
      *abort_flag = 1;
      set_error(err, MOE_DEVERR_TIMEOUT);
      return false;
    }
  }
}

MOE_DEV bool warp_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err, uint64_t limit) {
  bool ok = true;
  if (lane_id() == 0) ok = wait_bounded(bar, parity, abort_flag, err, limit);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// One 64-k stage: four k16 MMAs, both operands in shared memory; each step advances both
// descriptors' start address by 32 bytes (+2 in the address >> 4 field) inside the swizzle row.
MOE_DEV void mma4_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, q;\n .reg .b64 a1, a2, a3, b1, b2, b3;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.b32 q, 0, 0;\n"
      " add.s64 a1, %1, 2;\n add.s64 a2, %1, 4;\n add.s64 a3, %1, 6;\n"
      " add.s64 b1, %2, 2;\n add.s64 b2, %2, 4;\n add.s64 b3, %2, 6;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, q;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    dense_gemm_kernel(const __grid_constant__ CUtensorMap wmap0, const __grid_constant__ CUtensorMap wmap1,
                      const __grid_constant__ CUtensorMap bmap, const Args args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  constexpr int NS = C::NS;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (NS + s); };
  auto d_full = [&](int d) { return bar0 + 8u * (2 * NS + d); };
  auto d_empty = [&](int d) { return bar0 + 8u * (2 * NS + 2 + d); };
  const uint32_t drain_bar = bar0 + 8u * (2 * NS + 4);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t limit = args.wait_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(d_full(d), 1);
      mbar_init(d_empty(d), 4);  // the four epilogue warps
    }
    mbar_init(drain_bar, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(s_tmem), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int KA = (args.K + BK - 1) / BK;
  const int tiles_t = (int)gridDim.x;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&wmap0);
      prefetch_tmap(&bmap);
      if (args.nseg > 1) prefetch_tmap(&wmap1);
      int i = 0;
      bool ok = true;
      for (int g = blockIdx.x; ok && g < args.total; g += tiles_t) {
        const int tt = g / args.nt, nt = g - tt * args.nt;
        const bool seg1 = nt >= args.nt0;
        const CUtensorMap* wm = seg1 ? &wmap1 : &wmap0;
        const int row0 = (seg1 ? nt - args.nt0 : nt) * BM;
        const int tok0 = tt * C::BN;
        for (int kb = 0; kb < KA; ++kb, ++i) {
          const int s = i % NS;
          if (!wait_bounded(empty(s), ((i / NS) & 1) ^ 1, s_abort, args.err, limit)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full(s), C::STAGE);
          const uint32_t st = sbase + s * C::STAGE;
          tma_load_2d(st, wm, kb * BK, row0, full(s));
          tma_load_2d(st + A_STAGE, &bmap, kb * BK, tok0, full(s));
        }
      }
      if (!ok)  // every copy issued lands before the CTA leaves
        for (int j = std::max(0, i - NS); j < i; ++j) mbar_wait_drain(full(j % NS), (j / NS) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // the whole warp walks the schedule (warp-uniform descriptors), one elected lane issues
    {
      const uint32_t idesc = make_idesc_bf16(BM, C::BN);
      int i = 0, it = 0;
      bool ok = true;
      for (int g = blockIdx.x; ok && g < args.total; g += tiles_t, ++it) {
        const int db = it & 1;
        if (!warp_wait_bounded(d_empty(db), ((it >> 1) & 1) ^ 1, s_abort, args.err, limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(db * C::BN);
        for (int kb = 0; kb < KA; ++kb, ++i) {
          const int s = i % NS;
          if (!warp_wait_bounded(full(s), (i / NS) & 1, s_abort, args.err, limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + s * C::STAGE;
          if (elect_one()) {
            mma4_bf16_ss(d_tmem, make_sdesc_sw128(st), make_sdesc_sw128(st + A_STAGE), idesc, kb != 0);
            mma_commit(empty(s));
          }
          __syncwarp();
        }
        if (ok) {
          if (elect_one()) mma_commit(d_full(db));
          __syncwarp();
        }
      }
      if (!ok) {  // every issued MMA completes before TMEM is freed
        if (elect_one()) {
          mma_commit(drain_bar);
          mbar_wait_drain(drain_bar, 0);
        }
        __syncwarp();
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant of this warp
    uint8_t* stg = smem + C::OFF_EPI + (warp - 2) * C::EPI_WARP_BYTES;
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    int it = 0;
    for (int g = blockIdx.x; g < args.total; g += tiles_t, ++it) {
      const int tt = g / args.nt, nt = g - tt * args.nt;
      const bool seg1 = nt >= args.nt0;
      const int rows = seg1 ? args.rows[1] : args.rows[0];
      const int n0 = (seg1 ? nt - args.nt0 : nt) * BM + q * 32;  // this warp's first weight row
      const int col = (seg1 ? args.col[1] : args.col[0]) + n0;
      const int tok0 = tt * C::BN;
      const int cnt = min((int)C::BN, args.T - tok0);
      const int db = it & 1;
      if (!warp_wait_bounded(d_full(db), (it >> 1) & 1, s_abort, args.err, limit)) break;
      tc_fence_after();
      const uint32_t dcol = (uint32_t)(db * C::BN);
      for (int c0 = 0; c0 < cnt; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(lane_base + dcol + c0, v);
        tmem_wait_ld();
        if (c0 + 32 >= cnt) {  // the accumulator is free for the tile after next
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(d_empty(db));
        }
        // stage [token j][32 outputs] as BF16, then 16-byte stores of 8 outputs of one token
        __nv_bfloat16* s = reinterpret_cast<__nv_bfloat16*>(stg);
#pragma unroll
        for (int j = 0; j < 32; ++j) s[j * 32 + lane] = __float2bfloat16_rn(__uint_as_float(v[j]));
        __syncwarp();
        const int ntok = min(32, cnt - c0);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int c = lane + 32 * r;
          const int j = c >> 2, part = c & 3;
          if (j < ntok && n0 + part * 8 < rows) {
            const uint4 val = *reinterpret_cast<const uint4*>(stg + j * 64 + part * 16);
            *reinterpret_cast<uint4*>(args.C + (size_t)(tok0 + c0 + j) * args.ldc + col + part * 8) = val;
          }
        }
        __syncwarp();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <class C>
int launch_cfg(const DenseGemm& d, cudaStream_t stream) {
  CUtensorMap wmap[2], bmap;
  for (int s = 0; s < 2; ++s) {
    const int ss = s < d.nseg ? s : 0;  // an unused second map repeats the first
    const cuuint64_t dims[2] = {(cuuint64_t)d.K, (cuuint64_t)d.rows[ss]};
    const cuuint64_t strides[1] = {(cuuint64_t)d.ldw[ss] * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)BM};
    const cuuint32_t estr[2] = {1, 1};
    const int rc = encode_tmap(&wmap[s], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(d.W[ss]), dims,
                               strides, box, estr, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != MOE_OK) return rc;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)d.K, (cuuint64_t)d.T};
    const cuuint64_t strides[1] = {(cuuint64_t)d.ldb * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)C::BN};
    const cuuint32_t estr[2] = {1, 1};
    const int rc = encode_tmap(&bmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(d.B), dims, strides,
                               box, estr, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != MOE_OK) return rc;
  }
  Args a;
  a.T = d.T;
  a.K = d.K;
  a.nseg = d.nseg;
  a.nt0 = (d.rows[0] + BM - 1) / BM;
  a.nt = a.nt0;
  for (int s = 0; s < 2; ++s) {
    a.rows[s] = s < d.nseg ? d.rows[s] : 0;
    a.col[s] = s < d.nseg ? d.col[s] : 0;
  }
  if (d.nseg > 1) a.nt += (d.rows[1] + BM - 1) / BM;
  a.total = a.nt * ((d.T + C::BN - 1) / C::BN);
  a.C = d.C;
  a.ldc = d.ldc;
  a.err = device_error_word();
  a.wait_ns = gemm_wait_limit_ns();
  static std::atomic<int> configured[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (!configured[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(dense_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    configured[dev].store(1, std::memory_order_release);
  }
  const int nsm = device_sm_count();
  if (nsm <= 0) return MOE_ERR_CUDA;
  const int grid = std::max(1, std::min(a.total, nsm));
  dense_gemm_kernel<C><<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(wmap[0], wmap[1], bmap, a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace dg

// Token-tile width: the widest of 256, 128, 64 whose tiles still cover every SM (wide tiles
// halve the weight re-reads per token and keep each MMA large), else 64.
int dense_gemm_token_tile(int T, int weight_tiles, int nsm) {
  for (int bn : {256, 128}) {
    if ((long long)weight_tiles * ((T + bn - 1) / bn) >= nsm) return bn;
  }
  return 64;
}

int dense_gemm_launch(const DenseGemm& d, cudaStream_t stream) {
  if (d.T < 1 || d.K < 1 || d.nseg < 1 || d.nseg > 2 || d.K % 8 || d.ldb % 8 || d.ldc % 8) return MOE_ERR_INVALID_ARG;
  for (int s = 0; s < d.nseg; ++s)
    if (d.rows[s] < 1 || d.rows[s] % 8 || d.ldw[s] % 8 || d.col[s] % 8) return MOE_ERR_INVALID_ARG;
  int nt = 0;
  for (int s = 0; s < d.nseg; ++s) nt += (d.rows[s] + dg::BM - 1) / dg::BM;
  const int nsm = device_sm_count();
  if (nsm <= 0) return MOE_ERR_CUDA;
  switch (dense_gemm_token_tile(d.T, nt, nsm)) {
    case 256: return dg::launch_cfg<dg::Cfg<256>>(d, stream);
    case 128: return dg::launch_cfg<dg::Cfg<128>>(d, stream);
    default: return dg::launch_cfg<dg::Cfg<64>>(d, stream);
  }
}

}  // namespace moe
