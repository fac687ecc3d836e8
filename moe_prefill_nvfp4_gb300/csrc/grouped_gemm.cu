// grouped_gemm.cu -- persistent grouped W4A16 GEMM for sm_103a (tcgen05 + TMA + TMEM + clusters).
//
// One launch covers every expert ("Module forward_prefill_gemm", "What this replaces": one
// launch for all experts, an expert_offsets prefix sum, the A gather through
// sorted_token_ids inside the kernel).  For each expert e and sorted row p in
// [off[e], off[e+1]):  C[p, n] = sum_k A[g(p), k] * Wdq_e[n, k].
//
// Work decomposition ("swap AB"): a tile is (expert e, 128 weight rows, up to BN_MAX of the
// expert's rows).  The 128 weight rows are the MMA's M operand and live in TENSOR MEMORY:
// dequantisation warps turn the TMA-loaded NVFP4 bytes into BF16 and write them with tcgen05.st
// straight into TMEM (no shared-memory round trip for A).  The expert's rows (tokens) are the
// MMA's N operand (16..256 wide, padded to 16) in 128-byte-swizzled shared memory.  FP32
// accumulators stay in TMEM until the epilogue.
//
// Thread-block clusters of CL CTAs take CL consecutive 128-row weight blocks of the same
// (expert, token block): they need the same activation rows, so each CTA fetches 1/CL of them
// and multicasts them into all CL CTAs' shared memory (TMA gather4 for gathered rows, tiled
// 16-row boxes for contiguous rows).  This divides the per-SM activation fetch by CL.
//
// Tile order is (expert, n-block group, token block) with the token block fastest, so the
// clusters that share one expert's weights run at the same time and repeats hit L2: each
// expert's packed weights and scales are read from HBM once per launch.  The persistent
// scheduler is driven by expert_offsets on the device (no host round trip) and balances skew by
// splitting heavy experts into many token blocks.  By default it is a static round-robin walk
// over clusters; a launch that consumes a producer GEMM's output in the same forward (the down
// GEMM after the gate/up GEMM) claims tiles dynamically instead, so that its clusters that start
// early, on SMs the producer has already left, take more of the work (see tile_at below).
//
// A CTA owns NBLK (1 or 2) adjacent 128-row weight blocks that share the activation tile; each
// block has its own accumulator and its own MMA-issuing warp (one thread issues an MMA only every
// ~60-120 cycles, so small token tiles need more than one issuer per SM).
//
// Warp roles (16 warps):
//   0-3   epilogue: TMEM -> registers -> BF16/FP32 -> shared staging -> 16-byte global stores
//   4-11  dequantisation, two warpgroups taking alternate 64-k sub-stages (the 128-row token
//         tiles use one warpgroup, warps 4-7: measured 4-5% faster there, the second one mostly
//         competes with the MMA issuers for issue slots; warps 8-11 then idle)
//   12    weight producer (TMA: packed [128 x 128 B] swizzled + scales [128 x 16 B] per block)
//   13    activation producer (this CTA's share of each stage, multicast to the cluster)
//   14-15 MMA issuers (one thread each, block 0 / block 1); warp 14 owns TMEM
// When the activation ring and the TMEM A ring have the same depth, one "full" barrier per stage
// gathers both producers (the activation bytes as TMA transaction bytes, the four warps of the
// dequantising warpgroup as arrivals) and one commit per atom releases both, so the issuer waits
// once per 64-k atom.
// Every pipeline wait is bounded: on a timeout the CTA records MOE_DEVERR_TIMEOUT, drains its
// in-flight copies and MMAs, frees TMEM and exits.

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace gg {

constexpr int BM = 128;      // weight rows per tile = MMA M = TMEM lanes
constexpr int BKW = 256;     // k per weight stage (128 packed bytes per row)
constexpr int BKA = 64;      // k per activation stage and per TMEM A stage
constexpr int TMEM_COLS = 512;
constexpr int D_COL = 0;     // accumulators first, then the A stages
constexpr int WARP_WP = 12, WARP_AP = 13, WARP_MMA = 14;
constexpr int NUM_WARPS = 16;
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int MAX_E = 512;
constexpr int ID_BOX_ROWS = 16;  // rows per tiled box when the A rows are contiguous
constexpr int NTR = 8;           // tile-ring slots of the dynamic scheduler

// BN_MAX: token-tile width (MMA N, at most 256); NA/NW: activation/weight ring depths;
// ND: accumulator buffers per block (2 lets the epilogue of one tile overlap the next tile's
// MMAs); NBLK: 128-row weight blocks per CTA; NDQ: dequantising warpgroups (1 or 2); WU: the MMA
// warps walk their schedule warp-uniformly and one elected lane issues (else lane 0 alone runs
// the loop; measured per config: faster with the 48-row tiles, slower with the 128-row ones).  TMEM:
// ND*NBLK*BN_MAX accumulator columns, the rest holds NT A stages of 32*NBLK columns (64 k of
// every block).
template <int BN_MAX_, int NA_, int NW_, int ND_, int NBLK_, int NDQ_ = 2, bool WU_ = false>
struct Cfg {
  static constexpr bool WU = WU_;
  static constexpr int BN_MAX = BN_MAX_;
  static constexpr int NA = NA_;
  static constexpr int NW = NW_;
  static constexpr int ND = ND_;
  static constexpr int NBLK = NBLK_;
  static constexpr int NDQ = NDQ_;
  static constexpr int ROWS = BM * NBLK;
  static constexpr int A_COL = ND * NBLK * BN_MAX;
  static constexpr int NT = (TMEM_COLS - A_COL) / (32 * NBLK);
  static constexpr bool MERGED = (NA == NT);  // one "empty" barrier per stage for SMEM and TMEM
  static constexpr int ACT_STAGE = BN_MAX * 128;
  static constexpr int PK_STAGE = ROWS * 128;
  static constexpr int SC_STAGE = ROWS * 16;
  static constexpr int EPI_WARP_BYTES = 32 * 32 * 4;
  static constexpr int OFF_ACT = 0;
  static constexpr int OFF_PK = OFF_ACT + NA * ACT_STAGE;
  static constexpr int OFF_SC = OFF_PK + NW * PK_STAGE;
  static constexpr int OFF_EPI = OFF_SC + NW * SC_STAGE;
  static constexpr int OFF_OFFS = OFF_EPI + 4 * EPI_WARP_BYTES;
  static constexpr int OFF_TBASE = OFF_OFFS + (MAX_E + 1) * 4;
  static constexpr int OFF_BAR = (OFF_TBASE + (MAX_E + 1) * 4 + 7) & ~7;
  // barriers: w_full[NW] w_empty[NW] a_full[NA] a_empty[NA] t_full[NT] t_empty[NT] d_full[ND] d_empty[ND]
  // (t_full / t_empty idle when MERGED)
  // drain[NBLK]
  // + tile ring of the dynamic scheduler: tr_full[NTR] tr_empty[NTR]
  static constexpr int NBAR = 2 * NW + 2 * NA + 2 * NT + 2 * ND + NBLK + 2 * NTR;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int OFF_RING = OFF_MISC + 16;  // NTR tile indices
  static constexpr int BYTES = OFF_RING + NTR * 4;
  // units that read each tile index: weight producer, activation producer, the dequantising
  // warps, the MMA issuers and the epilogue warps (one arrival each)
  static constexpr int TILE_READERS = 2 + 4 * NDQ + NBLK + 4;
  static constexpr int SMEM_ALLOC = BYTES + 1024;  // slack to align the base to 1024
  static_assert(BN_MAX % 16 == 0 && BN_MAX <= 256 && A_COL % 32 == 0 && NT >= 2, "token tile / TMEM columns");
  static_assert(OFF_PK % 1024 == 0 && ACT_STAGE % 1024 == 0, "swizzled buffers need 1024-byte alignment");
  static_assert(BYTES + 1024 <= 232448, "shared memory");
  static_assert(NDQ == 1 || NDQ == 2, "dequantising warpgroups");
};

struct TileInfo {
  int e, nb, p0, cnt, bn;
};

// Group tile g of the cluster walk -> (expert, this CTA's first n-block, token block).  Expert e
// owns group tiles [s_tbase[e], s_tbase[e+1]); a group covers CL * NBLK consecutive n-blocks.
template <int BN_MAX, int NBLK>
MOE_DEV TileInfo decode_tile(int g, const int* s_tbase, const int* s_offs, int E, int CL, int rank) {
  int lo = 0, hi = E - 1;  // largest e in [0, E-1] with s_tbase[e] <= g
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_tbase[mid] <= g) lo = mid; else hi = mid - 1;
  }
  TileInfo ti;
  ti.e = lo;
  const int m = s_offs[lo + 1] - s_offs[lo];
  const int ntt = (m + BN_MAX - 1) / BN_MAX;
  const int local = g - s_tbase[lo];
  const int gb = local / ntt;
  const int tt = local - gb * ntt;
  ti.nb = (gb * CL + rank) * NBLK;
  const int chunk = (((m + ntt - 1) / ntt) + 15) & ~15;
  ti.p0 = s_offs[lo] + tt * chunk;
  ti.cnt = min(chunk, m - tt * chunk);
  ti.bn = (ti.cnt + 15) & ~15;
  return ti;
}

// First weight row of block b of a CTA whose first n-block is nb.  Plain GEMM: consecutive
// blocks.  Fused SwiGLU (half = I): block 0 is gate block j = nb / 2 (rows j*128..), block 1 the
// matching up block (rows I + j*128..), so one CTA holds both halves of 128 activation columns.
template <int NBLK>
MOE_DEV int weight_row(int nb, int b, int half) {
  return half ? (nb / NBLK) * BM + b * half : (nb + b) * BM;
}

// lane 0 waits, the result is broadcast so the whole warp takes the same branch
MOE_DEV bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err) {
  bool ok = true;
  if (lane_id() == 0) ok = mbar_wait(bar, parity, abort_flag, err);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

template <class C>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap amap, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);

  int* s_offs = reinterpret_cast<int*>(smem + C::OFF_OFFS);
  int* s_tbase = reinterpret_cast<int*>(smem + C::OFF_TBASE);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto w_full = [&](int s) { return bar0 + 8u * s; };
  auto w_empty = [&](int s) { return bar0 + 8u * (C::NW + s); };
  auto a_full = [&](int s) { return bar0 + 8u * (2 * C::NW + s); };
  auto a_empty = [&](int s) { return bar0 + 8u * (2 * C::NW + C::NA + s); };
  constexpr int NT = C::NT;
  auto t_full = [&](int s) { return bar0 + 8u * (2 * C::NW + 2 * C::NA + s); };
  auto t_empty = [&](int s) { return bar0 + 8u * (2 * C::NW + 2 * C::NA + NT + s); };
  auto d_full = [&](int d) { return bar0 + 8u * (2 * C::NW + 2 * C::NA + 2 * NT + d); };
  auto d_empty = [&](int d) { return bar0 + 8u * (2 * C::NW + 2 * C::NA + 2 * NT + C::ND + d); };
  auto drain_bar = [&](int b) { return bar0 + 8u * (2 * C::NW + 2 * C::NA + 2 * NT + 2 * C::ND + b); };
  auto tr_full = [&](int s) { return bar0 + 8u * (2 * C::NW + 2 * C::NA + 2 * NT + 2 * C::ND + C::NBLK + s); };
  auto tr_empty = [&](int s) {
    return bar0 + 8u * (2 * C::NW + 2 * C::NA + 2 * NT + 2 * C::ND + C::NBLK + NTR + s);
  };
  volatile int* s_ring = reinterpret_cast<volatile int*>(smem + C::OFF_RING);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  int* s_bad = reinterpret_cast<int*>(smem + C::OFF_MISC + 8);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = args.E;
  const int CL = (int)cluster_nctarank();
  const int rank = (int)cluster_ctarank();
  const int cid = (int)cluster_id_x();
  const int ncl = (int)cluster_count_x();
  const uint16_t mask = (uint16_t)((1u << CL) - 1u);

  if (tid == 0) {
    for (int s = 0; s < C::NW; ++s) {
      mbar_init(w_full(s), 1);
      mbar_init(w_empty(s), 8);
    }
    for (int s = 0; s < C::NA; ++s) {
      // the slot is ready when its activation bytes have landed (one expect-tx arrival) and,
      // when the rings coincide, the dequantisation warpgroup has filled the TMEM A stage (4)
      mbar_init(a_full(s), C::MERGED ? 5 : 1);
      mbar_init(a_empty(s), CL * C::NBLK);  // one commit from every MMA warp of the cluster
    }
    for (int s = 0; s < NT; ++s) {
      mbar_init(t_full(s), 4);
      mbar_init(t_empty(s), C::NBLK);
    }
    for (int d = 0; d < C::ND; ++d) {
      mbar_init(d_full(d), C::NBLK);
      mbar_init(d_empty(d), 4);
    }
    for (int b = 0; b < C::NBLK; ++b) mbar_init(drain_bar(b), 1);
    for (int sl = 0; sl < NTR; ++sl) {
      mbar_init(tr_full(sl), 1);                        // the scheduler's publication
      mbar_init(tr_empty(sl), C::TILE_READERS * CL);    // every reader of every CTA (CTA 0's copy)
    }
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(s_tmem), TMEM_COLS);
    tmem_relinquish();
  }
  // everything above overlaps the previous kernel of the stream; its outputs are read below.  A
  // consumer of a producer GEMM's per-expert readiness counters does not wait for that grid here
  // (it waits per expert before loading A rows, and for the whole grid at its end): the routing
  // outputs it reads come from the grid before the producer, which had completed before the
  // producer released this launch.
  if (args.ready_in == nullptr) griddep_wait();
  griddep_launch_dependents();
  for (int i = tid; i <= E; i += NUM_THREADS) s_offs[i] = args.offsets[i];
  __syncthreads();

  // group-tile table: expert e owns [s_tbase[e], s_tbase[e+1]); absent or empty experts own none
  const int NBG = (args.N + BM * CL * C::NBLK - 1) / (BM * CL * C::NBLK);  // n-block groups (CL*NBLK divides NB)
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int sum = 0;
    bool bad = false;
    for (int e = e0; e < e1; ++e) {
      const int m = s_offs[e + 1] - s_offs[e];
      if (m < 0) bad = true;
      if (m > 0 && args.packed[e] != nullptr) sum += NBG * ((m + C::BN_MAX - 1) / C::BN_MAX);
    }
    if (lane == 0 && (s_offs[0] != 0 || s_offs[E] > args.R || s_offs[E] < 0)) bad = true;
    bad = __any_sync(0xffffffffu, bad);
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int e = e0; e < e1; ++e) {
      s_tbase[e] = bad ? 0 : run;
      const int m = s_offs[e + 1] - s_offs[e];
      if (m > 0 && args.packed[e] != nullptr) run += NBG * ((m + C::BN_MAX - 1) / C::BN_MAX);
    }
    if (lane == 31) s_tbase[E] = bad ? 0 : incl;
    if (lane == 0) *s_bad = bad ? 1 : 0;
    if (bad && lane == 0 && blockIdx.x == 0) set_error(args.err, MOE_DEVERR_BAD_OFFSETS);
  }
  tc_fence_before();
  cluster_sync_all();  // barriers of every CTA initialised before any multicast reaches them
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int total = s_tbase[E];

  // Tile sequence of this cluster.  Static: tiles cid, cid + ncl, ...  Dynamic (a consumer GEMM):
  // CTA 0's weight producer claims each next tile from args.tile_counter and publishes it into
  // the tile ring of every CTA of the cluster; every role of every CTA reads the ring in order, so
  // the clusters that start early take more tiles.  tile_at(i) is called by one thread per
  // reading unit and returns the i-th tile, -1 after the last, -2 when the CTA aborts.
  const bool dyn = args.tile_counter != nullptr;
  auto tile_at = [&](int i) -> int {
    if (!dyn) {
      const int g = cid + i * ncl;
      return g < total ? g : -1;
    }
    const int sl = i % NTR;
    if (!mbar_wait_cluster(tr_full(sl), (i / NTR) & 1, s_abort, args.err)) return -2;
    const int g = s_ring[sl];
    mbar_arrive_remote(tr_empty(sl), 0);
    return g;
  };
  // CTA 0's weight producer claims and publishes the cluster's tiles: one ahead of its own use
  // while more than four rounds of tiles remain (the claim's round trip to global memory then
  // overlaps the current tile; measured +1.4% at 2048 rows), at the point of use after that (a
  // claim made early near the end can strand a tile on a busy cluster: -1.3% at 256 rows, which
  // has fewer than four rounds).  Returns false on abort.
  int n_pub = 0, last_claim = 0;
  bool pub_end = false;
  auto publish_upto = [&](int last) -> bool {
    for (; !pub_end && n_pub <= last; ++n_pub) {
      const int sl = n_pub % NTR;
      if (n_pub >= NTR && !mbar_wait_cluster(tr_empty(sl), ((n_pub / NTR) - 1) & 1, s_abort, args.err)) return false;
      int g = atomicAdd(args.tile_counter, 1);
      last_claim = g;
      if (g >= total) {
        g = -1;
        pub_end = true;
      }
      for (int r = 0; r < CL; ++r) {
        st_shared_cluster_u32(sbase + C::OFF_RING + 4 * sl, r, (uint32_t)g);
        mbar_arrive_remote(tr_full(sl), r);
      }
    }
    return true;
  };
  const int KA = args.K / BKA;  // activation / TMEM stages per tile
  const int KW = args.K / BKW;  // weight stages per tile

  if (warp < 4) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp;
    uint8_t* stg = smem + C::OFF_EPI + q * C::EPI_WARP_BYTES;
    const bool f32 = args.c_dtype == MOE_DTYPE_F32;
    const int esz = f32 ? 4 : 2;
    // rows of absent experts are written as zeros (the pages' zeroed routed-output rows)
    const int out_cols = args.swiglu_half ? args.swiglu_half : args.N;
    if (!*s_bad) {
      const int chunks_per_row = out_cols * esz / 16;
      for (int e = 0; e < E; ++e) {
        if (args.packed[e] != nullptr) continue;
        int nz = 0;
        for (int r = s_offs[e] + blockIdx.x; r < s_offs[e + 1]; r += gridDim.x, ++nz) {
          uint8_t* row = reinterpret_cast<uint8_t*>(args.C) + (size_t)r * args.ldc * esz;
          for (int c = tid; c < chunks_per_row; c += 128) *reinterpret_cast<uint4*>(row + c * 16) = make_uint4(0, 0, 0, 0);
        }
        if (args.ready_out != nullptr && nz > 0) {  // each epilogue warp publishes its own stores
          __threadfence();
          __syncwarp();
          if (lane == 0) counter_add_release(args.ready_out + e, nz * args.ready_need);
        }
      }
    }
    for (int it = 0;; ++it) {
      int g = 0;
      if (lane == 0) g = tile_at(it);
      g = __shfl_sync(0xffffffffu, g, 0);
      if (g < 0) break;
      const TileInfo ti = decode_tile<C::BN_MAX, C::NBLK>(g, s_tbase, s_offs, E, CL, rank);
      const int db = it % C::ND;
      if (!warp_wait(d_full(db), (it / C::ND) & 1, s_abort, args.err)) break;
      tc_fence_after();
      if (C::NBLK == 2 && args.swiglu_half) {
        // fused SwiGLU: act[p, n] = silu(min(g, L)) * clamp(u, -L, L) from the FP32 accumulators
        // of the gate block (b = 0) and the up block (b = 1), each rounded to BF16 first (the
        // pages' BF16 gate/up buffers); BF16 out, [R, swiglu_half]
        const int n0 = (ti.nb / C::NBLK) * BM + q * 32;
        const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
        const uint32_t dg = D_COL + (db * C::NBLK) * C::BN_MAX;
        const uint32_t du = dg + C::BN_MAX;
        for (int c0 = 0; c0 < ti.cnt; c0 += 32) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(lane_base + dg + c0, g);
          tmem_ld_32x32b_x32(lane_base + du + c0, u);
          tmem_wait_ld();
          if (c0 + 32 >= ti.cnt) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(d_empty(db));
          }
          __syncwarp();
          __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(stg);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            st[j * 32 + lane] = __float2bfloat16_rn(swiglu_clamped(
                __bfloat162float(__float2bfloat16_rn(__uint_as_float(g[j]))),
                __bfloat162float(__float2bfloat16_rn(__uint_as_float(u[j]))), args.limit));
          __syncwarp();
          const int rows = min(32, ti.cnt - c0);
          for (int c = lane; c < 32 * 4; c += 32) {
            const int r = c >> 2, cc = c & 3;
            if (r < rows) {
              const uint4 val = *reinterpret_cast<const uint4*>(stg + r * 64 + cc * 16);
              uint16_t* dst = reinterpret_cast<uint16_t*>(args.C) + (size_t)(ti.p0 + c0 + r) * args.ldc + n0 + cc * 8;
              *reinterpret_cast<uint4*>(dst) = val;
            }
          }
        }
        if (args.ready_out != nullptr) {  // this warp's part of the tile's rows is stored
          __threadfence();
          __syncwarp();
          if (lane == 0) counter_add_release(args.ready_out + ti.e, ti.cnt);
        }
        continue;
      }
      for (int b = 0; b < C::NBLK; ++b) {
        const int n0 = (ti.nb + b) * BM + q * 32;
        const uint32_t dcol = D_COL + (db * C::NBLK + b) * C::BN_MAX;
        for (int c0 = 0; c0 < ti.cnt; c0 += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + dcol + c0, v);
          tmem_wait_ld();
          if (b == C::NBLK - 1 && c0 + 32 >= ti.cnt) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(d_empty(db));
          }
          __syncwarp();
          if (f32) {
            float* s = reinterpret_cast<float*>(stg);
#pragma unroll
            for (int j = 0; j < 32; ++j) s[j * 32 + lane] = __uint_as_float(v[j]);
          } else {
            __nv_bfloat16* s = reinterpret_cast<__nv_bfloat16*>(stg);
#pragma unroll
            for (int j = 0; j < 32; ++j) s[j * 32 + lane] = __float2bfloat16_rn(__uint_as_float(v[j]));
          }
          __syncwarp();
          const int rows = min(32, ti.cnt - c0);
          const int cpr = 32 * esz / 16;  // 16-byte chunks per staged row (4 bf16, 8 f32)
          for (int c = lane; c < 32 * cpr; c += 32) {
            const int r = c / cpr, cc = c - r * cpr;
            const int n = n0 + cc * (16 / esz);
            if (r < rows && n < args.N) {
              const uint4 val = *reinterpret_cast<const uint4*>(stg + r * 32 * esz + cc * 16);
              uint8_t* dst = reinterpret_cast<uint8_t*>(args.C) + ((size_t)(ti.p0 + c0 + r) * args.ldc + n) * esz;
              *reinterpret_cast<uint4*>(dst) = val;
            }
          }
        }
      }
      if (args.ready_out != nullptr) {  // this warp's part of the tile's rows is stored
        __threadfence();
        __syncwarp();
        if (lane == 0) counter_add_release(args.ready_out + ti.e, ti.cnt);
      }
    }
  } else if (warp < 4 + 4 * C::NDQ) {
    // ------------------------------------------------------------------ dequantisation
    // Two warpgroups take alternate 64-k sub-stages of each weight stage (warpgroup wg: subs wg,
    // wg + 2); one warpgroup takes all four in order, two per pass over the stage.  Every pass
    // arrives once on the stage's "empty" barrier (8 arrivals per stage either way).
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    int wi = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      int g = 0;
      if (lane == 0) g = tile_at(i);
      g = __shfl_sync(0xffffffffu, g, 0);
      if (g < 0) break;
      const TileInfo ti = decode_tile<C::BN_MAX, C::NBLK>(g, s_tbase, s_offs, E, CL, rank);
      const float s2 = args.scale2[ti.e];
      for (int ks = 0; ok && ks < KW; ++ks, ++wi)
      for (int pass = 0; pass < 2 / C::NDQ; ++pass) {
        const int s = wi % C::NW;
        if (!warp_wait(w_full(s), (wi / C::NW) & 1, s_abort, args.err)) { ok = false; break; }
        uint4 chunk[C::NBLK][4];
        uint4 scv[C::NBLK];
#pragma unroll
        for (int b = 0; b < C::NBLK; ++b) {
          const int wr = b * BM + row;  // row of the stage (block b)
          const uint8_t* pk = smem + C::OFF_PK + s * C::PK_STAGE + wr * 128;
          scv[b] = *reinterpret_cast<const uint4*>(smem + C::OFF_SC + s * C::SC_STAGE + wr * 16);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int sub = C::NDQ == 2 ? wg + 2 * h : 2 * pass + h;
            chunk[b][2 * h] = *reinterpret_cast<const uint4*>(pk + (((2 * sub) ^ (wr & 7)) << 4));
            chunk[b][2 * h + 1] = *reinterpret_cast<const uint4*>(pk + (((2 * sub + 1) ^ (wr & 7)) << 4));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(w_empty(s));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int sub = C::NDQ == 2 ? wg + 2 * h : 2 * pass + h;
          const int tix = wi * 4 + sub;
          const int ts = tix % NT;
          if (!warp_wait(C::MERGED ? a_empty(ts) : t_empty(ts), ((tix / NT) & 1) ^ 1, s_abort, args.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int b = 0; b < C::NBLK; ++b) {
            const uint32_t w[8] = {chunk[b][2 * h].x,     chunk[b][2 * h].y,     chunk[b][2 * h].z,
                                   chunk[b][2 * h].w,     chunk[b][2 * h + 1].x, chunk[b][2 * h + 1].y,
                                   chunk[b][2 * h + 1].z, chunk[b][2 * h + 1].w};
            const uint32_t sc = sub == 0 ? scv[b].x : sub == 1 ? scv[b].y : sub == 2 ? scv[b].z : scv[b].w;
            uint32_t out[32];
            dequant64(w, sc, s2, out);
            tmem_st_32x32b_x32(tmem_base + lane_addr + C::A_COL + ts * 32 * C::NBLK + b * 32, out);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(C::MERGED ? a_full(ts) : t_full(ts));
        }
        if (!ok) break;
      }
    }
  } else if (warp == WARP_WP) {
    // ------------------------------------------------------------------ weight producer
    if (lane == 0) {
      int wi = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        if (dyn && rank == 0 && !publish_upto(last_claim + 4 * ncl < total ? i + 1 : i)) { ok = false; break; }
        const int g = tile_at(i);
        if (g == -2) ok = false;
        if (g < 0) break;
        const TileInfo ti = decode_tile<C::BN_MAX, C::NBLK>(g, s_tbase, s_offs, E, CL, rank);
        const CUtensorMap* mp = args.wmaps + 2 * ti.e;
        const CUtensorMap* ms = mp + 1;
        prefetch_tmap(mp);
        prefetch_tmap(ms);
        for (int ks = 0; ks < KW; ++ks, ++wi) {
          const int s = wi % C::NW;
          if (!mbar_wait(w_empty(s), ((wi / C::NW) & 1) ^ 1, s_abort, args.err)) { ok = false; break; }
          mbar_arrive_expect_tx(w_full(s), C::PK_STAGE + C::SC_STAGE);
#pragma unroll
          for (int b = 0; b < C::NBLK; ++b) {
            const int row = weight_row<C::NBLK>(ti.nb, b, args.swiglu_half);
            tma_load_2d(sbase + C::OFF_PK + s * C::PK_STAGE + b * BM * 128, mp, ks * 128, row, w_full(s));
            tma_load_2d(sbase + C::OFF_SC + s * C::SC_STAGE + b * BM * 16, ms, ks * 16, row, w_full(s));
          }
        }
      }
      if (!ok)
        for (int j = max(0, wi - C::NW); j < wi; ++j) mbar_wait_drain(w_full(j % C::NW), (j / C::NW) & 1);
    }
  } else if (warp == WARP_AP) {
    // ------------------------------------------------------------------ activation producer
    // This CTA fetches the row groups grp with grp % CL == rank of each stage and multicasts them.
    // Gathered rows: groups of 4 rows (TMA gather4); contiguous rows: 16-row tiled boxes.
    constexpr int NH = (C::BN_MAX + 127) / 128;  // gather4 groups per lane per stage (CL = 1)
    const bool gathered = args.gather != nullptr;
    int ai = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      int g = 0;
      if (lane == 0) g = tile_at(i);
      g = __shfl_sync(0xffffffffu, g, 0);
      if (g == -2) ok = false;
      if (g < 0) break;
      const TileInfo ti = decode_tile<C::BN_MAX, C::NBLK>(g, s_tbase, s_offs, E, CL, rank);
      const int ng = gathered ? (ti.bn >> 2) : (ti.bn / ID_BOX_ROWS);  // row groups per stage
      int rows[NH * 4];
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const int grp = rank + CL * (lane + 32 * h);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int p = ti.p0 + min(4 * grp + r, ti.cnt - 1);
          int src = gathered ? args.gather[p] : p;
          if ((unsigned)src >= (unsigned)args.a_rows) {
            if (gathered && grp < ng) set_error(args.err, MOE_DEVERR_BAD_GATHER);
            src = 0;
          }
          rows[4 * h + r] = src;
        }
      }
      if (args.ready_in != nullptr) {
        // the producer GEMM has stored every row of this expert (all its column blocks; each of
        // its 4 epilogue warps publishes separately)
        bool rdy = true;
        if (lane == 0)
          rdy = wait_counter_geq(args.ready_in + ti.e, (s_offs[ti.e + 1] - s_offs[ti.e]) * args.ready_need * 4,
                                 s_abort, args.err);
        if (__shfl_sync(0xffffffffu, rdy ? 1 : 0, 0) == 0) { ok = false; break; }
        fence_proxy_async_global();  // every lane issues TMA loads of those rows below
      }
      for (int kb = 0; kb < KA; ++kb, ++ai) {
        const int s = ai % C::NA;
        if (!warp_wait(a_empty(s), ((ai / C::NA) & 1) ^ 1, s_abort, args.err)) { ok = false; break; }
        if (lane == 0) mbar_arrive_expect_tx(a_full(s), ti.bn * 128);
        __syncwarp();
        const uint32_t dst0 = sbase + C::OFF_ACT + s * C::ACT_STAGE;
        const int x = kb * BKA;
        if (gathered) {
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const int grp = rank + CL * (lane + 32 * h);
            if (grp < ng) {
              if (CL > 1)
                tma_gather4_mc(dst0 + grp * 512, &amap, x, rows[4 * h], rows[4 * h + 1], rows[4 * h + 2],
                               rows[4 * h + 3], a_full(s), mask);
              else
                tma_gather4(dst0 + grp * 512, &amap, x, rows[4 * h], rows[4 * h + 1], rows[4 * h + 2],
                            rows[4 * h + 3], a_full(s));
            }
          }
        } else {
          for (int grp = rank + CL * lane; grp < ng; grp += CL * 32) {
            const int y = ti.p0 + grp * ID_BOX_ROWS;
            if (CL > 1)
              tma_load_2d_mc(dst0 + grp * ID_BOX_ROWS * 128, &amap, x, y, a_full(s), mask);
            else
              tma_load_2d(dst0 + grp * ID_BOX_ROWS * 128, &amap, x, y, a_full(s));
          }
        }
      }
    }
    if (!ok && lane == 0)
      for (int j = max(0, ai - C::NA); j < ai; ++j) mbar_wait_drain(a_full(j % C::NA), (j / C::NA) & 1);
  } else {
    // ------------------------------------------------------------------ MMA issuers
    const int b = warp - WARP_MMA;  // weight block of this issuer (b < 0: a warp without a role)
    if constexpr (C::WU) {
      if (b >= 0 && b < C::NBLK) {
        int ai = 0;
        bool ok = true;
        for (int it = 0; ok; ++it) {
          int g = 0;
          if (lane == 0) g = tile_at(it);
          g = __shfl_sync(0xffffffffu, g, 0);
          if (g == -2) ok = false;
          if (g < 0) break;
          const TileInfo ti = decode_tile<C::BN_MAX, C::NBLK>(g, s_tbase, s_offs, E, CL, rank);
          const int db = it % C::ND;
          if (!warp_wait(d_empty(db), ((it / C::ND) & 1) ^ 1, s_abort, args.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t idesc = make_idesc_bf16(BM, ti.bn);
          const uint64_t bdesc0 = make_sdesc_sw128(sbase + C::OFF_ACT);
          const uint32_t a_tmem0 = tmem_base + C::A_COL + b * 32;
          const uint32_t d_tmem = tmem_base + D_COL + (db * C::NBLK + b) * C::BN_MAX;
          for (int kb = 0; kb < KA; ++kb, ++ai) {
            const int s = ai % C::NA;
            const int ts = ai % NT;
            if (!warp_wait(a_full(s), (ai / C::NA) & 1, s_abort, args.err)) { ok = false; break; }
            if (!C::MERGED && !warp_wait(t_full(ts), (ai / NT) & 1, s_abort, args.err)) { ok = false; break; }
            tc_fence_after();
            const uint64_t bdesc = bdesc0 + (uint64_t)((s * C::ACT_STAGE) >> 4);
            if (elect_one()) {
              mma4_bf16_ts(d_tmem, a_tmem0 + ts * 32 * C::NBLK, bdesc, idesc, kb != 0);
              if (CL > 1) mma_commit_mc(a_empty(s), mask);
              else mma_commit(a_empty(s));
              if (!C::MERGED) mma_commit(t_empty(ts));
            }
            __syncwarp();
          }
          if (ok) {
            if (elect_one()) mma_commit(d_full(db));
            __syncwarp();
          }
        }
        if (!ok) {
          if (elect_one()) {
            mma_commit(drain_bar(b));
            mbar_wait_drain(drain_bar(b), 0);
          }
          __syncwarp();
        }
      }
    } else if (lane == 0 && b >= 0 && b < C::NBLK) {
      int ai = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int g = tile_at(it);
        if (g == -2) ok = false;
        if (g < 0) break;
        const TileInfo ti = decode_tile<C::BN_MAX, C::NBLK>(g, s_tbase, s_offs, E, CL, rank);
        const int db = it % C::ND;
        if (!mbar_wait(d_empty(db), ((it / C::ND) & 1) ^ 1, s_abort, args.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t idesc = make_idesc_bf16(BM, ti.bn);
        const uint64_t bdesc0 = make_sdesc_sw128(sbase + C::OFF_ACT);
        const uint32_t a_tmem0 = tmem_base + C::A_COL + b * 32;
        const uint32_t d_tmem = tmem_base + D_COL + (db * C::NBLK + b) * C::BN_MAX;
        for (int kb = 0; kb < KA; ++kb, ++ai) {
          const int s = ai % C::NA;
          const int ts = ai % NT;
          if (!mbar_wait(a_full(s), (ai / C::NA) & 1, s_abort, args.err)) { ok = false; break; }
          if (!C::MERGED && !mbar_wait(t_full(ts), (ai / NT) & 1, s_abort, args.err)) { ok = false; break; }
          tc_fence_after();
          // the descriptor's start-address field is the byte address >> 4: a stage offset adds to it
          const uint64_t bdesc = bdesc0 + (uint64_t)((s * C::ACT_STAGE) >> 4);
          mma4_bf16_ts(d_tmem, a_tmem0 + ts * 32 * C::NBLK, bdesc, idesc, kb != 0);
          // One commit releases the activation slot in every CTA of the cluster; when the two
          // rings have the same depth it also releases the TMEM A stage (the dequantisation warps
          // then wait on the slot's barrier), otherwise a second commit does.
          if (CL > 1) mma_commit_mc(a_empty(s), mask);
          else mma_commit(a_empty(s));
          if (!C::MERGED) mma_commit(t_empty(ts));
        }
        if (ok) mma_commit(d_full(db));
      }
      if (!ok) {
        mma_commit(drain_bar(b));
        mbar_wait_drain(drain_bar(b), 0);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
  cluster_sync_all();  // no CTA leaves while another may still multicast into it or signal it
  // a consumer completes only after its producer grid (stream order for the launches after it)
  if (args.ready_in != nullptr) griddep_wait();
}

// token tiles of 48 / 64 / 128 / 256 rows; the 48- to 128-row configs pair two weight blocks per CTA
using CfgT2 = Cfg<48, 5, 4, 2, 2, 2, true>;  // NT = 5; two accumulator buffers (mean rows per expert <= 32)
using CfgS2 = Cfg<64, 6, 4, 1, 2>;   // NT = 6
using CfgS2D = Cfg<64, 4, 4, 2, 2>;  // NT = 4; two accumulator buffers (contiguous rows)
using CfgM2 = Cfg<128, 4, 3, 1, 2, 1>;  // NT = 4; one dequantising warpgroup
using CfgS1 = Cfg<64, 12, 6, 2, 1>;  // NT = 12
using CfgM1 = Cfg<128, 8, 4, 2, 1>;  // NT = 8
using CfgL1 = Cfg<256, 3, 4, 1, 1>;

template <class C>
int launch_cfg(const CUtensorMap& amap, const GemmArgs& args, cudaStream_t stream) {
  // per-device caches of idempotent facts (several host threads may fill them concurrently)
  static std::atomic<int> configured[64];
  static std::atomic<int> max_clusters[64][9];  // per cluster width
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (!configured[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(grouped_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    configured[dev].store(1, std::memory_order_release);
  }
  const int nsm = device_sm_count();
  if (nsm <= 0) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = C::SMEM_ALLOC;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // the occupancy queries below take the cluster attribute alone
  // cluster width: gathered rows are bound by the TMA gather4 issue rate of each SM (~80-150
  // cycles per 4-row copy), so wider multicast (any width up to 8 that divides the weight-block
  // groups, not only powers of two) makes each tile cheaper.  Wide clusters leave SMs idle (8-CTA
  // clusters fit on 120 of 152 SMs, 6-CTA on 138), which measured as the lesser cost down to ~90%
  // coverage: gathered rows take the widest width whose clusters cover >= 90% of the SMs.
  // Contiguous rows in tiled boxes use pairs.  args.max_cluster caps the width (1: every CTA
  // loads its own activation tiles, no multicast).
  const int nblocks = (args.N + BM - 1) / BM;
  const int groups = nblocks / C::NBLK;
  const bool gathered = args.gather != nullptr;
  int CL = 1, ncl_max = 0;
  for (int cl = std::min(gathered ? 8 : 2, std::max(1, args.max_cluster)); cl >= 1; --cl) {
    if (groups % cl != 0) continue;
    int n = max_clusters[dev][cl].load(std::memory_order_relaxed);
    if (n == 0) {
      attr[0].val.clusterDim.x = cl;
      cfg.gridDim = dim3(cl * nsm);
      if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_kernel<C>, &cfg) != cudaSuccess || n < 1) return MOE_ERR_CUDA;
      max_clusters[dev][cl].store(n, std::memory_order_relaxed);
    }
    if (n * cl * 10 >= nsm * 9 || cl == 1) {
      CL = cl;
      break;
    }
  }
  ncl_max = max_clusters[dev][CL].load(std::memory_order_relaxed);
  attr[0].val.clusterDim.x = CL;
  const long long nbg = groups / CL;
  const long long max_groups = nbg * ((long long)args.E + (args.R + C::BN_MAX - 1) / C::BN_MAX);
  const int ncl = (int)std::max<long long>(1, std::min<long long>(ncl_max, max_groups));
  cfg.gridDim = dim3(ncl * CL);
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<C>, amap, args) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace gg

// ------------------------------------------------------------------------------------------------
// host side

int grouped_gemm_launch(const GemmArgs& args, const void* A, int a_rows, int lda, cudaStream_t stream) {
  const bool gathered = args.gather != nullptr;
  CUtensorMap amap;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)args.K, (cuuint64_t)a_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)lda * 2};
    const cuuint32_t box[2] = {64, gathered ? 1u : (cuuint32_t)gg::ID_BOX_ROWS};
    const cuuint32_t estr[2] = {1, 1};
    int rc = encode_tmap(&amap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(A), dims, strides, box, estr,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != MOE_OK) return rc;
  }
  // token-tile width from the mean rows per expert (the distribution itself is on the device);
  // two weight blocks per CTA when the number of 128-row blocks is even
  const double mean_rows = (double)args.R / args.E;
  const bool pairs = ((args.N + gg::BM - 1) / gg::BM) % 2 == 0;
  // measured at <= 32 rows per expert (256-row chunk, 64 experts): 48-row tiles with a second
  // accumulator buffer (the epilogue overlaps the next tile) beat 64-row tiles by ~3% on both
  // GEMMs; the few experts above 48 rows take a second token tile
  if (args.swiglu_half) {
    // the fused SwiGLU needs the gate/up pair in one CTA: two-block configs only
    if (mean_rows <= 32.0) return gg::launch_cfg<gg::CfgT2>(amap, args, stream);
    if (mean_rows <= 48.0) return gg::launch_cfg<gg::CfgS2>(amap, args, stream);
    return gg::launch_cfg<gg::CfgM2>(amap, args, stream);
  }
  // measured: gathered rows keep six activation stages at the cost of a second accumulator
  // buffer; contiguous rows prefer the overlap of the epilogue with the next tile; above ~48 rows
  // per expert two 128-row token tiles per weight-block pair beat one 256-row tile
  if (mean_rows <= 48.0) {
    if (!pairs) return gg::launch_cfg<gg::CfgS1>(amap, args, stream);
    if (mean_rows <= 32.0) return gg::launch_cfg<gg::CfgT2>(amap, args, stream);
    return gathered ? gg::launch_cfg<gg::CfgS2>(amap, args, stream) : gg::launch_cfg<gg::CfgS2D>(amap, args, stream);
  }
  if (pairs) return gg::launch_cfg<gg::CfgM2>(amap, args, stream);
  return mean_rows <= 160.0 ? gg::launch_cfg<gg::CfgM1>(amap, args, stream) : gg::launch_cfg<gg::CfgL1>(amap, args, stream);
}

}  // namespace moe
