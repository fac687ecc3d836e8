// pair_gemm.cu -- grouped W4A16 GEMM on CTA pairs (tcgen05.mma.cta_group::2) for sm_103a.
//
// One launch covers every expert ("Module forward_prefill_gemm", "What this replaces": one launch
// for all experts over an expert_offsets prefix sum, the A gather through sorted_token_ids inside
// the kernel).  For each expert e and sorted row p in [off[e], off[e+1]):
//     C[p, n] = sum_k A[g(p), k] * Wdq_e[n, k],   Wdq = bf16(fp32(E2M1 * E4M3) * scale2).
//
// Work decomposition ("swap AB", as in the single-CTA kernel): the weight rows are the MMA's M
// operand, the expert's token rows its N operand.  Two CTAs of a cluster form a pair whose MMA has
// M = 256: each CTA dequantises its own 128 weight rows into its TENSOR MEMORY (tcgen05.st), each
// holds half of the token tile (N/2 rows of B) in its shared memory, and one thread of the even CTA
// issues the pair's MMAs; both CTAs' TMEM receive their 128 rows x N of the FP32 accumulator.  A
// tile is (expert, 256 weight rows, up to BN token rows); a 256 x 192 MMA instruction does three
// times the work of a 128 x 128 one, which is what keeps the tensor pipe busy: one thread issues
// an MMA only every ~70-120 cycles, and the dequantising warps on its sub-partition make it
// slower, so small MMAs leave the tensor pipe idle.  A short tile costs nearly as much as a full
// one (dequantising its weights sets its pace), so busy experts take tiles of up to 384 rows (two
// MMAs of N = 192 per k16 step into 384 accumulator columns): an expert with m rows costs
// ceil(m / 384) weight passes instead of ceil(m / 256).
//
// B rows are contiguous: the down GEMM's activation rows are already in expert order, and the
// gate/up GEMM's gathered token rows are stored into expert order by this kernel's own epilogue
// warps, which have nothing to drain until the first accumulators are complete (GemmArgs::row_src;
// a TMA gather4 moves only ~12 B/cycle per SM and a 256-token tile needs ~32 B/cycle, 16-byte
// cp.async gathers from two warps measured ~8 B/cycle, so the tiles do not gather).  The rows are
// stored in sorted order by all epilogue warps of the grid; an expert's tiles start once its row
// count is published.  Each CTA loads the rows it holds with one tiled TMA box per atom and MMA
// (BN/(2 NH) rows x 64 k, 128-byte swizzle) whose transaction bytes complete on the even CTA's
// barrier (the .cta_group::2 form).  There is no cluster multicast.
//
// Warp roles (16 warps, 20 with a second epilogue warpgroup):
//   0-3   epilogue: TMEM -> registers -> BF16/FP32 (or the fused clamped SwiGLU) -> global;
//         between accumulators, the token rows in expert order (GemmArgs::row_src); 16-19 the
//         second epilogue warpgroup
//   4-7   dequantisation (8-11 a second warpgroup taking alternate turns of atoms when NDQ = 2)
//   12    weight producer (TMA: packed 2 x [64 rows x 128 B] swizzled + scales 2 x [64 x 16 B])
//   13    B producer (TMA: this CTA's half of the token tile)
//   14    MMA issuer (even CTA, one thread); TMEM allocation in both CTAs
// Per atom (64 k) the even CTA's "full" barrier collects the 4 dequantising warps of each CTA (the
// odd CTA's arrive remotely), the even CTA's B producer (arrival with the expected bytes of both
// CTAs' boxes) and both CTAs' TMA transaction bytes; one multicast commit then releases the
// atom's B and A slots in both CTAs.
// The gate/up projection with the fused SwiGLU maps each CTA's 128 rows as 64 gate rows + the 64
// matching up rows, interleaved in 16-row groups so that each warp of the epilogue holds a gate
// row and its up row in lanes l and l + 16 of the same warp.
//
// Every pipeline wait is bounded (GemmArgs::wait_ns): on a timeout the CTA records
// MOE_DEVERR_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM and returns.

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace pg {

constexpr int BM = 128;          // weight rows per CTA (TMEM lanes); the pair's MMA has M = 256
constexpr int PAIR_ROWS = 256;
constexpr int BKW = 256;         // k per weight stage (128 packed bytes per row)
constexpr int BKA = 64;          // k per atom: one B stage, one TMEM A stage, four MMAs
constexpr int TMEM_COLS = 512;
constexpr int WARP_WP = 12, WARP_BP = 13, WARP_MMA = 14;
constexpr int MAX_E = 512;

// BN: token-tile width (each CTA holds BN/2 rows of B); NH: MMAs per k16 step across the tile
// (each of N = BN/NH <= 256, into its own accumulator columns); ND: accumulator buffers (2 lets
// the epilogue of one tile overlap the next tile's MMAs); NDQ: dequantising warpgroups.  TMEM:
// ND*BN accumulator columns, then NS A slots of 32 columns.
template <int BN_, int ND_, int NDQ_, int NEPI_ = 1, int NH_ = 1>
struct Cfg {
  static constexpr int BN = BN_;
  static constexpr int ND = ND_;
  static constexpr int NDQ = NDQ_;
  static constexpr int NEPI = NEPI_;  // epilogue warpgroups (2: alternate 32-column chunks)
  static constexpr int NH = NH_;
  static constexpr int HN = BN / NH;      // one MMA's N
  static constexpr int BOXH = HN / 2;     // B rows of one MMA in each CTA (one TMA box per atom)
  // warps: 0-3 epilogue, 4-7 (and 8-11) dequantisation, 12-14 producers and MMA, 16-19 the second
  // epilogue warpgroup when NEPI = 2
  static constexpr int THREADS = (NEPI == 2 ? 20 : 16) * 32;
  static constexpr int BH = BN / 2;
  static constexpr int A_COL = ND * BN;
  static constexpr int NS = (TMEM_COLS - A_COL) / 32;  // A slots = B slots; atom ai takes slot ai % NS
  // The dequantising warpgroups split every weight stage (four atoms): warpgroup wg takes the APW
  // atoms wg*APW.. of each stage, so each warpgroup waits on every phase of the weight ring in
  // order and both release each stage.  With NS a multiple of four every A slot then has a
  // single dequantising writer, whose successive uses of it are one completed phase apart.
  static constexpr int APW = 4 / NDQ;
  static constexpr int NW = 3;
  static constexpr int B_STAGE = BH * 128;  // NH boxes of BOXH rows
  static constexpr int PK_STAGE = BM * 128;
  static constexpr int SC_STAGE = BM * 16;
  static constexpr int EPI_WARP_BYTES = 32 * 32 * 4;
  static constexpr int OFF_B = 0;
  static constexpr int OFF_PK = OFF_B + NS * B_STAGE;
  static constexpr int OFF_SC = OFF_PK + NW * PK_STAGE;
  static constexpr int OFF_EPI = OFF_SC + NW * SC_STAGE;
  static constexpr int OFF_OFFS = OFF_EPI + 4 * NEPI * EPI_WARP_BYTES;
  static constexpr int OFF_TBASE = OFF_OFFS + (MAX_E + 1) * 4;
  static constexpr int OFF_BAR = (OFF_TBASE + (MAX_E + 1) * 4 + 7) & ~7;
  // barriers: full[NS] empty[NS] w_full[NW] w_empty[NW] d_full[ND] d_empty[ND] drain
  static constexpr int NBAR = 2 * NS + 2 * NW + 2 * ND + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 32;
  static constexpr int SMEM_ALLOC = BYTES + 1024;
  static constexpr int FULL_COUNT = 2 * 4 + 1;  // dequantising warps of both CTAs + the B producer
  static_assert(BN == NH * HN && HN % 32 == 0 && HN <= 256 && (NH == 1 || NH == 2) && NS >= 2,
                "token tile / TMEM columns");
  static_assert((BOXH * 128) % 1024 == 0, "B box of one MMA: whole 1 KB swizzle atoms");
  static_assert(OFF_PK % 1024 == 0 && B_STAGE % 1024 == 0 && OFF_SC % 128 == 0, "TMA / swizzle alignment");
  static_assert(BYTES + 1024 <= 232448, "shared memory");
  static_assert((NDQ == 1 || NDQ == 2) && (NEPI == 1 || NEPI == 2), "warpgroups");
  // A slot (or a weight stage) that two warpgroups take in alternation would let one's parity
  // wait pass on the phase before the one it needs (the other's use still pending), which breaks
  // the barriers' arrival and transaction counts.
  static_assert(NS % 4 == 0, "A slots per dequantising warpgroup");
};

struct Tile {
  int e, ng, p0, cnt;
};

// Tile g -> (expert, n-group of 256 weight rows, token rows).  Expert e owns tiles
// [tbase[e], tbase[e+1]): ntt token tiles x NG n-groups, n-group fastest, so the pairs running at
// the same time share token rows (and the expert's weights) in L2.  An expert's token rows are
// split into equal chunks (multiples of 32) over its ntt token tiles.
template <int BN>
MOE_DEV Tile decode(int g, const int* tbase, const int* offs, int E, int NG) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tbase[mid] <= g) lo = mid; else hi = mid - 1;
  }
  Tile t;
  t.e = lo;
  const int m = offs[lo + 1] - offs[lo];
  const int ntt = (m + BN - 1) / BN;
  const int local = g - tbase[lo];
  const int tt = local / NG;
  t.ng = local - tt * NG;
  const int chunk = (((m + ntt - 1) / ntt) + 31) & ~31;
  t.p0 = offs[lo] + tt * chunk;
  t.cnt = min(chunk, m - tt * chunk);
  return t;
}

// ------------------------------------------------------------------------- bounded waits

MOE_DEV bool wait_local(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err, uint64_t limit) {
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

// for barriers that CTAs of the cluster arrive on remotely (acquire at cluster scope)
MOE_DEV bool wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err, uint64_t limit) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit) {
      *abort_flag = 1;
      set_error(err, MOE_DEVERR_TIMEOUT);
      return false;
    }
  }
}

MOE_DEV bool warp_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err, uint64_t limit) {
  bool ok = true;
  if (lane_id() == 0) ok = wait_cluster(bar, parity, abort_flag, err, limit);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

MOE_DEV bool warp_wait_local(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err, uint64_t limit) {
  bool ok = true;
  if (lane_id() == 0) ok = wait_local(bar, parity, abort_flag, err, limit);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

MOE_DEV bool wait_counter(const int* p, int need, volatile int* abort_flag, int* err, uint64_t limit) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= need) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit) {
      *abort_flag = 1;
      set_error(err, MOE_DEVERR_TIMEOUT);
      return false;
    }
    __nanosleep(200);
  }
}

// Non-blocking probe of a local barrier's phase (acquire at CTA scope when it has completed).
MOE_DEV bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Arrive on the barrier at offset `bar` of the even CTA (local when this is the even CTA).  The
// remote arrive keeps the instruction's default semantics (release at CTA scope): the data it
// publishes is tensor memory written by tcgen05.st, ordered by the tcgen05 fences around the
// barrier, not generic memory (a release at cluster scope cost ~0.5 us per arrive here).
MOE_DEV void arrive_leader(uint32_t bar, uint32_t rank) {
  if (rank == 0) {
    mbar_arrive(bar);
  } else {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(bar), "r"(0));
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(ra) : "memory");
  }
}

// Address of the barrier at offset `bar` in the even CTA, in the shared::cluster window.
MOE_DEV uint32_t leader_addr(uint32_t bar) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(bar), "r"(0));
  return ra;
}

// Tiled 2D TMA load into this CTA's shared memory whose transaction bytes complete on `bar`, a
// barrier of either CTA of the pair (shared::cluster address).
MOE_DEV void tma_load_2d_pair(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// ------------------------------------------------------------------------- dequantisation, 32 k

// 32 consecutive codes of one weight row (w[j]: codes 8j..8j+7, low nibble first) with the two
// E4M3 block scales in the low two bytes of `sc` -> 16 BF16 pairs; the arithmetic of dequant64.
MOE_DEV void dequant32(const uint32_t (&w)[4], uint32_t sc, float s2, uint32_t (&out)[16]) {
  uint32_t a01, a23;
  e4m3x4_to_f16x2(sc, a01, a23);
  const uint32_t blk[2] = {a01, a01 >> 16};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t h[4];
    e2m1x8_to_f16x2(w[j], h);
#pragma unroll
    for (int q = 0; q < 4; ++q) out[4 * j + q] = dequant_pair(h[q], blk[j >> 1], s2);
  }
}

MOE_DEV void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

MOE_DEV float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// 16 TMEM lanes x 32 columns: register 4i + k of thread t holds lane (t / 4) + 8 (k / 2), column
// 8i + 2 (t % 4) + (k % 2) relative to taddr (the layout of an m16n8 MMA accumulator fragment).
MOE_DEV void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Four 8x8 BF16 matrices, each held as one register per thread in the m16n8 fragment layout
// (thread t: row t / 4, columns 2 (t % 4) and + 1), stored transposed: row j of matrix m goes to
// the 16 bytes at the address thread 8m + j supplies (column j of the fragment).
MOE_DEV void stmatrix_x4_trans(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}

// ------------------------------------------------------------------------- tcgen05, pair form

MOE_DEV void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
MOE_DEV void tmem_relinquish_pair() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;"); }
MOE_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// One 64-k atom on the pair: four k16 MMAs, A (256 rows: 128 in each CTA's TMEM) advancing 8
// columns per step, B (N rows: the first N/2 in the even CTA's shared memory, the rest at the
// same offset in the odd CTA's) advancing 32 bytes (+2 in the descriptor's address field).
MOE_DEV void mma4_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, q;\n .reg .b64 b1, b2, b3;\n .reg .b32 a1, a2, a3;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.b32 q, 0, 0;\n"
      " add.s64 b1, %2, 2;\n add.s64 b2, %2, 4;\n add.s64 b3, %2, 6;\n"
      " add.u32 a1, %1, 8;\n add.u32 a2, %1, 16;\n add.u32 a3, %1, 24;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], [a1], b1, %3, q;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], [a2], b2, %3, q;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], [a3], b3, %3, q;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the barrier at offset `bar` in both CTAs of the pair when every tcgen05 op issued
// so far by this thread has completed.
MOE_DEV void commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap bmap, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);

  int* s_offs = reinterpret_cast<int*>(smem + C::OFF_OFFS);
  int* s_tbase = reinterpret_cast<int*>(smem + C::OFF_TBASE);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  constexpr int NS = C::NS, NW = C::NW, ND = C::ND;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (NS + s); };
  auto w_full = [&](int s) { return bar0 + 8u * (2 * NS + s); };
  auto w_empty = [&](int s) { return bar0 + 8u * (2 * NS + NW + s); };
  auto d_full = [&](int d) { return bar0 + 8u * (2 * NS + 2 * NW + d); };
  auto d_empty = [&](int d) { return bar0 + 8u * (2 * NS + 2 * NW + ND + d); };
  const uint32_t drain_bar = bar0 + 8u * (2 * NS + 2 * NW + 2 * ND);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  int* s_bad = reinterpret_cast<int*>(smem + C::OFF_MISC + 8);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = args.E;
  const uint32_t rank = cluster_ctarank();  // 0: even CTA (issues the MMAs), 1: odd CTA
  const int pid = (int)cluster_id_x();
  const int npairs = (int)cluster_count_x();
  const uint64_t limit = args.wait_ns;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full(s), C::FULL_COUNT);
      mbar_init(empty(s), 1);
    }
    for (int s = 0; s < NW; ++s) {
      mbar_init(w_full(s), 1);
      mbar_init(w_empty(s), 4 * C::NDQ);  // the dequantising warps (every warpgroup reads every stage)
    }
    for (int d = 0; d < ND; ++d) {
      mbar_init(d_full(d), 1);
      mbar_init(d_empty(d), 8 * C::NEPI);  // the epilogue warps of both CTAs
    }
    mbar_init(drain_bar, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == WARP_MMA) {
    tmem_alloc_pair(smem_u32(s_tmem), TMEM_COLS);
    tmem_relinquish_pair();
  }
  // everything above overlaps the previous kernel of the stream; its outputs are read below (a
  // consumer of a producer GEMM's per-expert counters waits per expert instead, and for the whole
  // producer grid at its end)
  if (args.ready_in == nullptr) griddep_wait();
  griddep_launch_dependents();
  for (int i = tid; i <= E; i += C::THREADS) s_offs[i] = args.offsets[i];
  __syncthreads();

  const int NG = args.N / PAIR_ROWS;  // n-groups of 256 weight rows (gate/up: 128 act columns)
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int sum = 0;
    bool bad = false;
    for (int e = e0; e < e1; ++e) {
      const int m = s_offs[e + 1] - s_offs[e];
      if (m < 0) bad = true;
      if (m > 0 && args.packed[e] != nullptr) sum += NG * ((m + C::BN - 1) / C::BN);
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
      if (m > 0 && args.packed[e] != nullptr) run += NG * ((m + C::BN - 1) / C::BN);
    }
    if (lane == 31) s_tbase[E] = bad ? 0 : incl;
    if (lane == 0) *s_bad = bad ? 1 : 0;
    if (bad && lane == 0 && blockIdx.x == 0) set_error(args.err, MOE_DEVERR_BAD_OFFSETS);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int total = s_tbase[E];
  const int KA = args.K / BKA;
  const int KW = args.K / BKW;
  const int half = args.swiglu_half;
  // the tiles of this pair: pid, pid + npairs, ... (both CTAs walk the same list)
  auto tile_at = [&](int i) -> int {
    const int g = pid + i * npairs;
    return g < total ? g : -1;
  };

  if (warp < 4 || warp >= 16) {
    // ------------------------------------------------------------------ epilogue
    // Warpgroup h of NEPI takes the 32-column chunks c0 = 32 (h + NEPI j) of each tile; a warp
    // releases the accumulator after its last chunk's load, and publishes the tile's rows (to a
    // consumer GEMM) after its stores, like every other epilogue warp.
    const int q = warp & 3;
    const int h = warp >= 16 ? 1 : 0;
    uint8_t* stg = smem + C::OFF_EPI + (h * 4 + q) * C::EPI_WARP_BYTES;
    const uint32_t stg_u32 = smem_u32(stg);
    const bool f32 = args.c_dtype == MOE_DTYPE_F32;
    const int esz = f32 ? 4 : 2;
    const int out_cols = half ? half : args.N;
    if (!*s_bad && h == 0) {
      // rows of absent experts are written as zeros (the pages' zeroed routed-output rows)
      const int chunks_per_row = out_cols * esz / 16;
      for (int e = 0; e < E; ++e) {
        if (args.packed[e] != nullptr) continue;
        int nz = 0;
        for (int r = s_offs[e] + blockIdx.x; r < s_offs[e + 1]; r += gridDim.x, ++nz) {
          uint8_t* row = reinterpret_cast<uint8_t*>(args.C) + (size_t)r * args.ldc * esz;
          for (int c = tid; c < chunks_per_row; c += 128) *reinterpret_cast<uint4*>(row + c * 16) = make_uint4(0, 0, 0, 0);
        }
        if (args.ready_out != nullptr && nz > 0) {
          __threadfence();
          __syncwarp();
          if (lane == 0) counter_add_release(args.ready_out + e, nz * args.ready_need);
        }
      }
    }
    // Token rows in expert order (row_src set): the epilogue warps of the grid take the sorted
    // rows round robin (this warp: rows w, w + nw, ...), so the rows are stored roughly in sorted
    // order, the order in which the pairs reach the experts' tiles.  A warp stores 4 KB of a row
    // at a time while its next accumulator is not complete (a complete one waits for at most one
    // such piece), and the rest after its last tile; the stores wait on nothing, so every row is
    // stored even while B producers wait for them.
    const int nepw = 4 * C::NEPI;
    const int row_step = (int)gridDim.x * nepw;
    const int nrows = (args.row_src != nullptr && !*s_bad) ? s_offs[E] : 0;
    const int nv = args.K / 8;  // 16-byte vectors of a row (K % 256 == 0: whole warps)
    int next_row = (int)blockIdx.x * nepw + h * 4 + q, cur_v = 0;
    // store rows until the barrier's phase `parity` completes (poll) or none is left
    auto store_rows = [&](uint32_t bar, uint32_t parity, bool poll) {
      while (next_row < nrows) {
        int stop = 0;
        if (lane == 0) stop = (*s_abort != 0 || (poll && mbar_test_wait(bar, parity))) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, stop, 0)) return;
        const int p = next_row;
        int lo = 0, hi = E - 1;  // the expert of sorted row p: the last e with offs[e] <= p
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (s_offs[mid] <= p) lo = mid; else hi = mid - 1;
        }
        if (args.packed[lo] == nullptr) {  // no tile reads an absent expert's rows
          next_row += row_step;
          continue;
        }
        int tok = __ldg(args.row_ids + p);
        if ((unsigned)tok >= (unsigned)args.row_src_rows) {
          if (lane == 0 && cur_v == 0) set_error(args.err, MOE_DEVERR_BAD_GATHER);
          tok = 0;
        }
        const uint4* src = reinterpret_cast<const uint4*>(args.row_src + (size_t)tok * args.row_src_ld) + cur_v;
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(const_cast<void*>(args.A)) + (size_t)p * args.lda) +
                     cur_v;
        const int n = nv - cur_v;
        uint4 r[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (32 * j + lane < n) r[j] = __ldg(src + 32 * j + lane);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (32 * j + lane < n) dst[32 * j + lane] = r[j];
        cur_v += 256;
        if (cur_v >= nv) {  // the row is stored: publish it
          __threadfence();
          __syncwarp();
          if (lane == 0) counter_add_release(args.rows_ready + lo, 1);
          cur_v = 0;
          next_row += row_step;
        }
      }
    };
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    for (int it = 0;; ++it) {
      const int g = tile_at(it);
      if (g < 0) break;
      const Tile t = decode<C::BN>(g, s_tbase, s_offs, E, NG);
      const int db = it % ND;
      store_rows(d_full(db), (it / ND) & 1, true);
      if (!warp_wait_local(d_full(db), (it / ND) & 1, s_abort, args.err, limit)) break;
      tc_fence_after();
      const uint32_t dcol = (uint32_t)(db * C::BN);
      constexpr int CSTEP = 32 * C::NEPI;
      if (32 * h >= t.cnt) {  // no chunk for this warp in this tile
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_leader(d_empty(db), rank);
      }
      if (half) {
        // fused clamped SwiGLU.  TMEM lanes 32q..32q+15 hold 16 gate rows, 32q+16..32q+31 the
        // matching up rows (act columns a0..a0+15): two 16x256b loads give each thread the gate
        // and the up accumulator of the same (act column, token) pairs.  g and u are rounded to
        // BF16 (the pages' BF16 gate/up buffers), act = silu(min(g, L)) * clamp(u, -L, L) rounded
        // to BF16; transposing matrix stores stage [token][16 act columns] for 16-byte rows out.
        const int a0 = t.ng * 128 + (int)rank * 64 + q * 16;
        for (int c0 = 32 * h; c0 < t.cnt; c0 += CSTEP) {
          uint32_t vg[16], vu[16];
          tmem_ld_16x256b_x4(lane_base + dcol + c0, vg);
          tmem_ld_16x256b_x4(lane_base + (16u << 16) + dcol + c0, vu);
          tmem_wait_ld();
          if (c0 + CSTEP >= t.cnt) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_leader(d_empty(db), rank);
          }
          // register 4i + k: act column (lane / 4) + 8 (k / 2), token 8i + 2 (lane % 4) + (k % 2)
          uint32_t pk[4][2];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float a[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
              a[k] = swiglu_clamped(bf16_round(__uint_as_float(vg[4 * i + k])),
                                    bf16_round(__uint_as_float(vu[4 * i + k])), args.limit);
            pk[i][0] = pack_bf16x2(a[0], a[1]);
            pk[i][1] = pack_bf16x2(a[2], a[3]);
          }
          __syncwarp();
          // matrix m of instruction k2: token block 2 k2 + (m >> 1), act columns 8 (m & 1) + 0..7;
          // this lane addresses row (lane & 7) of matrix lane >> 3; the 16-byte half of a 32-byte
          // staged row is swizzled by bit 2 of the token (conflict-free stores)
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const int m = lane >> 3;
            const int j = 8 * (2 * k2 + (m >> 1)) + (lane & 7);
            const uint32_t addr = stg_u32 + j * 32 + (((m & 1) ^ ((j >> 2) & 1)) << 4);
            stmatrix_x4_trans(addr, pk[2 * k2][0], pk[2 * k2][1], pk[2 * k2 + 1][0], pk[2 * k2 + 1][1]);
          }
          __syncwarp();
          const int rows = min(32, t.cnt - c0);
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int c = lane + 32 * r;
            const int j = c >> 1, p = c & 1;
            if (j < rows) {
              const uint4 val = *reinterpret_cast<const uint4*>(stg + j * 32 + ((p ^ ((j >> 2) & 1)) << 4));
              uint16_t* dst = reinterpret_cast<uint16_t*>(args.C) + (size_t)(t.p0 + c0 + j) * args.ldc + a0 + p * 8;
              *reinterpret_cast<uint4*>(dst) = val;
            }
          }
          __syncwarp();
        }
      } else if (!f32) {
        // BF16 output: two 16x256b loads (TMEM lanes 32q + 0..15 and + 16..31) give each thread
        // pairs of adjacent tokens of one weight row; transposing matrix stores stage [token][32
        // outputs] (64-byte rows, 16-byte chunks swizzled by bits 1-2 of the token) for 16-byte
        // rows out
        const int n0 = t.ng * PAIR_ROWS + (int)rank * BM + q * 32;
        for (int c0 = 32 * h; c0 < t.cnt; c0 += CSTEP) {
          uint32_t va[16], vb[16];
          tmem_ld_16x256b_x4(lane_base + dcol + c0, va);
          tmem_ld_16x256b_x4(lane_base + (16u << 16) + dcol + c0, vb);
          tmem_wait_ld();
          if (c0 + CSTEP >= t.cnt) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_leader(d_empty(db), rank);
          }
          __syncwarp();
          // instruction i: token block i; matrix m: output columns 8m..8m+7 (va: m < 2, vb: m >= 2)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t p0 = pack_bf16x2(__uint_as_float(va[4 * i]), __uint_as_float(va[4 * i + 1]));
            const uint32_t p1 = pack_bf16x2(__uint_as_float(va[4 * i + 2]), __uint_as_float(va[4 * i + 3]));
            const uint32_t p2 = pack_bf16x2(__uint_as_float(vb[4 * i]), __uint_as_float(vb[4 * i + 1]));
            const uint32_t p3 = pack_bf16x2(__uint_as_float(vb[4 * i + 2]), __uint_as_float(vb[4 * i + 3]));
            const int m = lane >> 3;
            const int j = 8 * i + (lane & 7);
            stmatrix_x4_trans(stg_u32 + j * 64 + ((m ^ ((j >> 1) & 3)) << 4), p0, p1, p2, p3);
          }
          __syncwarp();
          const int rows = min(32, t.cnt - c0);
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int c = lane + 32 * r;
            const int j = c >> 2, p = c & 3;
            if (j < rows) {
              const uint4 val = *reinterpret_cast<const uint4*>(stg + j * 64 + ((p ^ ((j >> 1) & 3)) << 4));
              uint16_t* dst = reinterpret_cast<uint16_t*>(args.C) + (size_t)(t.p0 + c0 + j) * args.ldc + n0 + p * 8;
              *reinterpret_cast<uint4*>(dst) = val;
            }
          }
          __syncwarp();
        }
      } else {
        // FP32 output (tests and standalone calls): stage [token][32 outputs] through registers
        const int n0 = t.ng * PAIR_ROWS + (int)rank * BM + q * 32;
        for (int c0 = 32 * h; c0 < t.cnt; c0 += CSTEP) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(lane_base + dcol + c0, v);
          tmem_wait_ld();
          if (c0 + CSTEP >= t.cnt) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_leader(d_empty(db), rank);
          }
          __syncwarp();
          float* sf = reinterpret_cast<float*>(stg);
#pragma unroll
          for (int j = 0; j < 32; ++j) sf[j * 32 + lane] = __uint_as_float(v[j]);
          __syncwarp();
          const int rows = min(32, t.cnt - c0);
          for (int c = lane; c < 32 * 8; c += 32) {
            const int r = c >> 3, cc = c & 7;
            if (r < rows) {
              const uint4 val = *reinterpret_cast<const uint4*>(stg + r * 128 + cc * 16);
              float* dst = reinterpret_cast<float*>(args.C) + (size_t)(t.p0 + c0 + r) * args.ldc + n0 + cc * 4;
              *reinterpret_cast<uint4*>(dst) = val;
            }
          }
          __syncwarp();
        }
      }
      if (args.ready_out != nullptr) {  // this warp's part of the tile's rows is stored
        __threadfence();
        __syncwarp();
        if (lane == 0) counter_add_release(args.ready_out + t.e, t.cnt);
      }
    }
    store_rows(0, 0, false);
  } else if (warp >= 4 && warp < 4 + 4 * C::NDQ) {
    // ------------------------------------------------------------------ dequantisation
    // Warp quadrant q dequantises TMEM lanes 32q..32q+31.  Shared-memory row of lane l: plain
    // GEMM 32q + l; fused SwiGLU (gate rows 0-63, up rows 64-127 of the stage) 16q + l for l < 16,
    // 64 + 16q + (l - 16) otherwise.  Warpgroup wg takes atoms wg*APW .. wg*APW + APW-1 of every
    // weight stage: it reads their packed bytes and scales into registers once, releases the
    // stage, then writes the atoms' BF16 tiles into their TMEM slots and publishes them after one
    // wait for all their stores.
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;
    const int sr = half ? (lane < 16 ? 16 * q + lane : 64 + 16 * q + (lane - 16)) : 32 * q + lane;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    constexpr int APW = C::APW;
    const int a_lo = wg * APW;  // this warpgroup's first atom of each stage
    int wi = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int g = tile_at(it);
      if (g < 0) break;
      const Tile t = decode<C::BN>(g, s_tbase, s_offs, E, NG);
      const float s2 = args.scale2[t.e];
      for (int ks = 0; ks < KW; ++ks, ++wi) {
        const int ws = wi % NW;
        if (!warp_wait_local(w_full(ws), (wi / NW) & 1, s_abort, args.err, limit)) {
          ok = false;
          break;
        }
        // 16-byte chunks 2a, 2a + 1 of the row hold atom a's 64 codes; scale bytes 4a..4a+3
        const uint8_t* pk = smem + C::OFF_PK + ws * C::PK_STAGE + sr * 128;
        uint4 pkv[2 * APW];
#pragma unroll
        for (int c = 0; c < 2 * APW; ++c)
          pkv[c] = *reinterpret_cast<const uint4*>(pk + (((2 * a_lo + c) ^ (sr & 7)) << 4));
        const uint8_t* sc = smem + C::OFF_SC + ws * C::SC_STAGE + sr * 16 + 4 * a_lo;
        uint32_t scw[APW];
        if constexpr (APW == 4) {
          const uint4 v = *reinterpret_cast<const uint4*>(sc);
          scw[0] = v.x, scw[1] = v.y, scw[2] = v.z, scw[3] = v.w;
        } else {
          const uint2 v = *reinterpret_cast<const uint2*>(sc);
          scw[0] = v.x, scw[1] = v.y;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(w_empty(ws));
#pragma unroll
        for (int j = 0; j < APW; ++j) {
          const int a = a_lo + j;
          const int ai = wi * 4 + a;
          const int s = ai % NS;
          if (!warp_wait_local(empty(s), ((ai / NS) & 1) ^ 1, s_abort, args.err, limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ta = tmem_base + lane_addr + C::A_COL + s * 32;
          {
            const uint32_t w4[4] = {pkv[2 * j].x, pkv[2 * j].y, pkv[2 * j].z, pkv[2 * j].w};
            uint32_t out[16];
            dequant32(w4, scw[j], s2, out);
            tmem_st_32x32b_x16(ta, out);
          }
          {
            const uint32_t w4[4] = {pkv[2 * j + 1].x, pkv[2 * j + 1].y, pkv[2 * j + 1].z, pkv[2 * j + 1].w};
            uint32_t out[16];
            dequant32(w4, scw[j] >> 16, s2, out);
            tmem_st_32x32b_x16(ta + 16, out);
          }
        }
        if (!ok) break;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
          for (int j = 0; j < APW; ++j) arrive_leader(full((wi * 4 + a_lo + j) % NS), rank);
      }
    }
    if (!ok) tmem_wait_st();  // no TMEM store of this warp outlives it
  } else if (warp == WARP_WP) {
    // ------------------------------------------------------------------ weight producer
    if (lane == 0) {
      int wi = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int g = tile_at(it);
        if (g < 0) break;
        const Tile t = decode<C::BN>(g, s_tbase, s_offs, E, NG);
        const CUtensorMap* mp = args.wmaps64 + 2 * t.e;
        const CUtensorMap* ms = mp + 1;
        prefetch_tmap(mp);
        prefetch_tmap(ms);
        // this CTA's 128 weight rows as two 64-row boxes
        const int r0 = half ? t.ng * 128 + (int)rank * 64 : t.ng * PAIR_ROWS + (int)rank * BM;
        const int r1 = half ? half + r0 : r0 + 64;
        for (int ks = 0; ks < KW; ++ks, ++wi) {
          const int s = wi % NW;
          if (!wait_local(w_empty(s), ((wi / NW) & 1) ^ 1, s_abort, args.err, limit)) { ok = false; break; }
          mbar_arrive_expect_tx(w_full(s), C::PK_STAGE + C::SC_STAGE);
          const uint32_t pk = sbase + C::OFF_PK + s * C::PK_STAGE;
          const uint32_t sc = sbase + C::OFF_SC + s * C::SC_STAGE;
          tma_load_2d(pk, mp, ks * 128, r0, w_full(s));
          tma_load_2d(pk + 64 * 128, mp, ks * 128, r1, w_full(s));
          tma_load_2d(sc, ms, ks * 16, r0, w_full(s));
          tma_load_2d(sc + 64 * 16, ms, ks * 16, r1, w_full(s));
        }
      }
      if (!ok)
        for (int j = max(0, wi - NW); j < wi; ++j) mbar_wait_drain(w_full(j % NW), (j / NW) & 1);
    }
  } else if (warp == WARP_BP) {
    // ------------------------------------------------------------------ B producer
    // Both CTAs: for each atom, one tiled box of BH rows starting at this CTA's first row p0 +
    // rank*BH of the tile, k [64 kb, 64 kb + 64), whose bytes complete on the even CTA's full
    // barrier; the even CTA's thread arrives there with the bytes of both CTAs' boxes (one box
    // per atom: a producer thread issues a TMA copy only every ~100-150 cycles).  The MMA always
    // has N = BN (accumulator column j = token row p0 + j): rows past the tile's count belong to
    // the next expert (or lie past the tensor and are zero-filled) and reach only accumulator
    // columns the epilogue never stores.  Narrower MMAs for short tiles measured slower.
    if (lane == 0) {
      int ai = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int g = tile_at(it);
        if (g < 0) break;
        const Tile t = decode<C::BN>(g, s_tbase, s_offs, E, NG);
        const int nh = (C::NH == 2 && t.cnt > C::HN) ? 2 : 1;  // MMAs per k16 step for this tile
        const int y0 = t.p0 + (int)rank * C::BOXH;
        if (args.ready_in != nullptr) {
          // the producer GEMM has stored every row of this expert (all its CTA tiles' epilogue warps)
          if (!wait_counter(args.ready_in + t.e, (s_offs[t.e + 1] - s_offs[t.e]) * args.ready_need * 4, s_abort,
                            args.err, limit)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
        }
        if (args.row_src != nullptr) {
          // every row of this expert is stored in expert order (the grid's epilogue warps)
          if (!wait_counter(args.rows_ready + t.e, s_offs[t.e + 1] - s_offs[t.e], s_abort, args.err, limit)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
        }
        for (int kb = 0; kb < KA; ++kb, ++ai) {
          const int s = ai % NS;
          if (!wait_local(empty(s), ((ai / NS) & 1) ^ 1, s_abort, args.err, limit)) { ok = false; break; }
          if (rank == 0) mbar_arrive_expect_tx(full(s), 2u * (uint32_t)(nh * C::BOXH * 128));
          for (int hh = 0; hh < nh; ++hh)
            tma_load_2d_pair(sbase + C::OFF_B + s * C::B_STAGE + hh * (C::BOXH * 128), &bmap, kb * BKA, y0 + hh * C::HN,
                             leader_addr(full(s)));
        }
      }
      if (!ok) {
        // let this CTA's copies land before it leaves: its last NS atoms' boxes complete on the
        // even CTA's barriers, which both CTAs keep alive until the final cluster barrier
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------------------------ MMA issuer (even CTA)
    // The whole warp walks the schedule (its descriptors and addresses stay warp-uniform); one
    // elected lane issues each MMA and commit.
    if (rank == 0) {
      int ai = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int g = tile_at(it);
        if (g < 0) break;
        const int db = it % ND;
        // MMAs per k16 step: the second (accumulator columns HN..) only when the tile has rows there
        const int nh = C::NH == 2 && decode<C::BN>(g, s_tbase, s_offs, E, NG).cnt > C::HN ? 2 : 1;
        if (!warp_wait_cluster(d_empty(db), ((it / ND) & 1) ^ 1, s_abort, args.err, limit)) { ok = false; break; }
        tc_fence_after();
        const uint32_t idesc = make_idesc_bf16(PAIR_ROWS, C::HN);
        const uint64_t bdesc0 = make_sdesc_sw128(sbase + C::OFF_B);
        const uint32_t d_tmem = tmem_base + (uint32_t)(db * C::BN);
        for (int kb = 0; kb < KA; ++kb, ++ai) {
          const int s = ai % NS;
          if (!warp_wait_cluster(full(s), (ai / NS) & 1, s_abort, args.err, limit)) { ok = false; break; }
          tc_fence_after();
          const uint64_t bdesc = bdesc0 + (uint64_t)((s * C::B_STAGE) >> 4);
          if (elect_one()) {
            for (int hh = 0; hh < nh; ++hh)
              mma4_pair(d_tmem + hh * C::HN, tmem_base + C::A_COL + s * 32,
                        bdesc + (uint64_t)((hh * C::BOXH * 128) >> 4), idesc, kb != 0);
            commit_pair(empty(s));
          }
          __syncwarp();
        }
        if (ok) {
          if (elect_one()) commit_pair(d_full(db));
          __syncwarp();
        }
      }
      if (!ok) {  // let every issued MMA finish before TMEM is freed
        if (elect_one()) {
          commit_pair(drain_bar);
          mbar_wait_drain(drain_bar, 0);
        }
        __syncwarp();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA frees TMEM or leaves while its peer may still signal it
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
  // a consumer completes only after its producer grid (stream order for the launches after it)
  if (args.ready_in != nullptr) griddep_wait();
}

// 384-token tiles for experts averaging more than 128 rows: two MMAs of N = 192 per k16 step into
// 384 accumulator columns, four A slots (the two dequantising warpgroups take alternate halves of
// every weight stage), one accumulator.  An expert's m rows take ceil(m / 384) tiles, each
// dequantising the expert's weights once; 256-token tiles (ceil(m / 256) passes, eight A slots)
// measured 7% slower on the 8192-row chunk's gate/up launch and 6% on its down launch.
using CfgWide = Cfg<384, 1, 2, 2, 2>;
using CfgPair = Cfg<128, 2, 2>;   // 128-token tiles, two accumulator buffers

template <class C>
int launch_cfg(const GemmArgs& args, cudaStream_t stream) {
  CUtensorMap bmap;
  {  // A rows (contiguous, expert order): boxes of BN/2 rows x 64 k, 128-byte swizzle
    const cuuint64_t dims[2] = {(cuuint64_t)args.K, (cuuint64_t)args.a_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)args.lda * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BKA, (cuuint32_t)C::BOXH};
    const cuuint32_t estr[2] = {1, 1};
    const int rc = encode_tmap(&bmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(args.A), dims, strides, box,
                               estr, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != MOE_OK) return rc;
  }
  static std::atomic<int> configured[64];
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (!configured[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(pair_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    configured[dev].store(1, std::memory_order_release);
  }
  const int nsm = device_sm_count();
  if (nsm <= 0) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_ALLOC;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = max_clusters[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    cfg.gridDim = dim3(nsm);
    if (cudaOccupancyMaxActiveClusters(&n, pair_gemm_kernel<C>, &cfg) != cudaSuccess || n < 1) return MOE_ERR_CUDA;
    max_clusters[dev].store(n, std::memory_order_relaxed);
  }
  // upper bound of the tiles: every expert's token tiles times the n-groups
  const long long ng = args.N / PAIR_ROWS;
  const long long max_tiles = ng * ((long long)args.E + (args.R + C::BN - 1) / C::BN);
  const int npairs = (int)std::max<long long>(1, std::min<long long>(n, max_tiles));
  cfg.gridDim = dim3(2 * npairs);
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, pair_gemm_kernel<C>, bmap, args) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace pg

bool pair_gemm_shape_ok(int N, int K, int E, int swiglu_half) {
  return N % pg::PAIR_ROWS == 0 && K % pg::BKW == 0 && E <= pg::MAX_E && (swiglu_half == 0 || swiglu_half * 2 == N);
}

// Measured on GLM widths: the pair kernel's wide tiles beat the single-CTA kernel once experts
// average more than 128 rows (the 8192-row Zipf chunk, with 256-token tiles: gate/up 1.81 vs
// 2.33 ms, down 1.14 vs 1.23 ms); at ~100 rows per expert (2048 rows, 160 experts) and below the
// single-CTA kernel's multicast activation tiles are faster (gate/up 0.74 vs 0.95 ms).
bool pair_gemm_preferred(int R, int E) { return (double)R / E > 128.0; }

namespace {
bool wide_tiles(const GemmArgs& args) { return (double)args.R / args.E > 128.0; }
}  // namespace

int pair_gemm_epilogue_groups(const GemmArgs& args) {
  return wide_tiles(args) ? pg::CfgWide::NEPI : pg::CfgPair::NEPI;
}

bool pair_gemm_supported(const GemmArgs& args) {
  return args.wmaps64 != nullptr && args.gather == nullptr && pair_gemm_shape_ok(args.N, args.K, args.E, args.swiglu_half);
}

int pair_gemm_launch(const GemmArgs& args, cudaStream_t stream) {
  if (!pair_gemm_supported(args)) return MOE_ERR_UNSUPPORTED_SHAPE;
  // token-tile width from the mean rows per expert (the distribution itself stays on the device)
  if (wide_tiles(args)) return pg::launch_cfg<pg::CfgWide>(args, stream);
  return pg::launch_cfg<pg::CfgPair>(args, stream);
}

}  // namespace moe
