// common.cuh -- device helpers shared by the sm_103a kernels of the MoE prefill library:
// bounded mbarrier waits, TMA (cp.async.bulk.tensor) loads, tcgen05 (TMEM, MMA) wrappers and
// the packed NVFP4 -> BF16 dequantisation.  Inline PTX only; no CUTLASS/CuTe.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe_prefill.h"

#define MOE_DEV __device__ __forceinline__

namespace moe {

// ------------------------------------------------------------------------------------------------
// device error word (sticky, first error wins)

MOE_DEV void set_error(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

MOE_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

MOE_DEV uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

MOE_DEV uint32_t lane_id() { return threadIdx.x & 31u; }

// true in exactly one lane of the converged warp.  An issuing role (MMA, TMA) that walks its
// schedule with the whole warp and issues from the elected lane keeps its descriptors and
// addresses warp-uniform (measured faster in the CTA-pair GEMM than the loop run by lane 0 alone).
MOE_DEV bool elect_one() {
  uint32_t pred;
  asm volatile("{\n .reg .b32 r;\n .reg .pred p;\n elect.sync r|p, 0xffffffff;\n selp.b32 %0, 1, 0, p;\n}"
               : "=r"(pred));
  return pred != 0;
}

// ------------------------------------------------------------------------------------------------
// mbarrier

MOE_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

MOE_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(bar) : "memory");
}

MOE_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

MOE_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: the thread sleeps until the phase completes or about
// `hint_ns` pass, instead of re-issuing the poll (idle roles then take no issue slots).
MOE_DEV bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Upper bound of any single pipeline wait.  A wait that exceeds it means the pipeline is
// broken; the kernel records MOE_DEVERR_TIMEOUT and unwinds instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kSleepHintNs = 20000u;         // 20 us per suspended poll

// Waits for the phase of `parity` to complete.  Returns false when the CTA-wide abort flag is
// raised (by this or another role) or when the wait limit is exceeded (then it raises the
// flag and records the error).
MOE_DEV bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      set_error(err, MOE_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// Waits until the counter at p (global memory, written by other CTAs or grids) reaches `need`,
// with acquire ordering at GPU scope; the same bounds as mbar_wait.
MOE_DEV bool wait_counter_geq(const int* p, int need, volatile int* abort_flag, int* err) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= need) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      set_error(err, MOE_DEVERR_TIMEOUT);
      return false;
    }
    __nanosleep(200);
  }
}

// Adds v to the counter at p with release ordering at GPU scope.
MOE_DEV void counter_add_release(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Orders this thread's earlier generic-proxy accesses (e.g. an acquire of data that other threads
// stored) before its later async-proxy (TMA) accesses of global memory.
MOE_DEV void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Cluster-scope mbarrier operations on the barrier at the same shared offset in CTA `rank`:
// arrive with release (orders this thread's earlier st.shared::cluster), and a local wait with
// acquire at cluster scope.
MOE_DEV void mbar_arrive_remote(uint32_t bar, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(bar), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(ra) : "memory");
}
MOE_DEV bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, "
      "p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
MOE_DEV bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      set_error(err, MOE_DEVERR_TIMEOUT);
      return false;
    }
  }
}
MOE_DEV void st_shared_cluster_u32(uint32_t local_addr, uint32_t rank, uint32_t v) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(ra), "r"(v) : "memory");
}

// Wait used while unwinding: bounded, ignores the abort flag.
MOE_DEV bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

MOE_DEV void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

MOE_DEV void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------------------------------------
// TMA

MOE_DEV void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

MOE_DEV void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Four rows (y0..y3) of a box one row high, written to four consecutive box slots at dst.
MOE_DEV void tma_gather4(uint32_t dst, const void* tmap, int x, int y0, int y1, int y2, int y3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar)
      : "memory");
}

// Multicast forms: the same shared-memory offset and mbarrier offset in every CTA of `mask`
// (thread-block cluster) receive the data and its complete_tx.
MOE_DEV void tma_load_2d_mc(uint32_t dst, const void* tmap, int x, int y, uint32_t bar, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar), "h"(mask)
      : "memory");
}

MOE_DEV void tma_gather4_mc(uint32_t dst, const void* tmap, int x, int y0, int y1, int y2, int y3, uint32_t bar,
                            uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.multicast::cluster "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar), "h"(mask)
      : "memory");
}

// ------------------------------------------------------------------------------------------------
// thread-block clusters

MOE_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
MOE_DEV uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
MOE_DEV uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
MOE_DEV uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Store to the shared memory of CTA `rank` of the cluster, at the offset of `local_addr` in ours.
MOE_DEV void st_shared_cluster_f32(uint32_t local_addr, uint32_t rank, float v) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ra), "f"(v) : "memory");
}
// All threads of all CTAs of the cluster (also orders this CTA's shared-memory writes, e.g.
// mbarrier initialisation, before the other CTAs' later accesses).
MOE_DEV void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------------------------------------------
// tcgen05 (tensor memory and 5th-generation MMA), cta_group::1

MOE_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
MOE_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;"); }
MOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
MOE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem desc]; kind::f16 (BF16 operands, FP32 accumulator).
// One 64-k atom: four k16 MMAs; A advances 8 TMEM columns (16 BF16 k) per step and B's
// descriptor start address 32 bytes (+2 in its address >> 4 field) inside the 128-byte swizzle
// row.  The first step overwrites D unless `accumulate`; the others accumulate.
MOE_DEV void mma4_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, q;\n .reg .b64 b1, b2, b3;\n .reg .b32 a1, a2, a3;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.b32 q, 0, 0;\n"
      " add.s64 b1, %2, 2;\n add.s64 b2, %2, 4;\n add.s64 b3, %2, 6;\n"
      " add.u32 a1, %1, 8;\n add.u32 a2, %1, 16;\n add.u32 a3, %1, 24;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, q;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier completes one arrival once every tcgen05 op issued so far by this thread is done.
MOE_DEV void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// ... on the mbarrier at the same offset in every CTA of `mask`.
MOE_DEV void mma_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   bar),
               "h"(mask)
               : "memory");
}

MOE_DEV void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
MOE_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

MOE_DEV void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
MOE_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Instruction descriptor of tcgen05.mma kind::f16: D FP32 (bits 4-5 = 1), A BF16 (bits 7-9 = 1),
// B BF16 (bits 10-12 = 1), both K-major (bits 15/16 = 0), N>>3 at bits 17-22, M>>4 at bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a K-major operand in the canonical 128-byte-swizzled
// layout: rows of 128 B, 8-row groups 1024 B apart (stride byte offset), leading byte offset
// unused for this layout (encoded 1), descriptor version 1 (bit 46), swizzle mode 2 (128 B).
MOE_DEV uint64_t make_sdesc_sw128(uint32_t smem_addr) {
  return (uint64_t)((smem_addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// ------------------------------------------------------------------------------------------------
// NVFP4 -> BF16 dequantisation of 64 consecutive k of one weight row.
//
// Value of code c with block scale byte a ("Module forward_prefill_gemm", "What is NOT
// bit-identical", item 2): bf16( fp32( fp32(E2M1[c] * e4m3(a)) * scale2 ) ).
// E2M1[c] * e4m3(a) has at most 6 significant bits and lies in [2^-10, 2688], so it is exact
// in f16: the two packed converts and the f16 multiply are exact, the fp32 multiply by scale2
// is the one rounding before the BF16 rounding -- the same two roundings as the definition.
//
// w[j] holds codes 8j..8j+7 (byte b of w[j]: code 8j+2b in the low nibble, 8j+2b+1 in the high
// nibble); sc holds the 4 E4M3 scale bytes of the four 16-code blocks (byte i = block i).
// out[m] = BF16 pair (elements 2m, 2m+1), the lower k in the low half.
MOE_DEV uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

MOE_DEV void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

MOE_DEV void e4m3x4_to_f16x2(uint32_t sc, uint32_t& a01, uint32_t& a23) {
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
      : "=r"(a01), "=r"(a23)
      : "r"(sc));
}

// lut (f16 pair) * scale (one f16) -> two exact fp32 products (mixed-precision FMA with a -0
// addend, so code 8 keeps its sign as -0), times
// scale2 (packed fp32 multiply, the one rounding), -> BF16 pair (round to nearest even).
MOE_DEV uint32_t dequant_pair(uint32_t lut2, uint32_t scale_h, float s2) {
  uint32_t out;
  asm("{\n .reg .b16 lo, hi, a, unused;\n .reg .f32 flo, fhi;\n .reg .b64 p, q, s;\n"
      " mov.b32 {lo, hi}, %1;\n mov.b32 {a, unused}, %2;\n"
      " fma.rn.f32.f16 flo, lo, a, 0f80000000;\n fma.rn.f32.f16 fhi, hi, a, 0f80000000;\n"
      " mov.b64 p, {flo, fhi};\n mov.b64 s, {%3, %3};\n mul.rn.f32x2 q, p, s;\n"
      " mov.b64 {flo, fhi}, q;\n cvt.rn.bf16x2.f32 %0, fhi, flo;\n}"
      : "=r"(out)
      : "r"(lut2), "r"(scale_h), "f"(s2));
  return out;
}

// f16 pair (two E2M1 values) times one f16 (the block scale, low half of scale_h): two exact
// FP32 products (mixed-precision FMA with a -0 addend, as in dequant_pair).
MOE_DEV void f16x2_times_f16(uint32_t lut2, uint32_t scale_h, float& lo, float& hi) {
  asm("{\n .reg .b16 l, h, a, unused;\n mov.b32 {l, h}, %2;\n mov.b32 {a, unused}, %3;\n"
      " fma.rn.f32.f16 %0, l, a, 0f80000000;\n fma.rn.f32.f16 %1, h, a, 0f80000000;\n}"
      : "=f"(lo), "=f"(hi)
      : "r"(lut2), "r"(scale_h));
}

MOE_DEV void dequant64(const uint32_t (&w)[8], uint32_t sc, float s2, uint32_t (&out)[32]) {
  uint32_t a01, a23;
  e4m3x4_to_f16x2(sc, a01, a23);
  // block b's f16 scale in the low half of blk[b]
  const uint32_t blk[4] = {a01, a01 >> 16, a23, a23 >> 16};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t h[4];
    e2m1x8_to_f16x2(w[j], h);
#pragma unroll
    for (int q = 0; q < 4; ++q) out[4 * j + q] = dequant_pair(h[q], blk[j >> 1], s2);
  }
}

// ------------------------------------------------------------------------------------------------
// programmatic dependent launch: kernels launched with programmatic stream serialization may
// start before the previous kernel of the stream has finished.  griddep_wait() blocks until that
// kernel has completed and its memory is visible (a no-op without the launch attribute);
// griddep_launch_dependents() lets the next kernel be scheduled (it still waits for our end).

MOE_DEV void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEV void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------------------------------------
// clamped SwiGLU of one element: silu(min(g, L)) * clamp(u, -L, L), silu(z) = z / (1 + e^-z)
// ("glm5next_mlp/forward.rs" (metrale), swiglu_rows).  Shared by the standalone SwiGLU kernel,
// the fused gate/up GEMM epilogue and the small-row products.  The exponential and the division
// use the hardware approximations (a few FP32 ulp; the result is rounded to BF16, 2^-9): the
// accurate forms cost ~10% of the fused gate/up GEMM at 256 rows, where the epilogue shares the
// sub-partitions with the dequantisation warps.  For z -> -inf, 1 + e^-z overflows to +inf and
// the quotient is -0, the limit of silu.

MOE_DEV float swiglu_clamped(float g, float u, float L) {
  const float gm = fminf(g, L);
  const float uc = fminf(fmaxf(u, -L), L);
  return __fdividef(gm, 1.0f + __expf(-gm)) * uc;
}

// ------------------------------------------------------------------------------------------------
// BF16 helpers for the SIMT kernels

MOE_DEV float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
MOE_DEV float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
MOE_DEV uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t out;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
  return out;
}

}  // namespace moe
