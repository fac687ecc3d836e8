// api.cu -- the C ABI (include/moe_prefill.h): argument checks, NVFP4 expert tables (per-expert
// TMA descriptors built once at load), workspace layout, launches, and the fused forward.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

struct moe_expert_table {
  int E, N, K;
  int device;
  CUtensorMap* d_maps;    // [E][2] (128-row boxes)
  CUtensorMap* d_maps64;  // [E][2] (64-row boxes, the CTA-pair kernel)
  const void** d_packed;  // [E]
  const void** d_scales;  // [E]
  float* d_scale2;        // [E]
};

namespace moe {

__device__ int g_device_error;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// Filled once per device under g_mu; g_arch_ok is published last (release) and read first
// (acquire), so a thread that sees 1 also sees the error word and the SM count.
int* g_err_addr[kMaxDevices] = {nullptr};
int g_sm_count[kMaxDevices] = {0};
std::atomic<int> g_arch_ok[kMaxDevices];  // 0 unknown, 1 ok, -1 not sm_103
std::atomic<PFN_cuTensorMapEncodeTiled_v12000> g_encode{nullptr};

int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

// Once per device: the compute capability check, the SM count and the error word address.
int ensure_device() {
  const int d = current_device();
  if (d < 0) return MOE_ERR_CUDA;
  if (g_arch_ok[d].load(std::memory_order_acquire) == 1) return MOE_OK;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_arch_ok[d].load(std::memory_order_relaxed) == 0) {
    cudaDeviceProp p;
    if (cudaGetDeviceProperties(&p, d) != cudaSuccess) return MOE_ERR_CUDA;
    if (!(p.major == 10 && p.minor == 3)) {
      g_arch_ok[d].store(-1, std::memory_order_release);
    } else {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_device_error) != cudaSuccess) return MOE_ERR_CUDA;
      g_err_addr[d] = static_cast<int*>(addr);
      g_sm_count[d] = p.multiProcessorCount;
      g_arch_ok[d].store(1, std::memory_order_release);
    }
  }
  return g_arch_ok[d].load(std::memory_order_relaxed) == 1 ? MOE_OK : MOE_ERR_NOT_BUILT_FOR_DEVICE;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Where p points, for the current device: kMemDevice (device or managed memory), kMemHost (host
// memory kernels can read and write: page-locked host memory, which unified addressing maps at
// the same address, or any host memory on a device with pageable memory access, a coherent
// CPU-GPU node), or kMemNone.  The pointer query is not a stream operation, so it runs in relaxed
// capture mode while a CUDA graph is being captured.
enum MemKind { kMemNone, kMemDevice, kMemHost };

MemKind memory_kind(const void* p) {
  cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
  if (cudaThreadExchangeStreamCaptureMode(&mode) != cudaSuccess) return kMemNone;
  cudaPointerAttributes a{};
  const cudaError_t e = cudaPointerGetAttributes(&a, p);
  cudaThreadExchangeStreamCaptureMode(&mode);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return kMemNone;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return kMemDevice;
  if (a.type == cudaMemoryTypeHost) return a.devicePointer == p ? kMemHost : kMemNone;
  int pageable = 0;
  const int d = current_device();
  return d >= 0 && cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, d) == cudaSuccess &&
                 pageable != 0
             ? kMemHost
             : kMemNone;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

int device_sm_count() {
  const int d = current_device();
  return d < 0 ? 0 : g_sm_count[d];
}

int* device_error_word() {
  const int d = current_device();
  return d < 0 ? nullptr : g_err_addr[d];
}

int encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, void* base, const cuuint64_t* dims,
                const cuuint64_t* strides_bytes, const cuuint32_t* box, const cuuint32_t* elem_strides,
                CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = g_encode.load(std::memory_order_acquire);
  if (encode == nullptr) {
    std::lock_guard<std::mutex> lk(g_mu);
    encode = g_encode.load(std::memory_order_relaxed);
    if (encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return MOE_ERR_CUDA;
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      g_encode.store(encode, std::memory_order_release);
    }
  }
  const CUresult r = encode(map, dtype, (cuuint32_t)rank, base, dims, strides_bytes, box, elem_strides,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace moe

// Which grouped GEMM kernel runs: the CTA-pair kernel wherever its shapes allow (the default), or
// the single-CTA kernel (a debug/test setting, moe_debug_set_gemm_kernel).
namespace moe {
namespace {
std::atomic<int> g_gemm_kernel{MOE_GEMM_KERNEL_AUTO};
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};
}  // namespace
uint64_t gemm_wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
}  // namespace moe

using namespace moe;

// ==================================================================================================
// C ABI

extern "C" {

const char* moe_version(void) { return "moe_prefill_nvfp4_gb300 0.1 (sm_103a)"; }

const char* moe_status_string(int s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
    case MOE_ERR_NOT_BUILT_FOR_DEVICE: return "MOE_ERR_NOT_BUILT_FOR_DEVICE";
    case MOE_ERR_SCRATCH_LIMIT: return "MOE_ERR_SCRATCH_LIMIT";
    default: return "MOE_ERR_UNKNOWN";
  }
}

// ------------------------------------------------------------------------------------------ tables

int moe_expert_table_create(const void* const* packed, const void* const* scales, const float* scale2, int E, int N,
                            int K, moe_expert_table** out) {
  if (out == nullptr || packed == nullptr || scales == nullptr || scale2 == nullptr) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (E < 1 || E > 512 || N < 8 || N % 8 != 0 || K < 256 || K % 256 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((long long)N * K / 2 > (1ll << 40)) return MOE_ERR_UNSUPPORTED_SHAPE;
  int any = 0;
  for (int e = 0; e < E; ++e) {
    if (packed[e] == nullptr) continue;
    if (scales[e] == nullptr || !aligned16(packed[e]) || !aligned16(scales[e])) return MOE_ERR_INVALID_ARG;
    any = 1;
  }
  if (!any) return MOE_ERR_INVALID_ARG;
  int rc = ensure_device();
  if (rc != MOE_OK) return rc;

  // two tensor maps per expert and box height: 128-row boxes (single-CTA kernel), 64-row boxes
  // (CTA-pair kernel)
  std::vector<CUtensorMap> maps(2 * (size_t)E), maps64(2 * (size_t)E);
  std::memset(maps.data(), 0, maps.size() * sizeof(CUtensorMap));
  std::memset(maps64.data(), 0, maps64.size() * sizeof(CUtensorMap));
  for (int e = 0; e < E; ++e) {
    if (packed[e] == nullptr) continue;
    const cuuint32_t estr[2] = {1, 1};
    for (int v = 0; v < 2; ++v) {
      const cuuint32_t rows = v == 0 ? 128u : 64u;
      std::vector<CUtensorMap>& dst = v == 0 ? maps : maps64;
      {  // packed nibbles [N, K/2] bytes: box 128 B x rows, 128-byte swizzle
        const cuuint64_t dims[2] = {(cuuint64_t)K / 2, (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)K / 2};
        const cuuint32_t box[2] = {128, rows};
        rc = encode_tmap(&dst[2 * e], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(packed[e]), dims, strides,
                         box, estr, CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc != MOE_OK) return rc;
      }
      {  // E4M3 scales [N, K/16] bytes: box 16 B x rows
        const cuuint64_t dims[2] = {(cuuint64_t)K / 16, (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)K / 16};
        const cuuint32_t box[2] = {16, rows};
        rc = encode_tmap(&dst[2 * e + 1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(scales[e]), dims,
                         strides, box, estr, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (rc != MOE_OK) return rc;
      }
    }
  }
  moe_expert_table* t = new moe_expert_table();
  t->E = E;
  t->N = N;
  t->K = K;
  t->device = current_device();
  t->d_maps = nullptr;
  t->d_maps64 = nullptr;
  t->d_packed = nullptr;
  t->d_scales = nullptr;
  t->d_scale2 = nullptr;
  bool ok = cudaMalloc(&t->d_maps, maps.size() * sizeof(CUtensorMap)) == cudaSuccess &&
            cudaMalloc(&t->d_maps64, maps64.size() * sizeof(CUtensorMap)) == cudaSuccess &&
            cudaMalloc(&t->d_packed, (size_t)E * sizeof(void*)) == cudaSuccess &&
            cudaMalloc(&t->d_scales, (size_t)E * sizeof(void*)) == cudaSuccess &&
            cudaMalloc(&t->d_scale2, (size_t)E * sizeof(float)) == cudaSuccess;
  ok = ok && cudaMemcpy(t->d_maps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice) == cudaSuccess;
  ok = ok &&
       cudaMemcpy(t->d_maps64, maps64.data(), maps64.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice) == cudaSuccess;
  ok = ok && cudaMemcpy(t->d_packed, packed, (size_t)E * sizeof(void*), cudaMemcpyHostToDevice) == cudaSuccess;
  ok = ok && cudaMemcpy(t->d_scales, scales, (size_t)E * sizeof(void*), cudaMemcpyHostToDevice) == cudaSuccess;
  ok = ok && cudaMemcpy(t->d_scale2, scale2, (size_t)E * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess;
  if (!ok) {
    moe_expert_table_destroy(t);
    return MOE_ERR_CUDA;
  }
  *out = t;
  return MOE_OK;
}

int moe_expert_table_destroy(moe_expert_table* t) {
  if (t == nullptr) return MOE_OK;
  cudaDeviceSynchronize();
  cudaFree(t->d_maps);
  cudaFree(t->d_maps64);
  cudaFree(t->d_packed);
  cudaFree(t->d_scales);
  cudaFree(t->d_scale2);
  delete t;
  return MOE_OK;
}

int moe_expert_table_shape(const moe_expert_table* t, int* E, int* N, int* K) {
  if (t == nullptr) return MOE_ERR_INVALID_ARG;
  if (E) *E = t->E;
  if (N) *N = t->N;
  if (K) *K = t->K;
  return MOE_OK;
}

// ------------------------------------------------------------------------------------------ routing

int moe_router_logits(const uint16_t* x, const uint16_t* w_router, int T, int H, int E, float* logits, void* stream) {
  if (x == nullptr || w_router == nullptr || logits == nullptr) return MOE_ERR_INVALID_ARG;
  if (T < 1 || E < 1 || E > 1024 || H < 8 || H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(w_router) || (reinterpret_cast<uintptr_t>(logits) & 3u)) return MOE_ERR_INVALID_ARG;
  const int rc = ensure_device();
  if (rc != MOE_OK) return rc;
  return router_logits_launch(x, w_router, T, H, E, logits, as_stream(stream));
}

int moe_route_topk(const float* logits, const float* bias, int T, int E, int k, int renormalize, float routed_scale,
                   int32_t* ids, float* wts, void* stream) {
  if (logits == nullptr || ids == nullptr || wts == nullptr) return MOE_ERR_INVALID_ARG;
  if (T < 1 || E < 1 || E > 1024 || k < 1 || k > E || k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int rc = ensure_device();
  if (rc != MOE_OK) return rc;
  return route_topk_launch(logits, bias, T, E, k, renormalize, routed_scale, ids, wts, device_error_word(),
                           as_stream(stream));
}

// ------------------------------------------------------------------------------------------ sort

size_t moe_sort_workspace_bytes(int T, int k, int E) {
  if (T < 1 || k < 1 || E < 1 || E > 1024 || (long long)T * k >= (1ll << 31)) return 0;
  return sort_scratch_bytes(T * k, E);
}

int moe_sort_by_expert(const int32_t* ids, int T, int k, int E, int32_t* sorted_token_ids, int32_t* sorted_expert_ids,
                       int32_t* expert_offsets, int32_t* token_to_perm, void* ws, size_t ws_bytes, void* stream) {
  if (!ids || !sorted_token_ids || !sorted_expert_ids || !expert_offsets || !token_to_perm || !ws)
    return MOE_ERR_INVALID_ARG;
  if (T < 1 || k < 1 || k > 32 || E < 1 || E > 1024 || (long long)T * k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (ws_bytes < moe_sort_workspace_bytes(T, k, E)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  int rc = ensure_device();
  if (rc != MOE_OK) return rc;
  const int R = T * k;
  int32_t* cnt = static_cast<int32_t*>(ws);
  return sort_launch(ids, R, k, E, cnt, sorted_token_ids, sorted_expert_ids, expert_offsets, token_to_perm,
                     device_error_word(), as_stream(stream));
}

// Fixed scratch of moe_sort_by_expert_noalloc: part of the module's device image, one copy per
// device, so no call allocates.  Its address is looked up once per device.
static __device__ __align__(256) int32_t g_sort_noalloc_scratch[MOE_SORT_NOALLOC_MAX_INTS];

namespace {
int32_t* g_sort_noalloc_addr[kMaxDevices] = {nullptr};

int sort_noalloc_scratch(int32_t** out) {
  const int d = current_device();
  if (d < 0) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sort_noalloc_addr[d] == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_sort_noalloc_scratch) != cudaSuccess || addr == nullptr) return MOE_ERR_CUDA;
    g_sort_noalloc_addr[d] = static_cast<int32_t*>(addr);
  }
  *out = g_sort_noalloc_addr[d];
  return MOE_OK;
}
}  // namespace

int moe_sort_by_expert_noalloc(const int32_t* ids, int T, int k, int E, int32_t* sorted_token_ids,
                               int32_t* sorted_expert_ids, int32_t* expert_offsets, int32_t* token_to_perm,
                               void* stream) {
  if (!ids || !sorted_token_ids || !sorted_expert_ids || !expert_offsets || !token_to_perm) return MOE_ERR_INVALID_ARG;
  if (T < 1 || k < 1 || k > 32 || E < 1 || E > 1024 || (long long)T * k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (sort_scratch_bytes(T * k, E) > sizeof(g_sort_noalloc_scratch)) return MOE_ERR_SCRATCH_LIMIT;
  int rc = ensure_device();
  if (rc != MOE_OK) return rc;
  int32_t* cnt = nullptr;
  rc = sort_noalloc_scratch(&cnt);
  if (rc != MOE_OK) return rc;
  const int R = T * k;
  return sort_launch(ids, R, k, E, cnt, sorted_token_ids, sorted_expert_ids, expert_offsets, token_to_perm,
                     device_error_word(), as_stream(stream));
}

// ------------------------------------------------------------------------------------------ GEMM

// swiglu_half = 0: plain GEMM into C [R, ldc >= N]; otherwise the fused SwiGLU epilogue with
// I = swiglu_half = N / 2 writing BF16 act [R, ldc >= I].
// tiles_per_row (out, optional): how many CTA tiles of this launch cover one output row (the
// producer side of the forward's GEMM overlap)
static int gemm_checked(const uint16_t* A, int a_rows, int lda, const int32_t* gather_ids, const moe_expert_table* W,
                        const int32_t* expert_offsets, int R, void* C, int ldc, int c_dtype, cudaStream_t st,
                        int swiglu_half = 0, float limit = 0.f, int* ready_out = nullptr,
                        const int* ready_in = nullptr, int ready_need = 0, int* tile_counter = nullptr,
                        int* tiles_per_row = nullptr, bool no_multicast = false,
                        const uint16_t* row_src = nullptr, int row_src_rows = 0, const int32_t* row_ids = nullptr,
                        int* rows_ready = nullptr) {
  if (A == nullptr || W == nullptr || expert_offsets == nullptr || C == nullptr) return MOE_ERR_INVALID_ARG;
  if (c_dtype != MOE_DTYPE_BF16 && c_dtype != MOE_DTYPE_F32) return MOE_ERR_INVALID_ARG;
  if (swiglu_half && (c_dtype != MOE_DTYPE_BF16 || W->N != 2 * swiglu_half || swiglu_half % 128 != 0))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  const int out_cols = swiglu_half ? swiglu_half : W->N;
  if (a_rows < 1 || R < 1 || lda < W->K || lda % 8 != 0 || ldc < out_cols || ldc % 8 != 0)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(A) || !aligned16(C)) return MOE_ERR_INVALID_ARG;
  int rc = ensure_device();
  if (rc != MOE_OK) return rc;
  if (current_device() != W->device) return MOE_ERR_INVALID_ARG;
  GemmArgs a;
  a.wmaps = W->d_maps;
  a.packed = W->d_packed;
  a.scale2 = W->d_scale2;
  a.gather = gather_ids;
  a.offsets = expert_offsets;
  a.C = C;
  a.E = W->E;
  a.N = W->N;
  a.K = W->K;
  a.R = R;
  a.a_rows = a_rows;
  a.ldc = ldc;
  a.c_dtype = c_dtype;
  a.err = device_error_word();
  a.swiglu_half = swiglu_half;
  a.limit = limit;
  a.ready_out = ready_out;
  a.ready_in = ready_in;
  a.ready_need = ready_need;
  a.tile_counter = tile_counter;
  a.wmaps64 = W->d_maps64;
  a.A = A;
  a.lda = lda;
  a.wait_ns = gemm_wait_limit_ns();
  a.max_cluster = no_multicast ? 1 : 8;
  a.row_src = row_src;
  a.row_src_rows = row_src_rows;
  a.row_src_ld = lda;
  a.row_ids = row_ids;
  a.rows_ready = rows_ready;
  const int mode = g_gemm_kernel.load(std::memory_order_relaxed);
  const bool pair = pair_gemm_supported(a) &&
                    (mode == MOE_GEMM_KERNEL_PAIR || (mode == MOE_GEMM_KERNEL_AUTO && pair_gemm_preferred(R, W->E)));
  if (mode == MOE_GEMM_KERNEL_PAIR && !pair) return MOE_ERR_UNSUPPORTED_SHAPE;
  // only the pair kernel stores its rows in expert order itself
  if (row_src != nullptr && (!pair || row_ids == nullptr || rows_ready == nullptr || !aligned16(row_src)))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  // CTA tiles of this launch covering one output row (counted once per epilogue warpgroup): the
  // producer side of the forward's GEMM overlap publishes per tile and warp (and, for absent
  // experts' zero rows, this many per row and warp)
  const int tiles = pair ? 2 * (W->N / 256) * pair_gemm_epilogue_groups(a) : (W->N + 255) / 256;
  if (tiles_per_row) *tiles_per_row = tiles;
  if (ready_out != nullptr) a.ready_need = tiles;
  if (pair) return pair_gemm_launch(a, st);
  return grouped_gemm_launch(a, A, a_rows, lda, st);
}

int moe_w4a16_grouped_gemm(const uint16_t* A, int a_rows, int lda, const int32_t* gather_ids,
                           const moe_expert_table* W, const int32_t* expert_offsets, int R, void* C, int ldc,
                           int c_dtype, void* stream) {
  return gemm_checked(A, a_rows, lda, gather_ids, W, expert_offsets, R, C, ldc, c_dtype, as_stream(stream));
}

int moe_w4a16_grouped_gemm_swiglu(const uint16_t* A, int a_rows, int lda, const int32_t* gather_ids,
                                  const moe_expert_table* W, const int32_t* expert_offsets, int R, uint16_t* act,
                                  int ld_act, float limit, void* stream) {
  if (W == nullptr) return MOE_ERR_INVALID_ARG;
  if (!(limit > 0.f)) return MOE_ERR_INVALID_ARG;
  return gemm_checked(A, a_rows, lda, gather_ids, W, expert_offsets, R, act, ld_act, MOE_DTYPE_BF16, as_stream(stream),
                      W->N / 2, limit);
}

static int gemv_checked(const uint16_t* A, int a_rows, int lda, const int32_t* gather_ids, const moe_expert_table* W,
                        const int32_t* expert_offsets, int R, uint16_t* C, int ldc, int swiglu_half, float limit,
                        cudaStream_t st) {
  if (A == nullptr || W == nullptr || expert_offsets == nullptr || C == nullptr) return MOE_ERR_INVALID_ARG;
  if (swiglu_half && (W->N != 2 * swiglu_half || !(limit > 0.f))) return MOE_ERR_INVALID_ARG;
  const int out_cols = swiglu_half ? swiglu_half : W->N;
  if (a_rows < 1 || R < 1 || lda < W->K || lda % 8 != 0 || ldc < out_cols) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(A)) return MOE_ERR_INVALID_ARG;
  int rc = ensure_device();
  if (rc != MOE_OK) return rc;
  if (current_device() != W->device) return MOE_ERR_INVALID_ARG;
  SmallRowsArgs a;
  a.A = A;
  a.lda = lda;
  a.a_rows = a_rows;
  a.gather = gather_ids;
  a.packed = W->d_packed;
  a.scales = W->d_scales;
  a.scale2 = W->d_scale2;
  a.offsets = expert_offsets;
  a.E = W->E;
  a.N = W->N;
  a.K = W->K;
  a.R = R;
  a.swiglu_half = swiglu_half;
  a.limit = limit;
  a.C = C;
  a.ldc = ldc;
  a.err = device_error_word();
  return small_rows_launch(a, st);
}

int moe_w4a16_grouped_gemv(const uint16_t* A, int a_rows, int lda, const int32_t* gather_ids,
                           const moe_expert_table* W, const int32_t* expert_offsets, int R, uint16_t* C, int ldc,
                           void* stream) {
  return gemv_checked(A, a_rows, lda, gather_ids, W, expert_offsets, R, C, ldc, 0, 0.f, as_stream(stream));
}

int moe_w4a16_grouped_gemv_swiglu(const uint16_t* A, int a_rows, int lda, const int32_t* gather_ids,
                                  const moe_expert_table* W, const int32_t* expert_offsets, int R, uint16_t* act,
                                  int ld_act, float limit, void* stream) {
  if (W == nullptr) return MOE_ERR_INVALID_ARG;
  return gemv_checked(A, a_rows, lda, gather_ids, W, expert_offsets, R, act, ld_act, W->N / 2, limit,
                      as_stream(stream));
}

int moe_dequant_nvfp4(const void* packed, const void* scales, float scale2, int N, int K, uint16_t* out,
                      void* stream) {
  if (packed == nullptr || scales == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
  if (N < 1 || K < 64 || K % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(packed) || !aligned16(out) || (reinterpret_cast<uintptr_t>(scales) & 3u) || (K / 16) % 4 != 0)
    return MOE_ERR_INVALID_ARG;
  const int rc = ensure_device();
  if (rc != MOE_OK) return rc;
  return dequant_launch(static_cast<const uint8_t*>(packed), static_cast<const uint8_t*>(scales), scale2, N, K, out,
                        as_stream(stream));
}

// ------------------------------------------------------------------------------------------ elementwise

int moe_swiglu_clamp(const uint16_t* gate, const uint16_t* up, int64_t rows, int64_t width, int64_t ld_in,
                     uint16_t* out, int64_t ld_out, float limit, void* stream) {
  if (gate == nullptr || up == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
  if (rows < 0 || width < 1 || width % 8 != 0 || ld_in % 8 != 0 || ld_out % 8 != 0 || ld_in < width || ld_out < width)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(gate) || !aligned16(up) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  const int rc = ensure_device();
  if (rc != MOE_OK) return rc;
  return swiglu_launch(gate, up, rows, width, ld_in, out, ld_out, limit, as_stream(stream));
}

int moe_combine_indexed(const uint16_t* Y, const int32_t* token_to_perm, const float* wts, const uint16_t* shared_out,
                        int T, int k, int H, uint16_t* out, void* stream) {
  if (Y == nullptr || token_to_perm == nullptr || wts == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
  if (T < 1 || k < 1 || k > 32 || H < 8 || H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(Y) || !aligned16(out) || (shared_out && !aligned16(shared_out))) return MOE_ERR_INVALID_ARG;
  const int rc = ensure_device();
  if (rc != MOE_OK) return rc;
  return combine_launch(Y, token_to_perm, wts, shared_out, T, k, H, out, as_stream(stream));
}

// ------------------------------------------------------------------------------------ shared expert

size_t moe_shared_expert_workspace_bytes(int T, int H, int I) {
  if (T < 1 || H < 8 || H % 8 != 0 || I < 8 || I % 8 != 0) return 0;
  size_t a, b;
  return shared_expert_ws_layout(T, I, &a, &b);
}

int moe_shared_expert_forward(const uint16_t* x, int T, int H, int I, const uint16_t* w_gate, const uint16_t* w_up,
                              const uint16_t* w_down, float limit, void* ws, size_t ws_bytes, uint16_t* shared_out,
                              void* stream) {
  if (!x || !w_gate || !w_up || !w_down || !ws || !shared_out || !(limit > 0.f)) return MOE_ERR_INVALID_ARG;
  if (T < 1 || H < 8 || H % 8 != 0 || I < 8 || I % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) || !aligned16(shared_out) ||
      (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_shared_expert_workspace_bytes(T, H, I)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int rc = ensure_device();
  if (rc != MOE_OK) return rc;
  return shared_expert_launch(x, T, H, I, w_gate, w_up, w_down, limit, ws, shared_out, as_stream(stream));
}

// ------------------------------------------------------------------------------------------ forward

static bool cfg_ok(const moe_prefill_config* c) {
  return c != nullptr && c->hidden >= 256 && c->hidden % 256 == 0 && c->moe_intermediate >= 256 &&
         c->moe_intermediate % 256 == 0 && c->num_experts >= 1 && c->num_experts <= 512 && c->top_k >= 1 &&
         c->top_k <= 32 && c->top_k <= c->num_experts &&
         (c->flags & ~(MOE_FWD_SEPARATE_SWIGLU | MOE_FWD_SMALL_ROWS | MOE_FWD_NO_MULTICAST)) == 0;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int moe_workspace_layout(const moe_prefill_config* c, int max_rows, moe_workspace_layout_t* L) {
  if (L == nullptr || !cfg_ok(c) || max_rows < 1) return MOE_ERR_INVALID_ARG;
  const size_t T = (size_t)max_rows, E = (size_t)c->num_experts, k = (size_t)c->top_k;
  const size_t H = (size_t)c->hidden, I = (size_t)c->moe_intermediate, R = T * k;
  if (R >= (1ull << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  L->logits = take(T * E * 4);
  L->ids = take(R * 4);
  L->wts = take(R * 4);
  L->sorted_token_ids = take(R * 4);
  L->sorted_expert_ids = take(R * 4);
  L->expert_offsets = take((E + 1) * 4);
  L->token_to_perm = take(R * 4);
  L->sort_scratch = take(sort_scratch_bytes((int)R, (int)E));
  L->ready = take((2 * E + 1) * 4);
  L->G = take((c->flags & MOE_FWD_SEPARATE_SWIGLU) ? R * 2 * I * 2 : 0);
  L->act = take(R * I * 2);
  L->Y = take(R * H * 2);
  L->x_stage = take(T * H * 2);
  L->x_sorted = take(R * H * 2);
  L->total = o;
  return MOE_OK;
}

size_t moe_workspace_bytes(const moe_prefill_config* cfg, int max_rows) {
  moe_workspace_layout_t L;
  return moe_workspace_layout(cfg, max_rows, &L) == MOE_OK ? L.total : 0;
}

int moe_prefill_forward(const moe_prefill_config* cfg, const uint16_t* x, int T, const uint16_t* w_router,
                        const float* logits_in, const float* router_bias, const moe_expert_table* w_gate_up,
                        const moe_expert_table* w_down, void* ws, size_t ws_bytes, uint16_t* out,
                        const uint16_t* shared_out, void* shared_ready, void* const* stage_events, void* stream) {
  if (!cfg_ok(cfg) || x == nullptr || out == nullptr || ws == nullptr || w_gate_up == nullptr || w_down == nullptr)
    return MOE_ERR_INVALID_ARG;
  if ((w_router == nullptr) == (logits_in == nullptr)) return MOE_ERR_INVALID_ARG;
  if (T < 1) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int H = cfg->hidden, I = cfg->moe_intermediate, E = cfg->num_experts, k = cfg->top_k;
  if (!aligned16(x) || !aligned16(out) || (reinterpret_cast<uintptr_t>(ws) & 255u) ||
      (w_router && !aligned16(w_router)) || (shared_out && !aligned16(shared_out)))
    return MOE_ERR_INVALID_ARG;
  if (w_gate_up->E != E || w_gate_up->N != 2 * I || w_gate_up->K != H) return MOE_ERR_INVALID_ARG;
  if (w_down->E != E || w_down->N != H || w_down->K != I) return MOE_ERR_INVALID_ARG;
  moe_workspace_layout_t L;
  int rc = moe_workspace_layout(cfg, T, &L);
  if (rc != MOE_OK) return rc;
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  rc = ensure_device();
  if (rc != MOE_OK) return rc;
  if (current_device() != w_gate_up->device || current_device() != w_down->device) return MOE_ERR_INVALID_ARG;
  // x and logits_in may be host memory the device can read, out host memory it can write: the
  // router kernel stages a host x into the workspace as it reads it (without a router, a staging
  // kernel does, or, when the CTA-pair gate/up GEMM takes the rows in expert order, the kernel
  // that stores each token row to its sorted positions reads it from the host once), the top-k
  // reads host logits directly, the combine stores into host memory
  const MemKind x_kind = memory_kind(x);
  if (x_kind == kMemNone || memory_kind(out) == kMemNone) return MOE_ERR_INVALID_ARG;
  if (logits_in && memory_kind(logits_in) == kMemNone) return MOE_ERR_INVALID_ARG;

  cudaStream_t st = as_stream(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  float* logits = reinterpret_cast<float*>(base + L.logits);
  int32_t* ids = reinterpret_cast<int32_t*>(base + L.ids);
  float* wts = reinterpret_cast<float*>(base + L.wts);
  int32_t* sti = reinterpret_cast<int32_t*>(base + L.sorted_token_ids);
  int32_t* sei = reinterpret_cast<int32_t*>(base + L.sorted_expert_ids);
  int32_t* off = reinterpret_cast<int32_t*>(base + L.expert_offsets);
  int32_t* t2p = reinterpret_cast<int32_t*>(base + L.token_to_perm);
  int32_t* cnt = reinterpret_cast<int32_t*>(base + L.sort_scratch);
  uint16_t* G = reinterpret_cast<uint16_t*>(base + L.G);
  uint16_t* act = reinterpret_cast<uint16_t*>(base + L.act);
  uint16_t* Y = reinterpret_cast<uint16_t*>(base + L.Y);
  uint16_t* x_stage = x_kind == kMemHost ? reinterpret_cast<uint16_t*>(base + L.x_stage) : nullptr;
  const uint16_t* xg = x_stage ? x_stage : x;  // the rows the expert GEMMs read
  const int R = T * k;
  int* err = device_error_word();
  // inside a stream capture the events become timestamp nodes of the graph (external records)
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (stage_events && cudaStreamIsCapturing(st, &cap) != cudaSuccess) return MOE_ERR_CUDA;
  auto ev = [&](int i) {
    if (stage_events && stage_events[i])
      cudaEventRecordWithFlags(static_cast<cudaEvent_t>(stage_events[i]), st,
                               cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault);
  };

  ev(0);
  if (w_router && E <= kRouterTopkMaxE) {
    // router GEMM and top-k in one launch (stage 1 -> 2 is empty): same results as the two
    // standalone entry points
    rc = router_topk_launch(x, w_router, T, H, E, router_bias, k, cfg->renormalize, cfg->routed_scale, logits, ids,
                            wts, err, st, x_stage);
    if (rc != MOE_OK) return rc;
    ev(1);
  } else {
    const float* lg = logits_in;
    if (w_router) {
      if ((rc = router_logits_launch(x, w_router, T, H, E, logits, st, x_stage)) != MOE_OK) return rc;
      lg = logits;
    }
    ev(1);
    rc = route_topk_launch(lg, router_bias, T, E, k, cfg->renormalize, cfg->routed_scale, ids, wts, err, st);
    if (rc != MOE_OK) return rc;
  }
  ev(2);
  // The fused-SwiGLU tensor-core path runs the down GEMM alongside the gate/up GEMM's last tiles:
  // the down GEMM loads an expert's activation rows once every gate/up CTA tile of them is stored
  // (per-expert counters ready[0..E)), and its clusters take tiles dynamically (counter ready[E]),
  // so the SMs the gate/up launch leaves early take more of the down work.  The CTA-pair gate/up
  // GEMM stores its token rows in expert order itself and counts them per expert in
  // ready[E+1..2E+1).  The sort clears all of them.
  const bool small = T <= 8 && (cfg->flags & MOE_FWD_SMALL_ROWS) && !(cfg->flags & MOE_FWD_SEPARATE_SWIGLU);
  const bool overlap = !small && !(cfg->flags & MOE_FWD_SEPARATE_SWIGLU);
  const bool no_mc = (cfg->flags & MOE_FWD_NO_MULTICAST) != 0;
  int32_t* ready = overlap ? reinterpret_cast<int32_t*>(base + L.ready) : nullptr;
  int producer_tiles = 0;
  if ((rc = sort_launch(ids, R, k, E, cnt, sti, sei, off, t2p, err, st, ready, 2 * E + 1)) != MOE_OK) return rc;
  // the fused gate/up GEMM on CTA pairs reads its token rows in expert order
  const int gemm_mode = g_gemm_kernel.load(std::memory_order_relaxed);
  const bool pair_gu = overlap && pair_gemm_shape_ok(2 * I, H, E, I) &&
                       (gemm_mode == MOE_GEMM_KERNEL_PAIR ||
                        (gemm_mode == MOE_GEMM_KERNEL_AUTO && pair_gemm_preferred(R, E)));
  uint16_t* x_sorted = reinterpret_cast<uint16_t*>(base + L.x_sorted);
  // the pair GEMM stores the rows in expert order from device rows (x, or x_stage written by the
  // router); a host x without a router is read over the link once instead, each row stored k times
  const bool host_scatter = pair_gu && x_stage && !w_router;
  if (host_scatter) {
    if ((rc = scatter_rows_launch(x, T, H, t2p, k, R, x_sorted, st)) != MOE_OK) return rc;
  } else if (x_stage && !w_router && (rc = stage_rows_launch(x, T, H, x_stage, st)) != MOE_OK) {
    return rc;
  }
  ev(3);
  // at most 8 rows per expert (top-k ids of a token are distinct): the small-row products
  if (small) {
    rc = gemv_checked(xg, T, H, sti, w_gate_up, off, R, act, I, I, cfg->swiglu_limit, st);
    if (rc != MOE_OK) return rc;
    ev(4);
  } else if (cfg->flags & MOE_FWD_SEPARATE_SWIGLU) {
    if ((rc = gemm_checked(xg, T, H, sti, w_gate_up, off, R, G, 2 * I, MOE_DTYPE_BF16, st, 0, 0.f, nullptr, nullptr, 0,
                           nullptr, nullptr, no_mc)) != MOE_OK)
      return rc;
    ev(4);
    if ((rc = swiglu_launch(G, G + I, R, I, 2 * I, act, I, cfg->swiglu_limit, st)) != MOE_OK) return rc;
  } else if (pair_gu) {
    // CTA-pair kernel: it loads contiguous rows in expert order (x_sorted) with tiled TMA boxes,
    // and stores them there itself unless the host rows were scattered above
    rc = gemm_checked(x_sorted, R, H, nullptr, w_gate_up, off, R, act, I, MOE_DTYPE_BF16, st, I, cfg->swiglu_limit,
                      ready, nullptr, 0, nullptr, &producer_tiles, no_mc, host_scatter ? nullptr : xg, T, sti,
                      ready + E + 1);
    if (rc != MOE_OK) return rc;
    ev(4);
  } else {
    // the gate/up launch reports how many of its CTA tiles cover one activation row (single-CTA
    // kernel: one per 128 activation columns; CTA pairs: two per 128)
    rc = gemm_checked(xg, T, H, sti, w_gate_up, off, R, act, I, MOE_DTYPE_BF16, st, I, cfg->swiglu_limit, ready,
                      nullptr, 0, nullptr, &producer_tiles, no_mc);
    if (rc != MOE_OK) return rc;
    ev(4);
  }
  ev(5);
  rc = small ? gemv_checked(act, R, I, nullptr, w_down, off, R, Y, H, 0, 0.f, st)
             : gemm_checked(act, R, I, nullptr, w_down, off, R, Y, H, MOE_DTYPE_BF16, st, 0, 0.f, nullptr, ready,
                            producer_tiles, ready ? ready + E : nullptr, nullptr, no_mc);
  if (rc != MOE_OK) return rc;
  ev(6);
  if (shared_ready && cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(shared_ready), 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  if ((rc = combine_launch(Y, t2p, wts, shared_out, T, k, H, out, st)) != MOE_OK) return rc;
  ev(7);
  return MOE_OK;
}

// ------------------------------------------------------------------------------------------ debug

int moe_debug_set_gemm_kernel(int which) {
  if (which != MOE_GEMM_KERNEL_AUTO && which != MOE_GEMM_KERNEL_SINGLE && which != MOE_GEMM_KERNEL_PAIR)
    return MOE_ERR_INVALID_ARG;
  g_gemm_kernel.store(which, std::memory_order_relaxed);
  return MOE_OK;
}

int moe_debug_grouped_gemm_after(const uint16_t* A, int a_rows, int lda, const int32_t* gather_ids,
                                 const moe_expert_table* W, const int32_t* expert_offsets, int R, void* C, int ldc,
                                 int c_dtype, const int32_t* ready, int ready_need, void* stream) {
  if (ready == nullptr || ready_need < 1) return MOE_ERR_INVALID_ARG;
  return gemm_checked(A, a_rows, lda, gather_ids, W, expert_offsets, R, C, ldc, c_dtype, as_stream(stream), 0, 0.f,
                      nullptr, ready, ready_need, nullptr);
}

unsigned long long moe_debug_set_wait_limit_ns(unsigned long long ns) {
  if (ns == 0) ns = 2000000000ull;
  if (ns > 2000000000ull) ns = 2000000000ull;
  return g_wait_limit_ns.exchange(ns, std::memory_order_relaxed);
}

// ------------------------------------------------------------------------------------------ errors

int moe_get_device_error(void* stream, int* code) {
  if (code == nullptr) return MOE_ERR_INVALID_ARG;
  *code = 0;
  const int rc = ensure_device();
  if (rc != MOE_OK) return rc;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  *code = v;
  return v == 0 ? MOE_OK : MOE_ERR_DEVICE;
}

}  // extern "C"
