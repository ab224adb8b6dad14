// api.cu -- the extern "C" boundary of libgqa.so: argument checks, per-device
// workspace, tensor-map encoding, host-buffer variants and status reporting.
// Declarations and their contracts are in include/gqa.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/gqa.h"
#include "internal.h"
#include "ptx.cuh"

namespace {

thread_local std::string g_cuda_msg;
std::mutex g_mu;
std::atomic<unsigned long long> g_wait_limit_ns{0};  // 0: kWaitLimitNs
std::atomic<int> g_fail_allocs{0};                   // workspace allocations still to fail

struct DeviceCtx {
  bool ready = false;
  int sm_count = 0;
  float* ws_part = nullptr;
  size_t ws_part_cap = 0;
  int* counters = nullptr;
  size_t counters_cap = 0;
  unsigned* err = nullptr;
  cudaEvent_t last_evt = nullptr;
  cudaStream_t last_stream = nullptr;
  bool evt_pending = false;
  void* stage = nullptr;  // host-call staging
  size_t stage_cap = 0;
};
std::vector<DeviceCtx> g_dev;

int cuda_fail(cudaError_t e) {
  g_cuda_msg = std::string(cudaGetErrorName(e)) + ": " + cudaGetErrorString(e);
  return GQA_ERR_CUDA;
}

// A workspace allocation, or the failure a test asked for.
cudaError_t ws_malloc(void** p, size_t bytes) {
  if (gqa::take_injected_alloc_failure()) return cudaErrorMemoryAllocation;
  return cudaMalloc(p, bytes);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Current device's context, created on first use.  Caller holds g_mu.
int get_ctx(DeviceCtx** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cuda_fail(e);
    return GQA_ERR_NO_DEVICE;
  }
  if ((int)g_dev.size() <= dev) g_dev.resize(dev + 1);
  DeviceCtx& c = g_dev[dev];
  if (!c.ready) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&c.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e);
    if (major != 10 || minor != 3) {
      g_cuda_msg = "device is sm_" + std::to_string(major) + std::to_string(minor) +
                   "; libgqa.so is built for sm_103a only";
      return GQA_ERR_NO_DEVICE;
    }
    if ((e = cudaMalloc(&c.err, sizeof(unsigned))) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMemset(c.err, 0, sizeof(unsigned))) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaEventCreateWithFlags(&c.last_evt, cudaEventDisableTiming)) != cudaSuccess)
      return cuda_fail(e);
    c.ready = true;
  }
  *out = &c;
  return GQA_OK;
}

// True while `s` is being captured into a CUDA graph: nothing may then
// synchronise, allocate, or wait on an event recorded outside the capture.
bool capturing(cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  return cudaStreamIsCapturing(s, &st) == cudaSuccess && st != cudaStreamCaptureStatusNone;
}

// Orders this call after the previous workspace user if it ran on another
// stream.  A captured call is not ordered here: replays of a graph are
// ordered against other users of the workspace by the caller.
cudaError_t order_after_previous(DeviceCtx& c, cudaStream_t s) {
  if (capturing(s)) return cudaSuccess;
  if (c.evt_pending && c.last_stream != s) return cudaStreamWaitEvent(s, c.last_evt, 0);
  return cudaSuccess;
}

cudaError_t mark_used(DeviceCtx& c, cudaStream_t s) {
  if (capturing(s)) return cudaSuccess;
  c.last_stream = s;
  c.evt_pending = true;
  return cudaEventRecord(c.last_evt, s);
}

int capture_needs_growth() {
  g_cuda_msg = "the workspace must grow, which cannot happen during stream capture: make one call with these "
               "sizes (or larger) before capturing";
  return GQA_ERR_CUDA;
}

int check_decode_args(const void* q, const void* k, const void* v, const int32_t* seqlens,
                      const void* out, int B, int Hq, int Hkv, int D, int Lmax, float scale) {
  if (!q || !k || !v || !seqlens || !out) return GQA_ERR_NULL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Lmax <= 0 || Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return GQA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(seqlens) & 3u))
    return GQA_ERR_MISALIGNED;
  gqa::DecodePlan plan;
  if (!gqa::decode_plan(B, Hq, Hkv, D, Lmax, 148, &plan)) return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

int check_prefill_args(const void* q, const void* k, const void* v, const void* out, int B, int L,
                       int Hq, int Hkv, int D, int causal) {
  if (!q || !k || !v || !out) return GQA_ERR_NULL;
  if (B <= 0 || L <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return GQA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return GQA_ERR_MISALIGNED;
  if (!gqa::prefill_supported(D)) return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

struct PagedCache {
  const int32_t* block_table = nullptr;
  int page_size = 0, num_pages = 0, max_pages = 0;
};

int decode_locked(DeviceCtx& c, const void* q, const void* k, const void* v, const int32_t* seqlens,
                  void* out, int B, int Hq, int Hkv, int D, int Lmax, float scale, cudaStream_t s,
                  const float* k_scale = nullptr, const float* v_scale = nullptr, PagedCache pc = PagedCache()) {
  const bool kv8 = k_scale != nullptr;
  gqa::DecodePlan plan;
  if (!gqa::decode_plan(B, Hq, Hkv, D, Lmax, c.sm_count, &plan, 0, kv8)) return GQA_ERR_UNSUPPORTED;
  cudaError_t e;
  if (plan.ws_part_floats > c.ws_part_cap || plan.ws_counters > c.counters_cap) {
    if (capturing(s)) return capture_needs_growth();
    // Growing the workspace: cudaFree waits for work that still uses the old one.
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e);
    if (plan.ws_part_floats > c.ws_part_cap) {
      if (c.ws_part) cudaFree(c.ws_part);
      c.ws_part = nullptr;
      c.ws_part_cap = 0;
      if ((e = ws_malloc(reinterpret_cast<void**>(&c.ws_part), plan.ws_part_floats * sizeof(float))) != cudaSuccess)
        return cuda_fail(e);
      c.ws_part_cap = plan.ws_part_floats;
    }
    if (plan.ws_counters > c.counters_cap) {
      if (c.counters) cudaFree(c.counters);
      c.counters = nullptr;
      c.counters_cap = 0;
      if ((e = ws_malloc(reinterpret_cast<void**>(&c.counters), plan.ws_counters * sizeof(int))) != cudaSuccess)
        return cuda_fail(e);
      if ((e = cudaMemset(c.counters, 0, plan.ws_counters * sizeof(int))) != cudaSuccess) return cuda_fail(e);
      c.counters_cap = plan.ws_counters;
    }
  }
  if ((e = order_after_previous(c, s)) != cudaSuccess) return cuda_fail(e);
  gqa::DecodeArgs a{q, k, v, seqlens, out, B, Hq, Hkv, D, Lmax, scale, c.ws_part, c.counters, c.err, k_scale, v_scale,
                    pc.block_table, pc.page_size, pc.num_pages, pc.max_pages};
  if ((e = gqa::decode_launch(plan, a, s)) != cudaSuccess) return cuda_fail(e);
  if ((e = mark_used(c, s)) != cudaSuccess) return cuda_fail(e);
  return GQA_OK;
}

cudaError_t ensure_stage(DeviceCtx& c, size_t bytes, cudaStream_t s) {
  if (bytes <= c.stage_cap) return cudaSuccess;
  if (capturing(s)) return cudaErrorStreamCaptureUnsupported;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  if (c.stage) cudaFree(c.stage);
  c.stage = nullptr;
  c.stage_cap = 0;
  if ((e = cudaMalloc(&c.stage, bytes)) != cudaSuccess) return e;
  c.stage_cap = bytes;
  return cudaSuccess;
}

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

namespace gqa {

unsigned long long pipeline_wait_limit_ns() {
  const unsigned long long v = g_wait_limit_ns.load(std::memory_order_relaxed);
  return v ? v : kWaitLimitNs;
}

bool pipeline_starved() { return g_wait_limit_ns.load(std::memory_order_relaxed) != 0; }

bool take_injected_alloc_failure() {
  int n = g_fail_allocs.load();
  while (n > 0)
    if (g_fail_allocs.compare_exchange_weak(n, n - 1)) return true;
  return false;
}

CUresult encode_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t dim0, uint64_t dim1,
                             uint64_t dim2, uint64_t stride1, uint64_t stride2, uint32_t box0,
                             uint32_t box1, uint32_t box2) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[3] = {dim0, dim1, dim2};
  cuuint64_t strides[2] = {stride1, stride2};
  cuuint32_t box[3] = {box0, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_tmap_u8_3d(CUtensorMap* map, const void* base, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                           uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1, uint32_t box2) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[3] = {dim0, dim1, dim2};
  cuuint64_t strides[2] = {stride1, stride2};
  cuuint32_t box[3] = {box0, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = box0 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace gqa

extern "C" {

int gqa_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* seqlens,
               void* out, int B, int Hq, int Hkv, int D, int Lmax, float scale, void* stream) {
  int st = check_decode_args(q, k_cache, v_cache, seqlens, out, B, Hq, Hkv, D, Lmax, scale);
  if (st != GQA_OK) return st;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceCtx* c = nullptr;
  if ((st = get_ctx(&c)) != GQA_OK) return st;
  return decode_locked(*c, q, k_cache, v_cache, seqlens, out, B, Hq, Hkv, D, Lmax, scale,
                       static_cast<cudaStream_t>(stream));
}

int gqa_decode_fp8(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                   const float* v_scale, const int32_t* seqlens, void* out, int B, int Hq, int Hkv, int D,
                   int Lmax, float scale, void* stream) {
  if (!q || !k_cache || !v_cache || !k_scale || !v_scale || !seqlens || !out) return GQA_ERR_NULL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Lmax <= 0 || Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return GQA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(seqlens) & 3u) || (reinterpret_cast<uintptr_t>(k_scale) & 3u) ||
      (reinterpret_cast<uintptr_t>(v_scale) & 3u))
    return GQA_ERR_MISALIGNED;
  gqa::DecodePlan plan;
  if (!gqa::decode_plan(B, Hq, Hkv, D, Lmax, 148, &plan, 0, true)) return GQA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceCtx* c = nullptr;
  int st = get_ctx(&c);
  if (st != GQA_OK) return st;
  return decode_locked(*c, q, k_cache, v_cache, seqlens, out, B, Hq, Hkv, D, Lmax, scale,
                       static_cast<cudaStream_t>(stream), k_scale, v_scale);
}

int gqa_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                     const int32_t* seqlens, void* out, int B, int Hq, int Hkv, int D, int num_pages, int page_size,
                     int max_pages, float scale, void* stream) {
  if (!q || !k_pages || !v_pages || !block_table || !seqlens || !out) return GQA_ERR_NULL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || num_pages <= 0 || page_size <= 0 || max_pages <= 0 ||
      Hq % Hkv != 0)
    return GQA_ERR_INVALID_ARG;
  if ((long long)max_pages * page_size > 0x7fffffffLL) return GQA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return GQA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(seqlens) & 3u) || (reinterpret_cast<uintptr_t>(block_table) & 3u))
    return GQA_ERR_MISALIGNED;
  const int Lcap = max_pages * page_size;
  gqa::DecodePlan plan;
  if (!gqa::decode_plan(B, Hq, Hkv, D, Lcap, 148, &plan)) return GQA_ERR_UNSUPPORTED;
  if (page_size % plan.tile_keys != 0) return GQA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceCtx* c = nullptr;
  int st = get_ctx(&c);
  if (st != GQA_OK) return st;
  PagedCache pc;
  pc.block_table = block_table;
  pc.page_size = page_size;
  pc.num_pages = num_pages;
  pc.max_pages = max_pages;
  return decode_locked(*c, q, k_pages, v_pages, seqlens, out, B, Hq, Hkv, D, Lcap, scale,
                       static_cast<cudaStream_t>(stream), nullptr, nullptr, pc);
}

int gqa_decode_fp8_paged(const void* q, const void* k_pages, const void* v_pages, const float* k_scale,
                         const float* v_scale, const int32_t* block_table, const int32_t* seqlens, void* out, int B,
                         int Hq, int Hkv, int D, int num_pages, int page_size, int max_pages, float scale,
                         void* stream) {
  if (!q || !k_pages || !v_pages || !k_scale || !v_scale || !block_table || !seqlens || !out) return GQA_ERR_NULL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || num_pages <= 0 || page_size <= 0 || max_pages <= 0 ||
      Hq % Hkv != 0)
    return GQA_ERR_INVALID_ARG;
  if ((long long)max_pages * page_size > 0x7fffffffLL) return GQA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return GQA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(seqlens) & 3u) || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
    return GQA_ERR_MISALIGNED;
  const int Lcap = max_pages * page_size;
  gqa::DecodePlan plan;
  if (!gqa::decode_plan(B, Hq, Hkv, D, Lcap, 148, &plan, 0, true)) return GQA_ERR_UNSUPPORTED;
  if (page_size % plan.tile_keys != 0) return GQA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceCtx* c = nullptr;
  int st = get_ctx(&c);
  if (st != GQA_OK) return st;
  PagedCache pc;
  pc.block_table = block_table;
  pc.page_size = page_size;
  pc.num_pages = num_pages;
  pc.max_pages = max_pages;
  return decode_locked(*c, q, k_pages, v_pages, seqlens, out, B, Hq, Hkv, D, Lcap, scale,
                       static_cast<cudaStream_t>(stream), k_scale, v_scale, pc);
}

int gqa_rope_append(const void* q, const void* k_new, const void* v_new, void* q_out, void* k_cache,
                    void* v_cache, int32_t* seqlens, int B, int Hq, int Hkv, int D, int Lmax, double base,
                    void* stream) {
  if (!q || !k_new || !v_new || !q_out || !k_cache || !v_cache || !seqlens) return GQA_ERR_NULL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Lmax <= 0 || Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (!(base > 1.0) || !isfinite(base)) return GQA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(q_out) || !aligned16(k_cache) ||
      !aligned16(v_cache) || (reinterpret_cast<uintptr_t>(seqlens) & 3u))
    return GQA_ERR_MISALIGNED;
  if (!gqa::rope_supported(D)) return GQA_ERR_UNSUPPORTED;
  DeviceCtx* c = nullptr;
  int st;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = get_ctx(&c)) != GQA_OK) return st;
  }
  gqa::RopeArgs a{static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_new),
                  static_cast<const __nv_bfloat16*>(v_new), static_cast<__nv_bfloat16*>(q_out),
                  static_cast<__nv_bfloat16*>(k_cache), static_cast<__nv_bfloat16*>(v_cache),
                  seqlens, B, Hq, Hkv, D, Lmax, base, c->err};
  cudaError_t e = gqa::rope_append_launch(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GQA_OK : cuda_fail(e);
}

int gqa_meanpool_kv_heads(const void* w, void* w_out, int H, int Hkv, int rows, int cols, int mode,
                          void* stream) {
  if (!w || !w_out) return GQA_ERR_NULL;
  if (H <= 0 || Hkv <= 0 || rows <= 0 || cols <= 0 || H % Hkv != 0 || (mode != 0 && mode != 1))
    return GQA_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(w_out)) return GQA_ERR_MISALIGNED;
  const long long n = (long long)rows * cols;
  const char* wb = static_cast<const char*>(w);
  const char* ob = static_cast<const char*>(w_out);
  if (ob < wb + (size_t)H * n * 2 && wb < ob + (size_t)Hkv * n * 2) return GQA_ERR_INVALID_ARG;  // overlap
  DeviceCtx* c = nullptr;
  int st;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = get_ctx(&c)) != GQA_OK) return st;
  }
  cudaError_t e = gqa::meanpool_heads_launch(w, w_out, H, Hkv, n, mode, c->sm_count, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GQA_OK : cuda_fail(e);
}

int gqa_prefill(const void* q, const void* k, const void* v, void* out, int B, int L, int Hq, int Hkv,
                int D, int causal, void* stream) {
  int st = check_prefill_args(q, k, v, out, B, L, Hq, Hkv, D, causal);
  if (st != GQA_OK) return st;
  DeviceCtx* c = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = get_ctx(&c)) != GQA_OK) return st;
  }
  gqa::PrefillArgs a{q, k, v, out, B, L, Hq, Hkv, D, causal, c->err};
  cudaError_t e = gqa::prefill_launch(a, c->sm_count, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GQA_OK : cuda_fail(e);
}

int gqa_prefill_chunk(const void* q, const void* k, const void* v, void* out, int B, int Lq, int Lk, int Hq,
                      int Hkv, int D, int causal, void* stream) {
  int st = check_prefill_args(q, k, v, out, B, Lq, Hq, Hkv, D, causal);
  if (st != GQA_OK) return st;
  if (Lk < Lq) return GQA_ERR_INVALID_ARG;
  DeviceCtx* c = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = get_ctx(&c)) != GQA_OK) return st;
  }
  gqa::PrefillArgs a{q, k, v, out, B, Lq, Hq, Hkv, D, causal, c->err, Lk};
  cudaError_t e = gqa::prefill_launch(a, c->sm_count, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GQA_OK : cuda_fail(e);
}

int gqa_decode_host(const void* q_host, const void* k_cache_host, const void* v_cache_host,
                    const int32_t* seqlens_host, void* out_host, int B, int Hq, int Hkv, int D,
                    int Lmax, float scale, void* stream) {
  if (!q_host || !k_cache_host || !v_cache_host || !seqlens_host || !out_host) return GQA_ERR_NULL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Lmax <= 0 || Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return GQA_ERR_INVALID_ARG;
  gqa::DecodePlan plan;
  if (!gqa::decode_plan(B, Hq, Hkv, D, Lmax, 148, &plan)) return GQA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t qb = (size_t)B * Hq * D * 2, kb = (size_t)B * Hkv * Lmax * D * 2, sb = (size_t)B * 4;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceCtx* c = nullptr;
  int st = get_ctx(&c);
  if (st != GQA_OK) return st;
  cudaError_t e;
  if ((e = ensure_stage(*c, al256(qb) * 2 + al256(kb) * 2 + al256(sb), s)) != cudaSuccess) return cuda_fail(e);
  char* base = static_cast<char*>(c->stage);
  char* dq = base;
  char* dk = dq + al256(qb);
  char* dv = dk + al256(kb);
  char* dsl = dv + al256(kb);
  char* dout = dsl + al256(sb);
  if ((e = order_after_previous(*c, s)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaMemcpyAsync(dq, q_host, qb, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
      (e = cudaMemcpyAsync(dk, k_cache_host, kb, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
      (e = cudaMemcpyAsync(dv, v_cache_host, kb, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
      (e = cudaMemcpyAsync(dsl, seqlens_host, sb, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e);
  st = decode_locked(*c, dq, dk, dv, reinterpret_cast<const int32_t*>(dsl), dout, B, Hq, Hkv, D, Lmax,
                     scale, s);
  if (st != GQA_OK) return st;
  if ((e = cudaMemcpyAsync(out_host, dout, qb, cudaMemcpyDeviceToHost, s)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e);
  return GQA_OK;
}

int gqa_prefill_host(const void* q_host, const void* k_host, const void* v_host, void* out_host, int B,
                     int L, int Hq, int Hkv, int D, int causal, void* stream) {
  if (!q_host || !k_host || !v_host || !out_host) return GQA_ERR_NULL;
  if (B <= 0 || L <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return GQA_ERR_INVALID_ARG;
  if (!gqa::prefill_supported(D)) return GQA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t qb = (size_t)B * Hq * L * D * 2, kb = (size_t)B * Hkv * L * D * 2;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceCtx* c = nullptr;
  int st = get_ctx(&c);
  if (st != GQA_OK) return st;
  cudaError_t e;
  if ((e = ensure_stage(*c, al256(qb) * 2 + al256(kb) * 2, s)) != cudaSuccess) return cuda_fail(e);
  char* dq = static_cast<char*>(c->stage);
  char* dk = dq + al256(qb);
  char* dv = dk + al256(kb);
  char* dout = dv + al256(kb);
  if ((e = order_after_previous(*c, s)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaMemcpyAsync(dq, q_host, qb, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
      (e = cudaMemcpyAsync(dk, k_host, kb, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
      (e = cudaMemcpyAsync(dv, v_host, kb, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e);
  gqa::PrefillArgs a{dq, dk, dv, dout, B, L, Hq, Hkv, D, causal, c->err};
  if ((e = gqa::prefill_launch(a, c->sm_count, s)) != cudaSuccess) return cuda_fail(e);
  if ((e = mark_used(*c, s)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaMemcpyAsync(out_host, dout, qb, cudaMemcpyDeviceToHost, s)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e);
  return GQA_OK;
}

const char* gqa_status_string(int status) {
  switch (status) {
    case GQA_OK: return "GQA_OK";
    case GQA_ERR_INVALID_ARG: return "GQA_ERR_INVALID_ARG: a size is <= 0, Hq % Hkv != 0, causal is not 0/1 or scale is not finite and > 0";
    case GQA_ERR_UNSUPPORTED: return "GQA_ERR_UNSUPPORTED: shape not implemented (decode: D = 128 with Hq/Hkv <= 128, or D = 64 with Hq/Hkv <= 8, 16 or 32; B <= 1024; prefill: D = 64 or 128)";
    case GQA_ERR_NULL: return "GQA_ERR_NULL: a required pointer is NULL";
    case GQA_ERR_MISALIGNED: return "GQA_ERR_MISALIGNED: tensor pointers must be 16-byte aligned (seqlens 4-byte)";
    case GQA_ERR_CUDA: {
      static thread_local std::string s;
      s = "GQA_ERR_CUDA: " + (g_cuda_msg.empty() ? std::string("unknown CUDA error") : g_cuda_msg);
      return s.c_str();
    }
    case GQA_ERR_NO_DEVICE: {
      static thread_local std::string s;
      s = "GQA_ERR_NO_DEVICE: " + (g_cuda_msg.empty() ? std::string("no sm_103 device") : g_cuda_msg);
      return s.c_str();
    }
    case GQA_ERR_TOO_LARGE: return "GQA_ERR_TOO_LARGE: the sizes need more workspace than the fixed scratch of gqa_decode_noalloc";
    default: return "unknown gqa status";
  }
}

int gqa_get_device_status(void* stream, uint32_t* flags) {
  if (!flags) return GQA_ERR_NULL;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceCtx* c = nullptr;
  int st = get_ctx(&c);
  if (st != GQA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  unsigned v = 0;
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaMemcpy(&v, c->err, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaMemset(c->err, 0, sizeof v)) != cudaSuccess) return cuda_fail(e);
  unsigned na = 0;
  if ((e = gqa::noalloc_take_status(&na)) != cudaSuccess) return cuda_fail(e);
  v |= na;
  if ((v & GQA_DEV_WAIT_TIMEOUT) && c->counters) {
    // A decode that gave up may have left arrival counters half counted.
    if ((e = cudaMemset(c->counters, 0, c->counters_cap * sizeof(int))) != cudaSuccess) return cuda_fail(e);
  }
  *flags = v;
  return GQA_OK;
}

int gqa_decode_plan(int B, int Hq, int Hkv, int D, int Lmax, int* tile_keys, int* num_ctas) {
  if (!tile_keys || !num_ctas) return GQA_ERR_NULL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Lmax <= 0 || Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  int sm = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) sm = v;
  } else {
    cudaGetLastError();
  }
  gqa::DecodePlan plan;
  if (!gqa::decode_plan(B, Hq, Hkv, D, Lmax, sm, &plan)) return GQA_ERR_UNSUPPORTED;
  *tile_keys = plan.tile_keys;
  *num_ctas = plan.num_ctas;
  return GQA_OK;
}

void gqa_test_set_wait_limit_ns(unsigned long long ns) { g_wait_limit_ns.store(ns); }

void gqa_test_fail_workspace_allocs(int n) { g_fail_allocs.store(n > 0 ? n : 0); }

void gqa_release(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int cur = -1;
  bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
  for (size_t d = 0; d < g_dev.size(); ++d) {
    DeviceCtx& c = g_dev[d];
    if (!c.ready) continue;
    cudaSetDevice((int)d);
    cudaDeviceSynchronize();
    if (c.ws_part) cudaFree(c.ws_part);
    if (c.counters) cudaFree(c.counters);
    if (c.err) cudaFree(c.err);
    if (c.stage) cudaFree(c.stage);
    if (c.last_evt) cudaEventDestroy(c.last_evt);
    c = DeviceCtx();
  }
  if (have_cur) cudaSetDevice(cur);
  cudaGetLastError();
}

}  // extern "C"
