// noalloc.cu -- gqa_decode_noalloc: the decode step of gqa_decode with its
// scratch memory in a fixed-size device array that is part of the library
// image, so that the call itself never allocates.
//
// Who needs this: a caller that owns every byte of device memory through its
// own pool -- e.g. a serving engine that reserves HBM for its KV cache at
// start-up -- cannot let a library cudaMalloc behind its back (the call may
// fail, or fragment the pool), and a caller on a latency-critical loop may not
// allocate after start-up at all, because cudaMalloc / cudaFree can
// synchronise the device and stall every stream.  Such callers pass inputs
// and outputs as with gqa_decode; the merge workspace comes from the array
// below instead of from the library's allocator.
#include <cuda_runtime.h>
#include <math.h>

#include <mutex>

#include "../../include/gqa.h"
#include "internal.h"

namespace {

// Scratch layout: [0, 256) status word; then the arrival counters (one per
// (b, kv head) pair, two spare); then the partial results (fp32).  Total
// about 5 MiB + 33 KiB.
constexpr size_t kMaxPairs = GQA_NOALLOC_MAX_PAIRS;
constexpr size_t kMaxPartFloats = GQA_NOALLOC_MAX_PART_FLOATS;
constexpr size_t kCountersOff = 256;
constexpr size_t kPartOff = (kCountersOff + 4 * (kMaxPairs + 2) + 255) / 256 * 256;
constexpr size_t kScratchBytes = kPartOff + 4 * kMaxPartFloats;
static_assert(kScratchBytes == GQA_NOALLOC_SCRATCH_BYTES, "gqa.h states the scratch size callers plan for");

// Every GPU on which this array's module is loaded (at the first
// gqa_decode_noalloc call there, see scratch_for_current_device) holds it
// until the process exits.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_na_mu;
void* g_na_ptr[kMaxDevices];  // device address of g_decode_scratch, per device
int g_na_sms[kMaxDevices];

// Once per device, with that device current: resolve the array's device
// address (in host code the symbol is only a host-side stand-in).  With the
// CUDA runtime's lazy module loading (the default) this lookup is also what
// loads the module holding the array, and so what commits its
// GQA_NOALLOC_SCRATCH_BYTES of device memory on this device: the first call
// on a device belongs at start-up.
int scratch_for_current_device(void** ptr, int* sms) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GQA_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_na_mu);
  if (!g_na_ptr[dev]) {
    int major = 0, minor = 0, sm = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return GQA_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return GQA_ERR_NO_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return GQA_ERR_CUDA;
    }
    g_na_sms[dev] = sm;
    g_na_ptr[dev] = p;
  }
  *ptr = g_na_ptr[dev];
  *sms = g_na_sms[dev];
  return GQA_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace gqa {

cudaError_t noalloc_take_status(unsigned* flags) {
  *flags = 0;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return cudaSuccess;
  }
  void* p = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_na_mu);
    p = g_na_ptr[dev];
  }
  if (!p) return cudaSuccess;
  unsigned v = 0;
  cudaError_t e = cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return e;
  if (v && (e = cudaMemset(p, 0, sizeof v)) != cudaSuccess) return e;
  *flags = v;
  return cudaSuccess;
}

}  // namespace gqa

extern "C" int gqa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* seqlens, void* out, int B, int Hq, int Hkv, int D,
                                  int Lmax, float scale, void* stream) {
  if (!q || !k_cache || !v_cache || !seqlens || !out) return GQA_ERR_NULL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Lmax <= 0 || Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return GQA_ERR_INVALID_ARG;
  if (!al16(q) || !al16(k_cache) || !al16(v_cache) || !al16(out) || (reinterpret_cast<uintptr_t>(seqlens) & 3u))
    return GQA_ERR_MISALIGNED;
  void* base = nullptr;
  int sms = 0;
  int st = scratch_for_current_device(&base, &sms);
  if (st != GQA_OK) return st;
  gqa::DecodePlan plan;
  if ((size_t)B * Hkv > kMaxPairs) return GQA_ERR_TOO_LARGE;
  if (!gqa::decode_plan(B, Hq, Hkv, D, Lmax, sms, &plan)) return GQA_ERR_UNSUPPORTED;
  if (plan.ws_counters > kMaxPairs + 2 || plan.ws_part_floats > kMaxPartFloats) return GQA_ERR_TOO_LARGE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* b = static_cast<unsigned char*>(base);
  // The array keeps the previous call's contents: the status word and the
  // counters this call uses must start at zero.
  if (cudaMemsetAsync(b, 0, kCountersOff + 4 * plan.ws_counters, s) != cudaSuccess) {
    cudaGetLastError();
    return GQA_ERR_CUDA;
  }
  gqa::DecodeArgs a{q, k_cache, v_cache, seqlens, out, B, Hq, Hkv, D, Lmax, scale,
                    reinterpret_cast<float*>(b + kPartOff), reinterpret_cast<int*>(b + kCountersOff),
                    reinterpret_cast<unsigned*>(b)};
  if (gqa::decode_launch(plan, a, s) != cudaSuccess) {
    cudaGetLastError();
    return GQA_ERR_CUDA;
  }
  return GQA_OK;
}
