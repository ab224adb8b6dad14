// convert.cu -- MHA -> GQA checkpoint conversion of a key or value projection.
//
// The GQA paper notes on 51969.com, section "Uptraining" (figure 1) and the
// checkpoint-conversion experiment (figure 4): an H-head checkpoint becomes a
// GQA checkpoint with Hkv groups by giving group j, which serves query heads
// j*G .. j*G + G - 1 (G = H / Hkv, the h -> h / G grouping of the decode and
// prefill kernels), one key and one value head whose projection is the mean
// of those G heads' projections ("Mean"; the notes also compare taking the
// group's first head, "First").  Hkv = 1 is the MHA -> MQA conversion.
//
// Data: the projection as H contiguous per-head blocks of n = rows * cols
// bf16 values (an nn.Linear weight [H * head_dim, d_model] viewed as
// [H, head_dim, d_model], or a bias [H * head_dim] with cols = 1); the result
// is Hkv blocks.  This is a bandwidth-bound streaming reduction (every input
// byte read once, every output byte written once): one thread per 8
// consecutive values of an output block (16-byte loads of the G input
// blocks, coalesced across the warp, streaming cache hints), fp32 sum in
// head order, one correctly rounded division by G, bf16 round to nearest
// even.  "First" copies bits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace gqa {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void unpack8(const uint4 v, float (&x)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// kVec: n % 8 == 0 (16-byte chunks); otherwise one value per item.
template <bool kVec>
__global__ void __launch_bounds__(kThreads) meanpool_kernel(const __nv_bfloat16* __restrict__ w,
                                                            __nv_bfloat16* __restrict__ out, long long n, int G,
                                                            int Hkv, int mode) {
  const long long per = kVec ? n / 8 : n;  // items per output block
  const long long items = (long long)Hkv * per;
  const float g_f = (float)G;
  for (long long it = (long long)blockIdx.x * kThreads + threadIdx.x; it < items;
       it += (long long)gridDim.x * kThreads) {
    const long long j = it / per, c = it - j * per;
    const __nv_bfloat16* src = w + (size_t)j * G * n;
    if constexpr (kVec) {
      const uint4* s4 = reinterpret_cast<const uint4*>(src) + c;
      uint4* d4 = reinterpret_cast<uint4*>(out + (size_t)j * n) + c;
      if (mode == 1) {
        __stcs(d4, __ldcs(s4));
        continue;
      }
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int g = 0; g < G; ++g) {
        float x[8];
        unpack8(__ldcs(s4 + (size_t)g * (n / 8)), x);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += x[e];
      }
      uint4 r;
      r.x = pack2(acc[0] / g_f, acc[1] / g_f);
      r.y = pack2(acc[2] / g_f, acc[3] / g_f);
      r.z = pack2(acc[4] / g_f, acc[5] / g_f);
      r.w = pack2(acc[6] / g_f, acc[7] / g_f);
      __stcs(d4, r);
    } else {
      if (mode == 1) {
        out[(size_t)j * n + c] = src[c];
        continue;
      }
      float acc = 0.f;
      for (int g = 0; g < G; ++g) acc += __bfloat162float(src[(size_t)g * n + c]);
      out[(size_t)j * n + c] = __float2bfloat16_rn(acc / g_f);
    }
  }
}

}  // namespace

cudaError_t meanpool_heads_launch(const void* w, void* out, int H, int Hkv, long long n, int mode, int sm_count,
                                  cudaStream_t stream) {
  if (H <= 0 || Hkv <= 0 || H % Hkv != 0 || n <= 0 || (mode != 0 && mode != 1)) return cudaErrorInvalidValue;
  const int G = H / Hkv;
  const bool vec = n % 8 == 0;
  const long long items = (long long)Hkv * (vec ? n / 8 : n);
  const long long want = (items + kThreads - 1) / kThreads;
  const long long cap = 8LL * (sm_count > 0 ? sm_count : 148);  // 8 resident CTAs of 256 threads per SM
  const int grid = (int)(want < cap ? want : cap);
  const auto* src = static_cast<const __nv_bfloat16*>(w);
  auto* dst = static_cast<__nv_bfloat16*>(out);
  if (vec)
    meanpool_kernel<true><<<grid, kThreads, 0, stream>>>(src, dst, n, G, Hkv, mode);
  else
    meanpool_kernel<false><<<grid, kThreads, 0, stream>>>(src, dst, n, G, Hkv, mode);
  return cudaGetLastError();
}

}  // namespace gqa
