// rope.cu -- the step before a decode: rotary position embedding of the new
// token's query and key heads, and the append of its key and value heads to
// the KV cache.
//
// The attention code of the GQA paper notes on 51969.com ("QA 相关") rotates
// query_states and key_states with apply_rotary_pos_emb(.., cos, sin) before
// repeat_kv; the Huawei Cloud post "多头注意力机制的代码实现（MQA和GQA）",
// sections 2 and 5, concatenates each step's K and V to the layer's cache.
// Here the cache is the preallocated bf16 [B, Hkv, Lmax, D] tensor of the
// decode path, the new token of sequence b sits at position p = seqlens[b],
// and the rotation is the Llama "rotate half" form (the pages do not spell it
// out): for i < D/2 the pair (x[i], x[i + D/2]) turns by p * base^(-2i/D).
//
// One CTA per sequence: the D/2 frequencies base^(-2i/D) come in fp64 from
// the host (the device then needs no fp64 transcendental), the angles p *
// freq are formed and reduced modulo 2 pi in fp64 before an fp32 sincos (so
// positions in the tens of thousands keep full precision); then every thread
// rotates chunks of 8 pairs of the query and key heads with 16-byte loads,
// writes the key and value rows into the cache, and one thread advances
// seqlens[b] after a barrier.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kRopeThreads = 256;
constexpr int kMaxHalf = 128;  // D <= 256

__global__ void __launch_bounds__(kRopeThreads) rope_append_kernel(const __grid_constant__ RopeArgs a) {
  __shared__ float cs[kMaxHalf], sn[kMaxHalf];
  __shared__ int pos_s;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int half = a.D / 2;
  if (tid == 0) {
    const int p = a.seqlens[b];
    pos_s = p < 0 ? 0 : p;
    if (pos_s >= a.Lmax) atomicOr(a.err, GQA_DEV_CACHE_FULL);
  }
  __syncthreads();
  const int p = pos_s;
  for (int i = tid; i < half; i += kRopeThreads) {
    const double theta = (double)p * a.inv_freq[i];
    const double two_pi = 6.283185307179586476925286766559;
    const double inv_two_pi = 0.15915494309189533576888376337251;
    const double r = theta - two_pi * rint(theta * inv_two_pi);  // in [-pi, pi] up to rounding
    float s, c;
    sincosf((float)r, &s, &c);
    cs[i] = c;
    sn[i] = s;
  }
  __syncthreads();
  const bool write_row = p < a.Lmax;
  const int chunks = half / 8;  // 8 pairs per item
  const int items = (a.Hq + a.Hkv) * chunks;
  for (int e = tid; e < items; e += kRopeThreads) {
    const int h = e / chunks, i0 = (e % chunks) * 8;
    const __nv_bfloat16* src;
    __nv_bfloat16* dst;
    if (h < a.Hq) {
      src = a.q + ((size_t)b * a.Hq + h) * a.D;
      dst = a.q_out + ((size_t)b * a.Hq + h) * a.D;
    } else {
      const int j = h - a.Hq;
      src = a.k_new + ((size_t)b * a.Hkv + j) * a.D;
      if (!write_row) continue;
      dst = a.k_cache + (((size_t)b * a.Hkv + j) * a.Lmax + p) * a.D;
    }
    const uint4 lo = *reinterpret_cast<const uint4*>(src + i0);
    const uint4 hi = *reinterpret_cast<const uint4*>(src + i0 + half);
    const uint32_t lw[4] = {lo.x, lo.y, lo.z, lo.w}, hw[4] = {hi.x, hi.y, hi.z, hi.w};
    uint32_t ol[4], oh[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float x1[2], x2[2], y1[2], y2[2];
      x1[0] = __uint_as_float(lw[w] << 16);
      x1[1] = __uint_as_float(lw[w] & 0xFFFF0000u);
      x2[0] = __uint_as_float(hw[w] << 16);
      x2[1] = __uint_as_float(hw[w] & 0xFFFF0000u);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int i = i0 + 2 * w + t;
        y1[t] = x1[t] * cs[i] - x2[t] * sn[i];
        y2[t] = x2[t] * cs[i] + x1[t] * sn[i];
      }
      ol[w] = pack_bf16x2(y1[0], y1[1]);
      oh[w] = pack_bf16x2(y2[0], y2[1]);
    }
    *reinterpret_cast<uint4*>(dst + i0) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
    *reinterpret_cast<uint4*>(dst + i0 + half) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
  }
  // V rows: a copy into row p.
  if (write_row) {
    const int vchunks = a.Hkv * (a.D / 8);
    for (int e = tid; e < vchunks; e += kRopeThreads) {
      const int j = e / (a.D / 8), c = (e % (a.D / 8)) * 8;
      *reinterpret_cast<uint4*>(a.v_cache + (((size_t)b * a.Hkv + j) * a.Lmax + p) * a.D + c) =
          *reinterpret_cast<const uint4*>(a.v_new + ((size_t)b * a.Hkv + j) * a.D + c);
    }
  }
  __syncthreads();
  if (tid == 0 && write_row) a.seqlens[b] = p + 1;
}

}  // namespace

bool rope_supported(int D) { return D >= 16 && D <= 2 * kMaxHalf && D % 16 == 0; }

cudaError_t rope_append_launch(const RopeArgs& args, cudaStream_t stream) {
  if (!rope_supported(args.D)) return cudaErrorInvalidValue;
  RopeArgs a = args;
  for (int i = 0; i < a.D / 2; ++i) a.inv_freq[i] = std::pow(a.base, -2.0 * i / a.D);
  rope_append_kernel<<<a.B, kRopeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gqa
