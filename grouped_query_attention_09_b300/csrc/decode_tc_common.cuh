// decode_tc_common.cuh -- pieces of the tcgen05 decode kernel (decode_tc.cu)
// kept apart from its main loop: the walk over the flattened
// (b, kv head, 128-key block) space, the owner of a block under the equal
// contiguous split, a bounded drain wait, and the log-sum-exp merge of the
// pieces of a (b, kv head) pair that the split cut apart.
//
// Split-KV is the "分块计算与内存优化" passage of the gsyq.cn page on xformers
// (K/V cut into blocks that are computed apart and reduced); the merge is the
// log-sum-exp reduction of those blocks' partial softmax states.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace gqa {
namespace tcd {

constexpr int kD = 128;
constexpr int kBN = 128;                   // keys per block
constexpr int kBlockBytes = kBN * kD * 2;  // one K or V block: 32 KiB
constexpr int kHalf = kBlockBytes / 2;     // one 64-column half (128-byte rows)
constexpr int kMaxBatch = 1024;
constexpr int kMaxCtas = 160;
constexpr int kSmemLimit = 232448;
constexpr float kRebase = 8.0f;            // log2 units a score may pass the reference max by

// Position in the flattened (b, kv head j, block) space.
struct Iter {
  int b, j, lt, nb;
};

__device__ inline void it_next(Iter& it, const int* pre, int B, int Hkv) {
  if (++it.lt < it.nb) return;
  it.lt = 0;
  if (++it.j < Hkv) return;
  it.j = 0;
  do { ++it.b; } while (it.b < B && pre[it.b + 1] == pre[it.b]);
  it.nb = it.b < B ? pre[it.b + 1] - pre[it.b] : 0;
}

// The equal contiguous split in 32-bit arithmetic (no 64-bit division on the
// kernel's start-up path): T < 2^31 / kMaxCtas blocks, P <= kMaxCtas shares,
// share c = [start(c), start(c + 1)) with start(c) = floor(c T / P)
// = c base + floor(c rem / P).
struct Split {
  int T, P, base, rem;
};

__device__ inline Split make_split(int T, int P) {
  Split s;
  s.T = T;
  s.P = P;
  s.base = P > 0 ? T / P : 0;
  s.rem = P > 0 ? T - s.base * P : 0;
  return s;
}

__device__ inline int share_start(const Split& s, int c) { return s.base * c + (s.rem * c) / s.P; }

// CTA whose share holds block t (0 <= t < T): the largest c with start(c) <= t.
__device__ inline int share_owner(const Split& s, int t) {
  int c = (int)((float)t * (float)s.P / (float)s.T);
  c = c < 0 ? 0 : (c >= s.P ? s.P - 1 : c);
  while (c + 1 < s.P && share_start(s, c + 1) <= t) ++c;
  while (c > 0 && share_start(s, c) > t) --c;
  return c;
}

__device__ inline void it_seek32(Iter& it, int t, const int* pre, int B, int Hkv) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (Hkv * pre[mid] <= t) lo = mid; else hi = mid - 1;
  }
  it.b = lo;
  it.nb = pre[lo + 1] - pre[lo];
  const int r = t - Hkv * pre[lo];
  it.j = r / it.nb;
  it.lt = r - it.j * it.nb;
}

__device__ inline int clamp_seq(int len, int Lmax) { return len < 0 ? 0 : (len > Lmax ? Lmax : len); }

// A wait bounded by the default limit only (draining in-flight work on exit).
__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity, unsigned* err) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, GQA_DEV_WAIT_TIMEOUT);
      return;
    }
  }
}

// Merge of the nseg pieces of one pair, held in the partial slots of CTAs
// c_lo .. c_lo + nseg - 1 (slot 1 for the piece that starts the pair, slot 0
// after it): part_acc [slot][G][D] unnormalised sums, part_ml [slot][2][G]
// (running max in log2 units, then the sum of weights).  out = sum_s
// 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s, rounded to bf16.  Run by nthr
// threads (r = 0 .. nthr - 1, nthr a multiple of 4): thread r covers heads
// h0 + r / 4 (h0 stepping by nthr / 4) and columns [32 (r % 4), 32 (r % 4) + 32).
// Up to four pieces have every load of the thread issued at once (one round
// trip to L2 -- the partials were written by other SMs, possibly on the other
// die); more take a two-pass loop.
static __device__ __noinline__ void merge_pieces(const float* part_acc, const float* part_ml, int G, int c_lo,
                                                int nseg, __nv_bfloat16* outp, int r, int nthr = 128) {
  constexpr int kFastSeg = 4;
  for (int h0 = 0; h0 < G && nseg <= kFastSeg; h0 += nthr / 4) {
    const int h = h0 + (r >> 2), cg = r & 3;
    if (h < G) {
      float ms[kFastSeg], ls[kFastSeg];
      float4 x[kFastSeg][8];
#pragma unroll
      for (int s2 = 0; s2 < kFastSeg; ++s2) {
        if (s2 < nseg) {
          const size_t si = (size_t)(c_lo + s2) * 2 + (s2 == 0 ? 1 : 0);
          ms[s2] = __ldcg(part_ml + (si * 2 + 0) * G + h);
          ls[s2] = __ldcg(part_ml + (si * 2 + 1) * G + h);
          const float4* src = reinterpret_cast<const float4*>(part_acc + (si * G + h) * kD + cg * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v) x[s2][v] = __ldcg(src + v);
        } else {
          ms[s2] = -INFINITY;
          ls[s2] = 0.f;
#pragma unroll
          for (int v = 0; v < 8; ++v) x[s2][v] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float M = ms[0];
#pragma unroll
      for (int s2 = 1; s2 < kFastSeg; ++s2) M = fmaxf(M, ms[s2]);
      const float Mu = M == -INFINITY ? 0.f : M;
      float Ls = 0.f, f[kFastSeg];
#pragma unroll
      for (int s2 = 0; s2 < kFastSeg; ++s2) {
        f[s2] = fast_exp2(ms[s2] - Mu);
        Ls += f[s2] * ls[s2];
      }
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(outp + (size_t)h * kD + cg * 32);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
#pragma unroll
        for (int s2 = 0; s2 < kFastSeg; ++s2) {
          const float4 y0 = x[s2][2 * v], y1 = x[s2][2 * v + 1];
          a0.x += f[s2] * y0.x;
          a0.y += f[s2] * y0.y;
          a0.z += f[s2] * y0.z;
          a0.w += f[s2] * y0.w;
          a1.x += f[s2] * y1.x;
          a1.y += f[s2] * y1.y;
          a1.z += f[s2] * y1.z;
          a1.w += f[s2] * y1.w;
        }
        dst[v] = make_uint4(pack_bf16x2(a0.x * inv, a0.y * inv), pack_bf16x2(a0.z * inv, a0.w * inv),
                            pack_bf16x2(a1.x * inv, a1.y * inv), pack_bf16x2(a1.z * inv, a1.w * inv));
      }
    }
  }
  for (int h0 = 0; h0 < G && nseg > kFastSeg; h0 += nthr / 4) {
    const int h = h0 + (r >> 2), cg = r & 3;
    if (h < G) {
      float M = -INFINITY;
#pragma unroll 4
      for (int s2 = 0; s2 < nseg; ++s2) {
        const size_t si = (size_t)(c_lo + s2) * 2 + (s2 == 0 ? 1 : 0);
        M = fmaxf(M, __ldcg(part_ml + (si * 2 + 0) * G + h));
      }
      const float Mu = M == -INFINITY ? 0.f : M;
      float Ls = 0.f;
      float4 acc4[8];
#pragma unroll
      for (int v = 0; v < 8; ++v) acc4[v] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
      for (int s2 = 0; s2 < nseg; ++s2) {
        const size_t si = (size_t)(c_lo + s2) * 2 + (s2 == 0 ? 1 : 0);
        const float f = fast_exp2(__ldcg(part_ml + (si * 2 + 0) * G + h) - Mu);
        Ls += f * __ldcg(part_ml + (si * 2 + 1) * G + h);
        const float4* src = reinterpret_cast<const float4*>(part_acc + (si * G + h) * kD + cg * 32);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float4 x = __ldcg(src + v);
          acc4[v].x += f * x.x;
          acc4[v].y += f * x.y;
          acc4[v].z += f * x.z;
          acc4[v].w += f * x.w;
        }
      }
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(outp + (size_t)h * kD + cg * 32);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const float4 a0 = acc4[2 * v], a1 = acc4[2 * v + 1];
        dst[v] = make_uint4(pack_bf16x2(a0.x * inv, a0.y * inv), pack_bf16x2(a0.z * inv, a0.w * inv),
                            pack_bf16x2(a1.x * inv, a1.y * inv), pack_bf16x2(a1.z * inv, a1.w * inv));
      }
    }
  }
}

}  // namespace tcd
}  // namespace gqa
