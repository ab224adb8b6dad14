// prefill.cu -- causal (or full) grouped-query attention over a prompt of L
// tokens on the tcgen05 tensor cores (row a4 of the hot path), and its
// generalisation to a chunk of Lq queries that follows a cached prefix of
// Lk - Lq tokens (Lk keys in all; the causal mask aligned at the bottom right:
// chunk row i is token Lk - Lq + i and sees keys t <= Lk - Lq + i).
//
// Per head: out = softmax(QK^T / sqrt(D)) V with keys t <= i visible to query
// i when causal (the Huawei Cloud post "多头注意力机制的代码实现（MQA和GQA）",
// section 5 code: Q @ K^T, / sqrt(head_size), triu(ones, 1) -> -inf, softmax,
// @ V), where query head h reads KV head h / G (G = Hq / Hkv; the GQA paper
// notes on 51969.com, "分组查询注意力（GQA）"; `repeat_interleave` of
// "手把手教你用PyTorch实现GQA", section 1.3).  K/V are never expanded: one
// K/V block in shared memory serves two query heads of its group at once.
//
// Work unit: (b, kv head j, two query heads of group j, 128-row query block
// qb).  Each CTA is persistent and walks units heaviest first (causal units
// with a large qb see the most keys) in a snake order over the grid.
//
// Head dimension D = 128 or 64 (a template parameter; rows of 128 or 64 bf16
// are loaded as D / 64 boxes of 64 columns, 128 bytes per row).
//
// Warp roles (320 threads, one CTA per SM):
//   warps 0-3  softmax of query tile 0 (thread = one query row = one TMEM lane)
//   warps 4-7  softmax of query tile 1
//   warp  8    TMA producer: the two Q tiles of a unit, then K/V blocks into a
//              ring of slots of 128 x D bf16 (32 KiB at D = 128, 16 KiB at
//              D = 64; 5 or 8 slots; a slot holds one K or one V block)
//   warp  9    TMEM owner and tcgen05.mma issuer (the whole warp walks the
//              schedule, one elected lane issues)
//
// Per KV block j of a unit:
//   S_t = Q_t K_j^T           SS MMA: A = Q_t (smem, K-major), B = K_j (smem,
//                             K-major), fp32 accumulator in TMEM columns
//                             [128t, 128t + 128)
//   softmax_t                 thread r loads row r of S_t from TMEM, masks the
//                             diagonal block, keeps a running max (re-based only
//                             when it grows by more than 2^8 in log2 units, so O
//                             is rescaled rarely) and the running sum, and writes
//                             P = exp2(S*scale*log2e - m) as bf16 pairs back into
//                             the first 64 TMEM columns of S_t
//   O_t += P_t V_j            TS MMA: A = P_t read from TMEM, B = V_j (smem,
//                             MN-major), fp32 accumulator in TMEM columns
//                             [256 + 128t, 256 + 128t + D)
// The MMA warp interleaves the two tiles (S0, S1, PV0, S0', PV1, S1', ...),
// so that the tensor pipe works on one tile while the other tile's softmax
// runs.  TMEM: S0, S1, O0, O1 = 512 columns.  At the end of a unit each
// softmax thread reads its O row, divides by the running sum and stores bf16
// to global memory.
//
// Every wait is bounded; on expiry the kernel flags GQA_DEV_WAIT_TIMEOUT,
// every role leaves its loop, in-flight copies and MMAs are waited for (again
// bounded), and the TMEM is freed before the CTA exits.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>

#include "internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace gqa {
namespace {

constexpr int kBM = 128;         // query rows per tile
constexpr int kBN = 128;         // keys per block
constexpr int kBoxBytes = kBM * 128;  // one 64-column box of a tile (128-byte rows): 16 KiB
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kRebaseLog2 = 8.0f;  // re-base the running max when it grows by more

// Shared memory of the D instantiation (offsets from a 1024-byte aligned base).
template <int D>
struct Cfg {
  static constexpr int kTileBytes = kBM * D * 2;  // one Q tile, K or V block
  static constexpr int kStages = D == 64 ? 8 : 5;  // K/V ring depth (a slot holds one K or one V block)
  static constexpr int kOffQ = 0;                  // 2 query tiles
  static constexpr int kOffRing = kOffQ + 2 * kTileBytes;
  static constexpr int kOffBars = kOffRing + kStages * kTileBytes;
  static constexpr int kNumBars = 2 + 2 + kStages + kStages + 2 + 2 + 2 + 1;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;  // TMEM base, abort flag
  static constexpr size_t kSmemBytes = (size_t)kOffMisc + 16 + 1024;  // + alignment slack
};

struct Params {
  __nv_bfloat16* out;
  int B, Lq, Lk, Hq, Hkv, G;
  int prefix;       // Lk - Lq: cached tokens before the first query
  int nqb, nkb;     // query blocks ceil(Lq / 128), key blocks ceil(Lk / 128)
  int causal;
  int two;          // 1: a unit holds two heads of one group (G even)
  int per_group;    // units per (b, j, qb): G / 2 or G
  int units;
  float scale_log2;  // (1 / sqrt(D)) * log2(e)
  unsigned* err;
  unsigned long long wait_ns;  // pipeline-wait limit
  int starve;                  // test hook: the producer issues no loads
};

struct Unit {
  int b, j, h0, qb, n;
};

__device__ __forceinline__ Unit unit_at(const Params& p, int u) {
  const int per_qb = p.B * p.Hkv * p.per_group;
  const int rank = u / per_qb;
  const int rem = u - rank * per_qb;
  Unit x;
  x.qb = p.causal ? p.nqb - 1 - rank : rank;
  const int pr = rem % p.per_group;
  const int bj = rem / p.per_group;
  x.j = bj % p.Hkv;
  x.b = bj / p.Hkv;
  x.h0 = x.j * p.G + (p.two ? 2 * pr : pr);
  // causal: keys up to the last row of the block, token prefix + min(128 qb + 127, Lq - 1)
  x.n = p.causal ? min((p.prefix + min(x.qb * kBM + kBM - 1, p.Lq - 1)) / kBN + 1, p.nkb) : p.nkb;
  return x;
}

// The i-th unit of this CTA (snake order over the grid), or -1.
__device__ __forceinline__ int my_unit(const Params& p, int i) {
  const int w = i;
  const int c = (w & 1) ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
  const int u = w * (int)gridDim.x + c;
  return u < p.units ? u : -1;
}

// A wait that is bounded by time only (used while draining on exit).
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity, unsigned* err) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, GQA_DEV_WAIT_TIMEOUT);
      return;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const Params p) {
  using C = Cfg<D>;
  constexpr int kTileBytes = C::kTileBytes, kStages = C::kStages;
  constexpr int kOffQ = C::kOffQ, kOffRing = C::kOffRing, kOffBars = C::kOffBars, kOffMisc = C::kOffMisc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 2;
  uint64_t* kv_full = bars + 4;
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_full = kv_empty + kStages;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = p_full + 2;
  uint64_t* mma_done = o_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&q_empty[t], 1);
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
      mbar_init(&o_full[t], 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && !p.starve) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      uint32_t kv_it = 0;
      uint32_t slot_used = 0, slot_par = 0;  // bit s: slot s was loaded / its last parity
      int q_used = 0;
      bool ok = true;
      int i = 0;
      for (int u = my_unit(p, 0); u >= 0 && ok; u = my_unit(p, ++i)) {
        const Unit x = unit_at(p, u);
        for (int t = 0; t < 1 + p.two && ok; ++t) {
          ok = mbar_wait_bounded(&q_empty[t], (i & 1) ^ 1, abort_flag, p.err, p.wait_ns);
          if (!ok) break;
          uint8_t* dst = smem + kOffQ + t * kTileBytes;
          mbar_arrive_expect_tx(&q_full[t], kTileBytes);
          const int row = x.b * p.Hq + x.h0 + t;
#pragma unroll
          for (int box = 0; box < D / 64; ++box)
            tma_load_3d(dst + box * kBoxBytes, &tm_q, box * 64, x.qb * kBM, row, &q_full[t], pol_q);
          q_used = i + 1;
        }
        const int kvrow = x.b * p.Hkv + x.j;
        for (int jb = 0; jb < x.n && ok; ++jb) {
          for (int kv = 0; kv < 2; ++kv) {
            const int s = kv_it % kStages;
            const uint32_t par = (kv_it / kStages) & 1;
            ok = mbar_wait_bounded(&kv_empty[s], par ^ 1, abort_flag, p.err, p.wait_ns);
            if (!ok) break;
            uint8_t* dst = smem + kOffRing + s * kTileBytes;
            const CUtensorMap* m = kv ? &tm_v : &tm_k;
            mbar_arrive_expect_tx(&kv_full[s], kTileBytes);
#pragma unroll
            for (int box = 0; box < D / 64; ++box)
              tma_load_3d(dst + box * kBoxBytes, m, box * 64, jb * kBN, kvrow, &kv_full[s], pol_kv);
            slot_used |= 1u << s;
            slot_par = (slot_par & ~(1u << s)) | (par << s);
            ++kv_it;
          }
        }
      }
      // Drain: every copy this thread started has landed before the CTA exits.
      for (int s = 0; s < kStages; ++s)
        if (slot_used >> s & 1u) mbar_wait_drain(&kv_full[s], slot_par >> s & 1u, p.err);
      if (q_used)
        for (int t = 0; t < 1 + p.two; ++t) mbar_wait_drain(&q_full[t], (q_used - 1) & 1, p.err);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp walks the schedule and waits on the barriers, so that
    // every descriptor is a warp-uniform value; one elected lane issues the
    // MMAs and the commits that track them.
    constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kBM, kBN, false);
    constexpr uint32_t idesc_o = tc::idesc_bf16_f32(kBM, D, true);
    const bool leader = elect_one_sync();
    // Descriptors of the tile bases; the address field (bits 0-13, in 16-byte
    // units) is advanced by adding the byte offset >> 4 (no carry: smem < 256 KiB).
    const uint64_t dq = tc::sdesc_sw128(smem_u32(smem + kOffQ), 16, 1024);
    const uint64_t dk = tc::sdesc_sw128(smem_u32(smem + kOffRing), 16, 1024);
    // (the leading-byte offset steps between 64-column boxes along N = D)
    const uint64_t dv = tc::sdesc_sw128(smem_u32(smem + kOffRing), kBoxBytes, 1024);
    auto issue_s = [&](int t, int slot) {
      const uint64_t a0 = dq + (uint64_t)((t * kTileBytes) >> 4);
      const uint64_t b0 = dk + (uint64_t)((slot * kTileBytes) >> 4);
      if (leader) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t off = (uint64_t)(((k >> 2) * kBoxBytes + (k & 3) * 32) >> 4);
          tc::mma_ss(tmem + t * 128, a0 + off, b0 + off, idesc_s, k > 0);
        }
      }
    };
    // P_t sits in TMEM columns [128t, 128t + 64) (over the S_t it came
    // from), 16 keys = 8 columns per instruction.
    auto issue_pv = [&](int t, int slot, bool acc) {
      const uint64_t b0 = dv + (uint64_t)((slot * kTileBytes) >> 4);
      if (leader) {
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)
          tc::mma_ts(tmem + 256 + t * 128, tmem + t * 128 + k * 8, b0 + (uint64_t)((k * 16 * 128) >> 4), idesc_o,
                     (acc || k > 0) ? 1u : 0u);
      }
    };
    auto commit = [&](uint64_t* bar) {
      if (leader) tc::commit(bar);
    };
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      const bool w = mbar_wait_bounded(bar, parity, abort_flag, p.err, p.wait_ns);
      return __all_sync(0xffffffffu, w);
    };
    uint32_t kv_it = 0, pc0 = 0, pc1 = 0;
    bool ok = true;
    int i = 0;
    for (int u = my_unit(p, 0); u >= 0 && ok; u = my_unit(p, ++i)) {
      const Unit x = unit_at(p, u);
      const int nt = 1 + p.two;
      for (int t = 0; t < nt && ok; ++t) ok = wait(&q_full[t], i & 1);
      if (!ok) break;
      int ks = kv_it % kStages;
      ok = wait(&kv_full[ks], (kv_it / kStages) & 1);
      if (!ok) break;
      ++kv_it;
      tc::fence_after_sync();
      for (int t = 0; t < nt; ++t) {
        issue_s(t, ks);
        commit(&s_full[t]);
        if (x.n == 1) commit(&q_empty[t]);
      }
      commit(&kv_empty[ks]);
      for (int jb = 0; jb < x.n && ok; ++jb) {
        // V of this block and K of the next one first: both were usually
        // loaded long ago, and P0 is the wait on the critical path.
        const int vs = kv_it % kStages;
        ok = wait(&kv_full[vs], (kv_it / kStages) & 1);
        if (!ok) break;
        ++kv_it;
        int ks2 = -1;
        if (jb + 1 < x.n) {
          ks2 = kv_it % kStages;
          ok = wait(&kv_full[ks2], (kv_it / kStages) & 1);
          if (!ok) break;
          ++kv_it;
        }
        ok = wait(&p_full[0], pc0 & 1);
        if (!ok) break;
        ++pc0;
        tc::fence_after_sync();
        issue_pv(0, vs, jb > 0);
        if (ks2 >= 0) {
          issue_s(0, ks2);
          commit(&s_full[0]);
          if (jb + 2 == x.n) commit(&q_empty[0]);
        } else {
          commit(&o_full[0]);
        }
        if (!p.two) {
          commit(&kv_empty[vs]);
          if (ks2 >= 0) commit(&kv_empty[ks2]);
          continue;
        }
        ok = wait(&p_full[1], pc1 & 1);
        if (!ok) break;
        ++pc1;
        tc::fence_after_sync();
        issue_pv(1, vs, jb > 0);
        commit(&kv_empty[vs]);
        if (ks2 >= 0) {
          issue_s(1, ks2);
          commit(&s_full[1]);
          if (jb + 2 == x.n) commit(&q_empty[1]);
          commit(&kv_empty[ks2]);
        } else {
          commit(&o_full[1]);
        }
      }
    }
    // Drain: every MMA issued has completed before TMEM is freed.
    commit(mma_done);
    mbar_wait_drain(mma_done, 0, p.err);
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;           // query tile 0 or 1
    const int r = (warp & 3) * 32 + lane;  // row of the tile = TMEM lane
    const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_tm = tmem + lane_addr + t * 128;
    const uint32_t o_tm = tmem + lane_addr + 256 + t * 128;
    uint32_t sc = 0, oc = 0;
    bool ok = (t == 0) || p.two;
    int i = 0;
    for (int u = ok ? my_unit(p, 0) : -1; u >= 0 && ok; u = my_unit(p, ++i)) {
      const Unit x = unit_at(p, u);
      const int h = x.h0 + t;
      const int qi = x.qb * kBM + r;  // query position of this row
      float m_use = -INFINITY, l = 0.f;
      for (int jb = 0; jb < x.n; ++jb) {
        ok = mbar_wait_bounded(&s_full[t], sc & 1, abort_flag, p.err, p.wait_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ++sc;
        tc::fence_after_sync();
        uint32_t s[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::ld_32x32b_x32(s_tm + c * 32, s[c]);
        tc::wait_ld_regs(s[0]);
        tc::pin_regs(s[1]);
        tc::pin_regs(s[2]);
        tc::pin_regs(s[3]);
        const int key0 = jb * kBN;
        // Mask where some key of the block lies past the first row's token
        // (causal) or past the last key.
        if ((p.causal && key0 + kBN - 1 > p.prefix + x.qb * kBM) || key0 + kBN > p.Lk) {
          const int lim = p.causal ? min(p.prefix + qi, p.Lk - 1) : p.Lk - 1;  // last visible key
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (key0 + c * 32 + e > lim) s[c][e] = __float_as_uint(-INFINITY);
        }
        // Row max: 8 independent chains of 3-input max, then a tree.
        float mxv[8];
#define SV(i) __uint_as_float(s[(i) >> 5][(i) & 31])
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          // chain e takes elements e + 8m, m = 0..15
          float m = fmax3(SV(e), SV(e + 8), SV(e + 16));
#pragma unroll
          for (int q = 3; q < 15; q += 2) m = fmax3(m, SV(e + 8 * q), SV(e + 8 * (q + 1)));
          mxv[e] = fmaxf(m, SV(e + 120));
        }
#undef SV
        mxv[0] = fmax3(mxv[0], mxv[1], mxv[2]);
        mxv[3] = fmax3(mxv[3], mxv[4], mxv[5]);
        mxv[6] = fmaxf(mxv[6], mxv[7]);
        mxv[0] = fmax3(mxv[0], mxv[3], mxv[6]);
        const float mx = mxv[0];
        const float mxs = mx * p.scale_log2;
        const bool rebase = mxs > m_use + kRebaseLog2;
        const bool any_rebase = __any_sync(0xffffffffu, rebase);
        const float m_new = rebase ? mxs : m_use;
        const float alpha = rebase ? fast_exp2(m_use - m_new) : 1.f;
        m_use = m_new;
        const float ref = (m_use == -INFINITY) ? 0.f : m_use;
        // P = exp2(S * scale * log2e - ref) as bf16 pairs, written over the
        // first 64 TMEM columns of S_t (row r = lane r).
        float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const float sl = p.scale_log2, nref = -ref;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pw[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float x0, x1;
            fma2(x0, x1, __uint_as_float(s[c][2 * e]), __uint_as_float(s[c][2 * e + 1]), sl, sl, nref, nref);
            const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
            ls[2 * (e & 3)] += p0;
            ls[2 * (e & 3) + 1] += p1;
            pw[e] = pack_bf16x2(p0, p1);
          }
          tc::st_32x32b_x16(s_tm + c * 16, pw);
        }
        const float lsum = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        l = l * alpha + lsum;
        // O holds the blocks before this one (the commit that signalled S
        // also covered the previous P V); bring it to the new reference.
        if (any_rebase && jb > 0) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tc::ld_32x32b_x32(o_tm + c * 32, o);
            tc::wait_ld_regs(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tc::st_32x32b_x32(o_tm + c * 32, o);
          }
        }
        tc::wait_st();
        tc::fence_before_sync();
        mbar_arrive(&p_full[t]);
      }
      if (!ok) break;
      ok = mbar_wait_bounded(&o_full[t], oc & 1, abort_flag, p.err, p.wait_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ++oc;
      tc::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.out + ((size_t)(x.b * p.Hq + h) * p.Lq + qi) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tc::ld_32x32b_x32(o_tm + c * 32, o);
        tc::wait_ld_regs(o);
        if (qi < p.Lq) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(o[v * 8 + 2 * e]) * inv, __uint_as_float(o[v * 8 + 2 * e + 1]) * inv);
            dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool prefill_supported(int D) { return D == 64 || D == 128; }

template <int D>
cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const Params& p, int grid,
                     cudaStream_t stream) {
  static std::atomic<unsigned long long> attr_set{0};  // one bit per device ordinal < 64
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(attr_set.load() >> dev & 1ull)) {
    e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set.fetch_or(1ull << dev);
  }
  prefill_kernel<D><<<grid, kThreads, Cfg<D>::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

cudaError_t prefill_launch(const PrefillArgs& a, int sm_count, cudaStream_t stream) {
  if (!prefill_supported(a.D)) return cudaErrorNotSupported;
  const int Lk = a.Lk > 0 ? a.Lk : a.L;
  if (Lk < a.L) return cudaErrorInvalidValue;
  const uint64_t rowb = (uint64_t)a.D * 2, qheadb = (uint64_t)a.L * a.D * 2, kheadb = (uint64_t)Lk * a.D * 2;
  CUtensorMap tq, tk, tv;
  if (encode_tmap_bf16_3d(&tq, a.q, a.D, a.L, (uint64_t)a.B * a.Hq, rowb, qheadb, 64, kBM, 1) != CUDA_SUCCESS ||
      encode_tmap_bf16_3d(&tk, a.k, a.D, Lk, (uint64_t)a.B * a.Hkv, rowb, kheadb, 64, kBN, 1) != CUDA_SUCCESS ||
      encode_tmap_bf16_3d(&tv, a.v, a.D, Lk, (uint64_t)a.B * a.Hkv, rowb, kheadb, 64, kBN, 1) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  Params p;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.B = a.B;
  p.Lq = a.L;
  p.Lk = Lk;
  p.prefix = Lk - a.L;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.Hq / a.Hkv;
  p.nqb = (a.L + kBM - 1) / kBM;
  p.nkb = (Lk + kBN - 1) / kBN;
  p.causal = a.causal;
  p.two = (p.G % 2 == 0) ? 1 : 0;
  p.per_group = p.two ? p.G / 2 : p.G;
  const long long units = (long long)a.B * a.Hkv * p.per_group * p.nqb;
  if (units > 0x7fffffff) return cudaErrorInvalidValue;
  p.units = (int)units;
  p.scale_log2 = (1.0f / sqrtf((float)a.D)) * 1.4426950408889634f;
  p.err = a.err;
  p.wait_ns = pipeline_wait_limit_ns();
  p.starve = pipeline_starved() ? 1 : 0;
  const int grid = (int)std::min<long long>(units, sm_count);
  return a.D == 64 ? launch_d<64>(tq, tk, tv, p, grid, stream) : launch_d<128>(tq, tk, tv, p, grid, stream);
}

}  // namespace gqa
