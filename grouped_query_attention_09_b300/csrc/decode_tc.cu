// decode_tc.cu -- split-KV GQA decode on the tcgen05 tensor cores, for wide
// groups (9 <= G <= 128 query heads per KV head at D = 128, e.g. multi-query
// attention).
//
// Same computation as decode.cu: for every sequence b and query head h, the
// new query attends to the first seqlens[b] rows of KV head j = h / G of the
// bf16 [B, Hkv, Lmax, D] cache (the GQA paper notes on 51969.com, "分组查询
// 注意力（GQA）"; the Huawei Cloud post "多头注意力机制的代码实现（MQA和GQA）",
// section 5: scores q.k / sqrt(d), softmax, weighted sum of V).  With a wide
// group the warp-level MMA path re-reads every K/V tile from shared memory once
// per head slice; here the G query heads of a (b, j) pair are the M rows of one
// tcgen05.mma (rows G..127 are padding and never read back), so each K/V block
// crosses HBM once and shared memory once.
//
// Split ("Split-KV": the gsyq.cn page on xformers, "分块计算与内存优化"): the
// flattened (b, j, 128-key block) space is cut into equal contiguous shares,
// one per persistent CTA; a pair cut by share boundaries is merged by
// log-sum-exp by the CTA that completes its last piece (arrival counter), as
// in decode.cu, with the same workspace layout.
//
// Per block i of the share (warp roles, 256 threads):
//   warp 0  TMA producer: the pair's Q tile [128 x D] once per piece (rows >=
//           G are out of range and arrive as zeros), then K_i and V_i into a
//           ring of 32 KiB stages.
//   warp 1  TMEM owner and MMA issuer (all lanes walk the schedule, one
//           elected lane issues): S_i = Q K_i^T into S buffer i % 2, then
//           O += P_{i-1} V_{i-1} -- the next block's scores are computed while
//           the softmax of the current one runs.
//   warps 2-3  bf16 cache: publisher of the cut pieces before the share's
//           last one (count the piece in; the CTA that completes a pair's
//           count merges it).  FP8 cache: E4M3 -> fp16 converters (below).
//   warps 4-7  softmax and epilogue, one thread per query head (TMEM lane):
//           mask keys past seqlens[b], running max (re-based only when it
//           grows by more than 2^8), P = exp2(.) as bf16 over the S buffer,
//           running sum; at the end of a piece, O / l to the output or the
//           partial slot (publishing the share's last cut piece itself).
//           Warps whose 32 lanes are all padding rows skip the TMEM work but
//           keep the barrier protocol.
// TMEM: S buffers at columns [0, 128) and [128, 256), O at [256, 384).
//
// Every wait is bounded; on expiry GQA_DEV_WAIT_TIMEOUT is flagged, the roles
// leave their loops, in-flight copies and MMAs are drained (bounded) and the
// TMEM is freed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "decode_tc_common.cuh"
#include "tcgen05.cuh"

namespace gqa {
namespace {

using namespace tcd;

constexpr int kQBytes = 128 * kD * 2;         // Q tile: 32 KiB
constexpr int kThreads = 256;
constexpr int kColO = 256;

struct TcParams {
  const __nv_bfloat16* q;  // read directly only for an FP8 cache (else through tmQ)
  __nv_bfloat16* out;
  const int32_t* seqlens;
  float* part_acc;  // [num_ctas][2][G][D]
  float* part_ml;   // [num_ctas][2][2][G]
  int* counters;    // [B * Hkv]
  unsigned* err;
  int B, Hq, Hkv, G, Lmax, stages, num_ctas;
  float scale_log2;
  const int32_t* block_table;  // paged cache (else null): [B][max_pages]
  int page_size, max_pages, num_pages;
  unsigned long long wait_ns;  // pipeline-wait limit
  int starve;                  // test hook: the producer issues no loads
  // FP8 (E4M3) cache: per (b, kv head) scales of K and V, and the depth of
  // the ring the E4M3 blocks land in before their conversion.
  const float* k_scale;
  const float* v_scale;
  int stages8;
};

constexpr int kBlockBytes8 = kBN * kD;  // one E4M3 K or V block: 16 KiB

struct TcLayout {
  int ring_off, ring8_off, pre_off, bar_off, misc_off, total;
};

// stages: the ring the MMAs read (bf16, or fp16 converted from E4M3);
// stages8: the ring E4M3 blocks land in (0 for a bf16 cache).
__host__ __device__ inline TcLayout tc_layout(int stages, int stages8) {
  TcLayout l;
  l.ring_off = kQBytes;
  l.ring8_off = l.ring_off + stages * kBlockBytes;
  l.pre_off = l.ring8_off + stages8 * kBlockBytes8;
  l.bar_off = l.pre_off + ((kMaxBatch + 1) * 4 + 7) / 8 * 8;
  // q_full, q_empty, kv_full[S], kv_empty[S], s_full[2], p_full[2], o_done, o_full, mma_done,
  // e8_full[S8], e8_empty[S8], pub_full[2]
  l.misc_off = l.bar_off + (2 + 2 * stages + 2 + 2 + 3 + 2 * stages8 + 2) * 8;
  l.total = l.misc_off + 4 * 40 + 1024;  // flags + scan scratch, + alignment slack
  return l;
}

// KV8: the cache holds E4M3 bytes.  The producer then lands each K or V
// block in an E4M3 ring; warps 2-3 convert it (exactly) to fp16 in the
// 128-byte-swizzled layout the MMAs read, zeroing the V rows past the
// sequence end, and also write the pair's q as fp16 into the Q tile; the
// MMAs run in fp16 (kind::f16 with f16 operands), P is fp16, the K scale
// joins the logit scale and the V scale the output.
template <bool KV8>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const TcParams p) {
  const int S8 = KV8 ? p.stages8 : 1;  // (1 keeps the bf16 instantiation free of a modulo by zero)
  const TcLayout L = tc_layout(p.stages, KV8 ? p.stages8 : 0);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_tile = smem;
  uint8_t* ring = smem + L.ring_off;
  uint8_t* ring8 = smem + L.ring8_off;
  int* pre = reinterpret_cast<int*>(smem + L.pre_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* kv_full = bars + 2;
  uint64_t* kv_empty = kv_full + p.stages;
  uint64_t* s_full = kv_empty + p.stages;  // [2]
  uint64_t* p_full = s_full + 2;           // [2]
  uint64_t* o_done = p_full + 2;
  uint64_t* o_full = o_done + 1;
  uint64_t* mma_done = o_full + 1;
  // (The E4M3 ring's barriers exist only with KV8: tc_layout reserves 2 S8
  // of them then and none for a bf16 cache, so the pointers step by 0 there.)
  const int S8b = KV8 ? p.stages8 : 0;
  uint64_t* e8_full = mma_done + 1;    // [S8] an E4M3 block landed (KV8)
  uint64_t* e8_empty = e8_full + S8b;  // [S8] ... and was converted (KV8)
  uint64_t* pub_full = e8_empty + S8b;  // [2] partial slot 0 / 1 written (bf16 cache: merged by warps 2-3)
  int* misc = reinterpret_cast<int*>(smem + L.misc_off);
  volatile int* abort_flag = misc;
  volatile int* merge_flags = misc + 4;  // [2][2]: last-piece flag and owner of the last piece, per publisher
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 3);
  int* scan = misc + 8;  // [8]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.B, Hkv = p.Hkv, G = p.G;

  // The sequence lengths first: their cold read overlaps the set-up below.
  constexpr int kLensPerThread = kMaxBatch / kThreads;
  const int per = (B + kThreads - 1) / kThreads;
  const int lo = tid * per, hi = min(B, lo + per);
  int lens[kLensPerThread];
#pragma unroll
  for (int k = 0; k < kLensPerThread; ++k) lens[k] = (lo + k < hi) ? __ldg(p.seqlens + lo + k) : 0;

  // With KV8 the Q tile and the blocks the MMAs read are written by the 64
  // converter threads (warps 2-3) instead of by TMA.
  constexpr int kConv = 64;
  if (tid == 0) {
    mbar_init(q_full, KV8 ? kConv : 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&kv_full[s], KV8 ? kConv : 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; KV8 && s < S8; ++s) {
      mbar_init(&e8_full[s], 1);
      mbar_init(&e8_empty[s], kConv);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&s_full[k], 1);
      mbar_init(&p_full[k], 128);
    }
    mbar_init(o_done, 1);
    mbar_init(o_full, 1);
    mbar_init(mma_done, 1);
    mbar_init(&pub_full[0], 128);
    mbar_init(&pub_full[1], 128);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }

  // ---- blocks per sequence and their exclusive prefix pre[0..B]
  {
    int local = 0;
    unsigned flags = 0;
#pragma unroll
    for (int k = 0; k < kLensPerThread; ++k) {
      if (lo + k < hi) {
        if (lens[k] > p.Lmax) flags |= GQA_DEV_SEQLEN_CLAMPED;
        if (lens[k] <= 0) flags |= GQA_DEV_EMPTY_CONTEXT;
        local += (clamp_seq(lens[k], p.Lmax) + kBN - 1) / kBN;
      }
    }
    if (flags && blockIdx.x == 0) atomicOr(p.err, flags);
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) scan[warp] = incl;
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) {
      const int w = lane < kThreads / 32 ? scan[lane] : 0;
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += v;
      }
      if (lane < kThreads / 32) scan[lane] = wi - w;
    }
    __syncthreads();
    int run = scan[warp] + incl - local;
#pragma unroll
    for (int k = 0; k < kLensPerThread; ++k) {
      if (lo + k < hi) {
        pre[lo + k] = run;
        run += (clamp_seq(lens[k], p.Lmax) + kBN - 1) / kBN;
      }
    }
    if (lo < B && hi == B) pre[B] = run;
  }
  __syncthreads();
  const uint32_t tmem = *tmem_slot;

  // Shares in 32-bit arithmetic (the host guarantees T < 2^31 / 160): no
  // 64-bit division on the start-up path.  CTAs that take a share: about one
  // per six blocks, at most one per SM.  Longer shares mean fewer cut pairs
  // (each a merge through L2) and a gentler burst of ring fills at launch; a
  // sweep over ragged G = 32 batches of 134 to 1018 blocks put six blocks per
  // CTA within a few percent of the best count at every size (134 blocks:
  // 25.6 us on 23 CTAs against 30.5 us on 134; 287 blocks: 26.8 us on 48
  // against 33.3 us on 148).  The others only zero-fill.
  const int T = Hkv * pre[B];
  const int P = min(p.num_ctas, (T + 5) / 6);
  const Split sp = make_split(T, P);
  const bool active = (int)blockIdx.x < P;
  const int s_c = active ? share_start(sp, blockIdx.x) : 0;
  const int e_c = active ? share_start(sp, blockIdx.x + 1) : 0;

  // Zero the outputs of sequences with an empty context.
  for (int b = blockIdx.x; b < B; b += p.num_ctas) {
    if (pre[b + 1] != pre[b]) continue;
    __nv_bfloat16* o = p.out + (size_t)b * p.Hq * kD;
    for (int e = tid; e < p.Hq * kD; e += kThreads) o[e] = __float2bfloat16_rn(0.f);
  }

  // The piece of pair (it.b, it.j) that ends here sits in this CTA's partial
  // slot: count it in; the CTA whose piece completes the pair's count merges
  // all the pieces into the output.  Run by the nthr threads r = 0 .. nthr-1
  // that meet at named barrier bar_id (every one of them, also after an
  // abort, so that the barrier counts always match); flag 0 or 1 picks the
  // shared words it broadcasts through (the softmax group and warps 2-3 may
  // publish at the same time).
  auto publish_merge = [&](const Iter& it, __nv_bfloat16* outp, int r, int nthr, int bar_id, int flag) {
    volatile int* merge_flag = merge_flags + 2 * flag;
    volatile int* chi_flag = merge_flag + 1;
    named_bar_sync(bar_id, nthr);
    if (r == 0 && !*abort_flag) {
      const int o_p = Hkv * pre[it.b] + it.j * it.nb;
      const int c_lo = share_owner(sp, o_p);
      const int c_hi = share_owner(sp, o_p + it.nb - 1);
      const int pair = it.b * Hkv + it.j;
      const int old = atomic_add_acq_rel_gpu(&p.counters[pair], 1);
      const bool lastc = old == c_hi - c_lo;
      if (lastc) p.counters[pair] = 0;  // ready for the next call (ordered by the kernel boundary)
      *merge_flag = lastc ? c_lo + 1 : 0;
      *chi_flag = c_hi;
    } else if (r == 0) {
      *merge_flag = 0;
    }
    named_bar_sync(bar_id, nthr);
    const int lf = *merge_flag;
    if (lf) {
      const int c_lo = lf - 1, nseg = *chi_flag - c_lo + 1;
      merge_pieces(p.part_acc, p.part_ml, G, c_lo, nseg, outp, r, nthr);
    }
    named_bar_sync(bar_id, nthr);
  };

  auto kslot = [&](int i) { return (2 * i) % p.stages; };
  auto kpar = [&](int i) { return (uint32_t)(((2 * i) / p.stages) & 1); };
  auto vslot = [&](int i) { return (2 * i + 1) % p.stages; };
  auto vpar = [&](int i) { return (uint32_t)(((2 * i + 1) / p.stages) & 1); };

  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0 && s_c < e_c && !p.starve) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t pol = l2_policy_evict_first();
      Iter it;
      it_seek32(it, s_c, pre, B, Hkv);
      int seg = 0;
      int issued = 0;
      bool ok = true;
      int pg_b = -1, pg_lp = -1, pg = 0;  // last block-table entry read (paged cache)
      for (int t = s_c; t < e_c && ok; ++t) {
        const int i = t - s_c;
        const int z = it.b * Hkv + it.j;
        int kvz = z, kvy = it.lt * kBN;
        if (p.block_table) {
          // Paged cache: an out-of-range page index is flagged and sent
          // outside the tensor map, where TMA reads zeros.
          const int lp = kvy / p.page_size;
          if (it.b != pg_b || lp != pg_lp) {
            pg_b = it.b;
            pg_lp = lp;
            pg = __ldg(p.block_table + (size_t)it.b * p.max_pages + lp);
            if (pg < 0 || pg >= p.num_pages) {
              atomicOr(p.err, GQA_DEV_BAD_PAGE);
              pg = -1;
            }
          }
          kvz = pg < 0 ? -1 : pg * Hkv + it.j;
          kvy -= lp * p.page_size;
        }
        if (KV8) {
          // E4M3 blocks into their own ring; the converters take them on
          for (int kv = 0; kv < 2 && ok; ++kv) {
            const int n = 2 * i + kv, s8 = n % S8;
            if (n >= S8) {
              ok = mbar_wait_bounded(&e8_empty[s8], (uint32_t)(((n / S8) & 1) ^ 1), abort_flag, p.err, p.wait_ns);
              if (!ok) break;
            }
            mbar_arrive_expect_tx(&e8_full[s8], kBlockBytes8);
            tma_load_3d(ring8 + s8 * kBlockBytes8, kv ? &tmV : &tmK, 0, kvy, kvz, &e8_full[s8], pol);
            issued = n + 1;
          }
          it_next(it, pre, B, Hkv);
          continue;
        }
        if (t == s_c || it.lt == 0) {
          ok = mbar_wait_bounded(q_empty, (seg & 1) ^ 1, abort_flag, p.err, p.wait_ns);
          if (!ok) break;
          mbar_arrive_expect_tx(q_full, kQBytes);
          tma_load_3d(q_tile, &tmQ, 0, 0, z, q_full, pol);
          tma_load_3d(q_tile + kHalf, &tmQ, 64, 0, z, q_full, pol);
          ++seg;
        }
        for (int kv = 0; kv < 2 && ok; ++kv) {
          const int s = kv ? vslot(i) : kslot(i);
          const uint32_t par = kv ? vpar(i) : kpar(i);
          if (2 * i + kv >= p.stages) {
            ok = mbar_wait_bounded(&kv_empty[s], par ^ 1, abort_flag, p.err, p.wait_ns);
            if (!ok) break;
          }
          uint8_t* dst = ring + s * kBlockBytes;
          const CUtensorMap* m = kv ? &tmV : &tmK;
          mbar_arrive_expect_tx(&kv_full[s], kBlockBytes);
          tma_load_3d(dst, m, 0, kvy, kvz, &kv_full[s], pol);
          tma_load_3d(dst + kHalf, m, 64, kvy, kvz, &kv_full[s], pol);
          issued = 2 * i + kv + 1;
        }
        it_next(it, pre, B, Hkv);
      }
      // Drain: the last `stages` loads hold the latest use of every slot.
      if (KV8) {
        for (int n = issued > S8 ? issued - S8 : 0; n < issued; ++n)
          wait_drain(&e8_full[n % S8], (uint32_t)((n / S8) & 1), p.err);
      } else {
        for (int n = issued > p.stages ? issued - p.stages : 0; n < issued; ++n)
          wait_drain(&kv_full[n % p.stages], (uint32_t)((n / p.stages) & 1), p.err);
        if (seg > 0) wait_drain(q_full, (seg - 1) & 1, p.err);
      }
    }
  } else if (warp == 1) {
    // ================================================================ MMA
    constexpr uint32_t idesc_s = KV8 ? tc::idesc_f16_f32(128, kBN, false) : tc::idesc_bf16_f32(128, kBN, false);
    constexpr uint32_t idesc_o = KV8 ? tc::idesc_f16_f32(128, kD, true) : tc::idesc_bf16_f32(128, kD, true);
    const bool leader = elect_one_sync();
    const uint64_t dq = tc::sdesc_sw128(smem_u32(q_tile), 16, 1024);
    const uint64_t dk = tc::sdesc_sw128(smem_u32(ring), 16, 1024);
    const uint64_t dv = tc::sdesc_sw128(smem_u32(ring), kHalf, 1024);
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      const bool w = mbar_wait_bounded(bar, parity, abort_flag, p.err, p.wait_ns);
      return __all_sync(0xffffffffu, w);
    };
    auto commit = [&](uint64_t* bar) {
      if (leader) tc::commit(bar);
    };
    auto issue_s = [&](int i) {
      const uint64_t b0 = dk + (uint64_t)((kslot(i) * kBlockBytes) >> 4);
      const uint32_t d = tmem + (uint32_t)(i & 1) * 128;
      if (leader) {
#pragma unroll
        for (int k = 0; k < kD / 16; ++k) {
          const uint64_t off = (uint64_t)(((k >> 2) * kHalf + (k & 3) * 32) >> 4);
          tc::mma_ss(d, dq + off, b0 + off, idesc_s, k > 0);
        }
      }
    };
    auto issue_pv = [&](int i, bool acc) {
      const uint64_t b0 = dv + (uint64_t)((vslot(i) * kBlockBytes) >> 4);
      const uint32_t a = tmem + (uint32_t)(i & 1) * 128;
      if (leader) {
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)
          tc::mma_ts(tmem + kColO, a + k * 8, b0 + (uint64_t)((k * 16 * 128) >> 4), idesc_o, (acc || k > 0) ? 1u : 0u);
      }
    };
    Iter it;
    if (s_c < e_c) it_seek32(it, s_c, pre, B, Hkv);
    int seg = 0;
    bool ok = true;
    bool prev_first = false, prev_last = false;
    for (int t = s_c; t < e_c && ok; ++t) {
      const int i = t - s_c;
      const bool first = (t == s_c) || it.lt == 0;
      const bool last = (t == e_c - 1) || it.lt == it.nb - 1;
      if (first) {
        ok = wait(q_full, seg & 1);
        if (!ok) break;
        ++seg;
      }
      ok = wait(&kv_full[kslot(i)], kpar(i));
      if (!ok) break;
      tc::fence_after_sync();
      issue_s(i);
      commit(&s_full[i & 1]);
      commit(&kv_empty[kslot(i)]);
      if (last) commit(q_empty);
      if (i > 0) {
        // P V of the previous block (its scores were signalled one block ago)
        ok = wait(&p_full[(i - 1) & 1], (uint32_t)(((i - 1) >> 1) & 1));
        if (!ok) break;
        ok = wait(&kv_full[vslot(i - 1)], vpar(i - 1));
        if (!ok) break;
        tc::fence_after_sync();
        issue_pv(i - 1, !prev_first);
        commit(&kv_empty[vslot(i - 1)]);
        commit(o_done);
        if (prev_last) commit(o_full);
      }
      prev_first = first;
      prev_last = last;
      it_next(it, pre, B, Hkv);
    }
    if (ok && e_c > s_c) {
      const int i = e_c - s_c;  // P V of the share's last block
      ok = wait(&p_full[(i - 1) & 1], (uint32_t)(((i - 1) >> 1) & 1));
      if (ok) ok = wait(&kv_full[vslot(i - 1)], vpar(i - 1));
      if (ok) {
        tc::fence_after_sync();
        issue_pv(i - 1, !prev_first);
        commit(&kv_empty[vslot(i - 1)]);
        commit(o_done);
        commit(o_full);
      }
    }
    commit(mma_done);
    wait_drain(mma_done, 0, p.err);
  } else if (KV8 && warp < 4) {
    // ================================================================ E4M3 -> fp16 converters
    const int ct = tid - 64;  // 0 .. 63
    // Rows G..127 of the Q tile are padding MMA rows: zero once.
    for (int e = ct; e < (128 - G) * 16; e += kConv) {
      const int row = G + (e >> 4), c16 = e & 15;
      *reinterpret_cast<uint4*>(q_tile + (c16 >> 3) * kHalf + row * 128 + (((c16 & 7) ^ (row & 7)) << 4)) =
          make_uint4(0, 0, 0, 0);
    }
    Iter it;
    if (s_c < e_c) it_seek32(it, s_c, pre, B, Hkv);
    int seg = 0, len_b = 0;
    bool ok = true;
    for (int t = s_c; t < e_c && ok; ++t) {
      const int i = t - s_c;
      if (t == s_c || it.lt == 0) {
        // The pair's query heads as fp16 rows of the Q tile (128-byte swizzle,
        // two 64-column halves), once the previous piece's scores are done.
        // Eight 16-byte pieces of q per thread are loaded at once (all of
        // them for G <= 32, before the wait), so the global-load latency is
        // paid once per batch, not once per piece.
        const __nv_bfloat16* qb = p.q + ((size_t)it.b * p.Hq + (size_t)it.j * G) * kD;
        const int nq = G * 16;  // 16-byte pieces of the group's q
        uint4 x[8];
        auto load_q = [&](int e0) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int e = e0 + ct + u * kConv;
            x[u] = e < nq ? __ldg(reinterpret_cast<const uint4*>(qb + (size_t)(e >> 4) * kD + (e & 15) * 8))
                          : make_uint4(0, 0, 0, 0);
          }
        };
        auto store_q = [&](int e0) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int e = e0 + ct + u * kConv, row = e >> 4, c16 = e & 15;
            if (e < nq) {
              const uint4 h = make_uint4(
                  pack_f16x2(__uint_as_float(x[u].x << 16), __uint_as_float(x[u].x & 0xFFFF0000u)),
                  pack_f16x2(__uint_as_float(x[u].y << 16), __uint_as_float(x[u].y & 0xFFFF0000u)),
                  pack_f16x2(__uint_as_float(x[u].z << 16), __uint_as_float(x[u].z & 0xFFFF0000u)),
                  pack_f16x2(__uint_as_float(x[u].w << 16), __uint_as_float(x[u].w & 0xFFFF0000u)));
              *reinterpret_cast<uint4*>(q_tile + (c16 >> 3) * kHalf + row * 128 + (((c16 & 7) ^ (row & 7)) << 4)) = h;
            }
          }
        };
        load_q(0);
        const int seq_len = __ldg(p.seqlens + it.b);
        ok = mbar_wait_bounded(q_empty, (seg & 1) ^ 1, abort_flag, p.err, p.wait_ns);
        if (!ok) break;
        store_q(0);
        for (int e0 = 8 * kConv; e0 < nq; e0 += 8 * kConv) {
          load_q(e0);
          store_q(e0);
        }
        fence_proxy_async_smem();
        mbar_arrive(q_full);
        ++seg;
        len_b = clamp_seq(seq_len, p.Lmax);
      }
      const int valid = min(kBN, len_b - it.lt * kBN);
      for (int kv = 0; kv < 2 && ok; ++kv) {
        const int n = 2 * i + kv, s8 = n % S8, s = n % p.stages;
        ok = mbar_wait_bounded(&e8_full[s8], (uint32_t)((n / S8) & 1), abort_flag, p.err, p.wait_ns);
        if (ok && n >= p.stages)
          ok = mbar_wait_bounded(&kv_empty[s], (uint32_t)(((n / p.stages) & 1) ^ 1), abort_flag, p.err, p.wait_ns);
        if (!ok) break;
        // 16 E4M3 bytes (d = 16c .. 16c + 15 of row r) become two 16-byte
        // fp16 chunks of the row's half c / 4.  V rows at and past the
        // sequence end become zeros (the cache may hold NaN bytes there).
        // Thread ct takes chunk c = ct % 8 of rows ct / 8 + 8u (u < 16), all
        // in the same swizzle phase; the 16 loads go out before any
        // conversion, and the row test selects after it (no branch).
        const uint8_t* src = ring8 + s8 * kBlockBytes8;
        uint8_t* dst = ring + s * kBlockBytes;
        const int zero_from = kv ? valid : kBN;
        constexpr int kIt = kBN * 8 / kConv;
        const int c = ct & 7, r0 = ct >> 3, sw = r0 & 7;
        uint4 wv[kIt];
#pragma unroll
        for (int u = 0; u < kIt; ++u)
          wv[u] = *reinterpret_cast<const uint4*>(src + (r0 + 8 * u) * 128 + ((c ^ sw) << 4));
        const int cc = 2 * (c & 3);
        uint8_t* base = dst + (c >> 2) * kHalf + r0 * 128;
#pragma unroll
        for (int u = 0; u < kIt; ++u) {
          uint4 lo, hi;
          e4m3x4_to_f16x2x2(wv[u].x, lo.x, lo.y);
          e4m3x4_to_f16x2x2(wv[u].y, lo.z, lo.w);
          e4m3x4_to_f16x2x2(wv[u].z, hi.x, hi.y);
          e4m3x4_to_f16x2x2(wv[u].w, hi.z, hi.w);
          if (r0 + 8 * u >= zero_from) lo = hi = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(base + u * 1024 + ((cc ^ sw) << 4)) = lo;
          *reinterpret_cast<uint4*>(base + u * 1024 + (((cc + 1) ^ sw) << 4)) = hi;
        }
        fence_proxy_async_smem();
        mbar_arrive(&e8_empty[s8]);
        mbar_arrive(&kv_full[s]);
      }
      it_next(it, pre, B, Hkv);
    }
  } else if (!KV8 && warp < 4) {
    // ================================================================ piece publisher / merger
    // bf16 cache: warps 2-3 take the cross-CTA step of every cut piece off
    // the softmax group's path.  The group writes the piece's partial,
    // arrives on pub_full[slot] (release at CTA scope) and goes on with the
    // next piece; here the arrival is awaited (acquire), the pair's counter
    // is bumped with an acquire-release atomic at GPU scope (which carries
    // the group's partial stores with it), and the last piece's CTA merges.
    // Each slot holds at most one piece per launch (slot 0: the share's
    // first piece when it starts inside a pair; slot 1: a piece that starts
    // a pair and is cut), so each barrier completes once, at parity 0.
    const int ct = tid - 64;  // 0 .. 63
    Iter it;
    if (s_c < e_c) it_seek32(it, s_c, pre, B, Hkv);
    int seg_lt0 = 0;
    for (int t = s_c; t < e_c; ++t) {
      if (t == s_c || it.lt == 0) seg_lt0 = it.lt;
      const bool last = (t == e_c - 1) || it.lt == it.nb - 1;
      // cut pieces before the share's last one (that one the softmax group
      // publishes itself)
      if (last && t != e_c - 1 && !(seg_lt0 == 0 && it.lt == it.nb - 1)) {
        mbar_wait_bounded(&pub_full[seg_lt0 == 0 ? 1 : 0], 0, abort_flag, p.err, p.wait_ns);
        __nv_bfloat16* outp = p.out + ((size_t)it.b * p.Hq + (size_t)it.j * G) * kD;
        publish_merge(it, outp, ct, 64, 2, 1);
      }
      it_next(it, pre, B, Hkv);
    }
  } else if (warp >= 4) {
    // ================================================================ softmax + epilogue
    const int r = tid - 128;                 // query head within the group = TMEM lane
    const int wq = warp - 4;                 // lane quarter
    const bool rows = wq * 32 < G;           // this warp holds at least one real head
    const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
    const uint32_t o_tm = tmem + lane_addr + kColO;
    Iter it;
    if (s_c < e_c) it_seek32(it, s_c, pre, B, Hkv);
    int seg = 0, seg_lt0 = 0, len_b = 0;
    float m_use = -INFINITY, l = 0.f;
    float slp = p.scale_log2, v_mul = 1.f;  // logit scale, output factor (FP8 cache: times its scales)
    // After a timeout the group keeps walking the share with every wait
    // returning at once (the abort flag is up), so that all four warps always
    // meet the same named barriers; only the memory work is skipped.
    bool ok = true;
    for (int t = s_c; t < e_c; ++t) {
      const int i = t - s_c;
      const bool first = (t == s_c) || it.lt == 0;
      const bool last = (t == e_c - 1) || it.lt == it.nb - 1;
      if (first) {
        seg_lt0 = it.lt;
        len_b = clamp_seq(p.seqlens[it.b], p.Lmax);
        m_use = -INFINITY;
        l = 0.f;
        if (KV8) {
          slp = p.scale_log2 * __ldg(p.k_scale + it.b * Hkv + it.j);
          v_mul = __ldg(p.v_scale + it.b * Hkv + it.j);
        }
      }
      const int valid = min(kBN, len_b - it.lt * kBN);  // keys of this block that exist (>= 1)
      {
        const bool w = mbar_wait_bounded(&s_full[i & 1], (uint32_t)((i >> 1) & 1), abort_flag, p.err, p.wait_ns);
        ok = __all_sync(0xffffffffu, w) && ok;
      }
      tc::fence_after_sync();
      const uint32_t s_tm = tmem + lane_addr + (uint32_t)(i & 1) * 128;
      if (rows && ok) {
        uint32_t s[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::ld_32x32b_x32(s_tm + c * 32, s[c]);
        tc::wait_ld_regs(s[0]);
        tc::pin_regs(s[1]);
        tc::pin_regs(s[2]);
        tc::pin_regs(s[3]);
        if (valid < kBN) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c * 32 + e >= valid) s[c][e] = __float_as_uint(-INFINITY);
        }
        float mxv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float m = fmax3(__uint_as_float(s[0][e]), __uint_as_float(s[0][e + 8]), __uint_as_float(s[0][e + 16]));
          m = fmaxf(m, __uint_as_float(s[0][e + 24]));
#pragma unroll
          for (int c = 1; c < 4; ++c)
            m = fmax3(m, fmaxf(__uint_as_float(s[c][e]), __uint_as_float(s[c][e + 8])),
                      fmaxf(__uint_as_float(s[c][e + 16]), __uint_as_float(s[c][e + 24])));
          mxv[e] = m;
        }
        const float mx = fmaxf(fmax3(mxv[0], mxv[1], mxv[2]), fmax3(fmax3(mxv[3], mxv[4], mxv[5]), mxv[6], mxv[7]));
        const float mxs = mx * slp;
        const bool rebase = mxs > m_use + kRebase;
        const bool any_rebase = __any_sync(0xffffffffu, rebase);
        const float m_new = rebase ? mxs : m_use;
        const float alpha = rebase ? fast_exp2(m_use - m_new) : 1.f;
        m_use = m_new;
        const float ref = m_use == -INFINITY ? 0.f : m_use;
        const float sl = slp, nref = -ref;
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pw[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float x0, x1;
            fma2(x0, x1, __uint_as_float(s[c][2 * e]), __uint_as_float(s[c][2 * e + 1]), sl, sl, nref, nref);
            const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
            ls[e & 3] += p0 + p1;
            pw[e] = KV8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
          }
          tc::st_32x32b_x16(s_tm + c * 16, pw);
        }
        l = l * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
        if (any_rebase && !first) {
          // O holds blocks up to i - 1: wait for that P V, then re-base it.
          const bool w = mbar_wait_bounded(o_done, (uint32_t)((i - 1) & 1), abort_flag, p.err, p.wait_ns);
          if (__all_sync(0xffffffffu, w)) {
            tc::fence_after_sync();
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              uint32_t o[32];
              tc::ld_32x32b_x32(o_tm + c * 32, o);
              tc::wait_ld_regs(o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tc::st_32x32b_x32(o_tm + c * 32, o);
            }
          }
        }
        tc::wait_st();
      }
      if (!KV8 && valid < kBN) {
        // Cache rows at and past seqlens[b] may hold anything (NaN included):
        // zero them in the V block so that P = 0 there contributes exactly 0
        // (an FP8 cache's converters already wrote zeros there).
        uint8_t* vb = ring + vslot(i) * kBlockBytes;
        const bool w = mbar_wait_bounded(&kv_full[vslot(i)], vpar(i), abort_flag, p.err, p.wait_ns);
        ok = __all_sync(0xffffffffu, w) && ok;
        if (ok) {
          const int nchunks = (kBN - valid) * 16;  // 16-byte chunks over both halves
          for (int e = r; e < nchunks; e += 128) {
            const int row = valid + (e >> 4), rem = e & 15;
            *reinterpret_cast<uint4*>(vb + (rem >> 3) * kHalf + row * 128 + (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
      }
      tc::fence_before_sync();
      mbar_arrive(&p_full[i & 1]);

      if (last) {
        // ---- end of a piece: O / l to the output, or a partial for the merge
        {
          const bool w = mbar_wait_bounded(o_full, (uint32_t)(seg & 1), abort_flag, p.err, p.wait_ns);
          ok = __all_sync(0xffffffffu, w) && ok;
        }
        ++seg;
        tc::fence_after_sync();
        const bool complete = (seg_lt0 == 0) && (it.lt == it.nb - 1);
        const int slot = seg_lt0 == 0 ? 1 : 0;
        const size_t slot_idx = (size_t)blockIdx.x * 2 + slot;
        __nv_bfloat16* outp = p.out + ((size_t)it.b * p.Hq + (size_t)it.j * G) * kD;
        if (rows && ok) {
          // the partial and the output carry the V scale (1 for a bf16 cache)
          const float inv = l > 0.f ? v_mul / l : 0.f;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tc::ld_32x32b_x32(o_tm + c * 32, o);
            tc::wait_ld_regs(o);
            if (KV8 && !complete) {
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * v_mul);
            }
            if (r < G) {
              if (complete) {
                uint4* dst = reinterpret_cast<uint4*>(outp + (size_t)r * kD + c * 32);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                  uint32_t w[4];
#pragma unroll
                  for (int e = 0; e < 4; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(o[v * 8 + 2 * e]) * inv, __uint_as_float(o[v * 8 + 2 * e + 1]) * inv);
                  dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
                }
              } else {
                float4* dst = reinterpret_cast<float4*>(p.part_acc + (slot_idx * G + r) * kD + c * 32);
#pragma unroll
                for (int v = 0; v < 8; ++v)
                  dst[v] = make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]),
                                       __uint_as_float(o[4 * v + 2]), __uint_as_float(o[4 * v + 3]));
              }
            }
          }
          if (!complete && r < G) {
            p.part_ml[(slot_idx * 2 + 0) * G + r] = m_use;
            p.part_ml[(slot_idx * 2 + 1) * G + r] = l;
          }
        }
        tc::fence_before_sync();
        if (!complete) {
          if (KV8 || t == e_c - 1) {
            // the share's last piece (nothing left to overlap with): this
            // group of 128 threads counts it in and merges, one head per
            // four threads
            publish_merge(it, outp, r, 128, 1, 0);
          } else {
            // warps 2-3 count the piece in and merge; this group goes on
            mbar_arrive(&pub_full[slot]);
          }
        }
      }
      it_next(it, pre, B, Hkv);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool decode_tc_plan(int B, int Hq, int Hkv, int D, int Lmax, int sm_count, DecodePlan* plan, bool kv8) {
  if (B < 1 || B > kMaxBatch || Hkv < 1 || Hq % Hkv != 0 || Lmax < 1 || D != kD) return false;
  const int G = Hq / Hkv;
  if (G < 1 || G > 128) return false;
  plan->kind = 1;
  plan->kv8 = kv8;
  plan->D = D;
  plan->G = G;
  plan->Gpad = 128;
  plan->NT = 0;
  plan->HS = 0;
  plan->tile_keys = kBN;
  plan->threads = kThreads;
  const long long blocks_max = (long long)B * Hkv * ((Lmax + kBN - 1) / kBN);
  if (blocks_max >= (1LL << 31) / kMaxCtas) return false;  // the kernel's split arithmetic is 32-bit
  plan->num_ctas = (int)std::min<long long>(blocks_max, std::min(kMaxCtas, std::max(1, sm_count)));
  const TcLayout l0 = tc_layout(0, 0);
  int stages, stages8 = 0;
  if (kv8) {
    // three fp16 blocks for the MMAs (one K, V pair and the next K), the
    // rest of shared memory for E4M3 blocks in flight from HBM
    stages = 3;
    stages8 = std::min((kSmemLimit - l0.total - stages * kBlockBytes - 32 * 8) / kBlockBytes8, 8);
    if (stages8 < 2) return false;
  } else {
    stages = std::min((kSmemLimit - l0.total - 16 * 8) / kBlockBytes, 8);
    if (stages < 2) return false;
  }
  plan->stages = stages;
  plan->stages8 = stages8;
  plan->smem_bytes = (size_t)tc_layout(stages, stages8).total;
  plan->ws_part_floats = (size_t)plan->num_ctas * 2 * G * (D + 2);
  plan->chunk_tiles = 0;
  plan->chunks_max = plan->num_ctas;
  plan->ws_counters = (size_t)B * Hkv;
  return true;
}

cudaError_t decode_tc_launch(const DecodePlan& plan, const DecodeArgs& a, cudaStream_t stream) {
  CUtensorMap tq, tk, tv;
  const uint64_t pairs = (uint64_t)a.B * a.Hkv;
  const int G = plan.G;
  const bool paged = a.block_table != nullptr;
  if (paged && (a.page_size % kBN != 0 || a.page_size <= 0)) return cudaErrorInvalidValue;
  if (plan.kv8 && (!a.k_scale || !a.v_scale)) return cudaErrorInvalidValue;
  const uint64_t planes = paged ? (uint64_t)a.num_pages * a.Hkv : pairs;
  const uint64_t rows = paged ? (uint64_t)a.page_size : (uint64_t)a.Lmax;
  // Q viewed as [B * Hkv][G][D]: a 128-row box starting at row 0 reads the
  // group's G heads and zero-fills rows G..127.  An E4M3 cache is a byte
  // tensor: one 128-byte box (a whole row of D = 128) per K or V block.
  CUresult r1 =
      encode_tmap_bf16_3d(&tq, a.q, kD, (uint64_t)G, pairs, (uint64_t)kD * 2, (uint64_t)G * kD * 2, 64, 128, 1);
  CUresult r2, r3;
  if (plan.kv8) {
    r2 = encode_tmap_u8_3d(&tk, a.k_cache, kD, rows, planes, (uint64_t)kD, rows * kD, kD, kBN, 1);
    r3 = encode_tmap_u8_3d(&tv, a.v_cache, kD, rows, planes, (uint64_t)kD, rows * kD, kD, kBN, 1);
  } else {
    r2 = encode_tmap_bf16_3d(&tk, a.k_cache, kD, rows, planes, (uint64_t)kD * 2, rows * kD * 2, 64, kBN, 1);
    r3 = encode_tmap_bf16_3d(&tv, a.v_cache, kD, rows, planes, (uint64_t)kD * 2, rows * kD * 2, 64, kBN, 1);
  }
  if (r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS || r3 != CUDA_SUCCESS) return cudaErrorInvalidValue;
  TcParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.seqlens = a.seqlens;
  p.part_acc = a.ws_part;
  p.part_ml = a.ws_part + (size_t)plan.num_ctas * 2 * G * kD;
  p.counters = a.ws_counters;
  p.err = a.err;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = G;
  p.Lmax = a.Lmax;
  p.stages = plan.stages;
  p.num_ctas = plan.num_ctas;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.block_table = a.block_table;
  p.page_size = a.page_size;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.wait_ns = pipeline_wait_limit_ns();
  p.starve = pipeline_starved() ? 1 : 0;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.stages8 = plan.stages8;
  auto kern = plan.kv8 ? decode_tc_kernel<true> : decode_tc_kernel<false>;
  static std::atomic<unsigned long long> attr_set[2] = {{0}, {0}};
  std::atomic<unsigned long long>& done = attr_set[plan.kv8 ? 1 : 0];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(done.load() >> dev & 1ull)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return e;
    if (dev < 64) done.fetch_or(1ull << dev);
  }
  kern<<<plan.num_ctas, kThreads, plan.smem_bytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace gqa
