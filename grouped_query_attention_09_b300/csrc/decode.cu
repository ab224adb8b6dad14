// decode.cu -- split-KV GQA decode on sm_103a.
//
// One decode step: for every sequence b and query head h, one query vector
// attends to the first seqlens[b] rows of KV head j = h / G of a bf16
// [B, Hkv, Lmax, D] cache (G = Hq / Hkv query heads per KV head; the grouping
// of the GQA paper notes, "分组查询注意力（GQA）", and of the Huawei Cloud post
// "多头注意力机制的代码实现（MQA和GQA）", section 5).  Decode is bound by reading
// the KV cache (the paper notes, "QA 相关": the saving of GQA is the smaller
// cache read from HBM), so the design goal is that every cache byte crosses
// HBM exactly once and is reused from shared memory by all G query heads of
// its group -- K/V are never expanded to Hq heads.
//
// Work split ("Split-KV": the gsyq.cn page on xformers, "分块计算与内存优化",
// cuts K/V into blocks computed apart and reduced afterwards):
//   * the (b, j, key tile) space is flattened pair-major (pair = b*Hkv + j)
//     and cut into num_ctas contiguous, equal shares; each persistent CTA
//     streams its share, crossing pair boundaries;
//   * a pair wholly inside one CTA is normalised and written directly; a pair
//     cut by a share boundary leaves one partial (running max m, sum l,
//     unnormalised acc) per piece in a workspace, and the CTA that finishes
//     the last piece of that pair (an arrival counter) merges the pieces by
//     log-sum-exp and writes the output -- no second kernel.
//
// CTA layout: warps 0..NC-1 consume, warps NC.. produce.
//   producers: one lane of a warp streams K and V tiles [tile_keys x D] of
//     the cache into a ring of shared-memory stages with 3-D TMA loads
//     (128-byte swizzle, evict-first L2 policy), an mbarrier pair per stage;
//     for an 8-bit cache or whole contiguous pairs each tile group has its own
//     producer warp and ring part, otherwise one producer fills both; with one
//     CTA per (b, kv head) pair the first producer prefetches the pair's
//     opening tiles into L2 while the prologue reads seqlens;
//   consumers: NG tile groups (two for G <= 8) of a 4 x HS grid of warps take
//     alternate tiles, each group from a private part of the ring and walking
//     only its own tiles; warp (ks, hs) owns keys [16 ks, 16 ks + 16) of its
//     group's tiles and query heads [8 NT hs, 8 NT (hs+1)) of the group.
//     Scores are computed transposed, S^T = K q^T, with mma.sync m16n8k16
//     (keys in M, heads in N, D in K); the online softmax runs on the
//     accumulator fragments, with a per-head reference max that moves only
//     when a score passes it by more than 2^8 (then the column max by warp
//     shuffles and the rescale); P^T is turned into the B operand of
//     O^T = V^T P^T with movmatrix; V^T comes from the swizzled V tile through
//     ldmatrix.trans (an FP8 cache: both come from E4M3 bytes converted in
//     registers).  The key-slice states of a head are merged in shared memory
//     at the end of each piece.
//   Decode intensity is G flop per cache byte (<= 64), far below the tensor
//   ridge point, so the warp-level MMA is not the bound; HBM is.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kBN = 64;            // keys per tile
constexpr int kKW = kBN / 16;      // key-slice warps
constexpr int kMaxBatch = 1024;    // batches whose tile prefix fits in shared memory
constexpr int kMaxStages = 8;
constexpr int kSmemLimit = 232448; // opt-in dynamic shared memory per CTA on sm_100-class parts
constexpr int kMaxCtas = 160;      // persistent CTAs at most (one per SM; B300 has 148)
constexpr float kRebase = 8.f;     // log2 units a score may exceed a head's reference max by

struct Params {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  const int32_t* seqlens;
  float* part_acc;  // [P][2][G][D]
  float* part_ml;   // [P][2][2][G]  (m then l; m in log2 units)
  int* counters;    // [B*Hkv]
  unsigned* err;
  int B, Hq, Hkv, G, Lmax;
  int HS, NC, stages, num_ctas;
  float scale_log2;
  const float* k_scale;  // FP8 cache: per (b, kv head) scales of K and V
  const float* v_scale;
  const int32_t* block_table;  // paged cache (else null): [B][max_pages] page of each logical page
  int page_size, max_pages, num_pages;
  int prefetch_tiles;  // > 0: one CTA per (b, kv head) pair; prefetch its first tiles into L2 at launch
  int NP;              // producer warps: 1, or NG (one per tile group)
  unsigned long long wait_ns;  // pipeline-wait limit
  int starve;                  // test hook: the producer issues no loads
};

struct SmemLayout {
  int stage_bytes, k_bytes;
  int epi_off, red_off, q_off, pre_off, bar_off, flag_off, total;
};

__host__ __device__ inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

// NG: groups of consumer warps that take alternate tiles (each group keeps
// its own running state, merged at the end of a piece like the key slices).
// kv8: the ring holds FP8 E4M3 tiles (one byte per element); the consumers
// convert them in registers.
template <int D>
__host__ __device__ inline SmemLayout smem_layout(int stages, int Gpad, int NG, bool kv8, int G) {
  SmemLayout s;
  const int slices = kKW * NG;
  s.k_bytes = kv8 ? kBN * D : (D / 64) * kBN * 128;
  s.stage_bytes = 2 * s.k_bytes;
  s.epi_off = stages * s.stage_bytes;
  // epi holds the key-slice accumulators, later the merge statistics (2 x pieces x G)
  // epi: one row of D + 4 floats per (key slice, real head) -- sized by G, not
  // the padded head count, which leaves room for one more ring stage at G = 4
  s.red_off = s.epi_off + (slices * (D + 4) > 2 * kMaxCtas ? slices * (D + 4) : 2 * kMaxCtas) * G * 4;
  s.q_off = s.red_off + 2 * slices * Gpad * 4;  // [Gpad][D + 8] bf16 (NT = 2 only)
  s.pre_off = round_up(s.q_off + Gpad * (D + 8) * 2, 16);
  s.bar_off = round_up(s.pre_off + (kMaxBatch + 1) * 4, 8);
  s.flag_off = s.bar_off + 2 * stages * 8;
  s.total = s.flag_off + 4 * (4 + 32) + 1024;  // flags + scan scratch, + slack to align the base

  return s;
}

// Position in the flattened (b, j, tile) space.
struct TileIter {
  int b, j, lt, nb;
};

__device__ inline void iter_seek(TileIter& it, long long t, const int* pre, int B, int Hkv) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if ((long long)Hkv * pre[mid] <= t) lo = mid; else hi = mid - 1;
  }
  it.b = lo;
  it.nb = pre[lo + 1] - pre[lo];
  long long r = t - (long long)Hkv * pre[lo];
  it.j = (int)(r / it.nb);
  it.lt = (int)(r % it.nb);
}

__device__ inline void iter_next(TileIter& it, const int* pre, int B, int Hkv) {
  if (++it.lt < it.nb) return;
  it.lt = 0;
  if (++it.j < Hkv) return;
  it.j = 0;
  do { ++it.b; } while (it.b < B && pre[it.b + 1] == pre[it.b]);
  it.nb = it.b < B ? pre[it.b + 1] - pre[it.b] : 0;
}

// CTA whose share [floor(c T / P), floor((c+1) T / P)) holds tile t.
__device__ inline int cta_of(long long t, long long T, int P) {
  return (int)(((t + 1) * P + T - 1) / T) - 1;
}

__device__ inline int clamp_len(int len, int Lmax) { return len < 0 ? 0 : (len > Lmax ? Lmax : len); }

// E4M3 tiles (rows of D bytes, as TMA lands them): the 16-byte chunk c of row
// r sits at chunk c ^ (r & 7) with D = 128 (128-byte swizzle) and at
// c ^ ((r >> 1) & 3) with D = 64 (64-byte swizzle; a 128-byte line holds two
// rows).  Rows r and r + 8 share the pattern in both.
template <int D>
__device__ __forceinline__ int e4m3_chunk(int c, int r) {
  return D == 128 ? (c ^ (r & 7)) : (c ^ ((r >> 1) & 3));
}

// V bytes a lane takes from one row of an E4M3 tile: 16 bytes (d = 16 g ..
// 16 g + 15) at D = 128, 8 bytes (d = 8 g .. 8 g + 7) at D = 64 -- the output
// rows of the lane's m-rows g and g + 8 (see the PV product).
template <int D>
struct V8Frag {
  uint32_t w[D / 32];
};
template <int D>
__device__ __forceinline__ V8Frag<D> load_v8(const uint8_t* tile, int row, int g) {
  V8Frag<D> f;
  if constexpr (D == 128) {
    const uint4 x = *reinterpret_cast<const uint4*>(tile + row * 128 + (e4m3_chunk<128>(g, row) << 4));
    f.w[0] = x.x;
    f.w[1] = x.y;
    f.w[2] = x.z;
    f.w[3] = x.w;
  } else {
    const uint2 x = *reinterpret_cast<const uint2*>(tile + row * 64 + (e4m3_chunk<64>(g >> 1, row) << 4) + 8 * (g & 1));
    f.w[0] = x.x;
    f.w[1] = x.y;
  }
  return f;
}

// Consumer warp groups per CTA: with one n-tile per warp (G <= 8) a single
// group leaves one consumer warp per SM sub-partition, whose per-tile
// dependency chain then sets the pace; two groups on alternate tiles overlap
// two chains.
template <int NT>
__host__ __device__ constexpr int tile_groups() { return NT == 1 ? 2 : 1; }

template <int D, int NT, bool KV8>
__global__ void __launch_bounds__(320, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const Params p) {
  constexpr int KT = D / 16;  // 16-wide k-steps over D (QK) and m-tiles over D (PV)
  constexpr int NG = tile_groups<NT>();
  constexpr int KS = kKW * NG;  // key-slice states merged at the end of a piece
  static_assert(!KV8 || NT == 1, "the FP8 cache path is built for G <= 8");
  const int Gpad = p.HS * 8 * NT;
  const SmemLayout L = smem_layout<D>(p.stages, Gpad, NG, KV8, p.G);
  // Each tile group has a private ring of SG stages: tile i belongs to group
  // i % NG and takes stage (i % NG) * SG + (i / NG) % SG.  A group therefore
  // waits on use u of a stage only after it consumed use u - 1 itself, so a
  // parity wait can never be satisfied by the phase before the one it wants
  // (which could happen if two groups alternated on one stage and a load
  // completed out of order).
  const int SG = p.stages / NG;
  auto stage_of = [&](long long i) { return (int)((i % NG) * SG + (i / NG) % SG); };
  auto parity_of = [&](long long i) { return (uint32_t)(((i / NG) / SG) & 1); };

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* epi = reinterpret_cast<float*>(smem + L.epi_off);          // [KS][G][D+4]
  float* red_m = reinterpret_cast<float*>(smem + L.red_off);        // [KW][Gpad]
  float* red_l = red_m + KS * Gpad;                                  // [KS][Gpad]
  int* pre = reinterpret_cast<int*>(smem + L.pre_off);               // [B+1]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty = full + p.stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.flag_off);
  volatile int* last_flag = abort_flag + 1;
  volatile int* chi_flag = abort_flag + 2;
  int* warp_tot = reinterpret_cast<int*>(smem + L.flag_off) + 4;  // [32]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NC = p.NC, nthr = blockDim.x;
  const int B = p.B, Hkv = p.Hkv, G = p.G;

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NC / NG);
    }
    *abort_flag = 0;
    *last_flag = 0;
    fence_mbar_init();
  }
  if (warp == NC && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    // One CTA per pair (the host's choice for nearly SM-filling pair counts):
    // when the lengths are equal this CTA's share is exactly pair blockIdx.x,
    // so its first tiles are pulled into L2 while the prologue below reads
    // seqlens (with unequal lengths the prefetch is merely wasted).  The rows
    // stay inside the tensor map: at most Lmax.  A paged cache maps each
    // tile through the block table first (row t kBN of pair (b, j) sits in
    // page block_table[b][t kBN / page_size]); an entry outside the page pool
    // is skipped here (the producer flags it when it loads the tile).
    const int pb = (int)blockIdx.x / Hkv, pj = (int)blockIdx.x - pb * Hkv;
    int pg_lp = -1, pg = -1;
    for (int t = 0; t < p.prefetch_tiles; ++t) {
      int y = t * kBN, z = (int)blockIdx.x;
      if (p.block_table) {
        const int lp = y / p.page_size;
        if (lp != pg_lp) {
          pg_lp = lp;
          pg = __ldg(p.block_table + (size_t)pb * p.max_pages + lp);
        }
        if (pg < 0 || pg >= p.num_pages) continue;
        z = pg * Hkv + pj;
        y -= lp * p.page_size;
      }
      if constexpr (KV8) {
        tma_prefetch_l2_3d(&tmK, 0, y, z);
        tma_prefetch_l2_3d(&tmV, 0, y, z);
      } else {
#pragma unroll
        for (int box = 0; box < D / 64; ++box) {
          tma_prefetch_l2_3d(&tmK, box * 64, y, z);
          tma_prefetch_l2_3d(&tmV, box * 64, y, z);
        }
      }
    }
  }

  // ---- tile count per batch and its exclusive prefix pre[0..B] (block scan)
  {
    const int per = (B + nthr - 1) / nthr;
    const int lo = tid * per, hi = min(B, lo + per);
    int local = 0;
    unsigned flags = 0;
    for (int i = lo; i < hi; ++i) {
      int len = p.seqlens[i];
      if (len > p.Lmax) flags |= GQA_DEV_SEQLEN_CLAMPED;
      if (len <= 0) flags |= GQA_DEV_EMPTY_CONTEXT;
      local += (clamp_len(len, p.Lmax) + kBN - 1) / kBN;
    }
    if (flags && blockIdx.x == 0) atomicOr(p.err, flags);
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int nw = nthr >> 5;
      int w = lane < nw ? warp_tot[lane] : 0;
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += v;
      }
      if (lane < nw) warp_tot[lane] = wi - w;  // exclusive warp offsets
    }
    __syncthreads();
    int run = warp_tot[warp] + incl - local;
    for (int i = lo; i < hi; ++i) {
      pre[i] = run;
      run += (clamp_len(p.seqlens[i], p.Lmax) + kBN - 1) / kBN;
    }
    if (lo < B && hi == B) pre[B] = run;
  }
  __syncthreads();

  // Shares: the first P = min(CTAs, tiles) CTAs each take a non-empty,
  // contiguous share [s_c, e_c) of the T tiles; the others only zero-fill.
  const long long T = (long long)Hkv * pre[B];
  const int P = (int)(T < p.num_ctas ? T : p.num_ctas);
  const bool active = (int)blockIdx.x < P;
  const long long s_c = active ? T * blockIdx.x / P : 0;
  const long long e_c = active ? T * (blockIdx.x + 1) / P : 0;

  if (warp >= NC) {
    // ============================== producers =============================
    // With p.NP == NG producer warps, warp NC + g fills the ring of tile
    // group g: it walks every tile (so that the ring counters and the page
    // position stay exact) and issues the loads of tiles i with i % NG == g.
    // With one producer (p.NP == 1) warp NC issues every tile.  Two pay with
    // 8-bit tiles, which one lane cannot issue fast enough for both groups,
    // and with whole contiguous pairs; with cut pairs or bf16 pages the
    // extra warp costs more than it brings (measured).
    const int pgrp = warp - NC;
    if (lane == 0 && s_c < e_c && !p.starve) {
      const uint64_t pol = l2_policy_evict_first();
      TileIter it;
      iter_seek(it, s_c, pre, B, Hkv);
      long long issued = 0;
      int pg_b = -1, pg_lp = -1, pg = 0;  // last block-table entry read (paged cache)
      // the previous tile's page and row offset in it: along a pair they
      // advance by one tile without a division (with 8-bit tiles this loop
      // runs close to the consumers' pace, so a division by page_size on
      // every tile shows in the step time)
      int pv_b = -1, pv_j = -1, pv_lt = -2, pv_lp = 0, pv_off = 0;
      // tile i: group ig = i % NG, use us = (i / NG) % SG of that group's
      // ring, lap = i / (NG SG) (kept incrementally: no divisions per tile)
      int ig = 0, us = 0, lap = 0;
      for (long long t = s_c; t < e_c; ++t) {
        const int i = (int)(t - s_c);
        const int s = ig * SG + us;
        const bool mine = p.NP == 1 || ig == pgrp;
        if (mine && lap > 0) {
          if (!mbar_wait_bounded(&empty[s], (uint32_t)((lap - 1) & 1), abort_flag, p.err, p.wait_ns)) break;
        }
        if (++ig == NG) {
          ig = 0;
          if (++us == SG) {
            us = 0;
            ++lap;
          }
        }
        uint8_t* kdst = smem + s * L.stage_bytes;
        uint8_t* vdst = kdst + L.k_bytes;
        int z = it.b * Hkv + it.j, y = it.lt * kBN;
        if (p.block_table) {
          // Paged cache: logical page y / page_size of sequence b; the entry
          // is reloaded only when the page changes.  A page index out of range
          // is flagged and sent outside the tensor map, where TMA reads zeros.
          int lp, off;
          if (it.b == pv_b && it.j == pv_j && it.lt == pv_lt + 1) {
            lp = pv_lp;
            off = pv_off + kBN;
            if (off == p.page_size) {  // page_size is a multiple of kBN
              off = 0;
              ++lp;
            }
          } else {
            lp = y / p.page_size;
            off = y - lp * p.page_size;
          }
          pv_b = it.b;
          pv_j = it.j;
          pv_lt = it.lt;
          pv_lp = lp;
          pv_off = off;
          if (mine && (it.b != pg_b || lp != pg_lp)) {
            pg_b = it.b;
            pg_lp = lp;
            pg = __ldg(p.block_table + (size_t)it.b * p.max_pages + lp);
            if (pg < 0 || pg >= p.num_pages) {
              atomicOr(p.err, GQA_DEV_BAD_PAGE);
              pg = -1;
            }
          }
          z = pg < 0 ? -1 : pg * Hkv + it.j;
          y = off;
        }
        if (!mine) {
          iter_next(it, pre, B, Hkv);
          continue;
        }
        mbar_arrive_expect_tx(&full[s], L.stage_bytes);
        if constexpr (KV8) {
          // one 128-byte-wide box per tensor: a row of D = 128 E4M3 bytes
          tma_load_3d(kdst, &tmK, 0, y, z, &full[s], pol);
          tma_load_3d(vdst, &tmV, 0, y, z, &full[s], pol);
        } else {
#pragma unroll
          for (int box = 0; box < D / 64; ++box) {
            tma_load_3d(kdst + box * kBN * 128, &tmK, box * 64, y, z, &full[s], pol);
            tma_load_3d(vdst + box * kBN * 128, &tmV, box * 64, y, z, &full[s], pol);
          }
        }
        issued = i + 1;
        iter_next(it, pre, B, Hkv);
      }
      // Wait (bounded) until every copy this thread issued has landed.
      // The last NG * SG tiles hold the latest use of every stage; this
      // producer waits for those of its own group.
      const long long first = issued > NG * SG ? issued - NG * SG : 0;
      for (long long i = first; i < issued; ++i) {
        if (p.NP != 1 && (int)(i % NG) != pgrp) continue;
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(&full[stage_of(i)], parity_of(i))) {
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(p.err, GQA_DEV_WAIT_TIMEOUT);
            break;
          }
        }
      }
    }
  } else {
    // ============================== consumers =============================
    const int grp = warp / (kKW * p.HS);  // tile group: tiles i with i % NG == grp
    const int wig = warp % (kKW * p.HS);
    const int ks = wig % kKW;             // key slice
    const int hs = wig / kKW;             // head slice
    const int slice = grp * kKW + ks;     // index of this warp's state in the merge
    const int key0 = ks * 16;
    const int cthreads = NC * 32;

    // Zero output rows of sequences with an empty context (this CTA's share).
    for (int b = blockIdx.x; b < B; b += p.num_ctas) {
      if (pre[b + 1] != pre[b]) continue;
      __nv_bfloat16* o = p.out + (size_t)b * p.Hq * D;
      for (int e = tid; e < p.Hq * D; e += cthreads) o[e] = __float2bfloat16_rn(0.f);
    }

    // Per-lane constants of the ldmatrix addressing (128-byte swizzle: the
    // 16-byte chunk c of row r sits at chunk c ^ (r & 7)).
    const int sw = lane & 7;
    const int k_row = key0 + (lane & 7) + ((lane >> 3) & 1) * 8;  // K: M0..M3 = (k0-7,c),(k8-15,c),(k0-7,c+1),(k8-15,c+1)
    const int k_chunk_add = lane >> 4;
    const int v_row = key0 + (lane & 7) + (lane >> 4) * 8;        // V^T: (k0-7,c),(k0-7,c+1),(k8-15,c),(k8-15,c+1)
    const int v_chunk_add = (lane >> 3) & 1;

    float acc[KT][NT][4];
    float m_run[NT][2], l_run[NT][2];
    // NT = 1 keeps the group's q fragments in registers; NT = 2 (G = 16, 32)
    // reads them from a padded copy in shared memory with ldmatrix, which
    // keeps the per-thread state of the wider head slice out of local memory.
    constexpr int kQReg = NT == 1 ? KT : 1;
    uint32_t qf[kQReg][NT][2];
    __nv_bfloat16* q_s = reinterpret_cast<__nv_bfloat16*>(smem + L.q_off);
    constexpr int kQRow = D + 8;  // padded row (elements): rows 16 B apart in the bank map
    int seg_lt0 = 0, len_b = 0;
    // logit scale in log2 units of accumulator columns 2 (lane % 4) and + 1
    // (an FP8 cache: times the K scale and the inverse of each head's q scale)
    float sl_col0 = p.scale_log2, sl_col1 = p.scale_log2;
    float v_mul = 1.f;  // V scale of an FP8 cache
    bool live = true;

    // The share is walked piece by piece (a piece: the share's tiles of one
    // (b, j) pair).  Tile i of the share (i = t - s_c) belongs to tile group
    // i % NG; a group visits only its own tiles, so its u-th tile takes
    // stage grp SG + u % SG with parity (u / SG) & 1, counted as it goes.
    TileIter it;
    if (s_c < e_c) iter_seek(it, s_c, pre, B, Hkv);
    int us = 0;       // u % SG
    uint32_t ph = 0;  // (u / SG) & 1
    long long t = s_c;
    while (t < e_c) {
      const int n_piece = (int)min((long long)(it.nb - it.lt), e_c - t);
      const int pair = it.b * Hkv + it.j;

      {
        // ---- piece start: this pair's q, scales and a fresh running state
        seg_lt0 = it.lt;
        len_b = clamp_len(p.seqlens[it.b], p.Lmax);
        if constexpr (KV8) v_mul = __ldg(p.v_scale + pair);
        const __nv_bfloat16* qb = p.q + ((size_t)it.b * p.Hq + (size_t)it.j * G) * D;
        if constexpr (NT == 1 && !KV8) {
#pragma unroll
          for (int kk = 0; kk < KT; ++kk) {
            const int hg = (lane >> 2);
            if (hg < G) {
              const uint32_t* qp = reinterpret_cast<const uint32_t*>(qb + (size_t)hg * D + kk * 16 + 2 * (lane & 3));
              qf[kk][0][0] = __ldg(qp);
              qf[kk][0][1] = __ldg(qp + 4);
            } else {
              qf[kk][0][0] = 0u;
              qf[kk][0][1] = 0u;
            }
          }
        } else if constexpr (KV8) {
          // fp16 q in the permuted contraction order of the FP8 K fragments
          // (see the QK product): k-step kk, k = 2c, 2c+1 | 2c+8, 2c+9 read
          // d = 64 (kk / 4) + 16c + 4 (kk % 4) + 0, 1 | 2, 3
          const int hg = lane >> 2;
#pragma unroll
          for (int kk = 0; kk < KT; ++kk) {
            uint2 qv = make_uint2(0u, 0u);
            if (hg < G)
              qv = __ldg(reinterpret_cast<const uint2*>(qb + (size_t)hg * D + 64 * (kk >> 2) + 16 * (lane & 3) +
                                                        4 * (kk & 3)));
            qf[kk][0][0] = pack_f16x2(__uint_as_float(qv.x << 16), __uint_as_float(qv.x & 0xFFFF0000u));
            qf[kk][0][1] = pack_f16x2(__uint_as_float(qv.y << 16), __uint_as_float(qv.y & 0xFFFF0000u));
          }
          sl_col0 = sl_col1 = p.scale_log2 * __ldg(p.k_scale + pair);
        } else {
          // The previous piece's last named barrier has passed: q_s is free.
          for (int e = tid; e < G * (D / 8); e += cthreads) {
            const int h = e / (D / 8), c = e % (D / 8);
            *reinterpret_cast<uint4*>(q_s + h * kQRow + c * 8) =
                __ldg(reinterpret_cast<const uint4*>(qb + (size_t)h * D + c * 8));
          }
          named_bar_sync(1, cthreads);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            m_run[nt][e] = -INFINITY;
            l_run[nt][e] = 0.f;
          }
#pragma unroll
          for (int kk = 0; kk < KT; ++kk)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[kk][nt][e] = 0.f;
        }
      }

      const int first = (int)((((long long)grp - (t - s_c)) % NG + NG) % NG);
      for (int k = first; k < n_piece; k += NG) {
      const int lt = seg_lt0 + k;  // tile of the pair
      const int s = grp * SG + us;
      const uint32_t par = ph;
      if (++us == SG) {
        us = 0;
        ph ^= 1u;
      }
      if (live) live = mbar_wait_bounded(&full[s], par, abort_flag, p.err, p.wait_ns);
      if (live) {
        uint32_t kbase = smem_u32(smem + s * L.stage_bytes);
        uint32_t vbase = kbase + L.k_bytes;
        const int valid = min(kBN, len_b - lt * kBN);  // >= 1

        // FP8 cache: this warp's E4M3 K bytes go to registers at the start of
        // the tile, its V bytes before the PV product, and the stage is
        // released once both are held (no converted copy in shared memory).
        //   K rows g, g + 8 (g = key0 + lane / 4), 16-byte chunks c and 4 + c
        //     (c = lane % 4): in k-step kk the fragment's k = 2c, 2c+1 | 2c+8,
        //     2c+9 read bytes 4 (kk % 4) .. +3 of chunk 4 (kk / 4) + c -- a
        //     permutation of the contraction index that q's fragments share;
        //   V rows key0 + 2c, +1, +8, +9, chunk lane / 4 (d = 16 (lane / 4) ..
        //     + 15): the A fragment of V^T in m-tile mt pairs the bytes of two
        //     rows at columns 2 mt, 2 mt + 1 -- a permutation of the output
        //     rows d undone when the accumulators are stored.
        //   V rows at or past seqlens[b] read as zeros (the cache may hold
        //   anything there, NaN included).
        uint4 k8[D / 64][2];
        V8Frag<D> v8[4];
        if constexpr (KV8) {
          const uint8_t* kt = smem + s * L.stage_bytes;
          const int g = key0 + (lane >> 2);
#pragma unroll
          for (int hd = 0; hd < D / 64; ++hd) {
            const int ch = e4m3_chunk<D>(4 * hd + (lane & 3), g) << 4;  // rows g and g + 8 share the swizzle
            k8[hd][0] = *reinterpret_cast<const uint4*>(kt + g * D + ch);
            k8[hd][1] = *reinterpret_cast<const uint4*>(kt + (g + 8) * D + ch);
          }
        } else if (valid < key0 + 16) {
          // Rows past the sequence end hold whatever the cache holds there
          // (possibly NaN); zero this warp's V rows so P = 0 stays 0.
          const int r0 = max(valid, key0);
          const int nrows = key0 + 16 - r0;
          uint8_t* vtile = smem + s * L.stage_bytes + L.k_bytes;
          for (int e = lane; e < nrows * (D / 64) * 8; e += 32) {
            const int row = r0 + e / ((D / 64) * 8);
            const int rem = e % ((D / 64) * 8);
            const int box = rem / 8, chunk = rem % 8;
            *reinterpret_cast<uint4*>(vtile + box * kBN * 128 + row * 128 + chunk * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }

        // ---- S^T = K q^T over this warp's 16 keys
        float sc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[nt][e] = 0.f;
        float sc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};  // two MMA chains (even, odd k-steps)
        if constexpr (KV8) {
          // k-step kk: rows g and g + 8 of word kk % 4 of chunk 4 (kk / 4) + c;
          // bytes 0, 1 are the fragment's k = 2c, 2c+1 and bytes 2, 3 its
          // k = 2c+8, 2c+9 (the order q's fragments were loaded in)
#pragma unroll
          for (int kk = 0; kk < KT; ++kk) {
            const uint4& kg = k8[kk >> 2][0];
            const uint4& kh = k8[kk >> 2][1];
            const uint32_t w0 = (kk & 3) == 0 ? kg.x : (kk & 3) == 1 ? kg.y : (kk & 3) == 2 ? kg.z : kg.w;
            const uint32_t w1 = (kk & 3) == 0 ? kh.x : (kk & 3) == 1 ? kh.y : (kk & 3) == 2 ? kh.z : kh.w;
            uint32_t a[4];
            e4m3x4_to_f16x2x2(w0, a[0], a[2]);
            e4m3x4_to_f16x2x2(w1, a[1], a[3]);
            mma_f16_16816(sc2[kk & 1], a, qf[kk][0][0], qf[kk][0][1]);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[0][e] = sc2[0][e] + sc2[1][e];
        } else {
#pragma unroll
          for (int kk = 0; kk < KT; ++kk) {
            uint32_t a[4];
            const int chunk = (kk & 3) * 2 + k_chunk_add;
            ldmatrix_x4(a, kbase + (kk >> 2) * kBN * 128 + k_row * 128 + ((chunk ^ sw) << 4));
            if constexpr (NT == 1) {
              mma_bf16_16816(sc2[kk & 1], a, qf[kk][0][0], qf[kk][0][1]);
              if (kk == KT - 1)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[0][e] = sc2[0][e] + sc2[1][e];
            } else {
              // B fragments of both n-tiles for this k-step: matrices
              // (nt, d-lo), (nt, d-hi) for nt = 0, 1; lane l addresses head
              // row l % 8 of matrix l / 8.
              uint32_t b[4];
              const int m = lane >> 3;
              const int hrow = (hs * NT + (m >> 1)) * 8 + (lane & 7);
              ldmatrix_x4(b, smem_u32(q_s + hrow * kQRow + kk * 16 + (m & 1) * 8));
              mma_bf16_16816(sc[0], a, b[0], b[1]);
              mma_bf16_16816(sc[1], a, b[2], b[3]);
            }
          }
        }

        // ---- online softmax (log2 domain); rows = keys, columns = heads.
        // The reference point m_run of a head moves only when a score
        // exceeds it by more than kRebase (or on the first tile), so most
        // tiles skip the rescale of the accumulators; p stays <= 2^kRebase,
        // and the merges below take m_run as the base of (l, acc) whatever
        // its distance from the true maximum.
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float x[4];
          x[0] = sc[nt][0] * sl_col0;
          x[1] = sc[nt][1] * sl_col1;
          x[2] = sc[nt][2] * sl_col0;
          x[3] = sc[nt][3] * sl_col1;
          if (valid < key0 + 16) {  // rows past the sequence end (warp-uniform test)
            if (key0 + (lane >> 2) >= valid) x[0] = x[1] = -INFINITY;
            if (key0 + (lane >> 2) + 8 >= valid) x[2] = x[3] = -INFINITY;
          }
          // each lane tests its own scores; only a tile that moves some
          // head's reference point pays for the column max (shuffles over
          // the 8 lanes that share a column) and the rescale
          float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
          if (__any_sync(0xffffffffu, mx0 > m_run[nt][0] + kRebase || mx1 > m_run[nt][1] + kRebase)) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
              mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
              mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mn0 = fmaxf(m_run[nt][0], mx0), mn1 = fmaxf(m_run[nt][1], mx1);
            const float al0 = fast_exp2(m_run[nt][0] - (mn0 == -INFINITY ? 0.f : mn0));
            const float al1 = fast_exp2(m_run[nt][1] - (mn1 == -INFINITY ? 0.f : mn1));
            m_run[nt][0] = mn0;
            m_run[nt][1] = mn1;
            l_run[nt][0] *= al0;
            l_run[nt][1] *= al1;
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
              acc[kk][nt][0] *= al0;
              acc[kk][nt][1] *= al1;
              acc[kk][nt][2] *= al0;
              acc[kk][nt][3] *= al1;
            }
          }
          const float mu0 = m_run[nt][0] == -INFINITY ? 0.f : m_run[nt][0];
          const float mu1 = m_run[nt][1] == -INFINITY ? 0.f : m_run[nt][1];
          const float p0 = fast_exp2(x[0] - mu0), p1 = fast_exp2(x[1] - mu1);
          const float p2 = fast_exp2(x[2] - mu0), p3 = fast_exp2(x[3] - mu1);
          l_run[nt][0] += p0 + p2;
          l_run[nt][1] += p1 + p3;
          if constexpr (KV8) {
            pb[nt][0] = movmatrix_trans(pack_f16x2(p0, p1));
            pb[nt][1] = movmatrix_trans(pack_f16x2(p2, p3));
          } else {
            pb[nt][0] = movmatrix_trans(pack_bf16x2(p0, p1));
            pb[nt][1] = movmatrix_trans(pack_bf16x2(p2, p3));
          }
        }

        if constexpr (KV8) {
          const uint8_t* vt = smem + s * L.stage_bytes + L.k_bytes;
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int row = key0 + 2 * (lane & 3) + (r & 1) + 8 * (r >> 1);
            v8[r] = row < valid ? load_v8<D>(vt, row, lane >> 2) : V8Frag<D>{};
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
        }
        // ---- O^T += V^T P^T
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
          uint32_t a[4];
          if constexpr (KV8) {
            // bytes (row 2c, row 2c+1) and (row 2c+8, row 2c+9) at columns
            // 2 mt (m-row g) and 2 mt + 1 (m-row g + 8)
            const int w = mt >> 1;
            const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
            const uint32_t r0 = v8[0].w[w], r1 = v8[1].w[w], r8 = v8[2].w[w], r9 = v8[3].w[w];
            e4m3x4_to_f16x2x2(__byte_perm(r0, r1, sel), a[0], a[1]);
            e4m3x4_to_f16x2x2(__byte_perm(r8, r9, sel), a[2], a[3]);
          } else {
            const int chunk = (mt & 3) * 2 + v_chunk_add;
            ldmatrix_x4_trans(a, vbase + (mt >> 2) * kBN * 128 + v_row * 128 + ((chunk ^ sw) << 4));
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if constexpr (KV8)
              mma_f16_16816(acc[mt][nt], a, pb[nt][0], pb[nt][1]);
            else
              mma_bf16_16816(acc[mt][nt], a, pb[nt][0], pb[nt][1]);
          }
        }
        __syncwarp();
        if (!KV8 && lane == 0) mbar_arrive(&empty[s]);
      }
      }

      {
        // ---- piece end: merge the key-slice states, then output or partial
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float l = l_run[nt][e];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            const int hg = (hs * NT + nt) * 8 + 2 * (lane & 3) + e;
            if ((lane >> 2) == 0) {
              red_m[slice * Gpad + hg] = m_run[nt][e];
              red_l[slice * Gpad + hg] = l;
            }
          }
#pragma unroll
          for (int mt = 0; mt < KT; ++mt) {
            const int hg = (hs * NT + nt) * 8 + 2 * (lane & 3);
            float* e0 = epi + (size_t)(slice * G + hg) * (D + 4);  // rows of padding heads are not kept
            float* e1 = e0 + (D + 4);
            if constexpr (KV8) {
              // m-rows g, g + 8 of m-tile mt are d = (D / 8) g + 2 mt and + 1;
              // the FP8 cache's V scale is applied here, once per piece
              const int d = (D / 8) * (lane >> 2) + 2 * mt;
              if (hg < G)
                *reinterpret_cast<float2*>(e0 + d) = make_float2(acc[mt][nt][0] * v_mul, acc[mt][nt][2] * v_mul);
              if (hg + 1 < G)
                *reinterpret_cast<float2*>(e1 + d) = make_float2(acc[mt][nt][1] * v_mul, acc[mt][nt][3] * v_mul);
            } else {
              const int d = mt * 16 + (lane >> 2);
              if (hg < G) {
                e0[d] = acc[mt][nt][0];
                e0[d + 8] = acc[mt][nt][2];
              }
              if (hg + 1 < G) {
                e1[d] = acc[mt][nt][1];
                e1[d + 8] = acc[mt][nt][3];
              }
            }
          }
        }
        // The running state now lives in shared memory; resetting it here
        // (the next piece starts from it anyway) frees its registers for the
        // merge below.
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            m_run[nt][e] = -INFINITY;
            l_run[nt][e] = 0.f;
          }
#pragma unroll
          for (int kk = 0; kk < KT; ++kk)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[kk][nt][e] = 0.f;
        }
        named_bar_sync(1, cthreads);

        const bool complete = (seg_lt0 == 0) && (seg_lt0 + n_piece == it.nb);
        const int slot = seg_lt0 == 0 ? 1 : 0;
        const size_t slot_idx = (size_t)blockIdx.x * 2 + slot;
        __nv_bfloat16* outp = p.out + ((size_t)it.b * p.Hq + (size_t)it.j * G) * D;

        // Per head: the piece's max M, the key slices' weights 2^(m_k - M)
        // (stored over red_m) and the piece's sum L (stored in red_l[0]).
        for (int h = tid; h < G; h += cthreads) {
          float M = -INFINITY;
#pragma unroll
          for (int k = 0; k < KS; ++k) M = fmaxf(M, red_m[k * Gpad + h]);
          const float Mu = M == -INFINITY ? 0.f : M;
          float Ls = 0.f;
#pragma unroll
          for (int k = 0; k < KS; ++k) {
            const float f = fast_exp2(red_m[k * Gpad + h] - Mu);
            Ls += f * red_l[k * Gpad + h];
            red_m[k * Gpad + h] = f;
          }
          red_l[h] = Ls;
          red_l[Gpad + h] = M;
        }
        named_bar_sync(1, cthreads);
        for (int e = tid; e < G * (D / 4); e += cthreads) {
          const int h = e / (D / 4), d = 4 * (e % (D / 4));
          float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int k = 0; k < KS; ++k) {
            const float f = red_m[k * Gpad + h];
            const float4 x = *reinterpret_cast<const float4*>(epi + (size_t)(k * G + h) * (D + 4) + d);
            acc4.x += f * x.x;
            acc4.y += f * x.y;
            acc4.z += f * x.z;
            acc4.w += f * x.w;
          }
          if (complete) {
            const float inv = 1.f / red_l[h];
            uint2 pk;
            pk.x = pack_bf16x2(acc4.x * inv, acc4.y * inv);
            pk.y = pack_bf16x2(acc4.z * inv, acc4.w * inv);
            *reinterpret_cast<uint2*>(outp + (size_t)h * D + d) = pk;
          } else {
            *reinterpret_cast<float4*>(p.part_acc + (slot_idx * G + h) * D + d) = acc4;
            if (d == 0) {
              p.part_ml[(slot_idx * 2 + 0) * G + h] = red_l[Gpad + h];
              p.part_ml[(slot_idx * 2 + 1) * G + h] = red_l[h];
            }
          }
        }

        if (!complete) {
          // Publish this piece: the barrier orders every thread's partial
          // stores before thread 0's acquire-release arrival.
          named_bar_sync(1, cthreads);
          if (tid == 0) {
            const long long o_p = (long long)Hkv * pre[it.b] + (long long)it.j * it.nb;
            const int c_lo = cta_of(o_p, T, P);
            const int c_hi = cta_of(o_p + it.nb - 1, T, P);
            const int old = atomic_add_acq_rel_gpu(&p.counters[pair], 1);
            const bool last = old == c_hi - c_lo;
            if (last) p.counters[pair] = 0;  // ready for the next call (ordered by the kernel boundary)
            *last_flag = last ? (c_lo + 1) : 0;  // encodes c_lo
            *chi_flag = c_hi;
          }
          named_bar_sync(1, cthreads);
          const int lf = *last_flag;
          if (lf) {
            // This CTA finished the pair's last piece: merge all pieces.
            // Piece s of the pair sits in CTA c_lo + s, slot 1 for s = 0
            // (the piece that starts the pair) and slot 0 after it.
            const int c_lo = lf - 1, nseg = *chi_flag - c_lo + 1;
            float* wm = epi;              // [nseg][G] piece max, then merge weight
            float* wl = epi + nseg * G;   // [nseg][G] piece sum
            for (int e = tid; e < nseg * G; e += cthreads) {
              const int s2 = e / G, h = e % G;
              const size_t si = (size_t)(c_lo + s2) * 2 + (s2 == 0 ? 1 : 0);
              wm[e] = __ldcg(p.part_ml + (si * 2 + 0) * G + h);
              wl[e] = __ldcg(p.part_ml + (si * 2 + 1) * G + h);
            }
            named_bar_sync(1, cthreads);
            for (int h = tid; h < G; h += cthreads) {
              float M = -INFINITY;
              for (int s2 = 0; s2 < nseg; ++s2) M = fmaxf(M, wm[s2 * G + h]);
              const float Mu = M == -INFINITY ? 0.f : M;
              float Ls = 0.f;
              for (int s2 = 0; s2 < nseg; ++s2) {
                const float f = fast_exp2(wm[s2 * G + h] - Mu);
                Ls += f * wl[s2 * G + h];
                wm[s2 * G + h] = f;
              }
              const float inv = 1.f / Ls;
              for (int s2 = 0; s2 < nseg; ++s2) wm[s2 * G + h] *= inv;
            }
            named_bar_sync(1, cthreads);
            // Every thread owns up to 4 float4 chunks of the [G][D] output and
            // loads its chunks of all pieces without waiting in between.
            constexpr int kChunksMax = 4;
            const int nchunk = G * (D / 4);
            float4 a4[kChunksMax];
#pragma unroll
            for (int u = 0; u < kChunksMax; ++u) a4[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
            for (int s2 = 0; s2 < nseg; ++s2) {
              const size_t si = (size_t)(c_lo + s2) * 2 + (s2 == 0 ? 1 : 0);
              const float* base = p.part_acc + si * G * D;
#pragma unroll
              for (int u = 0; u < kChunksMax; ++u) {
                const int e = tid + u * cthreads;
                if (e < nchunk) {
                  const int h = e / (D / 4), d = 4 * (e % (D / 4));
                  const float f = wm[s2 * G + h];
                  const float4 x = __ldcg(reinterpret_cast<const float4*>(base + (size_t)h * D + d));
                  a4[u].x += f * x.x;
                  a4[u].y += f * x.y;
                  a4[u].z += f * x.z;
                  a4[u].w += f * x.w;
                }
              }
            }
#pragma unroll
            for (int u = 0; u < kChunksMax; ++u) {
              const int e = tid + u * cthreads;
              if (e < nchunk) {
                const int h = e / (D / 4), d = 4 * (e % (D / 4));
                uint2 pk;
                pk.x = pack_bf16x2(a4[u].x, a4[u].y);
                pk.y = pack_bf16x2(a4[u].z, a4[u].w);
                *reinterpret_cast<uint2*>(outp + (size_t)h * D + d) = pk;
              }
            }
          }
        }
        named_bar_sync(1, cthreads);
      }
      t += n_piece;
      it.lt = seg_lt0 + n_piece - 1;  // the piece's last tile: step to the next pair
      iter_next(it, pre, B, Hkv);
    }
  }
  __syncthreads();
}

// Tensor maps of recently used caches.  A map encodes only the base address,
// shape and strides, so an entry with the same key is always valid (even if
// the memory was freed and reallocated in between).  Serving loops call
// decode with the same cache every step; this skips two driver encodes.
struct TmapEntry {
  const void* k;
  const void* v;
  int D, Lmax, kv8;
  uint64_t pairs;
  CUtensorMap tk, tv;
};
constexpr int kTmapCacheSize = 8;
std::mutex g_tmap_mu;
TmapEntry g_tmap_cache[kTmapCacheSize];
int g_tmap_n = 0, g_tmap_next = 0;

cudaError_t cache_tensor_maps(const DecodeArgs& a, int D, bool kv8, CUtensorMap* tk, CUtensorMap* tv) {
  // Contiguous cache: planes (b, j) of Lmax rows; paged: planes (page, j) of page_size rows.
  const bool paged = a.block_table != nullptr;
  const uint64_t pairs = paged ? (uint64_t)a.num_pages * a.Hkv : (uint64_t)a.B * a.Hkv;
  const int rows = paged ? a.page_size : a.Lmax;
  std::lock_guard<std::mutex> lk(g_tmap_mu);
  for (int e = 0; e < g_tmap_n; ++e) {
    const TmapEntry& c = g_tmap_cache[e];
    if (c.k == a.k_cache && c.v == a.v_cache && c.D == D && c.Lmax == rows && c.pairs == pairs &&
        c.kv8 == (int)kv8) {
      *tk = c.tk;
      *tv = c.tv;
      return cudaSuccess;
    }
  }
  TmapEntry n;
  n.k = a.k_cache;
  n.v = a.v_cache;
  n.D = D;
  n.Lmax = rows;
  n.kv8 = (int)kv8;
  n.pairs = pairs;
  if (kv8) {
    // E4M3 bytes: one box of D bytes covers a row (128- or 64-byte swizzle)
    const uint64_t s1 = (uint64_t)D, s2 = (uint64_t)rows * D;
    if (encode_tmap_u8_3d(&n.tk, a.k_cache, D, rows, pairs, s1, s2, D, kBN, 1) != CUDA_SUCCESS ||
        encode_tmap_u8_3d(&n.tv, a.v_cache, D, rows, pairs, s1, s2, D, kBN, 1) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  } else {
    const uint64_t s1 = (uint64_t)D * 2, s2 = (uint64_t)rows * D * 2;
    if (encode_tmap_bf16_3d(&n.tk, a.k_cache, D, rows, pairs, s1, s2, 64, kBN, 1) != CUDA_SUCCESS ||
        encode_tmap_bf16_3d(&n.tv, a.v_cache, D, rows, pairs, s1, s2, 64, kBN, 1) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  g_tmap_cache[g_tmap_next] = n;
  g_tmap_next = (g_tmap_next + 1) % kTmapCacheSize;
  if (g_tmap_n < kTmapCacheSize) ++g_tmap_n;
  *tk = n.tk;
  *tv = n.tv;
  return cudaSuccess;
}

template <int D, int NT, bool KV8>
cudaError_t launch_t(const DecodePlan& plan, const DecodeArgs& a, cudaStream_t stream) {
  CUtensorMap tmK, tmV;
  cudaError_t e = cache_tensor_maps(a, D, KV8, &tmK, &tmV);
  if (e != cudaSuccess) return e;
  Params p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.seqlens = a.seqlens;
  p.part_acc = a.ws_part;
  p.part_ml = a.ws_part + (size_t)plan.num_ctas * 2 * plan.G * D;
  p.counters = a.ws_counters;
  p.err = a.err;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = plan.G;
  p.Lmax = a.Lmax;
  p.HS = plan.HS;
  p.NC = kKW * plan.HS * tile_groups<NT>();
  p.stages = plan.stages;
  p.num_ctas = plan.num_ctas;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.block_table = a.block_table;
  p.page_size = a.page_size;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.wait_ns = pipeline_wait_limit_ns();
  p.starve = pipeline_starved() ? 1 : 0;
  p.prefetch_tiles = 0;
  if (plan.num_ctas == a.B * a.Hkv) p.prefetch_tiles = std::min(plan.stages, (a.Lmax + kBN - 1) / kBN);
  // One producer warp per tile group for an 8-bit cache and for whole
  // contiguous pairs, else one (the measured better choice in each case).
  p.NP = (KV8 || (!a.block_table && plan.num_ctas == a.B * a.Hkv)) ? tile_groups<NT>() : 1;
  if (a.block_table && (a.page_size % kBN != 0 || a.page_size <= 0)) return cudaErrorInvalidValue;
  auto kern = decode_kernel<D, NT, KV8>;
  // The opt-in shared-memory size is a per-device function attribute: set it
  // once per device to the largest size any plan can ask for.
  static std::atomic<unsigned long long> attr_set{0};  // bit d: set on device d (< 64)
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev >= 64 || !(attr_set.load() >> dev & 1ull)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set.fetch_or(1ull << dev);
  }
  kern<<<plan.num_ctas, 32 * (p.NC + p.NP), plan.smem_bytes, stream>>>(tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace

bool decode_plan(int B, int Hq, int Hkv, int D, int Lmax, int sm_count, DecodePlan* plan, size_t max_part_floats,
                 bool kv8) {
  if (B < 1 || B > kMaxBatch || Hkv < 1 || Hq % Hkv != 0 || Lmax < 1) return false;
  if (D != 64 && D != 128) return false;
  const int G = Hq / Hkv;
  // An FP8 cache: D = 128 (every G <= 128) or D = 64 (G <= 8).
  if (kv8 && D == 64 && G > 8) return false;
  // Wide groups at D = 128 go to the tcgen05 kernel: its tensor core reads
  // each K/V block from shared memory once for all G heads.
  if (D == 128 && G > 8 && G <= 128) {
    if (!decode_tc_plan(B, Hq, Hkv, D, Lmax, sm_count, plan, kv8)) return false;
    if (max_part_floats > 0 && plan->ws_part_floats > max_part_floats) return false;
    return true;
  }
  plan->kind = 0;
  plan->kv8 = kv8;
  int Gpad, NT, HS;
  if (G <= 8) {
    Gpad = 8; NT = 1; HS = 1;
  } else if (G == 16 || G == 32) {
    Gpad = G; NT = 2; HS = G / 16;
  } else {
    return false;
  }
  plan->D = D;
  plan->G = G;
  plan->Gpad = Gpad;
  plan->NT = NT;
  plan->HS = HS;
  plan->tile_keys = kBN;
  const int NG = NT == 1 ? tile_groups<1>() : tile_groups<2>();
  plan->threads = 32 * (kKW * HS * NG + NG);  // at most: NG groups of 4 x HS consumer warps, a producer warp each
  const long long tiles_max = (long long)B * Hkv * ((Lmax + kBN - 1) / kBN);
  plan->num_ctas = (int)std::min<long long>(tiles_max, std::min(kMaxCtas, std::max(1, sm_count)));
  {
    // One CTA per (b, kv head) pair when the pairs nearly fill the GPU: with
    // equal lengths every share is then exactly one pair, so no pair is cut
    // and no cross-CTA merge runs (each SM's ring still keeps its share of
    // HBM bandwidth in flight).  Ragged lengths are still balanced by the
    // tile split, at the cost of some cuts.  Short caches (at most 8 tiles
    // per pair) also take one CTA per pair: a cut would save less time than
    // the merge it adds (a partial write, an arrival atomic and a chain of
    // L2 reads).
    const long long pairs = (long long)B * Hkv;
    const long long tiles_per_pair = (Lmax + kBN - 1) / kBN;
    if (pairs <= plan->num_ctas && (pairs * 4 >= (long long)plan->num_ctas * 3 || tiles_per_pair <= 8))
      plan->num_ctas = (int)pairs;
  }
  SmemLayout l0 = D == 64 ? smem_layout<64>(0, Gpad, NG, kv8, G) : smem_layout<128>(0, Gpad, NG, kv8, G);
  int stages = std::min(kMaxStages, (kSmemLimit - l0.total - 2 * kMaxStages * 8) / l0.stage_bytes);
  stages = stages / NG * NG;  // every tile group gets a private ring of stages / NG
  if (stages / NG < 2) return false;
  plan->stages = stages;
  plan->smem_bytes = (size_t)(D == 64 ? smem_layout<64>(stages, Gpad, NG, kv8, G) : smem_layout<128>(stages, Gpad, NG, kv8, G)).total;
  plan->ws_part_floats = (size_t)plan->num_ctas * 2 * G * (D + 2);
  if (max_part_floats > 0 && plan->ws_part_floats > max_part_floats) return false;
  plan->chunk_tiles = 0;  // static split: one contiguous share per CTA
  plan->chunks_max = plan->num_ctas;
  plan->ws_counters = (size_t)B * Hkv;
  return true;
}

cudaError_t decode_launch(const DecodePlan& plan, const DecodeArgs& a, cudaStream_t stream) {
  if (plan.kind == 1) return decode_tc_launch(plan, a, stream);
  if (plan.kv8) {
    if (plan.NT != 1 || !a.k_scale || !a.v_scale) return cudaErrorInvalidValue;
    return plan.D == 128 ? launch_t<128, 1, true>(plan, a, stream) : launch_t<64, 1, true>(plan, a, stream);
  }
  if (plan.D == 128) {
    // groups wider than 8 at D = 128 run on the tcgen05 kernel (decode_plan)
    if (plan.NT != 1) return cudaErrorInvalidValue;
    return launch_t<128, 1, false>(plan, a, stream);
  }
  return plan.NT == 1 ? launch_t<64, 1, false>(plan, a, stream) : launch_t<64, 2, false>(plan, a, stream);
}

}  // namespace gqa
