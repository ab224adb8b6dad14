// internal.h -- host-side declarations shared by the translation units of libgqa.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <cuda_bf16.h>

namespace gqa {

// Limit of the kernels' pipeline waits for launches made now (nanoseconds):
// kWaitLimitNs unless gqa_test_set_wait_limit_ns chose another; in that case
// pipeline_starved() is true and the kernels' producers issue no loads, so
// that the waits for them run out.
unsigned long long pipeline_wait_limit_ns();
bool pipeline_starved();

// Test hook of gqa_test_fail_workspace_allocs: true if this workspace
// allocation is to fail (consumes one of the requested failures).
bool take_injected_alloc_failure();

// Reads and clears the status word of gqa_decode_noalloc's fixed scratch on
// the current device (0 if that entry point was never set up there).
// Synchronous; allocates nothing.
cudaError_t noalloc_take_status(unsigned* flags);

// Encodes a 3-D bf16 tiled tensor map (dims innermost first, strides in bytes
// for dims 1 and 2) with 128-byte swizzle and zero fill outside the tensor.
CUresult encode_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t dim0, uint64_t dim1,
                             uint64_t dim2, uint64_t stride1, uint64_t stride2, uint32_t box0,
                             uint32_t box1, uint32_t box2);
// The same for a byte tensor (FP8 cache stored as uint8); a 64-byte inner box
// takes the 64-byte swizzle instead.
CUresult encode_tmap_u8_3d(CUtensorMap* map, const void* base, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                           uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1, uint32_t box2);

// ------------------------------------------------------------------ decode
struct DecodePlan {
  int kind;                // 0: warp-level MMA kernel (decode.cu), 1: tcgen05 kernel (decode_tc.cu)
  bool kv8;                // FP8 E4M3 cache (D = 128)
  int D, G, Gpad, NT, HS;  // head dim, group size, padded group, n-tiles/warp, head slices
  int tile_keys;           // keys per pipeline tile
  int chunk_tiles;         // tiles per scheduling chunk (unit of work a CTA claims)
  int chunks_max;          // chunks of a full cache (sizes the partial-result slots)
  int num_ctas;            // persistent CTAs
  int threads;             // threads per CTA
  int stages;              // pipeline depth
  int stages8 = 0;         // tcgen05 kernel with an FP8 cache: depth of the E4M3 ring
  size_t smem_bytes;       // dynamic shared memory per CTA
  size_t ws_part_floats;   // partial-result floats (acc + m + l)
  size_t ws_counters;      // per-(b, kv head) arrival counters
};

// Chooses tile and chunk size, persistent grid and pipeline depth; returns
// false if the shape is not supported by the decode kernels.  A non-zero
// max_part_floats bounds the partial-result workspace: the chunks grow
// coarser until it fits.
bool decode_plan(int B, int Hq, int Hkv, int D, int Lmax, int sm_count, DecodePlan* plan,
                 size_t max_part_floats = 0, bool kv8 = false);

struct DecodeArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* seqlens;
  void* out;
  int B, Hq, Hkv, D, Lmax;
  float scale;
  float* ws_part;     // >= plan.ws_part_floats floats
  int* ws_counters;   // >= plan.ws_counters ints, zero on entry, zero on exit
  unsigned* err;      // device status word
  const float* k_scale = nullptr;  // FP8 cache: [B * Hkv] scales of K and V
  const float* v_scale = nullptr;
  // Paged cache (block_table != nullptr): k_cache / v_cache are pools of
  // pages [num_pages, Hkv, page_size, D]; row t of sequence b is row
  // t % page_size of page block_table[b * max_pages + t / page_size]; Lmax is
  // then max_pages * page_size.
  const int32_t* block_table = nullptr;
  int page_size = 0, num_pages = 0, max_pages = 0;
};

cudaError_t decode_launch(const DecodePlan& plan, const DecodeArgs& a, cudaStream_t stream);

// The tcgen05 decode for wide groups (D = 128, 1 <= G <= 128, bf16 or FP8
// E4M3 cache); decode_plan routes G > 8 to it.  Same workspace layout as the
// warp-level kernel.
bool decode_tc_plan(int B, int Hq, int Hkv, int D, int Lmax, int sm_count, DecodePlan* plan, bool kv8 = false);
cudaError_t decode_tc_launch(const DecodePlan& plan, const DecodeArgs& a, cudaStream_t stream);

// ------------------------------------------------------------------ prefill
// ------------------------------------------------------------------ rope + append
struct RopeArgs {
  const __nv_bfloat16* q;      // [B, Hq, D]
  const __nv_bfloat16* k_new;  // [B, Hkv, D]
  const __nv_bfloat16* v_new;  // [B, Hkv, D]
  __nv_bfloat16* q_out;        // [B, Hq, D] (may be q)
  __nv_bfloat16* k_cache;      // [B, Hkv, Lmax, D]
  __nv_bfloat16* v_cache;
  int32_t* seqlens;            // [B], advanced by one per appended row
  int B, Hq, Hkv, D, Lmax;
  double base;
  unsigned* err;
  double inv_freq[128];  // base^(-2i/D), i < D/2: filled on the host by rope_append_launch
};

bool rope_supported(int D);
cudaError_t rope_append_launch(const RopeArgs& a, cudaStream_t stream);

// MHA -> GQA conversion of a K/V projection: H blocks of n bf16 values ->
// Hkv blocks (mode 0: mean of each group's G = H / Hkv blocks; 1: its first).
cudaError_t meanpool_heads_launch(const void* w, void* out, int H, int Hkv, long long n, int mode, int sm_count,
                                  cudaStream_t stream);

struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  int B, L, Hq, Hkv, D, causal;  // L: query rows (Lq)
  unsigned* err;
  int Lk = 0;  // key rows; 0 means L (plain prefill).  Lk > L: a chunk after Lk - L cached tokens
};

bool prefill_supported(int D);
cudaError_t prefill_launch(const PrefillArgs& a, int sm_count, cudaStream_t stream);

}  // namespace gqa
