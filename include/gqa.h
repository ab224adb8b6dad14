/*
 * gqa.h -- C ABI of libgqa.so, a single-GPU grouped-query attention (GQA)
 * engine for NVIDIA B300 (sm_103a).
 *
 * Grouped-query attention: Hq query heads are split into Hkv groups; every
 * group shares one K head and one V head, and query head h reads KV head
 * h / (Hq / Hkv) (the GQA paper notes on 51969.com, section "分组查询注意力
 * （GQA）"; the grouping `head_index // n_head_per_group` of the Huawei Cloud
 * post "多头注意力机制的代码实现（MQA和GQA）", section 5; the
 * `repeat_interleave` of "手把手教你用PyTorch实现GQA", section 1.3).
 * Hkv == Hq is multi-head attention and Hkv == 1 is multi-query attention.
 * Per head, out = softmax(scale * q K^T) V (Huawei Cloud post, section 5 code:
 * Q @ K^T, divide by sqrt(head_size), softmax, @ V).
 *
 * Conventions for every entry point
 *   - Tensors are dense, row-major, bf16 unless stated; pointers are DEVICE
 *     pointers of the current CUDA device unless the name says "host", and
 *     must be 16-byte aligned.  The caller allocates and owns every tensor and
 *     the stream; the library only borrows the pointers until the enqueued
 *     work has run.  K/V are never expanded to Hq heads in memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device entry points are asynchronous: they enqueue kernels on
 *     `stream` and return without synchronising.
 *   - Every function returns a gqa_status (0 = GQA_OK).  Argument errors are
 *     detected on the host before anything is enqueued; nothing traps.
 *   - Conditions seen on the device (a sequence length above the cache
 *     capacity, an empty context, a bounded wait that gave up) never trap:
 *     the kernel takes the documented fallback and sets a bit in a per-device
 *     status word that gqa_get_device_status() returns.
 *   - Thread safety: calls may come from several host threads; the library
 *     serialises access to its per-device workspace.  Two decode calls that
 *     share the workspace must not run concurrently on different streams; the
 *     library orders them on the stream of the later call.
 *   - CUDA graphs: the device entry points can be captured (stream capture)
 *     once a call with the same or larger sizes has run outside the capture,
 *     so that nothing has to be allocated; a call that would have to grow the
 *     workspace during capture returns GQA_ERR_CUDA and enqueues nothing.
 *     Captured calls are not ordered against other users of the workspace by
 *     the library: the caller orders a graph's replays against decode calls
 *     on other streams (replays on the capturing stream's successors, or on
 *     the stream the direct calls use, need nothing).  Every replay reads the
 *     inputs' current contents (new q, cache rows and seqlens values in the
 *     same buffers) and the in-launch merge counters return to zero at the
 *     end of each launch, so a graph replays any number of times.
 */
#ifndef GQA_H_
#define GQA_H_

#include <stdint.h>

#if defined(__GNUC__)
#define GQA_API __attribute__((visibility("default")))
#else
#define GQA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gqa_status {
  GQA_OK = 0,
  GQA_ERR_INVALID_ARG = 1, /* a size <= 0, Hq % Hkv != 0, causal not 0/1, bad scale */
  GQA_ERR_UNSUPPORTED = 2, /* a shape the kernels do not implement (see each call) */
  GQA_ERR_NULL = 3,        /* a required pointer is NULL */
  GQA_ERR_MISALIGNED = 4,  /* a tensor pointer is not 16-byte aligned */
  GQA_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed; see gqa_status_string */
  GQA_ERR_NO_DEVICE = 6,   /* no usable sm_103 device, or the kernels are not loadable */
  GQA_ERR_TOO_LARGE = 7    /* gqa_decode_noalloc: sizes need more than its fixed scratch */
} gqa_status;

/* Bits of the per-device status word (gqa_get_device_status). */
#define GQA_DEV_SEQLEN_CLAMPED 0x1u /* some seqlens[b] > Lmax; Lmax keys were used */
#define GQA_DEV_EMPTY_CONTEXT 0x2u  /* some seqlens[b] <= 0; that row of out is zero */
#define GQA_DEV_WAIT_TIMEOUT 0x4u   /* a pipeline wait gave up; results are invalid */
#define GQA_DEV_CACHE_FULL 0x8u     /* gqa_rope_append: some seqlens[b] >= Lmax; no row appended */
#define GQA_DEV_BAD_PAGE 0x10u      /* gqa_decode_paged: a needed block-table entry is out of range; its rows read as 0 */

/*
 * gqa_decode -- one decode step: every sequence b has one new query token per
 * query head, attending to the first seqlens[b] cached keys of its group.
 *
 *   q        [B, Hq, D]          bf16, device
 *   k_cache  [B, Hkv, Lmax, D]   bf16, device; row t of (b, j) at element
 *   v_cache  [B, Hkv, Lmax, D]     offset ((b*Hkv + j)*Lmax + t)*D
 *   seqlens  [B]                 int32, device; keys visible to sequence b
 *                                (the new token's own K/V already appended).
 *                                Read only on the device: no host sync.
 *   out      [B, Hq, D]          bf16, device, written (RNE from fp32)
 *   scale    logit scale, finite and > 0 (usually 1/sqrt(D))
 *
 * There is no mask inside [0, seqlens[b]); cache rows at or beyond seqlens[b]
 * are never read into the result (they may hold anything, NaN included).
 * seqlens[b] > Lmax is clamped to Lmax; seqlens[b] <= 0 gives a zero output
 * row; both set a device status bit.
 *
 * Supported: D = 128 with 1 <= G <= 128 (G = Hq/Hkv); D = 64 with G in
 * {1..8, 16, 32}; 1 <= B <= 1024.  Otherwise GQA_ERR_UNSUPPORTED.  G <= 8
 * (and D = 64) runs a warp-level MMA kernel; wider groups at D = 128 run a
 * tcgen05 kernel with the group's heads as the rows of each MMA.
 *
 * Work is split across a persistent grid: the (b, j, key-tile) space is cut
 * into equal contiguous shares, one per CTA (split-KV, the gsyq.cn page on
 * xformers, "分块计算与内存优化"), and the pieces of a (b, j) that landed in
 * different CTAs are merged by log-sum-exp in the same launch.  The partial
 * results live in a library-owned device workspace that is allocated on the
 * first call on a device (and grown when a later call needs more), kept until
 * gqa_release(); this first call allocates and so must not be made during
 * stream capture.
 */
GQA_API int gqa_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* seqlens,
               void* out, int B, int Hq, int Hkv, int D, int Lmax, float scale, void* stream);

/*
 * gqa_decode_fp8 -- gqa_decode over a KV cache stored in 8 bits: OCP FP8 E4M3
 * bytes (sign, 4 exponent bits with bias 7, 3 mantissa bits; largest 448)
 * with one fp32 scale per (sequence, KV head) for K and one for V, so the
 * real entry is e4m3(byte) * scale ("InputsFp8", FP8 KV storage, on the
 * gsyq.cn page on xformers, "混合精度计算加速"; the scale granularity is this
 * library's choice).  It halves the bytes the bandwidth-bound decode reads.
 *
 *   k_cache, v_cache  [B, Hkv, Lmax, D]  uint8 (E4M3 bytes), device
 *   k_scale, v_scale  [B, Hkv]            fp32, device (4-byte aligned)
 *   everything else as gqa_decode.
 *
 * Arithmetic: the E4M3 values are converted exactly to fp16 (in registers);
 * q is rounded to fp16 (so |q| must stay below 65504), scores and softmax are
 * fp32, P is rounded to fp16, accumulation is fp32; the K scale multiplies
 * the logit scale and the V scale the output.  Cache rows at or beyond
 * seqlens[b] are never used (they may hold anything, NaN bytes included).
 *
 * Supported: D == 128 with 1 <= G = Hq/Hkv <= 128, or D == 64 with G <= 8;
 * 1 <= B <= 1024.  Otherwise GQA_ERR_UNSUPPORTED.  G <= 8 runs the
 * warp-level kernel (E4M3 bytes converted in registers); wider groups run the
 * tcgen05 kernel, whose converter warps turn each E4M3 block into fp16 in
 * shared memory for fp16 MMAs.  Workspace, streams and device status as
 * gqa_decode.
 */
GQA_API int gqa_decode_fp8(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                           const float* v_scale, const int32_t* seqlens, void* out, int B, int Hq, int Hkv,
                           int D, int Lmax, float scale, void* stream);

/*
 * gqa_prefill -- attention of L query tokens over the same L keys (prompt
 * processing), causal or not.
 *
 *   q, out   [B, Hq, L, D]   bf16, device
 *   k, v     [B, Hkv, L, D]  bf16, device
 *   causal   1: query i sees keys t <= i (the square mask triu(ones, 1) ->
 *               -inf of the Huawei Cloud post, section 5, applied);
 *            0: every query sees all L keys.
 *   scale    fixed at 1/sqrt(D) (the post divides by head_size ** 0.5).
 *
 * QK^T and PV are dense bf16 contractions on the tcgen05 tensor cores with
 * fp32 accumulators in tensor memory; the softmax is fp32; P is rounded to
 * bf16 before PV; out is rounded RNE.
 *
 * Supported: D == 128 or D == 64, any L >= 1, any G.  Otherwise
 * GQA_ERR_UNSUPPORTED.
 * Needs no workspace and allocates nothing.
 */
GQA_API int gqa_prefill(const void* q, const void* k, const void* v, void* out, int B, int L, int Hq,
                int Hkv, int D, int causal, void* stream);

/*
 * gqa_decode_paged -- gqa_decode over a paged KV cache: the cache is a pool of
 * fixed-size pages and a block table maps each sequence's logical pages to
 * pool pages (the split-K heuristic of the gsyq.cn page on xformers takes
 * `page_size` and `is_paged` arguments; the layout is this library's choice).
 *
 *   k_pages, v_pages  [num_pages, Hkv, page_size, D]  bf16, device
 *   block_table       [B, max_pages]  int32, device: row t of sequence b is
 *                     row t % page_size of page block_table[b][t / page_size]
 *   seqlens           [B] int32, device, at most max_pages * page_size
 *                     (larger values are clamped and flagged)
 *   everything else as gqa_decode.
 *
 * page_size must be a multiple of the kernel's key tile: 64 for G <= 8 (or
 * D = 64), 128 for wider groups at D = 128.  Entries past a sequence's last
 * page are never read; a needed entry outside [0, num_pages) sets
 * GQA_DEV_BAD_PAGE and its rows read as zeros (never out-of-bounds memory).
 * Supported shapes, workspace and streams as gqa_decode.
 */
GQA_API int gqa_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                             const int32_t* seqlens, void* out, int B, int Hq, int Hkv, int D, int num_pages,
                             int page_size, int max_pages, float scale, void* stream);

/*
 * gqa_decode_fp8_paged -- gqa_decode_paged over pages of FP8 E4M3 bytes: the
 * two cache forms above combined (the usual layout of a serving engine's
 * quantised cache).  Pages are cut from the sequences' caches, so the scales
 * stay per (sequence, KV head):
 *
 *   k_pages, v_pages  [num_pages, Hkv, page_size, D]  uint8 (E4M3 bytes), device
 *   k_scale, v_scale  [B, Hkv]  fp32, device (4-byte aligned)
 *   block_table, seqlens, num_pages, page_size, max_pages as gqa_decode_paged;
 *   everything else as gqa_decode.
 *
 * Arithmetic as gqa_decode_fp8, page rules and GQA_DEV_BAD_PAGE as
 * gqa_decode_paged; supported shapes as gqa_decode_fp8.  The result is
 * bit-identical to gqa_decode_fp8 on the contiguous cache the pages hold.
 */
GQA_API int gqa_decode_fp8_paged(const void* q, const void* k_pages, const void* v_pages, const float* k_scale,
                                 const float* v_scale, const int32_t* block_table, const int32_t* seqlens, void* out,
                                 int B, int Hq, int Hkv, int D, int num_pages, int page_size, int max_pages,
                                 float scale, void* stream);

/*
 * gqa_rope_append -- the step before a decode: rotary position embedding of
 * the new token and the append of its K/V heads to the cache.  The attention
 * code of the GQA paper notes on 51969.com ("QA 相关") rotates the query and
 * key heads with apply_rotary_pos_emb before repeat_kv, and the Huawei Cloud
 * post "多头注意力机制的代码实现（MQA和GQA）", sections 2 and 5, concatenates
 * each step's K and V to the cache; the rotation is read as the Llama "rotate
 * half" form: for i < D/2 the pair (x[i], x[i + D/2]) turns by the angle
 * p * base^(-2i/D), p = seqlens[b] the new token's position.
 *
 *   q        [B, Hq, D]          bf16, device: the new token's query heads
 *   k_new    [B, Hkv, D]         bf16, device: its key heads (before rotation)
 *   v_new    [B, Hkv, D]         bf16, device: its value heads
 *   q_out    [B, Hq, D]          bf16, device: rotated query (may equal q)
 *   k_cache, v_cache             [B, Hkv, Lmax, D] bf16, device: row p of
 *                                (b, j) receives the rotated key / the value
 *   seqlens  [B]                 int32, device: read as p, then set to p + 1
 *   base     rotary base (10000 for Llama), finite and > 1
 *
 * Afterwards gqa_decode on q_out, the caches and seqlens attends over the new
 * token too.  A sequence with seqlens[b] >= Lmax gets its query rotated but
 * no row appended and its length unchanged, and GQA_DEV_CACHE_FULL is set.
 * The frequencies base^(-2i/D) are computed on the host in fp64, the angles
 * in fp64 on the device and reduced modulo 2 pi before an fp32 sincos;
 * the rotation itself is fp32, results rounded to bf16 (RNE).
 *
 * Supported: D a multiple of 16 up to 256.  Otherwise GQA_ERR_UNSUPPORTED.
 * Allocates nothing; asynchronous on `stream`.
 */
GQA_API int gqa_rope_append(const void* q, const void* k_new, const void* v_new, void* q_out, void* k_cache,
                            void* v_cache, int32_t* seqlens, int B, int Hq, int Hkv, int D, int Lmax,
                            double base, void* stream);

/*
 * gqa_prefill_chunk -- prefill of a chunk of Lq new tokens that follows
 * Lk - Lq tokens already in the cache (chunked prefill): the queries are the
 * chunk's, the keys and values all Lk tokens' (prefix then chunk).  Causal:
 * chunk row i is token Lk - Lq + i and sees keys t <= Lk - Lq + i -- the
 * square mask of the Huawei Cloud post, section 5, aligned at the bottom
 * right, where a query that follows a cached prefix sits; otherwise every row
 * sees all Lk keys.  Lq == Lk is gqa_prefill.
 *
 *   q, out   [B, Hq, Lq, D]   bf16, device
 *   k, v     [B, Hkv, Lk, D]  bf16, device (Lk >= Lq)
 *
 * Same kernel, arithmetic, scale (1/sqrt(D)) and support (D == 64 or 128) as
 * gqa_prefill.  Allocates nothing.
 */
GQA_API int gqa_prefill_chunk(const void* q, const void* k, const void* v, void* out, int B, int Lq, int Lk,
                              int Hq, int Hkv, int D, int causal, void* stream);

/*
 * gqa_meanpool_kv_heads -- MHA -> GQA checkpoint conversion of one key or
 * value projection (the GQA paper notes on 51969.com, section "Uptraining",
 * figure 1, and the checkpoint-conversion experiment, figure 4): group j of
 * the converted model serves query heads j*G .. j*G + G - 1 (G = H / Hkv, the
 * h -> h / G grouping of every attention entry point here) and its K (or V)
 * head's projection is
 *   mode 0 ("Mean", the method the notes adopt): the mean of those G heads'
 *          projections;
 *   mode 1 ("First"): the projection of head j*G.
 * Hkv == 1 is the MHA -> MQA conversion; Hkv == H copies.
 *
 *   w      [H, rows, cols]    bf16, device: head h's block of the projection
 *                             (an nn.Linear weight [H * head_dim, d_model]
 *                             viewed as [H, head_dim, d_model]; a bias with
 *                             cols = 1)
 *   w_out  [Hkv, rows, cols]  bf16, device, written; must not overlap w
 *
 * Arithmetic: fp32 sum over the group in head order, one correctly rounded
 * division by G, bf16 round to nearest even (mode 1 copies bits).  Both
 * pointers 16-byte aligned (else GQA_ERR_MISALIGNED); H % Hkv != 0, a mode
 * outside {0, 1}, a non-positive size or overlapping buffers give
 * GQA_ERR_INVALID_ARG.  Allocates nothing; asynchronous on `stream`.
 */
GQA_API int gqa_meanpool_kv_heads(const void* w, void* w_out, int H, int Hkv, int rows, int cols, int mode,
                                  void* stream);

/*
 * gqa_decode_host / gqa_prefill_host -- the same computations on HOST
 * buffers (pageable or pinned).  The call copies the inputs to library-owned
 * device buffers on `stream`, runs the device entry point, copies `out` back
 * and synchronises `stream` before returning, so the host output is ready.
 * Shapes, layouts and errors are those of the device calls; seqlens_host is
 * host memory here.  The staging buffers are kept (and grown) until
 * gqa_release().
 */
GQA_API int gqa_decode_host(const void* q_host, const void* k_cache_host, const void* v_cache_host,
                    const int32_t* seqlens_host, void* out_host, int B, int Hq, int Hkv, int D,
                    int Lmax, float scale, void* stream);
GQA_API int gqa_prefill_host(const void* q_host, const void* k_host, const void* v_host, void* out_host,
                     int B, int L, int Hq, int Hkv, int D, int causal, void* stream);

/*
 * gqa_decode_noalloc -- gqa_decode for callers that must not have the library
 * allocate device memory: callers that manage all device memory through their
 * own pool (a serving engine that reserves HBM for its KV cache at start-up,
 * where a cudaMalloc from a library could fail or fragment the pool), and
 * callers on a latency-critical path that may not allocate after start-up
 * because cudaMalloc / cudaFree can synchronise the device.
 * The paper pages have no counterpart of this call; it is a deployment
 * variant of gqa_decode.
 *
 * Arguments, layouts, results and device-side fallbacks are those of
 * gqa_decode.  Differences:
 *   - the split workspace is a fixed device array inside libgqa.so of
 *     GQA_NOALLOC_SCRATCH_BYTES; the call makes no cudaMalloc / cudaFree and
 *     calls no allocating routine;
 *   - the first call on a device sets the array up there, with that device
 *     current: it looks up the array's device address, and with the CUDA
 *     runtime's default lazy module loading that lookup loads the module
 *     holding the array, which commits GQA_NOALLOC_SCRATCH_BYTES of device
 *     memory on that device until the process exits.  Make that first call at
 *     start-up, before a memory pool reserves the free HBM and before any
 *     stream capture; later calls change no device-memory total;
 *   - sizes whose workspace exceeds the array return GQA_ERR_TOO_LARGE: at
 *     most GQA_NOALLOC_MAX_PAIRS (b, kv head) pairs (B * Hkv) and
 *     GQA_NOALLOC_MAX_PART_FLOATS partial floats (persistent CTAs x 2 x G x
 *     (D + 2), the CTAs at most 160); every workload with G <= 32, D = 128 and
 *     B * Hkv <= 8192 fits;
 *   - every call, on every stream, shares the one array: calls that overlap
 *     on the GPU race and give wrong results -- order them (one stream, or
 *     events).  Each call clears the parts that must start at zero;
 *   - the device status bits of these calls are kept in the array and are
 *     reported (and cleared) by gqa_get_device_status together with the
 *     library's own word; that read allocates nothing.
 */
#define GQA_NOALLOC_MAX_PAIRS 8192
#define GQA_NOALLOC_MAX_PART_FLOATS 1331200
#define GQA_NOALLOC_SCRATCH_BYTES \
  ((256 + 4 * (GQA_NOALLOC_MAX_PAIRS + 2) + 255) / 256 * 256 + 4 * GQA_NOALLOC_MAX_PART_FLOATS)
GQA_API int gqa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* seqlens, void* out, int B, int Hq, int Hkv, int D,
                               int Lmax, float scale, void* stream);

/* Human-readable text of a status (for GQA_ERR_CUDA it names the CUDA error
 * of the last failure on this host thread).  Never NULL. */
GQA_API const char* gqa_status_string(int status);

/* Synchronises `stream`, then reads and clears the current device's status
 * word (GQA_DEV_* bits) into *flags -- the OR of the word every entry point
 * but gqa_decode_noalloc writes and, once gqa_decode_noalloc has run on the
 * device, the word in its fixed scratch.  After GQA_DEV_WAIT_TIMEOUT it also
 * zeroes the decode workspace's arrival counters.  Returns GQA_OK or
 * GQA_ERR_CUDA.  (The status comes back through a pointer, not as the return
 * value, so that a failure to read it is told apart from the bits.) */
GQA_API int gqa_get_device_status(void* stream, uint32_t* flags);

/* Number of key tiles of the decode split and persistent CTAs the next
 * gqa_decode with these sizes would use, for tests and tuning:
 * *tile_keys, *num_ctas.  Returns GQA_OK or an argument error. */
GQA_API int gqa_decode_plan(int B, int Hq, int Hkv, int D, int Lmax, int* tile_keys, int* num_ctas);

/*
 * Test hooks: failure injection for the error paths (the paper pages have
 * no counterpart).  Not for production use.
 *
 * gqa_test_set_wait_limit_ns -- with ns > 0, kernels launched after this
 * call issue none of their pipeline loads (the TMA copies of Q, K and V) and
 * every pipeline wait (a consumer waiting for its data, the MMA issuer for
 * the softmax, ...) gives up after ns nanoseconds instead of the default
 * 2 s: the waits for the loads that never come run out, the kernel sets
 * GQA_DEV_WAIT_TIMEOUT and returns early with its output invalid; nothing
 * traps.  The waits with which a CTA lets its own copies and MMAs land
 * before it exits keep the 2 s limit.  0 restores normal operation.
 *
 * gqa_test_fail_workspace_allocs -- the next `n` allocations of the decode
 * workspace (made when a decode needs a larger one) fail as out of memory
 * without calling cudaMalloc, so the call returns GQA_ERR_CUDA; n <= 0
 * cancels.
 */
GQA_API void gqa_test_set_wait_limit_ns(unsigned long long ns);
GQA_API void gqa_test_fail_workspace_allocs(int n);

/* Frees every device buffer the library holds on every device it touched.
 * No call may be in flight.  Safe to call more than once. */
GQA_API void gqa_release(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_H_ */
