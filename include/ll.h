/*
 * ll.h -- C ABI of the short-window + frame-sink attention library (sm_103a).
 *
 * Operation (from "LongLive: Real-time Interactive Long Video Generation",
 * §3.3 Efficient Long Inference, "Short window attention" and "Frame sink";
 * §3.1 KV Recache; §4 Implementation; §4.4 Table 4):
 *
 *   A causal, chunk-by-chunk video generator keeps, per transformer layer, a
 *   KV cache of latent frames.  The first S frames (the first frame chunk) are
 *   a sink that is never evicted; the other cached frames form a rolling
 *   window of the W most recent frames, evicted first-in first-out.  A chunk
 *   of C frames (C*T query tokens) attends, per head, to
 *       [sink frames' K/V || window frames' K/V || the chunk's own K/V]
 *   with softmax(Q K^T / sqrt(d)) V and no mask inside that list.  When a
 *   pass commits, the chunk's K/V enter the cache (evicting the oldest
 *   window frames).  At a prompt switch the resident frames' K/V are
 *   recomputed ("recache") and written back in place.
 *
 * Conventions for every call:
 *   - Shapes: T = tokens_per_frame, C = chunk_frames, S = sink_frames,
 *     W = window_frames, H = heads, d = head_dim (64 or 128).
 *   - Token tensors (q, k, v, out, *_win) are caller-owned DEVICE pointers,
 *     contiguous [tokens][H][d] in the cache dtype (bf16 or fp32), 16-byte
 *     aligned.  They are borrowed until the work enqueued on `stream`
 *     completes.  No call keeps a pointer after that.
 *   - Calls on one cache are not thread-safe.  Host metadata (frames
 *     committed, frame-to-slot map) is updated when a call is enqueued, so
 *     calls must be issued in stream order on a single stream.
 *   - Argument and state errors are detected on the host before anything is
 *     enqueued; the call then returns the error and changes nothing.
 *   - Kernel launch failures return LL_ERR_CUDA.  A device-side wait that
 *     runs out of time sets an error word that the next call (or
 *     ll_cache_state / ll_sync) reports as LL_ERR_DEVICE_TIMEOUT.
 *   - No call synchronises the device except ll_cache_read, ll_sync and
 *     ll_cache_state (which checks the device error word).
 */
#ifndef LL_H_
#define LL_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LL_API __attribute__((visibility("default")))
#else
#define LL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ll_cache ll_cache; /* opaque */

/*
 * Element type of the cache and of every token tensor.
 *   LL_BF16, LL_FP32: tokens and both caches in that type.  At head_dim 64 an
 *     LL_FP32 cache runs on the tensor cores with tf32 operands
 *     (tcgen05.mma kind::tf32): Q K^T sums three tf32 products of split
 *     operands (x = tf32(x) + tf32(x - tf32(x)), the dropped term below 2^-22
 *     of each product), so the scores keep fp32 accuracy; P V reads P and V
 *     rounded to tf32 (nearest).  At head_dim 128 it runs on CUDA cores in fp32.
 *   LL_BF16_K8: token tensors (q, k, v, out, windows) and the V cache in bf16;
 *     the K cache holds every key rounded to FP8 e4m3 (one byte: round to
 *     nearest even, saturating at +-448), and Q K^T runs on the FP8 tensor-core
 *     path (tcgen05.mma kind::f8f6f4) with q and the fresh keys rounded the same
 *     way; P V, the softmax statistics and out are as in LL_BF16.  The K cache
 *     takes half the bytes.  head_dim 128 only.  (The pages report INT8
 *     inference (Abstract, §5 Conclusion); rounding the keys is a defined input
 *     step, so results match attention over the rounded q and k.)
 *   LL_FP8: as LL_BF16_K8, and the V cache holds every value rounded to e4m3
 *     the same way: both caches take half the bytes of bf16.  P V runs on the
 *     tensor cores with fp16 operands (kind::f16): each V tile is widened to
 *     fp16 (exact for e4m3) in shared memory and P is rounded to fp16.  Results
 *     match attention over the rounded q, k and v.  head_dim 128 only.
 */
typedef enum { LL_BF16 = 0, LL_FP32 = 1, LL_BF16_K8 = 2, LL_FP8 = 3 } ll_dtype;

typedef enum {
  LL_OK = 0,
  LL_ERR_INVALID_ARG = 1,   /* bad shape, null or misaligned pointer, layer out of range */
  LL_ERR_UNSUPPORTED = 2,   /* valid request the library does not implement (e.g. d not 64/128) */
  LL_ERR_OOM = 3,           /* device allocation failed in ll_cache_create */
  LL_ERR_STATE = 4,         /* call not allowed in the cache's state (e.g. recache of an empty layer) */
  LL_ERR_CUDA = 5,          /* a CUDA runtime call or kernel launch failed */
  LL_ERR_DEVICE_TIMEOUT = 6 /* a bounded device-side wait gave up (reported by a later call) */
} ll_status;

/* Human-readable name of a status code (static storage). */
LL_API const char* ll_status_str(ll_status s);

/*
 * ll_cache_create -- allocate the per-layer KV caches.
 * §3.3 "Short window attention": the cache is sized by the window, not by the
 * video length: K and V each hold layers * H * (S + W) * T * d elements,
 * head-major [layer][head][slot][token][d] (K one byte per element with
 * LL_BF16_K8, K and V with LL_FP8).  The memory is cudaMalloc'ed on the
 * current device and
 * zero-filled; ll_cache_destroy frees it.
 * Requirements: layers, heads, tokens_per_frame, chunk_frames >= 1;
 * sink_frames, window_frames >= 0; head_dim in {64, 128} (128 for
 * LL_BF16_K8 and LL_FP8).  Limits of the
 * library, beyond which the call returns LL_ERR_UNSUPPORTED: S + W <= 512 and
 * C <= 512 frames, heads <= 127 (the commit copy runs 512 x heads blocks at
 * most), (S + W + C) * T <= 2^30 tokens.  Returns LL_ERR_OOM if the
 * allocation fails.  On any error *out is NULL.
 */
LL_API ll_status ll_cache_create(ll_cache** out, int layers, int heads, int head_dim,
                          int tokens_per_frame, int sink_frames, int window_frames,
                          int chunk_frames, ll_dtype dtype);

/* Free the cache (waits for the device to finish with it).  NULL is ignored. */
LL_API void ll_cache_destroy(ll_cache* cache);

/*
 * ll_attend_chunk -- one query pass of the chunk that starts at frame
 * t0 = frames committed so far in `layer`.
 * §3.3 "Frame sink" + "Short window attention": per head h,
 *   out_h = softmax(q_h K_h^T / sqrt(d)) V_h,
 *   K/V = [frames 0..min(S,t0)-1 || frames max(S,t0-W)..t0-1 || k/v of this chunk].
 * q, k, v: [C*T][H][d] device buffers in the cache dtype; out: [C*T][H][d] in
 * the output dtype (see ll_set_output_dtype); out may share no byte with q,
 * k or v (LL_ERR_INVALID_ARG).
 * commit != 0: after the attention, the chunk's K/V are written into the
 * cache: frame f < S into sink slot f, frame f >= S into ring slot
 * S + ((f - S) mod W), replacing the frame W positions older; frames that
 * would be evicted within the same commit (W < C) are not written.  Frames
 * committed += C.  Softmax statistics are fp32; out is rounded to the dtype.
 */
LL_API ll_status ll_attend_chunk(ll_cache* cache, int layer, const void* q, const void* k,
                          const void* v, void* out, int commit, void* stream);

/*
 * ll_recache -- §3.1 "KV recache": replace the K/V of the R frames resident
 * in `layer` (R = min(S,n) + min(W, max(0, n - S)), n = frames committed) by
 * k_win/v_win, [R*T][H][d], given in list order (sink frames ascending, then
 * window frames ascending).  Frame indices and n do not change.
 * Returns LL_ERR_STATE if the layer is empty (n = 0).  With
 * ll_set_recache_scope(LL_RECACHE_WINDOW) only the window frames are given
 * and rewritten.
 */
LL_API ll_status ll_recache(ll_cache* cache, int layer, const void* k_win, const void* v_win,
                     void* stream);

/*
 * ll_recache_attend -- the recache prefill: block-causal attention over the
 * R resident frames' fresh q/k/v (list cut into blocks of C frames; query
 * rows of block g see key blocks 0..g), written to out_win [R*T][H][d]
 * (sharing no byte with q_win, k_win or v_win: LL_ERR_INVALID_ARG);
 * then the same K/V write as ll_recache.
 */
LL_API ll_status ll_recache_attend(ll_cache* cache, int layer, const void* q_win, const void* k_win,
                            const void* v_win, void* out_win, void* stream);

/*
 * ll_recache_tokens -- the token rows that a recache of `layer` reads from
 * k_win and v_win (and, for ll_recache_attend, from q_win and writes to
 * out_win) in the cache's current state and recache scope: R * T, where R is
 * the number of frames the recache rewrites (0 when it would return
 * LL_ERR_STATE).  Host metadata only: no device work, no synchronisation.
 * The recache calls take raw pointers and cannot see a buffer's length, so
 * callers check theirs against this.
 */
LL_API ll_status ll_recache_tokens(const ll_cache* cache, int layer, int64_t* tokens);

/*
 * ll_set_output_dtype -- element type of `out` / `out_win` in later calls.
 * Default: the cache dtype.  LL_FP32 on a bf16 cache returns the fp32
 * accumulator result unrounded (bf16 rounding alone costs up to |o| * 2^-9,
 * which passes 1e-2 once |o| >= 4).  LL_BF16 on an fp32 cache is rejected.
 */
LL_API ll_status ll_set_output_dtype(ll_cache* cache, ll_dtype dtype);

/*
 * Options for two readings the pages leave open; both default to the first value.
 *
 * ll_set_chunk_mask -- which of the chunk's own keys a query sees.
 *   LL_MASK_CHUNK: all of them (chunk-level block causality; the default).
 *   LL_MASK_FRAME: the model is called "frame-level autoregressive", so a query
 *     of chunk frame t0 + i sees the cached frames and the chunk's frames
 *     t0 .. t0 + i only; the recache prefill then uses one-frame blocks.
 * Applies to later ll_attend_chunk / ll_recache_attend calls of this cache.
 */
typedef enum { LL_MASK_CHUNK = 0, LL_MASK_FRAME = 1 } ll_chunk_mask;
LL_API ll_status ll_set_chunk_mask(ll_cache* cache, int mode);

/*
 * ll_set_recache_scope -- which frames a recache rewrites.
 *   LL_RECACHE_RESIDENT: every resident frame, sink and window (the default).
 *   LL_RECACHE_WINDOW: §3.3 "rebuild the cache only from the most recent W
 *     frames": the sink keeps its K/V; k_win / v_win (and q_win, out_win) hold
 *     the Rw = min(W, max(0, n - S)) window frames, ascending; the prefill
 *     queries see every cached sink frame plus the fresh window, block-causal
 *     over the window list from its first frame.  A recache with no window
 *     frame resident returns LL_ERR_STATE.
 */
typedef enum { LL_RECACHE_RESIDENT = 0, LL_RECACHE_WINDOW = 1 } ll_recache_scope;
LL_API ll_status ll_set_recache_scope(ll_cache* cache, int scope);

/* §4.4 Table 4 ("no KV cache"): drop every frame of every layer (metadata only). */
LL_API ll_status ll_reset(ll_cache* cache);

/*
 * ll_cache_state -- host copy of one layer's bookkeeping: frames committed and
 * frame_of_slot[S + W] (-1 = empty slot).  Synchronises the device first and
 * returns LL_ERR_DEVICE_TIMEOUT if a device-side wait gave up since the last
 * check.  Either output pointer may be NULL.
 */
LL_API ll_status ll_cache_state(ll_cache* cache, int layer, int64_t* frames_committed,
                         int64_t* frame_of_slot);

/*
 * ll_cache_read -- copy one layer's raw cache to HOST buffers, each
 * H * (S + W) * T * d elements in the head-major slot layout (for tests;
 * synchronises the device).  With LL_BF16_K8 host_k receives the e4m3 bytes
 * (one per element) and host_v bf16; with LL_FP8 both receive e4m3 bytes.
 */
LL_API ll_status ll_cache_read(ll_cache* cache, int layer, void* host_k, void* host_v);

/* Wait for all work on the device; report a pending device error, if any. */
LL_API ll_status ll_sync(ll_cache* cache);

/* Sizes of a cache: S + W slots, bytes of one layer's K cache and the size of a K element
 * (V: the same, except LL_BF16_K8, whose V elements take 2 bytes and K elements 1).
 * With LL_FP8 K and V elements both take 1 byte. */
LL_API ll_status ll_cache_info(const ll_cache* cache, int* slots, size_t* layer_bytes, int* elem_bytes);

/*
 * Host-side index logic, exported for tests (no device needed):
 * ll_frame_slot: slot of frame f (-1 if f can not be resident, i.e. f >= S and W = 0).
 * ll_resident_frames: frames resident after n commits in list order
 * (sink asc, window asc) into frames[] (capacity >= S + W); returns the count.
 */
LL_API int ll_frame_slot(int sink_frames, int window_frames, int64_t f);
LL_API int ll_resident_frames(int sink_frames, int window_frames, int64_t n, int64_t* frames);

/*
 * Number of kernel launches this library has made since it was loaded
 * (all caches, all devices).  Benchmarks read it to count launches.
 */
LL_API uint64_t ll_launch_count(void);

/*
 * Per-kernel timing.  ll_profile_enable(cache, n) with n > 0 brackets one
 * launch in every n of each kind (the first, the (n+1)-th, ...) with two CUDA
 * events on its stream; n = 1 brackets every launch, n <= 0 switches timing
 * off.  ll_profile_read synchronises, returns for one kernel kind the number of
 * bracketed launches and their summed device time (milliseconds) since timing
 * was switched on, and clears that kind.  An attend bracket also holds the
 * merge of split work items that follows the attention kernel.
 */
typedef enum {
  LL_KERNEL_ATTEND = 0,  /* chunk attention (tensor-core or CUDA-core kernel) */
  LL_KERNEL_PREFILL = 1, /* recache prefill attention */
  LL_KERNEL_COPY = 2,    /* commit / recache K,V write */
  LL_KERNEL_KINDS = 3
} ll_kernel_kind;
LL_API ll_status ll_profile_enable(ll_cache* cache, int enable);
LL_API ll_status ll_profile_read(ll_cache* cache, int kind, int64_t* launches, double* total_ms);

/*
 * Test hook: a non-zero value makes the next tensor-core attention launch of
 * this cache skip one barrier arrival so its bounded waits run out after
 * `timeout_us` microseconds; the kernel then returns early and the next call
 * reports LL_ERR_DEVICE_TIMEOUT.  0 disarms it.  The CUDA-core kernel (fp32
 * at head_dim 128) has no barriers and ignores it.
 */
LL_API ll_status ll_debug_inject_stall(ll_cache* cache, int enable, int timeout_us);

/*
 * Test hook: a non-zero value routes this cache's bf16 or fp32 attention
 * through the CUDA-core kernel (one warp per query row; the one fp32 at
 * head_dim 128 runs on) instead of the tensor-core kernel, so tests can compare
 * the two CUDA kernels.  LL_BF16_K8 and LL_FP8 caches ignore it (their keys need
 * the FP8 tensor-core path).
 */
LL_API ll_status ll_debug_use_simt(ll_cache* cache, int enable);

/*
 * Test hook: a non-zero value routes this cache's bf16 attention at head_dim 128
 * through the CTA-pair tensor-core kernel (two SMs share every MMA, M = 256;
 * slower than the default one-CTA kernel on B300) instead of the one-CTA
 * kernel, so tests and benchmarks can run both on the same inputs.  Other
 * head dims and the e4m3 caches (LL_BF16_K8, LL_FP8) ignore it.
 */
LL_API ll_status ll_debug_pair_kernel(ll_cache* cache, int enable);

/*
 * Test hook: a non-zero value fills every slot of this cache that holds no
 * resident frame with all-ones bytes (NaN in bf16, fp32 and e4m3), now and after
 * every ll_reset, so that an attention that read a slot it should not read
 * returns NaN.  Synchronises the device.  The environment variable LL_POISON
 * (any value but 0) turns it on for every cache at ll_cache_create.
 */
LL_API ll_status ll_debug_poison(ll_cache* cache, int enable);

/*
 * Fault injection on the host, process-wide: the n-th next device allocation
 * (LL_FAULT_ALLOC: cudaMalloc / mapped host allocation in ll_cache_create) or
 * kernel launch step (LL_FAULT_LAUNCH: the attention of a call, or its commit /
 * recache copy) of the library fails as if the CUDA call had failed, without
 * making it.  The call then returns LL_ERR_OOM (allocation), LL_ERR_CUDA
 * (mapped host allocation, launch) and changes no cache state.  n = 0 disarms.
 * The environment variable LL_FAULT="alloc:N" and/or "launch:N" (comma-separated)
 * arms the same when the library loads.  Returns LL_ERR_INVALID_ARG for an
 * unknown kind or n < 0.
 */
typedef enum { LL_FAULT_ALLOC = 1, LL_FAULT_LAUNCH = 2 } ll_fault_kind;
LL_API ll_status ll_debug_inject_fault(int kind, int n);

/*
 * Test hook (host only, no device needed): replay the work schedule of a
 * tensor-core attention launch with Lq queries, La cached and Lb fresh keys
 * per head and at most max_ctas CTAs; mode 0 = chunk attend (persistent:
 * whole rounds, then the left-over items split into runs of key tiles),
 * mode 1 = recache prefill (La cached keys all visible, the Lb fresh keys
 * block-causal in blocks of block_tokens; persistent, items longest first in
 * zigzag rounds, none split), mode 2 = frame-causal chunk attend (the mode 0
 * schedule; its mask is applied inside the tiles).  Writes the
 * CTA count to *grid, the pieces of work as (cta, item, first key tile, end key
 * tile, partial, scratch slot) sextuples into pieces[cap], and the items split
 * across CTAs as (item, parts, slot of each part ...) into splits[split_cap]
 * (*split_ints = ints written).  Returns the number of pieces (-1 on bad
 * arguments: a size below 1, a mode other than 0-2, block_tokens < 1 in
 * modes 1 and 2).  Items are (head, 256-row query block): head-major in mode 0,
 * last query block first in mode 1; key tiles hold 128 keys.
 */
LL_API int ll_debug_attend_schedule(int Lq, int La, int Lb, int heads, int max_ctas, int mode, int block_tokens,
                                    int* grid, int* pieces, int cap, int* splits, int split_cap, int* split_ints);

/*
 * ll_attend_chunk_noalloc -- the attention of ll_attend_chunk (no commit) for
 * callers that may not allocate device memory.  The paper has no counterpart:
 * this entry point exists for deployment.
 *
 * Who cannot allocate: a host program whose memory manager owns the GPU's
 * whole budget (e.g. a serving runtime that reserves nearly all of HBM in its
 * own pool and hands out slices: a cudaMalloc behind its back fails or breaks
 * its accounting), a plugin interface that hands a library a stream and
 * buffers and forbids it to allocate, and real-time loops whose per-frame
 * deadline cannot absorb cudaMalloc / cudaFree, which may block the host and
 * synchronise the device.  ll_cache_create allocates, so these callers keep
 * the cache in memory they own and place frames with ll_frame_slot /
 * ll_resident_frames.  This call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *
 * Per head h: out_h = softmax(q_h K_h^T / sqrt(d)) V_h over the keys
 * [cached rows || the chunk's own rows], every query seeing every key (the
 * default chunk mask), bf16 in and out, fp32 softmax.
 *   q, k, v, out: [chunk_tokens][heads][head_dim] bf16 device buffers (16-byte
 *                 aligned; out may share no byte with q, k, v or the
 *                 cached rows: LL_ERR_INVALID_ARG).
 *   k_cached, v_cached: the resident rows, head-major: head h's cached_tokens
 *                 rows of head_dim elements start at element
 *                 h * cached_head_stride (16-byte aligned, stride a multiple
 *                 of 8).  The cache layout of ll_cache_read qualifies, with
 *                 the resident frames in slots [0, R) and
 *                 cached_tokens = R * T.  Ignored when cached_tokens = 0.
 *   err_word: optional device-visible 4-byte word; a device wait that runs
 *             out (2 s) writes 1 into it and out is then undefined.  The
 *             caller zeroes it and reads it after the stream completes.
 *             NULL: such an event is not reported.
 *   stream: CUDA stream (cudaStream_t) of the work.
 * The scratch for the split work items' partial results is a file-scope
 * device array of LL_NOALLOC_SCRATCH_BYTES (37.6 MiB), which every GPU that
 * loads the library holds until the process exits: two partial results of 256
 * query rows per CTA for up to LL_NOALLOC_PARTIAL_SLOTS / 2 = 148 CTAs at
 * head_dim 128 (one per SM of a B300).  At head_dim 64 the array would hold
 * 291 CTAs' partial results, but no attend launch uses more than 256 CTAs.  A request that
 * would need more (a GPU with more SMs and more work items than that) returns
 * LL_ERR_UNSUPPORTED before anything is enqueued; so do head_dim not in
 * {64, 128} and cached_tokens + chunk_tokens > 2^30.  Bad pointers, strides or
 * sizes return LL_ERR_INVALID_ARG.
 * The first call on a device, with that device current, looks up the array's
 * device address (cudaGetSymbolAddress); make it before any stream capture.
 * Every call on a device shares the array, and it keeps the previous call's
 * contents: nothing in it needs to start at zero, since each call writes
 * every partial result it later reads.  Calls whose work may overlap on the
 * GPU (unordered streams, other host threads) race on the array and give
 * wrong results: order them, e.g. on one stream.
 */
#define LL_NOALLOC_PARTIAL_SLOTS 296
#define LL_NOALLOC_SCRATCH_BYTES (256 + (size_t)LL_NOALLOC_PARTIAL_SLOTS * 256 * 130 * 4)
LL_API ll_status ll_attend_chunk_noalloc(const void* q, const void* k_cached, const void* v_cached,
                                         int cached_tokens, int64_t cached_head_stride, const void* k,
                                         const void* v, int chunk_tokens, void* out, int heads, int head_dim,
                                         unsigned* err_word, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LL_H_ */
