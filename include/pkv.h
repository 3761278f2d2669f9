/*
 * pkv.h - paged KV cache for streaming 3D reconstruction on one GB300 (sm_103a).
 *
 * What the library computes
 * -------------------------
 * "LingBot-Map Paged KV Cache: 3D reconstruction managed like LLM memory",
 * section 2: each layer's KV is cut into fixed-size pages handed out from a free
 * list. A stream's cache has three page types:
 *   - scale pages: the patch tokens of the first num_scale frames, never evicted;
 *   - sliding-window pages: the patch tokens of the most recent `window` frames;
 *     a page that leaves the window goes straight back to the free list, where
 *     the next frame reuses it;
 *   - special pages: each frame's n_special special tokens (camera / register /
 *     scale), appended floor(page_size / n_special) frames to a page (42 x 6 in a
 *     256-slot page), never recycled.
 * Attention runs over a visible page table built in the order scale -> window ->
 * special; the fill of the last page is last_page_len. Section 3: a non-keyframe
 * is appended, attended, then rolled back. Section 4: in windowed mode the cache
 * is reset once per window of window_slots KV slots, and the last
 * overlap_keyframes keyframes carry over into the next window.
 *
 * vLLM-Omni RFC "Reconstruction Engine" (issue 2727), sections 2.3 and 3.3:
 * chunked sliding-window global attention. Frames are grouped in chunks of
 * chunk_size; the current chunk's tokens attend over the KV of the most recent
 * sliding_window_num chunks (itself included); the oldest chunk is then evicted.
 *
 * Conventions (every call)
 * ------------------------
 *  - Tensors q, k, v, out are caller-owned DEVICE buffers of bf16, layout
 *    [tokens][heads][head_dim], contiguous, 16-byte aligned. Values must be finite.
 *  - `cuda_stream` is a cudaStream_t (NULL = legacy default stream). Every call
 *    that touches the device is asynchronous and ordered on that stream. All
 *    calls on one handle must be issued on one CUDA stream, or ordered by the
 *    caller: the handle's device metadata and scratch are shared by its calls.
 *  - The library owns the page pool, the free list and all page-id metadata in
 *    device memory (allocated by create / stream_open, freed by close / destroy).
 *    The host keeps only counters, so argument, capacity (OOM) and call-order
 *    (STATE) errors are detected before anything is launched: a call that
 *    returns an error has changed nothing. Kernels that find an inconsistency
 *    (a page id outside the pool) record it in a device error word instead of
 *    faulting; pkv_sync reports it as PKV_ERR_DEVICE.
 *  - Non-zero statuses come with a message from pkv_last_error.
 *  - head_dim must be 64; page_size a multiple of 16 in [16, 256] that divides
 *    or is divided by 64.
 *  - There is no CPU fallback and no other backend.
 *
 * Pool layout (documented for callers that read the pool directly)
 * ------------------------------------------------------------------
 * pool[layer][page][kv][head][slot][64] bf16, kv = 0 for K, 1 for V. Inside each
 * [slot][64] block (one 128-byte row per slot) the eight 16-byte chunks of a row
 * are stored XOR-swizzled: logical chunk c of slot s sits at chunk (c ^ (s & 7)).
 * This is the 128-byte-swizzled operand layout the tensor cores read, so a page
 * block is copied into shared memory as-is. Every slot of a held page is either a
 * valid token or zero.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_ctx* pkv_t;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID = 1, /* bad argument or shape                                  */
  PKV_ERR_OOM = 2,     /* the free list (or the stream table) cannot cover the call */
  PKV_ERR_STATE = 3,   /* call order: e.g. rollback with nothing to roll back    */
  PKV_ERR_CUDA = 4,    /* a CUDA runtime call failed                             */
  PKV_ERR_TIMEOUT = 5, /* a bounded device wait gave up                          */
  PKV_ERR_DEVICE = 6   /* a kernel recorded an inconsistency in the error word   */
} pkv_status;

enum { PKV_MODE_FRAME = 0, PKV_MODE_CHUNKED = 1 };

/* Per-stream configuration. Fields of the other mode are ignored. */
typedef struct {
  int mode;              /* PKV_MODE_FRAME or PKV_MODE_CHUNKED                      */
  /* frame mode (LingBot-Map) */
  int num_scale;         /* scale frames kept forever (8)                           */
  int window;            /* sliding-window frames, including the current one (64)   */
  int n_patch;           /* patch tokens per frame; must equal page_size (256)      */
  int n_special;         /* special tokens per frame (6)                            */
  int window_slots;      /* windowed mode: KV slots (cached keyframes) per window; 0 = off */
  int overlap_keyframes; /* keyframes carried into the next window; <= num_scale    */
  /* chunked mode (VGGT RFC) */
  int chunk_size;        /* frames per chunk (8)                                    */
  int sliding_window_num;/* chunks visible, including the current one (4)           */
  int tokens_per_frame;  /* tokens appended per frame (1374)                        */
} pkv_stream_cfg;

/* Create a cache of `pool_pages` pages of `page_size` slots for one layer
 * ("LingBot-Map Paged KV Cache", section 2: each layer's KV lives in fixed-size
 * pages handed out from a free list).
 * Equivalent to pkv_create_ex(pool_pages, page_size, heads, head_dim, 1, 64, out).
 * Errors: as pkv_create_ex. */
pkv_status pkv_create(int pool_pages, int page_size, int heads, int head_dim, pkv_t* out);

/* Create with `layers` page sets ("LingBot-Map Paged KV Cache", section 2: the
 * cache is kept per layer, in fixed-size pages taken from a free list; here all
 * layers share one page table, so a page id names the same page in every layer,
 * and the metadata is updated once per frame) and room for
 * `max_streams` concurrent streams sharing the pool and its free list.
 * Allocates layers*pool_pages*2*heads*page_size*head_dim bf16 (zeroed), plus, for
 * pkv_attend_blocksparse, a cache of each page's mean key per layer (fp32,
 * layers*pool_pages*heads*head_dim values: 1/page_size of the pool's bytes) and a
 * few KB of scratch. The free list is a stack that initially hands out pages
 * 0, 1, 2, ... *out receives the handle, which the caller releases with pkv_destroy.
 * Errors: INVALID (null out; head_dim != 64; page_size not a multiple of 16 in
 * 16..256 that divides or is divisible by 64; pool_pages, heads (<= 32), layers or
 * max_streams (<= 1024) out of range); OOM or CUDA if the device allocations fail
 * (nothing is left allocated). The message is pkv_last_error(NULL). */
pkv_status pkv_create_ex(int pool_pages, int page_size, int heads, int head_dim, int layers,
                         int max_streams, pkv_t* out);

/* As pkv_create_ex, but the pages hold FP8 keys and values (vLLM-Omni RFC
 * "Reconstruction Engine", section 3.4, acceleration dimension 5: KV cache FP8,
 * about half the memory). Every stored row of head_dim = 64 values (one token,
 * one head, K or V) is kept as 64 OCP E4M3 codes (1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits; largest magnitude 448) of v * 2^-e and one exponent
 * byte e: the smallest integer with max|v| <= 448 * 2^e (0 for a zero row),
 * clamped to [-126, 126], codes rounded to nearest, ties to even. So a row holds decode(code) * 2^e,
 * which is exact in bf16, and the quantization is the format's only rounding.
 * A page takes 2 * heads * page_size * 65 bytes instead of * 128. Append,
 * rollback, eviction, the windowed reset and every attention call work as on
 * bf16 pages; the attention dequantizes each K/V tile in shared memory and
 * computes exactly what bf16 pages holding the dequantized values would give.
 * K and V must be finite with magnitude below 2^126.
 * Page layout (for callers that read the pool): per page, [kv][head] planes of
 * page_size rows, each plane in blocks of B = min(page_size, 64) rows: the B rows'
 * 64 code bytes (unswizzled), then their B exponent bytes (int8), so a block is
 * B * 65 bytes and one copy moves a block's codes with their exponents.
 * pkv_attend_blocksparse and pkv_read_page refuse FP8 caches (pkv_read_page_fp8
 * reads them).
 * Errors: as pkv_create_ex. */
pkv_status pkv_create_fp8(int pool_pages, int page_size, int heads, int head_dim, int layers,
                          int max_streams, pkv_t* out);

/* Free everything. Synchronises the device first. NULL is accepted. Always OK. */
pkv_status pkv_destroy(pkv_t h);

/* Open a stream; *stream_id receives the lowest unused id ("LingBot-Map Paged KV
 * Cache", section 2: a stream's cache is its scale, sliding-window and special
 * page lists, filled from the shared free list; section 4: windowed mode; vLLM-Omni
 * RFC "Reconstruction Engine", sections 2.3 and 3.3: a chunked stream keeps the
 * pages of its most recent sliding_window_num chunks). Allocates the stream's
 * page-id lists on the device (synchronously), and grows the handle's split-KV
 * scratch to what this stream's attention calls need at their natural query
 * count (frame mode: n_patch + n_special rows; chunked mode: chunk_size x
 * tokens_per_frame rows) for every table size the stream can reach, so that
 * those calls never allocate.
 * Errors: INVALID (null argument, a configuration field out of range: frame mode
 * needs n_patch == page_size, 1 <= n_special <= page_size, window >= 1,
 * overlap_keyframes <= num_scale; chunked mode 1 <= sliding_window_num <= 16),
 * OOM (max_streams already open), CUDA (the allocation failed). */
pkv_status pkv_stream_open(pkv_t h, const pkv_stream_cfg* cfg, int* stream_id);

/* Close a stream: its pages go back on the free stack (frame mode: scale pages,
 * window pages oldest first, then special pages in order; chunked mode: chunks
 * oldest first, pages in order). Synchronises cuda_stream before freeing the
 * stream's device lists. Errors: INVALID (the stream is not open), CUDA. */
pkv_status pkv_stream_close(pkv_t h, int stream_id, void* cuda_stream);

/* Return every page of the stream to the free stack (in pkv_stream_close's
 * order) and clear its counters, keeping the stream open and its device lists
 * allocated: the stream starts over as if just opened. No allocation and no
 * synchronisation, so it can sit inside a captured CUDA graph.
 * Errors: INVALID (the stream is not open), CUDA (the launch failed). */
pkv_status pkv_stream_reset(pkv_t h, int stream_id, void* cuda_stream);

/* Append one frame's K and V ("LingBot-Map Paged KV Cache", section 2; RFC
 * section 3.3 "KV Cache append").
 * k, v: device bf16 [n_tokens][heads][head_dim], tokens in frame order (frame
 * mode: n_patch patch tokens then n_special special tokens).
 * layer == 0 starts a new frame: pages are popped from the free list (frame mode:
 * the patch page first, then a new special page when the current one holds
 * floor(page_size/n_special) frames; chunked mode: as many pages as the chunk's
 * packed tokens need, a new chunk starting on a new page) and the tokens are
 * scattered into their slots. layer > 0 writes the same slots of that layer's
 * page set and must follow layer 0 of the same frame.
 * Errors: INVALID (shape / layer), OOM (too few free pages), STATE (frame mode:
 * the window already holds `window` pages, or layer == 0 while the previous frame
 * is still pending, i.e. neither rolled back nor committed by pkv_evict_window;
 * chunked: the chunk is full or the window holds sliding_window_num chunks;
 * layer > 0 without a pending frame). */
pkv_status pkv_append_frame(pkv_t h, int stream_id, int layer, const void* k, const void* v,
                            int n_tokens, void* cuda_stream);

/* Append one frame to each of `n` frame-mode streams (n <= 32) in one launch, in
 * the order given: stream i pops its pages after streams 0..i-1 (an exclusive
 * warp scan of the page needs gives each stream its place on the free stack).
 * stream_ids, k, v are HOST arrays of n entries; k[i], v[i] are device pointers.
 * The batch is validated as a whole: on error nothing is appended. */
pkv_status pkv_append_frames(pkv_t h, int n, const int* stream_ids, int layer,
                             const void* const* k, const void* const* v, int n_tokens,
                             void* cuda_stream);

/* Undo the last append (section 3: a non-keyframe is appended, attended, then
 * rolled back). Pages it popped are pushed back in reverse order, so the free
 * stack, the page lists and every valid slot are exactly as before the append.
 * Errors: STATE if no append is pending (already rolled back, or committed by
 * pkv_evict_window). */
pkv_status pkv_rollback_last_frame(pkv_t h, int stream_id, void* cuda_stream);

/* Commit the pending frame and evict (section 2; RFC 3.3 "evict oldest chunk").
 * Frame mode: window pages beyond window-1 go back on the free stack, oldest
 * first, so the next frame reuses them; no KV bytes move. In windowed mode, once
 * the stream holds window_slots cached keyframes, the window is reset (section 4):
 * the last overlap_keyframes held frames become the new window's scale frames
 * (their patch pages stay in place; their special tokens are copied, for every
 * layer, into freshly popped special pages) and all other pages are freed.
 * Chunked mode: closes the current chunk and frees the oldest chunks' pages until
 * sliding_window_num-1 chunks remain.
 * Errors: OOM if a reset cannot pop its special page. */
pkv_status pkv_evict_window(pkv_t h, int stream_id, void* cuda_stream);

/* A run of n_frames frames of one frame-mode stream, driven from native code
 * (sections 2-3 of "LingBot-Map Paged KV Cache": each new frame is appended,
 * attends over the visible pages, then is committed with pkv_evict_window when it
 * is a keyframe or undone with pkv_rollback_last_frame when it is not). For
 * every frame t in order it makes exactly these calls on cuda_stream:
 *   pkv_append_frame(h, stream_id, layer, k[t], v[t], tokens)
 *   pkv_attend(h, q[t], tokens, stream_id, layer, out[t], sm_scale)
 *   keyframe == NULL || keyframe[t] ? pkv_evict_window : pkv_rollback_last_frame
 * so results and state equal those of the separate calls; only the host work per
 * frame shrinks (no caller round trip between the calls).
 * q, k, v, out: device bf16 [n_frames][tokens][heads][64], contiguous, 16-byte
 * aligned, owned by the caller; keyframe: HOST array of n_frames bytes, or NULL
 * (every frame is a keyframe). tokens must be the stream's n_patch + n_special.
 * With several layers, a frame's evict or rollback follows its append and attend
 * of `layer` alone, so this drives one-layer streams (or callers that run one
 * layer per stream). n_frames = 0 is a no-op.
 * Errors: INVALID (null or unaligned pointer, tokens, layer, n_frames < 0), STATE
 * (a chunked-mode stream, or a frame of this stream is pending); else the first
 * failing call's status, with the frame's index in pkv_last_error. Frames before
 * the failing one stay applied (each call is all-or-nothing, the run is not). */
pkv_status pkv_stream_frames(pkv_t h, int stream_id, int layer, const void* q, const void* k,
                             const void* v, int n_frames, int tokens,
                             const unsigned char* keyframe, void* out, float sm_scale,
                             void* cuda_stream);

/* A run of n_frames frames of one frame-mode stream through n_layers layers,
 * driven from native code: the model-shaped step of "LingBot-Map Paged KV Cache"
 * sections 2-3 (each layer appends the new frame's K/V and attends its queries
 * over that layer's visible pages; the frame is then committed with
 * pkv_evict_window when it is a keyframe, or undone with pkv_rollback_last_frame).
 * For frame i (its index frame0 + i) it makes exactly these calls on cuda_stream:
 *   for l in 0 .. n_layers-1:
 *     pkv_append_frame(h, stream_id, l, k[l] + slot, v[l] + slot, tokens)
 *     pkv_attend(h, q[l] + slot, tokens, stream_id, l, out[l] + slot, sm_scale)
 *   keyframe == NULL || keyframe[i] ? pkv_evict_window : pkv_rollback_last_frame
 * where slot is frame (frame0 + i) % ring of the per-layer input rings: q[l], k[l],
 * v[l], out[l] are device bf16 [ring][tokens][heads][64] (HOST arrays of n_layers
 * device pointers, each 16-byte aligned). keyframe: HOST array of n_frames bytes,
 * or NULL. events: HOST array of n_frames + 1 cudaEvent_t, or NULL; events[i] is
 * recorded on cuda_stream before frame i's calls and events[n_frames] after the
 * last, so the caller can read each frame's device time.
 * Errors: INVALID (null or unaligned pointer, n_layers outside 1 .. layers,
 * n_frames < 0, ring < 1, frame0 < 0, tokens), STATE (a chunked-mode stream, or a
 * frame of this stream is pending); else the first failing call's status, with
 * the frame's index in pkv_last_error (the frames before it stay applied). */
pkv_status pkv_stream_frames_multi(pkv_t h, int stream_id, int n_layers, const void* const* q,
                                   const void* const* k, const void* const* v, int ring, int frame0,
                                   int n_frames, int tokens, const unsigned char* keyframe,
                                   void* const* out, float sm_scale, void* const* events,
                                   void* cuda_stream);

/* The model-shaped step over the cache, driven from native code: VGGT's aggregator
 * alternates each layer's frame attention (every frame's tokens over that frame's
 * own tokens) with its global attention (vLLM-Omni RFC "Reconstruction Engine",
 * sections 2.2 and 3.3); here the global attention is the cache's paged attention
 * ("LingBot-Map Paged KV Cache", sections 2-3). For frame i and layer l it makes
 * exactly these calls on cuda_stream:
 *   pkv_attend_frames(h, fq[l] + slot, fk[l] + slot, fv[l] + slot, 1, tokens,
 *                     fout[l] + slot, sm_scale)
 *   pkv_append_frame(h, stream_id, l, k[l] + slot, v[l] + slot, tokens)
 *   pkv_attend(h, q[l] + slot, tokens, stream_id, l, out[l] + slot, sm_scale)
 * then, per frame, pkv_evict_window (keyframe == NULL or keyframe[i]) or
 * pkv_rollback_last_frame, as pkv_stream_frames_multi. slot, the rings (fq, fk, fv,
 * fout, q, k, v, out: HOST arrays of n_layers device pointers to bf16
 * [ring][tokens][heads][64], each 16-byte aligned), keyframe and events are as in
 * pkv_stream_frames_multi. Errors: as pkv_stream_frames_multi, and INVALID for a
 * null or unaligned frame-attention pointer. */
pkv_status pkv_stream_model_frames(pkv_t h, int stream_id, int n_layers, const void* const* fq,
                                   const void* const* fk, const void* const* fv, void* const* fout,
                                   const void* const* q, const void* const* k, const void* const* v,
                                   void* const* out, int ring, int frame0, int n_frames, int tokens,
                                   const unsigned char* keyframe, float sm_scale, void* const* events,
                                   void* cuda_stream);

/* Write the visible page table (section 2, build_visible_page_table): page ids in
 * the order scale -> window (oldest first) -> special (allocation order); chunked
 * mode: chunks oldest first, pages in order.
 * d_idx, d_len: device int32[capacity] receiving page ids and valid slot counts;
 * d_n, d_last_page_len: device int32 scalars (may be NULL) receiving the entry
 * count and the last entry's length. Errors: INVALID if capacity is too small or a
 * buffer is null or not 4-byte aligned. */
pkv_status pkv_build_visible_page_table(pkv_t h, int stream_id, int32_t* d_idx, int32_t* d_len,
                                        int capacity, int32_t* d_n, int32_t* d_last_page_len,
                                        void* cuda_stream);

/* Frame-mode attention (sections 1-2): for every query row i < n_q and head h,
 * out[i][h] = softmax(sm_scale * q[i][h] . K^T) V over every valid slot of the
 * stream's visible pages (no mask besides page validity: bidirectional).
 * q, out: device bf16 [n_q][heads][64]; fp32 accumulation and softmax.
 * sm_scale <= 0 means 1/sqrt(head_dim). Errors: STATE if nothing is visible. */
pkv_status pkv_attend(pkv_t h, const void* q, int n_q, int stream_id, int layer, void* out,
                      float sm_scale, void* cuda_stream);

/* Chunked-mode attention (RFC 2.3 / 3.3): the current chunk's n_q tokens (n_q
 * must equal the tokens appended to the open chunk) attend over the visible
 * chunks. Same layouts and numerics as pkv_attend.
 * Errors: as pkv_attend; STATE for a frame-mode stream or no open chunk; INVALID
 * when n_q differs from the open chunk's tokens. */
pkv_status pkv_attend_chunked(pkv_t h, const void* q, int n_q, int stream_id, int layer,
                              void* out, float sm_scale, void* cuda_stream);

/* Frame-mode attention over a per-layer random subset of the visible pages.
 * vLLM-Omni RFC "Reconstruction Engine", section 5 (KV compression): AVGGT
 * samples a random KV subset per layer, different layers drawing different
 * subsets; FastVGGT keeps the initial frames as global anchors. Read at page
 * granularity on the visible table of "LingBot-Map Paged KV Cache", section 2:
 * the scale pages are always kept; the page at table position e (0-based, in
 * the order scale -> window -> special) is otherwise kept when the low 16 bits
 * of splitmix64(seed XOR (layer << 32) XOR e) are below keep, so each page is
 * kept with probability keep / 65536. splitmix64(x) is the first output of the
 * published generator seeded with x: z = x + 0x9E3779B97F4A7C15, then
 * z ^= z >> 30, z *= 0xBF58476D1CE4E5B9, z ^= z >> 27, z *= 0x94D049BB133111EB,
 * z ^= z >> 31. The attention is pkv_attend's over the kept pages' valid slots.
 * keep: 0 .. 65536 (65536 keeps every page). Errors: as pkv_attend; STATE for
 * a chunked-mode stream or an empty subset; INVALID for more than 1024 visible
 * pages. */
pkv_status pkv_attend_sampled(pkv_t h, const void* q, int n_q, int stream_id, int layer, void* out,
                              float sm_scale, unsigned long long seed, int keep,
                              void* cuda_stream);

/* Intra-frame attention: the tokens of every frame attend to that frame's own
 * tokens only, bidirectionally; no page, stream or table of the cache is read or
 * changed. vLLM-Omni RFC "Reconstruction Engine", section 2.2 (VGGT's aggregator
 * alternates frame self-attention with global self-attention in each of its 24
 * layers) and section 3.3 (the worker runs frame attention, per frame, before the
 * global attention over the in-window KV). For every frame f < n_frames, query
 * row i < tokens and head h:
 *   out[f][i][h] = softmax(sm_scale * q[f][i][h] . k[f][:][h]^T) v[f][:][h].
 * q, k, v, out: device bf16 [n_frames][tokens][heads][64], contiguous, each
 * 16-byte aligned (heads = the handle's); the caller owns them; out is written,
 * nothing else. fp32 accumulation and softmax, as pkv_attend; sm_scale <= 0
 * means 1/sqrt(head_dim). K and V are read by the Tensor Memory Accelerator
 * through tensor maps built by the driver's cuTensorMapEncodeTiled for each call.
 * n_frames = 0 is a no-op. Errors: INVALID for a null handle or pointer, an
 * unaligned pointer, tokens outside 1 .. 2^20, n_frames < 0, or n_frames x tokens
 * above 2^31 - 65; CUDA if the tensor maps cannot be built or the launch fails. */
pkv_status pkv_attend_frames(pkv_t h, const void* q, const void* k, const void* v, int n_frames,
                             int tokens, void* out, float sm_scale, void* cuda_stream);

/* Frame-mode attention over the visible pages with the highest estimated attention
 * mass. vLLM-Omni RFC "Reconstruction Engine", section 5 (KV compression):
 * Sparse-VGGT observes that global attention mass concentrates on a few blocks and
 * skips the low-weight ones; FastVGGT keeps the initial frames as anchors. Read at
 * page granularity on the visible table of "LingBot-Map Paged KV Cache", section 2:
 * the scale pages are always kept; every other visible page e gets the estimate
 *   score(e) = sum over h, d of qm[h][d] * km_e[h][d]
 * where qm is the mean over the call's n_q query rows and km_e the mean over page
 * e's valid slots of the layer's keys; the `keep` pages with the highest score are
 * kept (ties to the earlier table position; a NaN score ranks lowest). The score
 * decides which pages are kept, so it is computed in IEEE fp32 in a fixed order:
 * each mean a running sum in row (slot) order divided once, then one running sum
 * over h and d in that order of the rounded products (no fused multiply-add).
 * The attention is pkv_attend's over the kept pages' valid slots, in table order.
 * keep >= 0 (at least the number of non-anchor pages keeps them all). The
 * estimate, the selection and the attention all run on the device (no host
 * round trip, no allocation). A page's km depends only on its rows, so the handle
 * keeps it per layer and page, computed at the page's valid length: the append and
 * the windowed reset drop the cached value of every page they write, and a call
 * recomputes only pages whose cached length differs from their valid length (at
 * steady state the current frame's pages); cached and recomputed values are the
 * same bits. The handle's estimate scratch is shared by its calls: calls on one
 * handle must not overlap in time (on different CUDA streams).
 * Errors: as pkv_attend; STATE for a chunked-mode stream; INVALID for keep < 0,
 * more than 1024 visible pages, or an FP8 cache. */
pkv_status pkv_attend_blocksparse(pkv_t h, const void* q, int n_q, int stream_id, int layer,
                                  void* out, float sm_scale, int keep, void* cuda_stream);

/* The table positions kept by the last pkv_attend_blocksparse call on this handle,
 * in table order (a readback for tests and diagnostics). kept_out: HOST int array
 * of `capacity` entries; *n_out receives the count. Synchronizes the device.
 * Errors: INVALID (null pointer, capacity too small), STATE (no such call yet). */
pkv_status pkv_blocksparse_kept(pkv_t h, int* kept_out, int capacity, int* n_out);

/* Several streams' attention in one launch (the multi-stream pool of LingBot-Map
 * section 4; batching in the manner of the vLLM-Omni RFC's scheduler, section
 * 2.3). Equivalent to n calls of pkv_attend (frame-mode streams) or
 * pkv_attend_chunked (chunked-mode streams) on the same cuda_stream, each over
 * its own visible pages, with the same numerics; the split of the KV range into
 * parallel parts is chosen for the whole batch, so results may differ from the
 * separate calls by rounding.
 * q, out: device bf16 [q_off[n]][heads][64], the streams' query rows back to
 * back: rows q_off[i] .. q_off[i + 1] - 1 belong to stream sids[i].
 * q_off (n + 1 ints, q_off[0] = 0, increasing) and sids (n distinct open
 * streams) are host arrays; 1 <= n <= 32; every stream uses `layer`.
 * Errors: INVALID for bad arguments, STATE if a stream has nothing visible (or,
 * chunked, no open chunk); checked for every stream before anything is launched. */
pkv_status pkv_attend_batched(pkv_t h, const void* q, const int* q_off, const int* sids, int n,
                              int layer, void* out, float sm_scale, void* cuda_stream);

/* Attention that allocates nothing (no counterpart in the paper; it serves callers
 * of this library).
 * Same inputs, outputs, numerics and errors as pkv_attend (frame-mode streams) and
 * pkv_attend_chunked (chunked-mode streams, n_q = the open chunk's tokens), but the
 * split-KV partial results live in one fixed block of device memory compiled into
 * the library (a file-scope static __device__ array of 16 MiB), instead of the
 * scratch that pkv_attend grows with cudaMalloc the first time it needs more.
 * Some callers cannot allocate device memory at call time: code that runs while a
 * CUDA graph is being captured (an allocation would break the capture), real-time
 * frame loops that cannot afford the device-wide synchronisation cudaMalloc and
 * cudaFree imply, and hosts whose device memory belongs to another allocator. They
 * can create the handle and open the stream up front and then call this.
 *  - A call whose partial results need more than 16 MiB (num_splits x n_q x heads
 *    x 264 bytes; e.g. a whole 8 x 1374-token chunk over a window of 4 chunks,
 *    which runs in 3 KV splits) returns PKV_ERR_INVALID and launches nothing. The
 *    split count follows the call's shape (a call that runs unsplit needs none).
 *  - pkv_create_ex resolves the array's device address (cudaGetSymbolAddress,
 *    no allocation) for the device current at creation, which is the handle's
 *    device; a handle created after a device reset resolves it again. So the
 *    set-up happens once per handle, before any stream capture of its calls.
 *  - Every call, on every handle and stream, shares the one array, which keeps
 *    the last call's contents (nothing in it needs to start at zero: each call
 *    writes every partial it reads). Calls that overlap on the GPU race: order
 *    them on one CUDA stream. */
pkv_status pkv_attend_noalloc(pkv_t h, const void* q, int n_q, int stream_id, int layer, void* out,
                              float sm_scale, void* cuda_stream);

/* Wait for `cuda_stream` and report the device error word (PKV_ERR_DEVICE) or a
 * pending CUDA error (PKV_ERR_CUDA). */
pkv_status pkv_sync(pkv_t h, void* cuda_stream);

/* Host-side counts of the stream's visible table (no device access).
 * Errors: INVALID (the stream is not open, or a null pointer). */
pkv_status pkv_visible_count(pkv_t h, int stream_id, int* n_pages, int* n_tokens);

/* Number of free pages (host mirror of the free-stack depth). */
pkv_status pkv_free_pages(pkv_t h, int* n_free);

/* Debug / test export (synchronises the device). Writes int32 words to host_buf:
 *   [0] free-stack depth F, [1..F] free stack bottom to top,
 *   then the stream's visible table: n, idx[0..n), len[0..n),
 *   then mode-specific counters: frame mode {n_scale, n_window, n_special, sp_len,
 *   kept, pending}; chunked mode {n_chunks, open, pending, tokens of each chunk}.
 * cap_words is the capacity of host_buf; *used_words receives the count.
 * Errors: INVALID (stream not open, null pointer, cap_words too small), CUDA. */
pkv_status pkv_export_state(pkv_t h, int stream_id, int32_t* host_buf, size_t cap_words,
                            size_t* used_words);

/* Debug / test read of one page's K (kv = 0) or V (kv = 1) of one layer, copied to
 * host_dst as plain bf16 [heads][page_size][64] (un-swizzled). Synchronous.
 * Errors: INVALID (null pointer; layer, page or kv out of range; an FP8 cache), CUDA. */
pkv_status pkv_read_page(pkv_t h, int layer, int page, int kv, void* host_dst);

/* Debug / test read of one page's K (kv = 0) or V (kv = 1) of one layer of an FP8
 * cache (pkv_create_fp8), as stored: codes_dst receives uint8 [heads][page_size][64]
 * E4M3 codes, exps_dst int8 [heads][page_size] row exponents; both are HOST
 * buffers. Synchronous.
 * Errors: INVALID (null pointer; layer, page or kv out of range; a bf16 cache), CUDA. */
pkv_status pkv_read_page_fp8(pkv_t h, int layer, int page, int kv, void* codes_dst, void* exps_dst);

/* Synthetic input generator (not part of the cache): fills dst, a device bf16
 * array [n_frames][n_tokens][heads][head_dim], with the counter-based ~N(0,1)
 * values of frames frame0 .. frame0+n_frames-1: splitmix64 of the packed key
 * (seed, workload, stream, layer, frame, tensor, token0+t, head, d), four 16-bit
 * uniforms summed, centred, scaled by sqrt(3)*2^-16 in fp32, times `scale` (a
 * power of two), rounded to bf16.
 * Errors: INVALID (a field outside its key bits, a null or odd dst, a scale
 * that is not a power of two; the message is pkv_last_error(NULL)), CUDA. */
pkv_status pkv_synth_fill(void* dst, int n_frames, int n_tokens, int heads, int head_dim,
                          int seed, int workload, int stream, int layer, int frame0, int tensor,
                          int token0, float scale, void* cuda_stream);

/* Kernels this library has launched in the calling process so far (all handles). */
unsigned long long pkv_kernel_launches(void);

/* The handle's split-KV scratch: its current size in bytes and how many times it
 * has been (re)allocated. pkv_stream_open sizes it for the stream's natural query
 * count; a later attention call that needs more (another query count, or a
 * batched call) grows it, which synchronises the device and allocates.
 * Errors: INVALID (null argument). */
pkv_status pkv_scratch_info(pkv_t h, size_t* bytes, int* allocs);

/* Message of the last error on this handle ("" if none). h may be NULL for
 * errors of pkv_create. */
const char* pkv_last_error(pkv_t h);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
