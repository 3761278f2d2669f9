// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>                   // CUtensorMap (the type only; no driver call here)
#include <cuda_runtime.h>

#include <utility>
#include <stdint.h>

namespace pkv {

constexpr int kHeadDim = 64;        // bf16 elements per (slot, head) row: 128 bytes
constexpr int kTileSlots = 64;      // KV slots per tile of the attention kernel
constexpr int kChunksPerRow = 8;    // 16-byte chunks per row
constexpr int kMaxBatch = 32;       // streams per batched append
constexpr int kMaxChunks = 16;      // chunks visible at once (chunked mode)
constexpr int kMaxSegments = 20;    // page-id segments one push launch can return
constexpr int kMaxCarry = 64;       // overlap keyframes carried by a window reset

// Bits of the device error word.
enum : int {
  kErrPageRange = 1,   // a page id outside [0, pool_pages) was read from the metadata
  kErrTimeout = 2,     // a bounded wait gave up
};

// 128-byte-swizzled storage: logical 16-byte chunk c of slot s sits at c ^ (s & 7).
__host__ __device__ __forceinline__ int swizzle_chunk(int slot, int chunk) {
  return chunk ^ (slot & 7);
}

// One layer's page set. bf16 pages: pool[page][kv][head][slot][64] bf16, rows
// 128-byte swizzled. FP8 pages: per page and (kv, head) plane, row blocks of
// E4M3 codes (64-byte rows, unswizzled) each followed by its rows' exponent bytes
// (fp8_code_off, fp8_exp_off below): a row's values are decode(code) * 2^exponent.
struct PoolView {
  uint16_t* base;
  long long page_elems;   // bf16 pages: 2 * heads * page_size * 64
  int heads;
  int page_size;
  int pool_pages;
  int fp8;                // 1: E4M3 pages
  long long page_bytes;   // bytes per page (either format)
  int* km_len;            // bf16 pages: this layer's mean-key cache tags (per page), or null;
                          // a kernel that writes a page's rows sets its tag to -1
};

// ------------------------------------------------------------- FP8 rows
// vLLM-Omni RFC "Reconstruction Engine", section 3.4 (quantization: KV cache
// FP8). A row of 64 values is stored as OCP E4M3 codes of v * 2^-e with one
// exponent e per row: the smallest integer with amax <= 448 * 2^e (amax the
// row's largest magnitude; 0 for a zero row). With amax = f * 2^k, f in
// [0.5, 1), and 448 = 0.875 * 2^9, e = k - 9 + (f > 0.875). bf16 inputs give e
// in [-127, 120]; the exponent is clamped to [-126, 126], so that 2^e and 2^-e
// are normal fp32 values and v * 2^-e and code * 2^e are exact.
__device__ __forceinline__ int fp8_row_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  int k;
  const float f = frexpf(amax, &k);
  const int e = k - 9 + (f > 0.875f ? 1 : 0);
  return e < -126 ? -126 : (e > 126 ? 126 : e);
}

// Two floats to two E4M3 codes, round to nearest even (a in the low byte).
__device__ __forceinline__ uint32_t fp8_pack2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// FP8 page layout: for each (kv, head) plane of page_size rows, blocks of
// B = min(page_size, 64) rows, each the B rows' 64 code bytes followed by their B
// exponent bytes (B * 65 bytes, a multiple of 16), so that one bulk copy moves a
// block's codes and exponents together. B is 16, 32 or 64 (page sizes are
// multiples of 16 that divide or are divisible by 64).
__host__ __device__ __forceinline__ int fp8_block_rows(int page_size) {
  return page_size < 64 ? page_size : 64;
}
__host__ __device__ __forceinline__ long long fp8_block_off(int heads, int page_size, int kv,
                                                            int head, int slot) {
  const int B = fp8_block_rows(page_size);
  return (long long)(kv * heads + head) * page_size * (kHeadDim + 1) +
         (long long)(slot / B) * B * (kHeadDim + 1);
}
__host__ __device__ __forceinline__ long long fp8_code_off(int heads, int page_size, int kv, int head,
                                                           int slot) {
  return fp8_block_off(heads, page_size, kv, head, slot) +
         (long long)(slot % fp8_block_rows(page_size)) * kHeadDim;
}
__host__ __device__ __forceinline__ long long fp8_exp_off(int heads, int page_size, int kv, int head,
                                                          int slot) {
  const int B = fp8_block_rows(page_size);
  return fp8_block_off(heads, page_size, kv, head, slot) + (long long)B * kHeadDim + slot % B;
}

__device__ __forceinline__ uint8_t* fp8_row_codes(const PoolView& pv, int page, int kv, int head,
                                                  int slot) {
  return reinterpret_cast<uint8_t*>(pv.base) + (long long)page * pv.page_bytes +
         fp8_code_off(pv.heads, pv.page_size, kv, head, slot);
}
__device__ __forceinline__ int8_t* fp8_row_exp(const PoolView& pv, int page, int kv, int head,
                                               int slot) {
  return reinterpret_cast<int8_t*>(pv.base) + (long long)page * pv.page_bytes +
         fp8_exp_off(pv.heads, pv.page_size, kv, head, slot);
}

// Stores 16-byte chunk c (values 8c .. 8c + 7) of row (page, kv, head, slot).
// bf16 pages: at its swizzled place. FP8 pages: the eight lanes that hold a
// row's eight chunks (lanes 8g .. 8g + 7 of a warp, chunk = lane % 8) call this
// together; they share the row's largest magnitude and write their 8 codes, and
// chunk 0 writes the exponent.
__device__ __forceinline__ void store_row_chunk(const PoolView& pv, int page, int kv, int head,
                                                int slot, int c, const uint4& val) {
  if (!pv.fp8) {
    uint16_t* row = pv.base + (long long)page * pv.page_elems +
                    ((long long)(kv * pv.heads + head) * pv.page_size + slot) * kHeadDim;
    *reinterpret_cast<uint4*>(row + swizzle_chunk(slot, c) * 8) = val;
    return;
  }
  const uint32_t w[4] = {val.x, val.y, val.z, val.w};
  float f[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  const unsigned group = 0xFFu << (threadIdx.x & 24);
  amax = fmaxf(amax, __shfl_xor_sync(group, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(group, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(group, amax, 4));
  const int e = fp8_row_exponent(amax);
  const float inv = __uint_as_float((uint32_t)(127 - e) << 23);   // 2^-e
  const uint32_t lo = fp8_pack2(f[0] * inv, f[1] * inv) | (fp8_pack2(f[2] * inv, f[3] * inv) << 16);
  const uint32_t hi = fp8_pack2(f[4] * inv, f[5] * inv) | (fp8_pack2(f[6] * inv, f[7] * inv) << 16);
  *reinterpret_cast<uint2*>(fp8_row_codes(pv, page, kv, head, slot) + 8 * c) = make_uint2(lo, hi);
  if (c == 0) *fp8_row_exp(pv, page, kv, head, slot) = (int8_t)e;
}

// ------------------------------------------------------------------ append
struct AppendItem {                 // one frame-mode stream of a batched append
  const uint16_t* k;
  const uint16_t* v;
  int32_t* patch_slot;              // list entry that receives / holds the patch page id
  int32_t* special_list;            // the stream's special page list
  int sp_idx;                       // list index of the special page this frame writes
  int sp_off;                       // first special slot this frame writes
  int new_sp;                       // this frame opened special_list[sp_idx]
  int pad_;
};

struct FrameAppendArgs {
  PoolView pool;
  int n_patch;
  int n_special;
  int32_t* free_stack;
  int top;                          // free-stack depth before this batch's pops
  int is_meta;                      // pop pages and write the lists (first layer of the frame)
  int n;                            // streams in the batch
  int* err;
  AppendItem item[kMaxBatch];
};

struct ChunkAppendArgs {
  PoolView pool;
  const uint16_t* k;
  const uint16_t* v;
  int n_tokens;
  int32_t* free_stack;
  int top;
  int is_meta;
  int32_t* chunk_pages;             // the open chunk's page list
  int old_pages;                    // pages the chunk held before this append
  int n_new;                        // pages this append pops
  int pos0;                         // tokens the chunk held before this append
  int* err;
};

// ------------------------------------------------------------ push (free)
struct PushSegment {                // page ids src[(start + step*j) mod ring], j < count
  const int32_t* src;
  int start;
  int count;
  int step;                         // +1 or -1
  int ring;                         // 0: linear
};

struct PushArgs {
  int32_t* free_stack;
  int top;                          // depth before the pushes
  int n_seg;
  int pool_pages;
  int* err;
  PushSegment seg[kMaxSegments];
};

// ----------------------------------------------------------- window reset
struct ResetCopyArgs {              // copy carried frames' special tokens, all layers
  uint16_t* pool;                   // layer 0 base
  long long layer_elems;            // pool_pages * page_elems
  long long page_elems;
  int fp8;                          // E4M3 pages: rows are codes + an exponent byte
  long long layer_bytes, page_bytes;
  int layers, heads, page_size, pool_pages;
  int n_special, f_sp;
  const int32_t* special_list;      // old special list
  const int32_t* free_stack;
  int top;                          // depth after the eviction, before the reset's pops
  int n_carry;
  int src_sp_idx[kMaxCarry];        // special list index of carried frame i
  int src_sp_off[kMaxCarry];        // its first slot there
  int n_new;                        // special pages the reset pops
  int* km_len;                      // [layers][pool_pages] mean-key cache tags, or null
  int* err;
};

struct ResetMetaArgs {
  int32_t* free_stack;
  int top;                          // depth after the eviction, before the reset's pops
  int32_t* scale;                   // scale list
  int n_scale;
  int32_t* window;                  // window ring
  int win_head, win_count, win_cap;
  int32_t* special;
  int n_special_old;
  int n_carry;                      // the last n_carry held pages are carried
  int n_new;
  int pool_pages;
  int* err;
};

// ------------------------------------------------------------------ table
struct TableArgs {
  int mode;
  int n;                            // entries
  int page_size;
  int pool_pages;
  // frame mode
  const int32_t* scale;
  int n_scale;
  const int32_t* window;
  int win_head, win_count, win_cap;
  const int32_t* special;
  int n_special;
  int sp_full_len;
  int sp_last_len;
  // chunked mode (oldest chunk first)
  int n_chunks;
  const int32_t* chunk_pages[kMaxChunks];
  int chunk_npages[kMaxChunks];
  int chunk_len[kMaxChunks];
  // outputs
  int32_t* out_idx;
  int32_t* out_len;
  int32_t* out_n;                   // may be null
  int32_t* out_last;                // may be null
  int* err;
};

// Valid slots of entry e of a stream's visible table, from the table's counters
// alone (no device memory is read): patch pages are full; special pages hold
// sp_full_len slots, the last one sp_last_len; a chunk's pages are full but its last.
__host__ __device__ __forceinline__ int table_len(const TableArgs& t, int e) {
  if (t.mode == 0) {
    if (e < t.n_scale + t.win_count) return t.page_size;
    const int k = e - t.n_scale - t.win_count;
    return (k == t.n_special - 1) ? t.sp_last_len : t.sp_full_len;
  }
  int c = 0, base = 0;
  while (c < t.n_chunks - 1 && e >= base + t.chunk_npages[c]) {
    base += t.chunk_npages[c];
    ++c;
  }
  const int k = e - base;
  const int n = t.chunk_len[c] - k * t.page_size;
  return n < t.page_size ? n : t.page_size;
}

// Entry e of a stream's visible table (page id, valid slots): scale pages, window
// pages oldest first, special pages (frame mode); chunks oldest first (chunked).
__device__ __forceinline__ void table_entry(const TableArgs& t, int e, int& id, int& len) {
  if (t.mode == 0) {
    if (e < t.n_scale) {
      id = t.scale[e];
      len = t.page_size;
    } else if (e < t.n_scale + t.win_count) {
      id = t.window[(t.win_head + e - t.n_scale) % t.win_cap];
      len = t.page_size;
    } else {
      const int k = e - t.n_scale - t.win_count;
      id = t.special[k];
      len = (k == t.n_special - 1) ? t.sp_last_len : t.sp_full_len;
    }
  } else {
    int c = 0, base = 0;
    while (c < t.n_chunks - 1 && e >= base + t.chunk_npages[c]) {
      base += t.chunk_npages[c];
      ++c;
    }
    const int k = e - base;
    id = t.chunk_pages[c][k];
    len = min(t.page_size, t.chunk_len[c] - k * t.page_size);
  }
}

// ---------------------------------------------------------------- attend
struct AttendArgs {
  const uint16_t* q;                // [n_q][heads][64]
  uint16_t* out;                    // [n_q][heads][64] (written when num_splits == 1)
  int n_q;
  int heads;
  const uint16_t* pool;             // layer base
  long long page_elems;
  long long page_bytes;             // FP8 pages: bytes per page, and the exponents'
  int fp8;                          // 1: the pool holds E4M3 pages
  int page_size;
  int pool_pages;
  TableArgs tbl;                     // the visible table, computed on the fly by the producer
  // Per-layer random page subset (pkv_attend_sampled; sampled = 0 attends to
  // every visible page): the first sample_anchor table positions are kept, any
  // other position e when page_sample_kept(sample_key, e, sample_keep). Then
  // n_entries counts the kept pages and n_entries_all every visible one.
  int sampled;
  int sample_keep;
  int sample_anchor;
  int n_entries_all;
  unsigned long long sample_key;
  // A kept list computed on the device (pkv_attend_blocksparse): the first
  // n_entries table positions, in order; when set, it replaces the rule above.
  const uint16_t* kept_dev;
  int n_entries;
  int n_tiles;                      // 64-slot tiles covering the table's slots
  long long n_slots;                // flat slots up to the last valid one
  float scale_log2;                 // sm_scale * log2(e)
  int num_splits;
  float* part_o;                    // [split][n_q][heads][64]
  float* part_ml;                   // [split][n_q][heads][2]  (running max, sum), log2 domain
  int* err;
};

// Several attention calls in one launch (streams of one kernel shape). Item i
// owns CTAs cta_base[i] .. cta_base[i+1] - 1 of the attention kernel and
// (query row, head) pairs pair_base[i] .. pair_base[i+1] - 1 of the combine.
struct AttendBatch {
  int n;
  int cta_base[kMaxBatch + 1];
  long long pair_base[kMaxBatch + 1];
  int n_mgroups[kMaxBatch];
  int n_tiles[kMaxBatch];
  AttendArgs item[kMaxBatch];
};

// Intra-frame attention (pkv_attend_frames): n_frames independent problems,
// the tokens of frame f attending to frame f's own tokens. `a` holds the common
// fields: n_q = tokens per frame (the keys and values are the same tokens),
// num_splits = 1, no table. K and V are read through 3-D tensor maps over
// [n_frames * tokens][heads][64] bf16 whose box, 64 tokens x 1 head x 64
// elements with the 128-byte swizzle, lands as one tensor-core operand tile.
struct AttendDense {
  CUtensorMap k_map;
  CUtensorMap v_map;
  AttendArgs a;
};

// ------------------------------------------------------- page sampling
// vLLM-Omni RFC "Reconstruction Engine", section 5 (KV compression: AVGGT draws
// a random KV subset per layer): a non-anchor page at table position e is kept
// when the low 16 bits of splitmix64(key XOR e) are below keep (a fraction in
// 1/65536 units), key = seed XOR (layer << 32). splitmix64 as published by
// Steele, Lea and Flood (OOPSLA 2014): the state advances by the golden gamma,
// then is mixed.
constexpr int kMaxSampledEntries = 1024;   // visible pages a sampled call may hold
__host__ __device__ inline bool page_sample_kept(unsigned long long key, int e, int keep) {
  unsigned long long z = (key ^ (unsigned long long)e) + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  return (int)(z & 0xFFFFull) < keep;
}

// ------------------------------------------- page skipping by estimated mass
// vLLM-Omni RFC "Reconstruction Engine", section 5 (Sparse-VGGT skips the
// low-weight blocks; FastVGGT keeps anchors): each visible page of a frame-mode
// table gets an fp32 estimate (mean query . mean key, summed over heads, in a
// fixed order); the n_anchor scale pages and the `keep` best others are listed,
// in table order, in kept[].
constexpr int kMaxHeads = 32;
constexpr int kMaxPageSize = 256;
struct PageScoreArgs {
  const uint16_t* q;                // [n_q][heads][64]
  int n_q;
  int heads;
  PoolView pool;                    // the attended layer's page set
  TableArgs tbl;
  int n_entries;                    // visible pages (<= kMaxSampledEntries)
  int n_anchor;
  int keep;
  float* qm;                        // [heads][64] scratch
  float* scores;                    // [n_entries] scratch
  float* km;                        // this layer's mean-key cache: [pool_pages][heads][64]
  int* km_len;                      // its tags: the valid length km was computed at, or -1
  uint16_t* kept;                   // [n_anchor + keep] out
  unsigned* done;                   // score blocks finished (0 between calls)
  int* err;
};
cudaError_t launch_page_select(const PageScoreArgs& a, cudaStream_t s);

// Kernel launches made by this library in this process (every launcher counts).
// ---------------------------------------------------- dependent launches
// The frame path's kernels are launched with programmatic stream serialization:
// a kernel may start while the one before it on the stream finishes, does only
// CTA-private set-up (shared memory, TMEM, mbarriers) until pdl_wait(), and
// every thread of every CTA executes pdl_wait() before it touches global memory
// or exits. pdl_wait() returns once the previous kernel has completed and its
// writes are visible; since that kernel waited for its own predecessor before
// completing, the order of the whole stream is kept. pdl_trigger() lets the
// next kernel start launching early. Both are no-ops for a normal launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

unsigned long long launch_count();
void count_launches(int n);

// Launchers (each returns the launch's cudaError_t).
cudaError_t launch_frame_append(const FrameAppendArgs& a, cudaStream_t s);
cudaError_t launch_chunk_append(const ChunkAppendArgs& a, cudaStream_t s);
cudaError_t launch_push(const PushArgs& a, cudaStream_t s);
cudaError_t launch_reset_copy(const ResetCopyArgs& a, cudaStream_t s);
cudaError_t launch_reset_meta(const ResetMetaArgs& a, cudaStream_t s);
cudaError_t launch_table(const TableArgs& a, cudaStream_t s);
cudaError_t launch_attend(const AttendArgs& a, int num_sms, cudaStream_t s);
int attend_num_splits(int n_q, int heads, long long n_slots, int num_sms);
cudaError_t launch_attend_tc(const AttendArgs& a, cudaStream_t s);
// A batch whose items share one kernel shape (attend_tc_shape of their n_q),
// with the attention and, for splits > 1, the combine.
cudaError_t launch_attend_batch(const AttendBatch& b, cudaStream_t s);
cudaError_t launch_attend_tc_batch(const AttendBatch& b, cudaStream_t s);
int attend_tc_shape(int n_q);                  // kernel shape (M-tiles, extra rows): 0 .. 3
int attend_tc_mgroups(int n_q);
// Split-KV factor for `pairs` (M-group, head) pairs whose longest table has
// n_tiles tiles: fill the SMs in as few, as even waves as possible.
int attend_tc_splits_pairs(int pairs, int n_tiles, int num_sms);
int attend_tc_splits(int n_q, int heads, int n_tiles, int num_sms);
int attend_tc_tiles(long long n_slots);
// Intra-frame attention over n_frames frames (grid: M-groups x heads x frames).
cudaError_t launch_attend_dense(const AttendDense& d, int n_frames, cudaStream_t s);
cudaError_t launch_synth(uint16_t* dst, int n_frames, int n_tokens, int heads, int head_dim,
                         unsigned long long key_base, int frame0, int token0, float scale,
                         cudaStream_t s);

}  // namespace pkv
