// C-ABI entry points of libpkv: the handle, host-side counters and validation,
// and the launches. See include/pkv.h for each call's contract.
//
// Split of responsibilities: the device holds the page pool, the free stack's
// array and every stream's page-id lists; the host mirrors only counters (free
// stack depth, list lengths, ring heads, special fill, chunk lengths). All
// capacity and call-order checks run on the host before anything is launched,
// so an error return leaves the cache untouched, and every kernel gets the
// positions it reads and writes as arguments.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <memory>
#include <string>
#include <vector>

#include "../../include/pkv.h"
#include "pkv_internal.cuh"

using namespace pkv;

namespace {

struct Stream {
  bool open = false;
  pkv_stream_cfg cfg{};
  // device lists (one allocation)
  int32_t* d_mem = nullptr;
  int32_t* d_scale = nullptr;
  int32_t* d_window = nullptr;
  int32_t* d_special = nullptr;
  int32_t* d_chunks = nullptr;   // [sliding_window_num][ppc]
  int32_t* d_tbl_idx = nullptr;
  int32_t* d_tbl_len = nullptr;
  int tbl_cap = 0;
  // frame-mode counters
  int f_sp = 0;
  int n_scale = 0, win_head = 0, win_count = 0, n_special = 0, sp_len = 0, kept = 0;
  bool pending = false;
  bool u_to_scale = false, u_new_sp = false;
  int u_sp_before = 0, u_sp_off = 0, u_patch_pos = 0;
  // chunked-mode counters (by ring slot)
  int ppc = 0;
  int c_head = 0, n_chunks = 0;
  bool c_open = false;
  int c_len[kMaxChunks] = {0}, c_pages[kMaxChunks] = {0}, c_frames[kMaxChunks] = {0};
  int u_n_new = 0, u_old_pages = 0, u_pos0 = 0, u_slot = 0;
  bool u_new_chunk = false;
};

}  // namespace

struct pkv_ctx {
  int P = 0, Ps = 0, H = 0, D = 0, L = 0, max_streams = 0;
  long long page_elems = 0;      // bf16 elements per page (bf16 pools)
  int fp8 = 0;                   // 1: E4M3 pages with row exponents
  long long page_bytes = 0;      // bytes per page (either format)
  uint16_t* d_pool = nullptr;
  int32_t* d_free = nullptr;
  int* d_err = nullptr;
  int free_top = 0;
  std::vector<Stream> streams;
  float* d_scratch = nullptr;
  size_t scratch_bytes = 0;
  int scratch_allocs = 0;        // times the split-KV scratch was (re)allocated
  int device = 0;                // the device current at pkv_create_ex
  float* noalloc_scratch = nullptr;   // device address of the static scratch on `device`
  void* d_select = nullptr;      // page skipping: query means, page estimates, kept list
  float* d_km = nullptr;         // bf16 pages: mean key per (layer, page, head, d)
  int* d_km_len = nullptr;       // its tags per (layer, page): valid length, or -1
  int select_kept = -1;          // entries in that kept list (the last call's); -1: none yet
  int num_sms = 0;
  std::string last_error;
};

namespace {

std::string g_create_error;

constexpr size_t kStaticScratchBytes = size_t(16) << 20;   // 16 MiB
// The partial (o, m, l) results of pkv_attend_noalloc, shared by every call on
// every handle. In host code this name is only a stand-in for the symbol: kernels
// get the device address that pkv_create_ex resolves with cudaGetSymbolAddress.
static __device__ __align__(256) float g_noalloc_scratch[kStaticScratchBytes / sizeof(float)];

pkv_status fail(pkv_t h, pkv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (h) h->last_error = buf;
  else g_create_error = buf;
  return st;
}

pkv_status cuda_fail(pkv_t h, cudaError_t e, const char* what) {
  return fail(h, PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define PKV_CUDA(h, call)                                  \
  do {                                                     \
    cudaError_t e_ = (call);                               \
    if (e_ != cudaSuccess) return cuda_fail((h), e_, #call); \
  } while (0)

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Layer `layer`'s page set (a byte offset, so that it holds for either format).
inline uint16_t* layer_base(pkv_t h, int layer) {
  return reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(h->d_pool) +
                                     (long long)layer * h->P * h->page_bytes);
}

inline PoolView pool_view(pkv_t h, int layer) {
  PoolView pv;
  pv.base = layer_base(h, layer);
  pv.page_elems = h->page_elems;
  pv.heads = h->H;
  pv.page_size = h->Ps;
  pv.pool_pages = h->P;
  pv.fp8 = h->fp8;
  pv.page_bytes = h->page_bytes;
  pv.km_len = h->d_km_len ? h->d_km_len + (long long)layer * h->P : nullptr;
  return pv;
}

pkv_status get_stream(pkv_t h, int sid, Stream** out) {
  if (!h) return fail(h, PKV_ERR_INVALID, "null handle");
  if (sid < 0 || sid >= h->max_streams || !h->streams[sid].open)
    return fail(h, PKV_ERR_INVALID, "stream %d is not open", sid);
  *out = &h->streams[sid];
  return PKV_OK;
}

inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Visible table size from the counters.
void visible_counts(const pkv_ctx* h, const Stream& st, int* n_pages, int* n_tokens, int* last) {
  if (st.cfg.mode == PKV_MODE_FRAME) {
    const int np = st.n_scale + st.win_count + st.n_special;
    int nt = (st.n_scale + st.win_count) * h->Ps;
    if (st.n_special > 0) nt += (st.n_special - 1) * st.f_sp * st.cfg.n_special + st.sp_len;
    *n_pages = np;
    *n_tokens = nt;
    *last = st.n_special > 0 ? st.sp_len : (np > 0 ? h->Ps : 0);
  } else {
    int np = 0, nt = 0, lst = 0;
    for (int i = 0; i < st.n_chunks; ++i) {
      const int slot = (st.c_head + i) % st.cfg.sliding_window_num;
      np += st.c_pages[slot];
      nt += st.c_len[slot];
      lst = st.c_len[slot] - (st.c_pages[slot] - 1) * h->Ps;
    }
    *n_pages = np;
    *n_tokens = nt;
    *last = np > 0 ? lst : 0;
  }
}

TableArgs table_args(pkv_t h, Stream& st, int32_t* idx, int32_t* len, int32_t* out_n,
                     int32_t* out_last) {
  TableArgs t;
  std::memset(&t, 0, sizeof(t));
  int np, nt, last;
  visible_counts(h, st, &np, &nt, &last);
  t.mode = st.cfg.mode;
  t.n = np;
  t.page_size = h->Ps;
  t.pool_pages = h->P;
  if (st.cfg.mode == PKV_MODE_FRAME) {
    t.scale = st.d_scale;
    t.n_scale = st.n_scale;
    t.window = st.d_window;
    t.win_head = st.win_head;
    t.win_count = st.win_count;
    t.win_cap = st.cfg.window;
    t.special = st.d_special;
    t.n_special = st.n_special;
    t.sp_full_len = st.f_sp * st.cfg.n_special;
    t.sp_last_len = st.sp_len;
  } else {
    t.n_chunks = st.n_chunks;
    for (int i = 0; i < st.n_chunks; ++i) {
      const int slot = (st.c_head + i) % st.cfg.sliding_window_num;
      t.chunk_pages[i] = st.d_chunks + (long long)slot * st.ppc;
      t.chunk_npages[i] = st.c_pages[slot];
      t.chunk_len[i] = st.c_len[slot];
    }
  }
  t.out_idx = idx;
  t.out_len = len;
  t.out_n = out_n;
  t.out_last = out_last;
  t.err = h->d_err;
  return t;
}

pkv_status push_pages(pkv_t h, const PushSegment* segs, int n_seg, cudaStream_t s) {
  int total = 0;
  PushArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int i = 0; i < n_seg; ++i) {
    if (segs[i].count <= 0) continue;
    if (a.n_seg == kMaxSegments) return fail(h, PKV_ERR_INVALID, "too many page segments");
    a.seg[a.n_seg++] = segs[i];
    total += segs[i].count;
  }
  if (total == 0) return PKV_OK;
  if (h->free_top + total > h->P) return fail(h, PKV_ERR_STATE, "free stack overflow");
  a.free_stack = h->d_free;
  a.top = h->free_top;
  a.pool_pages = h->P;
  a.err = h->d_err;
  PKV_CUDA(h, launch_push(a, s));
  h->free_top += total;
  return PKV_OK;
}

PushSegment seg(const int32_t* src, int start, int count, int step = 1, int ring = 0) {
  PushSegment g;
  g.src = src;
  g.start = start;
  g.count = count;
  g.step = step;
  g.ring = ring;
  return g;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

unsigned long long pkv_kernel_launches(void) { return pkv::launch_count(); }

pkv_status pkv_scratch_info(pkv_t h, size_t* bytes, int* allocs) {
  if (!h || !bytes || !allocs) return fail(h, PKV_ERR_INVALID, "null argument");
  *bytes = h->scratch_bytes;
  *allocs = h->scratch_allocs;
  return PKV_OK;
}

const char* pkv_last_error(pkv_t h) { return h ? h->last_error.c_str() : g_create_error.c_str(); }

pkv_status pkv_create(int pool_pages, int page_size, int heads, int head_dim, pkv_t* out) {
  return pkv_create_ex(pool_pages, page_size, heads, head_dim, 1, 64, out);
}

}  // extern "C"

static pkv_status create_cache(int pool_pages, int page_size, int heads, int head_dim, int layers,
                               int max_streams, int fp8, pkv_t* out) {
  if (!out) return fail(nullptr, PKV_ERR_INVALID, "null output handle");
  *out = nullptr;
  if (head_dim != kHeadDim) return fail(nullptr, PKV_ERR_INVALID, "head_dim must be 64");
  if (page_size < 16 || page_size > 256 || page_size % 16 != 0 ||
      !(64 % page_size == 0 || page_size % 64 == 0))
    return fail(nullptr, PKV_ERR_INVALID,
                "page_size must be a multiple of 16 in [16, 256] dividing or divisible by 64");
  if (pool_pages < 1 || heads < 1 || heads > 32 || layers < 1 || max_streams < 1 ||
      max_streams > 1024)
    return fail(nullptr, PKV_ERR_INVALID, "bad pool/heads/layers/max_streams");
  pkv_t h = new pkv_ctx();
  h->P = pool_pages;
  h->Ps = page_size;
  h->H = heads;
  h->D = head_dim;
  h->L = layers;
  h->max_streams = max_streams;
  h->page_elems = 2LL * heads * page_size * head_dim;
  h->fp8 = fp8;
  // FP8 pages: 64 code bytes and one exponent byte per row; bf16 pages: 128 bytes per row
  h->page_bytes = fp8 ? 2LL * heads * page_size * (head_dim + 1) : 2LL * h->page_elems;
  h->streams.resize(max_streams);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  h->device = dev;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) {
    // the static scratch of pkv_attend_noalloc on this device (no allocation)
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    h->noalloc_scratch = static_cast<float*>(p);
  }
  const size_t pool_bytes = (size_t)layers * pool_pages * h->page_bytes;
  if (e == cudaSuccess) e = cudaMalloc(&h->d_pool, pool_bytes);
  if (e == cudaSuccess) e = cudaMemset(h->d_pool, 0, pool_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&h->d_free, sizeof(int32_t) * pool_pages);
  if (e == cudaSuccess) e = cudaMalloc(&h->d_err, sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(h->d_err, 0, sizeof(int));
  if (e == cudaSuccess) {
    // page skipping's scratch (query means, estimates, kept list)
    const size_t bytes = sizeof(float) * (kMaxHeads * kHeadDim + kMaxSampledEntries) +
                         sizeof(uint16_t) * kMaxSampledEntries + sizeof(unsigned);
    e = cudaMalloc(&h->d_select, bytes);
    if (e == cudaSuccess) e = cudaMemset(h->d_select, 0, bytes);
  }
  if (e == cudaSuccess && !fp8) {
    // the mean-key cache of page skipping (1 / page_size of the pool's bytes),
    // every tag -1 (nothing cached)
    e = cudaMalloc(&h->d_km, sizeof(float) * (size_t)layers * pool_pages * heads * head_dim);
    if (e == cudaSuccess) e = cudaMalloc(&h->d_km_len, sizeof(int) * (size_t)layers * pool_pages);
    if (e == cudaSuccess) e = cudaMemset(h->d_km_len, 0xFF, sizeof(int) * (size_t)layers * pool_pages);
  }
  if (e == cudaSuccess) {
    // free stack bottom..top = P-1 .. 0, so pops hand out 0, 1, 2, ...
    std::vector<int32_t> init(pool_pages);
    for (int i = 0; i < pool_pages; ++i) init[i] = pool_pages - 1 - i;
    e = cudaMemcpy(h->d_free, init.data(), sizeof(int32_t) * pool_pages, cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess) {
    std::string msg = std::string("pkv_create: ") + cudaGetErrorString(e);
    pkv_destroy(h);
    return fail(nullptr, e == cudaErrorMemoryAllocation ? PKV_ERR_OOM : PKV_ERR_CUDA, "%s",
                msg.c_str());
  }
  h->free_top = pool_pages;
  *out = h;
  return PKV_OK;
}

extern "C" {

pkv_status pkv_create_ex(int pool_pages, int page_size, int heads, int head_dim, int layers,
                         int max_streams, pkv_t* out) {
  return create_cache(pool_pages, page_size, heads, head_dim, layers, max_streams, 0, out);
}

pkv_status pkv_create_fp8(int pool_pages, int page_size, int heads, int head_dim, int layers,
                          int max_streams, pkv_t* out) {
  return create_cache(pool_pages, page_size, heads, head_dim, layers, max_streams, 1, out);
}

pkv_status pkv_destroy(pkv_t h) {
  if (!h) return PKV_OK;
  cudaDeviceSynchronize();
  for (auto& st : h->streams)
    if (st.d_mem) cudaFree(st.d_mem);
  if (h->d_pool) cudaFree(h->d_pool);
  if (h->d_free) cudaFree(h->d_free);
  if (h->d_err) cudaFree(h->d_err);
  if (h->d_scratch) cudaFree(h->d_scratch);
  if (h->d_select) cudaFree(h->d_select);
  if (h->d_km) cudaFree(h->d_km);
  if (h->d_km_len) cudaFree(h->d_km_len);
  delete h;
  return PKV_OK;
}

}  // extern "C"

namespace {

pkv_status ensure_scratch(pkv_t h, size_t bytes) {
  if (bytes <= h->scratch_bytes) return PKV_OK;
  PKV_CUDA(h, cudaDeviceSynchronize());
  if (h->d_scratch) cudaFree(h->d_scratch);
  h->d_scratch = nullptr;
  h->scratch_bytes = 0;
  PKV_CUDA(h, cudaMalloc(&h->d_scratch, bytes));
  h->scratch_bytes = bytes;
  h->scratch_allocs++;
  return PKV_OK;
}

// Split-KV scratch that the attention calls of a stream with this configuration
// need at their natural query count (a frame's n_patch + n_special rows, or a
// whole chunk), for the largest split count any reachable table size gives.
size_t stream_scratch_need(const pkv_ctx* h, const pkv_stream_cfg& c) {
  long long n_q = 0, max_slots = 0;
  if (c.mode == PKV_MODE_FRAME) {
    n_q = (long long)c.n_patch + c.n_special;
    max_slots = ((long long)c.num_scale + c.window + h->P) * h->Ps;
  } else {
    const long long chunk = (long long)c.chunk_size * c.tokens_per_frame;
    n_q = chunk;
    max_slots = (long long)c.sliding_window_num * ceil_div(chunk, h->Ps) * h->Ps;
  }
  if (n_q > (1 << 20)) return 0;
  const int max_tiles = attend_tc_tiles(max_slots);
  int max_splits = 1;
  for (int t = 1; t <= max_tiles; ++t)
    max_splits = std::max(max_splits, attend_tc_splits((int)n_q, h->H, t, h->num_sms));
  if (max_splits == 1) return 0;
  return (size_t)max_splits * n_q * h->H * (kHeadDim + 2) * sizeof(float);
}

}  // namespace

extern "C" {

pkv_status pkv_stream_open(pkv_t h, const pkv_stream_cfg* cfg, int* stream_id) {
  if (!h || !cfg || !stream_id) return fail(h, PKV_ERR_INVALID, "null argument");
  const pkv_stream_cfg c = *cfg;
  size_t words = 0;
  Stream st;
  st.cfg = c;
  if (c.mode == PKV_MODE_FRAME) {
    if (c.n_patch != h->Ps) return fail(h, PKV_ERR_INVALID, "n_patch must equal page_size");
    if (c.n_special < 1 || c.n_special > h->Ps)
      return fail(h, PKV_ERR_INVALID, "n_special must be in [1, page_size]");
    if (c.num_scale < 0 || c.window < 1)
      return fail(h, PKV_ERR_INVALID, "num_scale >= 0 and window >= 1 required");
    if (c.window_slots < 0) return fail(h, PKV_ERR_INVALID, "window_slots must be >= 0");
    if (c.window_slots > 0 &&
        !(c.overlap_keyframes >= 0 && c.overlap_keyframes <= c.num_scale &&
          c.overlap_keyframes < c.window_slots && c.overlap_keyframes <= kMaxCarry))
      return fail(h, PKV_ERR_INVALID, "overlap_keyframes must be <= num_scale and < window_slots");
    st.f_sp = h->Ps / c.n_special;
    st.tbl_cap = c.num_scale + c.window + h->P;
    words = (size_t)c.num_scale + c.window + h->P + 2 * (size_t)st.tbl_cap;
  } else if (c.mode == PKV_MODE_CHUNKED) {
    if (c.chunk_size < 1 || c.tokens_per_frame < 1 || c.sliding_window_num < 1 ||
        c.sliding_window_num > kMaxChunks)
      return fail(h, PKV_ERR_INVALID, "chunk_size, tokens_per_frame >= 1; sliding_window_num in [1,16]");
    if ((long long)c.chunk_size * c.tokens_per_frame > (1LL << 24))
      return fail(h, PKV_ERR_INVALID, "chunk too large");
    if (ceil_div(c.tokens_per_frame, h->Ps) + 1 > 256)
      return fail(h, PKV_ERR_INVALID, "a frame may not need more than 256 pages");
    st.ppc = ceil_div((long long)c.chunk_size * c.tokens_per_frame, h->Ps);
    st.tbl_cap = c.sliding_window_num * st.ppc;
    words = (size_t)st.tbl_cap + 2 * (size_t)st.tbl_cap;
  } else {
    return fail(h, PKV_ERR_INVALID, "unknown mode %d", c.mode);
  }
  int sid = -1;
  for (int i = 0; i < h->max_streams; ++i)
    if (!h->streams[i].open) {
      sid = i;
      break;
    }
  if (sid < 0) return fail(h, PKV_ERR_OOM, "no free stream id");
  if (pkv_status r = ensure_scratch(h, stream_scratch_need(h, c))) return r;
  cudaError_t e = cudaMalloc(&st.d_mem, words * sizeof(int32_t));
  if (e != cudaSuccess) return cuda_fail(h, e, "stream_open cudaMalloc");
  e = cudaMemset(st.d_mem, 0, words * sizeof(int32_t));
  if (e != cudaSuccess) {
    cudaFree(st.d_mem);
    return cuda_fail(h, e, "stream_open cudaMemset");
  }
  int32_t* p = st.d_mem;
  if (c.mode == PKV_MODE_FRAME) {
    st.d_scale = p;
    p += c.num_scale;
    st.d_window = p;
    p += c.window;
    st.d_special = p;
    p += h->P;
  } else {
    st.d_chunks = p;
    p += st.tbl_cap;
  }
  st.d_tbl_idx = p;
  p += st.tbl_cap;
  st.d_tbl_len = p;
  st.open = true;
  h->streams[sid] = st;
  *stream_id = sid;
  return PKV_OK;
}

static pkv_status free_stream_pages(pkv_t h, Stream* st, cudaStream_t s) {
  std::vector<PushSegment> segs;
  if (st->cfg.mode == PKV_MODE_FRAME) {
    segs.push_back(seg(st->d_scale, 0, st->n_scale));
    segs.push_back(seg(st->d_window, st->win_head, st->win_count, 1, st->cfg.window));
    segs.push_back(seg(st->d_special, 0, st->n_special));
  } else {
    for (int i = 0; i < st->n_chunks; ++i) {
      const int slot = (st->c_head + i) % st->cfg.sliding_window_num;
      segs.push_back(seg(st->d_chunks + (long long)slot * st->ppc, 0, st->c_pages[slot]));
    }
  }
  return push_pages(h, segs.data(), (int)segs.size(), s);
}

static void clear_counters(Stream* st) {
  Stream fresh;
  fresh.open = true;
  fresh.cfg = st->cfg;
  fresh.d_mem = st->d_mem;
  fresh.d_scale = st->d_scale;
  fresh.d_window = st->d_window;
  fresh.d_special = st->d_special;
  fresh.d_chunks = st->d_chunks;
  fresh.d_tbl_idx = st->d_tbl_idx;
  fresh.d_tbl_len = st->d_tbl_len;
  fresh.tbl_cap = st->tbl_cap;
  fresh.f_sp = st->f_sp;
  fresh.ppc = st->ppc;
  *st = fresh;
}

pkv_status pkv_stream_close(pkv_t h, int sid, void* cuda_stream) {
  Stream* st = nullptr;
  if (pkv_status r = get_stream(h, sid, &st)) return r;
  if (pkv_status r = free_stream_pages(h, st, as_stream(cuda_stream))) return r;
  // the list memory may still be read by the push just launched
  PKV_CUDA(h, cudaStreamSynchronize(as_stream(cuda_stream)));
  cudaFree(st->d_mem);
  *st = Stream();
  return PKV_OK;
}

pkv_status pkv_stream_reset(pkv_t h, int sid, void* cuda_stream) {
  Stream* st = nullptr;
  if (pkv_status r = get_stream(h, sid, &st)) return r;
  if (pkv_status r = free_stream_pages(h, st, as_stream(cuda_stream))) return r;
  clear_counters(st);
  return PKV_OK;
}

static pkv_status append_chunked(pkv_t h, Stream* st, int layer, const void* k, const void* v,
                                 int n_tokens, cudaStream_t s) {
  const int Wc = st->cfg.sliding_window_num;
  ChunkAppendArgs a;
  std::memset(&a, 0, sizeof(a));
  a.pool = pool_view(h, layer);
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.n_tokens = n_tokens;
  a.free_stack = h->d_free;
  a.err = h->d_err;
  if (layer == 0) {
    const bool new_chunk = !st->c_open;
    const int cur = (st->c_head + st->n_chunks - 1 + Wc) % Wc;
    if (new_chunk && st->n_chunks == Wc)
      return fail(h, PKV_ERR_STATE, "window holds sliding_window_num chunks: evict first");
    if (!new_chunk && st->c_frames[cur] == st->cfg.chunk_size)
      return fail(h, PKV_ERR_STATE, "chunk is full: evict before the next chunk");
    const int slot = new_chunk ? (st->c_head + st->n_chunks) % Wc : cur;
    const int len = new_chunk ? 0 : st->c_len[slot];
    const int have = new_chunk ? 0 : st->c_pages[slot];
    const int need = ceil_div(len + n_tokens, h->Ps) - have;
    if (need > h->free_top) return fail(h, PKV_ERR_OOM, "free list exhausted (%d pages needed, %d free)", need, h->free_top);
    a.top = h->free_top;
    a.is_meta = 1;
    a.chunk_pages = st->d_chunks + (long long)slot * st->ppc;
    a.old_pages = have;
    a.n_new = need;
    a.pos0 = len;
    PKV_CUDA(h, launch_chunk_append(a, s));
    h->free_top -= need;
    if (new_chunk) {
      st->n_chunks++;
      st->c_open = true;
      st->c_len[slot] = st->c_pages[slot] = st->c_frames[slot] = 0;
    }
    st->c_pages[slot] += need;
    st->c_len[slot] += n_tokens;
    st->c_frames[slot] += 1;
    st->pending = true;
    st->u_new_chunk = new_chunk;
    st->u_n_new = need;
    st->u_old_pages = have;
    st->u_pos0 = len;
    st->u_slot = slot;
  } else {
    if (!st->pending) return fail(h, PKV_ERR_STATE, "layer > 0 append without a pending frame");
    a.top = h->free_top;
    a.is_meta = 0;
    a.chunk_pages = st->d_chunks + (long long)st->u_slot * st->ppc;
    a.old_pages = st->u_old_pages;
    a.n_new = st->u_n_new;
    a.pos0 = st->u_pos0;
    PKV_CUDA(h, launch_chunk_append(a, s));
  }
  return PKV_OK;
}

// Plan one frame-mode layer-0 append: fills the batch item, returns pages needed.
static pkv_status plan_frame_append(pkv_t h, Stream* st, const void* k, const void* v,
                                    AppendItem* it, int* need) {
  const pkv_stream_cfg& c = st->cfg;
  if (st->pending)
    return fail(h, PKV_ERR_STATE,
                "a frame is pending: roll it back or commit it with pkv_evict_window first");
  const bool to_scale = st->n_scale < c.num_scale;
  if (!to_scale && st->win_count == c.window)
    return fail(h, PKV_ERR_STATE, "window is full: evict before appending");
  const bool new_sp = st->n_special == 0 || st->sp_len + c.n_special > st->f_sp * c.n_special;
  it->k = static_cast<const uint16_t*>(k);
  it->v = static_cast<const uint16_t*>(v);
  it->patch_slot = to_scale ? st->d_scale + st->n_scale
                            : st->d_window + (st->win_head + st->win_count) % c.window;
  it->special_list = st->d_special;
  it->sp_idx = new_sp ? st->n_special : st->n_special - 1;
  it->sp_off = new_sp ? 0 : st->sp_len;
  it->new_sp = new_sp ? 1 : 0;
  it->pad_ = 0;
  *need = 1 + (new_sp ? 1 : 0);
  return PKV_OK;
}

static void commit_frame_append(pkv_t h, Stream* st, const AppendItem& it) {
  const pkv_stream_cfg& c = st->cfg;
  const bool to_scale = st->n_scale < c.num_scale;
  st->u_to_scale = to_scale;
  st->u_new_sp = it.new_sp != 0;
  st->u_sp_before = st->sp_len;
  st->u_sp_off = it.sp_off;
  if (to_scale) {
    st->u_patch_pos = st->n_scale;
    st->n_scale++;
  } else {
    st->u_patch_pos = (st->win_head + st->win_count) % c.window;
    st->win_count++;
  }
  if (it.new_sp) {
    st->n_special++;
    st->sp_len = 0;
  }
  st->sp_len += c.n_special;
  st->kept++;
  st->pending = true;
  h->free_top -= 1 + it.new_sp;
}

static void pending_item(Stream* st, const void* k, const void* v, AppendItem* it) {
  it->k = static_cast<const uint16_t*>(k);
  it->v = static_cast<const uint16_t*>(v);
  it->patch_slot = (st->u_to_scale ? st->d_scale : st->d_window) + st->u_patch_pos;
  it->special_list = st->d_special;
  it->sp_idx = st->n_special - 1;
  it->sp_off = st->u_sp_off;
  it->new_sp = st->u_new_sp ? 1 : 0;
  it->pad_ = 0;
}

pkv_status pkv_append_frames(pkv_t h, int n, const int* sids, int layer, const void* const* k,
                             const void* const* v, int n_tokens, void* cuda_stream) {
  if (!h) return fail(h, PKV_ERR_INVALID, "null handle");
  if (n < 1 || n > kMaxBatch || !sids || !k || !v)
    return fail(h, PKV_ERR_INVALID, "batch of 1..32 streams with k and v arrays required");
  if (layer < 0 || layer >= h->L) return fail(h, PKV_ERR_INVALID, "layer %d out of range", layer);
  FrameAppendArgs a;
  std::memset(&a, 0, sizeof(a));
  a.pool = pool_view(h, layer);
  a.free_stack = h->d_free;
  a.top = h->free_top;
  a.is_meta = layer == 0 ? 1 : 0;
  a.n = n;
  a.err = h->d_err;
  int total_need = 0;
  Stream* sts[kMaxBatch];
  for (int i = 0; i < n; ++i) {
    Stream* st = nullptr;
    if (pkv_status r = get_stream(h, sids[i], &st)) return r;
    for (int j = 0; j < i; ++j)
      if (sids[j] == sids[i]) return fail(h, PKV_ERR_INVALID, "stream %d twice in one batch", sids[i]);
    if (st->cfg.mode != PKV_MODE_FRAME)
      return fail(h, PKV_ERR_STATE, "stream %d is not a frame-mode stream", sids[i]);
    if (n_tokens != st->cfg.n_patch + st->cfg.n_special)
      return fail(h, PKV_ERR_INVALID, "n_tokens %d != n_patch + n_special", n_tokens);
    if (!k[i] || !v[i] || !aligned16(k[i]) || !aligned16(v[i]))
      return fail(h, PKV_ERR_INVALID, "k/v must be 16-byte aligned device pointers");
    if (i > 0 && st->cfg.n_special != sts[0]->cfg.n_special)
      return fail(h, PKV_ERR_INVALID, "a batch must share n_special");
    sts[i] = st;
    if (layer == 0) {
      int need = 0;
      if (pkv_status r = plan_frame_append(h, st, k[i], v[i], &a.item[i], &need)) return r;
      total_need += need;
    } else {
      if (!st->pending) return fail(h, PKV_ERR_STATE, "layer > 0 append without a pending frame");
      pending_item(st, k[i], v[i], &a.item[i]);
    }
  }
  if (layer == 0 && total_need > h->free_top)
    return fail(h, PKV_ERR_OOM, "free list exhausted (%d pages needed, %d free)", total_need,
                h->free_top);
  a.n_patch = sts[0]->cfg.n_patch;
  a.n_special = sts[0]->cfg.n_special;
  PKV_CUDA(h, launch_frame_append(a, as_stream(cuda_stream)));
  if (layer == 0)
    for (int i = 0; i < n; ++i) commit_frame_append(h, sts[i], a.item[i]);
  return PKV_OK;
}

pkv_status pkv_append_frame(pkv_t h, int sid, int layer, const void* k, const void* v,
                            int n_tokens, void* cuda_stream) {
  Stream* st = nullptr;
  if (pkv_status r = get_stream(h, sid, &st)) return r;
  if (layer < 0 || layer >= h->L) return fail(h, PKV_ERR_INVALID, "layer %d out of range", layer);
  if (!k || !v || !aligned16(k) || !aligned16(v))
    return fail(h, PKV_ERR_INVALID, "k/v must be 16-byte aligned device pointers");
  if (st->cfg.mode == PKV_MODE_CHUNKED) {
    if (n_tokens != st->cfg.tokens_per_frame)
      return fail(h, PKV_ERR_INVALID, "n_tokens %d != tokens_per_frame", n_tokens);
    return append_chunked(h, st, layer, k, v, n_tokens, as_stream(cuda_stream));
  }
  const void* ks[1] = {k};
  const void* vs[1] = {v};
  return pkv_append_frames(h, 1, &sid, layer, ks, vs, n_tokens, cuda_stream);
}

pkv_status pkv_rollback_last_frame(pkv_t h, int sid, void* cuda_stream) {
  Stream* st = nullptr;
  if (pkv_status r = get_stream(h, sid, &st)) return r;
  if (!st->pending) return fail(h, PKV_ERR_STATE, "nothing to roll back");
  cudaStream_t s = as_stream(cuda_stream);
  if (st->cfg.mode == PKV_MODE_CHUNKED) {
    const int slot = st->u_slot;
    PushSegment g = seg(st->d_chunks + (long long)slot * st->ppc, st->u_old_pages + st->u_n_new - 1,
                        st->u_n_new, -1);
    if (pkv_status r = push_pages(h, &g, 1, s)) return r;
    st->c_pages[slot] -= st->u_n_new;
    st->c_len[slot] -= st->cfg.tokens_per_frame;
    st->c_frames[slot] -= 1;
    if (st->u_new_chunk) {
      st->n_chunks--;
      st->c_open = false;
    }
    st->pending = false;
    return PKV_OK;
  }
  // special page first (popped last), then the patch page: the LIFO inverse
  PushSegment segs[2];
  int ns = 0;
  if (st->u_new_sp) segs[ns++] = seg(st->d_special, st->n_special - 1, 1);
  segs[ns++] = seg(st->u_to_scale ? st->d_scale : st->d_window, st->u_patch_pos, 1);
  if (pkv_status r = push_pages(h, segs, ns, s)) return r;
  if (st->u_new_sp) st->n_special--;
  st->sp_len = st->u_sp_before;
  if (st->u_to_scale) st->n_scale--;
  else st->win_count--;
  st->kept--;
  st->pending = false;
  return PKV_OK;
}

static pkv_status window_reset(pkv_t h, Stream* st, cudaStream_t s) {
  const pkv_stream_cfg& c = st->cfg;
  const int n_held = st->n_scale + st->win_count;
  const int n_carry = std::min(c.overlap_keyframes, n_held);
  const int n_new = ceil_div(n_carry, st->f_sp);
  ResetCopyArgs ca;
  std::memset(&ca, 0, sizeof(ca));
  ca.pool = h->d_pool;
  ca.layer_elems = (long long)h->P * h->page_elems;
  ca.page_elems = h->page_elems;
  ca.fp8 = h->fp8;
  ca.layer_bytes = (long long)h->P * h->page_bytes;
  ca.page_bytes = h->page_bytes;
  ca.layers = h->L;
  ca.heads = h->H;
  ca.page_size = h->Ps;
  ca.pool_pages = h->P;
  ca.n_special = c.n_special;
  ca.f_sp = st->f_sp;
  ca.special_list = st->d_special;
  ca.free_stack = h->d_free;
  ca.top = h->free_top;
  ca.n_carry = n_carry;
  ca.n_new = n_new;
  ca.km_len = h->d_km_len;
  ca.err = h->d_err;
  for (int i = 0; i < n_carry; ++i) {
    const int j = n_held - n_carry + i;   // held position
    const int kept_idx = j < st->n_scale ? j : st->kept - st->win_count + (j - st->n_scale);
    ca.src_sp_idx[i] = kept_idx / st->f_sp;
    ca.src_sp_off[i] = (kept_idx % st->f_sp) * c.n_special;
  }
  PKV_CUDA(h, launch_reset_copy(ca, s));
  ResetMetaArgs ma;
  std::memset(&ma, 0, sizeof(ma));
  ma.free_stack = h->d_free;
  ma.top = h->free_top;
  ma.scale = st->d_scale;
  ma.n_scale = st->n_scale;
  ma.window = st->d_window;
  ma.win_head = st->win_head;
  ma.win_count = st->win_count;
  ma.win_cap = c.window;
  ma.special = st->d_special;
  ma.n_special_old = st->n_special;
  ma.n_carry = n_carry;
  ma.n_new = n_new;
  ma.pool_pages = h->P;
  ma.err = h->d_err;
  PKV_CUDA(h, launch_reset_meta(ma, s));
  h->free_top += -n_new + (n_held - n_carry) + st->n_special;
  st->n_scale = n_carry;
  st->win_head = 0;
  st->win_count = 0;
  st->n_special = n_new;
  st->sp_len = n_new ? (n_carry - (n_new - 1) * st->f_sp) * c.n_special : 0;
  st->kept = n_carry;
  return PKV_OK;
}

pkv_status pkv_evict_window(pkv_t h, int sid, void* cuda_stream) {
  Stream* st = nullptr;
  if (pkv_status r = get_stream(h, sid, &st)) return r;
  cudaStream_t s = as_stream(cuda_stream);
  const pkv_stream_cfg& c = st->cfg;
  if (c.mode == PKV_MODE_CHUNKED) {
    const int Wc = c.sliding_window_num;
    std::vector<PushSegment> segs;
    int n_drop = std::max(0, st->n_chunks - (Wc - 1));
    for (int i = 0; i < n_drop; ++i) {
      const int slot = (st->c_head + i) % Wc;
      segs.push_back(seg(st->d_chunks + (long long)slot * st->ppc, 0, st->c_pages[slot]));
    }
    if (pkv_status r = push_pages(h, segs.data(), (int)segs.size(), s)) return r;
    st->c_head = (st->c_head + n_drop) % Wc;
    st->n_chunks -= n_drop;
    st->c_open = false;
    st->pending = false;
    return PKV_OK;
  }
  const int n_evict = std::max(0, st->win_count - (c.window - 1));
  const bool reset = c.window_slots > 0 && st->kept >= c.window_slots;
  if (reset) {
    const int held = st->n_scale + st->win_count - n_evict;
    const int n_new = ceil_div(std::min(c.overlap_keyframes, held), st->f_sp);
    if (h->free_top + n_evict < n_new)
      return fail(h, PKV_ERR_OOM, "free list exhausted by the window reset");
    if (st->n_scale + st->win_count + st->n_special + n_new > 12 * 1024)
      return fail(h, PKV_ERR_INVALID, "stream too large for a window reset");
  }
  if (n_evict > 0) {
    PushSegment g = seg(st->d_window, st->win_head, n_evict, 1, c.window);
    if (pkv_status r = push_pages(h, &g, 1, s)) return r;
    st->win_head = (st->win_head + n_evict) % c.window;
    st->win_count -= n_evict;
  }
  st->pending = false;
  if (reset) return window_reset(h, st, s);
  return PKV_OK;
}

pkv_status pkv_build_visible_page_table(pkv_t h, int sid, int32_t* d_idx, int32_t* d_len,
                                        int capacity, int32_t* d_n, int32_t* d_last_page_len,
                                        void* cuda_stream) {
  Stream* st = nullptr;
  if (pkv_status r = get_stream(h, sid, &st)) return r;
  int np, nt, last;
  visible_counts(h, *st, &np, &nt, &last);
  if (np > 0 && (!d_idx || !d_len)) return fail(h, PKV_ERR_INVALID, "null table buffers");
  const auto misaligned4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) != 0; };
  if (misaligned4(d_idx) || misaligned4(d_len) || misaligned4(d_n) || misaligned4(d_last_page_len))
    return fail(h, PKV_ERR_INVALID, "table buffers must be 4-byte aligned");
  if (capacity < np) return fail(h, PKV_ERR_INVALID, "capacity %d < %d entries", capacity, np);
  TableArgs t = table_args(h, *st, d_idx, d_len, d_n, d_last_page_len);
  PKV_CUDA(h, launch_table(t, as_stream(cuda_stream)));
  return PKV_OK;
}

// The attention arguments of one call on one stream, split count and scratch
// aside.
static pkv_status attend_args(pkv_t h, Stream* st, const void* q, int n_q, int layer, void* out,
                              float sm_scale, AttendArgs* a) {
  if (!q || !out || !aligned16(q) || !aligned16(out))
    return fail(h, PKV_ERR_INVALID, "q/out must be 16-byte aligned device pointers");
  if (n_q < 1 || n_q > (1 << 20)) return fail(h, PKV_ERR_INVALID, "n_q %d out of range", n_q);
  if (layer < 0 || layer >= h->L) return fail(h, PKV_ERR_INVALID, "layer %d out of range", layer);
  int np, nt, last;
  visible_counts(h, *st, &np, &nt, &last);
  if (nt == 0) return fail(h, PKV_ERR_STATE, "nothing is visible");
  std::memset(a, 0, sizeof(*a));
  a->q = static_cast<const uint16_t*>(q);
  a->out = static_cast<uint16_t*>(out);
  a->n_q = n_q;
  a->heads = h->H;
  a->pool = layer_base(h, layer);
  a->page_elems = h->page_elems;
  a->page_bytes = h->page_bytes;
  a->fp8 = h->fp8;
  a->page_size = h->Ps;
  a->pool_pages = h->P;
  a->tbl = table_args(h, *st, st->d_tbl_idx, st->d_tbl_len, nullptr, nullptr);
  a->n_entries = np;
  a->n_slots = (long long)(np - 1) * h->Ps + last;
  a->n_tiles = attend_tc_tiles(a->n_slots);
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt((float)h->D);
  a->scale_log2 = scale * 1.4426950408889634f;
  a->num_splits = 1;
  a->err = h->d_err;
  return PKV_OK;
}

static size_t partial_bytes(const AttendArgs& a) {
  return (size_t)a.num_splits * a.n_q * a.heads * (kHeadDim + 2) * sizeof(float);
}

// The same rounded up to 256 bytes: the partials of several calls placed back to
// back each start 16-byte aligned (the kernels move O partials in 16-byte vectors,
// and splits x n_q x heads x 264 bytes is only a multiple of 8 when all three are odd).
static size_t partial_bytes_aligned(const AttendArgs& a) {
  return (partial_bytes(a) + 255) & ~static_cast<size_t>(255);
}

// Split-KV partials of `a` at `base`: O first, then the (max, sum) pairs.
static void place_partials(AttendArgs* a, float* base) {
  a->part_o = base;
  a->part_ml = base + (size_t)a->num_splits * a->n_q * a->heads * kHeadDim;
}

static pkv_status attend_common(pkv_t h, Stream* st, const void* q, int n_q, int layer, void* out,
                                float sm_scale, cudaStream_t s) {
  AttendArgs a;
  if (pkv_status r = attend_args(h, st, q, n_q, layer, out, sm_scale, &a)) return r;
  a.num_splits = attend_num_splits(n_q, h->H, a.n_slots, h->num_sms);
  if (a.num_splits > 1) {
    if (pkv_status r = ensure_scratch(h, partial_bytes(a))) return r;
    place_partials(&a, h->d_scratch);
  }
  PKV_CUDA(h, launch_attend(a, h->num_sms, s));
  return PKV_OK;
}

pkv_status pkv_attend(pkv_t h, const void* q, int n_q, int sid, int layer, void* out,
                      float sm_scale, void* cuda_stream) {
  Stream* st = nullptr;
  if (pkv_status r = get_stream(h, sid, &st)) return r;
  if (st->cfg.mode != PKV_MODE_FRAME)
    return fail(h, PKV_ERR_STATE, "pkv_attend needs a frame-mode stream (use pkv_attend_chunked)");
  return attend_common(h, st, q, n_q, layer, out, sm_scale, as_stream(cuda_stream));
}

pkv_status pkv_stream_frames(pkv_t h, int sid, int layer, const void* q, const void* k,
                             const void* v, int n_frames, int tokens,
                             const unsigned char* keyframe, void* out, float sm_scale,
                             void* cuda_stream) {
  Stream* st = nullptr;
  if (pkv_status r = get_stream(h, sid, &st)) return r;
  if (st->cfg.mode != PKV_MODE_FRAME)
    return fail(h, PKV_ERR_STATE, "pkv_stream_frames needs a frame-mode stream");
  if (st->pending) return fail(h, PKV_ERR_STATE, "a frame of stream %d is pending", sid);
  if (n_frames < 0) return fail(h, PKV_ERR_INVALID, "n_frames %d < 0", n_frames);
  if (layer < 0 || layer >= h->L) return fail(h, PKV_ERR_INVALID, "layer %d out of range", layer);
  if (tokens != st->cfg.n_patch + st->cfg.n_special)
    return fail(h, PKV_ERR_INVALID, "tokens %d != n_patch + n_special", tokens);
  if (n_frames == 0) return PKV_OK;
  if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(h, PKV_ERR_INVALID, "q/k/v/out must be 16-byte aligned device pointers");
  const size_t fb = (size_t)tokens * h->H * kHeadDim * sizeof(uint16_t);   // bytes per frame
  const char* qb = static_cast<const char*>(q);
  const char* kb = static_cast<const char*>(k);
  const char* vb = static_cast<const char*>(v);
  char* ob = static_cast<char*>(out);
  for (int t = 0; t < n_frames; ++t) {
    const size_t o = fb * (size_t)t;
    pkv_status r = pkv_append_frame(h, sid, layer, kb + o, vb + o, tokens, cuda_stream);
    if (r == PKV_OK) r = pkv_attend(h, qb + o, tokens, sid, layer, ob + o, sm_scale, cuda_stream);
    if (r == PKV_OK)
      r = (keyframe == nullptr || keyframe[t]) ? pkv_evict_window(h, sid, cuda_stream)
                                               : pkv_rollback_last_frame(h, sid, cuda_stream);
    if (r != PKV_OK) {
      h->last_error = "frame " + std::to_string(t) + ": " + h->last_error;
      return r;
    }
  }
  return PKV_OK;
}

// The native frame runner of pkv_stream_frames_multi and pkv_stream_model_frames:
// per frame and layer, the frame's intra-frame attention (when fq is given), then
// the layer's append and global attention; then the frame's evict or rollback.
static pkv_status run_frames(pkv_t h, const char* fn, int sid, int n_layers, const void* const* q,
                             const void* const* k, const void* const* v, const void* const* fq,
                             const void* const* fk, const void* const* fv, void* const* fout,
                             int ring, int frame0, int n_frames, int tokens,
                             const unsigned char* keyframe, void* const* out, float sm_scale,
                             void* const* events, void* cuda_stream) {
  Stream* st = nullptr;
  if (pkv_status r = get_stream(h, sid, &st)) return r;
  if (st->cfg.mode != PKV_MODE_FRAME)
    return fail(h, PKV_ERR_STATE, "%s needs a frame-mode stream", fn);
  if (st->pending) return fail(h, PKV_ERR_STATE, "a frame of stream %d is pending", sid);
  if (n_layers < 1 || n_layers > h->L)
    return fail(h, PKV_ERR_INVALID, "n_layers %d outside 1..%d", n_layers, h->L);
  if (n_frames < 0 || ring < 1 || frame0 < 0)
    return fail(h, PKV_ERR_INVALID, "n_frames %d, ring %d, frame0 %d", n_frames, ring, frame0);
  if (tokens != st->cfg.n_patch + st->cfg.n_special)
    return fail(h, PKV_ERR_INVALID, "tokens %d != n_patch + n_special", tokens);
  if (n_frames == 0) return PKV_OK;
  if (!q || !k || !v || !out) return fail(h, PKV_ERR_INVALID, "null pointer array");
  const bool frame_attn = fq != nullptr;
  if (frame_attn && (!fk || !fv || !fout)) return fail(h, PKV_ERR_INVALID, "null pointer array");
  for (int l = 0; l < n_layers; ++l) {
    if (!q[l] || !k[l] || !v[l] || !out[l] || !aligned16(q[l]) || !aligned16(k[l]) ||
        !aligned16(v[l]) || !aligned16(out[l]))
      return fail(h, PKV_ERR_INVALID, "layer %d: q/k/v/out must be 16-byte aligned device pointers", l);
    if (frame_attn && (!fq[l] || !fk[l] || !fv[l] || !fout[l] || !aligned16(fq[l]) ||
                       !aligned16(fk[l]) || !aligned16(fv[l]) || !aligned16(fout[l])))
      return fail(h, PKV_ERR_INVALID,
                  "layer %d: frame-attention q/k/v/out must be 16-byte aligned device pointers", l);
  }
  cudaStream_t s = as_stream(cuda_stream);
  const size_t fb = (size_t)tokens * h->H * kHeadDim * sizeof(uint16_t);   // bytes per frame
  for (int i = 0; i < n_frames; ++i) {
    if (events && events[i]) PKV_CUDA(h, cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s));
    const size_t o = fb * (size_t)((frame0 + i) % ring);
    pkv_status r = PKV_OK;
    for (int l = 0; l < n_layers && r == PKV_OK; ++l) {
      if (frame_attn)
        r = pkv_attend_frames(h, static_cast<const char*>(fq[l]) + o, static_cast<const char*>(fk[l]) + o,
                              static_cast<const char*>(fv[l]) + o, 1, tokens,
                              static_cast<char*>(fout[l]) + o, sm_scale, cuda_stream);
      if (r == PKV_OK)
        r = pkv_append_frame(h, sid, l, static_cast<const char*>(k[l]) + o,
                             static_cast<const char*>(v[l]) + o, tokens, cuda_stream);
      if (r == PKV_OK)
        r = pkv_attend(h, static_cast<const char*>(q[l]) + o, tokens, sid, l,
                       static_cast<char*>(out[l]) + o, sm_scale, cuda_stream);
    }
    if (r == PKV_OK)
      r = (keyframe == nullptr || keyframe[i]) ? pkv_evict_window(h, sid, cuda_stream)
                                               : pkv_rollback_last_frame(h, sid, cuda_stream);
    if (r != PKV_OK) {
      h->last_error = "frame " + std::to_string(frame0 + i) + ": " + h->last_error;
      return r;
    }
  }
  if (events && events[n_frames])
    PKV_CUDA(h, cudaEventRecord(static_cast<cudaEvent_t>(events[n_frames]), s));
  return PKV_OK;
}

pkv_status pkv_stream_frames_multi(pkv_t h, int sid, int n_layers, const void* const* q,
                                   const void* const* k, const void* const* v, int ring, int frame0,
                                   int n_frames, int tokens, const unsigned char* keyframe,
                                   void* const* out, float sm_scale, void* const* events,
                                   void* cuda_stream) {
  return run_frames(h, "pkv_stream_frames_multi", sid, n_layers, q, k, v, nullptr, nullptr, nullptr,
                    nullptr, ring, frame0, n_frames, tokens, keyframe, out, sm_scale, events,
                    cuda_stream);
}

pkv_status pkv_stream_model_frames(pkv_t h, int sid, int n_layers, const void* const* fq,
                                   const void* const* fk, const void* const* fv, void* const* fout,
                                   const void* const* q, const void* const* k, const void* const* v,
                                   void* const* out, int ring, int frame0, int n_frames, int tokens,
                                   const unsigned char* keyframe, float sm_scale, void* const* events,
                                   void* cuda_stream) {
  if (!fq || !fk || !fv || !fout) return fail(h, PKV_ERR_INVALID, "null pointer array");
  return run_frames(h, "pkv_stream_model_frames", sid, n_layers, q, k, v, fq, fk, fv, fout, ring,
                    frame0, n_frames, tokens, keyframe, out, sm_scale, events, cuda_stream);
}

pkv_status pkv_attend_chunked(pkv_t h, const void* q, int n_q, int sid, int layer, void* out,
                              float sm_scale, void* cuda_stream) {
  Stream* st = nullptr;
  if (pkv_status r = get_stream(h, sid, &st)) return r;
  if (st->cfg.mode != PKV_MODE_CHUNKED)
    return fail(h, PKV_ERR_STATE, "pkv_attend_chunked needs a chunked-mode stream");
  if (!st->c_open) return fail(h, PKV_ERR_STATE, "no open chunk");
  const int cur = (st->c_head + st->n_chunks - 1) % st->cfg.sliding_window_num;
  if (n_q != st->c_len[cur])
    return fail(h, PKV_ERR_INVALID, "n_q %d != the open chunk's %d tokens", n_q, st->c_len[cur]);
  return attend_common(h, st, q, n_q, layer, out, sm_scale, as_stream(cuda_stream));
}

pkv_status pkv_attend_sampled(pkv_t h, const void* q, int n_q, int sid, int layer, void* out,
                              float sm_scale, unsigned long long seed, int keep, void* cuda_stream) {
  Stream* st = nullptr;
  if (pkv_status r = get_stream(h, sid, &st)) return r;
  if (st->cfg.mode != PKV_MODE_FRAME)
    return fail(h, PKV_ERR_STATE, "pkv_attend_sampled needs a frame-mode stream");
  if (keep < 0 || keep > 65536) return fail(h, PKV_ERR_INVALID, "keep %d outside 0..65536", keep);
  AttendArgs a;
  if (pkv_status r = attend_args(h, st, q, n_q, layer, out, sm_scale, &a)) return r;
  const int np = a.n_entries;
  if (np > kMaxSampledEntries)
    return fail(h, PKV_ERR_INVALID, "%d visible pages; a sampled call takes at most %d", np,
                kMaxSampledEntries);
  // the same decisions the kernel's producer makes, to size the grid: the
  // kept pages and the length of the last one
  const TableArgs& t = a.tbl;
  const unsigned long long key = seed ^ ((unsigned long long)layer << 32);
  int n_kept = 0, last_len = 0;
  for (int e = 0; e < np; ++e) {
    if (e >= t.n_scale && !page_sample_kept(key, e, keep)) continue;
    ++n_kept;
    const int k = e - t.n_scale - t.win_count;          // special page index, if >= 0
    last_len = k < 0 ? h->Ps : (k == t.n_special - 1 ? t.sp_last_len : t.sp_full_len);
  }
  if (n_kept == 0) return fail(h, PKV_ERR_STATE, "the sampled subset of the visible pages is empty");
  a.sampled = 1;
  a.sample_keep = keep;
  a.sample_anchor = t.n_scale;
  a.sample_key = key;
  a.n_entries_all = np;
  a.n_entries = n_kept;
  a.n_slots = (long long)(n_kept - 1) * h->Ps + last_len;
  a.n_tiles = attend_tc_tiles(a.n_slots);
  a.num_splits = attend_num_splits(n_q, h->H, a.n_slots, h->num_sms);
  if (a.num_splits > 1) {
    if (pkv_status r = ensure_scratch(h, partial_bytes(a))) return r;
    place_partials(&a, h->d_scratch);
  }
  PKV_CUDA(h, launch_attend(a, h->num_sms, as_stream(cuda_stream)));
  return PKV_OK;
}

pkv_status pkv_attend_blocksparse(pkv_t h, const void* q, int n_q, int sid, int layer, void* out,
                                  float sm_scale, int keep, void* cuda_stream) {
  Stream* st = nullptr;
  if (pkv_status r = get_stream(h, sid, &st)) return r;
  if (st->cfg.mode != PKV_MODE_FRAME)
    return fail(h, PKV_ERR_STATE, "pkv_attend_blocksparse needs a frame-mode stream");
  if (keep < 0) return fail(h, PKV_ERR_INVALID, "keep %d < 0", keep);
  if (h->fp8) return fail(h, PKV_ERR_INVALID, "page skipping by mass reads bf16 pages; this cache holds FP8 pages");
  AttendArgs a;
  if (pkv_status r = attend_args(h, st, q, n_q, layer, out, sm_scale, &a)) return r;
  const int np = a.n_entries;
  if (np > kMaxSampledEntries)
    return fail(h, PKV_ERR_INVALID, "%d visible pages; this call takes at most %d", np,
                kMaxSampledEntries);
  float* qm = static_cast<float*>(h->d_select);
  float* scores = qm + kMaxHeads * kHeadDim;
  uint16_t* kept = reinterpret_cast<uint16_t*>(scores + kMaxSampledEntries);
  unsigned* done = reinterpret_cast<unsigned*>(kept + kMaxSampledEntries);   // 4-byte aligned
  const int n_anchor = a.tbl.n_scale;
  const int n_kept = n_anchor + std::min(keep, np - n_anchor);
  PageScoreArgs g;
  std::memset(&g, 0, sizeof(g));
  g.q = static_cast<const uint16_t*>(q);
  g.n_q = n_q;
  g.heads = h->H;
  g.pool = pool_view(h, layer);
  g.tbl = a.tbl;
  g.n_entries = np;
  g.n_anchor = n_anchor;
  g.keep = keep;
  g.qm = qm;
  g.scores = scores;
  g.km = h->d_km + (long long)layer * h->P * h->H * kHeadDim;
  g.km_len = h->d_km_len + (long long)layer * h->P;
  g.kept = kept;
  g.done = done;
  g.err = h->d_err;
  cudaStream_t s = as_stream(cuda_stream);
  PKV_CUDA(h, launch_page_select(g, s));
  h->select_kept = n_kept;
  // which pages are kept is known on the device only: unless every page is kept
  // (then the exact slot count of pkv_attend), the grid covers n_kept full pages,
  // and the slots past each kept page's length are masked
  a.sampled = 1;
  a.kept_dev = kept;
  a.n_entries_all = np;
  if (n_kept < np) a.n_slots = (long long)n_kept * h->Ps;
  a.n_entries = n_kept;
  a.n_tiles = attend_tc_tiles(a.n_slots);
  a.num_splits = attend_num_splits(n_q, h->H, a.n_slots, h->num_sms);
  if (a.num_splits > 1) {
    if (pkv_status r = ensure_scratch(h, partial_bytes(a))) return r;
    place_partials(&a, h->d_scratch);
  }
  PKV_CUDA(h, launch_attend(a, h->num_sms, s));
  return PKV_OK;
}

pkv_status pkv_blocksparse_kept(pkv_t h, int* kept_out, int capacity, int* n_out) {
  if (!h || !kept_out || !n_out) return fail(h, PKV_ERR_INVALID, "null argument");
  if (h->select_kept < 0) return fail(h, PKV_ERR_STATE, "no pkv_attend_blocksparse call yet");
  if (capacity < h->select_kept)
    return fail(h, PKV_ERR_INVALID, "capacity %d < %d entries", capacity, h->select_kept);
  std::vector<uint16_t> tmp(h->select_kept);
  const uint16_t* kept = reinterpret_cast<const uint16_t*>(
      static_cast<const float*>(h->d_select) + kMaxHeads * kHeadDim + kMaxSampledEntries);
  PKV_CUDA(h, cudaDeviceSynchronize());
  PKV_CUDA(h, cudaMemcpy(tmp.data(), kept, sizeof(uint16_t) * tmp.size(), cudaMemcpyDeviceToHost));
  for (size_t i = 0; i < tmp.size(); ++i) kept_out[i] = tmp[i];
  *n_out = h->select_kept;
  return PKV_OK;
}

// cuTensorMapEncodeTiled, looked up once through the runtime (the library
// does not link the driver library itself).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Tensor map over a dense [rows][heads][64] bf16 tensor: box of kTileSlots rows x 1
// head x 64 elements, 128-byte swizzle (the tensor-core operand layout), zero
// fill past the last row.
static bool encode_kv_map(CUtensorMap* m, const void* base, int heads, long long rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)heads * kHeadDim * 2};
  const cuuint32_t box[3] = {(cuuint32_t)kHeadDim, 1u, (cuuint32_t)kTileSlots};
  const cuuint32_t elem[3] = {1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

pkv_status pkv_attend_frames(pkv_t h, const void* q, const void* k, const void* v, int n_frames,
                             int tokens, void* out, float sm_scale, void* cuda_stream) {
  if (!h) return fail(h, PKV_ERR_INVALID, "null handle");
  if (n_frames < 0 || tokens < 1 || tokens > (1 << 20))
    return fail(h, PKV_ERR_INVALID, "n_frames %d / tokens %d out of range", n_frames, tokens);
  // the tensor copies address rows with 32-bit coordinates
  if ((long long)n_frames * tokens > (long long)INT_MAX - 64)
    return fail(h, PKV_ERR_INVALID, "n_frames x tokens exceeds 2^31 - 65 rows");
  if (n_frames == 0) return PKV_OK;
  if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(h, PKV_ERR_INVALID, "q/k/v/out must be 16-byte aligned device pointers");
  const long long grid = (long long)attend_tc_mgroups(tokens) * h->H * n_frames;
  if (grid > INT_MAX) return fail(h, PKV_ERR_INVALID, "too many frames for one launch");
  AttendDense d;
  std::memset(&d, 0, sizeof(d));
  const long long rows = (long long)n_frames * tokens;
  if (!encode_kv_map(&d.k_map, k, h->H, rows) || !encode_kv_map(&d.v_map, v, h->H, rows))
    return fail(h, PKV_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable or rejected the K/V tensors");
  AttendArgs& a = d.a;
  a.q = static_cast<const uint16_t*>(q);
  a.out = static_cast<uint16_t*>(out);
  a.n_q = tokens;
  a.heads = h->H;
  a.page_size = kTileSlots;         // no pages; keeps the kernel's page arithmetic defined
  a.n_slots = tokens;
  a.n_tiles = attend_tc_tiles(tokens);
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt((float)h->D);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.num_splits = 1;
  a.err = h->d_err;
  PKV_CUDA(h, launch_attend_dense(d, n_frames, as_stream(cuda_stream)));
  return PKV_OK;
}

pkv_status pkv_attend_batched(pkv_t h, const void* q, const int* q_off, const int* sids, int n,
                              int layer, void* out, float sm_scale, void* cuda_stream) {
  if (!h) return fail(h, PKV_ERR_INVALID, "null handle");
  if (n < 1 || n > kMaxBatch || !q_off || !sids || !q || !out)
    return fail(h, PKV_ERR_INVALID, "need 1..%d streams, offsets, ids, q and out", kMaxBatch);
  if (q_off[0] != 0) return fail(h, PKV_ERR_INVALID, "q_off[0] must be 0");
  const size_t row_bytes = (size_t)h->H * kHeadDim * sizeof(uint16_t);
  // every stream's call, validated before anything is launched
  std::vector<AttendArgs> calls(n);
  for (int i = 0; i < n; ++i) {
    for (int k = 0; k < i; ++k)
      if (sids[k] == sids[i]) return fail(h, PKV_ERR_INVALID, "stream %d listed twice", sids[i]);
    Stream* st = nullptr;
    if (pkv_status r = get_stream(h, sids[i], &st)) return r;
    const int n_q = q_off[i + 1] - q_off[i];
    if (n_q < 1 || q_off[i + 1] > (1 << 20))
      return fail(h, PKV_ERR_INVALID, "stream %d: query rows %d..%d", sids[i], q_off[i], q_off[i + 1]);
    if (st->cfg.mode == PKV_MODE_CHUNKED) {
      if (!st->c_open) return fail(h, PKV_ERR_STATE, "stream %d: no open chunk", sids[i]);
      const int cur = (st->c_head + st->n_chunks - 1) % st->cfg.sliding_window_num;
      if (n_q != st->c_len[cur])
        return fail(h, PKV_ERR_INVALID, "stream %d: n_q %d != the open chunk's %d tokens", sids[i],
                    n_q, st->c_len[cur]);
    }
    const char* qi = static_cast<const char*>(q) + (size_t)q_off[i] * row_bytes;
    char* oi = static_cast<char*>(out) + (size_t)q_off[i] * row_bytes;
    if (pkv_status r = attend_args(h, st, qi, n_q, layer, oi, sm_scale, &calls[i])) return r;
  }
  // one launch (attention, then combine) per kernel shape; one split count each
  std::vector<int> shape(n);
  for (int i = 0; i < n; ++i) shape[i] = attend_tc_shape(calls[i].n_q);
  size_t scratch = 0;
  std::vector<int> splits_of_shape(4, 1);
  for (int sh = 0; sh < 4; ++sh) {
    int pairs = 0, max_tiles = 0;
    for (int i = 0; i < n; ++i)
      if (shape[i] == sh) {
        pairs += attend_tc_mgroups(calls[i].n_q) * h->H;
        max_tiles = std::max(max_tiles, calls[i].n_tiles);
      }
    if (pairs == 0) continue;
    splits_of_shape[sh] = attend_tc_splits_pairs(pairs, max_tiles, h->num_sms);
    for (int i = 0; i < n; ++i)
      if (shape[i] == sh) {
        calls[i].num_splits = splits_of_shape[sh];
        if (calls[i].num_splits > 1) scratch += partial_bytes_aligned(calls[i]);
      }
  }
  if (scratch > 0) {
    if (pkv_status r = ensure_scratch(h, scratch)) return r;
    float* base = h->d_scratch;
    for (int i = 0; i < n; ++i)
      if (calls[i].num_splits > 1) {
        place_partials(&calls[i], base);
        base += partial_bytes_aligned(calls[i]) / sizeof(float);
      }
  }
  std::unique_ptr<AttendBatch> b(new AttendBatch);
  for (int sh = 0; sh < 4; ++sh) {
    std::memset(b.get(), 0, sizeof(AttendBatch));
    for (int i = 0; i < n; ++i) {
      if (shape[i] != sh) continue;
      const int k = b->n++;
      b->item[k] = calls[i];
      b->n_mgroups[k] = attend_tc_mgroups(calls[i].n_q);
      b->n_tiles[k] = calls[i].n_tiles;
      b->cta_base[k + 1] = b->cta_base[k] + b->n_mgroups[k] * h->H * calls[i].num_splits;
      b->pair_base[k + 1] = b->pair_base[k] + (long long)calls[i].n_q * h->H;
    }
    if (b->n > 0) PKV_CUDA(h, launch_attend_batch(*b, as_stream(cuda_stream)));
  }
  return PKV_OK;
}

pkv_status pkv_sync(pkv_t h, void* cuda_stream) {
  if (!h) return fail(h, PKV_ERR_INVALID, "null handle");
  PKV_CUDA(h, cudaStreamSynchronize(as_stream(cuda_stream)));
  PKV_CUDA(h, cudaGetLastError());
  int err = 0;
  PKV_CUDA(h, cudaMemcpy(&err, h->d_err, sizeof(int), cudaMemcpyDeviceToHost));
  if (err & kErrTimeout) return fail(h, PKV_ERR_TIMEOUT, "a bounded device wait gave up (0x%x)", err);
  if (err) return fail(h, PKV_ERR_DEVICE, "device error word 0x%x (page id outside the pool)", err);
  return PKV_OK;
}

pkv_status pkv_visible_count(pkv_t h, int sid, int* n_pages, int* n_tokens) {
  Stream* st = nullptr;
  if (pkv_status r = get_stream(h, sid, &st)) return r;
  int np, nt, last;
  visible_counts(h, *st, &np, &nt, &last);
  if (n_pages) *n_pages = np;
  if (n_tokens) *n_tokens = nt;
  return PKV_OK;
}

pkv_status pkv_free_pages(pkv_t h, int* n_free) {
  if (!h || !n_free) return fail(h, PKV_ERR_INVALID, "null argument");
  *n_free = h->free_top;
  return PKV_OK;
}

pkv_status pkv_export_state(pkv_t h, int sid, int32_t* host_buf, size_t cap_words,
                            size_t* used_words) {
  Stream* st = nullptr;
  if (pkv_status r = get_stream(h, sid, &st)) return r;
  if (!host_buf || !used_words) return fail(h, PKV_ERR_INVALID, "null argument");
  int np, nt, last;
  visible_counts(h, *st, &np, &nt, &last);
  const size_t need = 1 + (size_t)h->free_top + 1 + 2 * (size_t)np + 6 + 3 + kMaxChunks;
  if (cap_words < need) return fail(h, PKV_ERR_INVALID, "export needs %zu words", need);
  PKV_CUDA(h, cudaDeviceSynchronize());
  std::vector<int32_t> buf;
  buf.push_back(h->free_top);
  std::vector<int32_t> fs(h->free_top);
  if (h->free_top)
    PKV_CUDA(h, cudaMemcpy(fs.data(), h->d_free, sizeof(int32_t) * h->free_top, cudaMemcpyDeviceToHost));
  buf.insert(buf.end(), fs.begin(), fs.end());
  buf.push_back(np);
  if (np) {
    TableArgs t = table_args(h, *st, st->d_tbl_idx, st->d_tbl_len, nullptr, nullptr);
    PKV_CUDA(h, launch_table(t, 0));
    PKV_CUDA(h, cudaDeviceSynchronize());
    std::vector<int32_t> idx(np), len(np);
    PKV_CUDA(h, cudaMemcpy(idx.data(), st->d_tbl_idx, sizeof(int32_t) * np, cudaMemcpyDeviceToHost));
    PKV_CUDA(h, cudaMemcpy(len.data(), st->d_tbl_len, sizeof(int32_t) * np, cudaMemcpyDeviceToHost));
    buf.insert(buf.end(), idx.begin(), idx.end());
    buf.insert(buf.end(), len.begin(), len.end());
  }
  if (st->cfg.mode == PKV_MODE_FRAME) {
    int32_t w[6] = {st->n_scale, st->win_count, st->n_special, st->sp_len, st->kept, st->pending};
    buf.insert(buf.end(), w, w + 6);
  } else {
    buf.push_back(st->n_chunks);
    buf.push_back(st->c_open);
    buf.push_back(st->pending);
    for (int i = 0; i < st->n_chunks; ++i)
      buf.push_back(st->c_len[(st->c_head + i) % st->cfg.sliding_window_num]);
  }
  std::memcpy(host_buf, buf.data(), buf.size() * sizeof(int32_t));
  *used_words = buf.size();
  return PKV_OK;
}

pkv_status pkv_read_page(pkv_t h, int layer, int page, int kv, void* host_dst) {
  if (!h || !host_dst) return fail(h, PKV_ERR_INVALID, "null argument");
  if (layer < 0 || layer >= h->L || page < 0 || page >= h->P || (kv != 0 && kv != 1))
    return fail(h, PKV_ERR_INVALID, "layer/page/kv out of range");
  if (h->fp8) return fail(h, PKV_ERR_INVALID, "this cache holds FP8 pages: use pkv_read_page_fp8");
  const size_t n = (size_t)h->H * h->Ps * kHeadDim;
  std::vector<uint16_t> raw(n);
  PKV_CUDA(h, cudaDeviceSynchronize());
  const uint16_t* src = layer_base(h, layer) + (long long)page * h->page_elems + (long long)kv * n;
  PKV_CUDA(h, cudaMemcpy(raw.data(), src, n * sizeof(uint16_t), cudaMemcpyDeviceToHost));
  uint16_t* dst = static_cast<uint16_t*>(host_dst);
  for (int hh = 0; hh < h->H; ++hh)
    for (int s = 0; s < h->Ps; ++s)
      for (int c = 0; c < kChunksPerRow; ++c) {
        const size_t row = ((size_t)hh * h->Ps + s) * kHeadDim;
        std::memcpy(dst + row + c * 8, raw.data() + row + swizzle_chunk(s, c) * 8, 16);
      }
  return PKV_OK;
}

pkv_status pkv_read_page_fp8(pkv_t h, int layer, int page, int kv, void* codes_dst,
                             void* exps_dst) {
  if (!h || !codes_dst || !exps_dst) return fail(h, PKV_ERR_INVALID, "null argument");
  if (layer < 0 || layer >= h->L || page < 0 || page >= h->P || (kv != 0 && kv != 1))
    return fail(h, PKV_ERR_INVALID, "layer/page/kv out of range");
  if (!h->fp8) return fail(h, PKV_ERR_INVALID, "this cache holds bf16 pages: use pkv_read_page");
  // the kv half of the page (heads planes of page_size rows, in 65-byte row
  // blocks), then unpacked into [heads][page_size][64] codes and [heads][page_size]
  // exponents
  const size_t half = (size_t)h->H * h->Ps * (kHeadDim + 1);
  std::vector<uint8_t> raw(half);
  PKV_CUDA(h, cudaDeviceSynchronize());
  const uint8_t* pg = reinterpret_cast<const uint8_t*>(layer_base(h, layer)) + (long long)page * h->page_bytes;
  PKV_CUDA(h, cudaMemcpy(raw.data(), pg + (size_t)kv * half, half, cudaMemcpyDeviceToHost));
  uint8_t* codes = static_cast<uint8_t*>(codes_dst);
  uint8_t* exps = static_cast<uint8_t*>(exps_dst);
  for (int hh = 0; hh < h->H; ++hh)
    for (int s = 0; s < h->Ps; ++s) {
      const size_t row = (size_t)hh * h->Ps + s;
      std::memcpy(codes + row * kHeadDim, raw.data() + fp8_code_off(h->H, h->Ps, 0, hh, s), kHeadDim);
      exps[row] = raw[fp8_exp_off(h->H, h->Ps, 0, hh, s)];
    }
  return PKV_OK;
}

pkv_status pkv_synth_fill(void* dst, int n_frames, int n_tokens, int heads, int head_dim,
                          int seed, int workload, int stream, int layer, int frame0, int tensor,
                          int token0, float scale, void* cuda_stream) {
  if (!dst || n_frames < 0 || n_tokens < 0 || heads < 1 || heads > 32 || head_dim < 1 ||
      head_dim > 64 || seed < 0 || seed >= 128 || workload < 0 || workload >= 8 || stream < 0 ||
      stream >= 64 || layer < 0 || layer >= 32 || frame0 < 0 || frame0 + n_frames > 65536 ||
      tensor < 0 || tensor >= 4 || token0 < 0 || token0 + n_tokens > 16384)
    return fail(nullptr, PKV_ERR_INVALID, "pkv_synth_fill: argument out of range");
  if (reinterpret_cast<uintptr_t>(dst) & 1u)
    return fail(nullptr, PKV_ERR_INVALID, "pkv_synth_fill: dst must be 2-byte aligned");
  int e2;
  const float m = std::frexp(scale, &e2);
  if (m != 0.5f) return fail(nullptr, PKV_ERR_INVALID, "pkv_synth_fill: scale must be a power of two");
  const unsigned long long key_base =
      ((unsigned long long)seed << 57) | ((unsigned long long)workload << 54) |
      ((unsigned long long)stream << 48) | ((unsigned long long)layer << 43) |
      ((unsigned long long)tensor << 25);
  cudaError_t e = launch_synth(static_cast<uint16_t*>(dst), n_frames, n_tokens, heads, head_dim,
                               key_base, frame0, token0, scale, as_stream(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "pkv_synth_fill");
  return PKV_OK;
}

// ---------------------------------------------------------------------------
// Attention without allocation: the split-KV partials live in a fixed array.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace {

// Device address of the static scratch for the handle's device. pkv_create_ex
// resolved it with that device current; a handle created after a device reset
// resolves it again.
pkv_status noalloc_scratch(pkv_t h, float** out) {
  if (!h->noalloc_scratch)
    return fail(h, PKV_ERR_CUDA, "the static scratch's device address could not be resolved");
  *out = h->noalloc_scratch;
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_attend_noalloc(pkv_t h, const void* q, int n_q, int sid, int layer, void* out,
                              float sm_scale, void* cuda_stream) {
  Stream* st = nullptr;
  if (pkv_status r = get_stream(h, sid, &st)) return r;
  if (st->cfg.mode == PKV_MODE_CHUNKED) {
    if (!st->c_open) return fail(h, PKV_ERR_STATE, "no open chunk");
    const int cur = (st->c_head + st->n_chunks - 1) % st->cfg.sliding_window_num;
    if (n_q != st->c_len[cur])
      return fail(h, PKV_ERR_INVALID, "n_q %d != the open chunk's %d tokens", n_q, st->c_len[cur]);
  }
  AttendArgs a;
  if (pkv_status r = attend_args(h, st, q, n_q, layer, out, sm_scale, &a)) return r;
  a.num_splits = attend_num_splits(n_q, h->H, a.n_slots, h->num_sms);
  if (a.num_splits > 1) {
    if (partial_bytes(a) > kStaticScratchBytes)
      return fail(h, PKV_ERR_INVALID,
                  "this call needs %zu bytes of split-KV scratch; the static scratch holds %zu",
                  partial_bytes(a), kStaticScratchBytes);
    float* scratch = nullptr;
    if (pkv_status r = noalloc_scratch(h, &scratch)) return r;
    place_partials(&a, scratch);
  }
  cudaStream_t s = as_stream(cuda_stream);
  PKV_CUDA(h, launch_attend(a, h->num_sms, s));
  return PKV_OK;
}

}  // extern "C"
