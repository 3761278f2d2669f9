// Page-pool metadata and KV movement kernels: append/scatter (frame and chunked
// mode), pushes onto the free stack (rollback, eviction, close), the windowed
// reset, and the visible-page-table build.
//
// "LingBot-Map Paged KV Cache", section 2: pages come from a free list; a page
// that leaves the sliding window returns to it at once; special tokens are
// appended floor(page_size / n_special) frames to a page; the visible table is
// scale -> window -> special. Section 3: a non-keyframe's append is undone.
// Section 4: a window reset carries the last overlap keyframes over.
// vLLM-Omni RFC "Reconstruction Engine", section 3.3: chunk append / evict.
//
// The device holds page ids only (the free stack's array and each stream's
// lists). Every count and list position is mirrored on the host and passed in,
// so no kernel ever reads a count that another kernel is changing.
#include <atomic>

#include "pkv_internal.cuh"

namespace pkv {

namespace {

__device__ __forceinline__ bool page_ok(int p, int pool_pages) {
  return p >= 0 && p < pool_pages;
}

// Tokens moved by one append block (TPB): with several, each thread issues all
// its loads before its stores and the block's set-up (page-need scan, barrier)
// is shared; a single frame keeps one token per block so that it still spreads
// over the SMs.
template <int TPB>
constexpr int append_blocks(int tokens) { return (tokens + TPB - 1) / TPB; }
constexpr int kAppendBatchTokens = 8;
constexpr long long kAppendBatchMin = 4096;   // tokens x streams above which TPB = 8

// One batched frame-mode append. blockIdx.y selects the stream, blockIdx.x a
// group of TPB tokens; thread (kv, head, 16-byte chunk) moves one vector per
// token. Every block
// recomputes its stream's place on the free stack with an exclusive warp scan of
// the batch's page needs (1, or 2 when the frame opens a special page), so stream
// i pops after streams 0..i-1 exactly as sequential appends would.
template <int TPB>
__global__ void __launch_bounds__(512) frame_append_kernel(const FrameAppendArgs a) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.y;
  const AppendItem& it = a.item[b];
  const int H = a.pool.heads;
  const int hh = threadIdx.x >> 3, c = threadIdx.x & 7;
  const bool mover = hh < 2 * H;               // blocks have at least one full warp
  const int kv = hh >= H ? 1 : 0;
  const int h = hh - kv * H;
  const int T = a.n_patch + a.n_special;
  const int t0 = blockIdx.x * TPB;
  // The block's K/V rows are loaded first: they do not depend on the page pop
  // below, whose dependent loads then overlap them.
  uint4 val[TPB];
  if (mover) {
    const uint16_t* src = (kv ? it.v : it.k) + (long long)h * kHeadDim + c * 8;
#pragma unroll
    for (int i = 0; i < TPB; ++i)
      if (t0 + i < T)
        val[i] = __ldg(reinterpret_cast<const uint4*>(src + (long long)(t0 + i) * H * kHeadDim));
  }
  __shared__ int s_patch, s_sp;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int need = lane < a.n ? 1 + a.item[lane].new_sp : 0;
    int incl = need;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += y;
    }
    const int off = __shfl_sync(0xffffffffu, incl - need, b);
    if (lane == 0) {
      int patch, sp;
      if (a.is_meta) {
        patch = a.free_stack[a.top - 1 - off];
        sp = it.new_sp ? a.free_stack[a.top - 2 - off] : it.special_list[it.sp_idx];
      } else {
        patch = *it.patch_slot;
        sp = it.special_list[it.sp_idx];
      }
      const bool ok = page_ok(patch, a.pool.pool_pages) && page_ok(sp, a.pool.pool_pages);
      if (!ok) {
        atomicOr(a.err, kErrPageRange);
        patch = -1;
      } else {
        if (a.is_meta && blockIdx.x == 0) {
          *it.patch_slot = patch;
          if (it.new_sp) it.special_list[it.sp_idx] = sp;
        }
        // the rows of both pages change: their cached mean keys are stale
        if (blockIdx.x == 0 && a.pool.km_len) {
          a.pool.km_len[patch] = -1;
          a.pool.km_len[sp] = -1;
        }
      }
      s_patch = patch;
      s_sp = sp;
    }
  }
  __syncthreads();
  const int patch = s_patch, sp = s_sp;
  if (patch < 0 || !mover) return;
#pragma unroll
  for (int i = 0; i < TPB; ++i) {
    const int t = t0 + i;
    if (t < T) {
      const int page = t < a.n_patch ? patch : sp;
      const int slot = t < a.n_patch ? t : it.sp_off + (t - a.n_patch);
      store_row_chunk(a.pool, page, kv, h, slot, c, val[i]);
    }
    // a freshly opened special page gets its unused slots zeroed, so that every
    // slot of a held page is a token or zero (the grid covers page_size +
    // n_special > page_size - n_special token indices)
    if (it.new_sp && t < a.pool.page_size - a.n_special) {
      const int slot = a.n_special + t;
      store_row_chunk(a.pool, sp, kv, h, slot, c, make_uint4(0u, 0u, 0u, 0u));
    }
  }
}

// Chunked-mode append: the frame's tokens are packed after the chunk's pos0
// tokens; pages of the chunk past old_pages are popped by this append. One block
// per TPB tokens, as above; the blocks also zero the tail of a freshly popped
// last page.
template <int TPB>
__global__ void __launch_bounds__(512) chunk_append_kernel(const ChunkAppendArgs a) {
  pdl_wait();
  pdl_trigger();
  const int Ps = a.pool.page_size;
  if (a.is_meta && blockIdx.x == 0) {
    for (int i = threadIdx.x; i < a.n_new; i += blockDim.x) {
      const int p = a.free_stack[a.top - 1 - i];
      if (page_ok(p, a.pool.pool_pages)) a.chunk_pages[a.old_pages + i] = p;
      else atomicOr(a.err, kErrPageRange);
    }
  }
  const int end = a.pos0 + a.n_tokens;
  const int last_pi = (end - 1) / Ps;
  const int zero_slots = (last_pi >= a.old_pages && (end % Ps) != 0) ? Ps - (end % Ps) : 0;
  const int H = a.pool.heads;
  const int hh = threadIdx.x >> 3, c = threadIdx.x & 7;
  if (hh >= 2 * H) return;
  const int kv = hh >= H ? 1 : 0;
  const int h = hh - kv * H;
  // position pos of the chunk receives val (a token, or zero past the end)
  auto put = [&](int pos, const uint4& val) {
    const int pi = pos / Ps;
    const int slot = pos - pi * Ps;
    const int page = (pi < a.old_pages || !a.is_meta)
                         ? a.chunk_pages[pi]
                         : a.free_stack[a.top - 1 - (pi - a.old_pages)];
    if (!page_ok(page, a.pool.pool_pages)) {
      atomicOr(a.err, kErrPageRange);
      return;
    }
    store_row_chunk(a.pool, page, kv, h, slot, c, val);
  };
  // tokens t0 .. t0 + TPB - 1, loads first
  const int t0 = blockIdx.x * TPB;
  const uint16_t* src = (kv ? a.v : a.k) + (long long)h * kHeadDim + c * 8;
  uint4 val[TPB];
#pragma unroll
  for (int i = 0; i < TPB; ++i)
    if (t0 + i < a.n_tokens)
      val[i] = __ldg(reinterpret_cast<const uint4*>(src + (long long)(t0 + i) * H * kHeadDim));
#pragma unroll
  for (int i = 0; i < TPB; ++i)
    if (t0 + i < a.n_tokens) put(a.pos0 + t0 + i, val[i]);
  // the unused tail of a freshly popped last page, in groups of TPB slots
  for (int z0 = t0; z0 < zero_slots; z0 += (int)gridDim.x * TPB)
    for (int i = 0; i < TPB && z0 + i < zero_slots; ++i)
      put(end + z0 + i, make_uint4(0u, 0u, 0u, 0u));
}

// Push page ids onto the free stack: free[top + j] for j over the segments in
// order. Sources are stream lists, never the free stack itself.
__global__ void __launch_bounds__(256) push_kernel(const PushArgs a) {
  pdl_wait();
  pdl_trigger();
  int total = 0;
  for (int s = 0; s < a.n_seg; ++s) total += a.seg[s].count;
  for (int j = threadIdx.x; j < total; j += blockDim.x) {
    int s = 0, base = 0;
    while (j >= base + a.seg[s].count) {
      base += a.seg[s].count;
      ++s;
    }
    const PushSegment& g = a.seg[s];
    int pos = g.start + g.step * (j - base);
    if (g.ring) pos = ((pos % g.ring) + g.ring) % g.ring;
    const int p = g.src[pos];
    if (!page_ok(p, a.pool_pages)) {
      atomicOr(a.err, kErrPageRange);
      continue;
    }
    a.free_stack[a.top + j] = p;
  }
}

// Window reset, data part: copy each carried frame's special tokens (every
// layer, K and V) into the freshly popped special pages free[top-1-k], and zero
// those pages' unused slots.
__global__ void __launch_bounds__(256) reset_copy_kernel(const ResetCopyArgs a) {
  const int H = a.heads, Ps = a.page_size;
  // the popped pages' rows change: their cached mean keys are stale
  if (blockIdx.x == 0 && a.km_len)
    for (int i = threadIdx.x; i < a.layers * a.n_new; i += blockDim.x) {
      const int p = a.free_stack[a.top - 1 - i % a.n_new];
      if (page_ok(p, a.pool_pages)) a.km_len[(long long)(i / a.n_new) * a.pool_pages + p] = -1;
    }
  const long long per_slot = 2LL * H * kChunksPerRow;
  const long long copy_total = (long long)a.layers * a.n_carry * a.n_special * per_slot;
  const long long zero_total = (long long)a.layers * a.n_new * Ps * per_slot;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < copy_total + zero_total;
       i += stride) {
    const bool is_copy = i < copy_total;
    long long r = is_copy ? i : i - copy_total;
    const int c = (int)(r & 7);
    r >>= 3;
    const int h = (int)(r % H);
    r /= H;
    const int kv = (int)(r & 1);
    r >>= 1;
    int dst_page_k, dst_slot, layer;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (is_copy) {
      const int j = (int)(r % a.n_special);
      r /= a.n_special;
      const int ci = (int)(r % a.n_carry);
      layer = (int)(r / a.n_carry);
      const int src_page = a.special_list[a.src_sp_idx[ci]];
      if (!page_ok(src_page, a.pool_pages)) {
        atomicOr(a.err, kErrPageRange);
        continue;
      }
      const int src_slot = a.src_sp_off[ci] + j;
      if (a.fp8) {
        // FP8 pages: the row's codes (8 per chunk) and exponent move as they are
        const uint8_t* base = reinterpret_cast<const uint8_t*>(a.pool) + layer * a.layer_bytes +
                              (long long)src_page * a.page_bytes;
        const uint2 codes =
            *reinterpret_cast<const uint2*>(base + fp8_code_off(H, Ps, kv, h, src_slot) + 8 * c);
        val = make_uint4(codes.x, codes.y,
                         c == 0 ? (uint32_t)base[fp8_exp_off(H, Ps, kv, h, src_slot)] : 0u, 0u);
      } else {
        const uint16_t* src = a.pool + layer * a.layer_elems + (long long)src_page * a.page_elems +
                              ((long long)(kv * H + h) * Ps + src_slot) * kHeadDim +
                              swizzle_chunk(src_slot, c) * 8;
        val = *reinterpret_cast<const uint4*>(src);
      }
      dst_page_k = ci / a.f_sp;
      dst_slot = (ci % a.f_sp) * a.n_special + j;
    } else {
      const int slot = (int)(r % Ps);
      r /= Ps;
      dst_page_k = (int)(r % a.n_new);
      layer = (int)(r / a.n_new);
      const int frames_here = min(a.f_sp, a.n_carry - dst_page_k * a.f_sp);
      if (slot < frames_here * a.n_special) continue;   // written by the copy part
      dst_slot = slot;
    }
    const int dst_page = a.free_stack[a.top - 1 - dst_page_k];
    if (!page_ok(dst_page, a.pool_pages)) {
      atomicOr(a.err, kErrPageRange);
      continue;
    }
    if (a.fp8) {
      uint8_t* base = reinterpret_cast<uint8_t*>(a.pool) + layer * a.layer_bytes +
                      (long long)dst_page * a.page_bytes;
      *reinterpret_cast<uint2*>(base + fp8_code_off(H, Ps, kv, h, dst_slot) + 8 * c) =
          make_uint2(val.x, val.y);
      if (c == 0) base[fp8_exp_off(H, Ps, kv, h, dst_slot)] = (uint8_t)val.z;
      continue;
    }
    uint16_t* dst = a.pool + layer * a.layer_elems + (long long)dst_page * a.page_elems +
                    ((long long)(kv * H + h) * Ps + dst_slot) * kHeadDim +
                    swizzle_chunk(dst_slot, c) * 8;
    *reinterpret_cast<uint4*>(dst) = val;
  }
}

// Window reset, metadata part (one block): the last n_carry held pages become
// the scale list, the popped pages the special list, and the other held pages
// (scale, then window oldest first) and the old special pages are pushed.
__global__ void __launch_bounds__(256) reset_meta_kernel(const ResetMetaArgs a) {
  extern __shared__ int sm[];
  const int n_held = a.n_scale + a.win_count;
  int* held = sm;
  int* old_sp = held + n_held;
  int* new_sp = old_sp + a.n_special_old;
  for (int j = threadIdx.x; j < n_held; j += blockDim.x)
    held[j] = j < a.n_scale ? a.scale[j] : a.window[(a.win_head + j - a.n_scale) % a.win_cap];
  for (int j = threadIdx.x; j < a.n_special_old; j += blockDim.x) old_sp[j] = a.special[j];
  for (int k = threadIdx.x; k < a.n_new; k += blockDim.x) new_sp[k] = a.free_stack[a.top - 1 - k];
  __syncthreads();
  const int n_free_held = n_held - a.n_carry;
  const int top2 = a.top - a.n_new;
  for (int i = threadIdx.x; i < a.n_carry; i += blockDim.x) a.scale[i] = held[n_free_held + i];
  for (int k = threadIdx.x; k < a.n_new; k += blockDim.x) a.special[k] = new_sp[k];
  for (int j = threadIdx.x; j < n_free_held + a.n_special_old; j += blockDim.x) {
    const int p = j < n_free_held ? held[j] : old_sp[j - n_free_held];
    if (!page_ok(p, a.pool_pages)) {
      atomicOr(a.err, kErrPageRange);
      continue;
    }
    a.free_stack[top2 + j] = p;
  }
}

// Visible page table: page ids and valid slot counts in attention order.
__global__ void __launch_bounds__(256) table_kernel(const TableArgs a) {
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < a.n; e += gridDim.x * blockDim.x) {
    int id, len;
    table_entry(a, e, id, len);
    if (!page_ok(id, a.pool_pages)) {
      atomicOr(a.err, kErrPageRange);
      id = 0;
      len = 0;
    }
    a.out_idx[e] = id;
    a.out_len[e] = len;
  }
}

__global__ void table_tail_kernel(int32_t* out_n, int32_t* out_last, int n, int last) {
  if (out_n) *out_n = n;
  if (out_last) *out_last = last;
}

inline int blocks_for(long long work, int per_block, int cap) {
  long long b = (work + per_block - 1) / per_block;
  if (b < 1) b = 1;
  if (b > cap) b = cap;
  return (int)b;
}

}  // namespace

namespace {
std::atomic<unsigned long long> g_launches{0};
}

unsigned long long launch_count() { return g_launches.load(); }
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n); }

cudaError_t launch_frame_append(const FrameAppendArgs& a, cudaStream_t s) {
  const int T = a.n_patch + a.n_special;
  const dim3 block(16 * a.pool.heads < 32 ? 32 : 16 * a.pool.heads);
  const cudaError_t e =
      (long long)T * a.n >= kAppendBatchMin
          ? launch_pdl(frame_append_kernel<kAppendBatchTokens>,
                       dim3(append_blocks<kAppendBatchTokens>(T), a.n), block, 0, s, a)
          : launch_pdl(frame_append_kernel<1>, dim3(T, a.n), block, 0, s, a);
  count_launches(1);
  return e;
}

cudaError_t launch_chunk_append(const ChunkAppendArgs& a, cudaStream_t s) {
  const dim3 block(16 * a.pool.heads < 32 ? 32 : 16 * a.pool.heads);
  const cudaError_t e =
      a.n_tokens >= kAppendBatchMin
          ? launch_pdl(chunk_append_kernel<kAppendBatchTokens>,
                       dim3(append_blocks<kAppendBatchTokens>(a.n_tokens)), block, 0, s, a)
          : launch_pdl(chunk_append_kernel<1>, dim3(a.n_tokens), block, 0, s, a);
  count_launches(1);
  return e;
}

cudaError_t launch_push(const PushArgs& a, cudaStream_t s) {
  const cudaError_t e = launch_pdl(push_kernel, dim3(1), dim3(256), 0, s, a);
  count_launches(1);
  return e;
}

cudaError_t launch_reset_copy(const ResetCopyArgs& a, cudaStream_t s) {
  const long long work = (long long)a.layers * (a.n_carry * a.n_special + a.n_new * a.page_size) *
                         2 * a.heads * 8;
  if (work == 0) return cudaSuccess;
  reset_copy_kernel<<<blocks_for(work, 256 * 4, 4096), 256, 0, s>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_reset_meta(const ResetMetaArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(int) * (size_t)(a.n_scale + a.win_count + a.n_special_old + a.n_new);
  if (smem > 48 * 1024) return cudaErrorInvalidValue;
  reset_meta_kernel<<<1, 256, smem, s>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_table(const TableArgs& a, cudaStream_t s) {
  if (a.n > 0) {
    table_kernel<<<blocks_for(a.n, 256, 64), 256, 0, s>>>(a);
    count_launches(1);
  }
  if (a.out_n || a.out_last) {
    // the last entry's length is known on the host through the counts
    int last = 0;
    if (a.n > 0) {
      if (a.mode == 0) {
        last = a.n_special > 0 ? a.sp_last_len : a.page_size;
      } else {
        const int c = a.n_chunks - 1;
        last = a.chunk_len[c] - (a.chunk_npages[c] - 1) * a.page_size;
      }
    }
    table_tail_kernel<<<1, 1, 0, s>>>(a.out_n, a.out_last, a.n, last);
    count_launches(1);
  }
  return cudaGetLastError();
}

}  // namespace pkv
