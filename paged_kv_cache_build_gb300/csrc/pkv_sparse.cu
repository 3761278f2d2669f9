// Page skipping by estimated attention mass: the per-page estimate and the
// selection of the pages a frame attends to.
//
// vLLM-Omni RFC "Reconstruction Engine", section 5 (KV compression): Sparse-VGGT
// skips the low-weight blocks of global attention, whose mass concentrates on a
// few of them; FastVGGT keeps the initial frames as anchors. At page granularity
// on the visible table of "LingBot-Map Paged KV Cache", section 2: a page's
// estimate is the dot product of the frame's mean query with the page's mean key,
// summed over heads; the scale pages are always kept and of the others the `keep`
// highest estimates (ties to the earlier table position, NaN lowest).
//
// The estimate decides an integer (which pages are kept), so it is computed in
// one fixed fp32 order with every operation rounded once:
//   qm[h][d] = (sum over rows i in order of q[i][h][d]) / n_q
//   km[h][d] = (sum over valid slots s in order of K[s][h][d]) / len
//   s_h      = sum over d in order of (qm[h][d] * km[h][d])   (each head h)
//   score    = sum over h in order of s_h
// (__fadd_rn / __fmul_rn / __fdiv_rn: no contraction into fused multiply-adds).
// A page's km depends only on its rows, so each layer keeps a cache of km per
// page, tagged with the valid length it was computed at; the append and the
// windowed reset clear the tag of every page they write, and a call recomputes
// only the pages whose tag differs from their length (at steady state the
// frame's newest pages): two launches in all (the means; the scores and the
// selection).
#include <cuda_bf16.h>

#include "pkv_internal.cuh"

namespace pkv {

namespace {

// The means, block (x, h), 256 threads: x = n_entries computes qm[h]; x < n_entries
// recomputes km[h] of visible page x into the layer's mean-key cache if the
// page's tag differs from its valid length (else it has nothing to do). The rows
// go through shared memory (coalesced, many loads in flight), then thread d adds
// its column in row order. The tags are set by the next launch, which reads
// them after every block here has finished.
constexpr int kPoolRows = 320;
__global__ void __launch_bounds__(256) page_means_kernel(const PageScoreArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint4 rows[kPoolRows * kChunksPerRow];       // 320 rows x 64 bf16 (40 KB)
  const int e = blockIdx.x, h = blockIdx.y;
  const bool is_q = e == a.n_entries;
  int page = 0, len = a.n_q;
  if (!is_q) {
    table_entry(a.tbl, e, page, len);
    // a bad entry is reported by the score kernel
    if (page < 0 || page >= a.pool.pool_pages || len < 1 || len > a.pool.page_size) return;
    if (a.km_len[page] == len) return;
  }
  const uint16_t* plane = is_q ? a.q + (long long)h * kHeadDim
                               : a.pool.base + (long long)page * a.pool.page_elems +
                                     (long long)h * a.pool.page_size * kHeadDim;
  const long long row_stride = is_q ? (long long)a.heads * kHeadDim : kHeadDim;
  float acc = 0.f;
  for (int r0 = 0; r0 < len; r0 += kPoolRows) {
    const int nr = min(kPoolRows, len - r0);
    for (int i = threadIdx.x; i < nr * kChunksPerRow; i += blockDim.x)
      rows[i] = __ldg(reinterpret_cast<const uint4*>(plane + (r0 + i / kChunksPerRow) * row_stride) +
                      i % kChunksPerRow);
    __syncthreads();
    if (threadIdx.x < kHeadDim) {
      const int d = threadIdx.x;
      const uint16_t* base = reinterpret_cast<const uint16_t*>(rows);
#pragma unroll 8
      for (int r = 0; r < nr; ++r) {
        // page rows are 128-byte swizzled: value d of slot s sits in chunk
        // swizzle_chunk(s, d / 8)
        const int col = is_q ? d : swizzle_chunk(r0 + r, d >> 3) * 8 + (d & 7);
        acc = __fadd_rn(acc, __uint_as_float((uint32_t)base[r * kHeadDim + col] << 16));
      }
    }
    __syncthreads();
  }
  if (threadIdx.x < kHeadDim) {
    const float v = __fdiv_rn(acc, (float)len);
    if (is_q) a.qm[h * kHeadDim + threadIdx.x] = v;
    else a.km[((long long)page * a.heads + h) * kHeadDim + threadIdx.x] = v;
  }
}

// Kept table positions in table order: the anchors, then the `keep` best others
// (one block; every thread takes entries e, e + blockDim.x, ...).
__device__ void select_kept(const PageScoreArgs& a) {
  __shared__ float key[kMaxSampledEntries];
  __shared__ int flag[kMaxSampledEntries];
  const int n = a.n_entries;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const float s = __ldcg(a.scores + e);
    key[e] = isnan(s) ? -INFINITY : s;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    int kept = 1;
    if (e >= a.n_anchor) {
      int rank = 0;
      for (int o = a.n_anchor; o < n; ++o)
        rank += (o != e) && (key[o] > key[e] || (key[o] == key[e] && o < e));
      kept = rank < a.keep;
    }
    flag[e] = kept;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < n; e += blockDim.x)
    if (flag[e]) {
      int pos = 0;
      for (int o = 0; o < e; ++o) pos += flag[o];
      a.kept[pos] = (uint16_t)e;
    }
}

// Score of page e (block e): the products qm * km of its cached mean keys (all
// threads), each head's added over d in order (one thread per head), then the
// heads' sums in head order (one thread); the page's
// tag becomes its valid length (every stale km was recomputed by the launch
// before). A recomputed km is the same fp32 value as a cached one, bit for bit
// (same operations, same order), and every kernel that writes a page's rows sets
// its tag to -1, so a cached value is used only while the page's rows are the
// ones it was computed from. The block that finishes last (a counter, after a
// fence; no block waits for another) selects the kept pages and resets the
// counter for the next call.
__global__ void __launch_bounds__(256) page_score_kernel(const PageScoreArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ __align__(16) float prod[kMaxHeads * kHeadDim];
  __shared__ float head_sum[kMaxHeads];
  __shared__ int s_last;
  const int e = blockIdx.x, n = a.heads * kHeadDim;   // n: a multiple of 64
  int page = 0, len = 0;
  table_entry(a.tbl, e, page, len);
  const bool ok = page >= 0 && page < a.pool.pool_pages && len >= 1 && len <= a.pool.page_size;
  if (ok) {
    // the products, all at once; then one thread adds them in (h, d) order
    const float* cache = a.km + (long long)page * n;
    for (int i = threadIdx.x; i < n; i += blockDim.x)
      prod[i] = __fmul_rn(__ldcg(a.qm + i), __ldcg(cache + i));
  }
  __syncthreads();
  if (ok && threadIdx.x < a.heads) {
    const float4* p4 = reinterpret_cast<const float4*>(prod + threadIdx.x * kHeadDim);
    float s_h = 0.f;
#pragma unroll
    for (int i = 0; i < kHeadDim / 4; ++i) {
      const float4 v = p4[i];
      s_h = __fadd_rn(s_h, v.x);
      s_h = __fadd_rn(s_h, v.y);
      s_h = __fadd_rn(s_h, v.z);
      s_h = __fadd_rn(s_h, v.w);
    }
    head_sum[threadIdx.x] = s_h;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float acc = __int_as_float(0x7fc00000);               // NaN: ranks lowest
    if (ok) {
      a.km_len[page] = len;
      acc = 0.f;
      for (int hh = 0; hh < a.heads; ++hh) acc = __fadd_rn(acc, head_sum[hh]);
    } else {
      atomicOr(a.err, kErrPageRange);
    }
    a.scores[e] = acc;
    __threadfence();
    s_last = atomicAdd(a.done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  select_kept(a);
  if (threadIdx.x == 0) *a.done = 0u;
}

}  // namespace

cudaError_t launch_page_select(const PageScoreArgs& a, cudaStream_t s) {
  cudaError_t e =
      launch_pdl(page_means_kernel, dim3(a.n_entries + 1, a.heads), dim3(256), 0, s, a);
  if (e == cudaSuccess) e = launch_pdl(page_score_kernel, dim3(a.n_entries), dim3(256), 0, s, a);
  count_launches(2);
  return e;
}

}  // namespace pkv
