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
//   score    = sum over h, then d, in order of (qm[h][d] * km[h][d])
// (__fadd_rn / __fmul_rn / __fdiv_rn: no contraction into fused multiply-adds).
#include <cuda_bf16.h>

#include "pkv_internal.cuh"

namespace pkv {

namespace {

__device__ __forceinline__ float bf16_at(const uint16_t* p) {
  return __uint_as_float((uint32_t)__ldg(p) << 16);
}

// qm[h][d]: block h, thread d
__global__ void __launch_bounds__(kHeadDim) pool_q_kernel(const PageScoreArgs a) {
  pdl_wait();
  pdl_trigger();
  const int h = blockIdx.x, d = threadIdx.x;
  float acc = 0.f;
  for (int i = 0; i < a.n_q; ++i)
    acc = __fadd_rn(acc, bf16_at(a.q + ((long long)i * a.heads + h) * kHeadDim + d));
  a.qm[h * kHeadDim + d] = __fdiv_rn(acc, (float)a.n_q);
}

// score of visible page e: block e; thread (h, d) pools its key column, then
// thread 0 adds the products in (h, d) order
__global__ void __launch_bounds__(256) page_score_kernel(const PageScoreArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ float prod[kMaxHeads * kHeadDim];
  const int e = blockIdx.x;
  int page = 0, len = 0;
  table_entry(a.tbl, e, page, len);
  const bool ok = page >= 0 && page < a.pool.pool_pages && len >= 1 && len <= a.pool.page_size;
  const int n = a.heads * kHeadDim;
  for (int hd = threadIdx.x; hd < n; hd += blockDim.x) {
    const int h = hd / kHeadDim, d = hd % kHeadDim;
    float km = 0.f;
    if (ok) {
      const uint16_t* col = a.pool.base + (long long)page * a.pool.page_elems +
                            (long long)h * a.pool.page_size * kHeadDim + (d & 7);
      float acc = 0.f;
      for (int s = 0; s < len; ++s)
        acc = __fadd_rn(acc, bf16_at(col + (long long)s * kHeadDim + swizzle_chunk(s, d >> 3) * 8));
      km = __fdiv_rn(acc, (float)len);
    }
    prod[hd] = __fmul_rn(a.qm[hd], km);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!ok) atomicOr(a.err, kErrPageRange);
    float acc = 0.f;
    for (int hd = 0; hd < n; ++hd) acc = __fadd_rn(acc, prod[hd]);
    a.scores[e] = ok ? acc : __int_as_float(0x7fc00000);    // NaN ranks lowest
  }
}

// kept table positions in table order: the anchors, then the `keep` best others
__global__ void __launch_bounds__(kMaxSampledEntries) select_kernel(const PageScoreArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ float key[kMaxSampledEntries];
  __shared__ int flag[kMaxSampledEntries];
  const int e = threadIdx.x, n = a.n_entries;
  if (e < n) {
    const float s = a.scores[e];
    key[e] = isnan(s) ? -INFINITY : s;
  }
  __syncthreads();
  if (e < n) {
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
  if (e < n && flag[e]) {
    int pos = 0;
    for (int o = 0; o < e; ++o) pos += flag[o];
    a.kept[pos] = (uint16_t)e;
  }
}

}  // namespace

cudaError_t launch_page_select(const PageScoreArgs& a, cudaStream_t s) {
  cudaError_t e = launch_pdl(pool_q_kernel, dim3(a.heads), dim3(kHeadDim), 0, s, a);
  if (e == cudaSuccess) e = launch_pdl(page_score_kernel, dim3(a.n_entries), dim3(256), 0, s, a);
  if (e == cudaSuccess) e = launch_pdl(select_kernel, dim3(1), dim3(kMaxSampledEntries), 0, s, a);
  count_launches(3);
  return e;
}

}  // namespace pkv
