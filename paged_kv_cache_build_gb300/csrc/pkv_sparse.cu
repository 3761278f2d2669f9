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

// qm[h][d]: block h; the rows go through shared memory in chunks (coalesced,
// many loads in flight), then thread d adds its column in row order
constexpr int kPoolRows = 128;
__global__ void __launch_bounds__(256) pool_q_kernel(const PageScoreArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint4 rows[kPoolRows * kChunksPerRow];       // 128 rows x 64 bf16
  const int h = blockIdx.x;
  float acc = 0.f;
  for (int r0 = 0; r0 < a.n_q; r0 += kPoolRows) {
    const int nr = min(kPoolRows, a.n_q - r0);
    for (int i = threadIdx.x; i < nr * kChunksPerRow; i += blockDim.x)
      rows[i] = __ldg(reinterpret_cast<const uint4*>(
                          a.q + ((long long)(r0 + i / kChunksPerRow) * a.heads + h) * kHeadDim) +
                      i % kChunksPerRow);
    __syncthreads();
    if (threadIdx.x < kHeadDim) {
      const uint16_t* base = reinterpret_cast<const uint16_t*>(rows) + threadIdx.x;
#pragma unroll 8
      for (int r = 0; r < nr; ++r)
        acc = __fadd_rn(acc, __uint_as_float((uint32_t)base[r * kHeadDim] << 16));
    }
    __syncthreads();
  }
  if (threadIdx.x < kHeadDim)
    a.qm[h * kHeadDim + threadIdx.x] = __fdiv_rn(acc, (float)a.n_q);
}

// prod[e][h][d] = qm[h][d] * km[h][d] for page e (blockIdx.x), head h
// (blockIdx.y): the page's plane of head h (len rows of 128 bytes, swizzled) is
// copied to shared memory, then thread d adds its column in slot order
__global__ void __launch_bounds__(kHeadDim) pool_k_kernel(const PageScoreArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint4 plane[kMaxPageSize * kChunksPerRow];   // up to 256 rows x 64 bf16
  const int e = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  int page = 0, len = 0;
  table_entry(a.tbl, e, page, len);
  const bool ok = page >= 0 && page < a.pool.pool_pages && len >= 1 && len <= a.pool.page_size;
  float km = __int_as_float(0x7fc00000);                  // NaN: ranks lowest
  if (ok) {
    const uint4* src = reinterpret_cast<const uint4*>(
        a.pool.base + (long long)page * a.pool.page_elems + (long long)h * a.pool.page_size * kHeadDim);
    for (int i = d; i < len * kChunksPerRow; i += blockDim.x) plane[i] = __ldg(src + i);
  } else if (d == 0) {
    atomicOr(a.err, kErrPageRange);
  }
  __syncthreads();
  if (ok) {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(plane) + (d & 7);
    float acc = 0.f;
#pragma unroll 8
    for (int s = 0; s < len; ++s)
      acc = __fadd_rn(acc, __uint_as_float((uint32_t)p[s * kHeadDim + swizzle_chunk(s, d >> 3) * 8]
                                           << 16));
    km = __fdiv_rn(acc, (float)len);
  }
  a.prod[((long long)e * a.heads + h) * kHeadDim + d] = __fmul_rn(a.qm[h * kHeadDim + d], km);
}

// score of page e (block e): the products in (h, d) order, one running sum
__global__ void __launch_bounds__(256) page_score_kernel(const PageScoreArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ __align__(16) float prod[kMaxHeads * kHeadDim];
  const int e = blockIdx.x, n = a.heads * kHeadDim;   // a multiple of 64
  for (int i = threadIdx.x; i < n; i += blockDim.x) prod[i] = a.prod[(long long)e * n + i];
  __syncthreads();
  if (threadIdx.x == 0) {
    // the loads run ahead four at a time; the adds stay in order
    const float4* p4 = reinterpret_cast<const float4*>(prod);
    float acc = 0.f;
#pragma unroll 4
    for (int i = 0; i < n / 4; ++i) {
      const float4 v = p4[i];
      acc = __fadd_rn(acc, v.x);
      acc = __fadd_rn(acc, v.y);
      acc = __fadd_rn(acc, v.z);
      acc = __fadd_rn(acc, v.w);
    }
    a.scores[e] = acc;
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
  cudaError_t e = launch_pdl(pool_q_kernel, dim3(a.heads), dim3(256), 0, s, a);
  if (e == cudaSuccess)
    e = launch_pdl(pool_k_kernel, dim3(a.n_entries, a.heads), dim3(kHeadDim), 0, s, a);
  if (e == cudaSuccess) e = launch_pdl(page_score_kernel, dim3(a.n_entries), dim3(256), 0, s, a);
  if (e == cudaSuccess) e = launch_pdl(select_kernel, dim3(1), dim3(kMaxSampledEntries), 0, s, a);
  count_launches(4);
  return e;
}

}  // namespace pkv
