// Paged attention over a visible page table, and the split-KV combine.
//
// "LingBot-Map Paged KV Cache", sections 1-2: a frame's tokens attend to every
// valid slot of the visible pages (scale -> window -> special, the frame's own
// tokens included); the pages need no mask beyond their valid lengths. The
// attention is bidirectional. vLLM-Omni RFC "Reconstruction Engine", section
// 3.3: a chunk's tokens attend over the in-window chunks the same way.
//
// For query row i and head h: o = sum_j 2^(s_j - m) v_j / sum_j 2^(s_j - m),
// s_j = sm_scale*log2(e) * (q . k_j), accumulated in fp32 with an online
// (running-max) softmax over 64-slot tiles of the table's slots.
//
// This translation unit holds the first, register-tile version of the kernel
// (mma.sync m16n8k16 bf16 tensor-core tiles, cp.async double buffering).
#include <cuda_bf16.h>

#include "pkv_internal.cuh"

namespace pkv {

namespace {

constexpr int kBM = 64;     // query rows per CTA (4 warps x 16)
constexpr int kBN = 64;     // slots per KV tile
constexpr int kThreads = 128;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// smem address of logical 16-byte chunk c of row r in a [rows][64] bf16 tile
// stored with the pool's 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int r, int c) {
  return base + r * 128 + (swizzle_chunk(r, c) << 4);
}

#ifdef PKV_ATTEND_MMA_SYNC
__global__ void __launch_bounds__(kThreads) attend_mma_kernel(const AttendArgs a) {
  __shared__ __align__(1024) uint16_t sQ[kBM * kHeadDim];
  __shared__ __align__(1024) uint16_t sK[2][kBN * kHeadDim];
  __shared__ __align__(1024) uint16_t sV[2][kBN * kHeadDim];
  __shared__ uint32_t sMask[2][2];

  const int mb = blockIdx.x, h = blockIdx.y, split = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.heads, Ps = a.page_size;
  const int t0 = (int)((long long)a.n_tiles * split / a.num_splits);
  const int t1 = (int)((long long)a.n_tiles * (split + 1) / a.num_splits);

  // ---- Q tile (rows beyond n_q are zero)
  for (int i = tid; i < kBM * 8; i += kThreads) {
    const int r = i >> 3, c = i & 7;
    const int row = mb * kBM + r;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < a.n_q)
      v = __ldg(reinterpret_cast<const uint4*>(a.q + ((long long)row * H + h) * kHeadDim + c * 8));
    *reinterpret_cast<uint4*>(&sQ[r * kHeadDim + swizzle_chunk(r, c) * 8]) = v;
  }

  // ---- K/V tile loader: tile j covers flat slots [64j, 64j+64); invalid slots
  // are zero-filled and masked.
  auto load_tile = [&](int j, int buf) {
    const uint32_t k_base = smem_u32(sK[buf]), v_base = smem_u32(sV[buf]);
    for (int i = tid; i < kBN * 8; i += kThreads) {
      const int r = i >> 3, pc = i & 7;          // physical chunk: copied as stored
      const int f = j * kBN + r;
      const int e = f / Ps, slot = f - e * Ps;
      int page = 0;
      bool valid = false;
      if (e < a.n_entries && slot < __ldg(&a.tbl_len[e])) {
        page = __ldg(&a.tbl_idx[e]);
        valid = page >= 0 && page < a.pool_pages;
      }
      const uint16_t* kp = a.pool + (long long)(valid ? page : 0) * a.page_elems +
                           ((long long)h * Ps + slot) * kHeadDim + pc * 8;
      const uint16_t* vp = kp + (long long)H * Ps * kHeadDim;
      cp_async16(k_base + r * 128 + pc * 16, kp, valid ? 16 : 0);
      cp_async16(v_base + r * 128 + pc * 16, vp, valid ? 16 : 0);
    }
    if (tid < kBN) {
      const int f = j * kBN + tid;
      const int e = f / Ps, slot = f - e * Ps;
      const bool valid = e < a.n_entries && slot < __ldg(&a.tbl_len[e]);
      const uint32_t bits = __ballot_sync(0xffffffffu, valid);
      if (lane == 0) sMask[buf][warp] = bits;
    }
  };

  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  if (t0 < t1) load_tile(t0, 0);
  cp_async_commit();
  __syncthreads();

  // Q fragments for this warp's 16 rows, all four 16-wide k-steps.
  uint32_t qa[4][4];
  {
    const uint32_t q_base = smem_u32(sQ);
    const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      ldsm_x4(tile_addr(q_base, r, 2 * kk + (lane >> 4)), qa[kk][0], qa[kk][1], qa[kk][2],
              qa[kk][3]);
  }

  const int g = lane >> 2, tq = lane & 3;
  for (int j = t0; j < t1; ++j) {
    const int buf = (j - t0) & 1;
    if (j + 1 < t1) load_tile(j + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    const uint32_t k_base = smem_u32(sK[buf]), v_base = smem_u32(sV[buf]);
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        const int r = np * 16 + (lane & 7) + (lane >> 4) * 8;
        ldsm_x4(tile_addr(k_base, r, 2 * kk + ((lane >> 3) & 1)), b0, b1, b2, b3);
        mma_bf16(s[2 * np], qa[kk], b0, b1);
        mma_bf16(s[2 * np + 1], qa[kk], b2, b3);
      }
    }

    // mask, scale to log2 domain, online softmax
    const uint32_t mask0 = sMask[buf][0], mask1 = sMask[buf][1];
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = nt * 8 + 2 * tq + (e & 1);
        const uint32_t bits = col < 32 ? mask0 : mask1;
        const bool ok = (bits >> (col & 31)) & 1u;
        s[nt][e] = ok ? s[nt][e] * a.scale_log2 : -INFINITY;
        mx[e >> 1] = fmaxf(mx[e >> 1], s[nt][e]);
      }
    }
    float alpha[2], m_use[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
      mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
      const float m_new = fmaxf(m_run[rr], mx[rr]);
      m_use[rr] = m_new == -INFINITY ? 0.f : m_new;
      alpha[rr] = fast_exp2(m_run[rr] - m_use[rr]);
      m_run[rr] = m_new;
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = fast_exp2(s[nt][e] - m_use[e >> 1]);
        s[nt][e] = p;
        rs[e >> 1] += p;
      }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) l_run[rr] = l_run[rr] * alpha[rr] + rs[rr];
#pragma unroll
    for (int dt = 0; dt < 8; ++dt) {
      o[dt][0] *= alpha[0];
      o[dt][1] *= alpha[0];
      o[dt][2] *= alpha[1];
      o[dt][3] *= alpha[1];
    }
    // O += P V: P from the S accumulators (k = slots), V via transposed ldmatrix
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < 4; ++dp) {
        uint32_t b0, b1, b2, b3;
        const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        ldsm_x4_t(tile_addr(v_base, r, 2 * dp + (lane >> 4)), b0, b1, b2, b3);
        mma_bf16(o[2 * dp], pa, b0, b1);
        mma_bf16(o[2 * dp + 1], pa, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 1);
    l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 2);
  }
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int row = mb * kBM + warp * 16 + g + rr * 8;
    if (row >= a.n_q) continue;
    if (a.num_splits == 1) {
      const float inv = l_run[rr] > 0.f ? 1.f / l_run[rr] : 0.f;
      uint16_t* dst = a.out + ((long long)row * H + h) * kHeadDim;
#pragma unroll
      for (int dt = 0; dt < 8; ++dt)
        *reinterpret_cast<uint32_t*>(dst + dt * 8 + 2 * tq) =
            pack_bf16(o[dt][2 * rr] * inv, o[dt][2 * rr + 1] * inv);
    } else {
      const long long ro = ((long long)split * a.n_q + row) * H + h;
      float* dst = a.part_o + ro * kHeadDim;
#pragma unroll
      for (int dt = 0; dt < 8; ++dt)
        *reinterpret_cast<float2*>(dst + dt * 8 + 2 * tq) =
            make_float2(o[dt][2 * rr], o[dt][2 * rr + 1]);
      if (tq == 0) *reinterpret_cast<float2*>(a.part_ml + ro * 2) = make_float2(m_run[rr], l_run[rr]);
    }
  }
}

#endif  // PKV_ATTEND_MMA_SYNC

// Merge the splits' partial (o, m, l) of each (row, head): one warp per pair,
// two head_dim elements per lane.
__global__ void __launch_bounds__(256) combine_kernel(const AttendArgs a) {
  const int warps_per_block = blockDim.x >> 5;
  const long long pair = (long long)blockIdx.x * warps_per_block + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long n_pairs = (long long)a.n_q * a.heads;
  if (pair >= n_pairs) return;
  const long long split_stride = n_pairs;
  float m_max = -INFINITY;
  for (int s = 0; s < a.num_splits; ++s)
    m_max = fmaxf(m_max, a.part_ml[(s * split_stride + pair) * 2]);
  float l_sum = 0.f, o0 = 0.f, o1 = 0.f;
  for (int s = 0; s < a.num_splits; ++s) {
    const float2 ml = *reinterpret_cast<const float2*>(a.part_ml + (s * split_stride + pair) * 2);
    if (ml.y <= 0.f) continue;
    const float w = fast_exp2(ml.x - m_max);
    const float2 ov =
        *reinterpret_cast<const float2*>(a.part_o + (s * split_stride + pair) * kHeadDim + 2 * lane);
    l_sum += w * ml.y;
    o0 += w * ov.x;
    o1 += w * ov.y;
  }
  const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
  *reinterpret_cast<uint32_t*>(a.out + pair * kHeadDim + 2 * lane) = pack_bf16(o0 * inv, o1 * inv);
}

}  // namespace

int attend_num_splits(int n_q, int heads, long long n_slots, int num_sms) {
#ifdef PKV_ATTEND_MMA_SYNC
  const int n_tiles = (int)((n_slots + kBN - 1) / kBN);
  const int base = ((n_q + kBM - 1) / kBM) * heads;
  int s = (2 * num_sms + base - 1) / base;
  if (s > 16) s = 16;
  if (s > n_tiles) s = n_tiles;
  return s < 1 ? 1 : s;
#else
  return attend_tc_splits(n_q, heads, attend_tc_tiles(n_slots), num_sms);
#endif
}

cudaError_t launch_attend(const AttendArgs& a, int num_sms, cudaStream_t s) {
  (void)num_sms;
#ifdef PKV_ATTEND_MMA_SYNC
  dim3 grid((a.n_q + kBM - 1) / kBM, a.heads, a.num_splits);
  attend_mma_kernel<<<grid, kThreads, 0, s>>>(a);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
#else
  cudaError_t e = launch_attend_tc(a, s);
#endif
  if (e != cudaSuccess || a.num_splits == 1) return e;
  const long long pairs = (long long)a.n_q * a.heads;
  combine_kernel<<<(unsigned)((pairs + 7) / 8), 256, 0, s>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace pkv
