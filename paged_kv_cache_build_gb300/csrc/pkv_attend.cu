// Split-KV combine of the paged attention (the attention kernel itself is in
// pkv_attend_tc.cu), and the attention launcher.
//
// "LingBot-Map Paged KV Cache", sections 1-2: a frame's tokens attend to every
// valid slot of the visible pages (scale -> window -> special, the frame's own
// tokens included); the pages need no mask beyond their valid lengths. The
// attention is bidirectional. vLLM-Omni RFC "Reconstruction Engine", section
// 3.3: a chunk's tokens attend over the in-window chunks the same way.
//
// Each KV split leaves, per query row and head, o_s = sum_j 2^(s_j - m_s) v_j and
// l_s = sum_j 2^(s_j - m_s) over its slots (log2-domain scores). The merge is
// o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s with M = max_s m_s.
#include <cuda_bf16.h>

#include "pkv_internal.cuh"

namespace pkv {

namespace {

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Merge the splits' partial (o, m, l) of each (row, head): 16 threads per pair,
// four head_dim elements each; every thread reads all the splits' (m, l) (the 16
// threads of a pair share them through L1) and its four elements of each o.
constexpr int kMaxSplits = 16;

__global__ void __launch_bounds__(256) combine_kernel(const AttendArgs a) {
  const long long n_pairs = (long long)a.n_q * a.heads;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long pair = gid >> 4;
  const int q4 = (int)(gid & 15);
  if (pair >= n_pairs) return;
  const int S = a.num_splits;
  float m[kMaxSplits], l[kMaxSplits];
  float m_max = -INFINITY;
#pragma unroll
  for (int s = 0; s < kMaxSplits; ++s) {
    if (s < S) {
      const float2 ml = __ldg(reinterpret_cast<const float2*>(a.part_ml + (s * n_pairs + pair) * 2));
      m[s] = ml.x;
      l[s] = ml.y;
      if (ml.y > 0.f) m_max = fmaxf(m_max, ml.x);
    }
  }
  float l_sum = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int s = 0; s < kMaxSplits; ++s) {
    if (s < S && l[s] > 0.f) {
      const float w = fast_exp2(m[s] - m_max);
      const float4 ov =
          __ldg(reinterpret_cast<const float4*>(a.part_o + (s * n_pairs + pair) * kHeadDim) + q4);
      l_sum += w * l[s];
      o.x += w * ov.x;
      o.y += w * ov.y;
      o.z += w * ov.z;
      o.w += w * ov.w;
    }
  }
  const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
  *reinterpret_cast<uint2*>(a.out + pair * kHeadDim + 4 * q4) =
      make_uint2(pack_bf16(o.x * inv, o.y * inv), pack_bf16(o.z * inv, o.w * inv));
}

}  // namespace

int attend_num_splits(int n_q, int heads, long long n_slots, int num_sms) {
  return attend_tc_splits(n_q, heads, attend_tc_tiles(n_slots), num_sms);
}

cudaError_t launch_attend(const AttendArgs& a, int num_sms, cudaStream_t s) {
  (void)num_sms;
  cudaError_t e = launch_attend_tc(a, s);
  if (e != cudaSuccess || a.num_splits == 1) return e;
  const long long threads = (long long)a.n_q * a.heads * 16;
  combine_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace pkv
