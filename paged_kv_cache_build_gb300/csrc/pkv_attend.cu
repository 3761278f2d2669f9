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

// The call a thread's (query row, head) pair belongs to, and the pair's index in it.
__device__ __forceinline__ const AttendArgs& pair_call(const AttendArgs& a, long long& pair) {
  return a;
}
__device__ __forceinline__ const AttendArgs& pair_call(const AttendBatch& b, long long& pair) {
  int i = 0;
  while (i + 1 < b.n && pair >= b.pair_base[i + 1]) ++i;
  pair -= b.pair_base[i];
  return b.item[i];
}

template <typename Params>
__global__ void __launch_bounds__(256, 2) combine_kernel(const __grid_constant__ Params params,
                                                         long long total_pairs) {
  pdl_wait();
  pdl_trigger();
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  long long pair = gid >> 4;
  const int q4 = (int)(gid & 15);
  if (pair >= total_pairs) return;
  const AttendArgs& a = pair_call(params, pair);
  const long long n_pairs = (long long)a.n_q * a.heads;
  const int S = a.num_splits;
  // Up to kFold splits at a time (a frame's 9 splits in one round): their loads
  // are issued together, then folded into the running max, sum and O. Every
  // split writes its partials (an empty one as max -inf, sum 0, O 0).
  constexpr int kFold = 12;
  float m_run = -INFINITY, l_sum = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < S; s0 += kFold) {
    float2 ml[kFold];
    float4 ov[kFold];
#pragma unroll
    for (int i = 0; i < kFold; ++i) {
      ml[i] = make_float2(-INFINITY, 0.f);
      ov[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (s0 + i < S) {
        const long long sp = (long long)(s0 + i) * n_pairs + pair;
        ml[i] = __ldg(reinterpret_cast<const float2*>(a.part_ml + sp * 2));
        ov[i] = __ldg(reinterpret_cast<const float4*>(a.part_o + sp * kHeadDim) + q4);
      }
    }
#pragma unroll
    for (int i = 0; i < kFold; ++i) {
      if (ml[i].y > 0.f) {
        const float m_new = fmaxf(m_run, ml[i].x);
        const float c = fast_exp2(m_run - m_new);     // 0 while m_run is -inf
        const float w = fast_exp2(ml[i].x - m_new);
        l_sum = l_sum * c + w * ml[i].y;
        o.x = o.x * c + w * ov[i].x;
        o.y = o.y * c + w * ov[i].y;
        o.z = o.z * c + w * ov[i].z;
        o.w = o.w * c + w * ov[i].w;
        m_run = m_new;
      }
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
  const long long pairs = (long long)a.n_q * a.heads;
  e = launch_pdl(combine_kernel<AttendArgs>, dim3((unsigned)((pairs * 16 + 255) / 256)), dim3(256),
                 0, s, a, pairs);
  count_launches(1);
  return e;
}

cudaError_t launch_attend_batch(const AttendBatch& b, cudaStream_t s) {
  cudaError_t e = launch_attend_tc_batch(b, s);
  if (e != cudaSuccess || b.item[0].num_splits == 1) return e;
  const long long pairs = b.pair_base[b.n];
  e = launch_pdl(combine_kernel<AttendBatch>, dim3((unsigned)((pairs * 16 + 255) / 256)), dim3(256),
                 0, s, b, pairs);
  count_launches(1);
  return e;
}

}  // namespace pkv
