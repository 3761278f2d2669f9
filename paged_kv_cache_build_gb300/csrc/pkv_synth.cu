// Device-side synthetic input generator (not part of the cache).
//
// Each bf16 value is a function of a 64-bit key packing (seed, workload,
// stream, layer, frame, tensor, token, head, d): the splitmix64 output for that
// key (Steele, Lea and Flood, OOPSLA 2014; 64-bit finaliser constants as
// published by Vigna) is cut into four 16-bit uniforms whose centred sum is
// scaled by 2^-16 (exact) and by 1.7320508 (one fp32 round-to-nearest
// multiply), then by a power-of-two scale (exact), and rounded to bf16 with
// round-to-nearest-even. Every step is exact or one correctly rounded IEEE
// operation, so a faithful host implementation produces the same bits.
#include <cuda_bf16.h>

#include "pkv_internal.cuh"

namespace pkv {

namespace {

__device__ __forceinline__ unsigned long long splitmix64(unsigned long long x) {
  unsigned long long z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void __launch_bounds__(256) synth_kernel(uint16_t* dst, long long total, int n_tokens,
                                                    int heads, int head_dim,
                                                    unsigned long long key_base, int frame0,
                                                    int token0, float scale) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    long long r = i;
    const int d = (int)(r % head_dim);
    r /= head_dim;
    const int h = (int)(r % heads);
    r /= heads;
    const int t = (int)(r % n_tokens);
    const int f = (int)(r / n_tokens);
    const unsigned long long key = key_base | ((unsigned long long)(frame0 + f) << 27) |
                                   ((unsigned long long)(token0 + t) << 11) |
                                   ((unsigned long long)h << 6) | (unsigned long long)d;
    const unsigned long long z = splitmix64(key);
    const int s = (int)(z & 0xFFFF) + (int)((z >> 16) & 0xFFFF) + (int)((z >> 32) & 0xFFFF) +
                  (int)((z >> 48) & 0xFFFF);
    float x = __fmul_rn((float)(s - 131070), 1.52587890625e-05f);   // 2^-16, exact
    x = __fmul_rn(x, 1.7320508f);
    x = __fmul_rn(x, scale);                                          // power of two, exact
    dst[i] = __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
}

}  // namespace

cudaError_t launch_synth(uint16_t* dst, int n_frames, int n_tokens, int heads, int head_dim,
                         unsigned long long key_base, int frame0, int token0, float scale,
                         cudaStream_t s) {
  const long long total = (long long)n_frames * n_tokens * heads * head_dim;
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  synth_kernel<<<(unsigned)blocks, 256, 0, s>>>(dst, total, n_tokens, heads, head_dim, key_base,
                                                frame0, token0, scale);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace pkv
