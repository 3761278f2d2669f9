// Paged attention on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a.
//
// "LingBot-Map Paged KV Cache", sections 1-2: a frame's tokens attend to every
// valid slot of the visible pages (scale -> window -> special, the frame's own
// tokens included), bidirectionally, masked only by each page's valid length.
// vLLM-Omni RFC "Reconstruction Engine", section 3.3: a chunk's tokens attend over
// the in-window chunks the same way.
//
// One CTA computes, for one head, MT M-tiles of 128 query rows against a range of
// 64-slot KV tiles of the visible table (split-KV partials are merged by the
// combine kernel). Roles:
//   warp 0       producer: one 1-D bulk copy (cp.async.bulk) per page block of a
//                tile into a 4-stage shared-memory ring. Pages are stored in the
//                pool already 128-byte swizzled, so a block lands in shared memory
//                as a ready tensor-core operand; no tensor map is needed.
//   warp 1       MMA issuer (one thread): S_m = Q_m K^T into TMEM, then
//                O_m += P_m V into TMEM, software-pipelined so that QK of tile j
//                overlaps the softmax of tile j-1.
//   warps 4..    one warpgroup per M-tile (a thread per query row): reads its S
//                row from TMEM, masks invalid slots, keeps a running max (only
//                raised when it grows by more than 2^8, so O rarely needs
//                rescaling), writes P = 2^(S - m) as bf16 into shared memory and
//                finally reads O from TMEM.
// Every mbarrier wait is bounded; a wait that gives up sets the device error
// word, and the CTA drains its copies and MMAs and frees TMEM before returning.
#include <cuda_bf16.h>

#include "pkv_internal.cuh"

namespace pkv {

namespace {

constexpr int kBN = 64;            // slots per KV tile
constexpr int kStages = 4;         // KV ring depth
// TMEM columns: S_m at 64m, O_m at 64*MT + 64m; the allocation is a power of two.
template <int MT>
struct TmemCols {
  static constexpr int kO = 64 * MT;
  static constexpr int kAlloc = MT == 1 ? 128 : (MT == 2 ? 256 : 512);
};
constexpr uint32_t kSpinLimit = 1u << 25;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int MT>
struct __align__(1024) TcSmem {
  uint8_t q[MT][128 * 128];          // Q_m: 128 rows x 64 bf16, 128B-swizzled
  uint8_t k[kStages][kBN * 128];     // K tile: 64 slots x 64 bf16
  uint8_t v[kStages][kBN * 128];
  uint8_t p[MT][128 * 128];          // P_m: 128 rows x 64 slots bf16
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[MT];
  uint64_t p_full[MT];
  uint64_t o_done[MT];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------- mbarriers
__device__ __forceinline__ void mbar_init(uint64_t* bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Bounded wait: returns false (and raises the CTA's abort flag and the device
// error word) if the phase does not complete within the spin limit, or if
// another role has already aborted.
// Drain waits (in-flight copies and MMAs before TMEM is freed) pass
// honor_abort = false: they are bounded but never cut short.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* err, bool honor_abort = true) {
  const uint32_t addr = smem_u32(bar);
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(addr, parity)) return true;
    if ((i & 255u) == 255u) {
      if (honor_abort && *abort) return false;
      __nanosleep(128);
    }
  }
  atomicOr(err, kErrTimeout);
  *abort = 1;
  return false;
}

// --------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// Shared-memory operand descriptor: 128-byte swizzle, 8-row groups 1024 bytes
// apart (stride byte offset), leading byte offset unused for these shapes,
// descriptor version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;                       // leading byte offset (16 B)
  d |= (uint64_t)(1024u >> 4) << 32;             // stride byte offset
  d |= (uint64_t)1u << 46;                       // version
  d |= (uint64_t)2u << 61;                       // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, bool b_mn_major) {
  return (1u << 4)                                // D: f32
         | (1u << 7)                              // A: bf16
         | (1u << 10)                             // B: bf16
         | ((b_mn_major ? 1u : 0u) << 16)         // B major-ness
         | ((uint32_t)(n >> 3) << 17)             // N / 8
         | ((uint32_t)(m >> 4) << 24);            // M / 16
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_u32(bar))
      : "memory");
}

#define PKV_TMEM_LD16(taddr, r)                                                                  \
  asm volatile(                                                                                  \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"   \
      "%14,%15}, [%16];\n"                                                                       \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),     \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
        "=r"(r[14]), "=r"(r[15])                                                                 \
      : "r"(taddr))

#define PKV_TMEM_ST16(taddr, r)                                                                  \
  asm volatile(                                                                                  \
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"    \
      "%13,%14,%15,%16};\n" ::"r"(taddr),                                                        \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),   \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),         \
      "r"(r[15]))

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
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

// Validity bits of the 64 columns of tile `tile`: slot f = 64*tile + c is valid
// when its table entry exists and the slot is below that page's length.
__device__ __forceinline__ uint64_t tile_mask(const AttendArgs& a, int tile) {
  const int Ps = a.page_size;
  uint64_t mask = 0;
  if (Ps >= kBN) {
    const int f0 = tile * kBN;
    const int e = f0 / Ps, so = f0 - e * Ps;
    if (e < a.n_entries) {
      int n = __ldg(&a.tbl_len[e]) - so;
      n = n < 0 ? 0 : (n > kBN ? kBN : n);
      mask = n == kBN ? ~0ull : ((1ull << n) - 1ull);
    }
  } else {
    const int per = kBN / Ps;
    for (int pp = 0; pp < per; ++pp) {
      const int e = tile * per + pp;
      if (e >= a.n_entries) break;
      int n = __ldg(&a.tbl_len[e]);
      n = n < 0 ? 0 : (n > Ps ? Ps : n);
      const uint64_t bits = n >= 64 ? ~0ull : ((1ull << n) - 1ull);
      mask |= bits << (pp * Ps);
    }
  }
  return mask;
}

template <int MT>
__global__ void __launch_bounds__((4 + 4 * MT) * 32, 1)
    attend_tc_kernel(const AttendArgs a, int n_mgroups) {
  extern __shared__ uint8_t smem_raw[];
  TcSmem<MT>& sm = *reinterpret_cast<TcSmem<MT>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.heads, Ps = a.page_size;

  int bid = blockIdx.x;
  const int mg = bid % n_mgroups;
  bid /= n_mgroups;
  const int h = bid % H;
  const int split = bid / H;
  const int t0 = (int)((long long)a.n_tiles * split / a.num_splits);
  const int t1 = (int)((long long)a.n_tiles * (split + 1) / a.num_splits);
  const int nT = t1 - t0;
  const int row0 = mg * MT * 128;

  // ---- set-up: barriers, zeroed KV ring, Q tiles, TMEM
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int m = 0; m < MT; ++m) {
      mbar_init(&sm.s_full[m], 1);
      mbar_init(&sm.p_full[m], 128);
      mbar_init(&sm.o_done[m], 1);
    }
    mbar_init(&sm.mma_done, 1);
    sm.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  {
    uint4* kv = reinterpret_cast<uint4*>(&sm.k[0][0]);
    const int n16 = 2 * kStages * kBN * 128 / 16;     // k and v rings are contiguous
    for (int i = threadIdx.x; i < n16; i += blockDim.x) kv[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < MT * 128 * 8; i += blockDim.x) {
      const int m = i / (128 * 8), r = (i >> 3) & 127, c = i & 7;
      const int row = row0 + m * 128 + r;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (row < a.n_q)
        val = __ldg(reinterpret_cast<const uint4*>(a.q + ((long long)row * H + h) * kHeadDim + c * 8));
      *reinterpret_cast<uint4*>(&sm.q[m][r * 128 + (swizzle_chunk(r, c) << 4)]) = val;
    }
    fence_proxy_async();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     smem_u32(&sm.tmem_base)),
                 "r"(TmemCols<MT>::kAlloc));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;

  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      int issued_tiles = 0;
      for (int j = 0; j < nT; ++j) {
        const int s = j % kStages;
        if (!mbar_wait(&sm.kv_empty[s], ((j / kStages) & 1) ^ 1, abort, a.err)) break;
        const int tile = t0 + j;
        const int per = Ps >= kBN ? 1 : kBN / Ps;
        const int rows = Ps >= kBN ? kBN : Ps;
        uint32_t bytes = 0;
        for (int pp = 0; pp < per; ++pp)
          if (tile * kBN / Ps + pp < a.n_entries) bytes += 2u * rows * 128u;
        mbar_arrive_expect_tx(&sm.kv_full[s], bytes);
        for (int pp = 0; pp < per; ++pp) {
          const int f0 = tile * kBN + pp * rows;
          const int e = f0 / Ps, so = f0 - e * Ps;
          if (e >= a.n_entries) break;
          int page = __ldg(&a.tbl_idx[e]);
          if (page < 0 || page >= a.pool_pages) {
            atomicOr(a.err, kErrPageRange);
            page = 0;
          }
          const uint16_t* kp = a.pool + (long long)page * a.page_elems +
                               ((long long)h * Ps + so) * kHeadDim;
          const uint16_t* vp = kp + (long long)H * Ps * kHeadDim;
          const uint32_t dk = smem_u32(&sm.k[s][pp * rows * 128]);
          const uint32_t dv = smem_u32(&sm.v[s][pp * rows * 128]);
          const uint32_t mb = smem_u32(&sm.kv_full[s]);
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
              "[%3];\n" ::"r"(dk),
              "l"(kp), "r"((uint32_t)rows * 128u), "r"(mb)
              : "memory");
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
              "[%3];\n" ::"r"(dv),
              "l"(vp), "r"((uint32_t)rows * 128u), "r"(mb)
              : "memory");
        }
        issued_tiles = j + 1;
      }
      // make sure no copy is still landing in shared memory when the CTA ends
      for (int j = issued_tiles - 1; j >= 0 && j >= issued_tiles - kStages; --j)
        mbar_wait(&sm.kv_full[j % kStages], (j / kStages) & 1, abort, a.err, false);
    }
  } else if (warp == 1) {
    // ============================================================= MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdQK = idesc_bf16(128, kBN, false);
      constexpr uint32_t kIdPV = idesc_bf16(128, kHeadDim, true);
      bool ok = true;
      for (int j = 0; j < nT && ok; ++j) {
        const int s = j % kStages;
        if (!mbar_wait(&sm.kv_full[s], (j / kStages) & 1, abort, a.err)) break;
        tc_fence_after();
        const int sp = (j + kStages - 1) % kStages;   // stage of tile j - 1
        // S_m = Q_m K_j^T once the softmax has consumed S_m of tile j - 1
        for (int m = 0; m < MT; ++m) {
          if (j > 0) {
            if (!mbar_wait(&sm.p_full[m], (j - 1) & 1, abort, a.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const uint32_t qa = smem_u32(&sm.q[m][0]), kb = smem_u32(&sm.k[s][0]);
#pragma unroll
          for (int kk = 0; kk < kHeadDim / 16; ++kk)
            tc_mma(tmem + m * kBN, sdesc(qa + kk * 32), sdesc(kb + kk * 32), kIdQK, kk > 0);
          tc_commit(&sm.s_full[m]);
        }
        // O_m += P_m V_{j-1}
        if (ok && j > 0) {
          for (int m = 0; m < MT; ++m) {
            const uint32_t pa = smem_u32(&sm.p[m][0]), vb = smem_u32(&sm.v[sp][0]);
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              tc_mma(tmem + TmemCols<MT>::kO + m * kHeadDim, sdesc(pa + kk * 32), sdesc(vb + kk * 2048), kIdPV,
                     (j > 1 || kk > 0) ? 1u : 0u);
            tc_commit(&sm.o_done[m]);
          }
          tc_commit(&sm.kv_empty[sp]);
        }
      }
      if (ok && nT > 0 && !*abort) {
        const int jl = nT - 1, sl = jl % kStages;
        for (int m = 0; m < MT; ++m) {
          if (!mbar_wait(&sm.p_full[m], jl & 1, abort, a.err)) break;
          tc_fence_after();
          const uint32_t pa = smem_u32(&sm.p[m][0]), vb = smem_u32(&sm.v[sl][0]);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            tc_mma(tmem + TmemCols<MT>::kO + m * kHeadDim, sdesc(pa + kk * 32), sdesc(vb + kk * 2048), kIdPV,
                   (jl > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&sm.o_done[m]);
        }
      }
      // every MMA issued by this thread has completed once mma_done flips
      tc_commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0, abort, a.err, false);
    }
  } else if (warp >= 4) {
    // ================================================================ softmax
    const int m = (warp - 4) >> 2;
    const int wq = warp & 3;                       // TMEM lane quarter of this warp
    const int r = wq * 32 + lane;                  // row inside the M-tile
    const int row = row0 + m * 128 + r;
    const bool warp_active = row0 + m * 128 + wq * 32 < a.n_q;
    const uint32_t t_lane = (uint32_t)(wq * 32) << 16;
    const uint32_t t_s = tmem + t_lane + m * kBN;
    const uint32_t t_o = tmem + t_lane + TmemCols<MT>::kO + m * kHeadDim;
    uint8_t* p_row = &sm.p[m][r * 128];
    float m_run = -INFINITY, l_run = 0.f;
    bool alive = true;
    for (int j = 0; j < nT; ++j) {
      if (!mbar_wait(&sm.s_full[m], j & 1, abort, a.err)) {
        alive = false;
        break;
      }
      tc_fence_after();
      uint32_t packed[32];
      bool rescale = false;
      float alpha = 1.f;
      if (warp_active) {
        const uint64_t mask = tile_mask(a, t0 + j);
        float s[kBN];
#pragma unroll
        for (int c = 0; c < kBN; c += 16) {
          uint32_t* rr = reinterpret_cast<uint32_t*>(&s[c]);
          PKV_TMEM_LD16(t_s + c, rr);
        }
        tmem_wait_ld();
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kBN; ++c) {
          s[c] = ((mask >> c) & 1ull) ? s[c] * a.scale_log2 : -INFINITY;
          mx = fmaxf(mx, s[c]);
        }
        const float m_new = fmaxf(m_run, mx);
        if (m_run == -INFINITY) {
          m_run = m_new;
        } else if (m_new > m_run + kRescaleThreshold) {
          alpha = fast_exp2(m_run - m_new);
          l_run *= alpha;
          m_run = m_new;
          rescale = true;
        }
        const float m_ref = m_run == -INFINITY ? 0.f : m_run;
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < kBN; c += 2) {
          const uint32_t pk = pack_bf16(fast_exp2(s[c] - m_ref), fast_exp2(s[c + 1] - m_ref));
          packed[c >> 1] = pk;
          __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&pk);
          const float2 f = __bfloat1622float2(b);
          sum += f.x + f.y;
        }
        l_run += sum;
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) packed[c] = 0u;
      }
      if (j > 0) {
        if (!mbar_wait(&sm.o_done[m], (j - 1) & 1, abort, a.err)) {
          alive = false;
          break;
        }
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O_m *= alpha for this row (alpha = 1 for rows that keep their max)
#pragma unroll
        for (int c = 0; c < kHeadDim; c += 16) {
          uint32_t o[16];
          PKV_TMEM_LD16(t_o + c, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          PKV_TMEM_ST16(t_o + c, o);
        }
        tmem_wait_st();
      }
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(p_row + (swizzle_chunk(r, c) << 4)) =
            make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&sm.p_full[m]);
    }
    // ---- epilogue
    float o[kHeadDim];
#pragma unroll
    for (int c = 0; c < kHeadDim; ++c) o[c] = 0.f;
    if (alive && nT > 0) {
      if (mbar_wait(&sm.o_done[m], (nT - 1) & 1, abort, a.err)) {
        tc_fence_after();
        if (warp_active) {
#pragma unroll
          for (int c = 0; c < kHeadDim; c += 16) {
            uint32_t* rr = reinterpret_cast<uint32_t*>(&o[c]);
            PKV_TMEM_LD16(t_o + c, rr);
          }
          tmem_wait_ld();
        }
      } else {
        alive = false;
      }
    }
    if (row < a.n_q && alive) {
      if (a.num_splits == 1) {
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        uint4* dst = reinterpret_cast<uint4*>(a.out + ((long long)row * H + h) * kHeadDim);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          dst[c] = make_uint4(pack_bf16(o[8 * c] * inv, o[8 * c + 1] * inv),
                              pack_bf16(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                              pack_bf16(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                              pack_bf16(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
      } else {
        const long long ro = ((long long)split * a.n_q + row) * H + h;
        float4* dst = reinterpret_cast<float4*>(a.part_o + ro * kHeadDim);
#pragma unroll
        for (int c = 0; c < 16; ++c)
          dst[c] = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
        *reinterpret_cast<float2*>(a.part_ml + ro * 2) = make_float2(m_run, l_run);
      }
    }
  }

  // ---- teardown: every role has finished its waits; free TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                 "r"(TmemCols<MT>::kAlloc));
  }
}

template <int MT>
cudaError_t launch_mt(const AttendArgs& a, int n_mgroups, cudaStream_t s) {
  const size_t smem = sizeof(TcSmem<MT>) + 1024;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel<MT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int grid = n_mgroups * a.heads * a.num_splits;
  attend_tc_kernel<MT><<<grid, (4 + 4 * MT) * 32, smem, s>>>(a, n_mgroups);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

// M-tiles per CTA for n_q query rows.
int attend_tc_mt(int n_q) { return n_q <= 128 ? 1 : (n_q <= 256 ? 2 : 3); }

// Split-KV factor: fill the SMs in as few, as even waves as possible.
int attend_tc_splits(int n_q, int heads, int n_tiles, int num_sms) {
  const int mt = attend_tc_mt(n_q);
  const int groups = (n_q + mt * 128 - 1) / (mt * 128);
  const int base = groups * heads;
  int best = 1;
  double best_eff = 0.0;
  for (int s = 1; s <= 16; ++s) {
    if (s > 1 && n_tiles / s < 4) break;
    const int ctas = base * s;
    const int waves = (ctas + num_sms - 1) / num_sms;
    // a wave's time is proportional to the tiles each CTA handles
    const double t = (double)waves * ((double)n_tiles / s);
    const double eff = (double)base * n_tiles / (t * num_sms);
    if (eff > best_eff * 1.03) {
      best_eff = eff;
      best = s;
    }
  }
  return best;
}

cudaError_t launch_attend_tc(const AttendArgs& a, cudaStream_t s) {
  const int mt = attend_tc_mt(a.n_q);
  const int n_mgroups = (a.n_q + mt * 128 - 1) / (mt * 128);
  switch (mt) {
    case 1: return launch_mt<1>(a, n_mgroups, s);
    case 2: return launch_mt<2>(a, n_mgroups, s);
    default: return launch_mt<3>(a, n_mgroups, s);
  }
}

}  // namespace pkv
