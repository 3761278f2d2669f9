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
//   warp 2       producer: one 1-D bulk copy (cp.async.bulk) per page block of a
//                tile into a 4-stage shared-memory ring. Pages are stored in the
//                pool already 128-byte swizzled, so a block lands in shared memory
//                as a ready tensor-core operand; no tensor map is needed.
//   warp 3       MMA issuer (one thread): S_m = Q_m K^T into TMEM, then
//                O_m += P_m V into TMEM, software-pipelined so that QK of tile j
//                overlaps the softmax of tile j-1.
//   warps 4..    one warpgroup per M-tile (a thread per query row; warp 0 alone
//                for a last M-tile of at most 32 valid rows): reads its S
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
  uint64_t s_free[MT];
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
// Non-blocking probe of a phase.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
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

// Warp roles: warp 2 produces, warp 3 issues MMAs, warps 4.. are the softmax
// warpgroups of M-tiles 0, 1, ... (warp w reads TMEM lane quarter w % 4). When
// the last M-tile's valid rows fit in one 32-row lane quarter (LAST == 1, a
// frame's 262 rows), that tile gets a single softmax warp: warp 0. This keeps
// the block at 12 warps or fewer, i.e. at most 3 warps per SM sub-partition,
// so each thread may use up to 168 registers.
template <int MT, int LAST>
constexpr int tc_threads() { return (LAST == 1 ? 4 * MT : 4 + 4 * MT) * 32; }
constexpr int kProducerWarp = 2;
constexpr int kMmaWarp = 3;

template <int MT, int LAST>
__global__ void __launch_bounds__(tc_threads<MT, LAST>(), 1)
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
      const int arrivals = m == MT - 1 ? 32 * LAST : 128;
      mbar_init(&sm.s_free[m], arrivals);
      mbar_init(&sm.p_full[m], arrivals);
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
    if (LAST < 4) {
      // rows of the last P tile that no softmax warp writes stay zero
      uint4* pl = reinterpret_cast<uint4*>(&sm.p[MT - 1][32 * LAST * 128]);
      for (int i = threadIdx.x; i < (128 - 32 * LAST) * 8; i += blockDim.x)
        pl[i] = make_uint4(0u, 0u, 0u, 0u);
    }
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
  if (warp == kMmaWarp) {
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

  int m = -1, wq = 0;                              // softmax role: M-tile and lane quarter
  if (warp >= 4) {
    m = (warp - 4) >> 2;
    wq = warp & 3;
  } else if (LAST == 1 && warp == 0) {
    m = MT - 1;
  }

  if (warp == kProducerWarp) {
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
  } else if (warp == kMmaWarp) {
    // ============================================================= MMA issuer
    // Event-driven: each sweep issues every QK and PV whose inputs are ready,
    // so a slow M-tile never holds back the others.
    //   QK(m, j) needs tile j in shared memory and S_m released by the softmax
    //            (it copies S_m to registers before doing any arithmetic);
    //   PV(m, j) needs P_m of tile j written;
    //   stage of tile j is released once PV(m, j) is issued for every m.
    if (lane == 0) {
      constexpr uint32_t kIdQK = idesc_bf16(128, kBN, false);
      constexpr uint32_t kIdPV = idesc_bf16(128, kHeadDim, true);
      int qk_next[MT], pv_next[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) qk_next[m] = pv_next[m] = 0;
      int loaded = 0, released = 0, done = 0;
      uint32_t idle = 0;
      while (done < MT && !*abort) {
        bool progress = false;
        if (loaded < nT) {
          int lo = nT;
#pragma unroll
          for (int m = 0; m < MT; ++m) lo = min(lo, qk_next[m]);
          if (loaded <= lo + 1 &&
              mbar_test_wait(&sm.kv_full[loaded % kStages], (loaded / kStages) & 1)) {
            ++loaded;
            progress = true;
            tc_fence_after();
          }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const int j = qk_next[m];
          if (j < loaded && (j == 0 || mbar_test_wait(&sm.s_free[m], (j - 1) & 1))) {
            tc_fence_after();
            const uint32_t qa = smem_u32(&sm.q[m][0]);
            const uint32_t kb = smem_u32(&sm.k[j % kStages][0]);
#pragma unroll
            for (int kk = 0; kk < kHeadDim / 16; ++kk)
              tc_mma(tmem + m * kBN, sdesc(qa + kk * 32), sdesc(kb + kk * 32), kIdQK, kk > 0);
            tc_commit(&sm.s_full[m]);
            qk_next[m] = j + 1;
            progress = true;
          }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const int j = pv_next[m];
          if (j < qk_next[m] && mbar_test_wait(&sm.p_full[m], j & 1)) {
            tc_fence_after();
            const uint32_t pa = smem_u32(&sm.p[m][0]);
            const uint32_t vb = smem_u32(&sm.v[j % kStages][0]);
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              tc_mma(tmem + TmemCols<MT>::kO + m * kHeadDim, sdesc(pa + kk * 32),
                     sdesc(vb + kk * 2048), kIdPV, (j > 0 || kk > 0) ? 1u : 0u);
            tc_commit(&sm.o_done[m]);
            pv_next[m] = j + 1;
            if (j + 1 == nT) ++done;
            progress = true;
          }
        }
        int lo = nT;
#pragma unroll
        for (int m = 0; m < MT; ++m) lo = min(lo, pv_next[m]);
        while (released < lo) {
          tc_commit(&sm.kv_empty[released % kStages]);
          ++released;
        }
        if (nT == 0) break;
        if (progress) {
          idle = 0;
        } else if (++idle > kSpinLimit) {
          atomicOr(a.err, kErrTimeout);
          *abort = 1;
        } else if ((idle & 255u) == 255u) {
          __nanosleep(64);
        }
      }
      // every MMA issued by this thread has completed once mma_done flips
      tc_commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0, abort, a.err, false);
    }
  } else if (m >= 0) {
    // ================================================================ softmax
    const int r = wq * 32 + lane;                  // row inside the M-tile
    const int row = row0 + m * 128 + r;
    const bool warp_active = row0 + m * 128 + wq * 32 < a.n_q;
    const uint32_t t_lane = (uint32_t)(wq * 32) << 16;
    const uint32_t t_s = tmem + t_lane + m * kBN;
    const uint32_t t_o = tmem + t_lane + TmemCols<MT>::kO + m * kHeadDim;
    uint8_t* p_row = &sm.p[m][r * 128];
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;          // running max (log2 units) and sum
    bool alive = true;
    for (int j = 0; j < nT; ++j) {
      if (!mbar_wait(&sm.s_full[m], j & 1, abort, a.err)) {
        alive = false;
        break;
      }
      tc_fence_after();
      bool rescale = false;
      float alpha = 1.f;
      float s[kBN];
      if (warp_active) {
#pragma unroll
        for (int c = 0; c < kBN; c += 16) {
          uint32_t* rr = reinterpret_cast<uint32_t*>(&s[c]);
          PKV_TMEM_LD16(t_s + c, rr);
        }
        tmem_wait_ld();
      }
      // S_m is in registers: the next QK may overwrite it
      tc_fence_before();
      mbar_arrive(&sm.s_free[m]);
      if (warp_active) {
        const uint64_t mask = tile_mask(a, t0 + j);
        if (mask != ~0ull) {
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (!((mask >> c) & 1ull)) s[c] = -INFINITY;
        }
        float mx0 = s[0], mx1 = s[1];
#pragma unroll
        for (int c = 2; c < kBN; c += 2) {
          mx0 = fmaxf(mx0, s[c]);
          mx1 = fmaxf(mx1, s[c + 1]);
        }
        const float mx = fmaxf(mx0, mx1) * sl2;      // sl2 > 0: max commutes with scaling
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
        float sum0 = 0.f, sum1 = 0.f;
        // P packed as bf16 pairs, compacted in place into s[0 .. kBN/2)
#pragma unroll
        for (int c = 0; c < kBN; c += 2) {
          const float p0 = fast_exp2(fmaf(s[c], sl2, -m_ref));
          const float p1 = fast_exp2(fmaf(s[c + 1], sl2, -m_ref));
          s[c >> 1] = __uint_as_float(pack_bf16(p0, p1));
          sum0 += p0;
          sum1 += p1;
        }
        l_run += sum0 + sum1;
      } else {
#pragma unroll
        for (int c = 0; c < kBN / 2; ++c) s[c] = 0.f;
      }
      // PV of the previous tile must be done before P_m is overwritten and
      // before O_m is rescaled
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
            make_uint4(__float_as_uint(s[4 * c]), __float_as_uint(s[4 * c + 1]),
                       __float_as_uint(s[4 * c + 2]), __float_as_uint(s[4 * c + 3]));
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&sm.p_full[m]);
    }
    // ---- epilogue: O_m row to the output (or the split's partial), 16 columns at a time
    bool have_o = false;
    if (alive && nT > 0) {
      have_o = mbar_wait(&sm.o_done[m], (nT - 1) & 1, abort, a.err);
      if (have_o) tc_fence_after();
    }
    const bool write = alive && row < a.n_q && (have_o || nT == 0);
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    const long long ro = ((long long)split * a.n_q + row) * H + h;
#pragma unroll
    for (int c = 0; c < kHeadDim; c += 16) {
      uint32_t o[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i] = 0u;
      if (have_o && warp_active) {
        PKV_TMEM_LD16(t_o + c, o);
        tmem_wait_ld();
      }
      if (!write) continue;
      if (a.num_splits == 1) {
        uint4* dst = reinterpret_cast<uint4*>(a.out + ((long long)row * H + h) * kHeadDim + c);
#pragma unroll
        for (int q4 = 0; q4 < 2; ++q4) {
          const float* f = reinterpret_cast<const float*>(&o[8 * q4]);
          dst[q4] = make_uint4(pack_bf16(f[0] * inv, f[1] * inv), pack_bf16(f[2] * inv, f[3] * inv),
                               pack_bf16(f[4] * inv, f[5] * inv), pack_bf16(f[6] * inv, f[7] * inv));
        }
      } else {
        uint4* dst = reinterpret_cast<uint4*>(a.part_o + ro * kHeadDim + c);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          dst[q4] = make_uint4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
      }
    }
    if (write && a.num_splits > 1)
      *reinterpret_cast<float2*>(a.part_ml + ro * 2) = make_float2(m_run, l_run);
  }

  // ---- teardown: every role has finished its waits; free TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                 "r"(TmemCols<MT>::kAlloc));
  }
}

template <int MT, int LAST>
cudaError_t launch_mt(const AttendArgs& a, int n_mgroups, cudaStream_t s) {
  const size_t smem = sizeof(TcSmem<MT>) + 1024;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel<MT, LAST>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int grid = n_mgroups * a.heads * a.num_splits;
  attend_tc_kernel<MT, LAST><<<grid, tc_threads<MT, LAST>(), smem, s>>>(a, n_mgroups);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

// M-tiles per CTA for n_q query rows: one M-group of up to three tiles when the
// rows fit (a frame's tokens), else groups of two tiles (a chunk's tokens).
int attend_tc_mt(int n_q) { return n_q <= 128 ? 1 : (n_q <= 256 ? 2 : (n_q <= 384 ? 3 : 2)); }

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
  // one softmax warp for the last M-tile when a single M-group's last tile has <= 32 rows
  const bool thin = n_mgroups == 1 && a.n_q - (mt - 1) * 128 <= 32;
  switch (mt * 2 + (thin ? 1 : 0)) {
    case 3: return launch_mt<1, 1>(a, n_mgroups, s);
    case 2: return launch_mt<1, 4>(a, n_mgroups, s);
    case 5: return launch_mt<2, 1>(a, n_mgroups, s);
    case 4: return launch_mt<2, 4>(a, n_mgroups, s);
    case 7: return launch_mt<3, 1>(a, n_mgroups, s);
    default: return launch_mt<3, 4>(a, n_mgroups, s);
  }
}

}  // namespace pkv
