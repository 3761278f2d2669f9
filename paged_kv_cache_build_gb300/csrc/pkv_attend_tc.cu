// Paged attention on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a.
//
// "LingBot-Map Paged KV Cache", sections 1-2: a frame's tokens attend to every
// valid slot of the visible pages (scale -> window -> special, the frame's own
// tokens included), bidirectionally, masked only by each page's valid length.
// vLLM-Omni RFC "Reconstruction Engine", section 3.3: a chunk's tokens attend over
// the in-window chunks the same way. The same RFC, sections 2.2 and 3.3: frame
// attention, each frame's tokens attending to their own frame only, alternates
// with the global attention; here the keys and values are the frame's dense
// [tokens][heads][64] tensors, read by TMA through tensor maps.
//
// One CTA computes, for one head, MT (1 or 2) M-tiles of 128 query rows, plus
// up to 8 extra rows, against a range of 64-slot KV tiles of the visible table
// (split-KV partials are merged by the combine kernel). A frame's 262 tokens
// are two M-tiles plus 6 extra rows. Roles:
//   warp 2       producer: one 1-D bulk copy (cp.async.bulk) per page block of a
//                tile into an 8-stage shared-memory ring, plus the tile's 64-bit
//                slot-validity mask. Pages are stored in the pool already
//                128-byte swizzled, so a block lands in shared memory as a ready
//                tensor-core operand; no tensor map is needed. Frame attention
//                instead loads each 64-token K and V tile with one 3-D tensor
//                copy (cp.async.bulk.tensor) whose 128-byte swizzle gives the
//                same operand layout.
//   warps 3, 1   MMA issuers (one thread each, one per M-tile): S_m = Q_m K^T
//                (N = 64 slots) into one of three TMEM buffers, and O_m += P_m V
//                with P_m read from the same buffer, where the softmax wrote it.
//   warps 4..11  one warpgroup per M-tile (a thread per query row): reads its S
//                row from TMEM, masks invalid slots, exponentiates against the
//                row's running reference max (moved to the row max on the first
//                tile and when the row's sum would exceed 2^64), writes P =
//                2^(S - m) as bf16 into TMEM, where PV takes its A operand, and at
//                the end reads O from TMEM.
//   warps 0, 12-14  the extra rows (at most 8, if any), every fourth tile per
//                warp, through warp-level mma.sync tiles held in registers; an
//                M = 128 tensor-core tile for 6 rows would cost as much as a
//                full one.
//   FP8 pages    a staging ring of codes and row exponents, dequantized into the
//                bf16 ring by one more warp and either the producer (no extra
//                rows) or three of the extra-row warps.
// With three S buffers per M-tile (P written in place), QK of tile j+3 is
// issued as soon as the softmax releases tile j, and PV of tile j runs while the
// softmax works on tile j+1; the softmax and the tensor-core queue set the pace.
// Every mbarrier wait is bounded; a wait that gives up sets the device error
// word, and the CTA drains its copies and MMAs and frees TMEM before returning.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <type_traits>

#include "pkv_internal.cuh"

namespace pkv {

namespace {

constexpr int kBN = kTileSlots;    // slots per KV tile (64)
constexpr int kMaxMaskTiles = 512; // tiles of a CTA whose slot masks are precomputed
constexpr int kStages = 8;         // KV ring depth
constexpr int kXRows = 8;          // extra query rows handled with mma.sync
constexpr int kXWarps = 4;         // extra-row warps: every fourth tile each
static_assert(kStages % kXWarps == 0, "a stage's tiles belong to one extra-row warp");
// S buffers per M-tile: tile j uses buffer j % kSBufs, and P of the tile (bf16
// pairs) is written over the first 32 columns of its own S buffer.
constexpr int kSBufs = 3;
// TMEM columns: S_m buffer b (fp32, 64 columns) at 64 (kSBufs m + b), O_m (fp32)
// at 64 kSBufs MT + 64 m; 512 columns for two M-tiles, 256 for one.
template <int MT>
struct TmemCols {
  static __host__ __device__ constexpr int s(int m, int b) { return kBN * (kSBufs * m + b); }
  static __host__ __device__ constexpr int o(int m) { return kBN * kSBufs * MT + kHeadDim * m; }
  static constexpr int kAlloc = MT == 1 ? 256 : 512;
};
static_assert(TmemCols<2>::o(1) + kHeadDim <= 512 && TmemCols<1>::o(0) + kHeadDim <= 256 &&
                  TmemCols<2>::s(1, kSBufs - 1) + kBN <= 512,
              "TMEM plan");
constexpr uint32_t kSpinLimit = 1u << 25;
// A tile is exponentiated against the running reference max; if a row's sum of
// 2^(s - m) exceeds 2^64 (or overflows), the row's reference moves to its max.
constexpr float kSumLimit = 18446744073709551616.0f;   // 2^64

// FP8 pages: the producer bulk-copies a tile's E4M3 codes and row exponents into
// a staging ring, one copy per row block of K and of V (the page's layout: B rows
// of 64 code bytes, then their B exponents), and warps dequantize them into the
// bf16 operand ring. Without extra rows the producer converts the K rows and one
// more warp the V rows. With extra rows the producer only stages, and four warps
// (three extra-row warps and one more, one per SM sub-partition) each convert the
// K and V rows of one 16-slot quarter of the tile, one row per lane; the extra-row
// warps convert three tiles ahead of the tile they work on.
constexpr int kF8Stages = 4;
template <bool EXTRA>
constexpr int kF8Deq = EXTRA ? 4 : 2;      // dequantizing warps (arrivals per stage)
template <bool FP8>
struct __align__(128) F8Ring {
  alignas(128) uint8_t k[kF8Stages][kBN * (kHeadDim + 1)];   // K row blocks, as in the page
  alignas(128) uint8_t v[kF8Stages][kBN * (kHeadDim + 1)];
  int nblk[kF8Stages];                     // page blocks copied into the stage
  uint64_t full[kF8Stages];                // the stage's copies have landed
  uint64_t free_[kF8Stages];               // every dequantizing warp is done with it
};
template <>
struct F8Ring<false> {
  uint64_t unused;
};
static_assert(sizeof(F8Ring<true>) % 128 == 0, "staging ring alignment");


template <int MT, bool FP8 = false>
struct __align__(1024) TcSmem {
  uint8_t q[MT][128 * 128];          // Q_m: 128 rows x 64 bf16, 128B-swizzled
  uint8_t k[kStages][kBN * 128];     // K tile: 64 slots x 64 bf16
  uint8_t v[kStages][kBN * 128];
  float xo[kXWarps][kXRows][kHeadDim];  // extra rows: each warp's partial O ...
  float xml[kXWarps][kXRows][2];        // ... and its running max and sum
  uint64_t tmask[kMaxMaskTiles];     // slot validity of the CTA's tiles (precomputed)
  uint16_t kept[kMaxSampledEntries]; // a sampled call's kept table positions
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[MT][kSBufs];       // S_m of the buffer's latest tile is in TMEM
  uint64_t p_full[MT][kSBufs];       // P_m of the buffer's latest tile written, O_m rescaled
  uint64_t o_done[MT];               // a PV of the last three tiles has completed (to rescale O)
  uint64_t mma_done[MT];
  uint64_t x_done;                   // the extra-row warps have published their partials
  F8Ring<FP8> f8;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(TcSmem<2, true>) + 1024 <= 232448, "shared memory of the largest variant");

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
// Non-blocking test of a phase: far cheaper than try_wait when the phase has
// already completed (try_wait first suspends for a while even then).
__device__ __forceinline__ bool mbar_test(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
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
  if (mbar_test(addr, parity)) return true;
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
// Same, with the A operand in TMEM (128 lanes = rows, K packed two bf16 per column).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_u32(bar))
      : "memory");
}

// One box of a 3-D tensor map (coordinates innermost first) into shared memory,
// completing on `mbar` with the box's bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
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

#define PKV_TMEM_LD32(taddr, r)                                                                  \
  asm volatile(                                                                                  \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"   \
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"      \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),     \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),           \
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),           \
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])            \
      : "r"(taddr))

#define PKV_TMEM_ST32(taddr, r)                                                                  \
  asm volatile(                                                                                  \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"    \
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::  \
          "r"(taddr),                                                                            \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),   \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),         \
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),       \
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),       \
      "r"(r[29]), "r"(r[30]), "r"(r[31]))

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

// Legacy warp-level tensor-core helpers for the extra rows.
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
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// shared address of logical 16-byte chunk c of row r of a [rows][64] swizzled tile
__device__ __forceinline__ uint32_t sw_addr(uint32_t base, int r, int c) {
  return base + r * 128 + (swizzle_chunk(r, c) << 4);
}

// Warps: 0 extra rows, 1 MMA issuer (M-tile 1), 2 producer, 3 MMA issuer
// (M-tile 0), 4 .. 4 + 4 MT - 1 softmax, then kXWarps - 1 more extra-row warps,
// then (FP8 pages) one more dequantizing warp.
template <int MT, bool EXTRA, bool FP8 = false>
__host__ __device__ constexpr int tc_threads() {
  return (4 + 4 * MT + (EXTRA ? kXWarps - 1 : 0) + (FP8 ? 1 : 0)) * 32;
}
template <int MT, bool EXTRA>
__host__ __device__ constexpr int tc_conv_warp() {
  return 4 + 4 * MT + (EXTRA ? kXWarps - 1 : 0);
}
constexpr int kXWarp = 0;
constexpr int kProducerWarp = 2;
constexpr int kMmaWarp = 3;          // MMA issuer of M-tile 0 (and TMEM owner)
constexpr int kMmaWarp2 = 1;         // MMA issuer of M-tile 1

// The call a CTA works on: the launch's only one, or its stream's in a batch,
// or (frame attention) its frame.
struct CtaWork {
  const AttendArgs* a;
  int bid, n_mgroups, n_tiles;
  int frame;                        // frame attention: the CTA's frame; else 0
};
__device__ __forceinline__ CtaWork cta_work(const AttendArgs& a, int n_mgroups, int n_tiles) {
  return {&a, (int)blockIdx.x, n_mgroups, n_tiles, 0};
}
__device__ __forceinline__ CtaWork cta_work(const AttendBatch& b, int, int) {
  int i = 0;
  while (i + 1 < b.n && (int)blockIdx.x >= b.cta_base[i + 1]) ++i;
  return {&b.item[i], (int)blockIdx.x - b.cta_base[i], b.n_mgroups[i], b.n_tiles[i], 0};
}
__device__ __forceinline__ CtaWork cta_work(const AttendDense& d, int n_mgroups, int n_tiles) {
  const int per_frame = n_mgroups * d.a.heads;
  return {&d.a, (int)blockIdx.x % per_frame, n_mgroups, n_tiles, (int)blockIdx.x / per_frame};
}

// Valid slots of a tile (bit i: slot i): dense frames by the frame's token count;
// paged tables by each page block's valid length, from the table's counters and,
// for a sampled call, the kept list in shared memory. Reads no device memory
// beyond the kernel's parameters.
template <bool kDense>
__device__ __forceinline__ uint64_t tile_mask(const AttendArgs& a, const uint16_t* kept, int tile) {
  if (kDense) {
    const int n = min(kBN, a.n_q - tile * kBN);
    return n >= kBN ? ~0ull : ((1ull << n) - 1ull);
  }
  const int Ps = a.page_size;
  const int rows = Ps >= kBN ? kBN : Ps;
  const int per = kBN / rows;
  uint64_t bits = 0ull;
  for (int pp = 0; pp < per; ++pp) {
    const int f0 = tile * kBN + pp * rows;
    const int e = f0 / Ps, so = f0 - e * Ps;
    if (e >= a.n_entries) break;
    int n = table_len(a.tbl, a.sampled ? (int)kept[e] : e) - so;
    n = n < 0 ? 0 : (n > rows ? rows : n);
    if (n > 0) bits |= (n == 64 ? ~0ull : ((1ull << n) - 1ull)) << (pp * rows);
  }
  return bits;
}

// FP8 pages are staged as row blocks of B rows: the B rows' 64 code bytes, then
// their B exponents. decode(code) is exact in f16, f16 -> fp32 is exact, and the
// power-of-two scale and the final bf16 rounding are exact for these values (at
// most 4 significant bits).
__device__ __forceinline__ float fp8_row_scale(const uint8_t* blk, int B, int rb) {
  return __uint_as_float((uint32_t)(127 + (int8_t)blk[B * kHeadDim + rb]) << 23);   // 2^e, |e| <= 126
}
// 16 codes -> 16 bf16 (8 pairs)
__device__ __forceinline__ void fp8_convert16(uint4 in, float sc, uint32_t out[8]) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int hw = 0; hw < 2; ++hw) {
      const uint16_t pair = (uint16_t)(w[i] >> (16 * hw));
      uint32_t h2;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(h2) : "h"(pair));
      const float lo = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * sc;
      const float hi = __half2float(__ushort_as_half((unsigned short)(h2 >> 16))) * sc;
      out[2 * i + hw] = pack_bf16(lo, hi);
    }
  }
}
// values 16 q .. 16 q + 15 of row r, into their two 16-byte chunks of the
// 128-byte-swizzled bf16 row
__device__ __forceinline__ void fp8_store16(uint8_t* dst, int r, int q, const uint32_t out[8]) {
  uint8_t* row = dst + r * 128;
  *reinterpret_cast<uint4*>(row + (swizzle_chunk(r, 2 * q) << 4)) = make_uint4(out[0], out[1], out[2], out[3]);
  *reinterpret_cast<uint4*>(row + (swizzle_chunk(r, 2 * q + 1) << 4)) =
      make_uint4(out[4], out[5], out[6], out[7]);
}
// row r (64 values); the row's 64 codes are loaded before any is converted. One
// out-of-line copy serves every converting warp, which keeps the kernel's
// instruction footprint small.
__device__ __noinline__ void fp8_dequant_row(const uint8_t* stage, int B, uint8_t* dst, int r) {
  const uint8_t* blk = stage + (r / B) * B * (kHeadDim + 1);
  const int rb = r % B;
  const float sc = fp8_row_scale(blk, B, rb);
  uint4 in[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) in[q] = *reinterpret_cast<const uint4*>(blk + rb * kHeadDim + 16 * q);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t out[8];
    fp8_convert16(in[q], sc, out);
    fp8_store16(dst, r, q, out);
  }
}
// `rows` rows of one operand (K or V), two per lane of one warp (row lane, lane + 32).
__device__ __forceinline__ void fp8_dequant_rows(const uint8_t* stage, int B, uint8_t* dst, int rows,
                                                 int lane) {
  for (int r = lane; r < rows; r += 32) fp8_dequant_row(stage, B, dst, r);
}

// One tile's share of a quarter-converting warp (FP8 pages with extra rows):
// once the stage's codes have landed and the operand stage is free, the K rows
// (lanes 0-15) and the V rows (lanes 16-31) of slots 16 dq .. 16 dq + 15, then
// the warp's arrivals on the operand stage and on the staging stage.
template <int MT>
__device__ __forceinline__ bool fp8_dequant_quarter(TcSmem<MT, true>& sm, int j, int dq, int B,
                                                    int lane, volatile int* abort, int* err) {
  const int st8 = j % kF8Stages, s = j % kStages;
  if (!mbar_wait(&sm.f8.full[st8], (j / kF8Stages) & 1, abort, err)) return false;
  if (!mbar_wait(&sm.kv_empty[s], ((j / kStages) & 1) ^ 1, abort, err)) return false;
  const int r = 16 * dq + (lane & 15);
  if (r < sm.f8.nblk[st8] * B)
    fp8_dequant_row(lane < 16 ? sm.f8.k[st8] : sm.f8.v[st8], B, lane < 16 ? sm.k[s] : sm.v[s], r);
  fence_proxy_async();
  __syncwarp();
  if (lane == 0) {
    mbar_arrive(&sm.kv_full[s]);
    mbar_arrive(&sm.f8.free_[st8]);
  }
  return true;
}

template <int MT, bool EXTRA, bool FP8, typename Params>
__global__ void __launch_bounds__(tc_threads<MT, EXTRA, FP8>(), 1)
    attend_tc_kernel(const __grid_constant__ Params params, int n_mgroups_1, int n_tiles_1) {
  extern __shared__ uint8_t smem_raw[];
  TcSmem<MT, FP8>& sm = *reinterpret_cast<TcSmem<MT, FP8>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const CtaWork cw = cta_work(params, n_mgroups_1, n_tiles_1);
  const AttendArgs& a = *cw.a;
  const int n_mgroups = cw.n_mgroups, n_tiles = cw.n_tiles;
  const int H = a.heads, Ps = a.page_size;
  constexpr bool kDense = std::is_same<Params, AttendDense>::value;
  // this CTA's query and output rows (a frame's, in frame attention)
  const long long row_base = (long long)cw.frame * a.n_q;
  const uint16_t* const qg = a.q + row_base * H * kHeadDim;
  uint16_t* const og = a.out + row_base * H * kHeadDim;

  // The KV split varies fastest, so the splits of one (head, M-group) run in the
  // same wave and its query tile is fetched from DRAM once; the M-groups of a
  // head come next, so they share that head's pages through L2.
  int bid = cw.bid;
  const int split = bid % a.num_splits;
  bid /= a.num_splits;
  const int mg = bid % n_mgroups;
  const int h = bid / n_mgroups;
  const int t0 = (int)((long long)n_tiles * split / a.num_splits);
  const int t1 = (int)((long long)n_tiles * (split + 1) / a.num_splits);
  const int nT = t1 - t0;
  const int row0 = mg * MT * 128;

  // ---- set-up: barriers, zeroed KV ring, Q tiles, TMEM
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.kv_full[s], FP8 ? kF8Deq<EXTRA> : 1);   // copy (tx) or the dequantizers
      mbar_init(&sm.kv_empty[s], MT + (EXTRA ? 1 : 0));   // M-tiles (softmax), the tile's extra-row warp
    }
    if constexpr (FP8) {
      for (int s = 0; s < kF8Stages; ++s) {
        mbar_init(&sm.f8.full[s], 1);
        mbar_init(&sm.f8.free_[s], kF8Deq<EXTRA>);
      }
    }
    for (int m = 0; m < MT; ++m) {
      for (int b = 0; b < kSBufs; ++b) {
        mbar_init(&sm.s_full[m][b], 1);
        mbar_init(&sm.p_full[m][b], 4);               // one per softmax warp of the M-tile
      }
      mbar_init(&sm.o_done[m], 1);
      mbar_init(&sm.mma_done[m], 1);
    }
    mbar_init(&sm.x_done, kXWarps);
    sm.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  {
    // stale ring rows are multiplied by P = 0; zero keeps them finite
    uint4* kv = reinterpret_cast<uint4*>(&sm.k[0][0]);
    const int n16 = 2 * kStages * kBN * 128 / 16;     // k and v rings are contiguous
    for (int i = threadIdx.x; i < n16; i += blockDim.x) kv[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     smem_u32(&sm.tmem_base)),
                 "r"(TmemCols<MT>::kAlloc));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  // barriers initialised and the zeroed ring visible to the copy engine: from
  // here the producer may fill the ring
  fence_proxy_async();
  __syncthreads();
  // everything above is private to the CTA; inputs are read only after the
  // previous kernel on the stream has completed
  pdl_wait();
  pdl_trigger();
  if (warp != kProducerWarp) {
    // Q tiles: every load issued before the first store; the producer warp
    // meanwhile starts on the KV ring
    constexpr int kThreads = tc_threads<MT, EXTRA, FP8>() - 32;
    constexpr int kQ = MT * 128 * 8;               // 16-byte chunks
    constexpr int kQPer = (kQ + kThreads - 1) / kThreads;
    const int qt = warp < kProducerWarp ? (int)threadIdx.x : (int)threadIdx.x - 32;
    uint4 val[kQPer];
#pragma unroll
    for (int u = 0; u < kQPer; ++u) {
      const int i = qt + u * kThreads;
      const int row = row0 + (i >> 3);             // M-tile m rows follow m * 128
      val[u] = make_uint4(0u, 0u, 0u, 0u);
      if (i < kQ && row < a.n_q)
        val[u] = __ldg(reinterpret_cast<const uint4*>(qg + ((long long)row * H + h) * kHeadDim +
                                                      (i & 7) * 8));
    }
#pragma unroll
    for (int u = 0; u < kQPer; ++u) {
      const int i = qt + u * kThreads;
      if (i < kQ) {
        const int m = i / (128 * 8), r = (i >> 3) & 127, c = i & 7;
        *reinterpret_cast<uint4*>(&sm.q[m][r * 128 + (swizzle_chunk(r, c) << 4)]) = val[u];
      }
    }
    fence_proxy_async();
  }
  // A sampled call's kept table positions, in order (producer warp, a ballot
  // per 32 positions); the producer then indexes the kept pages only, and the
  // other roles read the list for the tiles' slot masks (hence the CTA barrier).
  if (a.sampled) {
    if (warp == kProducerWarp) {
      if (a.kept_dev) {
        // a list made on the device (page skipping by estimated mass)
        for (int i = lane; i < a.n_entries; i += 32) sm.kept[i] = __ldcg(a.kept_dev + i);
      } else {
        int count = 0;
        for (int e0 = 0; e0 < a.n_entries_all; e0 += 32) {
          const int e = e0 + lane;
          const bool keep = e < a.n_entries_all &&
                            (e < a.sample_anchor || page_sample_kept(a.sample_key, e, a.sample_keep));
          const unsigned ball = __ballot_sync(0xffffffffu, keep);
          if (keep) sm.kept[count + __popc(ball & ((1u << lane) - 1u))] = (uint16_t)e;
          count += __popc(ball);
        }
      }
    }
    __syncthreads();
  }
  // Slot masks of the CTA's tiles, computed once by the roles that read them
  // (the softmax and extra-row warps), so that the tile loops read neither the
  // kernel's parameters nor the stage's copy barrier for them.
  if (warp != kProducerWarp) {
    constexpr int kThreads = tc_threads<MT, EXTRA, FP8>() - 32;
    const int tt = warp < kProducerWarp ? (int)threadIdx.x : (int)threadIdx.x - 32;
    for (int j = tt; j < nT && j < kMaxMaskTiles; j += kThreads)
      sm.tmask[j] = tile_mask<kDense>(a, sm.kept, t0 + j);
  }
  // Visible-table entries for the producer, 32 at a time (one per lane): the
  // entry lookups are dependent global loads, so a batch costs one latency.
  // table position of the producer's e-th entry
  auto entry_of = [&](int e) { return a.sampled ? (int)sm.kept[e] : e; };
  const int e_first = kDense ? 0 : (int)((long long)t0 * kBN / Ps);
  int e_batch = e_first & ~31, e_page = 0, e_len = 0;
  if (warp == kProducerWarp && e_batch + lane < a.n_entries)
    table_entry(a.tbl, entry_of(e_batch + lane), e_page, e_len);
  // Q and the TMEM address published to every role but the producer, which
  // needs neither (named barrier 1: all warps but the producer)
  if (warp != kProducerWarp) {
    tc_fence_before();
    asm volatile("bar.sync 1, %0;\n" ::"r"(tc_threads<MT, EXTRA, FP8>() - 32) : "memory");
    tc_fence_after();
  }
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;

  if (warp == kProducerWarp) {
    // ================================================================ producer
    // The whole warp walks the tiles (its lanes hold the cached table entries);
    // lane 0 issues the copies.
    int issued_tiles = 0;
    if constexpr (kDense) {
      // frame attention: tile t is tokens 64 t .. 64 t + 63 of the CTA's frame,
      // one K and one V box of head h; the slots past the frame's last token
      // (the next frame's, or the tensor map's zero fill after the last frame)
      // are masked
      const int kv_row0 = cw.frame * a.n_q;
      for (int j = 0; j < nT; ++j) {
        const int s = j % kStages;
        if (!mbar_wait(&sm.kv_empty[s], ((j / kStages) & 1) ^ 1, abort, a.err)) break;
        const int tile = t0 + j;
        if (lane == 0) {
          const uint32_t mb = smem_u32(&sm.kv_full[s]);
          mbar_arrive_expect_tx(&sm.kv_full[s], 2u * kBN * 128u);
          tma_load_3d(smem_u32(&sm.k[s][0]), &params.k_map, 0, h, kv_row0 + tile * kBN, mb);
          tma_load_3d(smem_u32(&sm.v[s][0]), &params.v_map, 0, h, kv_row0 + tile * kBN, mb);
        }
        issued_tiles = j + 1;
      }
    }
    const int per = Ps >= kBN ? 1 : kBN / Ps;      // page blocks per tile
    const int rows = Ps >= kBN ? kBN : Ps;         // slots per block
    if constexpr (FP8 && !kDense) {
      // FP8 pages: each tile's codes and row exponents are copied into a staging
      // stage kF8Stages tiles ahead. Without extra rows this warp dequantizes the
      // K rows into the operand ring (one more warp the V rows) and refills the
      // stage once both are done with it; with extra rows it only stages
      // tiles are staged in order, so the table position (entry st_e, slot st_so)
      // of the next block advances by one block each time (no division per tile)
      int st_e = (int)((long long)t0 * kBN / Ps);
      int st_so = (int)((long long)t0 * kBN - (long long)st_e * Ps);
      auto issue_stage = [&](int j) {
        const int st8 = j % kF8Stages;
        int nblk = 0, blk_page[kBN / 16], blk_so[kBN / 16];
#pragma unroll
        for (int pp = 0; pp < kBN / 16; ++pp) {
          if (pp >= per) break;
          const int e = st_e, so = st_so;
          if (e >= a.n_entries) break;
          if ((e & ~31) != e_batch) {              // warp-uniform: next batch of entries
            e_batch = e & ~31;
            e_page = e_len = 0;
            if (e_batch + lane < a.n_entries) table_entry(a.tbl, entry_of(e_batch + lane), e_page, e_len);
          }
          blk_page[pp] = __shfl_sync(0xffffffffu, e_page, e - e_batch);
          blk_so[pp] = so;
          nblk = pp + 1;
          st_so += rows;
          if (st_so >= Ps) {
            st_so = 0;
            ++st_e;
          }
        }
        if (lane == 0) {
          sm.f8.nblk[st8] = nblk;
          const uint32_t mb = smem_u32(&sm.f8.full[st8]);
          mbar_arrive_expect_tx(&sm.f8.full[st8], (uint32_t)nblk * 2u * rows * (kHeadDim + 1));
#pragma unroll
          for (int pp = 0; pp < kBN / 16; ++pp) {
            if (pp >= nblk) break;
            int page = blk_page[pp];
            if (page < 0 || page >= a.pool_pages) {
              atomicOr(a.err, kErrPageRange);
              page = 0;
            }
            const uint8_t* pg = reinterpret_cast<const uint8_t*>(a.pool) + (long long)page * a.page_bytes;
            const uint32_t blk_bytes = (uint32_t)rows * (kHeadDim + 1);
            const uint32_t dsts[2] = {smem_u32(&sm.f8.k[st8][pp * blk_bytes]),
                                      smem_u32(&sm.f8.v[st8][pp * blk_bytes])};
            // blk_so is block-aligned, so the block starts at (plane row + blk_so) * 65
            const long long kb = ((long long)h * Ps + blk_so[pp]) * (kHeadDim + 1);
            const uint8_t* srcs[2] = {pg + kb, pg + kb + (long long)H * Ps * (kHeadDim + 1)};
#pragma unroll
            for (int c = 0; c < 2; ++c)
              asm volatile(
                  "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], "
                  "%2, [%3];\n" ::"r"(dsts[c]),
                  "l"(srcs[c]), "r"(blk_bytes), "r"(mb)
                  : "memory");
          }
        }
      };
      int issued = 0, consumed = 0;
      for (; issued < nT && issued < kF8Stages; ++issued) issue_stage(issued);
      if constexpr (EXTRA) {
        // staging only: a stage is refilled once the four quarter warps are done
        // with its previous tile
        for (; issued < nT; ++issued) {
          if (!mbar_wait(&sm.f8.free_[issued % kF8Stages], (issued / kF8Stages - 1) & 1, abort,
                         a.err))
            break;
          issue_stage(issued);
        }
        consumed = issued > kF8Stages ? issued - kF8Stages : 0;
      }
      for (int j = 0; !EXTRA && j < nT; ++j) {
        const int st8 = j % kF8Stages, s = j % kStages;
        if (!mbar_wait(&sm.f8.full[st8], (j / kF8Stages) & 1, abort, a.err)) break;
        consumed = j + 1;
        if (!mbar_wait(&sm.kv_empty[s], ((j / kStages) & 1) ^ 1, abort, a.err)) break;
        fp8_dequant_rows(sm.f8.k[st8], rows, sm.k[s], sm.f8.nblk[st8] * rows, lane);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sm.kv_full[s]);
          mbar_arrive(&sm.f8.free_[st8]);
        }
        if (issued < nT) {
          if (!mbar_wait(&sm.f8.free_[st8], (j / kF8Stages) & 1, abort, a.err)) break;
          issue_stage(issued);
          ++issued;
        }
      }
      // no copy may still be landing in shared memory when the CTA ends
      if (lane == 0)
        for (int j = consumed; j < issued; ++j)
          mbar_wait(&sm.f8.full[j % kF8Stages], (j / kF8Stages) & 1, abort, a.err, false);
    }
    for (int j = 0; !kDense && !FP8 && j < nT; ++j) {
      const int s = j % kStages;
      if (!mbar_wait(&sm.kv_empty[s], ((j / kStages) & 1) ^ 1, abort, a.err)) break;
      const int tile = t0 + j;
      int nblk = 0, blk_page[kBN / 16], blk_so[kBN / 16];
#pragma unroll
      for (int pp = 0; pp < kBN / 16; ++pp) {
        if (pp >= per) break;
        const int f0 = tile * kBN + pp * rows;
        const int e = f0 / Ps, so = f0 - e * Ps;
        if (e >= a.n_entries) break;
        if ((e & ~31) != e_batch) {                // warp-uniform: next batch of entries
          e_batch = e & ~31;
          e_page = e_len = 0;
          if (e_batch + lane < a.n_entries) table_entry(a.tbl, entry_of(e_batch + lane), e_page, e_len);
        }
        blk_page[pp] = __shfl_sync(0xffffffffu, e_page, e - e_batch);
        blk_so[pp] = so;
        nblk = pp + 1;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&sm.kv_full[s], (uint32_t)nblk * 2u * rows * 128u);
#pragma unroll
        for (int pp = 0; pp < kBN / 16; ++pp) {
          if (pp >= nblk) break;
          int page = blk_page[pp];
          if (page < 0 || page >= a.pool_pages) {
            atomicOr(a.err, kErrPageRange);
            page = 0;
          }
          const uint16_t* kp = a.pool + (long long)page * a.page_elems +
                               ((long long)h * Ps + blk_so[pp]) * kHeadDim;
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
      }
      issued_tiles = j + 1;
    }
    // make sure no copy is still landing in shared memory when the CTA ends
    if (lane == 0)
      for (int j = issued_tiles - 1; j >= 0 && j >= issued_tiles - kStages; --j)
        mbar_wait(&sm.kv_full[j % kStages], (j / kStages) & 1, abort, a.err, false);
  } else if (warp == kMmaWarp || (MT == 2 && warp == kMmaWarp2)) {
    // ============================================================ MMA issuers
    // One issuing thread per M-tile (warp 3: M-tile 0; warp 1: M-tile 1): an
    // issuing thread stalls on each tcgen05.mma until the tensor core takes it,
    // and two issuers keep the tensor core twice as busy. Each M-tile has three
    // S buffers in TMEM, tile j using buffer j % 3, its P written over the
    // buffer's first 32 columns. Per M-tile:
    //   QK(m, 0..2) up front; then for every tile j, once the softmax has read S
    //   and written P of tile j:
    //   PV(m, j)      O_m += P_m V;
    //   QK(m, j + 3)  into the buffer of tile j, so S of the next two tiles is
    //                 in TMEM while the softmax works and the loop from one
    //                 tile's P to the S it releases spans three tiles.
    if (lane == 0) {
      const int m = warp == kMmaWarp ? 0 : 1;
      constexpr uint32_t kIdQK = idesc_bf16(128, kBN, false);
      constexpr uint32_t kIdPV = idesc_bf16(128, kHeadDim, true);
      const uint64_t qa = sdesc(smem_u32(&sm.q[m][0]));
      const uint32_t t_o = tmem + TmemCols<MT>::o(m);
      auto issue_qk = [&](int j) -> bool {
        if (!mbar_wait(&sm.kv_full[j % kStages], (j / kStages) & 1, abort, a.err)) return false;
        tc_fence_after();
        const uint64_t kb = sdesc(smem_u32(&sm.k[j % kStages][0]));
        const uint32_t t_s = tmem + TmemCols<MT>::s(m, j % kSBufs);
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk)
          tc_mma(t_s, qa + 2 * kk, kb + 2 * kk, kIdQK, kk > 0);
        tc_commit(&sm.s_full[m][j % kSBufs]);
        return true;
      };
      bool ok = true;
      for (int j = 0; ok && j < kSBufs && j < nT; ++j) ok = issue_qk(j);
      for (int j = 0; ok && j < nT; ++j) {
        if (!mbar_wait(&sm.p_full[m][j % kSBufs], (j / kSBufs) & 1, abort, a.err)) break;
        tc_fence_after();
        const uint64_t vb = sdesc(smem_u32(&sm.v[j % kStages][0]));
        const uint32_t t_p = tmem + TmemCols<MT>::s(m, j % kSBufs);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          tc_mma_ts(t_o, t_p + 8 * kk, vb + 128 * kk, kIdPV, (j > 0 || kk > 0) ? 1u : 0u);
        // QK(j + 3) overwrites P of tile j: the tensor core runs this thread's
        // MMAs in issue order, so PV(j) has read P before it. Its commit (S of
        // tile j + 3) also announces that PV(j) has completed, which frees the
        // stage of tile j and lets O be rescaled; the last three PVs, which no
        // QK follows, are announced on o_done.
        if (j + kSBufs < nT) {
          if (!issue_qk(j + kSBufs)) break;
        } else {
          tc_commit(&sm.o_done[m]);
        }
      }
      // every MMA issued by this thread has completed once mma_done[m] flips
      tc_commit(&sm.mma_done[m]);
      mbar_wait(&sm.mma_done[m], 0, abort, a.err, false);
    }
  } else if (warp >= 4 && warp < 4 + 4 * MT) {
    // ================================================================ softmax
    const int m = (warp - 4) >> 2;
    const int wq = warp & 3;                       // TMEM lane quarter of this warp
    const int r = wq * 32 + lane;                  // row inside the M-tile
    const int row = row0 + m * 128 + r;
    const bool warp_active = row0 + m * 128 + wq * 32 < a.n_q;
    const uint32_t t_lane = (uint32_t)(wq * 32) << 16;
    const uint32_t t_o = tmem + t_lane + TmemCols<MT>::o(m);
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;          // running max (log2 units) and sum
    bool alive = true;
    // One wait per tile, for S of the tile (buffer b = j % 3, phase (j / 3) & 1).
    // The issuing thread issues QK(j) after PV(j - 3), and the commit that
    // announces S(j) covers every MMA it issued before, so S(j) also means that
    // PV(j - 3) has completed: the M-tile's first thread then releases the KV
    // stage of tile j - 3 (when a later tile needs it). PV(j - 1), and with it
    // every earlier PV, is waited for only when O must be rescaled: through S of
    // tile j + 2 (issued right after PV(j - 1)), or, for the last three tiles,
    // through o_done, whose phases are the PVs of those tiles; at most the
    // phases of PV(j - 2) and PV(j - 1) are open then, so waiting for them in
    // order is exact. The arrivals of tile j go to p_full[m][b]: a warp running
    // ahead arrives on the other buffers' barriers, and it reaches tile j + 3
    // only through S(j + 3), which the issuer starts after it has seen all four
    // arrivals of tile j, so no phase mixes two tiles.
    const int tail0 = nT > kSBufs ? nT - kSBufs : 0;   // first PV announced on o_done
    auto wait_pv = [&](int jj) -> bool {               // PV(jj) (and all before) done
      if (jj + kSBufs < nT)
        return mbar_wait(&sm.s_full[m][jj % kSBufs], (uint32_t)((jj / kSBufs + 1) & 1), abort,
                         a.err);
      if (jj - 1 >= tail0 && !mbar_wait(&sm.o_done[m], (uint32_t)((jj - 1 - tail0) & 1), abort, a.err))
        return false;
      return mbar_wait(&sm.o_done[m], (uint32_t)((jj - tail0) & 1), abort, a.err);
    };
    int b = 0;
    uint32_t ph = 0;
    for (int j = 0; j < nT; ++j, b = b == kSBufs - 1 ? 0 : b + 1, ph ^= (b == 0)) {
      const uint32_t t_s = tmem + t_lane + TmemCols<MT>::s(m, b);
      if (!mbar_wait(&sm.s_full[m][b], ph, abort, a.err)) {
        alive = false;
        break;
      }
      if (wq == 0 && lane == 0 && j >= kSBufs && j - kSBufs + kStages < nT)
        mbar_arrive(&sm.kv_empty[(j - kSBufs) % kStages]);
      tc_fence_after();
      const uint64_t bits = j < kMaxMaskTiles ? sm.tmask[j] : tile_mask<kDense>(a, sm.kept, t0 + j);
      const uint32_t t_p = t_s;                    // P over the S columns just read
      bool rescale = false;
      float alpha = 1.f;
      if (warp_active) {
        // Fast path: exponentiate against the running reference max. Any
        // reference keeps the result exact (it cancels in O / l); it only has
        // to keep 2^(s - m) finite, so a row whose sum exceeds 2^64 (or is not
        // finite), and every row on its first tile, takes the exact path: its
        // reference moves to its max and O and l are rescaled. S stays in TMEM
        // until this tile's arrival below, so the exact path reads it again.
        float v[kBN];
        PKV_TMEM_LD32(t_s, reinterpret_cast<uint32_t*>(v));
        PKV_TMEM_LD32(t_s + 32, reinterpret_cast<uint32_t*>(v + 32));
        tmem_wait_ld();
        if (bits != ~0ull) {
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (!((bits >> c) & 1ull)) v[c] = -INFINITY;
        }
        uint32_t pk[kBN / 2];
        float sum0 = 0.f, sum1 = 0.f;
        {
          const float m_ref = m_run == -INFINITY ? 0.f : m_run;
#pragma unroll
          for (int c = 0; c < kBN; c += 2) {
            const float p0 = fast_exp2(fmaf(v[c], sl2, -m_ref));
            const float p1 = fast_exp2(fmaf(v[c + 1], sl2, -m_ref));
            pk[c >> 1] = pack_bf16(p0, p1);
            sum0 += p0;
            sum1 += p1;
          }
        }
        const bool redo = m_run == -INFINITY || !(sum0 + sum1 <= kSumLimit);
        if (__any_sync(0xffffffffu, redo)) {
          // exact path for the rows that need it (the TMEM load is warp-wide)
          PKV_TMEM_LD32(t_s, reinterpret_cast<uint32_t*>(v));
          PKV_TMEM_LD32(t_s + 32, reinterpret_cast<uint32_t*>(v + 32));
          tmem_wait_ld();
          if (redo) {
            float x0 = -INFINITY, x1 = -INFINITY, x2 = -INFINITY, x3 = -INFINITY;
#pragma unroll
            for (int c = 0; c < kBN; c += 4) {
              if (!((bits >> c) & 1ull)) v[c] = -INFINITY;
              if (!((bits >> (c + 1)) & 1ull)) v[c + 1] = -INFINITY;
              if (!((bits >> (c + 2)) & 1ull)) v[c + 2] = -INFINITY;
              if (!((bits >> (c + 3)) & 1ull)) v[c + 3] = -INFINITY;
              x0 = fmaxf(x0, v[c]);
              x1 = fmaxf(x1, v[c + 1]);
              x2 = fmaxf(x2, v[c + 2]);
              x3 = fmaxf(x3, v[c + 3]);
            }
            const float tmax = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3)) * sl2;   // sl2 > 0
            if (tmax > m_run) {                    // -inf stays -inf: no valid slot yet
              if (m_run != -INFINITY) {
                alpha = fast_exp2(m_run - tmax);
                l_run *= alpha;
                rescale = true;
              }
              m_run = tmax;
            }
            const float m_ref = m_run == -INFINITY ? 0.f : m_run;
            sum0 = sum1 = 0.f;
#pragma unroll
            for (int c = 0; c < kBN; c += 2) {
              const float p0 = fast_exp2(fmaf(v[c], sl2, -m_ref));
              const float p1 = fast_exp2(fmaf(v[c + 1], sl2, -m_ref));
              pk[c >> 1] = pack_bf16(p0, p1);
              sum0 += p0;
              sum1 += p1;
            }
          }
        }
        l_run += sum0 + sum1;
        // P over the first half of the S buffer (all of S is in registers)
        PKV_TMEM_ST32(t_p, pk);
        tmem_wait_st();
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O_m *= alpha for this row (alpha = 1 for rows that keep their max),
        // once PV(j - 1) has completed
        if (j > 0 && !wait_pv(j - 1)) {
          alive = false;
          break;
        }
        tc_fence_after();
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
      // S_m read, P_m written, O_m rescaled: PV(m, j) and QK(m, j + 2) may go
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[m][b]);
    }
    // ---- epilogue: O_m row (64 columns, one TMEM read) to the output or the split's partial
    const bool have_o = alive && nT > 0 && mbar_wait(&sm.mma_done[m], 0, abort, a.err);
    if (have_o) tc_fence_after();
    const bool write = alive && row < a.n_q && (have_o || nT == 0);
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    const long long ro = ((long long)split * a.n_q + row) * H + h;
    uint32_t o[kHeadDim];
#pragma unroll
    for (int i = 0; i < kHeadDim; ++i) o[i] = 0u;
    if (have_o && warp_active) {
      PKV_TMEM_LD32(t_o, o);
      PKV_TMEM_LD32(t_o + 32, (o + 32));
      tmem_wait_ld();
    }
    if (write) {
      if (a.num_splits == 1) {
        uint4* dst = reinterpret_cast<uint4*>(og + ((long long)row * H + h) * kHeadDim);
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float* f = reinterpret_cast<const float*>(&o[8 * q4]);
          dst[q4] = make_uint4(pack_bf16(f[0] * inv, f[1] * inv), pack_bf16(f[2] * inv, f[3] * inv),
                               pack_bf16(f[4] * inv, f[5] * inv), pack_bf16(f[6] * inv, f[7] * inv));
        }
      } else {
        uint4* dst = reinterpret_cast<uint4*>(a.part_o + ro * kHeadDim);
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4)
          dst[q4] = make_uint4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
      }
    }
    if (write && a.num_splits > 1)
      *reinterpret_cast<float2*>(a.part_ml + ro * 2) = make_float2(m_run, l_run);
  } else if (FP8 && !kDense && warp == tc_conv_warp<MT, EXTRA>()) {
    // ============================ V dequantizer, or the fourth quarter warp (FP8)
    if constexpr (FP8 && !kDense) {
      const int rows = Ps >= kBN ? kBN : Ps;
      if constexpr (EXTRA)
        for (int j = 0; j < nT; ++j)
          if (!fp8_dequant_quarter<MT>(sm, j, kF8Deq<EXTRA> - 1, rows, lane, abort, a.err)) break;
      for (int j = 0; !EXTRA && j < nT; ++j) {
        const int st8 = j % kF8Stages, s = j % kStages;
        if (!mbar_wait(&sm.f8.full[st8], (j / kF8Stages) & 1, abort, a.err)) break;
        if (!mbar_wait(&sm.kv_empty[s], ((j / kStages) & 1) ^ 1, abort, a.err)) break;
        fp8_dequant_rows(sm.f8.v[st8], rows, sm.v[s], sm.f8.nblk[st8] * rows, lane);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sm.kv_full[s]);
          mbar_arrive(&sm.f8.free_[st8]);
        }
      }
    }
  } else if (EXTRA && (warp == kXWarp || (warp >= 4 + 4 * MT && warp < tc_conv_warp<MT, EXTRA>()))) {
    // ============================================== extra rows (mma.sync, regs)
    // Up to 8 query rows, shared by kXWarps warps: warp xi takes every kXWarps-th
    // tile (tiles xi, xi + kXWarps, ...; all 64 slots, so the four slot groups'
    // MMAs are independent and the softmax bookkeeping is paid once a tile) with
    // its own running max, sum and O, and the partial results are merged at the
    // end. A stage's tiles are kStages apart, a multiple of kXWarps, so each stage
    // is always released by the same warp. Transposed so that the 8 queries
    // are the N = 8 side of m16n8k16 tiles and the slots the M = 16 side:
    // S^T = K Q_x^T, then O^T += V^T P^T with P^T moved into B fragments by
    // movmatrix. Softmax runs over slots, i.e. across the 8 lanes that share a
    // query column.
    const int xi = warp == kXWarp ? 0 : warp - (4 + 4 * MT) + 1;
    // FP8 pages: warps 1..3 convert quarter xi - 1 of every tile, kF8Ahead tiles ahead
    constexpr int kF8Ahead = 3;
    const int dq = xi - 1;
    const int xr0 = row0 + MT * 128;               // first extra row
    const int g = lane >> 2, tq = lane & 3;
    // B fragments of Q_x^T: (k = d 2tq.., n = query g)
    uint32_t qb[4][2];
    {
      const int qrow = xr0 + g;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int i = 0; i < 2; ++i)
          qb[kk][i] = qrow < a.n_q ? __ldg(reinterpret_cast<const uint32_t*>(
                                         qg + ((long long)qrow * H + h) * kHeadDim + kk * 16 +
                                         i * 8 + 2 * tq))
                                   : 0u;
    }
    // per thread: queries 2tq and 2tq+1
    float m_x[2] = {-INFINITY, -INFINITY}, l_x[2] = {0.f, 0.f};
    float ox[4][4];                                // O^T: d-tile x (d g|g+8, query 2tq|2tq+1)
#pragma unroll
    for (int i = 0; i < 4; ++i) ox[i][0] = ox[i][1] = ox[i][2] = ox[i][3] = 0.f;
    const float sl2 = a.scale_log2;
    bool alive = true;
    if constexpr (FP8 && !kDense)
      for (int jj = 0; dq >= 0 && alive && jj < kF8Ahead && jj < nT; ++jj)
        alive = fp8_dequant_quarter<MT>(sm, jj, dq, Ps >= kBN ? kBN : Ps, lane, abort, a.err);
    // tiles xi, xi + kXWarps, ...: all 64 slots of each (four 16-slot groups)
    for (int j = FP8 && !kDense ? 0 : xi; alive && j < nT; j += FP8 && !kDense ? 1 : kXWarps) {
      if constexpr (FP8 && !kDense) {
        if (dq >= 0 && j + kF8Ahead < nT &&
            !fp8_dequant_quarter<MT>(sm, j + kF8Ahead, dq, Ps >= kBN ? kBN : Ps, lane, abort, a.err)) {
          alive = false;
          break;
        }
        if (j % kXWarps != xi) continue;
      }
      const int st = j % kStages;
      if (!mbar_wait(&sm.kv_full[st], (j / kStages) & 1, abort, a.err)) {
        alive = false;
        break;
      }
      const uint64_t bits = j < kMaxMaskTiles ? sm.tmask[j] : tile_mask<kDense>(a, sm.kept, t0 + j);
      const uint32_t kbase = smem_u32(&sm.k[st][0]), vbase = smem_u32(&sm.v[st][0]);
      // S^T: 64 slots (four groups of 16) x 8 queries
      float sc[4][4];
#pragma unroll
      for (int sg = 0; sg < 4; ++sg) {
        sc[sg][0] = sc[sg][1] = sc[sg][2] = sc[sg][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t ka[4];
          ldsm_x4(sw_addr(kbase, sg * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, 2 * kk + (lane >> 4)),
                  ka[0], ka[1], ka[2], ka[3]);
          mma_16816(sc[sg], ka, qb[kk][0], qb[kk][1]);
        }
      }
      // mask, scale, per-query max over the tile's slots
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int sg = 0; sg < 4; ++sg)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool ok = (bits >> (sg * 16 + g + (e >> 1) * 8)) & 1ull;
          sc[sg][e] = ok ? sc[sg][e] * sl2 : -INFINITY;
          mx[e & 1] = fmaxf(mx[e & 1], sc[sg][e]);
        }
      float alpha[2], m_use[2];
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        mx[qq] = fmaxf(mx[qq], __shfl_xor_sync(0xffffffffu, mx[qq], 4));
        mx[qq] = fmaxf(mx[qq], __shfl_xor_sync(0xffffffffu, mx[qq], 8));
        mx[qq] = fmaxf(mx[qq], __shfl_xor_sync(0xffffffffu, mx[qq], 16));
        const float m_new = fmaxf(m_x[qq], mx[qq]);
        m_use[qq] = m_new == -INFINITY ? 0.f : m_new;
        alpha[qq] = fast_exp2(m_x[qq] - m_use[qq]);
        m_x[qq] = m_new;
        l_x[qq] *= alpha[qq];
      }
#pragma unroll
      for (int dt = 0; dt < 4; ++dt) {
        ox[dt][0] *= alpha[0];
        ox[dt][1] *= alpha[1];
        ox[dt][2] *= alpha[0];
        ox[dt][3] *= alpha[1];
      }
      // P^T of each slot group, then O^T += V^T P^T over the group's 16 slots
#pragma unroll
      for (int sg = 0; sg < 4; ++sg) {
        const float p0 = fast_exp2(sc[sg][0] - m_use[0]);
        const float p1 = fast_exp2(sc[sg][1] - m_use[1]);
        const float p2 = fast_exp2(sc[sg][2] - m_use[0]);
        const float p3 = fast_exp2(sc[sg][3] - m_use[1]);
        l_x[0] += p0 + p2;
        l_x[1] += p1 + p3;
        // (slot g | g+8, query 2tq..) pairs -> transposed: (query g, slots 2tq..)
        uint32_t pb0 = pack_bf16(p0, p1), pb1 = pack_bf16(p2, p3);
        asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %0;\n" : "+r"(pb0));
        asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %0;\n" : "+r"(pb1));
#pragma unroll
        for (int dt = 0; dt < 4; ++dt) {
          uint32_t va[4];
          ldsm_x4_t(sw_addr(vbase, sg * 16 + (lane & 7) + (lane >> 4) * 8, 2 * dt + ((lane >> 3) & 1)),
                    va[0], va[1], va[2], va[3]);
          mma_16816(ox[dt], va, pb0, pb1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.kv_empty[st]);
    }
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
      l_x[qq] += __shfl_xor_sync(0xffffffffu, l_x[qq], 4);
      l_x[qq] += __shfl_xor_sync(0xffffffffu, l_x[qq], 8);
      l_x[qq] += __shfl_xor_sync(0xffffffffu, l_x[qq], 16);
    }
    // publish this warp's partial state; warp 0 merges the kXWarps of them
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
#pragma unroll
      for (int dt = 0; dt < 4; ++dt)
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) sm.xo[xi][2 * tq + qq][dt * 16 + g + hi * 8] = ox[dt][2 * hi + qq];
      if (g == 0) {
        sm.xml[xi][2 * tq + qq][0] = m_x[qq];
        sm.xml[xi][2 * tq + qq][1] = l_x[qq];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.x_done);
    if (xi == 0 && alive && mbar_wait(&sm.x_done, 0, abort, a.err)) {
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        const int xq = 2 * tq + qq;
        const int xrow = xr0 + xq;
        if (xrow >= a.n_q) continue;
        float mm = -INFINITY;
#pragma unroll
        for (int i = 0; i < kXWarps; ++i) mm = fmaxf(mm, sm.xml[i][xq][0]);
        float w[kXWarps], ll = 0.f;
#pragma unroll
        for (int i = 0; i < kXWarps; ++i) {
          w[i] = mm == -INFINITY ? 0.f : fast_exp2(sm.xml[i][xq][0] - mm);
          ll += w[i] * sm.xml[i][xq][1];
        }
        const float inv = ll > 0.f ? 1.f / ll : 0.f;
        const long long ro = ((long long)split * a.n_q + xrow) * H + h;
#pragma unroll
        for (int dt = 0; dt < 4; ++dt)
#pragma unroll
          for (int hi = 0; hi < 2; ++hi) {
            const int d = dt * 16 + g + hi * 8;
            float val = 0.f;
#pragma unroll
            for (int i = 0; i < kXWarps; ++i) val += w[i] * sm.xo[i][xq][d];
            if (a.num_splits == 1)
              og[((long long)xrow * H + h) * kHeadDim + d] =
                  __bfloat16_as_ushort(__float2bfloat16_rn(val * inv));
            else
              a.part_o[ro * kHeadDim + d] = val;
          }
        if (a.num_splits > 1 && g == 0)
          *reinterpret_cast<float2*>(a.part_ml + ro * 2) = make_float2(mm, ll);
      }
    }
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

template <int MT, bool EXTRA, bool FP8, typename Params>
cudaError_t launch_mt(const Params& p, int grid, int n_mgroups, int n_tiles, cudaStream_t s) {
  const size_t smem = sizeof(TcSmem<MT, FP8>) + 1024;
  // the shared-memory opt-in is a per-device function attribute: set it once for
  // every device this process launches on
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (dev >= 64 || !(configured.load() & bit)) {
    cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel<MT, EXTRA, FP8, Params>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured.fetch_or(bit);
  }
  const cudaError_t e = launch_pdl(attend_tc_kernel<MT, EXTRA, FP8, Params>, dim3(grid),
                                   dim3(tc_threads<MT, EXTRA, FP8>()), smem, s, p, n_mgroups, n_tiles);
  count_launches(1);
  return e;
}

struct TcShape {
  int mt, n_mgroups;
  bool extra;
};

// Query rows per CTA: up to two 128-row M-tiles, plus up to 8 extra rows when
// the whole query fits one group that way (a frame's 256 + 6 tokens); longer
// queries (a chunk's tokens) are cut into groups of 256 rows.
TcShape tc_shape(int n_q) {
  if (n_q <= 128) return {1, 1, false};
  if (n_q <= 128 + kXRows) return {1, 1, true};
  if (n_q <= 256) return {2, 1, false};
  if (n_q <= 256 + kXRows) return {2, 1, true};
  return {2, (n_q + 255) / 256, false};
}

}  // namespace

int attend_tc_tiles(long long n_slots) { return (int)((n_slots + kBN - 1) / kBN); }

// Split-KV factor: fill the SMs in as few, as even waves as possible.
int attend_tc_splits(int n_q, int heads, int n_tiles, int num_sms) {
  return attend_tc_splits_pairs(tc_shape(n_q).n_mgroups * heads, n_tiles, num_sms);
}

int attend_tc_shape(int n_q) {
  const TcShape sh = tc_shape(n_q);
  return (sh.mt - 1) * 2 + (sh.extra ? 1 : 0);
}

int attend_tc_mgroups(int n_q) { return tc_shape(n_q).n_mgroups; }

int attend_tc_splits_pairs(int pairs, int n_tiles, int num_sms) {
  // a wave's time is the tiles each CTA handles plus a CTA's fixed cost (set-up,
  // the first tile's cold start, epilogue), ~14 tile periods on a LingBot frame
  constexpr double kCtaFixedTiles = 14.0;
  int best = 1;
  double best_eff = 0.0;
  for (int s = 1; s <= 16; ++s) {
    if (s > 1 && n_tiles / s < 3) break;
    const int ctas = pairs * s;
    const int waves = (ctas + num_sms - 1) / num_sms;
    const double t = (double)waves * ((double)n_tiles / s + kCtaFixedTiles);
    const double eff = (double)pairs * n_tiles / (t * num_sms);
    if (eff > best_eff * 1.03) {
      best_eff = eff;
      best = s;
    }
  }
  return best;
}

template <bool FP8, typename Params>
static cudaError_t launch_shape(int shape, const Params& p, int grid, int n_mgroups, int n_tiles,
                                cudaStream_t s) {
  switch (shape) {
    case 0: return launch_mt<1, false, FP8>(p, grid, n_mgroups, n_tiles, s);
    case 1: return launch_mt<1, true, FP8>(p, grid, n_mgroups, n_tiles, s);
    case 2: return launch_mt<2, false, FP8>(p, grid, n_mgroups, n_tiles, s);
    default: return launch_mt<2, true, FP8>(p, grid, n_mgroups, n_tiles, s);
  }
}

cudaError_t launch_attend_tc(const AttendArgs& a, cudaStream_t s) {
  const TcShape sh = tc_shape(a.n_q);
  const int n_tiles = attend_tc_tiles(a.n_slots);
  if (a.fp8)
    return launch_shape<true>(attend_tc_shape(a.n_q), a, sh.n_mgroups * a.heads * a.num_splits,
                              sh.n_mgroups, n_tiles, s);
  return launch_shape<false>(attend_tc_shape(a.n_q), a, sh.n_mgroups * a.heads * a.num_splits,
                             sh.n_mgroups, n_tiles, s);
}

cudaError_t launch_attend_tc_batch(const AttendBatch& b, cudaStream_t s) {
  if (b.item[0].fp8)
    return launch_shape<true>(attend_tc_shape(b.item[0].n_q), b, b.cta_base[b.n], 0, 0, s);
  return launch_shape<false>(attend_tc_shape(b.item[0].n_q), b, b.cta_base[b.n], 0, 0, s);
}

cudaError_t launch_attend_dense(const AttendDense& d, int n_frames, cudaStream_t s) {
  const TcShape sh = tc_shape(d.a.n_q);
  return launch_shape<false>(attend_tc_shape(d.a.n_q), d, sh.n_mgroups * d.a.heads * n_frames,
                             sh.n_mgroups, d.a.n_tiles, s);
}

}  // namespace pkv
