// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// tensor loads, tcgen05 (MMA into tensor memory, TMEM loads/stores, alloc),
// and the shared-memory / instruction descriptors the MMA reads.
//
// Conventions used by every kernel in this library:
//  * operand tiles in shared memory use the 128-byte swizzle: rows of 128 B
//    (64 bf16), 8-row groups of 1024 B, 16-byte chunk index XOR (row % 8);
//    every tile base is 1024-byte aligned so TMA, the MMA descriptors and the
//    hand-written stores agree on the pattern;
//  * every mbarrier wait is bounded in time; on expiry the wait records a
//    timeout in the caller's status word and returns false, and the kernel
//    unwinds instead of spinning forever.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fm {

// ---------------------------------------------------------------- status word
// Device-side status bits, or-ed into a word in the caller's workspace.
enum : int {
  DEV_OK = 0,
  DEV_BOUNDS = 1,     // a bound value outside [0, Sq]
  DEV_TIMEOUT = 2,    // an mbarrier wait ran past its time limit
  DEV_LAYOUT = 4,     // shared memory not 1024-byte aligned: the kernel did nothing
};

#ifndef FM_WAIT_LIMIT_NS
#define FM_WAIT_LIMIT_NS 2000000000ull   // 2 s: far beyond any legitimate wait
#endif

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// `count` arrivals at once (on behalf of threads that have nothing to do in
// this phase).
__device__ __forceinline__ void mbar_arrive_count(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// One arrival for the whole calling warp, once every lane has reached it
// (barriers that consumer warps release count warps, not threads): the warp
// synchronisation orders each lane's earlier stores, fenced as their proxy
// requires, before lane 0's arrival.  Every lane of the warp must call it.
__device__ __forceinline__ void mbar_arrive_warp(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// One bounded attempt: the thread may be suspended for a system-dependent
// time while the phase is incomplete.  No suspend-time hint is given: with
// a long hint the waiter resumed measurably later after the phase completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait until the phase with the given parity has completed.  Returns false
// (and records DEV_TIMEOUT) if that takes longer than limit_ns nanoseconds
// (each launch passes its limit; FM_WAIT_LIMIT_NS unless a test shortened it).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* status,
                                          uint64_t limit_ns = FM_WAIT_LIMIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer() - t0 > limit_ns) {
      if (status) atomicOr(status, DEV_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}
// 4-D tiled load of one box into shared memory, completing `bar`'s tx count.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, uint32_t bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple
// of 16), completing `bar`'s tx count.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T-style product described by the descriptors.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same with 8-bit operands (kind::f8f6f4; K = 32 per MMA).
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem] (bf16): A read from tensor memory (lane = row of A).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same with 8-bit operands (kind::f8f6f4; K = 32 per MMA): A read from
// tensor memory, four e4m3 values of consecutive k per 32-bit column.
__device__ __forceinline__ void mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

#define FM_R8(b) "=r"(r[b + 0]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), \
                 "=r"(r[b + 4]), "=r"(r[b + 5]), "=r"(r[b + 6]), "=r"(r[b + 7])
#define FM_W8(b) "r"(r[b + 0]), "r"(r[b + 1]), "r"(r[b + 2]), "r"(r[b + 3]), \
                 "r"(r[b + 4]), "r"(r[b + 5]), "r"(r[b + 6]), "r"(r[b + 7])

// Each thread of a warp reads 32 consecutive 32-bit columns of its own TMEM
// lane (lane = warp's lane quarter * 32 + lane id).  Needs tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : FM_R8(0), FM_R8(8), FM_R8(16), FM_R8(24)
      : "r"(taddr));
}
#define FM_R32(b) FM_R8(b), FM_R8(b + 8), FM_R8(b + 16), FM_R8(b + 24)
// 64 consecutive columns in one instruction.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : FM_R32(0), FM_R32(32)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : FM_R8(0), FM_R8(8)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      FM_W8(0), FM_W8(8), FM_W8(16), FM_W8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      FM_W8(0), FM_W8(8)
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               FM_W8(0)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- registers
// Per-warpgroup register budget change (all warps of a warpgroup execute it).
// The sum of the budgets must stay within the registers the block was
// launched with, or setmaxnreg.inc waits forever: every caller documents the
// split and its launch checks the compiled register count.
template <uint32_t N>
__device__ __forceinline__ void regs_increase() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_decrease() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor for a 128B-swizzled operand.
//   K-major tile (rows of 64 bf16 along K): sbo = 1024 (next 8 rows);
//     lbo unused.  Step along K inside a 64-wide block by +32 B per 16
//     elements; the next 64-wide block of K is a separate 1024-aligned slab.
//   MN-major tile (rows of 64 bf16 along M/N, consecutive rows along K):
//     lbo = byte distance between 64-wide M/N slabs, sbo = 1024 (next 8 K rows).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}
// The same descriptor split in two words: every tile here has sbo = 1024,
// so the high word is one constant, and the low word holds the start address
// (address >> 4, 14 bits) and lbo.  Shared-memory addresses stay below 2^18,
// so adding (bytes >> 4) to a low word never carries out of the address
// field: with a tile's low word computed once, an MMA `bytes` further on in
// the tile needs one add.
constexpr uint32_t kSdescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__device__ __forceinline__ uint64_t sdesc_at(uint32_t lo, uint32_t bytes) {
  return (static_cast<uint64_t>(kSdescHi) << 32) | (lo + (bytes >> 4));
}
// Instruction descriptor, kind::f16 with bf16 A/B and fp32 accumulation.
// Instruction descriptor of a kind::f8f6f4 MMA with e4m3 A and B (format
// code 0 in both fields) and an f32 accumulator; both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4)                                  // D format: f32
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                                  // D format: f32
         | (1u << 7)                                // A format: bf16
         | (1u << 10)                               // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15)           // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16)           // B major-ness
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// Byte offset of element (row, col) of a 128B-swizzled bf16 tile made of
// 64-column slabs of `rows` rows each (slab-major).  Matches TMA SWIZZLE_128B
// for a 1024-aligned base.
__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t col,
                                                          uint32_t rows) {
  const uint32_t slab = col >> 6;
  const uint32_t c = col & 63u;
  const uint32_t chunk = (c >> 3) ^ (row & 7u);
  return slab * rows * 128u + row * 128u + chunk * 16u + (c & 7u) * 2u;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two floats to e4m3 (as pack_e4m3x4), x0 in the low byte of the result.
__device__ __forceinline__ uint32_t pack_e4m3x2(float x0, float x1) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(x1), "f"(x0));
  return r;
}
// Four floats to e4m3 (nearest, ties to even, saturating at +-448), x0 in
// the lowest byte: the order of consecutive K elements in a K-major tile.
__device__ __forceinline__ uint32_t pack_e4m3x4(float x0, float x1, float x2, float x3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Three-input maximum and packed (two-lane) fp32 arithmetic of sm_100+.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// (d0, d1) = (a0 * b + c, a1 * b + c)
__device__ __forceinline__ void fma2_bc(float& d0, float& d1, float a0, float a1, uint64_t b2,
                                        uint64_t c2) {
  uint64_t a, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b2), "l"(c2));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(d));
}
// (s0, s1) += (a0, a1)
__device__ __forceinline__ void add2_acc(float& s0, float& s1, float a0, float a1) {
  uint64_t s, a;
  asm("mov.b64 %0, {%1, %2};" : "=l"(s) : "f"(s0), "f"(s1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(s) : "l"(s), "l"(a));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(s));
}
// (d0, d1) = (a0 * b + c0, a1 * b + c1)
__device__ __forceinline__ void fma2_bv(float& d0, float& d1, float a0, float a1, uint64_t b2,
                                        float c0, float c1) {
  uint64_t a, c, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(c) : "f"(c0), "f"(c1));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b2), "l"(c));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(d));
}
// (d0, d1) = (p0 * (x0 - y0), p1 * (x1 - y1))
__device__ __forceinline__ void mulsub2(float& d0, float& d1, float p0, float p1, float x0,
                                        float x1, float y0, float y1) {
  uint64_t p, x, y, t;
  asm("mov.b64 %0, {%1, %2};" : "=l"(p) : "f"(p0), "f"(p1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(y0), "f"(y1));
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(t) : "l"(x), "l"(y));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(t) : "l"(p), "l"(t));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(t));
}
__device__ __forceinline__ uint64_t splat2(float x) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// One 32-byte global store (sm_100 and later; the address must be 32-byte
// aligned).  A warp's 32 lanes writing to 32 different rows touch as many
// cache lines per instruction as with 16-byte stores, so a row written in
// 32-byte pieces costs half the instructions and line accesses.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// Row-per-lane data (lane L holds NC chunks of W 32-bit words of row L, chunk
// i in c[W*i .. W*i + W-1]) regrouped for coalesced stores: within each
// group of NC lanes, an NC x NC transpose of the chunks in log2(NC)
// butterfly stages (stage b swaps bit b of the lane and of the chunk index
// through one exchange with lane ^ 2^b).  Afterwards lane NC*g + j holds in
// c[W*i ..] chunk j of row NC*g + i, so the i-th store of the warp writes NC
// rows of NC contiguous chunks each, instead of 32 rows of one chunk.
template <int NC, int W = 4>
__device__ __forceinline__ void transpose_chunks(uint32_t (&c)[W * NC]) {
  static_assert(NC == 2 || NC == 4 || NC == 8, "groups of 2, 4 or 8 lanes");
  const int j = threadIdx.x & (NC - 1);
#pragma unroll
  for (int b = 0; (1 << b) < NC; ++b) {
    const int m = 1 << b;
    const bool upper = ((j >> b) & 1) != 0;
#pragma unroll
    for (int k = 0; k < NC / 2; ++k) {
      // the pair of chunks whose indices differ in bit b only
      const int lo = ((k >> b) << (b + 1)) | (k & (m - 1));
      const int hi = lo | m;
      // a lane sends the chunk whose bit b differs from its own lane bit and
      // puts the partner's chunk in its place
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const uint32_t send = upper ? c[W * lo + w] : c[W * hi + w];
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, m);
        if (upper) c[W * lo + w] = recv;
        else c[W * hi + w] = recv;
      }
    }
  }
}

}  // namespace fm
