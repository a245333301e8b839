// Backward pass of masked attention on sm_103a.
//
// Gradients of exact attention by recomputation (FlashAttention-2 page,
// «Блочная обработка сохраняет общую нормализацию»: the probabilities are
// rebuilt from the saved row statistics instead of being stored; results
// match the plain definition up to floating-point order, «...поэтому выходы и
// градиенты проверяют с допусками»).  With P = exp(scale*S - LSE):
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  D_i = dO_i . O_i,
//   dK = scale dS^T Q,  dQ = scale dS K.
//
// Three kernels:
//   bwd_pre_kernel    D_i and -LSE_i*log2(e) per query row, padded to whole
//                     128-row tiles (-inf / 0 past Sq and on rows that see no
//                     key, so P = 0 there without a branch), and the zeroed
//                     fp32 dQ accumulator;
//   bwd_kernel        one unit = one (batch, head, k-tile): K and V stay in
//                     smem, the unit walks its column of non-empty q-tiles.
//                     Warps 0-7 (compute): thread r owns key row r (TMEM
//                     lane r, warp quarter w & 3) and half of the q columns
//                     (w >> 2) of S^T and dP^T, and half of dK / dV.
//                     Warps 8-11 (dQ): thread r owns q row r of the dQ tile
//                     and adds it into the fp32 accumulator.
//                     Warp 12: K/V loads, warp 14: Q/dO/LSE/D loads (TMA).
//                     Warp 13: one thread issues tcgen05:
//                       S^T = K Q^T, dP^T = V dO^T      (SS, both K-major)
//                       dV += P^T dO                     (P^T from TMEM, dO MN-major)
//                       dK += dS^T Q                     (dS^T smem K-major, Q MN-major)
//                       dQ  = dS K                       (dS smem MN-major, K MN-major)
//                     dQ tiles are added into an fp32 accumulator with
//                     vector atomics; dK, dV leave once per unit;
//   dq_convert_kernel fp32 accumulator -> bf16 dQ.
// TMEM (512 columns): [0,128) S^T then P^T (packed bf16, 64 columns);
// [128,256) dP^T then the dQ tile; [256,256+d) dV; [384,384+d) dK.
#include <cuda_bf16.h>

#include "fm_internal.h"
#include "fm_ptx.cuh"
#include "fm_tmap.h"

namespace fm {

// ------------------------------------------------------------------ preprocess
// One warp per 16 consecutive rows of one (b, h), over nQ*128 padded rows.
// Eight lanes share a row: lane (rr, part) = (lane >> 3, lane & 7) loads the
// 16-byte words part, part + 8, ... of row 4k + rr of O and of dO, so that a
// warp load covers four whole 128-byte segments; all 16 rows' loads are
// issued before any arithmetic (256 bytes in flight per thread).  The eight
// partial dot products of a row are summed with shuffles.  The warp also
// zeroes those rows of the fp32 dQ accumulator (the backward kernel adds
// into it), with the same coalesced pattern.
template <int D>
__global__ void __launch_bounds__(128) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dout,
                                                      int64_t os0, int64_t os1, int64_t os2,
                                                      const float* __restrict__ lse, int B, int H,
                                                      int Sq, int rows_pad, float* delta,
                                                      float* lse_log2, float* dq_acc) {
  constexpr int W = D / 64;  // 16-byte words per lane per row
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31, rr = lane >> 3, part = lane & 7;
  const int groups = rows_pad / 16;
  if (gw >= static_cast<long long>(B) * H * groups) return;
  const int bh = static_cast<int>(gw / groups);
  const int i0 = static_cast<int>(gw - static_cast<long long>(bh) * groups) * 16;
  const int b = bh / H, h = bh - b * H;
  uint4 a[4][W], g[4][W];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = i0 + 4 * k + rr;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      a[k][w] = make_uint4(0u, 0u, 0u, 0u);
      g[k][w] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (i < Sq) {
      const size_t at = static_cast<size_t>(b) * os0 + static_cast<size_t>(i) * os1 +
                        static_cast<size_t>(h) * os2;
      const uint4* a4 = reinterpret_cast<const uint4*>(o + at);
      const uint4* g4 = reinterpret_cast<const uint4*>(dout + at);
#pragma unroll
      for (int w = 0; w < W; ++w) {
        a[k][w] = __ldg(a4 + part + 8 * w);
        g[k][w] = __ldg(g4 + part + 8 * w);
      }
    }
  }
  float dot[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[k][w]);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g[k][w]);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 x = __bfloat1622float2(a2[t]);
        const float2 y = __bfloat1622float2(g2[t]);
        acc0 = fmaf(x.x, y.x, acc0);
        acc1 = fmaf(x.y, y.y, acc1);
      }
    }
    dot[k] = acc0 + acc1;
  }
#pragma unroll
  for (int sh = 1; sh < 8; sh <<= 1)
#pragma unroll
    for (int k = 0; k < 4; ++k) dot[k] += __shfl_xor_sync(0xffffffffu, dot[k], sh);
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = i0 + 4 * k + rr;
    if (i < Sq) {
      float4* acc_row = reinterpret_cast<float4*>(dq_acc + (static_cast<size_t>(bh) * Sq + i) * D);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) acc_row[part + 8 * c] = z;
    }
    if (part == 0) {
      float l2 = -INFINITY, dsum = 0.f;
      if (i < Sq) {
        const float L = lse[static_cast<size_t>(bh) * Sq + i];
        l2 = (L == -INFINITY) ? -INFINITY : -L * 1.4426950408889634f;
        dsum = dot[k];
      }
      delta[static_cast<size_t>(bh) * rows_pad + i] = dsum;
      lse_log2[static_cast<size_t>(bh) * rows_pad + i] = l2;
    }
  }
}

// ------------------------------------------------------------------ dQ convert
template <int D>
__global__ void dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* dq, int64_t s0,
                                  int64_t s1, int64_t s2, int H, int Sq, long long n_vec) {
  // one thread per 8 consecutive elements of one row
  for (long long v = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; v < n_vec;
       v += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long e = v * 8;
    const int c = static_cast<int>(e % D);
    const long long row = e / D;  // (b*H + h)*Sq + i
    const int i = static_cast<int>(row % Sq);
    const long long bh = row / Sq;
    const int h = static_cast<int>(bh % H);
    const int b = static_cast<int>(bh / H);
    const float4 x = *reinterpret_cast<const float4*>(acc + e);
    const float4 y = *reinterpret_cast<const float4*>(acc + e + 4);
    uint4 w;
    w.x = pack_bf16(x.x, x.y);
    w.y = pack_bf16(x.z, x.w);
    w.z = pack_bf16(y.x, y.y);
    w.w = pack_bf16(y.z, y.w);
    *reinterpret_cast<uint4*>(dq + b * s0 + static_cast<int64_t>(i) * s1 + h * s2 + c) = w;
  }
}

// ------------------------------------------------------------------ main kernel
template <int D>
struct BwdCfg {
  static constexpr int TILE = 128 * D * 2;   // one 128-row bf16 tile
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_Q = OFF_V + TILE;          // 2 stages
  static constexpr int OFF_DO = OFF_Q + 2 * TILE;     // 2 stages
  static constexpr int OFF_DS = OFF_DO + 2 * TILE;    // 128 x 128 bf16, [key][q]
  static constexpr int OFF_LD = OFF_DS + 128 * 128 * 2;  // 2 stages x (-LSE*log2e, D) fp32
  static constexpr int OFF_RING = OFF_LD + 2 * 1024;   // [UNIT_RING] claimed units
  static constexpr int OFF_BAR = OFF_RING + 16;
  static constexpr int NBAR = 24;
  static constexpr int SMEM_USED = OFF_BAR + NBAR * 8 + 16;
  // at least 120 KB so that one CTA (which takes all 512 TMEM columns) is
  // resident per SM
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  static constexpr uint32_t T_A = 0, T_B = 128, T_DV = 256, T_DK = 384, T_COLS = 512;
  // warpgroups 0-1: compute (P^T, dS^T, the dV/dK epilogue); warpgroup 2:
  // dQ drain; warpgroup 3: the K/V load warp, the MMA warp, the Q/dO load
  // warp and one idle warp
  static constexpr int THREADS = 512;
  // register split (setmaxnreg): 2 x 128 x REGS_COMPUTE + 128 x REGS_DQ +
  // 128 x REGS_PRODUCER = 65536 = THREADS x 128 registers at launch
  static constexpr uint32_t REGS_COMPUTE = 144, REGS_DQ = 152, REGS_PRODUCER = 72;
  static constexpr int MIN_LAUNCH_REGS =
      (2 * 128 * REGS_COMPUTE + 128 * REGS_DQ + 128 * REGS_PRODUCER + THREADS - 1) / THREADS;
};

enum { C_KVFULL = 0, C_KVEMPTY, C_QFULL0, C_QFULL1, C_QEMPTY0, C_QEMPTY1, C_SFULL, C_PREADY,
       C_DVDONE, C_DPFULL, C_DSREADY, C_DQFULL, C_DQEMPTY, C_ACCFULL, C_ACCEMPTY, C_DRAIN,
       C_UFULL0, C_UEMPTY0 = C_UFULL0 + 4 };
// Units are claimed at run time (one atomic counter per launch, in the
// workspace) by the Q/dO load warp, the first role to need the next unit,
// and handed to the other roles that walk units through a ring of
// UNIT_RING slots; U_READERS warps read every slot: the K/V load warp, the
// MMA warp, the eight compute warps and the four dQ warps.  Claiming just in
// time keeps the units in flight on all CTAs close together in the
// head-major order (Q/dO stay in L2).
constexpr int UNIT_RING = 4, U_READERS = 14;

struct BwdParams {
  int B, H, Hm, Sq, Skv, nQ, nK, n_units;
  float scale, scale_log2;
  const int32_t* bounds[4];
  const int32_t* col_count;
  const int32_t* col_list;
  const int32_t* order;
  int* next_unit;         // claim counter (zero at launch)
  const float* delta;     // [B][H][nQ*128]
  const float* lse_log2;  // [B][H][nQ*128]
  float* dq_acc;          // [B][H][Sq][D]
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int64_t k_stride[3], v_stride[3];
  int* status;
  uint64_t wait_ns;  // limit of every mbarrier wait
  int withhold;      // test hook: 2 = the compute warps withhold their first P-ready arrival
};

// Tile pipeline per q-tile t of a unit (MMA issue order on the left, other
// warps on the right; region A = TMEM [0,128), region B = [128,256)):
//   S^T(t) = K Q^T -> A       [after dV(t-1) read P^T(t-1) from A]
//                               dQ warps: dQ(t-1) from B to registers
//   dP^T(t) = V dO^T -> B     [after that read]
//                               compute: P^T(t) = exp2(S^T*scale*log2e - LSE*log2e) -> A
//                               dQ warps: atomics of dQ(t-1)
//   dV += P^T(t) dO           [after P^T(t)]
//                               compute: dS^T(t) = P^T o (dP^T - D) -> smem
//   dQ = dS K -> B, dK += dS^T Q   [after dS^T(t)]
// so the P, dS and dQ work overlaps S, dP and dV.
// Bits [a, b) of a 64-bit word, with a and b clipped to [0, 64].
__device__ __forceinline__ uint64_t row_span(int a, int b) {
  a = min(max(a, 0), 64);
  b = min(max(b, 0), 64);
  if (a >= b) return 0ull;
  const uint64_t below_b = b == 64 ? ~0ull : ((1ull << b) - 1ull);
  return below_b & ~((1ull << a) - 1ull);
}

template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    bwd_kernel(const __grid_constant__ BwdParams P, const __grid_constant__ CUtensorMap tmQ,
               const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __grid_constant__ CUtensorMap tmDO) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // swizzled tiles need a 1024-aligned base
    if (threadIdx.x == 0) atomicOr(P.status, DEV_LAYOUT);
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sDS = sbase + C::OFF_DS;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  volatile int* ring = reinterpret_cast<volatile int*>(smem + C::OFF_RING);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::NBAR * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8 + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int DQ_WARP0 = 8, TMA_WARP = 12, MMA_WARP = 13, QTMA_WARP = 14;

  if (tid == 0) {
    mbar_init(bar(C_KVFULL), 1);
    mbar_init(bar(C_KVEMPTY), 1);
    mbar_init(bar(C_QFULL0), 1);
    mbar_init(bar(C_QFULL1), 1);
    // a Q/dO stage is free once the tile's MMAs are done (commit) and the dQ
    // warps, which use its dO buffer as transpose scratch, are done (128)
    mbar_init(bar(C_QEMPTY0), 1 + 128);
    mbar_init(bar(C_QEMPTY1), 1 + 128);
    mbar_init(bar(C_SFULL), 1);
    mbar_init(bar(C_PREADY), 256);
    mbar_init(bar(C_DVDONE), 1);
    mbar_init(bar(C_DPFULL), 1);
    mbar_init(bar(C_DSREADY), 256);
    mbar_init(bar(C_DQFULL), 1);
    mbar_init(bar(C_DQEMPTY), 128);
    mbar_init(bar(C_ACCFULL), 1);
    mbar_init(bar(C_ACCEMPTY), 256);
    mbar_init(bar(C_DRAIN), 1);
    for (int r = 0; r < UNIT_RING; ++r) {
      mbar_init(bar(C_UFULL0 + r), 1);
      mbar_init(bar(C_UEMPTY0 + r), U_READERS);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), C::T_COLS);
    tmem_relinquish();
  }
  if (warp == TMA_WARP && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == QTMA_WARP && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmDO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const int rows_pad = P.nQ * kTile;

  auto wait = [&](int b, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (!mbar_wait(bar(b), parity, P.status, P.wait_ns)) {
      *abort_flag = 1;
      return false;
    }
    return true;
  };
  // for warps whose 32 lanes all take part: one answer per warp, so the
  // warp-collective TMEM instructions after it never run diverged
  auto wait_all = [&](int b, uint32_t parity) -> bool {
    const bool ok = wait(b, parity);
    return __all_sync(0xffffffffu, ok);
  };
  // unit u = (b*H + h)*nK + kj -> its column of q-tiles
  auto unit_info = [&](int idx, int& b, int& h, int& kj, const int32_t*& list) {
    const int u = P.order[idx];
    const int bh = u / P.nK;
    kj = u - bh * P.nK;
    b = bh / P.H;
    h = bh - b * P.H;
    const int col = (b * P.Hm + (P.Hm == 1 ? 0 : h)) * P.nK + kj;
    list = P.col_list + static_cast<size_t>(col) * P.nQ;
    return P.col_count[col];
  };
  // the n-th claimed unit (-1: none left, or the launch was aborted).
  // claimed_one: one thread of the warp reads and releases the ring slot;
  // claimed_all: all 32 lanes call it, lane 0 reads, the others get a copy
  auto claimed_one = [&](uint32_t& n) -> int {
    int idx = -1;
    const int r = n % UNIT_RING;
    if (wait(C_UFULL0 + r, (n / UNIT_RING) & 1)) {
      idx = ring[r];
      mbar_arrive(bar(C_UEMPTY0 + r));
    }
    ++n;
    return idx;
  };
  auto claimed_all = [&](uint32_t& n) -> int {
    uint32_t m = n;
    const int idx = lane == 0 ? claimed_one(m) : -1;
    ++n;
    return __shfl_sync(0xffffffffu, idx, 0);
  };

  if (warp >= TMA_WARP) {
  // producer warpgroup: small register budget (each role branch below runs
  // after the budget change, so the compiler allocates it within the budget)
  regs_decrease<C::REGS_PRODUCER>();
  if (warp == TMA_WARP) {
    // ------------------------------------------------------------ K / V loads
    // once per unit, after the previous unit's MMAs are done with K and V
    if (lane == 0) {
      uint32_t un = 0, cn = 0;
      while (true) {
        const int idx = claimed_one(cn);
        if (idx < 0) break;
        int b, h, kj;
        const int32_t* list;
        const int n = unit_info(idx, b, h, kj, list);
        if (n == 0) continue;
        if (un > 0 && !wait(C_KVEMPTY, (un - 1) & 1)) break;
        ++un;
        mbar_arrive_expect_tx(bar(C_KVFULL), 2 * C::TILE);
#pragma unroll
        for (int s = 0; s < D / 64; ++s) {
          tma_load_4d(sK + s * 16384, &tmK, bar(C_KVFULL), s * 64, h, kj * kTile, b);
          tma_load_4d(sV + s * 16384, &tmV, bar(C_KVFULL), s * 64, h, kj * kTile, b);
        }
      }
      // drain every issued copy before exit
      if (un > 0) mbar_wait(bar(C_KVFULL), (un - 1) & 1, P.status, P.wait_ns);
    }
    __syncwarp();
  } else if (warp == QTMA_WARP) {
    // ------------------------------------------------------------ Q / dO / LSE / D loads
    // its own warp, so the next unit's first tiles load as soon as a stage
    // is free, without waiting for the unit's K and V
    if (lane == 0) {
      uint32_t it = 0, cn = 0;
      bool ok = true;
      while (ok) {
        // claim the next unit and publish it to the other roles
        const int r = cn % UNIT_RING;
        const uint32_t use = cn / UNIT_RING;
        ++cn;
        if (use > 0 && !wait(C_UEMPTY0 + r, (use - 1) & 1)) break;
        int idx = atomicAdd(P.next_unit, 1);
        if (idx >= P.n_units) idx = -1;
        ring[r] = idx;
        mbar_arrive(bar(C_UFULL0 + r));
        if (idx < 0) break;
        int b, h, kj;
        const int32_t* list;
        const int n = unit_info(idx, b, h, kj, list);
        const size_t bh_row = (static_cast<size_t>(b) * P.H + h) * rows_pad;
        for (int t = 0; t < n; ++t, ++it) {
          const int qi = list[t] >> 2;
          const int st = it & 1;
          const uint32_t use = it >> 1;
          if (use > 0 && !wait(C_QEMPTY0 + st, (use - 1) & 1)) { ok = false; break; }
          const uint32_t fb = bar(C_QFULL0 + st);
          mbar_arrive_expect_tx(fb, 2 * C::TILE + 1024);
          const uint32_t sQ = sbase + C::OFF_Q + st * C::TILE;
          const uint32_t sDO = sbase + C::OFF_DO + st * C::TILE;
#pragma unroll
          for (int s = 0; s < D / 64; ++s) {
            tma_load_4d(sQ + s * 16384, &tmQ, fb, s * 64, h, qi * kTile, b);
            tma_load_4d(sDO + s * 16384, &tmDO, fb, s * 64, h, qi * kTile, b);
          }
          const uint32_t sLD = sbase + C::OFF_LD + st * 1024;
          bulk_load(sLD, P.lse_log2 + bh_row + qi * kTile, 512, fb);
          bulk_load(sLD + 512, P.delta + bh_row + qi * kTile, 512, fb);
        }
      }
      // drain every issued copy before exit
      for (uint32_t k = (it > 2u ? it - 2u : 0u); k < it; ++k)
        mbar_wait(bar(C_QFULL0 + (k & 1)), (k >> 1) & 1, P.status, P.wait_ns);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idSS = idesc_bf16(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t idKB = idesc_bf16(128, D, false, true);     // dV, dK (B MN-major)
      constexpr uint32_t idDQ = idesc_bf16(128, D, true, true);      // dQ (A, B MN-major)
      // operand descriptors of each buffer, computed once (each MMA adds a
      // constant offset); "k" = K-major view, "m" = MN-major view
      const uint32_t dKk = sdesc_lo(sK, 16), dKm = sdesc_lo(sK, 16384);
      const uint32_t dVk = sdesc_lo(sV, 16);
      const uint32_t dSk = sdesc_lo(sDS, 16), dSm = sdesc_lo(sDS, 16384);
      const uint32_t dQk0 = sdesc_lo(sbase + C::OFF_Q, 16), dQm0 = sdesc_lo(sbase + C::OFF_Q, 16384);
      const uint32_t dOk0 = sdesc_lo(sbase + C::OFF_DO, 16), dOm0 = sdesc_lo(sbase + C::OFF_DO, 16384);
      uint32_t it = 0, un = 0, cn = 0;
      bool ok = true;
      while (ok) {
        const int idx = claimed_one(cn);
        if (idx < 0) break;
        int b, h, kj;
        const int32_t* list;
        const int n = unit_info(idx, b, h, kj, list);
        if (n == 0) continue;
        if (!wait(C_KVFULL, un & 1)) break;
        for (int t = 0; t < n; ++t, ++it) {
          const int st = it & 1;
          const uint32_t stage = st * (C::TILE >> 4);
          const uint32_t dQk = dQk0 + stage, dQm = dQm0 + stage;
          const uint32_t dOk = dOk0 + stage, dOm = dOm0 + stage;
          if (!wait(C_QFULL0 + st, (it >> 1) & 1)) { ok = false; break; }
          // S^T overwrites P^T of the previous tile in region A: the dV that
          // reads it was issued earlier, and MMAs issued by this thread run in
          // issue order
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(tbase + C::T_A, sdesc_at(dKk, koff), sdesc_at(dQk, koff), idSS,
                   kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(C_SFULL));
          // dP^T into region B once the previous dQ tile was drained
          if (it > 0 && !wait(C_DQEMPTY, (it - 1) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(tbase + C::T_B, sdesc_at(dVk, koff), sdesc_at(dOk, koff), idSS,
                   kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(C_DPFULL));
          // dV += P^T dO once P^T is in TMEM (and the previous unit's dV/dK were read)
          if (!wait(C_PREADY, it & 1)) { ok = false; break; }
          if (t == 0 && un > 0 && !wait(C_ACCEMPTY, (un - 1) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // P^T of q columns 0..63 sits in TMEM columns [0,32), 64..127 in [64,96)
            const uint32_t acol = (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
            mma_ts(tbase + C::T_DV, tbase + C::T_A + acol,
                   sdesc_at(dOm, kk * 2048), idKB, (t > 0 || kk > 0) ? 1u : 0u);
          }
          // dQ = dS K and dK += dS^T Q once dS^T is in smem; dQ first, so its
          // drain (which frees region B for the next dP^T) starts earlier.
          // The dQ warps may then use this stage's dO buffer while dK runs:
          // dK reads Q and dS^T only
          if (!wait(C_DSREADY, it & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tbase + C::T_B, sdesc_at(dSm, kk * 2048), sdesc_at(dKm, kk * 2048), idDQ,
                   kk > 0 ? 1u : 0u);
          mma_commit(bar(C_DQFULL));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(tbase + C::T_DK, sdesc_at(dSk, aoff), sdesc_at(dQm, kk * 2048), idKB,
                   (t > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(C_QEMPTY0 + st));
        }
        if (!ok) break;
        mma_commit(bar(C_KVEMPTY));
        mma_commit(bar(C_ACCFULL));
        ++un;
      }
      mma_commit(bar(C_DRAIN));
      mbar_wait(bar(C_DRAIN), 0, P.status, P.wait_ns);
    }
    __syncwarp();
  }  // warp 15: spare warp of the producer warpgroup
  } else if (warp >= DQ_WARP0) {
    // ------------------------------------------------------------ dQ drain
    // Thread r holds q row r of the tile in region B (TMEM lane r): all D
    // columns in one TMEM round trip, region B released for the next dP^T.
    // Straight from registers each fp32 atomic of a warp would touch 32
    // different rows; instead the warp transposes 32 x 32 blocks through a
    // 4 KB patch so that every reduction instruction covers four rows x 128
    // contiguous bytes.  The patch lies in the dO buffer of this tile's Q/dO
    // stage: the tile's MMAs have finished with it (they committed before
    // the dQ tile), and the stage is refilled only after these warps arrive
    // on its release barrier.  These warps do nothing else, so the
    // reductions overlap the compute warps' P^T / dS^T work and the MMAs.
    regs_increase<C::REGS_DQ>();
    const int quarter = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t it = 0, cn = 0;
    bool ok = true;
    while (ok) {
      const int idx = claimed_all(cn);
      if (idx < 0) break;
      int b, h, kj;
      const int32_t* list;
      const int n = unit_info(idx, b, h, kj, list);
      float* acc_bh = P.dq_acc + (static_cast<size_t>(b) * P.H + h) * P.Sq * D;
      for (int t = 0; t < n; ++t, ++it) {
        const int qi = list[t] >> 2;
        const int st = it & 1;
        if (!wait_all(C_DQFULL, it & 1)) { ok = false; break; }
        tc_fence_after();
        uint32_t raw[D];
#pragma unroll
        for (int c = 0; c < D / 64; ++c) tmem_ld64(tbase + lane_off + C::T_B + 64 * c, raw + 64 * c);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(C_DQEMPTY));
        const uint32_t patch = sbase + C::OFF_DO + st * C::TILE + quarter * 4096;
        const int row0 = qi * kTile + quarter * 32;  // first q row of this warp
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {  // 32-column blocks
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t chunk = static_cast<uint32_t>(j) ^ static_cast<uint32_t>(lane & 7);
            const int e = c * 32 + j * 4;
            st_shared_v4(patch + lane * 128 + chunk * 16,
                         __float_as_uint(__uint_as_float(raw[e]) * P.scale),
                         __float_as_uint(__uint_as_float(raw[e + 1]) * P.scale),
                         __float_as_uint(__uint_as_float(raw[e + 2]) * P.scale),
                         __float_as_uint(__uint_as_float(raw[e + 3]) * P.scale));
          }
          __syncwarp();
          const int j = lane & 7;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rl = i * 4 + (lane >> 3);  // row within the warp's 32
            const uint32_t chunk = static_cast<uint32_t>(j) ^ static_cast<uint32_t>(rl & 7);
            float4 v;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                         : "r"(patch + rl * 128 + chunk * 16));
            if (row0 + rl < P.Sq)
              atomicAdd(reinterpret_cast<float4*>(acc_bh + static_cast<size_t>(row0 + rl) * D +
                                                  c * 32 + j * 4),
                        v);
          }
          __syncwarp();
        }
        // the stage may be refilled by TMA (async proxy) after these accesses
        fence_proxy_async_smem();
        mbar_arrive(bar(C_QEMPTY0 + st));
      }
    }
  } else {
    // ------------------------------------------------------------ compute warps
    regs_increase<C::REGS_COMPUTE>();
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;  // TMEM lane: key row (S^T, dP^T, dK, dV), q row (dQ)
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int c0 = half * 64;           // this thread's 64 of the 128 q columns
    uint32_t it = 0, un = 0, cn = 0;
    bool ok = true;
    while (ok) {
      const int idx = claimed_all(cn);
      if (idx < 0) break;
      int b, h, kj;
      const int32_t* list;
      const int n = unit_info(idx, b, h, kj, list);
      const int key = kj * kTile + r;
      __nv_bfloat16* dk_row = P.dk + b * P.k_stride[0] + static_cast<int64_t>(key) * P.k_stride[1] +
                              h * P.k_stride[2] + half * (D / 2);
      __nv_bfloat16* dv_row = P.dv + b * P.v_stride[0] + static_cast<int64_t>(key) * P.v_stride[1] +
                              h * P.v_stride[2] + half * (D / 2);
      if (n == 0) {
        if (key < P.Skv) {
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            reinterpret_cast<uint4*>(dk_row)[c] = z;
            reinterpret_cast<uint4*>(dv_row)[c] = z;
          }
        }
        continue;
      }
      // this thread's key column bounds (beyond Skv: hidden from every row)
      int lts = 0, lte = 0x7fffffff, uts = 0, ute = 0;
      if (key < P.Skv) {
        const size_t at = static_cast<size_t>(b * P.Hm + (P.Hm == 1 ? 0 : h)) * P.Skv + key;
        lts = __ldg(P.bounds[0] + at);
        lte = __ldg(P.bounds[1] + at);
        uts = __ldg(P.bounds[2] + at);
        ute = __ldg(P.bounds[3] + at);
      }
      const bool key_ragged = (kj == P.nK - 1) && (P.Skv & (kTile - 1));
      for (int t = 0; t < n; ++t, ++it) {
        const int e = list[t];
        const int qi = e >> 2;
        const bool partial = ((e & 3) == CLS_PARTIAL) || key_ragged;
        const int st = it & 1;
        const float* lse_s = reinterpret_cast<const float*>(smem + C::OFF_LD + st * 1024) + c0;
        const float* del_s = lse_s + 128;
        // ---- P^T = exp2(S^T * scale*log2e - LSE*log2e), hidden entries 0
        if (!wait_all(C_SFULL, it & 1)) { ok = false; break; }
        // the LSE/D of this stage arrived with the Q/dO tiles
        if (!wait_all(C_QFULL0 + st, (it >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        float p[64];
        {
          uint32_t raw[64];
          tmem_ld64(tbase + lane_off + C::T_A + c0, raw);
          tmem_wait_ld();
          // two columns per packed FMA: S^T * scale*log2e + (-LSE*log2e)
          const uint64_t sc2 = splat2(P.scale_log2);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 L = *reinterpret_cast<const float4*>(lse_s + 4 * i);
            float a0, a1, a2, a3;
            fma2_bv(a0, a1, __uint_as_float(raw[4 * i + 0]), __uint_as_float(raw[4 * i + 1]), sc2,
                    L.x, L.y);
            fma2_bv(a2, a3, __uint_as_float(raw[4 * i + 2]), __uint_as_float(raw[4 * i + 3]), sc2,
                    L.z, L.w);
            p[4 * i + 0] = ex2(a0);
            p[4 * i + 1] = ex2(a1);
            p[4 * i + 2] = ex2(a2);
            p[4 * i + 3] = ex2(a3);
          }
        }
        if (partial) {
          // the rows q0 .. q0+63 hidden from this key form at most two
          // intervals: one 64-bit mask, then a bit test per entry
          const int q0 = qi * kTile + c0;
          const uint64_t hm = row_span(lts - q0, lte - q0) | row_span(uts - q0, ute - q0);
          if (hm != 0) {
            const uint32_t m0 = static_cast<uint32_t>(hm), m1 = static_cast<uint32_t>(hm >> 32);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              p[c] = ((m0 >> c) & 1u) ? 0.f : p[c];
              p[c + 32] = ((m1 >> c) & 1u) ? 0.f : p[c + 32];
            }
          }
        }
        {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) pk[c] = pack_bf16(p[2 * c], p[2 * c + 1]);
          // into the TMEM columns this thread read: [c0, c0 + 32)
          tmem_st32(tbase + lane_off + C::T_A + c0, pk);
          tmem_wait_st();
        }
        tc_fence_before();
        // (a test of the wait limit withholds the first P-ready arrival: the
        // MMA thread then gives up on it and the launch unwinds with DEV_TIMEOUT)
        if (!(P.withhold == 2 && it == 0)) mbar_arrive(bar(C_PREADY));
        // ---- dS^T = P^T o (dP^T - D), to smem as bf16 [key][q] (slab = half)
        if (!wait_all(C_DPFULL, it & 1)) { ok = false; break; }
        tc_fence_after();
        {
          uint32_t raw[64];
          tmem_ld64(tbase + lane_off + C::T_B + c0, raw);
          tmem_wait_ld();
          const uint32_t row_base = sDS + half * 16384 + r * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float4 Dv = *reinterpret_cast<const float4*>(del_s + 8 * j + 4 * i);
              const int c = 8 * j + 4 * i;
              float s0, s1, s2, s3;
              mulsub2(s0, s1, p[c + 0], p[c + 1], __uint_as_float(raw[c + 0]),
                      __uint_as_float(raw[c + 1]), Dv.x, Dv.y);
              mulsub2(s2, s3, p[c + 2], p[c + 3], __uint_as_float(raw[c + 2]),
                      __uint_as_float(raw[c + 3]), Dv.z, Dv.w);
              w[2 * i] = pack_bf16(s0, s1);
              w[2 * i + 1] = pack_bf16(s2, s3);
            }
            const uint32_t chunk = static_cast<uint32_t>(j) ^ static_cast<uint32_t>(r & 7);
            st_shared_v4(row_base + chunk * 16, w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(C_DSREADY));
      }
      if (!ok) break;
      // ---- epilogue: dV and scale * dK, this thread's half of the columns;
      // both are read from TMEM first so the next unit's MMAs may start
      if (!wait_all(C_ACCFULL, un & 1)) { ok = false; break; }
      tc_fence_after();
      uint32_t rv[D / 2], rk[D / 2];
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tmem_ld32(tbase + lane_off + C::T_DV + half * (D / 2) + c * 32, rv + 32 * c);
        tmem_ld32(tbase + lane_off + C::T_DK + half * (D / 2) + c * 32, rk + 32 * c);
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(C_ACCEMPTY));
      if constexpr (D == 128) {
        // Each thread holds 64 columns of its key row of dV and of dK.
        // Stored straight from registers, every store instruction of a warp
        // would touch 32 rows; instead each 32 x 64 bf16 block goes through
        // this warp's 4 KB patch of the dS^T buffer (idle: the unit's MMAs
        // are done, and these warps write the next dS^T only afterwards), so
        // that an instruction stores four rows x 128 contiguous bytes.
        const uint32_t patch = sDS + half * 16384 + quarter * 4096;
        const int key0 = kj * kTile + quarter * 32;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const float sc = m ? P.scale : 1.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t* x = m ? rk + 8 * j : rv + 8 * j;
            const uint32_t chunk = static_cast<uint32_t>(j) ^ static_cast<uint32_t>(lane & 7);
            st_shared_v4(patch + lane * 128 + chunk * 16,
                         pack_bf16(__uint_as_float(x[0]) * sc, __uint_as_float(x[1]) * sc),
                         pack_bf16(__uint_as_float(x[2]) * sc, __uint_as_float(x[3]) * sc),
                         pack_bf16(__uint_as_float(x[4]) * sc, __uint_as_float(x[5]) * sc),
                         pack_bf16(__uint_as_float(x[6]) * sc, __uint_as_float(x[7]) * sc));
          }
          __syncwarp();
          __nv_bfloat16* base = m ? P.dk : P.dv;
          const int64_t* st3 = m ? P.k_stride : P.v_stride;
          const int jj = lane & 7;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rl = i * 4 + (lane >> 3);  // row within the warp's 32 keys
            const uint32_t chunk = static_cast<uint32_t>(jj) ^ static_cast<uint32_t>(rl & 7);
            uint4 val;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                         : "r"(patch + rl * 128 + chunk * 16));
            const int kr = key0 + rl;
            if (kr < P.Skv)
              *reinterpret_cast<uint4*>(base + b * st3[0] + static_cast<int64_t>(kr) * st3[1] +
                                        h * st3[2] + half * (D / 2) + jj * 8) = val;
          }
          __syncwarp();
        }
      } else if (key < P.Skv) {
        const float sc = P.scale;
        uint4* dv_dst = reinterpret_cast<uint4*>(dv_row);
        uint4* dk_dst = reinterpret_cast<uint4*>(dk_row);
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
          dv_dst[i] = make_uint4(pack_bf16(__uint_as_float(rv[8 * i + 0]), __uint_as_float(rv[8 * i + 1])),
                                 pack_bf16(__uint_as_float(rv[8 * i + 2]), __uint_as_float(rv[8 * i + 3])),
                                 pack_bf16(__uint_as_float(rv[8 * i + 4]), __uint_as_float(rv[8 * i + 5])),
                                 pack_bf16(__uint_as_float(rv[8 * i + 6]), __uint_as_float(rv[8 * i + 7])));
          dk_dst[i] = make_uint4(pack_bf16(__uint_as_float(rk[8 * i + 0]) * sc, __uint_as_float(rk[8 * i + 1]) * sc),
                                 pack_bf16(__uint_as_float(rk[8 * i + 2]) * sc, __uint_as_float(rk[8 * i + 3]) * sc),
                                 pack_bf16(__uint_as_float(rk[8 * i + 4]) * sc, __uint_as_float(rk[8 * i + 5]) * sc),
                                 pack_bf16(__uint_as_float(rk[8 * i + 6]) * sc, __uint_as_float(rk[8 * i + 7]) * sc));
        }
      }
      ++un;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tbase, C::T_COLS);
  }
}

template <int D>
static fm_status launch_bwd_d(const Plan& p, const fm_desc& desc, const TensorArgs& t, char* ws,
                              cudaStream_t s) {
  using C = BwdCfg<D>;
  const int rows_pad = p.nQ * kTile;
  float* delta = reinterpret_cast<float*>(ws + p.L.delta);
  float* lse2 = reinterpret_cast<float*>(ws + p.L.lse_log2);
  float* acc = reinterpret_cast<float*>(ws + p.L.dq_acc);
  {
    // four warps per block, one warp per 16 rows (rows_pad is a multiple of 128)
    const long long rows = static_cast<long long>(p.B) * p.H * rows_pad;
    const long long blocks = (rows / 16 + 3) / 4;
    prof_begin(K_BWD_PRE, s);
    bwd_pre_kernel<D><<<static_cast<unsigned>(blocks), 128, 0, s>>>(
        static_cast<const __nv_bfloat16*>(t.o), static_cast<const __nv_bfloat16*>(t.dout),
        desc.o_stride[0], desc.o_stride[1], desc.o_stride[2], t.lse_in, p.B, p.H, p.Sq, rows_pad,
        delta, lse2, acc);
    prof_end(K_BWD_PRE, s);
    if (cudaGetLastError() != cudaSuccess) return FM_ERR_CUDA;
  }
  CUtensorMap tq, tk, tv, tdo;
  if (!make_tmap_bshd(&tq, t.q, p.B, p.Sq, p.H, D, desc.q_stride, 128) ||
      !make_tmap_bshd(&tk, t.k, p.B, p.Skv, p.H, D, desc.k_stride, 128) ||
      !make_tmap_bshd(&tv, t.v, p.B, p.Skv, p.H, D, desc.v_stride, 128) ||
      !make_tmap_bshd(&tdo, t.dout, p.B, p.Sq, p.H, D, desc.o_stride, 128))
    return FM_ERR_CUDA;
  BwdParams P{};
  P.B = p.B; P.H = p.H; P.Hm = p.Hm; P.Sq = p.Sq; P.Skv = p.Skv; P.nQ = p.nQ; P.nK = p.nK;
  P.n_units = p.B * p.H * p.nK;
  P.scale = t.scale;
  P.scale_log2 = t.scale * 1.4426950408889634f;
  for (int i = 0; i < 4; ++i) P.bounds[i] = t.bounds[i];
  P.col_count = reinterpret_cast<const int32_t*>(ws + p.L.col_count);
  P.col_list = reinterpret_cast<const int32_t*>(ws + p.L.col_list);
  P.order = reinterpret_cast<const int32_t*>(ws + p.L.bwd_order);
  P.next_unit = reinterpret_cast<int*>(ws + p.L.status) + 1;
  P.delta = delta;
  P.lse_log2 = lse2;
  P.dq_acc = acc;
  P.dk = static_cast<__nv_bfloat16*>(t.dk);
  P.dv = static_cast<__nv_bfloat16*>(t.dv);
  for (int i = 0; i < 3; ++i) {
    P.k_stride[i] = desc.k_stride[i];
    P.v_stride[i] = desc.v_stride[i];
  }
  P.status = reinterpret_cast<int*>(ws + p.L.status);
  const TestHooks th = test_hooks();
  P.wait_ns = th.wait_ns;
  P.withhold = th.withhold;
  auto kern = bwd_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
      cudaSuccess)
    return FM_ERR_CUDA;
  {
    // the setmaxnreg split must fit in the registers the block launches with
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return FM_ERR_CUDA;
    if (fa.numRegs < C::MIN_LAUNCH_REGS) return FM_ERR_UNSUPPORTED;
  }
  const int grid = P.n_units < num_sms() ? P.n_units : num_sms();
  prof_begin(K_BWD, s);
  kern<<<grid, C::THREADS, C::SMEM, s>>>(P, tq, tk, tv, tdo);
  prof_end(K_BWD, s);
  if (cudaGetLastError() != cudaSuccess) return FM_ERR_CUDA;
  {
    const long long n_vec = static_cast<long long>(p.B) * p.H * p.Sq * (D / 8);
    const long long want = (n_vec + 255) / 256;
    const int blocks = static_cast<int>(want < 8192 ? want : 8192);
    prof_begin(K_DQ_CONVERT, s);
    dq_convert_kernel<D><<<blocks, 256, 0, s>>>(acc, static_cast<__nv_bfloat16*>(t.dq),
                                                desc.q_stride[0], desc.q_stride[1],
                                                desc.q_stride[2], p.H, p.Sq, n_vec);
    prof_end(K_DQ_CONVERT, s);
    if (cudaGetLastError() != cudaSuccess) return FM_ERR_CUDA;
  }
  return FM_OK;
}

fm_status launch_bwd(const Plan& p, const fm_desc& desc, const TensorArgs& t, char* ws,
                     cudaStream_t s) {
  if (p.d == 64) return launch_bwd_d<64>(p, desc, t, ws, s);
  if (p.d == 128) return launch_bwd_d<128>(p, desc, t, ws, s);
  return FM_ERR_UNSUPPORTED;
}

}  // namespace fm
