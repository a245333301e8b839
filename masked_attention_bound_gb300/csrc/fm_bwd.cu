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
// Three kernels, each over its own units:
//   bwd_pre_kernel  D_i and -LSE_i*log2(e) per query row, padded to whole
//                   128-row tiles (-inf / 0 past Sq and on rows that see no
//                   key, so P = 0 there without a branch);
//   bwd_kv_kernel   one unit = one (batch, head, k-tile): K and V stay in
//                   smem, the unit walks its column of non-empty q-tiles and
//                   accumulates dV and dK in TMEM (four GEMMs per tile);
//   bwd_dq_kernel   one unit = one (batch, head, q-tile): Q and dO stay in
//                   smem, the unit walks its row of non-empty k-tiles and
//                   accumulates dQ in TMEM (three GEMMs per tile), written
//                   once as bf16.
// dQ is not reduced across k-tiles through global memory: each q-tile row
// sums its own dQ on chip.  The price is S and dP computed twice (once per
// kernel); the gain is no fp32 accumulator to clear, reduce into and
// convert, and two kernels whose tensor-core work hides the softmax-side
// arithmetic.
#include <cuda_bf16.h>

#include "fm_internal.h"
#include "fm_ptx.cuh"
#include "fm_tmap.h"

namespace fm {

// ------------------------------------------------------------------ preprocess
// One warp per 4 consecutive rows of one (b, h), over nQ*128 padded rows.
// Eight lanes share a row: lane (rr, part) = (lane >> 3, lane & 7) loads the
// 16-byte words part, part + 8, ... of row rr of O and of dO, so that a warp
// load covers four whole 128-byte segments.  Many short warps keep more of
// HBM busy than fewer warps with more rows each (4 rows per warp measured
// 17 % faster than 16 on the 32K workload).  The eight partial dot products
// of a row are summed with shuffles.
template <int D>
__global__ void __launch_bounds__(128) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dout,
                                                      int64_t os0, int64_t os1, int64_t os2,
                                                      const float* __restrict__ lse, int B, int H,
                                                      int Sq, int rows_pad, float* delta,
                                                      float* lse_log2) {
  constexpr int W = D / 64;  // 16-byte words per lane
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31, rr = lane >> 3, part = lane & 7;
  const int groups = rows_pad / 4;
  if (gw >= static_cast<long long>(B) * H * groups) return;
  const int bh = static_cast<int>(gw / groups);
  const int i = static_cast<int>(gw - static_cast<long long>(bh) * groups) * 4 + rr;
  const int b = bh / H, h = bh - b * H;
  uint4 a[W], g[W];
#pragma unroll
  for (int w = 0; w < W; ++w) {
    a[w] = make_uint4(0u, 0u, 0u, 0u);
    g[w] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (i < Sq) {
    const size_t at = static_cast<size_t>(b) * os0 + static_cast<size_t>(i) * os1 +
                      static_cast<size_t>(h) * os2;
    const uint4* a4 = reinterpret_cast<const uint4*>(o + at);
    const uint4* g4 = reinterpret_cast<const uint4*>(dout + at);
#pragma unroll
    for (int w = 0; w < W; ++w) {
      a[w] = __ldg(a4 + part + 8 * w);
      g[w] = __ldg(g4 + part + 8 * w);
    }
  }
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[w]);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g[w]);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 x = __bfloat1622float2(a2[t]);
      const float2 y = __bfloat1622float2(g2[t]);
      acc0 = fmaf(x.x, y.x, acc0);
      acc1 = fmaf(x.y, y.y, acc1);
    }
  }
  float dot = acc0 + acc1;
#pragma unroll
  for (int sh = 1; sh < 8; sh <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, sh);
  if (part == 0) {
    float l2 = -INFINITY, dsum = 0.f;
    if (i < Sq) {
      const float L = lse[static_cast<size_t>(bh) * Sq + i];
      l2 = (L == -INFINITY) ? -INFINITY : -L * 1.4426950408889634f;
      dsum = dot;
    }
    delta[static_cast<size_t>(bh) * rows_pad + i] = dsum;
    lse_log2[static_cast<size_t>(bh) * rows_pad + i] = l2;
  }
}

// Units are claimed at run time (one atomic counter per kernel, in the
// workspace) by the warp that loads the per-unit operands, the first role to
// need the next unit, and handed to the roles that walk units through a
// ring of UNIT_RING slots.  Claiming just in time keeps the units in flight
// on all CTAs close together in the head-major order (the streamed operands
// stay in L2).
constexpr int UNIT_RING = 4;

struct BwdParams {
  int B, H, Hm, Sq, Skv, nQ, nK, n_units;
  int Hkv, G;  // K/V heads; query heads per K/V head (head h reads K/V head h / G)
  float scale, scale_log2;
  const int32_t* bounds[4];
  const int32_t* list_count;  // units' tile counts: columns (dK/dV) or rows (dQ)
  const int32_t* list;        // units' tile lists, entry = tile << 2 | class
  const int32_t* order;
  int* next_unit;             // claim counter (zero at launch)
  const float* delta;         // [B][H][nQ*128]
  const float* lse_log2;      // [B][H][nQ*128]
  const int32_t* row_mask;    // dQ: first visibility-mask slot of a q-tile row, -1: none
  const uint8_t* masks;       // dQ: 2 KB per slot, 128 rows x 128 column bits, set = hidden
  __nv_bfloat16* out0;        // dK (dK/dV kernel) or dQ (dQ kernel)
  __nv_bfloat16* out1;        // dV (dK/dV kernel)
  int64_t s0[3], s1[3];       // strides of out0, out1
  int* status;
  uint64_t wait_ns;  // limit of every mbarrier wait
  int withhold;      // test hook: 2 = the dK/dV compute warps withhold their first P-ready arrival,
                     // 3 = the dQ compute warps their first dS-ready arrival
};

// Bits [a, b) of a 64-bit word, with a and b clipped to [0, 64].
__device__ __forceinline__ uint64_t row_span(int a, int b) {
  a = min(max(a, 0), 64);
  b = min(max(b, 0), 64);
  if (a >= b) return 0ull;
  const uint64_t below_b = b == 64 ? ~0ull : ((1ull << b) - 1ull);
  return below_b & ~((1ull << a) - 1ull);
}

// ------------------------------------------------------------------ dK / dV kernel
template <int D>
struct KvCfg {
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
  // the K/V load warp, the MMA warp, the Q/dO load warp and one idle warp
  static constexpr int THREADS = 384;
  // register split (setmaxnreg): 2 x 128 x REGS_COMPUTE + 128 x REGS_PRODUCER
  // = 64512 = THREADS x 168 registers at launch
  static constexpr uint32_t REGS_COMPUTE = 216, REGS_PRODUCER = 72;
  static constexpr int MIN_LAUNCH_REGS =
      (2 * 128 * REGS_COMPUTE + 128 * REGS_PRODUCER + THREADS - 1) / THREADS;
};

enum { A_KFULL = 0, A_KEMPTY, A_VFULL, A_VEMPTY, A_QFULL0, A_QFULL1, A_QEMPTY0, A_QEMPTY1,
       A_SFULL, A_PREADY, A_DPFULL, A_DSREADY, A_ACCFULL, A_ACCEMPTY, A_DRAIN, A_UFULL0,
       A_UEMPTY0 = A_UFULL0 + 4 };
// every slot of the unit ring is read by the K/V load warp, the MMA warp and
// the eight compute warps
constexpr int A_READERS = 10;

// MMA issue order (region A = TMEM [0,128), region B = [128,256); t-1 is the
// previous tile of the same unit):
//   S^T(t) = K Q^T -> A       [after dV(t-1) read P^T(t-1) from A]
//   dK += dS^T(t-1) Q(t-1)     [after dS^T(t-1) is in smem]
//   dP^T(t) = V dO^T -> B     [B free: the compute warps read dP^T(t-1) before dS^T(t-1)]
//   dV += P^T(t) dO(t)        [after P^T(t) is in TMEM]
// and the unit's last dK after its last tile.  The compute warps work out
// P^T(t) while dK(t-1) and dP^T(t) run, and dS^T(t) while dV(t) and S^T(t+1)
// run, so the tensor pipe need not wait for them.  dS^T(t) goes into the
// one dS buffer only after dP^T(t) has completed, which implies dK(t-1),
// issued before it by the same thread, has completed too.
// WIDE: every dK and dV row starts on a 32-byte boundary (32-byte epilogue
// stores at d = 128)
template <int D, bool WIDE>
__global__ void __launch_bounds__(KvCfg<D>::THREADS, 1)
    bwd_kv_kernel(const __grid_constant__ BwdParams P, const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmDO) {
  using C = KvCfg<D>;
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
  constexpr int KV_WARP = 8, MMA_WARP = 9, Q_WARP = 10;

  if (tid == 0) {
    // K is read by the unit's S^T products only, V by its dP^T products: each
    // is free for the next unit as soon as its last reader is done
    mbar_init(bar(A_KFULL), 1);
    mbar_init(bar(A_KEMPTY), 1);
    mbar_init(bar(A_VFULL), 1);
    mbar_init(bar(A_VEMPTY), 1);
    mbar_init(bar(A_QFULL0), 1);
    mbar_init(bar(A_QFULL1), 1);
    mbar_init(bar(A_QEMPTY0), 1);  // the tile's last MMA (its dK) is done
    mbar_init(bar(A_QEMPTY1), 1);
    mbar_init(bar(A_SFULL), 1);
    mbar_init(bar(A_PREADY), 8);  // one arrival per compute warp
    mbar_init(bar(A_DPFULL), 1);
    mbar_init(bar(A_DSREADY), 8);
    mbar_init(bar(A_ACCFULL), 1);
    mbar_init(bar(A_ACCEMPTY), 8);
    mbar_init(bar(A_DRAIN), 1);
    for (int r = 0; r < UNIT_RING; ++r) {
      mbar_init(bar(A_UFULL0 + r), 1);
      mbar_init(bar(A_UEMPTY0 + r), A_READERS);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), C::T_COLS);
    tmem_relinquish();
  }
  if (warp == KV_WARP && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == Q_WARP && lane == 0) {
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
  // k-tile column kj of query head h (its mask head)
  auto col_of = [&](int b, int h, int kj) { return (b * P.Hm + (P.Hm == 1 ? 0 : h)) * P.nK + kj; };
  // unit u = (b*Hkv + hk)*nK + kj -> the columns of q-tiles of the G query
  // heads h = hk*G + j that read K/V head hk, walked one head after another;
  // returns their total tile count, and the first head's column and count
  // (so that a walk starts without loading them again)
  auto unit_info = [&](int idx, int& b, int& hk, int& kj, const int32_t*& list0, int& n0) {
    const int u = P.order[idx];
    const int bh = u / P.nK;
    kj = u - bh * P.nK;
    b = bh / P.Hkv;
    hk = bh - b * P.Hkv;
    const int col0 = col_of(b, hk * P.G, kj);
    list0 = P.list + static_cast<size_t>(col0) * P.nQ;
    n0 = P.list_count[col0];
    int n = n0;
    for (int j = 1; j < P.G; ++j) n += P.list_count[col_of(b, hk * P.G + j, kj)];
    return n;
  };
  // the n-th claimed unit (-1: none left, or the launch was aborted).
  // claimed_one: one thread of the warp reads and releases the ring slot;
  // claimed_all: all 32 lanes call it, lane 0 reads, the others get a copy
  auto claimed_one = [&](uint32_t& n) -> int {
    int idx = -1;
    const int r = n % UNIT_RING;
    if (wait(A_UFULL0 + r, (n / UNIT_RING) & 1)) {
      idx = ring[r];
      mbar_arrive(bar(A_UEMPTY0 + r));
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

  if (warp >= KV_WARP) {
  // producer warpgroup: small register budget (each role branch below runs
  // after the budget change, so the compiler allocates it within the budget)
  regs_decrease<C::REGS_PRODUCER>();
  if (warp == KV_WARP) {
    // ------------------------------------------------------------ K / V loads
    // once per unit, after the previous unit's MMAs are done with K and V
    if (lane == 0) {
      uint32_t un = 0, kn = 0, cn = 0;  // V and K loads issued
      while (true) {
        const int idx = claimed_one(cn);
        if (idx < 0) break;
        int b, h, kj, n0;  // h: the K/V head
        const int32_t* list0;
        const int n = unit_info(idx, b, h, kj, list0, n0);
        if (n == 0) continue;
        if (un > 0 && !wait(A_KEMPTY, (un - 1) & 1)) break;
        mbar_arrive_expect_tx(bar(A_KFULL), C::TILE);
#pragma unroll
        for (int s = 0; s < D / 64; ++s)
          tma_load_4d(sK + s * 16384, &tmK, bar(A_KFULL), s * 64, h, kj * kTile, b);
        if (un > 0 && !wait(A_VEMPTY, (un - 1) & 1)) {
          ++kn;
          break;
        }
        ++un;
        ++kn;
        mbar_arrive_expect_tx(bar(A_VFULL), C::TILE);
#pragma unroll
        for (int s = 0; s < D / 64; ++s)
          tma_load_4d(sV + s * 16384, &tmV, bar(A_VFULL), s * 64, h, kj * kTile, b);
      }
      // drain every issued copy before exit
      if (kn > 0) mbar_wait(bar(A_KFULL), (kn - 1) & 1, P.status, P.wait_ns);
      if (un > 0) mbar_wait(bar(A_VFULL), (un - 1) & 1, P.status, P.wait_ns);
    }
    __syncwarp();
  } else if (warp == Q_WARP) {
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
        if (use > 0 && !wait(A_UEMPTY0 + r, (use - 1) & 1)) break;
        int idx = atomicAdd(P.next_unit, 1);
        if (idx >= P.n_units) idx = -1;
        ring[r] = idx;
        mbar_arrive(bar(A_UFULL0 + r));
        if (idx < 0) break;
        int b, hk, kj, nj;
        const int32_t* list;
        unit_info(idx, b, hk, kj, list, nj);
        // the q-tile columns of the G query heads reading K/V head hk
        for (int j = 0; j < P.G && ok; ++j) {
          const int h = hk * P.G + j;
          if (j > 0) {
            const int col = col_of(b, h, kj);
            list = P.list + static_cast<size_t>(col) * P.nQ;
            nj = P.list_count[col];
          }
          const size_t bh_row = (static_cast<size_t>(b) * P.H + h) * rows_pad;
          for (int t = 0; t < nj; ++t, ++it) {
            const int qi = list[t] >> 2;
            const int st = it & 1;
            const uint32_t use = it >> 1;
            if (use > 0 && !wait(A_QEMPTY0 + st, (use - 1) & 1)) { ok = false; break; }
            const uint32_t fb = bar(A_QFULL0 + st);
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
      }
      // drain every issued copy before exit
      for (uint32_t k = (it > 2u ? it - 2u : 0u); k < it; ++k)
        mbar_wait(bar(A_QFULL0 + (k & 1)), (k >> 1) & 1, P.status, P.wait_ns);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idSS = idesc_bf16(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t idKB = idesc_bf16(128, D, false, true);     // dV, dK (B MN-major)
      // operand descriptors of each buffer, computed once (each MMA adds a
      // constant offset); "k" = K-major view, "m" = MN-major view
      const uint32_t dKk = sdesc_lo(sK, 16);
      const uint32_t dVk = sdesc_lo(sV, 16);
      const uint32_t dSk = sdesc_lo(sDS, 16);
      const uint32_t dQk0 = sdesc_lo(sbase + C::OFF_Q, 16), dQm0 = sdesc_lo(sbase + C::OFF_Q, 16384);
      const uint32_t dOk0 = sdesc_lo(sbase + C::OFF_DO, 16), dOm0 = sdesc_lo(sbase + C::OFF_DO, 16384);
      // dK += dS^T(i) Q(i) of tile i (global count), once its dS^T is in
      // smem; then the tile's Q/dO stage is free
      auto issue_dk = [&](uint32_t i, bool first_of_unit) -> bool {
        if (!wait(A_DSREADY, i & 1)) return false;
        tc_fence_after();
        const uint32_t dQm = dQm0 + (i & 1) * (C::TILE >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tbase + C::T_DK, sdesc_at(dSk, aoff), sdesc_at(dQm, kk * 2048), idKB,
                 (!first_of_unit || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(A_QEMPTY0 + (i & 1)));
        return true;
      };
      uint32_t it = 0, un = 0, cn = 0;
      bool ok = true;
      while (ok) {
        const int idx = claimed_one(cn);
        if (idx < 0) break;
        int b, h, kj, n0;
        const int32_t* list0;
        const int n = unit_info(idx, b, h, kj, list0, n0);
        if (n == 0) continue;
        if (!wait(A_KFULL, un & 1)) break;
        for (int t = 0; t < n; ++t, ++it) {
          const int st = it & 1;
          const uint32_t stage = st * (C::TILE >> 4);
          const uint32_t dQk = dQk0 + stage;
          const uint32_t dOk = dOk0 + stage, dOm = dOm0 + stage;
          if (!wait(A_QFULL0 + st, (it >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(tbase + C::T_A, sdesc_at(dKk, koff), sdesc_at(dQk, koff), idSS,
                   kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(A_SFULL));
          if (t == n - 1) mma_commit(bar(A_KEMPTY));  // the unit's last reader of K
          // the previous tile's dK, deferred until S^T of this tile is queued
          if (t > 0 && !issue_dk(it - 1, t == 1)) { ok = false; break; }
          if (t == 0 && !wait(A_VFULL, un & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(tbase + C::T_B, sdesc_at(dVk, koff), sdesc_at(dOk, koff), idSS,
                   kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(A_DPFULL));
          if (t == n - 1) mma_commit(bar(A_VEMPTY));  // the unit's last reader of V
          // dV += P^T dO once P^T is in TMEM (and the previous unit's dV/dK were read)
          if (!wait(A_PREADY, it & 1)) { ok = false; break; }
          if (t == 0 && un > 0 && !wait(A_ACCEMPTY, (un - 1) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // P^T of q columns 0..63 sits in TMEM columns [0,32), 64..127 in [64,96)
            const uint32_t acol = (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
            mma_ts(tbase + C::T_DV, tbase + C::T_A + acol, sdesc_at(dOm, kk * 2048), idKB,
                   (t > 0 || kk > 0) ? 1u : 0u);
          }
        }
        if (!ok) break;
        if (!issue_dk(it - 1, n == 1)) break;
        mma_commit(bar(A_ACCFULL));
        ++un;
      }
      mma_commit(bar(A_DRAIN));
      mbar_wait(bar(A_DRAIN), 0, P.status, P.wait_ns);
    }
    __syncwarp();
  }  // warp 11: spare warp of the producer warpgroup
  } else {
    // ------------------------------------------------------------ compute warps
    regs_increase<C::REGS_COMPUTE>();
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;  // TMEM lane: key row of S^T, dP^T, dK, dV
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int c0 = half * 64;           // this thread's 64 of the 128 q columns
    uint32_t it = 0, un = 0, cn = 0, ep = 0;  // ep: epilogues done
    bool pending = false;                      // the previous unit's dK, dV wait in TMEM
    int pb = 0, ph = 0, pkj = 0;               // the previous unit's batch, head, k-tile
    // ---- epilogue of the previous unit: dV and scale * dK, this thread's
    // half of the columns.  It runs after the next unit's first P^T, when
    // the previous unit's last dK has long completed: its TMEM read (which
    // lets the next dV start) then waits for nothing, and its stores overlap
    // the next unit's MMAs.
    auto epilogue = [&]() -> bool {
      const int b = pb, h = ph, kj = pkj;
      const int key = kj * kTile + r;
      if (!wait_all(A_ACCFULL, ep & 1)) return false;
      ++ep;
      tc_fence_after();
      uint32_t rv[D / 2], rk[D / 2];
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tmem_ld32(tbase + lane_off + C::T_DV + half * (D / 2) + c * 32, rv + 32 * c);
        tmem_ld32(tbase + lane_off + C::T_DK + half * (D / 2) + c * 32, rk + 32 * c);
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive_warp(bar(A_ACCEMPTY));
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
          __nv_bfloat16* base = m ? P.out0 : P.out1;
          const int64_t* st3 = m ? P.s0 : P.s1;
          if constexpr (WIDE) {
            // 32 bytes per lane: four lanes per row, eight rows per store
            const int jj = lane & 3;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rl = i * 8 + (lane >> 2);  // row within the warp's 32 keys
              const uint32_t c0 = static_cast<uint32_t>(2 * jj) ^ static_cast<uint32_t>(rl & 7);
              const uint32_t c1 = static_cast<uint32_t>(2 * jj + 1) ^ static_cast<uint32_t>(rl & 7);
              uint32_t w[8];
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                           : "r"(patch + rl * 128 + c0 * 16));
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                           : "r"(patch + rl * 128 + c1 * 16));
              const int kr = key0 + rl;
              if (kr < P.Skv)
                st_global_v8(base + b * st3[0] + static_cast<int64_t>(kr) * st3[1] + h * st3[2] +
                                 half * (D / 2) + jj * 16,
                             w);
            }
          } else {
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
          }
          __syncwarp();
        }
      } else if (key < P.Skv) {
        const float sc = P.scale;
        uint4* dv_dst = reinterpret_cast<uint4*>(P.out1 + b * P.s1[0] + static_cast<int64_t>(key) * P.s1[1] +
                                                 h * P.s1[2] + half * (D / 2));
        uint4* dk_dst = reinterpret_cast<uint4*>(P.out0 + b * P.s0[0] + static_cast<int64_t>(key) * P.s0[1] +
                                                 h * P.s0[2] + half * (D / 2));
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
      pending = false;
      return true;
    };
    bool ok = true;
    while (ok) {
      const int idx = claimed_all(cn);
      if (idx < 0) break;
      int b, hk, kj, nj;  // hk: the K/V head
      const int32_t* list;  // the walk's current query-head column, nj tiles
      const int n = unit_info(idx, b, hk, kj, list, nj);
      const int key = kj * kTile + r;
      __nv_bfloat16* dk_row = P.out0 + b * P.s0[0] + static_cast<int64_t>(key) * P.s0[1] +
                              hk * P.s0[2] + half * (D / 2);
      __nv_bfloat16* dv_row = P.out1 + b * P.s1[0] + static_cast<int64_t>(key) * P.s1[1] +
                              hk * P.s1[2] + half * (D / 2);
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
      // this thread's key column bounds (beyond Skv: hidden from every row),
      // read again when the walk moves to a query head with its own mask
      int lts = 0, lte = 0x7fffffff, uts = 0, ute = 0;
      auto load_bounds = [&](int h) {
        if (key < P.Skv) {
          const size_t at = static_cast<size_t>(b * P.Hm + (P.Hm == 1 ? 0 : h)) * P.Skv + key;
          lts = __ldg(P.bounds[0] + at);
          lte = __ldg(P.bounds[1] + at);
          uts = __ldg(P.bounds[2] + at);
          ute = __ldg(P.bounds[3] + at);
        }
      };
      load_bounds(hk * P.G);
      const bool key_ragged = (kj == P.nK - 1) && (P.Skv & (kTile - 1));
      // the walk over the group's query heads: head j's column, tile t of
      // the unit
      int t = 0;
      for (int j = 0; j < P.G && ok; ++j) {
        if (j > 0) {
          const int h = hk * P.G + j;
          const int col = col_of(b, h, kj);
          list = P.list + static_cast<size_t>(col) * P.nQ;
          nj = P.list_count[col];
          if (P.Hm > 1) load_bounds(h);
        }
        for (int i = 0; i < nj; ++i, ++t, ++it) {
          const int e = list[i];
          const int qi = e >> 2;
          const bool partial = ((e & 3) == CLS_PARTIAL) || key_ragged;
          const int st = it & 1;
          const float* lse_s = reinterpret_cast<const float*>(smem + C::OFF_LD + st * 1024) + c0;
          const float* del_s = lse_s + 128;
          // ---- P^T = exp2(S^T * scale*log2e - LSE*log2e), hidden entries 0
          if (!wait_all(A_SFULL, it & 1)) { ok = false; break; }
          // the LSE/D of this stage arrived with the Q/dO tiles
          if (!wait_all(A_QFULL0 + st, (it >> 1) & 1)) { ok = false; break; }
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
          if (!(P.withhold == 2 && it == 0)) mbar_arrive_warp(bar(A_PREADY));
          if (t == 0 && pending && !epilogue()) { ok = false; break; }
          // ---- dS^T = P^T o (dP^T - D), to smem as bf16 [key][q] (slab = half)
          if (!wait_all(A_DPFULL, it & 1)) { ok = false; break; }
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
          mbar_arrive_warp(bar(A_DSREADY));
        }
      }
      if (!ok) break;
      pending = true;
      pb = b;
      ph = hk;
      pkj = kj;
      ++un;
    }
    if (ok && pending) epilogue();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tbase, C::T_COLS);
  }
}

// ------------------------------------------------------------------ dQ kernel
template <int D>
struct DqCfg {
  static constexpr int TILE = 128 * D * 2;   // one 128-row bf16 tile
  static constexpr int KSTAGES = 3, VSTAGES = 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + TILE;
  static constexpr int OFF_K = OFF_DO + TILE;              // KSTAGES stages
  static constexpr int OFF_V = OFF_K + KSTAGES * TILE;     // VSTAGES stages
  static constexpr int OFF_MSK = OFF_V + VSTAGES * TILE;   // one partial tile's 128 rows x 16 bytes
  static constexpr int OFF_RING = OFF_MSK + kMaskBytes;
  static constexpr int OFF_BAR = OFF_RING + 16;
  static constexpr int NBAR = 34;
  static constexpr int SMEM_USED = OFF_BAR + NBAR * 8 + 16;
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  // TMEM: S of even / odd tiles (then dS as packed bf16 over it), dP, dQ
  static constexpr uint32_t T_S = 0, T_DP = 256, T_DQ = 384, T_COLS = 512;
  // warpgroups 0-1: compute (P, dS, the dQ epilogue); warpgroup 2: the
  // Q/dO/K/bits load warp, the MMA warp, the V load warp and one idle warp
  static constexpr int THREADS = 384;
  // register split (setmaxnreg): 2 x 128 x REGS_COMPUTE + 128 x REGS_PRODUCER
  // = 64512 = THREADS x 168 registers at launch
  static constexpr uint32_t REGS_COMPUTE = 216, REGS_PRODUCER = 72;
  static constexpr int MIN_LAUNCH_REGS =
      (2 * 128 * REGS_COMPUTE + 128 * REGS_PRODUCER + THREADS - 1) / THREADS;
};

enum { Q_QFULL = 0, Q_QEMPTY, Q_OFULL, Q_OEMPTY, Q_READY0, Q_KEMPTY0 = Q_READY0 + 3,
       Q_VEMPTY0 = Q_KEMPTY0 + 3, Q_BFULL = Q_VEMPTY0 + 2, Q_BEMPTY, Q_SFULL0,
       Q_DPFULL = Q_SFULL0 + 2, Q_DPFREE, Q_DSREADY0, Q_DQFULL = Q_DSREADY0 + 2, Q_DQEMPTY, Q_DRAIN_A,
       Q_DRAIN_B, Q_UFULL0, Q_UEMPTY0 = Q_UFULL0 + 4 };
// every slot of the unit ring is read by the two MMA warps and the eight
// compute warps
constexpr int Q_READERS = 10;

// One unit = q-tile qi of one (batch, head), walking its row of non-empty
// k-tiles (g = the CTA's running tile count: TMEM S region g & 1, K stage
// g mod 3, V stage g & 1).  MMA issue order, per tile t of the unit:
//   S(t+1) = Q K^T -> S[(t+1) & 1]  [the region's previous dS was read by dQ(t-1)]
//   dP(t+1) = dO V^T -> DP          [the compute warps have loaded dP(t)]
//   dQ += dS(t) K(t)                 [dS(t) is in S[t & 1]]
// so dS(t) has the time of S(t+1) and dP(t+1) to be ready.
// Two threads issue the MMAs: A the S and dP products, B the dQ products.  A
// barrier check waits behind the MMAs its thread has issued, and leaves the
// tensor pipe idle until the thread issues again; with two issuers the
// other's queued MMAs cover it.  B checks DSREADY(t) per tile.  A checks
// READY(t) before S(t) (ring of three, by g mod 3): the K and V copies of the
// tile (one expect-tx arrival of the loader) and B's commit after dQ(t-2),
// the last reader of the S region S(t) overwrites; and DPFREE before dP(t):
// one arrival per compute warp once it has loaded dP(t-1) out of the single
// dP region.  S(t) thus never waits for the compute warps.  K(t) is read by
// S(t) and dQ(t), a period apart: the
// loader fills tile t+1's K stage once dQ(t-2) is done and its V stage once
// dP(t-1) is done.  The bits
// of a partial tile have their own one-tile buffer, filled after the compute
// warps have read the previous partial tile's bits.  dS readiness has one
// barrier per S region: dP(t+1) is issued before the wait for dS(t), and a
// region's barrier cannot run two phases ahead of that wait (dS(t+2) needs
// S(t+2), issued only after dQ(t)).
// WIDE: every dQ row starts on a 32-byte boundary (32-byte epilogue stores;
// a template parameter because a run-time choice between the two store forms
// made the rest of the kernel slower)
template <int D, bool WIDE>
__global__ void __launch_bounds__(DqCfg<D>::THREADS, 1)
    bwd_dq_kernel(const __grid_constant__ BwdParams P, const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmDO) {
  using C = DqCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(P.status, DEV_LAYOUT);
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint4* msk = reinterpret_cast<uint4*>(smem + C::OFF_MSK);  // [128 rows]
  volatile int* ring = reinterpret_cast<volatile int*>(smem + C::OFF_RING);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::NBAR * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8 + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int LD_WARP = 8, MMA_WARP = 9, DQ_WARP = 10;

  if (tid == 0) {
    // Q is read by the unit's S products only, dO by its dP products: each is
    // free for the next unit as soon as its last reader is done
    mbar_init(bar(Q_QFULL), 1);
    mbar_init(bar(Q_QEMPTY), 1);
    mbar_init(bar(Q_OFULL), 1);
    mbar_init(bar(Q_OEMPTY), 1);
    for (int s = 0; s < C::KSTAGES; ++s) {
      // the loader's expect-tx and the dQ issuer's commit
      mbar_init(bar(Q_READY0 + s), 2);
      mbar_init(bar(Q_KEMPTY0 + s), 1);
    }
    for (int s = 0; s < C::VSTAGES; ++s) mbar_init(bar(Q_VEMPTY0 + s), 1);
    mbar_init(bar(Q_BFULL), 1);
    mbar_init(bar(Q_BEMPTY), 8);  // one arrival per compute warp
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(Q_SFULL0 + s), 1);
      mbar_init(bar(Q_DSREADY0 + s), 8);
    }
    mbar_init(bar(Q_DPFULL), 1);
    mbar_init(bar(Q_DPFREE), 8);  // one arrival per compute warp
    mbar_init(bar(Q_DQFULL), 1);
    mbar_init(bar(Q_DQEMPTY), 8);
    mbar_init(bar(Q_DRAIN_A), 1);
    mbar_init(bar(Q_DRAIN_B), 1);
    for (int r = 0; r < UNIT_RING; ++r) {
      mbar_init(bar(Q_UFULL0 + r), 1);
      mbar_init(bar(Q_UEMPTY0 + r), Q_READERS);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), C::T_COLS);
    tmem_relinquish();
  }
  if (warp == LD_WARP && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmDO);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const int rows_pad = P.nQ * kTile;
  const bool ragged = (P.Skv & (kTile - 1)) != 0;

  auto wait = [&](int b, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (!mbar_wait(bar(b), parity, P.status, P.wait_ns)) {
      *abort_flag = 1;
      return false;
    }
    return true;
  };
  auto wait_all = [&](int b, uint32_t parity) -> bool {
    const bool ok = wait(b, parity);
    return __all_sync(0xffffffffu, ok);
  };
  // unit u = (b*H + h)*nQ + qi -> its row of k-tiles
  auto unit_info = [&](int idx, int& b, int& h, int& qi, int& row, const int32_t*& list) {
    const int u = P.order[idx];
    const int bh = u / P.nQ;
    qi = u - bh * P.nQ;
    b = bh / P.H;
    h = bh - b * P.H;
    row = (b * P.Hm + (P.Hm == 1 ? 0 : h)) * P.nQ + qi;
    list = P.list + static_cast<size_t>(row) * P.nK;
    return P.list_count[row];
  };
  auto claimed_one = [&](uint32_t& n) -> int {
    int idx = -1;
    const int r = n % UNIT_RING;
    if (wait(Q_UFULL0 + r, (n / UNIT_RING) & 1)) {
      idx = ring[r];
      mbar_arrive(bar(Q_UEMPTY0 + r));
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
  // a tile is handled element by element when it is partial, or the ragged
  // last k-tile
  auto is_partial = [&](int ent) {
    return (ent & 3) == CLS_PARTIAL || (ragged && (ent >> 2) == P.nK - 1);
  };

  if (warp >= LD_WARP) {
  regs_decrease<C::REGS_PRODUCER>();
  if (warp == LD_WARP) {
    // ------------------------------------------------------------ Q / dO / K / bits loads
    // Bits of a partial tile without a precomputed mask, built from the
    // bounds: lane l holds columns l, l+32, l+64, l+96, so ballot x over the
    // lanes is word x of a row; lane (r mod 32) keeps row r's words.
    auto build_bits = [&](int bm, int kj, int qt, uint4* rows) {
      const size_t base = static_cast<size_t>(bm) * P.Skv;
      int4 v[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int j = kj * kTile + lane + 32 * x;
        if (j < P.Skv) {
          v[x].x = __ldg(P.bounds[0] + base + j);
          v[x].y = __ldg(P.bounds[1] + base + j);
          v[x].z = __ldg(P.bounds[2] + base + j);
          v[x].w = __ldg(P.bounds[3] + base + j);
        } else {
          v[x] = make_int4(0, 0x7fffffff, 0, 0);  // beyond the keys: hidden from every row
        }
      }
      for (int g = 0; g < 4; ++g) {
        uint4 mine = make_uint4(0u, 0u, 0u, 0u);
        for (int rr = 0; rr < 32; ++rr) {
          const int qrow = qt * kTile + g * 32 + rr;
          uint32_t w[4];
#pragma unroll
          for (int x = 0; x < 4; ++x)
            w[x] = __ballot_sync(0xffffffffu, (v[x].x <= qrow && qrow < v[x].y) ||
                                                  (v[x].z <= qrow && qrow < v[x].w));
          if (lane == rr) mine = make_uint4(w[0], w[1], w[2], w[3]);
        }
        rows[g * 32 + lane] = mine;
      }
    };
    // a q-tile row with no visible tile: its dQ rows are zero
    auto finish_empty_row = [&](int b, int h, int qi) {
      constexpr int WPR = D / 8;  // 16-byte words per dQ row
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      const int row0 = qi * kTile;
      for (int i = lane; i < kTile * WPR; i += 32) {
        const int row = row0 + i / WPR;
        if (row < P.Sq)
          reinterpret_cast<uint4*>(P.out0 + b * P.s0[0] + static_cast<int64_t>(row) * P.s0[1] +
                                   h * P.s0[2])[i % WPR] = z;
      }
    };
    uint32_t g = 0, un = 0, cn = 0, pc = 0;  // tiles, units, ring slots, partial tiles
    uint32_t qn = 0, on = 0;                 // Q and dO loads issued (lane 0)
    bool ok = true;
    while (ok) {
      // claim the next unit with tiles and publish it to the other roles;
      // rows without tiles are finished here and never published
      const int r = cn % UNIT_RING;
      const uint32_t use = cn / UNIT_RING;
      ++cn;
      if (lane == 0 && use > 0 && !wait(Q_UEMPTY0 + r, (use - 1) & 1)) ok = false;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      int idx, b = 0, h = 0, qi = 0, row = 0, n = 0;
      const int32_t* list = nullptr;
      while (true) {
        idx = -1;
        if (lane == 0) {
          idx = atomicAdd(P.next_unit, 1);
          if (idx >= P.n_units) idx = -1;
        }
        idx = __shfl_sync(0xffffffffu, idx, 0);
        if (idx < 0) break;
        n = unit_info(idx, b, h, qi, row, list);
        if (n > 0) break;
        finish_empty_row(b, h, qi);
      }
      if (lane == 0) {
        ring[r] = idx;
        mbar_arrive(bar(Q_UFULL0 + r));
      }
      if (idx < 0) break;
      if (lane == 0) {
        if (un > 0 && !wait(Q_QEMPTY, (un - 1) & 1)) ok = false;
        if (ok) {
          mbar_arrive_expect_tx(bar(Q_QFULL), C::TILE);
#pragma unroll
          for (int x = 0; x < D / 64; ++x)
            tma_load_4d(sbase + C::OFF_Q + x * 16384, &tmQ, bar(Q_QFULL), x * 64, h, qi * kTile, b);
          ++qn;
        }
        if (ok && un > 0 && !wait(Q_OEMPTY, (un - 1) & 1)) ok = false;
        if (ok) {
          mbar_arrive_expect_tx(bar(Q_OFULL), C::TILE);
#pragma unroll
          for (int x = 0; x < D / 64; ++x)
            tma_load_4d(sbase + C::OFF_DO + x * 16384, &tmDO, bar(Q_OFULL), x * 64, h, qi * kTile,
                        b);
          ++on;
        }
      }
      ++un;
      // lane 0 alone may have cleared ok: make it the warp's, so that no
      // lane stays in the unit loop after the others have left it
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const int mb = P.row_mask[row];
      int mo = 0;  // partial tiles of the row so far
      for (int t = 0; t < n; ++t, ++g) {
        const int ent = list[t];
        const int kj = ent >> 2;
        const int ks = static_cast<int>(g % C::KSTAGES);
        const uint32_t uk = g / C::KSTAGES;
        const int vs = static_cast<int>(g & 1);
        if (lane == 0) {
          // K stage: dQ(g-3) done; V stage: dP(g-2) done (not implied by the
          // former when tile g-2 opens a unit: its dP is issued after the
          // previous unit's last dQ)
          if (uk > 0 && !wait(Q_KEMPTY0 + ks, (uk - 1) & 1)) ok = false;
          if (ok && g >= 2 && !wait(Q_VEMPTY0 + vs, ((g >> 1) - 1) & 1)) ok = false;
          if (ok) {
            const uint32_t rb = bar(Q_READY0 + ks);
            mbar_arrive_expect_tx(rb, 2 * C::TILE);
#pragma unroll
            for (int x = 0; x < D / 64; ++x) {
              tma_load_4d(sbase + C::OFF_K + ks * C::TILE + x * 16384, &tmK, rb, x * 64,
                          h / P.G, kj * kTile, b);
              tma_load_4d(sbase + C::OFF_V + vs * C::TILE + x * 16384, &tmV, rb, x * 64,
                          h / P.G, kj * kTile, b);
            }
          }
        }
        ok = __all_sync(0xffffffffu, ok);  // the warp's, as above
        if (!ok) break;
        if (is_partial(ent)) {
          // the bits buffer, once the compute warps have read the previous
          // partial tile's
          if (pc > 0 && !wait_all(Q_BEMPTY, (pc - 1) & 1)) { ok = false; break; }
          if (mb >= 0) {
            if (lane == 0) {
              mbar_arrive_expect_tx(bar(Q_BFULL), kMaskBytes);
              bulk_load(smem_u32(msk), P.masks + static_cast<size_t>(mb + mo) * kMaskBytes,
                        kMaskBytes, bar(Q_BFULL));
            }
          } else {
            build_bits(row / P.nQ, kj, qi, msk);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Q_BFULL));
          }
          ++mo;
          ++pc;
        }
      }
    }
    // drain: every issued copy has landed before the CTA may exit (a tile's
    // READY phase completes after its copies have)
    if (lane == 0) {
      const uint32_t back = g > static_cast<uint32_t>(C::KSTAGES) ? C::KSTAGES : g;
      for (uint32_t x = g - back; x < g; ++x)
        mbar_wait(bar(Q_READY0 + x % C::KSTAGES), (x / C::KSTAGES) & 1, P.status, P.wait_ns);
      if (pc > 0) mbar_wait(bar(Q_BFULL), (pc - 1) & 1, P.status, P.wait_ns);
      if (qn > 0) mbar_wait(bar(Q_QFULL), (qn - 1) & 1, P.status, P.wait_ns);
      if (on > 0) mbar_wait(bar(Q_OFULL), (on - 1) & 1, P.status, P.wait_ns);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer A: S, dP
    if (lane == 0) {
      constexpr uint32_t idSS = idesc_bf16(128, 128, false, false);  // S, dP
      const uint32_t dQ = sdesc_lo(sbase + C::OFF_Q, 16);
      const uint32_t dO = sdesc_lo(sbase + C::OFF_DO, 16);
      const uint32_t dK0 = sdesc_lo(sbase + C::OFF_K, 16);
      const uint32_t dV0 = sdesc_lo(sbase + C::OFF_V, 16);
      auto issue_s = [&](uint32_t gt, bool last) -> bool {
        const uint32_t ks = gt % C::KSTAGES;
        if (!wait(Q_READY0 + ks, (gt / C::KSTAGES) & 1)) return false;
        tc_fence_after();
        const uint32_t dK = dK0 + ks * (C::TILE >> 4);
        const int x = gt & 1;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tbase + C::T_S + 128 * x, sdesc_at(dQ, koff), sdesc_at(dK, koff), idSS,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(Q_SFULL0 + x));
        if (last) mma_commit(bar(Q_QEMPTY));  // the unit's last reader of Q
        return true;
      };
      auto issue_dp = [&](uint32_t gt, bool last) -> bool {
        const int st = gt & 1;
        // the compute warps have loaded dP(gt - 1) out of the region
        if (gt > 0 && !wait(Q_DPFREE, (gt - 1) & 1)) return false;
        tc_fence_after();
        const uint32_t dV = dV0 + st * (C::TILE >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tbase + C::T_DP, sdesc_at(dO, koff), sdesc_at(dV, koff), idSS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(Q_DPFULL));
        mma_commit(bar(Q_VEMPTY0 + st));  // V(gt) is read by this dP only
        if (last) mma_commit(bar(Q_OEMPTY));  // the unit's last reader of dO
        return true;
      };
      uint32_t g = 0, un = 0, cn = 0;
      bool ok = true;
      while (ok) {
        const int idx = claimed_one(cn);
        if (idx < 0) break;
        int b, h, qi, row;
        const int32_t* list;
        const int n = unit_info(idx, b, h, qi, row, list);
        if (!wait(Q_QFULL, un & 1) || !issue_s(g, n == 1)) break;
        if (!wait(Q_OFULL, un & 1) || !issue_dp(g, n == 1)) break;
        for (int t = 1; t < n; ++t) {
          if (!issue_s(g + t, t + 1 == n) || !issue_dp(g + t, t + 1 == n)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        g += n;
        ++un;
      }
      mma_commit(bar(Q_DRAIN_A));
      mbar_wait(bar(Q_DRAIN_A), 0, P.status, P.wait_ns);
    }
    __syncwarp();
  } else if (warp == DQ_WARP) {
    // ------------------------------------------------------------ MMA issuer B: dQ
    if (lane == 0) {
      constexpr uint32_t idDQ = idesc_bf16(128, D, false, true);  // dQ (B = K MN-major)
      const uint32_t dKm0 = sdesc_lo(sbase + C::OFF_K, 128 * 128);
      // S(0) and S(1) overwrite no dS
      mbar_arrive(bar(Q_READY0));
      mbar_arrive(bar(Q_READY0 + 1));
      uint32_t g = 0, un = 0, cn = 0;
      bool ok = true;
      while (ok) {
        const int idx = claimed_one(cn);
        if (idx < 0) break;
        int b, h, qi, row;
        const int32_t* list;
        const int n = unit_info(idx, b, h, qi, row, list);
        for (int t = 0; t < n; ++t) {
          const uint32_t gt = g + t;
          if (!wait(Q_DSREADY0 + (gt & 1), (gt >> 1) & 1)) { ok = false; break; }
          // the previous unit's dQ has been read by the epilogue
          if (t == 0 && un > 0 && !wait(Q_DQEMPTY, (un - 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t ks = gt % C::KSTAGES;
          const uint32_t dKm = dKm0 + ks * (C::TILE >> 4);
          const uint32_t tS = tbase + C::T_S + 128 * (gt & 1);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // dS of keys 0..63 sits in TMEM columns [0,32), 64..127 in [64,96)
            const uint32_t acol = (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
            mma_ts(tbase + C::T_DQ, tS + acol, sdesc_at(dKm, kk * 2048), idDQ,
                   (t > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(Q_KEMPTY0 + ks));  // K(gt): read by S(gt) and this dQ
          // the S region of tile gt is free for S(gt + 2)
          mma_commit(bar(Q_READY0 + (gt + 2) % C::KSTAGES));
        }
        if (!ok) break;
        g += n;
        mma_commit(bar(Q_DQFULL));
        ++un;
      }
      mma_commit(bar(Q_DRAIN_B));
      mbar_wait(bar(Q_DRAIN_B), 0, P.status, P.wait_ns);
    }
    __syncwarp();
  }
  } else {
    // ------------------------------------------------------------ compute warps
    regs_increase<C::REGS_COMPUTE>();
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;  // TMEM lane: q row of S, dP, dQ
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int c0 = half * 64;           // this thread's 64 of the 128 key columns
    uint32_t g = 0, un = 0, cn = 0, ep = 0, pc = 0;  // ep: epilogues done, pc: partial tiles
    bool pending = false;                     // the previous unit's dQ waits in TMEM
    int pb = 0, ph = 0, prow = 0;             // its batch, head and this thread's q row
    // ---- epilogue of the previous unit: scale * dQ, this thread's half of
    // the columns.  It runs after the next unit's first P, when the previous
    // unit's last dQ has completed: its TMEM read then waits for nothing.
    auto epilogue = [&]() -> bool {
      if (!wait_all(Q_DQFULL, ep & 1)) return false;
      ++ep;
      tc_fence_after();
      uint32_t rq[D / 2];
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tmem_ld32(tbase + lane_off + C::T_DQ + half * (D / 2) + c * 32, rq + 32 * c);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive_warp(bar(Q_DQEMPTY));
      {
        // this thread's half row as NC 16-byte chunks, regrouped so that each
        // store instruction writes whole 16 * NC-byte runs of NC rows instead
        // of 16 bytes of 32 rows
        constexpr int NC = D / 16;
        uint32_t pk[4 * NC];
        const float sc = P.scale;
#pragma unroll
        for (int i = 0; i < 4 * NC; ++i)
          pk[i] = pack_bf16(__uint_as_float(rq[2 * i]) * sc, __uint_as_float(rq[2 * i + 1]) * sc);
        __nv_bfloat16* base = P.out0 + pb * P.s0[0] + ph * P.s0[2] + half * (D / 2);
        if constexpr (WIDE) {
          // 32-byte chunks where the layout allows: half the exchanges and
          // half the store instructions
          constexpr int N2 = NC / 2;
          transpose_chunks<N2, 8>(pk);
          const int row0 = prow - lane + (lane & ~(N2 - 1));  // q row of this lane group's first row
          base += (lane & (N2 - 1)) * 16;
#pragma unroll
          for (int i = 0; i < N2; ++i)
            if (row0 + i < P.Sq) st_global_v8(base + static_cast<int64_t>(row0 + i) * P.s0[1], pk + 8 * i);
        } else {
          transpose_chunks<NC>(pk);
          const int row0 = prow - lane + (lane & ~(NC - 1));  // q row of this lane group's first row
          base += (lane & (NC - 1)) * 8;
#pragma unroll
          for (int i = 0; i < NC; ++i)
            if (row0 + i < P.Sq)
              *reinterpret_cast<uint4*>(base + static_cast<int64_t>(row0 + i) * P.s0[1]) =
                  make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      pending = false;
      return true;
    };
    bool ok = true;
    while (ok) {
      const int idx = claimed_all(cn);
      if (idx < 0) break;
      int b, h, qi, row;
      const int32_t* list;
      const int n = unit_info(idx, b, h, qi, row, list);
      const int qrow = qi * kTile + r;
      const size_t bh_row = (static_cast<size_t>(b) * P.H + h) * rows_pad + qrow;
      const float lse2 = P.lse_log2[bh_row];  // -LSE*log2(e), -inf past Sq / no key
      const float drow = P.delta[bh_row];
      const uint64_t sc2 = splat2(P.scale_log2), l2 = splat2(lse2);
      for (int t = 0; t < n; ++t) {
        const uint32_t gt = g + t;
        const int ent = list[t];
        const bool partial = is_partial(ent);
        const int x = gt & 1;
        const uint32_t tS = tbase + lane_off + C::T_S + 128 * x;
        // ---- P = exp2(S * scale*log2e - LSE*log2e), hidden entries 0
        if (!wait_all(Q_SFULL0 + x, (gt >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        float p[64];
        {
          uint32_t raw[64];
          tmem_ld64(tS + c0, raw);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float a0, a1;
            fma2_bc(a0, a1, __uint_as_float(raw[2 * i]), __uint_as_float(raw[2 * i + 1]), sc2, l2);
            p[2 * i] = ex2(a0);
            p[2 * i + 1] = ex2(a1);
          }
        }
        if (partial) {
          // this row's 64 column bits of the tile (set = hidden)
          if (!wait_all(Q_BFULL, pc & 1)) { ok = false; break; }
          ++pc;
          const uint4 mw = msk[r];
          const uint32_t m0 = half ? mw.z : mw.x, m1 = half ? mw.w : mw.y;
          mbar_arrive_warp(bar(Q_BEMPTY));
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            p[c] = ((m0 >> c) & 1u) ? 0.f : p[c];
            p[c + 32] = ((m1 >> c) & 1u) ? 0.f : p[c + 32];
          }
        }
        if (t == 0 && pending && !epilogue()) { ok = false; break; }
        // ---- dS = P o (dP - D), packed bf16 over this thread's S columns
        if (!wait_all(Q_DPFULL, gt & 1)) { ok = false; break; }
        tc_fence_after();
        {
          uint32_t raw[64];
          tmem_ld64(tbase + lane_off + C::T_DP + c0, raw);
          tmem_wait_ld();
          // dP is in registers: the next dP may overwrite the region
          tc_fence_before();
          mbar_arrive_warp(bar(Q_DPFREE));
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            float s0, s1;
            mulsub2(s0, s1, p[2 * c], p[2 * c + 1], __uint_as_float(raw[2 * c]),
                    __uint_as_float(raw[2 * c + 1]), drow, drow);
            pk[c] = pack_bf16(s0, s1);
          }
          // keys c0 .. c0+63 packed two per column into the first half of
          // the columns this thread read, [c0, c0 + 32): the other half of
          // the warps may still be reading S from theirs
          tmem_st32(tS + c0, pk);
          tmem_wait_st();
        }
        tc_fence_before();
        // (a test of the wait limit withholds the first dS-ready arrival: the
        // dQ MMA thread then gives up on it and the launch unwinds with
        // DEV_TIMEOUT)
        if (!(P.withhold == 3 && gt == 0)) mbar_arrive_warp(bar(Q_DSREADY0 + x));
      }
      if (!ok) break;
      g += n;
      pending = true;
      pb = b;
      ph = h;
      prow = qrow;
      ++un;
    }
    if (ok && pending) epilogue();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tbase, C::T_COLS);
  }
}

template <typename Kern>
static fm_status prepare(Kern kern, int smem, int min_regs) {
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return FM_ERR_CUDA;
  // the setmaxnreg split must fit in the registers the block launches with
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return FM_ERR_CUDA;
  if (fa.numRegs < min_regs) return FM_ERR_UNSUPPORTED;
  return FM_OK;
}

template <int D>
static fm_status launch_bwd_d(const Plan& p, const fm_desc& desc, const TensorArgs& t, char* ws,
                              cudaStream_t s) {
  const int rows_pad = p.nQ * kTile;
  float* delta = reinterpret_cast<float*>(ws + p.L.delta);
  float* lse2 = reinterpret_cast<float*>(ws + p.L.lse_log2);
  {
    // four warps per block, one warp per 4 rows (rows_pad is a multiple of 128)
    const long long rows = static_cast<long long>(p.B) * p.H * rows_pad;
    const long long blocks = (rows / 4 + 3) / 4;
    prof_begin(K_BWD_PRE, s);
    bwd_pre_kernel<D><<<static_cast<unsigned>(blocks), 128, 0, s>>>(
        static_cast<const __nv_bfloat16*>(t.o), static_cast<const __nv_bfloat16*>(t.dout),
        desc.o_stride[0], desc.o_stride[1], desc.o_stride[2], t.lse_in, p.B, p.H, p.Sq, rows_pad,
        delta, lse2);
    prof_end(K_BWD_PRE, s);
    if (cudaGetLastError() != cudaSuccess) return FM_ERR_CUDA;
  }
  CUtensorMap tq, tk, tv, tdo;
  if (!make_tmap_bshd(&tq, t.q, p.B, p.Sq, p.H, D, desc.q_stride, 128) ||
      !make_tmap_bshd(&tk, t.k, p.B, p.Skv, p.Hkv, D, desc.k_stride, 128) ||
      !make_tmap_bshd(&tv, t.v, p.B, p.Skv, p.Hkv, D, desc.v_stride, 128) ||
      !make_tmap_bshd(&tdo, t.dout, p.B, p.Sq, p.H, D, desc.o_stride, 128))
    return FM_ERR_CUDA;
  const TestHooks th = test_hooks();
  BwdParams P{};
  P.B = p.B; P.H = p.H; P.Hm = p.Hm; P.Sq = p.Sq; P.Skv = p.Skv; P.nQ = p.nQ; P.nK = p.nK;
  P.Hkv = p.Hkv; P.G = p.G;
  P.scale = t.scale;
  P.scale_log2 = t.scale * 1.4426950408889634f;
  for (int i = 0; i < 4; ++i) P.bounds[i] = t.bounds[i];
  P.delta = delta;
  P.lse_log2 = lse2;
  P.status = reinterpret_cast<int*>(ws + p.L.status);
  P.wait_ns = th.wait_ns;
  fm_status st;
  {
    // dK, dV over k-tile columns
    BwdParams A = P;
    A.n_units = p.B * p.Hkv * p.nK;
    A.list_count = reinterpret_cast<const int32_t*>(ws + p.L.col_count);
    A.list = reinterpret_cast<const int32_t*>(ws + p.L.col_list);
    A.order = reinterpret_cast<const int32_t*>(ws + p.L.bwd_order);
    A.next_unit = reinterpret_cast<int*>(ws + p.L.status) + 1;
    A.out0 = static_cast<__nv_bfloat16*>(t.dk);
    A.out1 = static_cast<__nv_bfloat16*>(t.dv);
    for (int i = 0; i < 3; ++i) {
      A.s0[i] = desc.k_stride[i];
      A.s1[i] = desc.v_stride[i];
    }
    A.withhold = th.withhold;
    using C = KvCfg<D>;
    auto kern = rows_32b_aligned(t.dk, desc.k_stride) && rows_32b_aligned(t.dv, desc.v_stride)
                    ? bwd_kv_kernel<D, true>
                    : bwd_kv_kernel<D, false>;
    if ((st = prepare(kern, C::SMEM, C::MIN_LAUNCH_REGS)) != FM_OK) return st;
    const int grid = A.n_units < num_sms() ? A.n_units : num_sms();
    prof_begin(K_BWD, s);
    kern<<<grid, C::THREADS, C::SMEM, s>>>(A, tq, tk, tv, tdo);
    prof_end(K_BWD, s);
    if (cudaGetLastError() != cudaSuccess) return FM_ERR_CUDA;
  }
  {
    // dQ over q-tile rows
    BwdParams Q = P;
    Q.n_units = p.B * p.H * p.nQ;
    Q.list_count = reinterpret_cast<const int32_t*>(ws + p.L.row_count);
    Q.list = reinterpret_cast<const int32_t*>(ws + p.L.row_list);
    Q.order = reinterpret_cast<const int32_t*>(ws + p.L.row_order);
    Q.next_unit = reinterpret_cast<int*>(ws + p.L.status) + 4;
    Q.row_mask = reinterpret_cast<const int32_t*>(ws + p.L.row_mask);
    Q.masks = reinterpret_cast<const uint8_t*>(ws + p.L.masks);
    Q.out0 = static_cast<__nv_bfloat16*>(t.dq);
    for (int i = 0; i < 3; ++i) Q.s0[i] = desc.q_stride[i];
    Q.withhold = th.withhold;
    using C = DqCfg<D>;
    auto kern = rows_32b_aligned(t.dq, desc.q_stride) ? bwd_dq_kernel<D, true> : bwd_dq_kernel<D, false>;
    if ((st = prepare(kern, C::SMEM, C::MIN_LAUNCH_REGS)) != FM_OK) return st;
    const int grid = Q.n_units < num_sms() ? Q.n_units : num_sms();
    prof_begin(K_BWD_DQ, s);
    kern<<<grid, C::THREADS, C::SMEM, s>>>(Q, tq, tk, tv, tdo);
    prof_end(K_BWD_DQ, s);
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
