// Forward pass of masked attention on sm_103a.
//
// Exact attention with a streaming (rescaled) softmax over the k-tiles of
// each 128-row q-tile, in the spirit of the FlashAttention-2 page
// («Блочная обработка сохраняет общую нормализацию»: running max and sum,
// partial outputs rescaled, normalisation over the whole row), and the
// empty/full/partial tile classes of the column-wise mask (FlashMask-3 page,
// introduction): empty tiles never reach this kernel, full tiles skip the
// mask arithmetic, partial tiles test every (row, column).
//
// Work unit: one (batch, head, q-tile), 128 query rows.  A persistent grid of
// one CTA per SM walks the longest-first unit list.  Six warps per CTA:
//   warps 0-3  softmax: thread r owns query row r = TMEM lane r.  Reads S from
//              TMEM, masks partial tiles, keeps the running max m and sum l
//              (base-2 exponent domain), writes P (bf16) to TMEM, rescales O
//              in TMEM when the max moves, and writes O / LSE at the end;
//   warp 4     loads Q, K, V tiles with TMA into 128B-swizzled smem and, for
//              partial tiles, the 128 columns' bounds into smem;
//   warp 5     one thread issues tcgen05 MMAs: S = Q K^T (both K-major, smem),
//              O += P V (P from TMEM, V MN-major from smem).
// TMEM (512 columns): S double buffer [0,128) [128,256), O [256,256+D),
// P [384,448) as packed bf16 pairs.
#include <cuda_bf16.h>

#include "fm_internal.h"
#include "fm_ptx.cuh"
#include "fm_tmap.h"

namespace fm {

template <int D>
struct FwdCfg {
  static constexpr int SLABS = D / 64;
  static constexpr int TILE = 128 * D * 2;  // bytes of one 128-row tile
  static constexpr int OFF_Q = 0;                       // 2 slots
  static constexpr int OFF_K = OFF_Q + 2 * TILE;        // 2 stages
  static constexpr int OFF_V = OFF_K + 2 * TILE;        // 2 stages
  static constexpr int OFF_BND = OFF_V + 2 * TILE;      // 2 stages x 128 x int4
  static constexpr int OFF_BAR = OFF_BND + 2 * 128 * 16;
  static constexpr int NBAR = 24;
  static constexpr int SMEM_USED = OFF_BAR + NBAR * 8 + 16;
  // at least 120 KB so that one CTA (which takes all 512 TMEM columns) is
  // resident per SM
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  // TMEM: S of slot s at [128 s, 128 s + 128) (P packed into its first 64
  // columns), O of slot s at [256 + 128 s, 256 + 128 s + D)
  static constexpr uint32_t T_COLS = 512;
  // warpgroups 0 and 1: softmax of slot 0 / slot 1; warpgroup 2: the Q/K/
  // bounds load warp, the MMA warp, the V load warp and one idle warp
  static constexpr int THREADS = 384;
  // register split (setmaxnreg): 2 x 128 x REGS_SOFTMAX + 128 x REGS_PRODUCER
  // = 62464 <= THREADS x (compiled registers); the launch checks that the
  // kernel was compiled with at least MIN_LAUNCH_REGS registers per thread
  static constexpr uint32_t REGS_SOFTMAX = 216, REGS_PRODUCER = 56;
  static constexpr int MIN_LAUNCH_REGS =
      (2 * 128 * REGS_SOFTMAX + 128 * REGS_PRODUCER + THREADS - 1) / THREADS;
};

// barrier slots; "s" = q-tile slot (0/1), "st" = K/V stage (0/1)
enum {
  B_QFULL0 = 0, B_QEMPTY0 = 2, B_SFULL0 = 4, B_PFULL0 = 6, B_PVDONE0 = 8, B_OEMPTY0 = 10,
  B_KFULL0 = 12, B_KEMPTY0 = 14, B_VFULL0 = 16, B_VEMPTY0 = 18, B_BEMPTY0 = 20, B_DRAIN = 22
};

struct FwdParams {
  int B, H, Hm, Sq, Skv, nQ, nK, n_units;
  float scale_log2;  // scale * log2(e)
  const int32_t* bounds[4];
  const int32_t* row_count;
  const int32_t* row_list;
  const int32_t* order;
  const int32_t* row_mask;  // first visibility-mask slot of a row's partial tiles, -1: none
  const uint8_t* masks;     // 2 KB per slot: 128 rows x 128 column bits, set = hidden
  __nv_bfloat16* o;
  int64_t o_stride[3];
  float* lse;
  int* status;
};

__device__ __forceinline__ bool tile_partial(int e, int kj, int nK, int Skv) {
  return ((e & 3) == CLS_PARTIAL) || (kj == nK - 1 && (Skv & (kTile - 1)) != 0);
}

// The CTA's units are idx = blockIdx.x + k * gridDim.x, k = 0, 1, 2, ...;
// slot s takes the units with k % 2 == s.  A cursor walks one slot's
// non-empty tiles; the merge interleaves the two slots' tiles (alternating
// while both have tiles left).  The TMA warp, the MMA warp and both softmax
// warpgroups run identical merges, so they agree on which K/V stage and
// which barrier phase every tile uses.
struct Cursor {
  int k, t, n, row;
};
struct UnitInfo {
  int b, h, qi, row, n;
};

__device__ __forceinline__ UnitInfo unit_of(const FwdParams& P, int idx) {
  UnitInfo u;
  const int id = P.order[idx];
  const int bh = id / P.nQ;
  u.qi = id - bh * P.nQ;
  u.b = bh / P.H;
  u.h = bh - u.b * P.H;
  u.row = (u.b * P.Hm + (P.Hm == 1 ? 0 : u.h)) * P.nQ + u.qi;
  u.n = P.row_count[u.row];
  return u;
}

__device__ __forceinline__ void cursor_next_unit(const FwdParams& P, Cursor& c) {
  while (true) {
    c.k += 2;
    const int idx = blockIdx.x + c.k * gridDim.x;
    if (idx >= P.n_units) {
      c.n = -1;
      return;
    }
    const UnitInfo u = unit_of(P, idx);
    if (u.n > 0) {
      c.n = u.n;
      c.row = u.row;
      c.t = 0;
      return;
    }
  }
}

struct Merge {
  Cursor c0, c1;  // two scalars, not an array: no dynamically indexed local memory
  int turn;
  __device__ __forceinline__ void init(const FwdParams& P) {
    c0.k = -2;
    c0.t = 0;
    cursor_next_unit(P, c0);
    c1.k = -1;
    c1.t = 0;
    cursor_next_unit(P, c1);
    turn = 0;
  }
  __device__ __forceinline__ int peek() const {
    const bool a = c0.n > 0, b = c1.n > 0;
    return (a && b) ? turn : (a ? 0 : (b ? 1 : -1));
  }
  // Take the next merged tile: its slot, unit index k, tile t and whether it
  // is the first / last tile of its unit.
  __device__ __forceinline__ int next(const FwdParams& P, int& k, int& t, int& row, bool& first,
                                      bool& last) {
    const int s = peek();
    if (s < 0) return -1;
    if (c0.n > 0 && c1.n > 0) turn ^= 1;
    Cursor x = s ? c1 : c0;
    k = x.k;
    t = x.t;
    row = x.row;
    first = x.t == 0;
    last = x.t == x.n - 1;
    if (++x.t >= x.n) cursor_next_unit(P, x);
    if (s) c1 = x; else c0 = x;
    return s;
  }
};

// Two-entry per-slot state kept in registers (selected, never indexed).
template <typename T>
struct Pair {
  T v0, v1;
  __device__ __forceinline__ T get(int s) const { return s ? v1 : v0; }
  __device__ __forceinline__ void set(int s, T v) {
    if (s) v1 = v; else v0 = v;
  }
};

template <int D>
__global__ void __launch_bounds__(FwdCfg<D>::THREADS, 1)
    fwd_kernel(const __grid_constant__ FwdParams P, const __grid_constant__ CUtensorMap tmQ,
               const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // swizzled tiles need a 1024-aligned base
    if (threadIdx.x == 0) atomicOr(P.status, DEV_LAYOUT);
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  int4* bnd = reinterpret_cast<int4*>(smem + C::OFF_BND);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::NBAR * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8 + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int TMA_WARP = 8, MMA_WARP = 9, V_WARP = 10;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_QFULL0 + s), 1);
      mbar_init(bar(B_QEMPTY0 + s), 1);
      mbar_init(bar(B_SFULL0 + s), 1);
      mbar_init(bar(B_PFULL0 + s), 128);
      mbar_init(bar(B_PVDONE0 + s), 1);
      mbar_init(bar(B_OEMPTY0 + s), 128);
      mbar_init(bar(B_KFULL0 + s), 1);
      mbar_init(bar(B_KEMPTY0 + s), 1);
      mbar_init(bar(B_VFULL0 + s), 1);
      mbar_init(bar(B_VEMPTY0 + s), 1);
      mbar_init(bar(B_BEMPTY0 + s), 128);
    }
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), C::T_COLS);
    tmem_relinquish();
  }
  if (warp == TMA_WARP && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
  }
  if (warp == V_WARP && lane == 0) tma_prefetch_desc(&tmV);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  auto wait = [&](int b, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (!mbar_wait(bar(b), parity, P.status)) {
      *abort_flag = 1;
      return false;
    }
    return true;
  };
  // for warps whose 32 lanes all take part: every lane gets the same answer,
  // so warp-collective instructions after it never run diverged
  auto wait_all = [&](int b, uint32_t parity) -> bool {
    const bool ok = wait(b, parity);
    return __all_sync(0xffffffffu, ok);
  };

  if (warp >= 8) {
  // producer warpgroup: small register budget (each role branch below runs
  // after the budget change, so the compiler allocates it within the budget)
  regs_decrease<C::REGS_PRODUCER>();
  if (warp == TMA_WARP) {
    // ------------------------------------------------------------ TMA producer
    Merge mg;
    mg.init(P);
    uint32_t i = 0;
    Pair<uint32_t> qn{0, 0};
    Pair<int> mbase{-1, -1}, mord{0, 0};  // per slot: the unit's first mask slot, partials so far
    while (true) {
      int k, t, row;
      bool first, last;
      const int s = mg.next(P, k, t, row, first, last);
      if (s < 0) break;
      const UnitInfo u = unit_of(P, blockIdx.x + k * gridDim.x);
      if (first && lane == 0) {
        bool ok = qn.get(s) == 0 || wait(B_QEMPTY0 + s, (qn.get(s) - 1) & 1);
        if (ok) {
          mbar_arrive_expect_tx(bar(B_QFULL0 + s), C::TILE);
#pragma unroll
          for (int x = 0; x < C::SLABS; ++x)
            tma_load_4d(sbase + C::OFF_Q + s * C::TILE + x * 16384, &tmQ, bar(B_QFULL0 + s),
                        x * 64, u.h, u.qi * kTile, u.b);
        }
      }
      if (first) {
        qn.set(s, qn.get(s) + 1);
        mbase.set(s, P.row_mask[u.row]);
        mord.set(s, 0);
      }
      const int e = P.row_list[static_cast<size_t>(row) * P.nK + t];
      const int kj = e >> 2;
      const int st = i & 1;
      const uint32_t use = i >> 1;
      if (use > 0 && !wait_all(B_KEMPTY0 + st, (use - 1) & 1)) break;
      if (use > 0 && !wait_all(B_BEMPTY0 + st, (use - 1) & 1)) break;
      const bool partial = tile_partial(e, kj, P.nK, P.Skv);
      int mslot = -1;  // precomputed bit mask of this tile, if any
      if (partial && mbase.get(s) >= 0) {
        mslot = mbase.get(s) + mord.get(s);
        mord.set(s, mord.get(s) + 1);
      }
      if (partial && mslot < 0) {
        // no precomputed mask for this tile: build its bits here from the
        // bounds. Lane l holds columns l, l+32, l+64, l+96, so ballot x over
        // the lanes is word x of a row; lane (r mod 32) keeps row r's words.
        const size_t base = static_cast<size_t>(u.b * P.Hm + (P.Hm == 1 ? 0 : u.h)) * P.Skv;
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
        uint4* rows = reinterpret_cast<uint4*>(bnd + st * 128);
        for (int g = 0; g < 4; ++g) {
          uint4 mine = make_uint4(0u, 0u, 0u, 0u);
          for (int rr = 0; rr < 32; ++rr) {
            const int qrow = u.qi * kTile + g * 32 + rr;
            uint32_t w[4];
#pragma unroll
            for (int x = 0; x < 4; ++x)
              w[x] = __ballot_sync(0xffffffffu, (v[x].x <= qrow && qrow < v[x].y) ||
                                                    (v[x].z <= qrow && qrow < v[x].w));
            if (lane == rr) mine = make_uint4(w[0], w[1], w[2], w[3]);
          }
          rows[g * 32 + lane] = mine;
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(B_KFULL0 + st), C::TILE + (mslot >= 0 ? kMaskBytes : 0));
        if (mslot >= 0)
          bulk_load(smem_u32(bnd + st * 128), P.masks + static_cast<size_t>(mslot) * kMaskBytes,
                    kMaskBytes, bar(B_KFULL0 + st));
#pragma unroll
        for (int x = 0; x < C::SLABS; ++x)
          tma_load_4d(sbase + C::OFF_K + st * C::TILE + x * 16384, &tmK, bar(B_KFULL0 + st),
                      x * 64, u.h, kj * kTile, u.b);
      }
      ++i;
    }
    // drain: every issued copy has landed before the CTA may exit
    if (lane == 0) {
      for (uint32_t x = (i > 2u ? i - 2u : 0u); x < i; ++x)
        mbar_wait(bar(B_KFULL0 + (x & 1)), (x >> 1) & 1, P.status);
      if (qn.v0 > 0) mbar_wait(bar(B_QFULL0), (qn.v0 - 1) & 1, P.status);
      if (qn.v1 > 0) mbar_wait(bar(B_QFULL0 + 1), (qn.v1 - 1) & 1, P.status);
    }
    __syncwarp();
  } else if (warp == V_WARP) {
    // ------------------------------------------------------------ V producer
    // its own warp, so a V stage that is still in use never holds up K loads
    if (lane == 0) {
      Merge mg;
      mg.init(P);
      uint32_t i = 0;
      while (true) {
        int k, t, row;
        bool first, last;
        if (mg.next(P, k, t, row, first, last) < 0) break;
        const UnitInfo u = unit_of(P, blockIdx.x + k * gridDim.x);
        const int kj = P.row_list[static_cast<size_t>(row) * P.nK + t] >> 2;
        const int st = i & 1;
        const uint32_t use = i >> 1;
        if (use > 0 && !wait(B_VEMPTY0 + st, (use - 1) & 1)) break;
        mbar_arrive_expect_tx(bar(B_VFULL0 + st), C::TILE);
#pragma unroll
        for (int x = 0; x < C::SLABS; ++x)
          tma_load_4d(sbase + C::OFF_V + st * C::TILE + x * 16384, &tmV, bar(B_VFULL0 + st),
                      x * 64, u.h, kj * kTile, u.b);
        ++i;
      }
      for (uint32_t x = (i > 2u ? i - 2u : 0u); x < i; ++x)
        mbar_wait(bar(B_VFULL0 + (x & 1)), (x >> 1) & 1, P.status);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idPV = idesc_bf16(128, D, false, true);
      Merge mg;
      mg.init(P);
      uint32_t i = 0;
      Pair<uint32_t> js{0, 0}, jp{0, 0}, qn{0, 0}, un{0, 0}, pend_i{0, 0};
      Pair<bool> pend{false, false}, pend_first{false, false};
      bool ok = true;
      // S of slot s for the next merged tile(s) of that slot; returns false on abort
      auto issue_s_phase = [&](int want) -> bool {
        while (true) {
          const int s = mg.peek();
          if (s < 0 || pend.get(s) || (want >= 0 && s != want)) return true;
          int k, t, row;
          bool first, last;
          mg.next(P, k, t, row, first, last);
          if (first) {
            if (!wait(B_QFULL0 + s, qn.get(s) & 1)) return false;
            qn.set(s, qn.get(s) + 1);
          }
          // S of this slot overwrites P of its previous tile; MMAs issued by this
          // thread run in issue order, so the PV that reads P is done with it first
          const int st = i & 1;
          if (!wait(B_KFULL0 + st, (i >> 1) & 1)) return false;
          tc_fence_after();
          const uint32_t sQ = sbase + C::OFF_Q + s * C::TILE;
          const uint32_t sK = sbase + C::OFF_K + st * C::TILE;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(tbase + 128 * s, sdesc_sw128(sQ + koff, 16, 1024),
                   sdesc_sw128(sK + koff, 16, 1024), idS, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(B_SFULL0 + s));
          mma_commit(bar(B_KEMPTY0 + st));
          if (last) mma_commit(bar(B_QEMPTY0 + s));
          js.set(s, js.get(s) + 1);
          pend.set(s, true);
          pend_first.set(s, first);
          pend_i.set(s, i);
          ++i;
        }
      };
      auto issue_pv = [&](int s) -> bool {
        if (!wait(B_PFULL0 + s, jp.get(s) & 1)) return false;
        const bool first = pend_first.get(s);
        if (first) {
          // O of this slot is overwritten: its previous epilogue must be done
          if (un.get(s) > 0 && !wait(B_OEMPTY0 + s, (un.get(s) - 1) & 1)) return false;
          un.set(s, un.get(s) + 1);
        }
        const int st = pend_i.get(s) & 1;
        if (!wait(B_VFULL0 + st, (pend_i.get(s) >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t sV = sbase + C::OFF_V + st * C::TILE;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tbase + 256 + 128 * s, tbase + 128 * s + kk * 8,
                 sdesc_sw128(sV + kk * 2048, 128 * 128, 1024), idPV, (!first || kk > 0) ? 1u : 0u);
        mma_commit(bar(B_PVDONE0 + s));
        mma_commit(bar(B_VEMPTY0 + st));
        jp.set(s, jp.get(s) + 1);
        pend.set(s, false);
        return true;
      };
      // prologue: the first S of each slot (merged order)
      ok = issue_s_phase(-1);
      // ping-pong: PV of slot 0 then its next S, PV of slot 1 then its next S,
      // so one slot's softmax overlaps the other slot's MMAs
      while (ok && (pend.v0 || pend.v1)) {
#pragma unroll
        for (int s = 0; s < 2; ++s)
          if (ok && pend.get(s) && !issue_pv(s)) ok = false;
        if (ok && !issue_s_phase(-1)) ok = false;
      }
      mma_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, P.status);
    }
    __syncwarp();
  }  // warp 11: spare warp of the producer warpgroup, nothing to do
  } else {
    // ------------------------------------------------------------ softmax
    regs_increase<C::REGS_SOFTMAX>();
    const int slot = warp >> 2;              // warpgroup = slot
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;       // query row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tbase + lane_off + 128 * slot;
    const uint32_t tO = tbase + lane_off + 256 + 128 * slot;
    Merge mg;
    mg.init(P);
    uint32_t i = 0, j = 0;  // merged tile index, this slot's tile index
    bool ok = true;
    for (int k = slot; ok; k += 2) {
      const int idx = blockIdx.x + k * gridDim.x;
      if (idx >= P.n_units) break;
      const UnitInfo u = unit_of(P, idx);
      const int qrow = u.qi * kTile + r;
      __nv_bfloat16* orow = P.o + u.b * P.o_stride[0] + static_cast<int64_t>(qrow) * P.o_stride[1] +
                            u.h * P.o_stride[2];
      float* lse_out = P.lse + (static_cast<size_t>(u.b) * P.H + u.h) * P.Sq + qrow;
      if (u.n == 0) {
        if (qrow < P.Sq) {
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
          *lse_out = -INFINITY;
        }
        continue;
      }
      float m_used = -INFINITY, l = 0.f;  // running max (base-2 exponent domain) and sum
      for (int t = 0; t < u.n; ++t, ++j) {
        // the merged index of this tile: walk the merge past the other slot's tiles
        int mk, mt, mrow;
        bool mf, ml;
        int ms;
        while ((ms = mg.next(P, mk, mt, mrow, mf, ml)) != slot && ms >= 0) ++i;
        const uint32_t mi = i++;
        const int e = P.row_list[static_cast<size_t>(u.row) * P.nK + t];
        const int kj = e >> 2;
        const int st = mi & 1;
        if (!wait_all(B_SFULL0 + slot, j & 1)) { ok = false; break; }
        tc_fence_after();
        // the whole S row in one round trip: TMEM load latency (~670 cycles)
        // does not depend on the width, so issue both halves, wait once
        const bool partial = tile_partial(e, kj, P.nK, P.Skv);
        float sv[128];
        {
          uint32_t* raw = reinterpret_cast<uint32_t*>(sv);
#pragma unroll
          for (int x = 0; x < 4; ++x) tmem_ld32(tS + 32 * x, raw + 32 * x);
          if (partial && !wait_all(B_KFULL0 + st, (mi >> 1) & 1)) { ok = false; break; }
          tmem_wait_ld();
        }
        if (partial) {
          // this row's 128 column bits (set = hidden), one 16-byte load
          const uint4 mw = reinterpret_cast<const uint4*>(bnd + st * 128)[r];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            sv[c] = ((mw.x >> c) & 1u) ? -INFINITY : sv[c];
            sv[c + 32] = ((mw.y >> c) & 1u) ? -INFINITY : sv[c + 32];
            sv[c + 64] = ((mw.z >> c) & 1u) ? -INFINITY : sv[c + 64];
            sv[c + 96] = ((mw.w >> c) & 1u) ? -INFINITY : sv[c + 96];
          }
        }
        mbar_arrive(bar(B_BEMPTY0 + st));  // done with this stage's mask bits
        float mx8[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) mx8[x] = sv[x];
#pragma unroll
        for (int c = 8; c < 128; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], sv[c]);
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const float m_tile = mx * P.scale_log2;
        // lazy rescale: move the reference max only when it grows by more than
        // 8 (factor 256); below that the unnormalised p stay within bf16/fp32
        // range and the result is unchanged
        const bool grow = m_tile > m_used + 8.f;
        const float m_new = grow ? m_tile : m_used;
        const float alpha = grow ? ex2(m_used - m_new) : 1.f;  // m_used = -inf gives 0
        l *= alpha;
        m_used = m_new;
        const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
        // p = exp2(s * scale*log2e - m) from the registers, packed to bf16 into
        // the first 64 columns of S (the row was read whole above)
        float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const float p0 = ex2(fmaf(sv[c4 * 32 + 2 * x], P.scale_log2, -m_ref));
            const float p1 = ex2(fmaf(sv[c4 * 32 + 2 * x + 1], P.scale_log2, -m_ref));
            sum4[x & 3] += p0 + p1;
            pk[x] = pack_bf16(p0, p1);
          }
          tmem_st16(tS + c4 * 16, pk);
        }
        const float sum = (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
        // rescale O by alpha (after P: the S registers are free by now).  O
        // holds the PVs of the earlier tiles, all complete since S of this tile
        // completed after them
        if (t > 0 && __any_sync(0xffffffffu, grow)) {
          uint32_t raw[D];
#pragma unroll
          for (int x = 0; x < D / 32; ++x) tmem_ld32(tO + 32 * x, raw + 32 * x);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < D; ++x) raw[x] = __float_as_uint(__uint_as_float(raw[x]) * alpha);
#pragma unroll
          for (int x = 0; x < D / 32; ++x) tmem_st32(tO + 32 * x, raw + 32 * x);
        }
        l += sum;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(B_PFULL0 + slot));
      }
      if (!ok) break;
      // epilogue: O / l and LSE, after this unit's last PV.  O is read from
      // TMEM first and released, so the slot's next unit may overwrite it
      if (!wait_all(B_PVDONE0 + slot, (j - 1) & 1)) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint32_t ro[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tO + c * 32, ro + 32 * c);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(B_OEMPTY0 + slot));
      if (qrow < P.Sq) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int x = 0; x < D / 8; ++x)
          dst[x] = make_uint4(pack_bf16(__uint_as_float(ro[8 * x + 0]) * inv, __uint_as_float(ro[8 * x + 1]) * inv),
                              pack_bf16(__uint_as_float(ro[8 * x + 2]) * inv, __uint_as_float(ro[8 * x + 3]) * inv),
                              pack_bf16(__uint_as_float(ro[8 * x + 4]) * inv, __uint_as_float(ro[8 * x + 5]) * inv),
                              pack_bf16(__uint_as_float(ro[8 * x + 6]) * inv, __uint_as_float(ro[8 * x + 7]) * inv));
        const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
        *lse_out = l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994530942f : -INFINITY;
      }
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
static fm_status launch_fwd_d(const Plan& p, const fm_desc& desc, const TensorArgs& t, char* ws,
                              cudaStream_t s) {
  using C = FwdCfg<D>;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_bshd(&tq, t.q, p.B, p.Sq, p.H, D, desc.q_stride, 128) ||
      !make_tmap_bshd(&tk, t.k, p.B, p.Skv, p.H, D, desc.k_stride, 128) ||
      !make_tmap_bshd(&tv, t.v, p.B, p.Skv, p.H, D, desc.v_stride, 128))
    return FM_ERR_CUDA;
  FwdParams P{};
  P.B = p.B; P.H = p.H; P.Hm = p.Hm; P.Sq = p.Sq; P.Skv = p.Skv; P.nQ = p.nQ; P.nK = p.nK;
  P.n_units = p.B * p.H * p.nQ;
  P.scale_log2 = t.scale * 1.4426950408889634f;
  for (int i = 0; i < 4; ++i) P.bounds[i] = t.bounds[i];
  P.row_count = reinterpret_cast<const int32_t*>(ws + p.L.row_count);
  P.row_list = reinterpret_cast<const int32_t*>(ws + p.L.row_list);
  P.order = reinterpret_cast<const int32_t*>(ws + p.L.fwd_order);
  P.row_mask = reinterpret_cast<const int32_t*>(ws + p.L.row_mask);
  P.masks = reinterpret_cast<const uint8_t*>(ws + p.L.masks);
  P.o = static_cast<__nv_bfloat16*>(t.o_out);
  for (int i = 0; i < 3; ++i) P.o_stride[i] = desc.o_stride[i];
  P.lse = t.lse_out;
  P.status = reinterpret_cast<int*>(ws + p.L.status);
  auto kern = fwd_kernel<D>;
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
  prof_begin(K_FWD, s);
  kern<<<grid, C::THREADS, C::SMEM, s>>>(P, tq, tk, tv);
  prof_end(K_FWD, s);
  return cudaGetLastError() == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}

fm_status launch_fwd(const Plan& p, const fm_desc& desc, const TensorArgs& t, char* ws,
                     cudaStream_t s) {
  if (p.d == 64) return launch_fwd_d<64>(p, desc, t, ws, s);
  if (p.d == 128) return launch_fwd_d<128>(p, desc, t, ws, s);
  return FM_ERR_UNSUPPORTED;
}

}  // namespace fm
