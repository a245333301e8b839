// Forward pass of masked attention on sm_103a.
//
// Exact attention with a streaming (rescaled) softmax over the k-tiles of
// each 128-row q-tile, in the spirit of the FlashAttention-2 page
// («Блочная обработка сохраняет общую нормализацию»: running max and sum,
// partial outputs rescaled, normalisation over the whole row), and the
// empty/full/partial tile classes of the column-wise mask (FlashMask-3 page,
// introduction): empty tiles never reach this kernel, full tiles skip the
// mask arithmetic, partial tiles apply a 128 x 128 visibility bit mask.
//
// Work unit: one (batch, head) and two adjacent q-tiles 2p, 2p+1 (slots a
// and b, 256 query rows) that walk the union of their non-empty k-tiles, so
// each K/V tile is loaded once for both; the FlashAttention-2 page («Три
// способа повысить загрузку GPU», third point) gives each group of warps its
// own queries and shares K and V.  A persistent grid of one CTA per SM walks
// the longest-first unit list.  Twelve warps per CTA:
//   warps 0-3 / 4-7   softmax of slot a / b: thread r owns query row r =
//              TMEM lane r.  Reads S from TMEM, masks partial tiles, keeps
//              the running max m and sum l (base-2 exponent domain), writes
//              P (bf16) over S in TMEM, rescales O in TMEM when the max moves
//              by more than 2^8, and writes O / LSE at the end of the unit;
//   warp 8     loads Q (per slot), K and the partial tiles' bit masks; passes
//              each entry's classes and unit boundaries to the MMA warps;
//   warps 9/11 one thread each issues the tcgen05 MMAs of slot a / b:
//              S = Q K^T (both K-major, smem), O += P V (P from TMEM, V
//              MN-major from smem), per entry e PV(e) then S(e+1), so one
//              slot's softmax runs while the other slot's MMAs do;
//   warp 10    loads V.
// TMEM (512 columns): S/P of slot s at [128 s, 128 s + 128), O of slot s at
// [256 + 128 s, 256 + 128 s + D).
//
// FP8 variant (F8 = true, d = 128): Q and K are e4m3 codes with one scale per
// 128-row tile, V is e4m3 transposed per head ([d][key], a K-major operand)
// with one scale per 128-key tile and the head's largest tile scale.  Both
// products are kind::f8f6f4 MMAs (32 elements of k per MMA): S on K-major
// shared-memory operands, P V with P from tensor memory.  The softmax
// multiplies each S tile by scale * sq * sk, keeps its reference exponent
// integral (so rescales are exact powers of two), folds the V tile's scale
// ratio sv / sv_head into P, rounds P to e4m3 over the first 32 columns of
// the slot's S region (four values per column), and the epilogue multiplies
// O by sv_head / l.
#include <cuda_bf16.h>

#include "fm_internal.h"
#include "fm_ptx.cuh"
#include "fm_tmap.h"

namespace fm {

template <int D, bool F8 = false>
struct FwdCfg {
  static constexpr int ESIZE = F8 ? 1 : 2;          // bytes per element of Q, K, V
  static constexpr int SLABS = D * ESIZE / 128;     // 128-byte swizzle slabs per row
  static constexpr int SLAB_ELEMS = 128 / ESIZE;    // elements per slab row
  static constexpr int KSTEPS = D * ESIZE / 32;     // MMA steps of 32 bytes along d
  static constexpr int TILE = 128 * D * ESIZE;      // bytes of one 128-row tile
  static constexpr int OFF_Q = 0;                              // slots a, b
  static constexpr int OFF_K = OFF_Q + 2 * TILE;               // 2 stages
  static constexpr int OFF_V = OFF_K + 2 * TILE;               // 2 stages
  static constexpr int OFF_MSK = OFF_V + 2 * TILE;             // [stage][slot] bit masks
  static constexpr int OFF_DESC = OFF_MSK + 4 * kMaskBytes;    // [stage] entry word
  static constexpr int OFF_RING = OFF_DESC + 16;               // [UNIT_RING] claimed units
  static constexpr int OFF_BAR = OFF_RING + 16;
  static constexpr int NBAR = 32;
  static constexpr int SMEM_USED = OFF_BAR + NBAR * 8 + 16;
  // at least 120 KB so that one CTA (which takes all 512 TMEM columns) is
  // resident per SM
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  static constexpr uint32_t T_COLS = 512;
  // warpgroups 0 and 1: softmax of slot a / b; warpgroup 2: the Q/K/mask
  // load warp, the V load warp and the two MMA warps
  static constexpr int THREADS = 384;
  // register split (setmaxnreg): 2 x 128 x REGS_SOFTMAX + 128 x REGS_PRODUCER
  // = 64512 = THREADS x 168 (the compiled registers); the launch checks that
  // the kernel was compiled with at least MIN_LAUNCH_REGS registers per
  // thread.  With 56 for the producer warpgroup its roles spilled, and the
  // MMA threads' spills sat between their MMA groups.
  static constexpr uint32_t REGS_SOFTMAX = 216, REGS_PRODUCER = 72;
  static constexpr int MIN_LAUNCH_REGS =
      (2 * 128 * REGS_SOFTMAX + 128 * REGS_PRODUCER + THREADS - 1) / THREADS;
};

// barrier slots; "s" = q-tile slot (0 = a, 1 = b), "st" = K/V stage (0/1)
enum {
  B_QFULL0 = 0, B_QEMPTY0 = 2, B_SFULL0 = 4, B_PFULL0 = 6, B_PVDONE0 = 8, B_OEMPTY0 = 10,
  B_KFULL0 = 12, B_VFULL0 = 16, B_KVEMPTY0 = 18, B_MEMPTY0 = 20, B_DRAIN = 22,
  B_UFULL0 = 23, B_UEMPTY0 = 27
};
// Units are claimed at run time (one atomic counter per launch, in the
// workspace) by the K/mask load warp when it is ready to load the next one,
// and handed to the other roles that walk units through a ring of
// UNIT_RING slots; U_READERS warps read every slot: the V load warp and the
// eight softmax warps.  Only units with at least one tile go through the
// ring.  Claiming just in time keeps the units in flight on all CTAs close
// together in the head-major order (K/V stay in L2).
constexpr int UNIT_RING = 4, U_READERS = 9;

// entry word the load warp hands to the MMA warps: the pair-list classes in
// bits 0-3 (class_b bits 0-1, class_a bits 2-3), then whether this entry is
// the first / last non-empty tile of slot a (bits 4, 5) and of slot b (6, 7)
// within its unit
constexpr uint32_t E_A = 12u, E_B = 3u, E_FIRST_A = 16u, E_LAST_A = 32u, E_FIRST_B = 64u,
                   E_LAST_B = 128u;
// the word of the entry after the CTA's last one: no tiles, end of the stream
constexpr uint32_t E_END = 256u;

struct FwdParams {
  int B, H, Hm, Sq, Skv, nQ, nK, nP, n_units;
  int G;             // query heads per K/V head: head h reads K/V head h / G
  float scale_log2;  // scale * log2(e)
  const int32_t* bounds[4];
  const int4* pair_info;    // per pair row: entries, tiles of 2p, tiles of 2p+1, sum
  const int32_t* pair_list;
  const int32_t* order;
  int* next_unit;           // claim counter (zero at launch)
  const int32_t* row_mask;  // first visibility-mask slot of a q-tile row's partial tiles, -1: none
  const uint8_t* masks;     // 2 KB per slot: 128 rows x 128 column bits, set = hidden
  __nv_bfloat16* o;
  int64_t o_stride[3];
  float* lse;
  int* status;
  uint64_t wait_ns;  // limit of every mbarrier wait
  int withhold;      // test hook: 1 = slot a's softmax withholds its first P-ready arrival
  // FP8 variant: per-tile scales [B][H][nQ] (Q), [B][Hkv][nK] (K, V), and
  // the per-head V scale [B][Hkv]
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  const float* v_head_scale;
};

// Each CTA claims units idx = 0, 1, 2, ... of the longest-first order as it
// finishes earlier ones; every role walks the claimed units in claim order
// and their entries one by one, so all agree on the K/V stage (entry count
// mod 2) and the barrier phases.
struct PairUnit {
  int b, h, qa, prow, row_a, n, na, nb;
};

__device__ __forceinline__ PairUnit unit_of(const FwdParams& P, int idx) {
  PairUnit u;
  const int id = P.order[idx];
  const int bh = id / P.nP;
  const int p = id - bh * P.nP;
  u.b = bh / P.H;
  u.h = bh - u.b * P.H;
  const int bm = u.b * P.Hm + (P.Hm == 1 ? 0 : u.h);
  u.prow = bm * P.nP + p;
  u.row_a = bm * P.nQ + 2 * p;
  u.qa = 2 * p;
  const int4 inf = P.pair_info[u.prow];
  u.n = inf.x;
  u.na = inf.y;
  u.nb = inf.z;
  return u;
}

// Two-entry per-slot state kept in registers (selected, never indexed).
template <typename T>
struct Pair {
  T v0, v1;
  __device__ __forceinline__ T get(int s) const { return s ? v1 : v0; }
  __device__ __forceinline__ void set(int s, T v) {
    if (s) v1 = v; else v0 = v;
  }
};

// WIDE: every O row starts on a 32-byte boundary (32-byte epilogue stores)
template <int D, bool F8, bool WIDE>
__global__ void __launch_bounds__(FwdCfg<D, F8>::THREADS, 1)
    fwd_kernel(const __grid_constant__ FwdParams P, const __grid_constant__ CUtensorMap tmQ,
               const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using C = FwdCfg<D, F8>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // swizzled tiles need a 1024-aligned base
    if (threadIdx.x == 0) atomicOr(P.status, DEV_LAYOUT);
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint4* msk = reinterpret_cast<uint4*>(smem + C::OFF_MSK);  // [stage * 2 + slot][128 rows]
  volatile uint32_t* desc = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_DESC);
  volatile int* ring = reinterpret_cast<volatile int*>(smem + C::OFF_RING);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::NBAR * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8 + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int TMA_WARP = 8, MMA_WARP = 9, V_WARP = 10, MMA_WARP_B = 11;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_QFULL0 + s), 1);
      mbar_init(bar(B_QEMPTY0 + s), 1);
      mbar_init(bar(B_SFULL0 + s), 1);
      mbar_init(bar(B_PFULL0 + s), 4);  // one arrival per softmax warp of the slot
      mbar_init(bar(B_PVDONE0 + s), 1);
      mbar_init(bar(B_OEMPTY0 + s), 4);
      mbar_init(bar(B_KFULL0 + s), 1);
      mbar_init(bar(B_VFULL0 + s), 1);
      // stage s of K, V (and the bits) is free again once both MMA threads
      // are past its PV: one commit per MMA thread per entry
      mbar_init(bar(B_KVEMPTY0 + s), 2);
      // per stage: 4 arrivals for each slot, from its softmax warps when the
      // slot's tile there is partial (they read the bits), else from the load
      // warp on the slot's behalf
      mbar_init(bar(B_MEMPTY0 + s), 8);
    }
    mbar_init(bar(B_DRAIN), 2);
    for (int r = 0; r < UNIT_RING; ++r) {
      mbar_init(bar(B_UFULL0 + r), 1);
      mbar_init(bar(B_UEMPTY0 + r), U_READERS);
    }
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
    if (!mbar_wait(bar(b), parity, P.status, P.wait_ns)) {
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
  // the n-th claimed unit (-1: none left, or the launch was aborted); all 32
  // lanes call it, lane 0 reads the ring slot and releases it
  auto claimed = [&](uint32_t& n) -> int {
    int idx = -1;
    if (lane == 0) {
      const int r = n % UNIT_RING;
      if (wait(B_UFULL0 + r, (n / UNIT_RING) & 1)) {
        idx = ring[r];
        mbar_arrive(bar(B_UEMPTY0 + r));
      }
    }
    ++n;
    return __shfl_sync(0xffffffffu, idx, 0);
  };

  if (warp >= 8) {
  // producer warpgroup: small register budget (each role branch below runs
  // after the budget change, so the compiler allocates it within the budget)
  regs_decrease<C::REGS_PRODUCER>();
  if (warp == TMA_WARP) {
    // ------------------------------------------------------------ Q / K / mask loads
    // Bits of a partial tile without a precomputed mask, built from the
    // bounds: lane l holds columns l, l+32, l+64, l+96, so ballot x over the
    // lanes is word x of a row; lane (r mod 32) keeps row r's words.
    auto build_bits = [&](const PairUnit& u, int kj, int qt, uint4* rows) {
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
    // A pair with no visible tile at all (every row of both q-tiles hidden
    // from every key) is finished by this warp: zero O rows and -inf LSE.
    // Consecutive 16-byte words of a row go to consecutive lanes.
    auto finish_empty_pair = [&](const PairUnit& u) {
      constexpr int WPR = D / 8;  // 16-byte words per O row
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      for (int s = 0; s < 2 && u.qa + s < P.nQ; ++s) {
        const int row0 = (u.qa + s) * kTile;
        for (int i = lane; i < kTile * WPR; i += 32) {
          const int row = row0 + i / WPR;
          if (row < P.Sq)
            reinterpret_cast<uint4*>(P.o + u.b * P.o_stride[0] +
                                     static_cast<int64_t>(row) * P.o_stride[1] +
                                     u.h * P.o_stride[2])[i % WPR] = z;
        }
        for (int rr = lane; rr < kTile; rr += 32)
          if (row0 + rr < P.Sq)
            P.lse[(static_cast<size_t>(u.b) * P.H + u.h) * P.Sq + row0 + rr] = -INFINITY;
      }
    };
    uint32_t e = 0, un = 0;
    Pair<uint32_t> qn{0, 0};
    bool ok = true;
    while (ok) {
      // claim the next unit with tiles and publish it to the other roles.
      // Pairs without tiles are finished here and never published: the last
      // PV of a unit waits for the entry word after it, so the claim that
      // yields the next entry must not have to wait for a free ring slot,
      // and a run of published empty pairs could fill the ring before it.
      const int r = un % UNIT_RING;
      const uint32_t use = un / UNIT_RING;
      ++un;
      if (lane == 0 && use > 0 && !wait(B_UEMPTY0 + r, (use - 1) & 1)) ok = false;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      int idx;
      PairUnit u;
      while (true) {
        idx = -1;
        if (lane == 0) {
          idx = atomicAdd(P.next_unit, 1);
          if (idx >= P.n_units) idx = -1;
        }
        idx = __shfl_sync(0xffffffffu, idx, 0);
        if (idx < 0) break;
        u = unit_of(P, idx);
        if (u.n > 0) break;
        finish_empty_pair(u);
      }
      if (lane == 0) {
        ring[r] = idx;
        mbar_arrive(bar(B_UFULL0 + r));
      }
      if (idx < 0) break;
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        if ((s ? u.nb : u.na) == 0) continue;  // no tile of this slot: no Q
        if (lane == 0) {
          if (qn.get(s) > 0 && !wait(B_QEMPTY0 + s, (qn.get(s) - 1) & 1)) ok = false;
          if (ok) {
            mbar_arrive_expect_tx(bar(B_QFULL0 + s), C::TILE);
#pragma unroll
            for (int x = 0; x < C::SLABS; ++x)
              tma_load_4d(sbase + C::OFF_Q + s * C::TILE + x * 16384, &tmQ, bar(B_QFULL0 + s),
                          x * C::SLAB_ELEMS, u.h, (u.qa + s) * kTile, u.b);
          }
        }
        qn.set(s, qn.get(s) + 1);
      }
      // lane 0 alone may have cleared ok: make it the warp's (the end marker
      // below is written only if it is true, through warp-wide waits)
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const int mb0 = P.row_mask[u.row_a];
      const int mb1 = u.nb > 0 ? P.row_mask[u.row_a + 1] : -1;
      int mo0 = 0, mo1 = 0;      // partial tiles of each slot so far in this unit
      int seen0 = 0, seen1 = 0;  // non-empty tiles of each slot so far in this unit
      for (int t = 0; t < u.n; ++t, ++e) {
        const int ent = P.pair_list[static_cast<size_t>(u.prow) * P.nK + t];
        const int kj = ent >> 4, ca = (ent >> 2) & 3, cb = ent & 3;
        const int st = e & 1;
        const uint32_t use = e >> 1;
        if (use > 0 && !wait_all(B_KVEMPTY0 + st, (use - 1) & 1)) { ok = false; break; }
        if (use > 0 && !wait_all(B_MEMPTY0 + st, (use - 1) & 1)) { ok = false; break; }
        int ms0 = -1, ms1 = -1;  // precomputed mask slots (bulk-copied below)
        if (ca == CLS_PARTIAL) {
          if (mb0 >= 0) ms0 = mb0 + mo0;
          else build_bits(u, kj, u.qa, msk + (st * 2 + 0) * 128);
          ++mo0;
        }
        if (cb == CLS_PARTIAL) {
          if (mb1 >= 0) ms1 = mb1 + mo1;
          else build_bits(u, kj, u.qa + 1, msk + (st * 2 + 1) * 128);
          ++mo1;
        }
        uint32_t flags = static_cast<uint32_t>(ent & 15);
        if (ca != CLS_EMPTY) {
          flags |= (seen0 == 0 ? E_FIRST_A : 0u) | (seen0 == u.na - 1 ? E_LAST_A : 0u);
          ++seen0;
        }
        if (cb != CLS_EMPTY) {
          flags |= (seen1 == 0 ? E_FIRST_B : 0u) | (seen1 == u.nb - 1 ? E_LAST_B : 0u);
          ++seen1;
        }
        __syncwarp();
        if (lane == 0) {
          desc[st] = flags;
          const uint32_t bytes =
              C::TILE + (ms0 >= 0 ? kMaskBytes : 0u) + (ms1 >= 0 ? kMaskBytes : 0u);
          mbar_arrive_expect_tx(bar(B_KFULL0 + st), bytes);
          if (ms0 >= 0)
            bulk_load(smem_u32(msk + (st * 2 + 0) * 128),
                      P.masks + static_cast<size_t>(ms0) * kMaskBytes, kMaskBytes,
                      bar(B_KFULL0 + st));
          if (ms1 >= 0)
            bulk_load(smem_u32(msk + (st * 2 + 1) * 128),
                      P.masks + static_cast<size_t>(ms1) * kMaskBytes, kMaskBytes,
                      bar(B_KFULL0 + st));
#pragma unroll
          for (int x = 0; x < C::SLABS; ++x)
            tma_load_4d(sbase + C::OFF_K + st * C::TILE + x * 16384, &tmK, bar(B_KFULL0 + st),
                        x * C::SLAB_ELEMS, u.h / P.G, kj * kTile, u.b);
          // a slot whose tile here is not partial never reads this stage's bits
          if (ca != CLS_PARTIAL) mbar_arrive_count(bar(B_MEMPTY0 + st), 4);
          if (cb != CLS_PARTIAL) mbar_arrive_count(bar(B_MEMPTY0 + st), 4);
        }
      }
    }
    // drain: every issued copy has landed before the CTA may exit (before
    // the end marker below, which completes one more phase of a stage)
    if (lane == 0) {
      for (uint32_t x = (e > 2u ? e - 2u : 0u); x < e; ++x)
        mbar_wait(bar(B_KFULL0 + (x & 1)), (x >> 1) & 1, P.status, P.wait_ns);
      if (qn.v0 > 0) mbar_wait(bar(B_QFULL0), (qn.v0 - 1) & 1, P.status, P.wait_ns);
      if (qn.v1 > 0) mbar_wait(bar(B_QFULL0 + 1), (qn.v1 - 1) & 1, P.status, P.wait_ns);
    }
    // the end marker: one more entry word, no tiles, so the MMA warps stop.
    // Like any entry it waits until the entry two before has been read by
    // the MMAs and by the softmax threads that read its bits: those threads
    // wait on this stage's KFULL barrier, which must not run two phases
    // ahead of them.
    if (ok) {
      const int st = e & 1;
      const uint32_t use = e >> 1;
      if (use > 0) ok = wait_all(B_KVEMPTY0 + st, (use - 1) & 1);
      if (ok && use > 0) ok = wait_all(B_MEMPTY0 + st, (use - 1) & 1);
      if (ok && lane == 0) {
        desc[st] = E_END;
        mbar_arrive(bar(B_KFULL0 + st));
      }
    }
    __syncwarp();
  } else if (warp == V_WARP) {
    // ------------------------------------------------------------ V loads
    // its own warp, so a V stage that is still in use never holds up K loads
    uint32_t e = 0, un = 0;
    bool ok = true;
    while (ok) {
      const int idx = claimed(un);
      if (idx < 0) break;
      if (lane == 0) {
        const PairUnit u = unit_of(P, idx);
        for (int t = 0; t < u.n; ++t, ++e) {
          const int kj = P.pair_list[static_cast<size_t>(u.prow) * P.nK + t] >> 4;
          const int st = e & 1;
          const uint32_t use = e >> 1;
          if (use > 0 && !wait(B_KVEMPTY0 + st, (use - 1) & 1)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(B_VFULL0 + st), C::TILE);
          if constexpr (F8) {
            // V^T tile: 128 keys (contiguous) x d rows of the K/V head
            tma_load_4d(sbase + C::OFF_V + st * C::TILE, &tmV, bar(B_VFULL0 + st), kj * kTile,
                        0, u.h / P.G, u.b);
          } else {
#pragma unroll
            for (int x = 0; x < C::SLABS; ++x)
              tma_load_4d(sbase + C::OFF_V + st * C::TILE + x * 16384, &tmV, bar(B_VFULL0 + st),
                          x * 64, u.h / P.G, kj * kTile, u.b);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    // drain: every issued copy has landed before the CTA may exit
    if (lane == 0)
      for (uint32_t x = (e > 2u ? e - 2u : 0u); x < e; ++x)
        mbar_wait(bar(B_VFULL0 + (x & 1)), (x >> 1) & 1, P.status, P.wait_ns);
    __syncwarp();
  } else if (warp == MMA_WARP || warp == MMA_WARP_B) {
    // ------------------------------------------------------------ MMA issuers
    // One thread per slot (warp 9: slot a, warp 11: slot b).  The tensor
    // pipe accepts about one MMA ahead of the one it runs, so whatever the
    // issuing thread does between its MMA groups (barrier waits, the entry
    // word) leaves the pipe idle unless another thread issues meanwhile;
    // with one thread per slot, neither slot's waits hold up the other's
    // MMAs.  Both walk every entry: the K and V stages are released when
    // both have committed (their barriers count two arrivals).
    if (lane == 0) {
      const int s = warp == MMA_WARP ? 0 : 1;
      const uint32_t fA = s ? E_B : E_A, fFIRST = s ? E_FIRST_B : E_FIRST_A,
                     fLAST = s ? E_LAST_B : E_LAST_A;
      constexpr uint32_t idS = F8 ? idesc_e4m3(128, 128) : idesc_bf16(128, 128, false, false);
      constexpr uint32_t idPV = F8 ? idesc_e4m3(128, D) : idesc_bf16(128, D, false, true);
      const uint32_t sQ = sbase + C::OFF_Q + s * C::TILE;
      // operand descriptors of each buffer, computed once (each MMA adds a
      // constant offset): Q and K K-major, V MN-major
      const uint32_t dQ = sdesc_lo(sQ, 16);
      const uint32_t dK0 = sdesc_lo(sbase + C::OFF_K, 16);
      // V: MN-major [key][d] tiles, or (F8) K-major V^T [d][key] tiles
      const uint32_t dV0 = F8 ? sdesc_lo(sbase + C::OFF_V, 16) : sdesc_lo(sbase + C::OFF_V, 128 * 128);
      const uint32_t tS = tbase + 128 * s, tO = tbase + 256 + 128 * s;
      uint32_t qn = 0, np = 0, un = 0;
      // entry word of entry e, once its K tile (and bits) have landed
      auto entry = [&](uint32_t e, uint32_t& f) -> bool {
        if (!wait(B_KFULL0 + (e & 1), (e >> 1) & 1)) return false;
        f = desc[e & 1];
        return true;
      };
      // S of this slot for entry e.  It overwrites the slot's P of its
      // previous tile; MMAs issued by this thread run in issue order, so the
      // PV that reads that P (issued before) is done with it first.
      auto issue_s = [&](uint32_t e, uint32_t f) -> bool {
        if (f & fFIRST) {
          if (!wait(B_QFULL0 + s, qn & 1)) return false;
          ++qn;
        }
        tc_fence_after();
        const uint32_t dK = dK0 + (e & 1) * (C::TILE >> 4);
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
          const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
          if constexpr (F8) mma_ss_f8(tS, sdesc_at(dQ, koff), sdesc_at(dK, koff), idS, kk > 0 ? 1u : 0u);
          else mma_ss(tS, sdesc_at(dQ, koff), sdesc_at(dK, koff), idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(B_SFULL0 + s));
        if (f & fLAST) mma_commit(bar(B_QEMPTY0 + s));
        return true;
      };
      auto issue_pv = [&](uint32_t e, uint32_t f) -> bool {
        if (!wait(B_PFULL0 + s, np & 1)) return false;
        ++np;
        const bool first = (f & fFIRST) != 0;
        if (first) {
          // O of this slot is overwritten: its previous epilogue must be done
          if (un > 0 && !wait(B_OEMPTY0 + s, (un - 1) & 1)) return false;
          ++un;
        }
        const int st = e & 1;
        if (!wait(B_VFULL0 + st, (e >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t dV = dV0 + st * (C::TILE >> 4);
        if constexpr (F8) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // 128 keys, 32 per MMA (8 columns of P)
            mma_ts_f8(tO, tS + kk * 8, sdesc_at(dV, kk * 32), idPV, (!first || kk > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tO, tS + kk * 8, sdesc_at(dV, kk * 2048), idPV, (!first || kk > 0) ? 1u : 0u);
        }
        // the epilogue reads O after the unit's last PV only
        if (f & fLAST) mma_commit(bar(B_PVDONE0 + s));
        return true;
      };
      // entries arrive in order until the end marker; per entry: this
      // slot's PV of it, then its S of the next one
      uint32_t fc = 0;
      bool ok = entry(0, fc);
      if (ok && !(fc & E_END)) {
        if (fc & fA) ok = issue_s(0, fc);
        for (uint32_t j = 0; ok; ++j) {
          uint32_t fn = 0;
          // release V(j) only once it has landed, also when this slot does
          // not use it: then V(j) loaded means the release of V(j - 2) was
          // complete, so this thread's two arrivals never fill one phase of
          // the stage's barrier (the other thread may still be using V(j - 2))
          if (fc & fA) {
            if (!issue_pv(j, fc)) break;
          } else if (!wait(B_VFULL0 + (j & 1), (j >> 1) & 1)) {
            break;
          }
          mma_commit(bar(B_KVEMPTY0 + (j & 1)));
          if (!entry(j + 1, fn)) break;
          if (fn & E_END) break;
          if ((fn & fA) && !issue_s(j + 1, fn)) break;
          fc = fn;
        }
      }
      mma_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, P.status, P.wait_ns);
    }
    __syncwarp();
  }
  } else {
    // ------------------------------------------------------------ softmax
    regs_increase<C::REGS_SOFTMAX>();
    const int slot = warp >> 2;              // warpgroup = slot
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;       // query row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tbase + lane_off + 128 * slot;
    const uint32_t tO = tbase + lane_off + 256 + 128 * slot;
    uint32_t e = 0, j = 0, un = 0;  // entries walked, tiles of this slot done, units claimed
    uint32_t pd = 0;                // units of this slot with tiles (PV-done phases)
    bool ok = true;
    while (ok) {
      const int idx = claimed(un);
      if (idx < 0) break;
      const PairUnit u = unit_of(P, idx);
      const int qt = u.qa + slot;
      if (qt >= P.nQ) {  // odd nQ: the last pair has no second q-tile
        e += u.n;
        continue;
      }
      const int ns = slot ? u.nb : u.na;
      const int qrow = qt * kTile + r;
      __nv_bfloat16* orow = P.o + u.b * P.o_stride[0] + static_cast<int64_t>(qrow) * P.o_stride[1] +
                            u.h * P.o_stride[2];
      float* lse_out = P.lse + (static_cast<size_t>(u.b) * P.H + u.h) * P.Sq + qrow;
      if (ns == 0) {
        if (qrow < P.Sq) {
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
          *lse_out = -INFINITY;
        }
        e += u.n;
        continue;
      }
      float m_used = -INFINITY, l = 0.f;  // running max (base-2 exponent domain) and sum
      int done = 0;                       // tiles of this unit done
      // F8: this row's Q tile scale, the K/V head's scales
      const int hk = u.h / P.G;
      const float sq_row = F8 ? P.q_scale[(static_cast<size_t>(u.b) * P.H + u.h) * P.nQ + qt] : 1.f;
      const size_t kv_row = (static_cast<size_t>(u.b) * (P.H / P.G) + hk) * P.nK;
      const float sv_head = F8 ? P.v_head_scale[static_cast<size_t>(u.b) * (P.H / P.G) + hk] : 1.f;
      for (int t = 0; t < u.n; ++t, ++e) {
        const int ent = P.pair_list[static_cast<size_t>(u.prow) * P.nK + t];
        const int cls = slot ? (ent & 3) : ((ent >> 2) & 3);
        if (cls == CLS_EMPTY) continue;
        const int st = e & 1;
        const bool partial = cls == CLS_PARTIAL;
        if (!wait_all(B_SFULL0 + slot, j & 1)) { ok = false; break; }
        tc_fence_after();
        // the whole S row in one round trip: TMEM load latency does not
        // depend on the width, so issue all four quarters and wait once
        float sv[128];
        {
          uint32_t* raw = reinterpret_cast<uint32_t*>(sv);
#pragma unroll
          for (int x = 0; x < 4; ++x) tmem_ld32(tS + 32 * x, raw + 32 * x);
          if (partial && !wait_all(B_KFULL0 + st, (e >> 1) & 1)) {
            tmem_wait_ld();
            ok = false;
            break;
          }
          tmem_wait_ld();
        }
        if (partial) {
          // this row's 128 column bits (set = hidden), one 16-byte load
          const uint4 mw = msk[(st * 2 + slot) * 128 + r];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            sv[c] = ((mw.x >> c) & 1u) ? -INFINITY : sv[c];
            sv[c + 32] = ((mw.y >> c) & 1u) ? -INFINITY : sv[c + 32];
            sv[c + 64] = ((mw.z >> c) & 1u) ? -INFINITY : sv[c + 64];
            sv[c + 96] = ((mw.w >> c) & 1u) ? -INFINITY : sv[c + 96];
          }
          mbar_arrive_warp(bar(B_MEMPTY0 + st));  // done with this stage's bits
        }
        // row maximum: eight independent chains of three-input max
        float mx8[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) mx8[x] = fmax3(sv[x], sv[x + 8], sv[x + 16]);
#pragma unroll
        for (int c = 24; c < 120; c += 16)
#pragma unroll
          for (int x = 0; x < 8; ++x) mx8[x] = fmax3(mx8[x], sv[c + x], sv[c + 8 + x]);
#pragma unroll
        for (int x = 0; x < 8; ++x) mx8[x] = fmaxf(mx8[x], sv[120 + x]);
        const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                               fmaxf(mx8[6], mx8[7]));
        // S * scale * log2 e; F8: times the Q and K tile scales
        float ct = P.scale_log2, vr = 1.f;
        if constexpr (F8) {
          const int kj = ent >> 4;
          ct *= sq_row * P.k_scale[kv_row + kj];
          vr = P.v_scale[kv_row + kj] / sv_head;  // this V tile's scale ratio, <= 1
        }
        const float m_tile = mx * ct;
        // lazy rescale: move the reference max only when it grows by more than
        // 8 (factor 256); below that the unnormalised p stay within bf16/fp32
        // range and the result is unchanged
        const bool grow = m_tile > m_used + 8.f;
        // F8: an integral reference, so every rescale is a power of two and
        // P's e4m3 codes do not depend on when the reference moved
        const float m_new = grow ? (F8 ? ceilf(m_tile) : m_tile) : m_used;
        const float alpha = grow ? ex2(m_used - m_new) : 1.f;  // m_used = -inf gives 0
        l *= alpha;
        m_used = m_new;
        const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
        // p = exp2(s * scale*log2e - m) from the registers, packed to bf16 into
        // the first 64 columns of S (the row was read whole above)
        // two columns per packed FMA and per packed add
        const uint64_t sc2 = splat2(ct), nm2 = splat2(-m_ref);
        float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            float a0, a1;
            fma2_bc(a0, a1, sv[c4 * 32 + 2 * x], sv[c4 * 32 + 2 * x + 1], sc2, nm2);
            const float p0 = ex2(a0);
            const float p1 = ex2(a1);
            if (x & 1) add2_acc(sum4[2], sum4[3], p0, p1);
            else add2_acc(sum4[0], sum4[1], p0, p1);
            if constexpr (F8) {
              const uint32_t h = pack_e4m3x2(p0 * vr, p1 * vr);
              pk[x >> 1] = (x & 1) ? (pk[x >> 1] | (h << 16)) : h;
            } else {
              pk[x] = pack_bf16(p0, p1);
            }
          }
          if constexpr (F8) tmem_st8(tS + c4 * 8, pk);  // 32 keys, four per column
          else tmem_st16(tS + c4 * 16, pk);
        }
        const float sum = (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
        // rescale O by alpha (after P: the S registers are free by now).  O
        // holds the PVs of the earlier tiles, all complete since S of this tile
        // completed after them
        if (done > 0 && __any_sync(0xffffffffu, grow)) {
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
        // (a test of the wait limit withholds the first P-ready arrival of
        // slot a: the slot's MMA thread then gives up on it and the launch
        // unwinds with DEV_TIMEOUT)
        if (!(P.withhold == 1 && slot == 0 && j == 0)) mbar_arrive_warp(bar(B_PFULL0 + slot));
        ++j;
        ++done;
      }
      if (!ok) break;
      // epilogue: O / l and LSE, after this unit's last PV.  O is read from
      // TMEM first and released, so the slot's next unit may overwrite it
      if (!wait_all(B_PVDONE0 + slot, pd & 1)) break;
      ++pd;
      tc_fence_after();
      const float inv = l > 0.f ? sv_head / l : 0.f;
      uint32_t ro[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tO + c * 32, ro + 32 * c);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive_warp(bar(B_OEMPTY0 + slot));
      if (qrow < P.Sq) {
        // each lane writes its own row (32 rows per instruction): in 32-byte
        // pieces where the layout allows (WIDE), which halves the
        // instructions and the cache-line accesses of these uncoalesced
        // stores.  A template parameter, not a run-time branch: with both
        // forms in one kernel the rest of it was scheduled worse (6 % on
        // the full mask).
        if constexpr (WIDE) {
#pragma unroll
          for (int x = 0; x < D / 16; ++x) {
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              w[i] = pack_bf16(__uint_as_float(ro[16 * x + 2 * i]) * inv, __uint_as_float(ro[16 * x + 2 * i + 1]) * inv);
            st_global_v8(orow + 16 * x, w);
          }
        } else {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int x = 0; x < D / 8; ++x)
            dst[x] = make_uint4(pack_bf16(__uint_as_float(ro[8 * x + 0]) * inv, __uint_as_float(ro[8 * x + 1]) * inv),
                                pack_bf16(__uint_as_float(ro[8 * x + 2]) * inv, __uint_as_float(ro[8 * x + 3]) * inv),
                                pack_bf16(__uint_as_float(ro[8 * x + 4]) * inv, __uint_as_float(ro[8 * x + 5]) * inv),
                                pack_bf16(__uint_as_float(ro[8 * x + 6]) * inv, __uint_as_float(ro[8 * x + 7]) * inv));
        }
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

template <int D, bool F8>
static fm_status launch_fwd_d(const Plan& p, const fm_desc& desc, const TensorArgs& t, char* ws,
                              cudaStream_t s, const Fp8Args* f8 = nullptr) {
  using C = FwdCfg<D, F8>;
  CUtensorMap tq, tk, tv;
  if constexpr (F8) {
    if (!make_tmap_bshd8(&tq, f8->q8, p.B, p.Sq, p.H, D, 128) ||
        !make_tmap_bshd8(&tk, f8->k8, p.B, p.Skv, p.Hkv, D, 128) ||
        !make_tmap_vt8(&tv, f8->v8t, p.B, p.Hkv, D, p.nK * 128))
      return FM_ERR_CUDA;
  } else if (!make_tmap_bshd(&tq, t.q, p.B, p.Sq, p.H, D, desc.q_stride, 128) ||
             !make_tmap_bshd(&tk, t.k, p.B, p.Skv, p.Hkv, D, desc.k_stride, 128) ||
             !make_tmap_bshd(&tv, t.v, p.B, p.Skv, p.Hkv, D, desc.v_stride, 128)) {
    return FM_ERR_CUDA;
  }
  FwdParams P{};
  P.B = p.B; P.H = p.H; P.Hm = p.Hm; P.Sq = p.Sq; P.Skv = p.Skv; P.nQ = p.nQ; P.nK = p.nK;
  P.G = p.G;
  P.nP = p.nP;
  P.n_units = p.B * p.H * p.nP;
  P.scale_log2 = t.scale * 1.4426950408889634f;
  for (int i = 0; i < 4; ++i) P.bounds[i] = t.bounds[i];
  P.pair_info = reinterpret_cast<const int4*>(ws + p.L.pair_info);
  P.pair_list = reinterpret_cast<const int32_t*>(ws + p.L.pair_list);
  P.order = reinterpret_cast<const int32_t*>(ws + p.L.fwd_order);
  P.next_unit = reinterpret_cast<int*>(ws + p.L.status) + 1;
  P.row_mask = reinterpret_cast<const int32_t*>(ws + p.L.row_mask);
  P.masks = reinterpret_cast<const uint8_t*>(ws + p.L.masks);
  P.o = static_cast<__nv_bfloat16*>(t.o_out);
  for (int i = 0; i < 3; ++i) P.o_stride[i] = desc.o_stride[i];
  P.lse = t.lse_out;
  P.status = reinterpret_cast<int*>(ws + p.L.status);
  const TestHooks th = test_hooks();
  P.wait_ns = th.wait_ns;
  P.withhold = th.withhold;
  if (f8) {
    P.q_scale = f8->q_scale;
    P.k_scale = f8->k_scale;
    P.v_scale = f8->v_scale;
    P.v_head_scale = f8->v_head_scale;
  }
  // 32-byte O stores where every row allows them
  const bool wide = rows_32b_aligned(t.o_out, desc.o_stride);
  auto kern = wide ? fwd_kernel<D, F8, true> : fwd_kernel<D, F8, false>;
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
  prof_begin(F8 ? K_FWD8 : K_FWD, s);
  kern<<<grid, C::THREADS, C::SMEM, s>>>(P, tq, tk, tv);
  prof_end(F8 ? K_FWD8 : K_FWD, s);
  return cudaGetLastError() == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}

fm_status launch_fwd(const Plan& p, const fm_desc& desc, const TensorArgs& t, char* ws,
                     cudaStream_t s) {
  if (p.d == 64) return launch_fwd_d<64, false>(p, desc, t, ws, s);
  if (p.d == 128) return launch_fwd_d<128, false>(p, desc, t, ws, s);
  return FM_ERR_UNSUPPORTED;
}

fm_status launch_fwd_fp8(const Plan& p, const fm_desc& desc, const TensorArgs& t,
                         const Fp8Args& f, char* ws, cudaStream_t s) {
  if (p.d != 128) return FM_ERR_UNSUPPORTED;
  return launch_fwd_d<128, true>(p, desc, t, ws, s, &f);
}

}  // namespace fm
