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
  static constexpr int NST = 2;             // K/V pipeline stages
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE;
  static constexpr int OFF_V = OFF_K + NST * TILE;
  static constexpr int OFF_BND = OFF_V + NST * TILE;  // NST x 128 x int4
  static constexpr int OFF_BAR = OFF_BND + NST * 128 * 16;
  static constexpr int NBAR = 16;
  // + alignment slack; at least 120 KB so that one CTA (which takes all 512
  // TMEM columns) is resident per SM
  static constexpr int SMEM_USED = OFF_BAR + NBAR * 8 + 16 + 1024;
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  static constexpr uint32_t T_S = 0, T_O = 256, T_P = 384, T_COLS = 512;
};

// barrier slots
enum { B_QFULL = 0, B_QEMPTY, B_SFULL0, B_SFULL1, B_SEMPTY0, B_SEMPTY1, B_PFULL, B_PVDONE,
       B_OEMPTY, B_DRAIN, B_KVFULL0, B_KVEMPTY0 = B_KVFULL0 + 2 };

struct FwdParams {
  int B, H, Hm, Sq, Skv, nQ, nK, n_units;
  float scale_log2;  // scale * log2(e)
  const int32_t* bounds[4];
  const int32_t* row_count;
  const int32_t* row_list;
  const int32_t* order;
  __nv_bfloat16* o;
  int64_t o_stride[3];
  float* lse;
  int* status;
};

__device__ __forceinline__ bool tile_partial(int e, int kj, int nK, int Skv) {
  return ((e & 3) == CLS_PARTIAL) || (kj == nK - 1 && (Skv & (kTile - 1)) != 0);
}

template <int D>
__global__ void __launch_bounds__(192, 1)
    fwd_kernel(const __grid_constant__ FwdParams P, const __grid_constant__ CUtensorMap tmQ,
               const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::OFF_Q;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  int4* bnd = reinterpret_cast<int4*>(smem + C::OFF_BND);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::NBAR * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8 + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    mbar_init(bar(B_SFULL0), 1);
    mbar_init(bar(B_SFULL1), 1);
    mbar_init(bar(B_SEMPTY0), 128);
    mbar_init(bar(B_SEMPTY1), 128);
    mbar_init(bar(B_PFULL), 128);
    mbar_init(bar(B_PVDONE), 1);
    mbar_init(bar(B_OEMPTY), 128);
    mbar_init(bar(B_DRAIN), 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar(B_KVFULL0 + s), 1);
      mbar_init(bar(B_KVEMPTY0 + s), 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), C::T_COLS);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
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
  auto aborted_all = [&]() -> bool { return __any_sync(0xffffffffu, *abort_flag != 0); };

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    uint32_t it = 0, qn = 0;
    for (int idx = blockIdx.x; idx < P.n_units; idx += gridDim.x) {
      const int u = P.order[idx];
      const int bh = u / P.nQ, qi = u - bh * P.nQ;
      const int b = bh / P.H, h = bh - b * P.H;
      const int row = (b * P.Hm + (P.Hm == 1 ? 0 : h)) * P.nQ + qi;
      const int n = P.row_count[row];
      if (n == 0) continue;
      const int32_t* list = P.row_list + static_cast<size_t>(row) * P.nK;
      if (lane == 0) {
        bool ok = qn == 0 || wait(B_QEMPTY, (qn - 1) & 1);
        if (ok) {
          mbar_arrive_expect_tx(bar(B_QFULL), C::TILE);
#pragma unroll
          for (int s = 0; s < C::SLABS; ++s)
            tma_load_4d(sQ + s * 16384, &tmQ, bar(B_QFULL), s * 64, h, qi * kTile, b);
        }
      }
      ++qn;
      for (int t = 0; t < n; ++t, ++it) {
        if (aborted_all()) break;
        const int e = list[t];
        const int kj = e >> 2;
        const int st = it % C::NST;
        const uint32_t use = it / C::NST;
        if (use > 0 && !wait_all(B_KVEMPTY0 + st, (use - 1) & 1)) break;
        if (tile_partial(e, kj, P.nK, P.Skv)) {
          const size_t base = static_cast<size_t>(b * P.Hm + (P.Hm == 1 ? 0 : h)) * P.Skv;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = lane + 32 * i;
            const int j = kj * kTile + c;
            int4 v;
            if (j < P.Skv) {
              v.x = __ldg(P.bounds[0] + base + j);
              v.y = __ldg(P.bounds[1] + base + j);
              v.z = __ldg(P.bounds[2] + base + j);
              v.w = __ldg(P.bounds[3] + base + j);
            } else {
              v = make_int4(0, 0x7fffffff, 0, 0);  // beyond the keys: hidden from every row
            }
            bnd[st * 128 + c] = v;
          }
        }
        __syncwarp();
        if (lane == 0) {
          const uint32_t fb = bar(B_KVFULL0 + st);
          mbar_arrive_expect_tx(fb, 2 * C::TILE);
          const uint32_t sK = sbase + C::OFF_K + st * C::TILE;
          const uint32_t sV = sbase + C::OFF_V + st * C::TILE;
#pragma unroll
          for (int s = 0; s < C::SLABS; ++s) {
            tma_load_4d(sK + s * 16384, &tmK, fb, s * 64, h, kj * kTile, b);
            tma_load_4d(sV + s * 16384, &tmV, fb, s * 64, h, kj * kTile, b);
          }
        }
      }
      if (aborted_all()) break;
    }
    // drain: every issued copy has landed before the CTA may exit
    if (lane == 0) {
      for (uint32_t k = (it > (uint32_t)C::NST ? it - C::NST : 0); k < it; ++k)
        mbar_wait(bar(B_KVFULL0 + k % C::NST), (k / C::NST) & 1, P.status);
      if (qn > 0) mbar_wait(bar(B_QFULL), (qn - 1) & 1, P.status);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idPV = idesc_bf16(128, D, false, true);
      uint32_t it = 0, qn = 0, un = 0;
      auto issue_pv = [&](uint32_t jt, bool first) -> bool {
        if (!wait(B_PFULL, jt & 1)) return false;
        // O is overwritten by a unit's first PV: the previous epilogue must be done
        if (first) {
          if (un > 0 && !wait(B_OEMPTY, (un - 1) & 1)) return false;
          ++un;
        }
        tc_fence_after();
        const int st = jt % C::NST;
        const uint32_t sV = sbase + C::OFF_V + st * C::TILE;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd = sdesc_sw128(sV + kk * 2048, 128 * 128, 1024);
          mma_ts(tbase + C::T_O, tbase + C::T_P + kk * 8, bd, idPV, (!first || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(B_PVDONE));
        mma_commit(bar(B_KVEMPTY0 + st));
        return true;
      };
      for (int idx = blockIdx.x; idx < P.n_units; idx += gridDim.x) {
        const int u = P.order[idx];
        const int bh = u / P.nQ, qi = u - bh * P.nQ;
        const int b = bh / P.H, h = bh - b * P.H;
        const int row = (b * P.Hm + (P.Hm == 1 ? 0 : h)) * P.nQ + qi;
        const int n = P.row_count[row];
        if (n == 0) continue;
        if (!wait(B_QFULL, qn & 1)) break;
        ++qn;
        bool ok = true;
        for (int t = 0; t < n; ++t, ++it) {
          const int st = it % C::NST;
          const int sb = it & 1;
          if (!wait(B_KVFULL0 + st, (it / C::NST) & 1)) { ok = false; break; }
          if (it >= 2 && !wait(B_SEMPTY0 + sb, ((it >> 1) - 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sK = sbase + C::OFF_K + st * C::TILE;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(tbase + C::T_S + sb * 128, sdesc_sw128(sQ + koff, 16, 1024),
                   sdesc_sw128(sK + koff, 16, 1024), idS, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(B_SFULL0 + sb));
          if (t == n - 1) mma_commit(bar(B_QEMPTY));
          if (t > 0 && !issue_pv(it - 1, t == 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (!issue_pv(it - 1, n == 1)) break;
      }
      mma_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, P.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int r = tid;  // query row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t it = 0, un = 0;
    for (int idx = blockIdx.x; idx < P.n_units; idx += gridDim.x) {
      const int u = P.order[idx];
      const int bh = u / P.nQ, qi = u - bh * P.nQ;
      const int b = bh / P.H, h = bh - b * P.H;
      const int row = (b * P.Hm + (P.Hm == 1 ? 0 : h)) * P.nQ + qi;
      const int n = P.row_count[row];
      const int32_t* list = P.row_list + static_cast<size_t>(row) * P.nK;
      const int qrow = qi * kTile + r;
      __nv_bfloat16* orow = P.o + b * P.o_stride[0] + static_cast<int64_t>(qrow) * P.o_stride[1] +
                            h * P.o_stride[2];
      float* lse_out = P.lse + (static_cast<size_t>(b) * P.H + h) * P.Sq + qrow;
      if (n == 0) {
        if (qrow < P.Sq) {
          uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
          *lse_out = -INFINITY;
        }
        continue;
      }
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int t = 0; t < n; ++t, ++it) {
        const int e = list[t];
        const int kj = e >> 2;
        const int sb = it & 1;
        if (!wait_all(B_SFULL0 + sb, (it >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        float s[128];
        {
          uint32_t raw[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            tmem_ld32(tbase + lane_off + C::T_S + sb * 128 + c * 32, raw);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(raw[i]);
          }
        }
        tc_fence_before();
        mbar_arrive(bar(B_SEMPTY0 + sb));
        if (tile_partial(e, kj, P.nK, P.Skv)) {
          const int st = it % C::NST;
          if (!wait_all(B_KVFULL0 + st, (it / C::NST) & 1)) { ok = false; break; }
          const int4* bb = bnd + st * 128;
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            const int4 v = bb[c];
            const bool hid = (v.x <= qrow && qrow < v.y) || (v.z <= qrow && qrow < v.w);
            s[c] = hid ? -INFINITY : s[c];
          }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; ++c) mx = fmaxf(mx, s[c]);
        const float m_new = fmaxf(m, mx * P.scale_log2);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2(m - m_use);
        float sum = 0.f;
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float p0 = ex2(fmaf(s[2 * c], P.scale_log2, -m_use));
          const float p1 = ex2(fmaf(s[2 * c + 1], P.scale_log2, -m_use));
          sum += p0 + p1;
          pk[c] = pack_bf16(p0, p1);
        }
        l = l * alpha + sum;
        if (t > 0) {
          // the previous PV has finished: P may be overwritten and O is stable
          if (!wait_all(B_PVDONE, (it - 1) & 1)) { ok = false; break; }
          tc_fence_after();
          // TMEM loads/stores are warp-collective: the whole warp rescales
          // if any of its rows needs it (alpha == 1 leaves a row unchanged)
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
            uint32_t raw[32];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              const uint32_t ta = tbase + lane_off + C::T_O + c * 32;
              tmem_ld32(ta, raw);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) raw[i] = __float_as_uint(__uint_as_float(raw[i]) * alpha);
              tmem_st32(ta, raw);
            }
          }
        }
        tmem_st32(tbase + lane_off + C::T_P, pk);
        tmem_st32(tbase + lane_off + C::T_P + 32, pk + 32);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(B_PFULL));
        m = m_new;
      }
      if (!ok) break;
      // epilogue: O / l and LSE
      if (!wait_all(B_PVDONE, (it - 1) & 1)) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint32_t raw[32];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        tmem_ld32(tbase + lane_off + C::T_O + c * 32, raw);
        tmem_wait_ld();
        if (qrow < P.Sq) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16(__uint_as_float(raw[2 * i]) * inv, __uint_as_float(raw[2 * i + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (qrow < P.Sq) {
        const float m_use = (m == -INFINITY) ? 0.f : m;
        *lse_out = l > 0.f ? (m_use + __log2f(l)) * 0.69314718055994530942f : -INFINITY;
      }
      tc_fence_before();
      mbar_arrive(bar(B_OEMPTY));
      ++un;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
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
  P.o = static_cast<__nv_bfloat16*>(t.o_out);
  for (int i = 0; i < 3; ++i) P.o_stride[i] = desc.o_stride[i];
  P.lse = t.lse_out;
  P.status = reinterpret_cast<int*>(ws + p.L.status);
  auto kern = fwd_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
      cudaSuccess)
    return FM_ERR_CUDA;
  const int grid = P.n_units < num_sms() ? P.n_units : num_sms();
  prof_begin(K_FWD, s);
  kern<<<grid, 192, C::SMEM, s>>>(P, tq, tk, tv);
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
