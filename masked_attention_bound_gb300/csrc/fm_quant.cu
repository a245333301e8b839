// Per-tile e4m3 quantisation of Q, K and V for the FP8 forward.
//
// One CTA per (batch, head, 128-row tile) of one tensor: the tile's largest
// magnitude amax (block reduction), scale s = amax / 448 in fp32 (1 for an
// all-zero tile), codes e4m3(x / s) with an IEEE fp32 division and the
// saturating round-to-nearest-even conversion.  Q and K codes keep the BSHD
// layout (one byte per element); V codes are written transposed per head,
// [b][h][d][key] over a key axis padded to whole tiles (padding = 0), so that
// V^T tiles are K-major operands of the P V product.  V also records, per
// (b, h), the largest of its tile scales (the per-head scale of P V).
#include <cuda_bf16.h>

#include "fm_internal.h"
#include "fm_ptx.cuh"

namespace fm {

namespace {

constexpr int kQuantD = 128;  // head_dim of the FP8 path

struct QuantArgs {
  const __nv_bfloat16* x;
  int64_t xs[3];   // element strides of x for (b, s, h)
  int B, S, H, nT;
  uint8_t* out;    // codes
  int64_t os[3];   // byte strides of out for (b, s, h) (BSHD) - unused when transposed
  int S_pad;       // transposed: key-axis length of out
  float* scales;   // [B][H][nT]
  float* head_max; // transposed only: [B][H], zeroed before the launch
};

template <bool TRANSPOSE>
__global__ void __launch_bounds__(256) quant_kernel(const __grid_constant__ QuantArgs A) {
  __shared__ float red[8];
  __shared__ __align__(16) uint8_t tr[TRANSPOSE ? kQuantD * 128 : 16];  // [c][row]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bid = blockIdx.x;
  const int t = bid % A.nT, bh = bid / A.nT, b = bh / A.H, h = bh - b * A.H;
  const int r0 = t * 128;
  const int rows = min(128, A.S - r0);
  // thread: row (tid / 16) + 16 i, 8-column chunk (tid % 16): 8 rows x 8 values
  const int ch = tid & 15, rb = tid >> 4;
  float v[8][8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = rb + 16 * i;
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows)
      u = *reinterpret_cast<const uint4*>(A.x + b * A.xs[0] + static_cast<int64_t>(r0 + r) * A.xs[1] +
                                          h * A.xs[2] + ch * 8);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[i][2 * j] = __uint_as_float(w[j] << 16);
      v[i][2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
      amax = fmaxf(amax, fmaxf(fabsf(v[i][2 * j]), fabsf(v[i][2 * j + 1])));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  if (tid == 0) {
    A.scales[static_cast<size_t>(bh) * A.nT + t] = s;
    if (TRANSPOSE) atomicMax(reinterpret_cast<int*>(A.head_max) + bh, __float_as_int(s));
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = rb + 16 * i;
    const uint32_t lo = pack_e4m3x4(__fdiv_rn(v[i][0], s), __fdiv_rn(v[i][1], s),
                                    __fdiv_rn(v[i][2], s), __fdiv_rn(v[i][3], s));
    const uint32_t hi = pack_e4m3x4(__fdiv_rn(v[i][4], s), __fdiv_rn(v[i][5], s),
                                    __fdiv_rn(v[i][6], s), __fdiv_rn(v[i][7], s));
    if (!TRANSPOSE) {
      if (r < rows)
        *reinterpret_cast<uint2*>(A.out + b * A.os[0] + static_cast<int64_t>(r0 + r) * A.os[1] +
                                  h * A.os[2] + ch * 8) = make_uint2(lo, hi);
    } else {
      // column c = ch * 8 + k of row r goes to tr[c][r] (rows past S hold 0)
#pragma unroll
      for (int k = 0; k < 8; ++k)
        tr[(ch * 8 + k) * 128 + r] = static_cast<uint8_t>(((k < 4 ? lo : hi) >> (8 * (k & 3))) & 0xffu);
    }
  }
  if (TRANSPOSE) {
    __syncthreads();
    // d rows of 128 keys: 16-byte pieces, 8 per row
    uint8_t* dst = A.out + (static_cast<size_t>(bh) * kQuantD) * A.S_pad + r0;
    for (int i = tid; i < kQuantD * 8; i += 256) {
      const int c = i >> 3, piece = i & 7;
      *reinterpret_cast<uint4*>(dst + static_cast<size_t>(c) * A.S_pad + piece * 16) =
          *reinterpret_cast<const uint4*>(tr + c * 128 + piece * 16);
    }
  }
}

}  // namespace

fm_status launch_quantize_fp8(const Plan& p, const fm_desc& desc, const void* q, const void* k,
                              const void* v, void* q8, void* k8, void* v8t, float* q_scale,
                              float* k_scale, float* v_scale, float* v_head_scale,
                              cudaStream_t s) {
  if (p.d != kQuantD) return FM_ERR_UNSUPPORTED;
  const int S_pad = p.nK * 128;
  if (cudaMemsetAsync(v_head_scale, 0, sizeof(float) * p.B * p.Hkv, s) != cudaSuccess)
    return FM_ERR_CUDA;
  auto run = [&](const void* x, const int64_t* xs, int S, int H, int nT, uint8_t* out,
                 float* sc, bool transpose) -> bool {
    QuantArgs A{};
    A.x = static_cast<const __nv_bfloat16*>(x);
    for (int i = 0; i < 3; ++i) A.xs[i] = xs[i];
    A.B = p.B; A.S = S; A.H = H; A.nT = nT;
    A.out = out;
    A.os[0] = static_cast<int64_t>(S) * H * kQuantD;
    A.os[1] = static_cast<int64_t>(H) * kQuantD;
    A.os[2] = kQuantD;
    A.S_pad = S_pad;
    A.scales = sc;
    A.head_max = v_head_scale;
    const unsigned grid = static_cast<unsigned>(p.B) * H * nT;
    prof_begin(K_QUANT, s);
    if (transpose) quant_kernel<true><<<grid, 256, 0, s>>>(A);
    else quant_kernel<false><<<grid, 256, 0, s>>>(A);
    prof_end(K_QUANT, s);
    return cudaGetLastError() == cudaSuccess;
  };
  if (!run(q, desc.q_stride, p.Sq, p.H, p.nQ, static_cast<uint8_t*>(q8), q_scale, false) ||
      !run(k, desc.k_stride, p.Skv, p.Hkv, p.nK, static_cast<uint8_t*>(k8), k_scale, false) ||
      !run(v, desc.v_stride, p.Skv, p.Hkv, p.nK, static_cast<uint8_t*>(v8t), v_scale, true))
    return FM_ERR_CUDA;
  return FM_OK;
}

}  // namespace fm
