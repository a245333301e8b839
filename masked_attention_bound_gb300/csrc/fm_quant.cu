// Per-tile e4m3 quantisation of Q, K and V for the FP8 forward.
//
// One CTA per (batch, head, 128-row tile) of one tensor: the tile's largest
// magnitude amax (block reduction), scale s = amax / 448 and its reciprocal
// r = 448 / amax in fp32 (IEEE divisions, once per tile; both 1 for an
// all-zero tile), codes e4m3(x * r) with an fp32 product and the saturating
// round-to-nearest-even conversion.  Q and K codes keep the BSHD
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
__global__ void __launch_bounds__(256, TRANSPOSE ? 3 : 4) quant_kernel(const __grid_constant__ QuantArgs A) {
  __shared__ float red[8];
  // transposed: [c][row] with the 8-byte slots of row group g at slot
  // g xor (c / 8), so that the stores of a warp hit distinct banks
  __shared__ __align__(16) uint8_t tr[TRANSPOSE ? kQuantD * 128 : 16];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bid = blockIdx.x;
  const int t = bid % A.nT, bh = bid / A.nT, b = bh / A.H, h = bh - b * A.H;
  const int r0 = t * 128;
  const int rows = min(128, A.S - r0);
  // thread: rows 8 g .. 8 g + 7 (g = tid / 16), 8-column chunk tid % 16:
  // 8 rows x 8 values, kept as packed bf16 (unpacked once for the maximum
  // and once for the conversion) so that four CTAs fit on an SM
  const int ch = tid & 15, g = tid >> 4;
  uint4 raw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 8 * g + i;
    raw[i] = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows)
      raw[i] = *reinterpret_cast<const uint4*>(A.x + b * A.xs[0] + static_cast<int64_t>(r0 + r) * A.xs[1] +
                                               h * A.xs[2] + ch * 8);
  }
  // |x| of a bf16 is its bit pattern without the sign, and the order of the
  // magnitudes is the order of those patterns
  uint32_t mbits = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) mbits = max(mbits, max(w[j] & 0x7fffu, (w[j] >> 16) & 0x7fffu));
  }
  float amax = __uint_as_float(mbits << 16);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  const float rs = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
  if (tid == 0) {
    A.scales[static_cast<size_t>(bh) * A.nT + t] = s;
    if (TRANSPOSE) atomicMax(reinterpret_cast<int*>(A.head_max) + bh, __float_as_int(s));
  }
  uint32_t code[8][2];  // row i: columns 0-3, 4-7 of the chunk (byte k = column k mod 4)
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 8 * g + i;
    const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
    float v[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(w[j] << 16);
      v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
    const uint32_t lo = pack_e4m3x4(v[0] * rs, v[1] * rs, v[2] * rs, v[3] * rs);
    const uint32_t hi = pack_e4m3x4(v[4] * rs, v[5] * rs, v[6] * rs, v[7] * rs);
    if (!TRANSPOSE) {
      if (r < rows)
        *reinterpret_cast<uint2*>(A.out + b * A.os[0] + static_cast<int64_t>(r0 + r) * A.os[1] +
                                  h * A.os[2] + ch * 8) = make_uint2(lo, hi);
    }
    code[i][0] = lo;
    code[i][1] = hi;
  }
  if (TRANSPOSE) {
    // each 4 x 4 byte block (4 rows x 4 columns) transposed with byte
    // permutes, so that a column's 8 bytes of rows 8 g .. 8 g + 7 form one
    // 8-byte store into tile row c (rows past S hold 0)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {        // columns 0-3 / 4-7 of the chunk
      uint32_t colw[2][4];                  // [row half][column]: 4 row bytes
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        const uint32_t w0 = code[4 * rh][hf], w1 = code[4 * rh + 1][hf], w2 = code[4 * rh + 2][hf],
                       w3 = code[4 * rh + 3][hf];
        const uint32_t t0 = __byte_perm(w0, w1, 0x5140), t1 = __byte_perm(w2, w3, 0x5140);
        const uint32_t t2 = __byte_perm(w0, w1, 0x7362), t3 = __byte_perm(w2, w3, 0x7362);
        colw[rh][0] = __byte_perm(t0, t1, 0x5410);
        colw[rh][1] = __byte_perm(t0, t1, 0x7632);
        colw[rh][2] = __byte_perm(t2, t3, 0x5410);
        colw[rh][3] = __byte_perm(t2, t3, 0x7632);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = ch * 8 + 4 * hf + k;
        *reinterpret_cast<uint2*>(tr + c * 128 + ((g ^ (c >> 3)) << 3)) = make_uint2(colw[0][k], colw[1][k]);
      }
    }
    __syncthreads();
    // d rows of 128 keys: 16-byte pieces, 8 per row; piece p of tile row c is
    // the slot pair p xor (c / 16), its halves swapped when c / 8 is odd
    uint8_t* dst = A.out + (static_cast<size_t>(bh) * kQuantD) * A.S_pad + r0;
    for (int i = tid; i < kQuantD * 8; i += 256) {
      const int c = i >> 3, piece = i & 7, chc = c >> 3;
      uint4 v = *reinterpret_cast<const uint4*>(tr + c * 128 + ((piece ^ (chc >> 1)) << 4));
      if (chc & 1) v = make_uint4(v.z, v.w, v.x, v.y);
      *reinterpret_cast<uint4*>(dst + static_cast<size_t>(c) * A.S_pad + piece * 16) = v;
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
