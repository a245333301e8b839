// Host-side declarations shared by the library's translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "fm.h"

namespace fm {

constexpr int kTile = 128;            // q-tile and k-tile edge
constexpr int kMaxChunks = 128;       // fm_localize chunk limit
constexpr int kMaxMaskTiles = 65536;  // partial tiles with a precomputed bit mask
constexpr int kMaskBytes = 128 * 16;  // 128 rows x 128 column bits

enum : int { CLS_EMPTY = 0, CLS_PARTIAL = 1, CLS_FULL = 2 };

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// A bf16 [B][S][H][d] tensor whose every row (and every 16-element piece of
// one) starts on a 32-byte boundary: the base is 32-byte aligned and every
// stride (in elements) is a multiple of 16.
inline bool rows_32b_aligned(const void* base, const int64_t (&stride)[3]) {
  if (reinterpret_cast<uintptr_t>(base) % 32 != 0) return false;
  for (int i = 0; i < 3; ++i)
    if (stride[i] % 16 != 0) return false;
  return true;
}

struct Plan {
  int B, H, Hm, Sq, Skv, d, nQ, nK;
  int Hkv, G;    // K/V heads and query heads per K/V head (H = G * Hkv)
  int nP;        // q-tile pairs, ceil(nQ / 2)
  int mask_cap;  // forward: slots in the visibility-mask region
  fm_ws_layout L;
};

// Validates the description (shapes and strides) and computes the layout.
// limit: the most bytes the forward layout may take; the visibility-mask
// region shrinks to fit (rows without slots fall back to bits built in the
// forward kernel).  Other regions do not shrink.
// mode: FM_WS_FWD, FM_WS_BWD or FM_WS_STEP (both passes)
fm_status make_plan(const fm_desc* desc, int mode, Plan* p, size_t limit = SIZE_MAX);

// Mask analysis kernels (fm_mask.cu).
cudaError_t launch_summary(const Plan& p, const int32_t* lts, const int32_t* lte,
                           const int32_t* uts, const int32_t* ute, char* ws, cudaStream_t s);
cudaError_t launch_classify(const Plan& p, char* ws, int mode, cudaStream_t s);
// unit orders: ORDER_PAIRS (forward, q-tile pairs), ORDER_COLS (dK/dV, k-tile
// columns), ORDER_ROWS (dQ, q-tile rows)
enum : int { ORDER_PAIRS = 0, ORDER_COLS, ORDER_ROWS };
// builds the orders whose bits (1 << ORDER_*) are set in `which`, in one launch
cudaError_t launch_orders(const Plan& p, char* ws, unsigned which, cudaStream_t s);
cudaError_t launch_varlen_bounds(const int32_t* cu, int n, int total, int causal, int32_t* out,
                                 int* bad, cudaStream_t s);
cudaError_t launch_tile_masks(const Plan& p, const int32_t* lts, const int32_t* lte,
                              const int32_t* uts, const int32_t* ute, char* ws, cudaStream_t s);

struct ChunkMap {
  int n;
  int start[kMaxChunks];
  int len[kMaxChunks];
  int offset[kMaxChunks];
};
cudaError_t launch_localize(const int32_t* in, int32_t* out, long long n_values,
                            const ChunkMap& cm, cudaStream_t s);

// Attention kernels (fm_fwd.cu, fm_bwd.cu).
struct TensorArgs {
  const void* q; const void* k; const void* v; const void* o; const void* dout;
  void* o_out; float* lse_out; const float* lse_in;
  void* dq; void* dk; void* dv;
  const int32_t* bounds[4];
  float scale;
};
fm_status launch_fwd(const Plan& p, const fm_desc& desc, const TensorArgs& t, char* ws,
                     cudaStream_t s);
fm_status launch_bwd(const Plan& p, const fm_desc& desc, const TensorArgs& t, char* ws,
                     cudaStream_t s);
// FP8 forward: per-tile e4m3 quantisation (fm_quant.cu) and the forward
// kernel on the codes (fm_fwd.cu); d = 128 only
fm_status launch_quantize_fp8(const Plan& p, const fm_desc& desc, const void* q, const void* k,
                              const void* v, void* q8, void* k8, void* v8t, float* q_scale,
                              float* k_scale, float* v_scale, float* v_head_scale, cudaStream_t s);
struct Fp8Args {
  const void* q8; const void* k8; const void* v8t;
  const float* q_scale; const float* k_scale; const float* v_scale; const float* v_head_scale;
};
fm_status launch_fwd_fp8(const Plan& p, const fm_desc& desc, const TensorArgs& t,
                         const Fp8Args& f, char* ws, cudaStream_t s);

int num_sms();

// Settings of fm_test_hooks (process-wide): the limit of every device-side
// mbarrier wait, and which release a test withholds (0 none).
struct TestHooks {
  uint64_t wait_ns;
  int withhold;
};
TestHooks test_hooks();

// Kernel ids for the timing hooks (fm_profile_*).
enum KernelId : int { K_SUMMARY = 0, K_CLASSIFY, K_ORDER, K_LOCALIZE, K_FWD, K_BWD_PRE, K_BWD,
                      K_BWD_DQ, K_TILE_MASKS, K_QUANT, K_FWD8, K_COUNT };
void prof_begin(int id, cudaStream_t s);
void prof_end(int id, cudaStream_t s);

}  // namespace fm
