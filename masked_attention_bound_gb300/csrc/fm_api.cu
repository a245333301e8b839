// The C ABI of include/fm.h: argument validation, workspace layout, and the
// sequence of launches for each entry point.
#include <cstring>

#include "fm_internal.h"
#include "fm_ptx.cuh"

namespace fm {

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

namespace {
TestHooks g_hooks = {FM_WAIT_LIMIT_NS, 0};
}  // namespace

TestHooks test_hooks() { return g_hooks; }

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static bool strides_ok(const int64_t* st) {
  for (int i = 0; i < 3; ++i)
    if (st[i] <= 0 || (st[i] % 8) != 0 || st[i] >= (int64_t(1) << 36)) return false;
  return true;
}

fm_status make_plan(const fm_desc* desc, int mode, Plan* p, size_t limit) {
  if (!desc || !p) return FM_ERR_INVALID;
  if (mode < FM_WS_FWD || mode > FM_WS_STEP) return FM_ERR_INVALID;
  const fm_desc& D = *desc;
  if (D.B < 1 || D.H < 1 || D.Sq < 1 || D.Skv < 1 || D.d < 1) return FM_ERR_INVALID;
  if (D.Hm != 1 && D.Hm != D.H) return FM_ERR_INVALID;
  const int Hkv = D.Hkv == 0 ? D.H : D.Hkv;
  if (Hkv < 1 || Hkv > D.H || D.H % Hkv != 0) return FM_ERR_INVALID;
  if (D.d != 64 && D.d != 128) return FM_ERR_UNSUPPORTED;
  if (!strides_ok(D.q_stride) || !strides_ok(D.k_stride) || !strides_ok(D.v_stride) ||
      !strides_ok(D.o_stride))
    return FM_ERR_INVALID;
  if (D.Sq > (1 << 24) || D.Skv > (1 << 24)) return FM_ERR_UNSUPPORTED;
  p->B = D.B; p->H = D.H; p->Hm = D.Hm; p->Sq = D.Sq; p->Skv = D.Skv; p->d = D.d;
  p->Hkv = Hkv; p->G = D.H / Hkv;
  p->nQ = ceil_div(D.Sq, kTile);
  p->nK = ceil_div(D.Skv, kTile);
  p->nP = ceil_div(p->nQ, 2);
  const size_t BHm = static_cast<size_t>(D.B) * D.Hm;
  const size_t BH = static_cast<size_t>(D.B) * D.H;
  fm_ws_layout& L = p->L;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t at = off; off = align256(off + bytes); return at; };
  L.status = take(32);
  L.summary = take(BHm * p->nK * 8 * 4);
  L.table = take(BHm * p->nQ * p->nK);
  L.row_count = take(BHm * p->nQ * 4);
  L.row_list = take(BHm * p->nQ * p->nK * 4);
  L.col_count = take(BHm * p->nK * 4);
  L.col_list = take(BHm * p->nK * p->nQ * 4);
  L.fwd_order = take(BH * p->nQ * 4);
  L.bwd_order = take(BH * p->nK * 4);
  L.row_mask = take(BHm * p->nQ * 4);
  L.pair_info = L.pair_list = L.delta = L.lse_log2 = L.row_order = 0;
  if (mode != FM_WS_BWD) {
    L.pair_info = take(BHm * p->nP * 16);
    L.pair_list = take(BHm * p->nP * p->nK * 4);
  }
  if (mode != FM_WS_FWD) {
    L.delta = take(BH * p->nQ * kTile * 4);
    L.lse_log2 = take(BH * p->nQ * kTile * 4);
    L.row_order = take(BH * p->nQ * 4);
  }
  {
    // the mask region comes last and takes what the limit leaves, up to one
    // slot per tile and kMaxMaskTiles slots
    size_t cap = BHm * p->nQ * p->nK;
    if (cap > static_cast<size_t>(kMaxMaskTiles)) cap = kMaxMaskTiles;
    const size_t room = limit > off ? (limit - off) / kMaskBytes : 0;
    if (cap > room) cap = room;
    p->mask_cap = static_cast<int>(cap);
    L.masks = take(cap * kMaskBytes);
  }
  L.total = off;
  return FM_OK;
}

static fm_status check_ws(const Plan& p, const void* ws, size_t ws_bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return FM_ERR_WORKSPACE;
  if (ws_bytes < p.L.total) return FM_ERR_WORKSPACE;
  return FM_OK;
}

static bool aligned16(const void* ptr) {
  return ptr && (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0;
}

static fm_status run_plan(const Plan& p, const int32_t* lts, const int32_t* lte,
                          const int32_t* uts, const int32_t* ute, char* ws, int mode,
                          cudaStream_t s) {
  if (cudaMemsetAsync(ws + p.L.status, 0, 32, s) != cudaSuccess) return FM_ERR_CUDA;
  if (launch_summary(p, lts, lte, uts, ute, ws, s) != cudaSuccess) return FM_ERR_CUDA;
  if (launch_classify(p, ws, mode, s) != cudaSuccess) return FM_ERR_CUDA;
  if (launch_tile_masks(p, lts, lte, uts, ute, ws, s) != cudaSuccess) return FM_ERR_CUDA;
  unsigned orders = 0;
  if (mode != FM_WS_BWD) orders |= 1u << ORDER_PAIRS;
  if (mode != FM_WS_FWD) orders |= (1u << ORDER_COLS) | (1u << ORDER_ROWS);
  if (launch_orders(p, ws, orders, s) != cudaSuccess) return FM_ERR_CUDA;
  return FM_OK;
}

// Zero the status words that count the attention kernels' claimed units
// ([1]: the forward's and the dK/dV pass's, [4]: the dQ pass's), keeping the
// analysis' device status bits and mask-slot count.
static fm_status reset_claims(const Plan& p, char* ws, int bwd, cudaStream_t s) {
  if (cudaMemsetAsync(ws + p.L.status + 4, 0, 4, s) != cudaSuccess) return FM_ERR_CUDA;
  if (bwd && cudaMemsetAsync(ws + p.L.status + 16, 0, 4, s) != cudaSuccess) return FM_ERR_CUDA;
  return FM_OK;
}

}  // namespace fm

using namespace fm;

extern "C" {

size_t fm_workspace_size(const fm_desc* desc, int mode) {
  Plan p;
  if (make_plan(desc, mode, &p) != FM_OK) return 0;
  return p.L.total;
}

fm_status fm_workspace_layout(const fm_desc* desc, int mode, fm_ws_layout* out) {
  if (!out) return FM_ERR_INVALID;
  Plan p;
  fm_status st = make_plan(desc, mode, &p);
  if (st != FM_OK) return st;
  *out = p.L;
  return FM_OK;
}

fm_status fm_plan(const fm_desc* desc, const int32_t* lts, const int32_t* lte,
                  const int32_t* uts, const int32_t* ute, void* ws, size_t ws_bytes,
                  int mode, void* stream) {
  Plan p;
  fm_status st = make_plan(desc, mode, &p);
  if (st != FM_OK) return st;
  if (!lts || !lte || !uts || !ute) return FM_ERR_INVALID;
  if ((st = check_ws(p, ws, ws_bytes)) != FM_OK) return st;
  return run_plan(p, lts, lte, uts, ute, static_cast<char*>(ws), mode,
                  static_cast<cudaStream_t>(stream));
}

// The forward with its own analysis (planned = 0, FM_WS_FWD layout) or on a
// step workspace whose analysis fm_plan(FM_WS_STEP) made (planned = 1).
static fm_status run_forward(const fm_desc* desc, const void* q, const void* k, const void* v,
                         const int32_t* lts, const int32_t* lte, const int32_t* uts,
                         const int32_t* ute, float scale, void* o, float* lse, void* ws,
                         size_t ws_bytes, void* stream, int planned) {
  Plan p;
  fm_status st = make_plan(desc, planned ? FM_WS_STEP : FM_WS_FWD, &p);
  if (st != FM_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !lse) return FM_ERR_INVALID;
  if (!lts || !lte || !uts || !ute) return FM_ERR_INVALID;
  if ((st = check_ws(p, ws, ws_bytes)) != FM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  st = planned ? reset_claims(p, w, 0, s) : run_plan(p, lts, lte, uts, ute, w, FM_WS_FWD, s);
  if (st != FM_OK) return st;
  TensorArgs t{};
  t.q = q; t.k = k; t.v = v; t.o_out = o; t.lse_out = lse;
  t.bounds[0] = lts; t.bounds[1] = lte; t.bounds[2] = uts; t.bounds[3] = ute;
  t.scale = scale;
  return launch_fwd(p, *desc, t, w, s);
}

static fm_status run_backward(const fm_desc* desc, const void* q, const void* k, const void* v,
                          const void* o, const float* lse, const void* dout,
                          const int32_t* lts, const int32_t* lte, const int32_t* uts,
                          const int32_t* ute, float scale, void* dq, void* dk, void* dv,
                          void* ws, size_t ws_bytes, void* stream, int planned) {
  Plan p;
  fm_status st = make_plan(desc, planned ? FM_WS_STEP : FM_WS_BWD, &p);
  if (st != FM_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !lse)
    return FM_ERR_INVALID;
  if (!lts || !lte || !uts || !ute) return FM_ERR_INVALID;
  if ((st = check_ws(p, ws, ws_bytes)) != FM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  st = planned ? reset_claims(p, w, 1, s) : run_plan(p, lts, lte, uts, ute, w, FM_WS_BWD, s);
  if (st != FM_OK) return st;
  TensorArgs t{};
  t.q = q; t.k = k; t.v = v; t.o = o; t.dout = dout; t.lse_in = lse;
  t.dq = dq; t.dk = dk; t.dv = dv;
  t.bounds[0] = lts; t.bounds[1] = lte; t.bounds[2] = uts; t.bounds[3] = ute;
  t.scale = scale;
  return launch_bwd(p, *desc, t, w, s);
}

fm_status fm_fwd(const fm_desc* desc, const void* q, const void* k, const void* v,
                 const int32_t* lts, const int32_t* lte, const int32_t* uts,
                 const int32_t* ute, float scale, void* o, float* lse, void* ws,
                 size_t ws_bytes, void* stream) {
  return run_forward(desc, q, k, v, lts, lte, uts, ute, scale, o, lse, ws, ws_bytes, stream, 0);
}

fm_status fm_fwd_planned(const fm_desc* desc, const void* q, const void* k, const void* v,
                         const int32_t* lts, const int32_t* lte, const int32_t* uts,
                         const int32_t* ute, float scale, void* o, float* lse, void* ws,
                         size_t ws_bytes, void* stream) {
  return run_forward(desc, q, k, v, lts, lte, uts, ute, scale, o, lse, ws, ws_bytes, stream, 1);
}

fm_status fm_bwd(const fm_desc* desc, const void* q, const void* k, const void* v,
                 const void* o, const float* lse, const void* dout, const int32_t* lts,
                 const int32_t* lte, const int32_t* uts, const int32_t* ute, float scale,
                 void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, void* stream) {
  return run_backward(desc, q, k, v, o, lse, dout, lts, lte, uts, ute, scale, dq, dk, dv, ws,
                  ws_bytes, stream, 0);
}

fm_status fm_bwd_planned(const fm_desc* desc, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* dout,
                         const int32_t* lts, const int32_t* lte, const int32_t* uts,
                         const int32_t* ute, float scale, void* dq, void* dk, void* dv,
                         void* ws, size_t ws_bytes, void* stream) {
  return run_backward(desc, q, k, v, o, lse, dout, lts, lte, uts, ute, scale, dq, dk, dv, ws,
                  ws_bytes, stream, 1);
}

fm_status fm_quantize_fp8(const fm_desc* desc, const void* q, const void* k, const void* v,
                          void* q8, void* k8, void* v8t, float* q_scale, float* k_scale,
                          float* v_scale, float* v_head_scale, void* stream) {
  Plan p;
  fm_status st = make_plan(desc, FM_WS_FWD, &p);
  if (st != FM_OK) return st;
  if (p.d != 128) return FM_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q8) || !aligned16(k8) ||
      !aligned16(v8t) || !q_scale || !k_scale || !v_scale || !v_head_scale)
    return FM_ERR_INVALID;
  return launch_quantize_fp8(p, *desc, q, k, v, q8, k8, v8t, q_scale, k_scale, v_scale,
                             v_head_scale, static_cast<cudaStream_t>(stream));
}

fm_status fm_fwd_fp8(const fm_desc* desc, const void* q8, const void* k8, const void* v8t,
                     const float* q_scale, const float* k_scale, const float* v_scale,
                     const float* v_head_scale, const int32_t* lts, const int32_t* lte,
                     const int32_t* uts, const int32_t* ute, float scale, void* o, float* lse,
                     void* ws, size_t ws_bytes, void* stream) {
  Plan p;
  fm_status st = make_plan(desc, FM_WS_FWD, &p);
  if (st != FM_OK) return st;
  if (p.d != 128) return FM_ERR_UNSUPPORTED;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8t) || !aligned16(o) || !lse ||
      !q_scale || !k_scale || !v_scale || !v_head_scale)
    return FM_ERR_INVALID;
  if (!lts || !lte || !uts || !ute) return FM_ERR_INVALID;
  if ((st = check_ws(p, ws, ws_bytes)) != FM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  if ((st = run_plan(p, lts, lte, uts, ute, w, FM_WS_FWD, s)) != FM_OK) return st;
  TensorArgs t{};
  t.o_out = o; t.lse_out = lse;
  t.bounds[0] = lts; t.bounds[1] = lte; t.bounds[2] = uts; t.bounds[3] = ute;
  t.scale = scale;
  Fp8Args f{q8, k8, v8t, q_scale, k_scale, v_scale, v_head_scale};
  return launch_fwd_fp8(p, *desc, t, f, w, s);
}

fm_status fm_varlen_bounds(const int32_t* cu_seqlens, int n_seqs, int total, int causal,
                           int32_t* bounds, int* bad, void* stream) {
  if (!cu_seqlens || !bounds || n_seqs < 1 || total < 1 || total > (1 << 24)) return FM_ERR_INVALID;
  if (launch_varlen_bounds(cu_seqlens, n_seqs, total, causal != 0, bounds, bad,
                           static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FM_ERR_CUDA;
  return FM_OK;
}

fm_status fm_localize(const int32_t* bounds, int B, int Hm, int Skv,
                      const int32_t* chunk_start, const int32_t* chunk_len, int n_chunks,
                      int32_t* local_bounds, void* stream) {
  if (!bounds || !local_bounds || !chunk_start || !chunk_len) return FM_ERR_INVALID;
  if (B < 1 || Hm < 1 || Skv < 1 || n_chunks < 1 || n_chunks > kMaxChunks) return FM_ERR_INVALID;
  const long long n = 4LL * B * Hm * Skv;
  const char* a = reinterpret_cast<const char*>(bounds);
  const char* b = reinterpret_cast<const char*>(local_bounds);
  if (a < b + n * 4 && b < a + n * 4) return FM_ERR_INVALID;  // overlapping buffers
  ChunkMap cm;
  std::memset(&cm, 0, sizeof(cm));
  cm.n = n_chunks;
  long long off = 0, end = -1;
  for (int c = 0; c < n_chunks; ++c) {
    const int g = chunk_start[c], L = chunk_len[c];
    if (g < 0 || L <= 0 || g < end) return FM_ERR_INVALID;
    end = static_cast<long long>(g) + L;
    if (off + L > (1LL << 30)) return FM_ERR_INVALID;
    cm.start[c] = g;
    cm.len[c] = L;
    cm.offset[c] = static_cast<int>(off);
    off += L;
  }
  if (launch_localize(bounds, local_bounds, n, cm, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return FM_ERR_CUDA;
  return FM_OK;
}

fm_status fm_device_status(const void* ws, void* stream) {
  if (!ws) return FM_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int word = 0;
  if (cudaMemcpyAsync(&word, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FM_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FM_ERR_CUDA;
  if (word & DEV_LAYOUT) return FM_ERR_CUDA;
  if (word & DEV_TIMEOUT) return FM_ERR_TIMEOUT;
  if (word & DEV_BOUNDS) return FM_ERR_BOUNDS;
  return FM_OK;
}

fm_status fm_test_hooks(uint64_t wait_limit_ns, int withhold_release) {
  if (withhold_release < 0 || withhold_release > 3) return FM_ERR_INVALID;
  g_hooks.wait_ns = wait_limit_ns ? wait_limit_ns : FM_WAIT_LIMIT_NS;
  g_hooks.withhold = withhold_release;
  return FM_OK;
}

const char* fm_status_string(fm_status s) {
  switch (s) {
    case FM_OK: return "ok";
    case FM_ERR_INVALID: return "invalid argument";
    case FM_ERR_BOUNDS: return "bound value outside [0, Sq]";
    case FM_ERR_UNSUPPORTED: return "unsupported configuration";
    case FM_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case FM_ERR_CUDA: return "CUDA runtime error";
    case FM_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int fm_version(void) { return 100; }

}  // extern "C"
