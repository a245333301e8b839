// fm_fwd_static: the forward pass for callers that cannot hand the library a
// workspace.  Some callers cannot allocate device memory at the moment they
// need attention: a host framework may own every byte of device memory
// through its own caching allocator or fixed arena and give a plugin no way
// to ask for more, and a latency-critical path may forbid calls that can
// block or synchronise the device, as cudaMalloc/cudaFree can.  This entry
// point therefore keeps its scratch (status word, block summary, tile table,
// work lists, unit order) in a fixed array in device memory that is part of
// the library image: each GPU that loads the library holds those
// FM_STATIC_SCRATCH_BYTES until the process exits.
//
// The array is shared by every call on a device and keeps the previous
// call's contents; the status word is cleared at the start of each call and
// every other region is rewritten before it is read.  Two calls whose work
// overlaps on the GPU (different streams, or different host threads) race on
// the array and produce undefined outputs.
#include <mutex>

#include "fm_internal.h"

namespace fm {

static __device__ __align__(256) char g_static_scratch[FM_STATIC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
char* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the array on the current device.  On the host the name
// g_static_scratch is only a stand-in for the symbol, never a usable pointer.
fm_status scratch_for_current_device(char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return FM_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<char*>(p);
  }
  *out = g_scratch_ptr[dev];
  return FM_OK;
}
}  // namespace

}  // namespace fm

using namespace fm;

extern "C" fm_status fm_fwd_static(const fm_desc* desc, const void* q, const void* k,
                                   const void* v, const int32_t* lts, const int32_t* lte,
                                   const int32_t* uts, const int32_t* ute, float scale, void* o,
                                   float* lse, void* stream) {
  Plan p;
  fm_status st = make_plan(desc, 0, &p, FM_STATIC_SCRATCH_BYTES);
  if (st != FM_OK) return st;
  if (p.L.total > FM_STATIC_SCRATCH_BYTES) return FM_ERR_WORKSPACE;
  auto a16 = [](const void* x) { return x && (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
  if (!a16(q) || !a16(k) || !a16(v) || !a16(o) || !lse) return FM_ERR_INVALID;
  if (!lts || !lte || !uts || !ute) return FM_ERR_INVALID;
  char* ws = nullptr;
  if ((st = scratch_for_current_device(&ws)) != FM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws + p.L.status, 0, 32, s) != cudaSuccess) return FM_ERR_CUDA;
  if (launch_summary(p, lts, lte, uts, ute, ws, s) != cudaSuccess) return FM_ERR_CUDA;
  if (launch_classify(p, ws, 0, s) != cudaSuccess) return FM_ERR_CUDA;
  if (launch_tile_masks(p, lts, lte, uts, ute, ws, s) != cudaSuccess) return FM_ERR_CUDA;
  if (launch_orders(p, ws, 1u << ORDER_PAIRS, s) != cudaSuccess) return FM_ERR_CUDA;
  TensorArgs t{};
  t.q = q; t.k = k; t.v = v; t.o_out = o; t.lse_out = lse;
  t.bounds[0] = lts; t.bounds[1] = lte; t.bounds[2] = uts; t.bounds[3] = ute;
  t.scale = scale;
  return launch_fwd(p, *desc, t, ws, s);
}
