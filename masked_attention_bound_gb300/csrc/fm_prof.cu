// Timing hooks: CUDA events around each kernel launch while enabled.
#include <vector>

#include "fm_internal.h"
#include "fm_ptx.cuh"

namespace fm {

namespace {
struct Rec {
  int id;
  cudaEvent_t a, b;
};
constexpr int kMaxRecs = 65536;
bool g_on = false;
std::vector<cudaEvent_t> g_pool;  // events reused across reads
size_t g_pool_used = 0;
std::vector<Rec> g_recs;
int g_counts[K_COUNT] = {0};
int g_open = -1;  // index of the record waiting for its end event

cudaEvent_t take_event() {
  if (g_pool_used == g_pool.size()) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_pool.push_back(e);
  }
  return g_pool[g_pool_used++];
}
}  // namespace

void prof_begin(int id, cudaStream_t s) {
  g_open = -1;
  if (!g_on) return;
  g_counts[id] += 1;
  if (static_cast<int>(g_recs.size()) >= kMaxRecs) return;
  cudaEvent_t a = take_event(), b = take_event();
  if (!a || !b) return;
  cudaEventRecord(a, s);
  g_recs.push_back({id, a, b});
  g_open = static_cast<int>(g_recs.size()) - 1;
}

void prof_end(int id, cudaStream_t s) {
  if (!g_on || g_open < 0 || g_recs[g_open].id != id) return;
  cudaEventRecord(g_recs[g_open].b, s);
  g_open = -1;
}

// exp2 throughput: every thread runs eight independent chains of
// ex2.approx (the instruction the attention kernels use for P), so the
// MUFU, not the chains' latency, bounds the rate.
__global__ void __launch_bounds__(1024) ex2_rate_kernel(int iters, float* sink) {
  float x[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) x[j] = -1e-3f * static_cast<float>(threadIdx.x + j);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = ex2(x[j]) - 1.0f;
  }
  float t = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) t += x[j];
  if (t == 12345.0f) sink[blockIdx.x] = t;  // never true; keeps the chains live
}

}  // namespace fm

using namespace fm;

extern "C" {

fm_status fm_measure_exp2_rate(double* per_second, void* stream) {
  if (!per_second) return FM_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int blocks = num_sms(), threads = 1024, iters = 4096;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return FM_ERR_CUDA;
  fm_status st = FM_OK;
  ex2_rate_kernel<<<blocks, threads, 0, s>>>(iters / 8, nullptr);  // warm-up
  cudaEventRecord(e0, s);
  ex2_rate_kernel<<<blocks, threads, 0, s>>>(iters, nullptr);
  cudaEventRecord(e1, s);
  float ms = 0.f;
  if (cudaGetLastError() != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
      cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess || ms <= 0.f)
    st = FM_ERR_CUDA;
  else
    *per_second = static_cast<double>(blocks) * threads * iters * 8.0 / (ms * 1e-3);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return st;
}

fm_status fm_profile_enable(int on) {
  g_on = on != 0;
  return FM_OK;
}

fm_status fm_profile_read(double* total_ms, int* launches, int n) {
  if (n < 0) return FM_ERR_INVALID;
  double ms[K_COUNT] = {0};
  fm_status st = FM_OK;
  for (const Rec& r : g_recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) {
      st = FM_ERR_CUDA;
      continue;
    }
    ms[r.id] += t;
  }
  for (int i = 0; i < n && i < K_COUNT; ++i) {
    if (total_ms) total_ms[i] = ms[i];
    if (launches) launches[i] = g_counts[i];
  }
  for (int i = K_COUNT; i < n; ++i) {
    if (total_ms) total_ms[i] = 0;
    if (launches) launches[i] = 0;
  }
  g_recs.clear();
  g_pool_used = 0;
  g_open = -1;
  for (int i = 0; i < K_COUNT; ++i) g_counts[i] = 0;
  return st;
}

const char* fm_kernel_name(int id) {
  static const char* names[K_COUNT] = {"summary_kernel", "classify_kernel", "order_kernel",
                                       "localize_kernel", "fwd_kernel", "bwd_pre_kernel",
                                       "bwd_kv_kernel", "bwd_dq_kernel", "tile_mask_kernel",
                                       "quant_kernel", "fwd_fp8_kernel"};
  return (id >= 0 && id < K_COUNT) ? names[id] : "unknown";
}

}  // extern "C"
