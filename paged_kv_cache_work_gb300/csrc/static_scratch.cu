// pa_decode_step_static: a whole decode step on scratch that lives in a file-scope device
// array, for callers that cannot allocate device memory (see include/pa.h).
//
// The array's name is only a host-side stand-in in host code; its device address comes
// from cudaGetSymbolAddress, looked up once per device with that device current and cached.
// The three stages reuse the public entry points unchanged, so the kernels and their
// results are exactly those of pa_plan + pa_decode + pa_reduce.  The planner writes every
// word of the scratch the later stages read (header, flags, work list, unit table), so
// nothing needs clearing between calls.
#include <mutex>

#include "pa_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[PA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

pa_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return PA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_step_static(const pa_config* cfg, const void* q,
                                           const void* k_cache, const void* v_cache,
                                           const float* k_scale, const float* v_scale,
                                           const int32_t* block_tables,
                                           const int32_t* context_lens, const int32_t* q_lens,
                                           void* out, float* lse, pa_stream stream) {
  size_t need = 0;
  pa_status st = pa_workspace_size(cfg, &need);
  if (st != PA_OK) return st;
  if (need > PA_STATIC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
  void* ws = nullptr;
  if ((st = scratch_on_current_device(&ws)) != PA_OK) return st;
  const size_t cap = PA_STATIC_SCRATCH_BYTES;
  if ((st = pa_plan(cfg, block_tables, context_lens, q_lens, ws, cap, stream)) != PA_OK) return st;
  if ((st = pa_decode(cfg, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                      q_lens, out, lse, ws, cap, stream)) != PA_OK)
    return st;
  return pa_reduce(cfg, out, lse, ws, cap, stream);
}
