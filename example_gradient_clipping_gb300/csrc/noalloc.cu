// dp_layer_sqnorms_noalloc: per-example norms for callers that cannot allocate.
//
// The ghost and instantiated norm kernels write per-tile partial sums to scratch
// memory before reducing them per example.  dp_layer_sqnorms takes that scratch
// from a caller-provided workspace; this entry point instead uses one array that
// the library owns, declared below at file scope, so the caller passes only its
// inputs and outputs.
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace {

// 4 MiB of fp32 partials.  Every GPU that loads the library holds this array until
// the process exits.
constexpr size_t kScratchFloats = (size_t)1 << 20;
static __device__ __align__(256) float g_norm_scratch[kScratchFloats];

// Device address of g_norm_scratch on the current device.  In host code the name
// g_norm_scratch is only a host-side stand-in for the symbol, never a device
// address, so it must not be passed to a kernel; the address is looked up once per
// device with that device current, and cached.
float* scratch_on_current_device(dp_status* st) {
  static std::mutex mu;
  static float* cache[64] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    *st = dph::set_error(DP_ERR_CUDA, "dp_layer_sqnorms_noalloc: no current CUDA device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_norm_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      snprintf(msg, sizeof(msg), "dp_layer_sqnorms_noalloc: cudaGetSymbolAddress failed: %s",
               cudaGetErrorString(e));
      *st = dph::set_error(DP_ERR_CUDA, msg);
      return nullptr;
    }
    cache[dev] = static_cast<float*>(p);
  }
  return cache[dev];
}

}  // namespace

extern "C" dp_status dp_layer_sqnorms_noalloc(const dp_layer_desc* desc, const void* A,
                                              const void* G, int mode, float* sqnorm_out,
                                              int* chosen_mode_out, cudaStream_t stream) {
  int chosen = 0;
  dp_status st = dp_plan(desc, mode, &chosen, nullptr, nullptr);
  if (st != DP_OK) return st;
  if (!A || !G || !sqnorm_out)
    return dph::set_error(DP_ERR_INVALID_ARG, "A, G and sqnorm_out must be non-NULL");
  dpk::Geom g;
  st = dph::geom_from_desc(desc, &g);
  if (st != DP_OK) return st;
  cudaError_t e = cudaSuccess;
  if (chosen == DP_NORM_T1) {
    e = dph::launch_t1_norm(g, desc->dtype, A, G, sqnorm_out, stream);   // needs no scratch
  } else {
    const size_t need = chosen == DP_NORM_GHOST ? dph::simt_ghost_ws_floats(g)
                                                : dph::simt_inst_ws_floats(g);
    if (need > kScratchFloats) {
      char msg[256];
      snprintf(msg, sizeof(msg),
               "dp_layer_sqnorms_noalloc: this layer needs %zu bytes of scratch, above the %zu-byte "
               "static maximum; use dp_layer_sqnorms with a workspace",
               need * sizeof(float), kScratchFloats * sizeof(float));
      return dph::set_error(DP_ERR_UNSUPPORTED, msg);
    }
    float* scratch = scratch_on_current_device(&st);
    if (!scratch) return st;
    // Every partial the reduction reads is written earlier in the same call, so the
    // previous call's contents need no clearing.
    e = chosen == DP_NORM_GHOST
            ? dph::launch_simt_ghost(g, desc->dtype, A, G, sqnorm_out, scratch, stream)
            : dph::launch_simt_inst(g, desc->dtype, A, G, sqnorm_out, scratch, stream);
  }
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "dp_layer_sqnorms_noalloc launch: %s", cudaGetErrorString(e));
    return dph::set_error(DP_ERR_CUDA, msg);
  }
  if (chosen_mode_out) *chosen_mode_out = chosen;
  return DP_OK;
}
