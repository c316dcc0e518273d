// PatchGroupNorm + SiLU for callers that cannot allocate device memory.
//
// Some hosts own every byte of device memory through their own pool and hand a plugin nothing but
// its input and output buffers (no workspace argument, and a cudaMalloc from the plugin would either
// fail against the pool's reservation or synchronise the whole device in the middle of a pipeline).
// For them this file keeps the group-norm scratch (per-patch partial sums and the per-frame affine) in
// a fixed device array that is part of the library image: every GPU that loads the library holds it
// until the process exits, and no call here allocates anything.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "internal.h"

namespace vae {
namespace {

static __device__ __align__(256) unsigned char g_gn_scratch[VAE_GN_NOALLOC_SCRATCH_BYTES];

// Device address of g_gn_scratch on the current device.  The name is a host-side stand-in in host
// code; the address comes from cudaGetSymbolAddress, once per device, with that device current.
void* scratch_address(cudaError_t* err) {
  static void* addr[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_gn_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace
}  // namespace vae

using namespace vae;

extern "C" vae_status_t vae_patch_groupnorm_silu_noalloc(const void* x, const float* gamma, const float* beta, void* y,
                                                         const vae_gn_desc_t* d, void* stream) {
  if (!x || !gamma || !beta || !y || !d) return op_error(VAE_ERR_INVALID_ARG, "null argument");
  vae_status_t st = validate_gn_desc(x, y, d);
  if (st) return st;
  const size_t need = gn_workspace_bytes(d->n_patch_h, d->n_patch_w, d->B, d->T, d->groups, d->C);
  if (need > VAE_GN_NOALLOC_SCRATCH_BYTES) {
    char msg[160];
    snprintf(msg, sizeof(msg), "needs %zu bytes of group-norm scratch; the fixed array holds %d bytes", need,
             VAE_GN_NOALLOC_SCRATCH_BYTES);
    return op_error(VAE_ERR_UNSUPPORTED, msg);
  }
  cudaError_t e = cudaSuccess;
  void* scratch = scratch_address(&e);
  if (!scratch) return op_error(VAE_ERR_CUDA, cudaGetErrorString(e));
  GnArgs g{};
  g.B = d->B; g.T = d->T; g.H = d->H; g.W = d->W; g.C = d->C; g.groups = d->groups; g.eps = d->eps; g.silu = d->silu;
  g.nph = d->n_patch_h; g.npw = d->n_patch_w; g.ph_edges = d->patch_h_edges; g.pw_edges = d->patch_w_edges;
  g.x = x; g.x_f32 = d->in_dtype == VAE_FP32; g.y = y; g.y_f32 = d->out_dtype == VAE_FP32;
  g.y_fp8 = d->out_dtype == VAE_FP8;
  g.gamma = gamma; g.beta = beta; g.partials = scratch;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // launch_gn_stats clears the partial sums (they must start at zero) before it adds into them; the
  // affine region is fully rewritten by the finalize step.
  e = launch_gn_stats(g, s);
  if (e == cudaSuccess) e = launch_gn_apply(g, s);
  if (e != cudaSuccess) return op_error(VAE_ERR_CUDA, cudaGetErrorString(e));
  return VAE_OK;
}
