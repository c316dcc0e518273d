// Causal Conv3d on the CUDA cores: the fp32 storage mode and channel counts the tensor-core
// kernel's 64-channel K blocks do not take (tiny decoders, C_in % 64 != 0).
//
// Same arithmetic as the tensor-core path (DistVAE PR #14 "Add tiled VAE parallelism & extended
// model support", PatchConv3d padding commit): y[b,t,h,w,co] = bias[co] + sum over the 27 taps and
// C_in of W * x[b, max(t-2+kt,0) (or the cached frames), h-1+kh, w-1+kw, ci], zero outside the
// image, fp32 accumulation in a fixed (tap, channel) order; then residual and depth-to-space.
// Blocks own 8 x 16 pixel tiles of one patch (tiles never cross a patch edge) and 8 output
// channels per thread; halo taps read the neighbour patch's rows in place.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace vae {

struct SimtParams {
  int B, T, H, W, C_in, C_out, T_in, x_T_alloc, cache_frames, res_T_alloc, y_T_alloc;
  int nph, npw, n_trows, n_tcols;
  int trow_prefix[kMaxP + 1], tcol_prefix[kMaxP + 1];
  int ph_edges[kMaxP + 1], pw_edges[kMaxP + 1];
  const void* x;
  int x_f32;
  const float* w;
  const float* bias;
  const void* residual;
  int res_f32;
  void* y;
  int out_f32, out_ncthw;
  int d2s_t, d2s_h, d2s_w, drop, S, C_d2s, T_out, H_out, W_out;
};

namespace {
constexpr int kRows = 8, kCols = 16, kCo = 8;

__device__ int band_of(const int* prefix, int n, int idx) {
  int i = 0;
  while (i + 1 < n && prefix[i + 1] <= idx) ++i;
  return i;
}
}  // namespace

__global__ void __launch_bounds__(128) conv_simt_kernel(const __grid_constant__ SimtParams p) {
  const int per_frame = p.n_trows * p.n_tcols;
  const int frame = blockIdx.x / per_frame;
  const int r = blockIdx.x % per_frame;
  const int tr = r / p.n_tcols, tc = r % p.n_tcols;
  const int pi = band_of(p.trow_prefix, p.nph, tr), pj = band_of(p.tcol_prefix, p.npw, tc);
  const int h = p.ph_edges[pi] + (tr - p.trow_prefix[pi]) * kRows + threadIdx.x / kCols;
  const int w = p.pw_edges[pj] + (tc - p.tcol_prefix[pj]) * kCols + threadIdx.x % kCols;
  const int b = frame / p.T, t = frame % p.T;
  const int co0 = blockIdx.y * kCo;
  if (h >= p.ph_edges[pi + 1] || w >= p.pw_edges[pj + 1]) return;

  float acc[kCo];
#pragma unroll
  for (int i = 0; i < kCo; ++i) acc[i] = 0.f;
  const int nco = min(kCo, p.C_out - co0);
  for (int kt = 0; kt < 3; ++kt) {
    const int ti = max(t + kt - 2 + p.cache_frames, 0);
    for (int kh = 0; kh < 3; ++kh) {
      const int hi = h + kh - 1;
      for (int kw = 0; kw < 3; ++kw) {
        const int wi = w + kw - 1;
        const float* wt = p.w + (static_cast<int64_t>((kt * 3 + kh) * 3 + kw) * p.C_in) * p.C_out + co0;
        const bool inside = hi >= 0 && hi < p.H && wi >= 0 && wi < p.W;
        const int64_t xoff = (((static_cast<int64_t>(b) * p.x_T_alloc + ti) * p.H + hi) * p.W + wi) * p.C_in;
        for (int ci = 0; ci < p.C_in; ++ci) {
          float xv = 0.f;
          if (inside)
            xv = p.x_f32 ? static_cast<const float*>(p.x)[xoff + ci]
                         : bf2f(static_cast<const __nv_bfloat16*>(p.x)[xoff + ci]);
          const float* wr = wt + static_cast<int64_t>(ci) * p.C_out;
#pragma unroll
          for (int i = 0; i < kCo; ++i)
            if (i < nco) acc[i] = fmaf(wr[i], xv, acc[i]);
        }
      }
    }
  }
  const int sh = p.d2s_h, sw = p.d2s_w;
  for (int i = 0; i < nco; ++i) {
    const int n = co0 + i;  // PyTorch channel order: c * S + sub
    const int c = n / p.S, sub = n - (n / p.S) * p.S;
    float v = acc[i] + (p.bias ? p.bias[n] : 0.f);
    if (p.residual) {
      const int64_t ridx = (((static_cast<int64_t>(b) * p.res_T_alloc + t) * p.H + h) * p.W + w) * p.C_out + n;
      v += p.res_f32 ? static_cast<const float*>(p.residual)[ridx]
                     : bf2f(static_cast<const __nv_bfloat16*>(p.residual)[ridx]);
    }
    const int dt = sub / (sh * sw), rem = sub - (sub / (sh * sw)) * sh * sw;
    const int dy = rem / sw, dx = rem - (rem / sw) * sw;
    const int to = p.d2s_t * t + dt - p.drop;
    if (to < 0) continue;
    const int ho = h * sh + dy, wo = w * sw + dx;
    int64_t oidx;
    if (p.out_ncthw)
      oidx = (((static_cast<int64_t>(b) * p.C_d2s + c) * p.y_T_alloc + to) * p.H_out + ho) * p.W_out + wo;
    else
      oidx = (((static_cast<int64_t>(b) * p.y_T_alloc + to) * p.H_out + ho) * p.W_out + wo) * p.C_d2s + c;
    if (p.out_f32) static_cast<float*>(p.y)[oidx] = v;
    else static_cast<__nv_bfloat16*>(p.y)[oidx] = f2bf(v);
  }
}

cudaError_t launch_conv_simt(const ConvSimtArgs& a, cudaStream_t s) {
  SimtParams p{};  // per call (launches from several host threads never share it)
  p.B = a.B; p.T = a.T; p.H = a.H; p.W = a.W; p.C_in = a.C_in; p.C_out = a.C_out;
  p.T_in = a.T_in; p.cache_frames = a.cache_frames;
  p.x_T_alloc = a.x_T_alloc ? a.x_T_alloc : a.T_in;
  if (a.nph > kMaxP || a.npw > kMaxP) return cudaErrorInvalidValue;
  p.nph = a.nph; p.npw = a.npw;
  for (int i = 0; i <= a.nph; ++i) p.ph_edges[i] = a.ph_edges[i];
  for (int j = 0; j <= a.npw; ++j) p.pw_edges[j] = a.pw_edges[j];
  p.trow_prefix[0] = p.tcol_prefix[0] = 0;
  for (int i = 0; i < a.nph; ++i)
    p.trow_prefix[i + 1] = p.trow_prefix[i] + (a.ph_edges[i + 1] - a.ph_edges[i] + kRows - 1) / kRows;
  for (int j = 0; j < a.npw; ++j)
    p.tcol_prefix[j + 1] = p.tcol_prefix[j] + (a.pw_edges[j + 1] - a.pw_edges[j] + kCols - 1) / kCols;
  p.n_trows = p.trow_prefix[a.nph];
  p.n_tcols = p.tcol_prefix[a.npw];
  p.x = a.x; p.x_f32 = a.x_f32; p.w = a.w; p.bias = a.bias;
  p.residual = a.residual; p.res_f32 = a.res_f32;
  p.y = a.y; p.out_f32 = a.out_f32; p.out_ncthw = a.out_ncthw;
  p.d2s_t = a.d2s_t; p.d2s_h = a.d2s_h; p.d2s_w = a.d2s_w;
  p.S = a.d2s_t * a.d2s_h * a.d2s_w;
  p.C_d2s = a.C_out / p.S;
  p.drop = a.drop_first ? a.d2s_t - 1 : 0;
  p.T_out = a.d2s_t * a.T - p.drop;
  p.H_out = a.H * a.d2s_h;
  p.W_out = a.W * a.d2s_w;
  p.res_T_alloc = a.res_T_alloc ? a.res_T_alloc : a.T;
  p.y_T_alloc = a.y_T_alloc ? a.y_T_alloc : p.T_out;
  if (a.residual && p.S != 1) return cudaErrorInvalidValue;
  const long long gx = static_cast<long long>(a.B) * a.T * p.n_trows * p.n_tcols;
  if (gx <= 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(gx), (a.C_out + kCo - 1) / kCo);
  conv_simt_kernel<<<grid, 128, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace vae
