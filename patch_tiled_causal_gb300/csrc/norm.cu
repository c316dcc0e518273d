// HBM-bound kernels: PatchGroupNorm (+ SiLU), tile blend, depth-to-space, layout changes,
// attention softmax, weight packing, and the watchdog self-test.
//
// PatchGroupNorm follows DistVAE PR #14 "Add tiled VAE parallelism & extended model support"
// (PatchGroupNorm commit: the exact global mean and the population variance, divide by the count;
// two-collective commit: per-patch counts and sums are merged before anything is normalised).
// Statistics are per (batch, frame, group).  Every element contributes q = round(x * 2^18) (|x| <
// 2^13, so q fits in 32 bits) to an int64 sum and q^2 to a 128-bit sum.  Integer addition is
// associative, so the totals are exact and identical whichever patch, block or warp adds which
// element: the normalised output does not change by one bit with the patch grid.  Each patch owns
// its own partial-sum slots; the merge adds them in patch order, then forms mean = S1 / (N 2^18) and
// var = S2 / (N 2^36) - mean^2 in fp64 (the exact totals carry the cancellation a float
// E[x^2] - E[x]^2 would suffer, so the two passes of the pages' estimator fold into one read).
//
// The tile blend follows TensorRT-LLM PR #15753 "LTX-2 tile-parallel VAE decode" (Approach: a
// per-tile mask built on the device from 1-D parts, weighted sum over the weight sum); here each
// output pixel gathers the tiles that cover it, in tile order, so the result is written once.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace vae {

// ============================================================================ group norm
struct GnPartial {
  unsigned long long s1;   // int64 sum of q (two's complement)
  unsigned long long s2a;  // sum of q^2 = s2a + s2b * 2^32: s2a sums the low 32 bits of each
  unsigned long long s2b;  // contribution and s2b the rest, so updates need no carry (plain atomics)
  unsigned long long pad;
};
static_assert(sizeof(GnPartial) == 32, "GnPartial layout is shared with the conv epilogue");

size_t gn_partials_bytes(int nph, int npw, int B, int T, int groups) {
  return static_cast<size_t>(nph) * npw * B * T * groups * sizeof(GnPartial);
}

size_t gn_workspace_bytes(int nph, int npw, int B, int T, int groups, int C) {
  const size_t parts = (gn_partials_bytes(nph, npw, B, T, groups) + 255) & ~size_t(255);
  return parts + static_cast<size_t>(B) * T * C * sizeof(float2);
}

struct GnParams {
  int B, T, H, W, C, groups, cpg;
  float eps;
  int silu;
  int nph, npw;
  int ph_edges[kMaxP + 1], pw_edges[kMaxP + 1];
  const void* x;
  int x_f32, x_T_alloc;
  void* y;
  int y_f32, y_T_alloc;
  const float* gamma;
  const float* beta;
  GnPartial* parts;
  float2* affine;  // [B*T, C] per-channel (scale, shift), after the partials in the workspace
  uint32_t* fault;
  int vec_per_px;   // C / 8
  int px_per_iter;  // blockDim / vec_per_px
  int rows_per_block, n_chunks;  // statistics: rows of one patch band per block, blocks per band
};

namespace {

VAE_DEV void add128(unsigned long long& lo, unsigned long long& hi, unsigned long long a_lo, unsigned long long a_hi) {
  const unsigned long long n = lo + a_lo;
  hi += a_hi + (n < lo ? 1ull : 0ull);
  lo = n;
}

// max(a, |x|) that is NaN when x is NaN (so a range test on the result also catches NaN)
VAE_DEV float max_abs_nan(float a, float x) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(fabsf(x)));
  return r;
}

// q = round(x * 2^18) for |x| < 16 (|q| < 2^22): adding 1.5 * 2^23 rounds x * 2^18 to the nearest
// integer (ties to even, as the float-to-int conversion below) and leaves it in the low mantissa bits.
VAE_DEV int quantize_small(float x) { return __float_as_int(fmaf(x, 262144.f, 12582912.f)) - 0x4B400000; }

VAE_DEV int quantize(float x, uint32_t* fault) {
  if (!(fabsf(x) < 8192.f)) {  // also catches NaN
    raise_fault(fault, FAULT_RANGE, 30);
    x = fminf(fmaxf(x, -8191.f), 8191.f);
    if (x != x) x = 0.f;
  }
  return __float2int_rn(x * 262144.f);  // exact scaling by 2^18
}

}  // namespace

// One block per (frame, patch, chunk of rows_per_block rows of the patch's band): everything a block
// reads lies in exactly one patch.  GPV = groups met by one 8-channel vector (1 when channels-per-
// group is a multiple of 8).
template <int GPV, typename T>
__global__ void __launch_bounds__(256) gn_stats_kernel(const __grid_constant__ GnParams p) {
  __shared__ unsigned long long sh_s1[1024], sh_lo[1024], sh_hi[1024];
  int rest = blockIdx.x;
  const int chunk = rest % p.n_chunks;
  rest /= p.n_chunks;
  const int j = rest % p.npw;
  rest /= p.npw;
  const int i = rest % p.nph;
  const int frame = rest / p.nph;
  const int fb = frame / p.T, ft = frame % p.T;
  const int h_beg = p.ph_edges[i] + chunk * p.rows_per_block;
  const int h_stop = min(p.ph_edges[i + 1], h_beg + p.rows_per_block);
  for (int g = threadIdx.x; g < p.groups; g += blockDim.x) sh_s1[g] = sh_lo[g] = sh_hi[g] = 0ull;
  __syncthreads();

  const int vid = threadIdx.x % p.vec_per_px;
  const int pxo = threadIdx.x / p.vec_per_px;
  const int c0 = vid * 8;
  const int w_beg = p.pw_edges[j], w_end = p.pw_edges[j + 1];
  long long s1[GPV];
  unsigned long long lo[GPV], hi[GPV];
#pragma unroll
  for (int k = 0; k < GPV; ++k) { s1[k] = 0; lo[k] = hi[k] = 0ull; }
  for (int h = h_beg; h < h_stop && threadIdx.x < p.vec_per_px * p.px_per_iter; ++h) {
    const T* xr = static_cast<const T*>(p.x) + ((static_cast<int64_t>(fb) * p.x_T_alloc + ft) * p.H + h) * p.W * p.C;
    // four pixels' vectors are loaded before any of them is summed (bytes in flight)
    for (int w = w_beg + pxo; w < w_end; w += 4 * p.px_per_iter) {
      float v[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int ww = w + u * p.px_per_iter;
        if (ww < w_end) load8(xr + static_cast<int64_t>(ww) * p.C + c0, v[u]);
        else {
#pragma unroll
          for (int e = 0; e < 8; ++e) v[u][e] = 0.f;
        }
      }
      float amax = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = max_abs_nan(amax, v[u][e]);
      if (amax < 16.f) {
        // every |q| < 2^22: 32-bit sums of q, q^2 summed in 64 bits (32 of them < 2^49)
#pragma unroll
        for (int k = 0; k < GPV; ++k) {
          int s1f = 0;
          unsigned long long sqf = 0;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
#pragma unroll
            for (int e = k * (8 / GPV); e < (k + 1) * (8 / GPV); ++e) {
              const int qv = quantize_small(v[u][e]);
              s1f += qv;
              sqf += static_cast<unsigned long long>(static_cast<long long>(qv) * qv);
            }
          }
          s1[k] += s1f;
          add128(lo[k], hi[k], sqf, 0ull);
        }
        continue;
      }
#pragma unroll
      for (int k = 0; k < GPV; ++k) {
        // q^2 < 2^62: four of them fit an unsigned 64-bit sum before the 128-bit carry
        unsigned long long sq4 = 0;
        int n4 = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
#pragma unroll
          for (int e = k * (8 / GPV); e < (k + 1) * (8 / GPV); ++e) {
            const int qv = quantize(v[u][e], p.fault);
            s1[k] += qv;
            sq4 += static_cast<unsigned long long>(static_cast<long long>(qv) * qv);
            if (++n4 == 4) {
              add128(lo[k], hi[k], sq4, 0ull);
              sq4 = 0;
              n4 = 0;
            }
          }
        }
        if (n4) add128(lo[k], hi[k], sq4, 0ull);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < GPV; ++k) {
    const int g = (GPV == 1) ? c0 / p.cpg : (c0 / p.cpg + k);
    if (s1[k] != 0 || lo[k] != 0 || hi[k] != 0) {  // plain adds: no returned values, no carries
      atomicAdd(&sh_s1[g], static_cast<unsigned long long>(s1[k]));
      atomicAdd(&sh_lo[g], lo[k] & 0xffffffffull);
      atomicAdd(&sh_hi[g], (lo[k] >> 32) | (hi[k] << 32));
    }
  }
  __syncthreads();
  const int patch = i * p.npw + j;
  const int b = fb, t = ft;
  for (int g = threadIdx.x; g < p.groups; g += blockDim.x) {
    GnPartial* d = p.parts + ((static_cast<int64_t>(patch) * p.B + b) * p.T + t) * p.groups + g;
    const unsigned long long a1 = sh_s1[g], a2 = sh_lo[g], b2 = sh_hi[g];
    if (a1 == 0 && a2 == 0 && b2 == 0) continue;
    atomicAdd(&d->s1, a1);
    atomicAdd(&d->s2a, a2);
    atomicAdd(&d->s2b, b2);
  }
}

// Merge the per-patch sums of one frame (patch order), then fold mean, rstd, gamma and beta into a
// per-channel affine y = x * a[c] + s[c]; one block per (batch, frame).
__global__ void __launch_bounds__(256) gn_finalize_kernel(const __grid_constant__ GnParams p) {
  __shared__ float sh_mean[1024], sh_rstd[1024];
  const int frame = blockIdx.x;
  const int b = frame / p.T, t = frame % p.T;
  const double n = static_cast<double>(p.cpg) * p.H * p.W;
  const int P = p.nph * p.npw;
  for (int g = threadIdx.x; g < p.groups; g += blockDim.x) {
    long long s1 = 0;
    unsigned long long lo = 0, hi = 0;
    for (int q = 0; q < P; ++q) {
      const GnPartial& d = p.parts[((static_cast<int64_t>(q) * p.B + b) * p.T + t) * p.groups + g];
      s1 += static_cast<long long>(d.s1);
      add128(lo, hi, d.s2a, 0ull);
      add128(lo, hi, d.s2b << 32, d.s2b >> 32);
    }
    const double mq = static_cast<double>(s1) / n;  // mean in units of 2^-18
    const double e2 = (static_cast<double>(hi) * 18446744073709551616.0 + static_cast<double>(lo)) / n;
    double var = (e2 - mq * mq) * (1.0 / 68719476736.0);  // / 2^36
    if (var < 0.0) var = 0.0;
    sh_mean[g] = static_cast<float>(mq * (1.0 / 262144.0));
    sh_rstd[g] = static_cast<float>(1.0 / sqrt(var + static_cast<double>(p.eps)));
  }
  __syncthreads();
  float2* aff = p.affine + static_cast<int64_t>(frame) * p.C;
  for (int c = threadIdx.x; c < p.C; c += blockDim.x) {
    const int g = c / p.cpg;
    const float a = sh_rstd[g] * p.gamma[c];
    aff[c] = make_float2(a, p.beta[c] - sh_mean[g] * a);
  }
}

// y = SiLU(x * a[c] + s[c]); grid (chunks of a frame, frames), 16-byte vectors.  Every thread
// issues all its loads (kept packed: 8 x 16 B of bf16 or 4 x 32 B of fp32) before any math, so that
// enough bytes are in flight to cover HBM latency at a register count that keeps 4 blocks per SM.
constexpr int kApplyBytesPerThread = 128;
template <typename TI> struct ApplyVec;
template <> struct ApplyVec<__nv_bfloat16> {
  static constexpr int kVecs = kApplyBytesPerThread / 16;
  uint4 raw;
  VAE_DEV void load(const __nv_bfloat16* p) { raw = *reinterpret_cast<const uint4*>(p); }
  VAE_DEV void get(float* v) const {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
};
template <> struct ApplyVec<float> {
  static constexpr int kVecs = kApplyBytesPerThread / 32;
  float4 a, b;
  VAE_DEV void load(const float* p) {
    a = reinterpret_cast<const float4*>(p)[0];
    b = reinterpret_cast<const float4*>(p)[1];
  }
  VAE_DEV void get(float* v) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

// SiLU z * sigmoid(z) in the output type's precision.  For e4m3 outputs (unit roundoff 2^-4) the sigmoid
// comes from one tanh.approx, sigmoid(z) = (1 + tanh(z / 2)) / 2 (relative error near 2^-11): one MUFU
// operation per element instead of two (exp and reciprocal), which a 3-byte-per-element e4m3 pass
// would otherwise saturate; every other output type keeps z / (1 + exp(-z)).
template <typename TO>
VAE_DEV float silu_to(float z) {
  if constexpr (sizeof(TO) == 1) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * z));
    return z * fmaf(0.5f, t, 0.5f);
  } else {
    return __fdividef(z, 1.0f + __expf(-z));
  }
}

// bf16 input keeps twice the vectors in flight per thread: 3 blocks per SM leave it room (measured:
// 0.201 -> 0.186 ms on [1,512,21,88,160]); fp32 input runs best at 4 (the decoders' case).
template <typename TI, typename TO>
__global__ void __launch_bounds__(256, sizeof(TI) == 2 ? 3 : 4) gn_apply_kernel(const __grid_constant__ GnParams p) {
  constexpr int VPT = ApplyVec<TI>::kVecs;
  extern __shared__ float2 sh_aff[];
  const int frame = blockIdx.y;
  const int b = frame / p.T, t = frame % p.T;
  const float2* aff = p.affine + static_cast<int64_t>(frame) * p.C;
  const int64_t fe = static_cast<int64_t>(p.H) * p.W * p.C;  // elements of one frame
  const TI* xf = static_cast<const TI*>(p.x) + (static_cast<int64_t>(b) * p.x_T_alloc + t) * fe;
  TO* yf = static_cast<TO*>(p.y) + (static_cast<int64_t>(b) * p.y_T_alloc + t) * fe;
  const int nvec = static_cast<int>(fe / 8);  // < 2^31 per frame (checked on the host)
  const int cvec = p.C / 8;
  const int v0 = blockIdx.x * blockDim.x * VPT + threadIdx.x;
  ApplyVec<TI> in[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = v0 + k * blockDim.x;
    if (v < nvec) in[k].load(xf + static_cast<int64_t>(v) * 8);
  }
  if (blockDim.x % cvec == 0) {
    // every vector of this thread covers the same 8 channels: their affine lives in registers
    const int c0 = (v0 % cvec) * 8;
    float2 m[8];
    const float4* a4 = reinterpret_cast<const float4*>(aff + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 q = __ldg(a4 + i);
      m[2 * i] = make_float2(q.x, q.y);
      m[2 * i + 1] = make_float2(q.z, q.w);
    }
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = v0 + k * blockDim.x;
      if (v >= nvec) break;
      float a[8];
      in[k].get(a);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float z = fmaf(a[e], m[e].x, m[e].y);
        a[e] = p.silu ? silu_to<TO>(z) : z;
      }
      vstore8(yf + static_cast<int64_t>(v) * 8, a, p.fault);
    }
    return;
  }
  for (int c = threadIdx.x; c < p.C; c += blockDim.x) sh_aff[c] = aff[c];
  __syncthreads();
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = v0 + k * blockDim.x;
    if (v >= nvec) break;
    const int c0 = ((cvec & (cvec - 1)) == 0 ? (v & (cvec - 1)) : (v % cvec)) * 8;
    float a[8];
    in[k].get(a);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float2 m = sh_aff[c0 + e];
      const float z = fmaf(a[e], m.x, m.y);
      a[e] = p.silu ? silu_to<TO>(z) : z;
    }
    vstore8(yf + static_cast<int64_t>(v) * 8, a, p.fault);
  }
}

namespace {
bool fill_gn(GnParams& p, const GnArgs& a) {
  p = GnParams{};
  p.B = a.B; p.T = a.T; p.H = a.H; p.W = a.W; p.C = a.C; p.groups = a.groups;
  if (a.groups <= 0 || a.groups > 1024 || a.C % a.groups) return false;
  p.cpg = a.C / a.groups;
  if (a.C % 8 || a.C > 6144 || !(p.cpg % 8 == 0 || 8 % p.cpg == 0)) return false;
  if (a.nph > kMaxP || a.npw > kMaxP) return false;
  p.eps = a.eps; p.silu = a.silu;
  p.nph = a.nph; p.npw = a.npw;
  for (int i = 0; i <= a.nph; ++i) p.ph_edges[i] = a.ph_edges[i];
  for (int j = 0; j <= a.npw; ++j) p.pw_edges[j] = a.pw_edges[j];
  p.x = a.x; p.x_f32 = a.x_f32; p.y = a.y; p.y_f32 = a.y_f32;
  p.x_T_alloc = a.x_T_alloc ? a.x_T_alloc : a.T;
  p.y_T_alloc = a.y_T_alloc ? a.y_T_alloc : a.T;
  p.gamma = a.gamma; p.beta = a.beta;
  p.parts = static_cast<GnPartial*>(a.partials);
  p.affine = reinterpret_cast<float2*>(static_cast<char*>(a.partials) +
                                       ((gn_partials_bytes(a.nph, a.npw, a.B, a.T, a.groups) + 255) & ~size_t(255)));
  p.fault = fault_word();
  p.vec_per_px = a.C / 8;
  p.px_per_iter = std::max(1, 256 / p.vec_per_px);
  return true;
}
}  // namespace

cudaError_t launch_gn_stats(const GnArgs& a, cudaStream_t s) {
  GnParams p;  // per call (several host threads may launch)
  if (!fill_gn(p, a)) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(a.partials, 0, gn_partials_bytes(a.nph, a.npw, a.B, a.T, a.groups), s);
  if (e != cudaSuccess) return e;
  int band_max = 1, pw_max = 1;
  for (int i = 0; i < a.nph; ++i) band_max = std::max(band_max, a.ph_edges[i + 1] - a.ph_edges[i]);
  for (int j = 0; j < a.npw; ++j) pw_max = std::max(pw_max, a.pw_edges[j + 1] - a.pw_edges[j]);
  p.rows_per_block = std::max(1, static_cast<int>(65536 / (static_cast<int64_t>(pw_max) * a.C)));
  p.n_chunks = (band_max + p.rows_per_block - 1) / p.rows_per_block;
  const long long nb = static_cast<long long>(a.B) * a.T * a.nph * a.npw * p.n_chunks;
  if (nb == 0) return cudaSuccess;
  const int threads = std::max(p.vec_per_px * p.px_per_iter, 32);
  if (threads > 1024) return cudaErrorInvalidValue;
  const int gpv = p.cpg >= 8 ? 1 : 8 / p.cpg;
  dim3 grid(static_cast<unsigned>(nb));
#define VAE_GN_STATS(G)                                                                   \
  if (a.x_f32) gn_stats_kernel<G, float><<<grid, threads, 0, s>>>(p);                     \
  else gn_stats_kernel<G, __nv_bfloat16><<<grid, threads, 0, s>>>(p);
  switch (gpv) {
    case 1: VAE_GN_STATS(1) break;
    case 2: VAE_GN_STATS(2) break;
    case 4: VAE_GN_STATS(4) break;
    default: VAE_GN_STATS(8) break;
  }
#undef VAE_GN_STATS
  return cudaGetLastError();
}

cudaError_t launch_gn_apply(const GnArgs& a, cudaStream_t s) {
  GnParams p;  // per call (several host threads may launch)
  if (!fill_gn(p, a)) return cudaErrorInvalidValue;
  const long long frames = static_cast<long long>(a.B) * a.T;
  if (frames == 0) return cudaSuccess;
  if (frames > 65535 || static_cast<int64_t>(a.H) * a.W * a.C / 8 > 0x7fffffffLL) return cudaErrorInvalidValue;
  gn_finalize_kernel<<<static_cast<unsigned>(frames), 256, 0, s>>>(p);
  const int64_t nvec = static_cast<int64_t>(a.H) * a.W * a.C / 8;
  const int64_t per_block = 256LL * (a.x_f32 ? ApplyVec<float>::kVecs : ApplyVec<__nv_bfloat16>::kVecs);
  dim3 grid(static_cast<unsigned>((nvec + per_block - 1) / per_block), static_cast<unsigned>(frames));
  const size_t sm = static_cast<size_t>(a.C) * sizeof(float2);
  if (a.y_fp8 && a.x_f32) gn_apply_kernel<float, __nv_fp8_e4m3><<<grid, 256, sm, s>>>(p);
  else if (a.y_fp8) gn_apply_kernel<__nv_bfloat16, __nv_fp8_e4m3><<<grid, 256, sm, s>>>(p);
  else if (a.x_f32 && a.y_f32) gn_apply_kernel<float, float><<<grid, 256, sm, s>>>(p);
  else if (a.x_f32) gn_apply_kernel<float, __nv_bfloat16><<<grid, 256, sm, s>>>(p);
  else if (a.y_f32) gn_apply_kernel<__nv_bfloat16, float><<<grid, 256, sm, s>>>(p);
  else gn_apply_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, 256, sm, s>>>(p);
  return cudaGetLastError();
}

// ============================================================================ channel RMS norm
// Per pixel r = 1 / sqrt(mean_c x^2 + eps), y = x * r * gamma[c] + beta[c] (then SiLU): the norm of
// the Wan / Qwen-Image, HunyuanVideo 1.5 and LTX-2 decoders, which reduces over channels only and so
// needs nothing from other patches.  A team of L = min(32, C/8) lanes (a power of two) owns a pixel:
// lane j of the team takes the 8-channel vectors j, j + L, ..., sums their squares in that order and
// the team adds its lanes by xor shuffles, so a pixel's result never depends on the patch grid or on
// which block runs it.  All lanes of a warp run every loop step (pixels past the end are masked), so
// the shuffles always see the full warp.
struct RmsParams {
  int B, T, H, W, C;
  float eps;
  int silu;
  const void* x;
  int x_T_alloc;
  void* y;
  int y_T_alloc;
  const float* gamma;
  const float* beta;
  int team, vpl;  // lanes per pixel, 8-channel vectors per lane
  uint32_t* fault;
};
constexpr int kRmsMaxVpl = 4;
constexpr int kRmsVecs = 4;  // 8-channel vectors a lane holds per step: kRmsVecs / VPL pixels per team

// Raw 8-element loads, converted only when used (so several can be in flight per thread).
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
  uint4 r;
  VAE_DEV void load(const __nv_bfloat16* p) { r = *reinterpret_cast<const uint4*>(p); }
  VAE_DEV void get(float* v) const {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
};
template <> struct Raw8<float> {
  float4 a, b;
  VAE_DEV void load(const float* p) {
    a = reinterpret_cast<const float4*>(p)[0];
    b = reinterpret_cast<const float4*>(p)[1];
  }
  VAE_DEV void get(float* v) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

// VPL vectors per lane per pixel; each team takes NP = kRmsVecs / VPL consecutive pixels per step and
// issues all their loads before any sum, then reduces the NP sums side by side.  A warp step covers
// one chunk of 32 / team * NP pixels of one frame, so a step costs one 32-bit division for its frame
// and chunk and none per pixel.
template <typename TI, typename TO, int VPL>
__global__ void __launch_bounds__(256) rms_apply_kernel(const __grid_constant__ RmsParams p) {
  constexpr int NP = kRmsVecs / VPL;
  const int lane = threadIdx.x & 31;
  const int L = p.team;
  const int sub = lane & (L - 1);
  const int per_step = (32 / L) * NP;  // pixels per warp step, all in one frame
  const int hw = p.H * p.W;
  const int n_chunks = (hw + per_step - 1) / per_step;
  const int items = p.B * p.T * n_chunks;
  const int warp_id = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int n_warps = static_cast<int>((gridDim.x * blockDim.x) >> 5);
  const float inv_c = 1.0f / static_cast<float>(p.C);
  for (int item = warp_id; item < items; item += n_warps) {
    const int f = item / n_chunks;
    const int r0 = (item - f * n_chunks) * per_step + (lane / L) * NP;
    const int b = f / p.T, t = f - b * p.T;
    const TI* xf = static_cast<const TI*>(p.x) + (static_cast<int64_t>(b) * p.x_T_alloc + t) * hw * p.C;
    TO* yf = static_cast<TO*>(p.y) + (static_cast<int64_t>(b) * p.y_T_alloc + t) * hw * p.C;
    Raw8<TI> raw[NP][VPL];
#pragma unroll
    for (int k = 0; k < NP; ++k)
      if (r0 + k < hw) {
#pragma unroll
        for (int j = 0; j < VPL; ++j) raw[k][j].load(xf + static_cast<int64_t>(r0 + k) * p.C + (j * L + sub) * 8);
      }
    float ss[NP];
#pragma unroll
    for (int k = 0; k < NP; ++k) {
      ss[k] = 0.f;
      if (r0 + k < hw) {
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          float v[8];
          raw[k][j].get(v);
#pragma unroll
          for (int e = 0; e < 8; ++e) ss[k] = fmaf(v[e], v[e], ss[k]);
        }
      }
    }
    for (int off = L >> 1; off > 0; off >>= 1)
#pragma unroll
      for (int k = 0; k < NP; ++k) ss[k] += __shfl_xor_sync(0xffffffffu, ss[k], off);
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int c0 = (j * L + sub) * 8;
      const float4* g4 = reinterpret_cast<const float4*>(p.gamma + c0);
      const float4* b4 = reinterpret_cast<const float4*>(p.beta + c0);
      const float4 g0 = __ldg(g4), g1 = __ldg(g4 + 1), b0 = __ldg(b4), b1 = __ldg(b4 + 1);
      const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int k = 0; k < NP; ++k) {
        if (r0 + k >= hw) continue;
        const float rr = 1.0f / sqrtf(ss[k] * inv_c + p.eps);
        float v[8], o[8];
        raw[k][j].get(v);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float z = fmaf(v[e] * rr, gg[e], bb[e]);
          o[e] = p.silu ? silu_to<TO>(z) : z;
        }
        vstore8(yf + static_cast<int64_t>(r0 + k) * p.C + c0, o, p.fault);
      }
    }
  }
}

bool rms_supported(int C) {
  if (C <= 0 || C % 8) return false;
  const int nv = C / 8;
  const int L = nv >= 32 ? 32 : nv;
  return (L & (L - 1)) == 0 && nv % L == 0 && nv / L <= kRmsMaxVpl;
}

cudaError_t launch_rms(const GnArgs& a, cudaStream_t s) {
  if (!rms_supported(a.C)) return cudaErrorInvalidValue;
  RmsParams p{};
  p.B = a.B; p.T = a.T; p.H = a.H; p.W = a.W; p.C = a.C; p.eps = a.eps; p.silu = a.silu;
  p.x = a.x; p.x_T_alloc = a.x_T_alloc ? a.x_T_alloc : a.T;
  p.y = a.y; p.y_T_alloc = a.y_T_alloc ? a.y_T_alloc : a.T;
  p.gamma = a.gamma; p.beta = a.beta;
  p.fault = fault_word();
  const int nv = a.C / 8;
  p.team = nv >= 32 ? 32 : nv;
  p.vpl = nv / p.team;
  const int64_t npx = static_cast<int64_t>(a.B) * a.T * a.H * a.W;
  if (npx == 0) return cudaSuccess;
  const int64_t per_warp = static_cast<int64_t>(32 / p.team) * (kRmsVecs / p.vpl);
  const int64_t warps = static_cast<int64_t>(a.B) * a.T * ((static_cast<int64_t>(a.H) * a.W + per_warp - 1) / per_warp);
  if (warps >= (1LL << 30) || static_cast<int64_t>(a.H) * a.W >= (1LL << 30)) return cudaErrorInvalidValue;  // 32-bit indexing
  const int blocks = static_cast<int>(std::min<int64_t>((warps + 7) / 8, 152LL * 8));
#define VAE_RMS(VPL)                                                                                     \
  if (a.y_fp8 && a.x_f32) rms_apply_kernel<float, __nv_fp8_e4m3, VPL><<<blocks, 256, 0, s>>>(p);         \
  else if (a.y_fp8) rms_apply_kernel<__nv_bfloat16, __nv_fp8_e4m3, VPL><<<blocks, 256, 0, s>>>(p);      \
  else if (a.x_f32 && a.y_f32) rms_apply_kernel<float, float, VPL><<<blocks, 256, 0, s>>>(p);            \
  else if (a.x_f32) rms_apply_kernel<float, __nv_bfloat16, VPL><<<blocks, 256, 0, s>>>(p);               \
  else if (a.y_f32) rms_apply_kernel<__nv_bfloat16, float, VPL><<<blocks, 256, 0, s>>>(p);               \
  else rms_apply_kernel<__nv_bfloat16, __nv_bfloat16, VPL><<<blocks, 256, 0, s>>>(p);
  switch (p.vpl) {
    case 1: VAE_RMS(1) break;
    case 2: VAE_RMS(2) break;
    default: VAE_RMS(4) break;
  }
#undef VAE_RMS
  return cudaGetLastError();
}

// ============================================================================ layouts
template <typename TO>
__global__ void latent_to_cl_kernel(const float* z, int B, int C, int T, int H, int W, int t0, int nt, int h0, int nh,
                                    int w0, int nw, int Cp, TO* y, int yTa) {
  const int64_t n = static_cast<int64_t>(B) * nt * nh * nw * Cp;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % Cp);
    int64_t r = i / Cp;
    const int w = static_cast<int>(r % nw); r /= nw;
    const int h = static_cast<int>(r % nh); r /= nh;
    const int t = static_cast<int>(r % nt);
    const int b = static_cast<int>(r / nt);
    float v = 0.f;
    if (c < C) v = z[((((static_cast<int64_t>(b) * C + c) * T + t0 + t) * H + h0 + h) * W) + w0 + w];
    y[(((static_cast<int64_t>(b) * yTa + t) * nh + h) * nw + w) * Cp + c] = from_f<TO>(v);
  }
}

cudaError_t launch_latent_to_cl(const float* z, int B, int C, int T, int H, int W, int t0, int nt, int h0, int nh, int w0,
                                int nw, int C_pad, void* y, int y_f32, int y_T_alloc, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(B) * nt * nh * nw * C_pad;
  if (n == 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 152 * 64));
  if (y_f32)
    latent_to_cl_kernel<float><<<blocks, 256, 0, s>>>(z, B, C, T, H, W, t0, nt, h0, nh, w0, nw, C_pad,
                                                       static_cast<float*>(y), y_T_alloc);
  else
    latent_to_cl_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(z, B, C, T, H, W, t0, nt, h0, nh, w0, nw, C_pad,
                                                               static_cast<__nv_bfloat16*>(y), y_T_alloc);
  return cudaGetLastError();
}

// depth-to-space, channels-last; one thread per 8 output channels (C % 8 == 0) or per element
template <typename T>
__global__ void d2s_kernel(const T* x, T* y, int B, int T_, int H, int W, int C, int st, int sh, int sw, int drop,
                           int vec) {
  const int To = st * T_ - drop, Ho = H * sh, Wo = W * sw;
  const int cw = vec ? 8 : 1;
  const int64_t n = static_cast<int64_t>(B) * To * Ho * Wo * (C / cw);
  const int S = st * sh * sw;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int cv = static_cast<int>(i % (C / cw));
    int64_t r = i / (C / cw);
    const int wo = static_cast<int>(r % Wo); r /= Wo;
    const int ho = static_cast<int>(r % Ho); r /= Ho;
    const int to = static_cast<int>(r % To);
    const int b = static_cast<int>(r / To);
    const int tf = to + drop;
    const int t = tf / st, dt = tf % st, h = ho / sh, dy = ho % sh, w = wo / sw, dx = wo % sw;
    const int sub = (dt * sh + dy) * sw + dx;
    const int64_t xpix = ((static_cast<int64_t>(b) * T_ + t) * H + h) * W + w;
    const int64_t ypix = ((static_cast<int64_t>(b) * To + to) * Ho + ho) * Wo + wo;
    for (int e = 0; e < cw; ++e) {
      const int c = cv * cw + e;
      y[ypix * C + c] = x[xpix * C * S + static_cast<int64_t>(c) * S + sub];
    }
  }
}

cudaError_t launch_d2s(const void* x, void* y, int B, int T, int H, int W, int C, int st, int sh, int sw,
                       int drop_first, int f32, cudaStream_t s) {
  const int drop = drop_first ? st - 1 : 0;
  const int64_t n = static_cast<int64_t>(B) * (st * T - drop) * H * sh * W * sw * C;
  if (n <= 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>((n / 8 + 255) / 256 + 1, 152 * 64));
  const int vec = (C % 8 == 0);
  if (f32) d2s_kernel<float><<<blocks, 256, 0, s>>>(static_cast<const float*>(x), static_cast<float*>(y), B, T, H, W, C, st, sh, sw, drop, vec);
  else d2s_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), B, T, H, W, C, st, sh, sw, drop, vec);
  return cudaGetLastError();
}

cudaError_t launch_copy_frames(const void* src, int src_T, int src_t0, void* dst, int dst_T, int dst_t0, int n_frames,
                               int B, int64_t frame_bytes, cudaStream_t s) {
  if (n_frames <= 0 || B <= 0) return cudaSuccess;
  const char* sp = static_cast<const char*>(src) + src_t0 * frame_bytes;
  char* dp = static_cast<char*>(dst) + dst_t0 * frame_bytes;
  return cudaMemcpy2DAsync(dp, dst_T * frame_bytes, sp, src_T * frame_bytes, n_frames * frame_bytes, B,
                           cudaMemcpyDeviceToDevice, s);
}

// ============================================================================ tile blend
struct BlendTile {
  const void* ptr;
  int t0, nt, h0, nh, w0, nw;
  unsigned short ovl[6];
};
struct BlendParams {
  int B, C, T, H, W, n;
  int tile_f32, out_f32;
  void* out;
  BlendTile tiles[VAE_MAX_TILES];
};

// Ramp of a tile of n pixels at local coordinate y: (y+1)/(lo+1) over the lo-pixel overlap with the
// previous tile, (n-y)/(hi+1) over the hi-pixel overlap with the next, 1 elsewhere.
VAE_DEV float ramp_w(int y, int n, int lo, int hi) {
  float w = 1.f;
  if (y < lo) w *= __fdividef(static_cast<float>(y + 1), static_cast<float>(lo + 1));
  if (y >= n - hi) w *= __fdividef(static_cast<float>(n - y), static_cast<float>(hi + 1));
  return w;
}

// One warp per output row (t, y), 8 rows per block, no block-wide synchronisation.  The warp lists
// the tiles covering (t, y) in tile order (32 tiles per ballot round) together with everything that
// does not depend on x or the plane (row offset, plane stride, x extent, overlaps, t/y weight); its
// lanes then take (plane, 8-pixel vector) jobs, consecutive lanes on consecutive vectors of one
// plane, and gather from the listed tiles.
struct RowTile {
  const void* ptr;
  long long rowoff, pstride;
  int w0, nw, lo, hi;
  float wty;
};
constexpr int kBlendRowsPerBlock = 8;
constexpr int kRowList = 64;  // covering tiles of one row kept in shared memory
template <typename TT, typename TO>
__global__ void __launch_bounds__(32 * kBlendRowsPerBlock) blend_kernel(const __grid_constant__ BlendParams p) {
  __shared__ RowTile rts[kBlendRowsPerBlock][kRowList];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_per_t = (p.H + kBlendRowsPerBlock - 1) / kBlendRowsPerBlock;
  const int pl = blockIdx.y;  // one (b, c) plane per block: a block's reads stay in few pages
  const int t = blockIdx.x / rows_per_t;
  const int y = (blockIdx.x - t * rows_per_t) * kBlendRowsPerBlock + warp;
  if (y >= p.H) return;
  RowTile* rt = rts[warp];
  int nk = 0;
  for (int i0 = 0; i0 < p.n; i0 += 32) {
    const int i = i0 + lane;
    bool cov = false;
    if (i < p.n) {
      const BlendTile& tl = p.tiles[i];
      cov = t >= tl.t0 && t < tl.t0 + tl.nt && y >= tl.h0 && y < tl.h0 + tl.nh;
    }
    const unsigned m = __ballot_sync(0xffffffffu, cov);
    if (cov) {
      const int k = nk + __popc(m & ((1u << lane) - 1u));
      if (k < kRowList) {
        const BlendTile& tl = p.tiles[i];
        RowTile r;
        r.ptr = tl.ptr;
        r.rowoff = (static_cast<long long>(t - tl.t0) * tl.nh + (y - tl.h0)) * tl.nw;
        r.pstride = static_cast<long long>(tl.nt) * tl.nh * tl.nw;
        r.w0 = tl.w0;
        r.nw = tl.nw;
        r.lo = tl.ovl[4];
        r.hi = tl.ovl[5];
        r.wty = ramp_w(t - tl.t0, tl.nt, tl.ovl[0], tl.ovl[1]) * ramp_w(y - tl.h0, tl.nh, tl.ovl[2], tl.ovl[3]);
        rt[k] = r;
      }
    }
    nk += __popc(m);
  }
  __syncwarp();
  const bool spill = nk > kRowList;  // more covering tiles than listed: read them from the table
  const int nv = (p.W + 7) / 8;
  const int jobs = nv;
  const int64_t plane_out = static_cast<int64_t>(p.T) * p.H * p.W;
  const int64_t row_out = (static_cast<int64_t>(t) * p.H + y) * p.W;
  constexpr int kJ = 1;  // jobs per lane whose loads are all issued before any is summed
  for (int job0 = lane; job0 < jobs; job0 += 32 * kJ) {
    // phase 1: for each job find (at most 2) covering tiles with whole aligned vectors and load them
    ApplyVec<TT> raw[kJ][2];
    int sel[kJ][2];
    int nsel[kJ];
#pragma unroll
    for (int u = 0; u < kJ; ++u) {
      nsel[u] = 0;
      const int job = job0 + 32 * u;
      if (job >= jobs || spill) {
        nsel[u] = job >= jobs ? 0 : -1;
        continue;
      }
      const int x0 = job * 8;
      for (int k = 0; k < nk; ++k) {
        const int lx = x0 - rt[k].w0;
        if (lx + 8 <= 0 || lx >= rt[k].nw) continue;
        const bool aligned = lx >= 0 && lx + 8 <= rt[k].nw && ((lx | rt[k].nw) & 7) == 0;
        if (!aligned || nsel[u] == 2) {
          nsel[u] = -1;  // generic path
          break;
        }
        const TT* src = static_cast<const TT*>(rt[k].ptr) + pl * rt[k].pstride + rt[k].rowoff + lx;
        if (nsel[u] == 0) {  // constant register indices only (no local-memory arrays)
          raw[u][0].load(src);
          sel[u][0] = k;
        } else {
          raw[u][1].load(src);
          sel[u][1] = k;
        }
        ++nsel[u];
      }
    }
    // phase 2: weights and sums
#pragma unroll
    for (int u = 0; u < kJ; ++u) {
      const int job = job0 + 32 * u;
      if (job >= jobs) break;
      const int x0 = job * 8;
      float acc[8], ws[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = ws[e] = 0.f;
      if (nsel[u] >= 0) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (j >= nsel[u]) break;
          const RowTile& r = rt[sel[u][j]];
          const int lx = x0 - r.w0;
          float v[8];
          raw[u][j].get(v);
          if (lx >= r.lo && lx + 8 <= r.nw - r.hi) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              acc[e] = fmaf(r.wty, v[e], acc[e]);
              ws[e] += r.wty;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float w = r.wty * ramp_w(lx + e, r.nw, r.lo, r.hi);
              acc[e] = fmaf(w, v[e], acc[e]);
              ws[e] += w;
            }
          }
        }
      } else {
        // generic: every covering tile, element by element
        const int nloop = spill ? p.n : nk;
        for (int k = 0; k < nloop; ++k) {
          RowTile r;
          if (!spill) {
            r = rt[k];
          } else {
            const BlendTile& tl = p.tiles[k];
            if (t < tl.t0 || t >= tl.t0 + tl.nt || y < tl.h0 || y >= tl.h0 + tl.nh) continue;
            r.ptr = tl.ptr;
            r.rowoff = (static_cast<long long>(t - tl.t0) * tl.nh + (y - tl.h0)) * tl.nw;
            r.pstride = static_cast<long long>(tl.nt) * tl.nh * tl.nw;
            r.w0 = tl.w0;
            r.nw = tl.nw;
            r.lo = tl.ovl[4];
            r.hi = tl.ovl[5];
            r.wty = ramp_w(t - tl.t0, tl.nt, tl.ovl[0], tl.ovl[1]) * ramp_w(y - tl.h0, tl.nh, tl.ovl[2], tl.ovl[3]);
          }
          const int lx = x0 - r.w0;
          if (lx + 8 <= 0 || lx >= r.nw) continue;
          const TT* src = static_cast<const TT*>(r.ptr) + pl * r.pstride + r.rowoff;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int xx = lx + e;
            if (xx < 0 || xx >= r.nw) continue;
            const float w = r.wty * ramp_w(xx, r.nw, r.lo, r.hi);
            acc[e] = fmaf(w, to_f<TT>(src[xx]), acc[e]);
            ws[e] += w;
          }
        }
      }
      TO* orow = static_cast<TO*>(p.out) + pl * plane_out + row_out;
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = ws[e] > 0.f ? __fdividef(acc[e], ws[e]) : 0.f;
      if (x0 + 8 <= p.W && (p.W & 7) == 0) {
        store8(orow + x0, o);
      } else {
        for (int e = 0; e < 8 && x0 + e < p.W; ++e) orow[x0 + e] = from_f<TO>(o[e]);
      }
    }
  }
}

// Blend for tile sets that form a grid (the tile plan's output): tile (a, b, c) is the product of the
// a-th temporal, b-th row and c-th column interval, and its weight the product of the three 1-D
// ramps, so out = sum_{a,b,c} w_a w_b w_c x_abc / (sum_a w_a)(sum_b w_b)(sum_c w_c).  One warp per
// output row of one plane at a time: the (a, b) pairs covering (t, y) are found once per row from the
// interval lists, the column intervals covering each 8-pixel vector once per block.
constexpr int kAxisMax = 64;
struct BlendGridParams {
  int B, C, T, H, W;
  int n[3];                       // intervals per axis (t, h, w)
  int s0[3][kAxisMax], len[3][kAxisMax];
  unsigned short lo[3][kAxisMax], hi[3][kAxisMax];
  void* out;
  const void* ptr[VAE_MAX_TILES];  // tile (a, b, c) at ptr[(a * n[1] + b) * n[2] + c]
};


// Rows per block of the grid blend (of every plane); the 8 warps take (plane, row) tasks in turn.
constexpr int kGridRows = 32;
constexpr int kGridMaxVec = 384;  // 8-pixel vectors per row with a shared-memory entry (W <= 3072)

// axis_cover with the (at most 2) results in scalars, so they stay in registers.
VAE_DEV int axis_cover2(const BlendGridParams& p, int ax, int x, int& i0, int& i1, float& w0, float& w1) {
  int k = 0;
  i0 = i1 = 0;
  w0 = w1 = 0.f;
  for (int i = 0; i < p.n[ax] && k < 2; ++i) {
    const int l = x - p.s0[ax][i];
    if (l < 0 || l >= p.len[ax][i]) continue;
    const float w = ramp_w(l, p.len[ax][i], p.lo[ax][i], p.hi[ax][i]);
    if (k == 0) {
      i0 = i;
      w0 = w;
    } else {
      i1 = i;
      w1 = w;
    }
    ++k;
  }
  const float inv = __fdividef(1.f, w0 + w1);
  w0 *= inv;
  w1 *= inv;
  return k;
}

// 16-byte asynchronous copy global -> shared (L2 only), and its group fences.
VAE_DEV void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
VAE_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> VAE_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Grid blend for grids with at most kG2Cols column intervals (others take the general kernel).  Per
// 8-pixel vector, built once per block: one packed shared-memory word (first column interval, count,
// offsets into both intervals' rows) and the first interval's normalised column weights (the
// second's are one minus them).  Per warp and (plane, row): the source row pointers of each (t, y)
// pair and column interval, and the pair weights in registers.  A lane issues every source load of
// its vector before summing; rows covered by more than two (t, y) pairs, and ragged or unaligned
// vectors, take the per-pixel loop.
constexpr int kG2Cols = 16;
constexpr int kBlendRing = 3;  // staged source vectors per lane: 2 in flight while one is summed (static smem <= 48 KB)
// Per 8-pixel vector of an output row, built once per block: one packed word (first column interval,
// count, fast-path flag, offsets into both intervals' rows) and the first interval's normalised column
// weights (the second's are one minus them).
VAE_DEV void build_vec_table(const BlendGridParams& p, int4* vinfo, float4 (*vw0)[2]) {
  const int nv = (p.W + 7) / 8;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    const int x0 = v * 8;
    int c0 = -1, nc = 0;
    for (int i = 0; i < p.n[2]; ++i) {
      const int l = x0 - p.s0[2][i];
      if (l + 8 <= 0 || l >= p.len[2][i]) continue;
      if (c0 < 0) c0 = i;
      ++nc;
    }
    if (c0 < 0) c0 = 0;
    int lx[2] = {0, 0};
    bool fast = nc >= 1 && nc <= 2 && x0 + 8 <= p.W;
    float w0[8];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (j < nc && nc <= 2) {
        lx[j] = x0 - p.s0[2][c0 + j];
        const int nw = p.len[2][c0 + j];
        fast = fast && lx[j] >= 0 && lx[j] + 8 <= nw && ((lx[j] | nw) & 7) == 0;
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float a0 = 0.f, a1 = 0.f;
      if (nc >= 1 && nc <= 2 && x0 + e < p.W) {
        const int l0 = lx[0] + e, n0 = p.len[2][c0];
        if (l0 >= 0 && l0 < n0) a0 = ramp_w(l0, n0, p.lo[2][c0], p.hi[2][c0]);
        if (nc == 2) {
          const int l1 = lx[1] + e, n1 = p.len[2][c0 + 1];
          if (l1 >= 0 && l1 < n1) a1 = ramp_w(l1, n1, p.lo[2][c0 + 1], p.hi[2][c0 + 1]);
        }
      }
      const float sum = a0 + a1;
      w0[e] = sum > 0.f ? __fdividef(a0, sum) : 0.f;
    }
    vinfo[v] = make_int4(c0 | (nc << 8) | (fast ? 1 << 12 : 0), lx[0], lx[1], 0);
    vw0[v][0] = make_float4(w0[0], w0[1], w0[2], w0[3]);
    vw0[v][1] = make_float4(w0[4], w0[5], w0[6], w0[7]);
  }
}

template <typename TT, typename TO>
__global__ void __launch_bounds__(256, 4) blend_grid2_kernel(const __grid_constant__ BlendGridParams p) {
  __shared__ int4 vinfo[kGridMaxVec];
  __shared__ float4 vw0[kGridMaxVec][2];
  __shared__ const TT* rowp[8][4][kG2Cols];
  // bf16 tiles, rows covered by one (t, y) pair: each lane's source vectors (one per column
  // interval) of its next kBlendRing - 1 vectors are copied here asynchronously while it sums the
  // current one
  __shared__ uint4 stage[sizeof(TT) == 2 ? 8 : 1][kBlendRing][2][32];
  const int nv = (p.W + 7) / 8;
  build_vec_table(p, vinfo, vw0);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blocks_per_t = (p.H + kGridRows - 1) / kGridRows;
  const int n_pl = p.B * p.C;
  const int t = blockIdx.x / blocks_per_t;
  const int y_base = (blockIdx.x - t * blocks_per_t) * kGridRows;
  int ia0, ia1;
  float wa0, wa1;
  const int na = axis_cover2(p, 0, t, ia0, ia1, wa0, wa1);
  const int n2 = p.n[2];
  for (int task = warp; task < n_pl * kGridRows; task += 8) {
    const int pl = task / kGridRows, r = task - (task / kGridRows) * kGridRows;
    const int y = y_base + r;
    if (y >= p.H) continue;
    int ib0, ib1;
    float wb0, wb1;
    const int nb = axis_cover2(p, 1, y, ib0, ib1, wb0, wb1);
    const int npair = na * nb;
    for (int e = lane; e < npair * n2; e += 32) {
      const int q = e / n2, cc = e - q * n2;
      const int qa = nb == 2 ? q >> 1 : q, qb = nb == 2 ? q & 1 : 0;
      const int a = qa ? ia1 : ia0, b = qb ? ib1 : ib0;
      const int64_t plane_in = static_cast<int64_t>(p.len[0][a]) * p.len[1][b];
      rowp[warp][q][cc] = static_cast<const TT*>(p.ptr[(a * p.n[1] + b) * n2 + cc]) +
                          ((pl * plane_in + static_cast<int64_t>(t - p.s0[0][a]) * p.len[1][b]) + (y - p.s0[1][b])) *
                              p.len[2][cc];
    }
    __syncwarp();
    float wq[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int qa = nb == 2 ? q >> 1 : q, qb = nb == 2 ? q & 1 : 0;
      wq[q] = q < npair ? (qa ? wa1 : wa0) * (qb ? wb1 : wb0) : 0.f;
    }
    TO* orow = static_cast<TO*>(p.out) + ((static_cast<int64_t>(pl) * p.T + t) * p.H + y) * p.W;
    if constexpr (sizeof(TT) == 2) {
      if (npair == 1) {
        // issue the copies of vector v's sources into buffer `buf`; returns whether v is on the fast path
        auto issue = [&](int v, int buf) -> bool {
          if (v >= nv) return false;
          const int4 inf = vinfo[v];
          if (!((inf.x >> 12) & 1)) return false;
          const int cv = inf.x & 255, ncv = (inf.x >> 8) & 15;
#pragma unroll
          for (int j = 0; j < 2; ++j)
            if (j < ncv) cp_async16(&stage[warp][buf][j][lane], rowp[warp][0][cv + j] + (j ? inf.z : inf.y));
          return true;
        };
        uint32_t fm = 0;  // bit k: ring slot k holds a fast-path vector
#pragma unroll
        for (int k = 0; k < kBlendRing - 1; ++k) {
          if (issue(lane + 32 * k, k)) fm |= 1u << k;
          cp_async_commit();
        }
        int buf = 0;
        for (int v = lane; v < nv; v += 32) {
          const int refill = buf == 0 ? kBlendRing - 1 : buf - 1;  // the slot consumed last step
          fm &= ~(1u << refill);
          if (issue(v + 32 * (kBlendRing - 1), refill)) fm |= 1u << refill;
          cp_async_commit();
          cp_async_wait<kBlendRing - 1>();  // this lane's copies for v have landed
          const bool fast_cur = (fm >> buf) & 1u;
          const int x0 = v * 8;
          float acc[8];
          if (fast_cur) {
            const int ncv = (vinfo[v].x >> 8) & 15;
            const float4 wl = vw0[v][0], wh = vw0[v][1];
            const float w0[8] = {wl.x, wl.y, wl.z, wl.w, wh.x, wh.y, wh.z, wh.w};
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              float val[8];
              if (j < ncv) {
                Raw8<TT> r;
                r.r = stage[warp][buf][j][lane];
                r.get(val);
              } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) val[e] = 0.f;
              }
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float wc = (j ? 1.f - w0[e] : w0[e]) * wq[0];
                acc[e] = j ? fmaf(wc, val[e], acc[e]) : wc * val[e];
              }
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              acc[e] = 0.f;
              const int x = x0 + e;
              if (x >= p.W) continue;
              int ic0, ic1;
              float wc0, wc1;
              const int ncx = axis_cover2(p, 2, x, ic0, ic1, wc0, wc1);
              for (int j = 0; j < ncx; ++j) {
                const int ci = j ? ic1 : ic0;
                acc[e] = fmaf(wq[0] * (j ? wc1 : wc0), to_f<TT>(rowp[warp][0][ci][x - p.s0[2][ci]]), acc[e]);
              }
            }
          }
          if (x0 + 8 <= p.W && (p.W & 7) == 0) {
            store8(orow + x0, acc);
          } else {
            for (int e = 0; e < 8 && x0 + e < p.W; ++e) orow[x0 + e] = from_f<TO>(acc[e]);
          }
          buf = buf + 1 == kBlendRing ? 0 : buf + 1;
        }
        cp_async_wait<0>();
        __syncwarp();
        continue;
      }
    }
    for (int v = lane; v < nv; v += 32) {
      const int4 inf = vinfo[v];
      const bool fast = (inf.x >> 12) & 1;
      const int x0 = v * 8;
      float acc[8];
      if (fast) {
        // up to 4 (t, y) pairs (frames and rows both in overlaps), taken two at a time: the loads of
        // two pairs are in flight together, the pair-weighted sums s[j] kept per column interval j
        const int cv = inf.x & 255, ncv = (inf.x >> 8) & 15;
        float s2[2][8];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 8; ++e) s2[j][e] = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (2 * h >= npair) break;
          Raw8<TT> raw[2][2];  // [pair][interval]
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int j = 0; j < 2; ++j)
              if (2 * h + q < npair && j < ncv) raw[q][j].load(rowp[warp][2 * h + q][cv + j] + (j ? inf.z : inf.y));
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int j = 0; j < 2; ++j)
              if (2 * h + q < npair && j < ncv) {
                float val[8];
                raw[q][j].get(val);
#pragma unroll
                for (int e = 0; e < 8; ++e) s2[j][e] = fmaf(wq[2 * h + q], val[e], s2[j][e]);
              }
        }
        const float4 wl = vw0[v][0], wh = vw0[v][1];
        const float w0[8] = {wl.x, wl.y, wl.z, wl.w, wh.x, wh.y, wh.z, wh.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(1.f - w0[e], s2[1][e], w0[e] * s2[0][e]);
      } else {
        // ragged or unaligned vector: per pixel (unrolled, so that acc stays in registers)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          acc[e] = 0.f;
          const int x = x0 + e;
          if (x >= p.W) continue;
          int ic0, ic1;
          float wc0, wc1;
          const int ncx = axis_cover2(p, 2, x, ic0, ic1, wc0, wc1);
          for (int q = 0; q < npair; ++q) {
            const int qa = nb == 2 ? q >> 1 : q, qb = nb == 2 ? q & 1 : 0;
            const float wqq = (qa ? wa1 : wa0) * (qb ? wb1 : wb0);  // (no dynamically indexed array)
            for (int j = 0; j < ncx; ++j) {
              const int ci = j ? ic1 : ic0;
              acc[e] = fmaf(wqq * (j ? wc1 : wc0), to_f<TT>(rowp[warp][q][ci][x - p.s0[2][ci]]), acc[e]);
            }
          }
        }
      }
      if (x0 + 8 <= p.W && (p.W & 7) == 0) {
        store8(orow + x0, acc);
      } else {
        for (int e = 0; e < 8 && x0 + e < p.W; ++e) orow[x0 + e] = from_f<TO>(acc[e]);
      }
    }
    __syncwarp();
  }
}


namespace {
// Recognise a grid: tiles in raster order over per-axis interval lists with per-axis overlaps, at most
// two intervals covering any coordinate (overlap shorter than the stride).
bool build_grid(const void* const* tiles, const vae_tile_t* meta, int n, const vae_blend_desc_t& d,
                BlendGridParams& g) {
  const int extent[3] = {d.T, d.H, d.W};
  for (int ax = 0; ax < 3; ++ax) {
    int cnt = 0;
    for (int i = 0; i < n; ++i) {
      const int s0 = meta[i].pix[2 * ax], ln = meta[i].pix[2 * ax + 1];
      bool seen = false;
      for (int k = 0; k < cnt; ++k)
        if (g.s0[ax][k] == s0 && g.len[ax][k] == ln) seen = true;
      if (seen) continue;
      if (cnt == kAxisMax) return false;
      g.s0[ax][cnt] = s0;
      g.len[ax][cnt] = ln;
      g.lo[ax][cnt] = static_cast<unsigned short>(meta[i].ovl[2 * ax]);
      g.hi[ax][cnt] = static_cast<unsigned short>(meta[i].ovl[2 * ax + 1]);
      ++cnt;
    }
    g.n[ax] = cnt;
    for (int k = 1; k < cnt; ++k)
      if (g.s0[ax][k] <= g.s0[ax][k - 1]) return false;           // sorted starts
    for (int k = 2; k < cnt; ++k)
      if (g.s0[ax][k] < g.s0[ax][k - 2] + g.len[ax][k - 2]) return false;  // <= 2 cover a point
    (void)extent;
  }
  if (static_cast<long long>(g.n[0]) * g.n[1] * g.n[2] != n) return false;
  for (int i = 0; i < n; ++i) {
    const int a = i / (g.n[1] * g.n[2]), b = (i / g.n[2]) % g.n[1], c = i % g.n[2];
    const int idx[3] = {a, b, c};
    for (int ax = 0; ax < 3; ++ax) {
      const int k = idx[ax];
      if (meta[i].pix[2 * ax] != g.s0[ax][k] || meta[i].pix[2 * ax + 1] != g.len[ax][k] ||
          meta[i].ovl[2 * ax] != g.lo[ax][k] || meta[i].ovl[2 * ax + 1] != g.hi[ax][k])
        return false;
    }
    g.ptr[i] = tiles[i];
  }
  return true;
}
}  // namespace

cudaError_t launch_blend(const void* const* tiles, const vae_tile_t* meta, int n_tiles, void* out,
                         const vae_blend_desc_t& d, cudaStream_t s) {
  // per call and per host thread (about 20 KB each, kept off the stack): concurrent launches never
  // share them, and a launch copies its parameters before returning
  thread_local BlendParams p;
  thread_local BlendGridParams g;
  p = BlendParams{};
  g = BlendGridParams{};
  if (n_tiles > VAE_MAX_TILES) return cudaErrorInvalidValue;
  if (static_cast<long long>(d.B) * d.C > 65535) return cudaErrorInvalidValue;
  if (d.W <= 8 * kGridMaxVec && build_grid(tiles, meta, n_tiles, d, g) && g.n[2] <= kG2Cols) {
    g.B = d.B; g.C = d.C; g.T = d.T; g.H = d.H; g.W = d.W; g.out = out;
    const long long nb = static_cast<long long>(d.T) * ((d.H + kGridRows - 1) / kGridRows);
    if (nb == 0) return cudaSuccess;
    if (nb > 0x7fffffffLL) return cudaErrorInvalidValue;
    const bool tf = d.tile_dtype == VAE_FP32, of = d.out_dtype == VAE_FP32;
    const dim3 grid(static_cast<unsigned>(nb));  // every plane of a (t, row chunk) in one block
    if (tf && of) blend_grid2_kernel<float, float><<<grid, 256, 0, s>>>(g);
    else if (tf) blend_grid2_kernel<float, __nv_bfloat16><<<grid, 256, 0, s>>>(g);
    else if (of) blend_grid2_kernel<__nv_bfloat16, float><<<grid, 256, 0, s>>>(g);
    else blend_grid2_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, s>>>(g);
    return cudaGetLastError();
  }
  p.B = d.B; p.C = d.C; p.T = d.T; p.H = d.H; p.W = d.W; p.n = n_tiles;
  p.tile_f32 = d.tile_dtype == VAE_FP32;
  p.out_f32 = d.out_dtype == VAE_FP32;
  p.out = out;
  for (int i = 0; i < n_tiles; ++i) {
    BlendTile& t = p.tiles[i];
    t.ptr = tiles[i];
    t.t0 = meta[i].pix[0]; t.nt = meta[i].pix[1];
    t.h0 = meta[i].pix[2]; t.nh = meta[i].pix[3];
    t.w0 = meta[i].pix[4]; t.nw = meta[i].pix[5];
    for (int k = 0; k < 6; ++k) t.ovl[k] = static_cast<unsigned short>(meta[i].ovl[k]);
  }
  const long long nb = static_cast<long long>(d.T) * ((d.H + kBlendRowsPerBlock - 1) / kBlendRowsPerBlock);
  if (nb == 0) return cudaSuccess;
  if (static_cast<long long>(d.B) * d.C > 65535) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(nb), static_cast<unsigned>(d.B * d.C));
  const int threads = 32 * kBlendRowsPerBlock;
  if (p.tile_f32 && p.out_f32) blend_kernel<float, float><<<grid, threads, 0, s>>>(p);
  else if (p.tile_f32) blend_kernel<float, __nv_bfloat16><<<grid, threads, 0, s>>>(p);
  else if (p.out_f32) blend_kernel<__nv_bfloat16, float><<<grid, threads, 0, s>>>(p);
  else blend_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, threads, 0, s>>>(p);
  return cudaGetLastError();
}

// ============================================================================ attention helpers
// softmax over each row's first `cols` entries; padded columns of P (up to ld_out) are zeroed
template <typename TO>
__global__ void __launch_bounds__(256) softmax_rows_kernel(const float* s, TO* p, int cols, int ld_out) {
  __shared__ float red[32];
  const float* row = s + static_cast<int64_t>(blockIdx.x) * cols;
  TO* out = p + static_cast<int64_t>(blockIdx.x) * ld_out;
  float m = -INFINITY;
  for (int i = threadIdx.x; i < cols; i += blockDim.x) m = fmaxf(m, row[i]);
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : -INFINITY;
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  m = red[0];
  __syncthreads();
  float sum = 0.f;
  for (int i = threadIdx.x; i < cols; i += blockDim.x) sum += expf(row[i] - m);
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float inv = 1.f / red[0];
  for (int i = threadIdx.x; i < ld_out; i += blockDim.x)
    out[i] = from_f<TO>(i < cols ? expf(row[i] - m) * inv : 0.f);
}

// Rows of at most 4096 columns (cols % 4 == 0, ld_out % 4 == 0): the row is read once, as float4
// vectors held in registers (NV per thread); exp is taken once per element and the row written from
// registers, padding columns as zeros.
template <typename TO, int NV>
__global__ void __launch_bounds__(256) softmax_rows_reg_kernel(const float* s, TO* p, int cols, int ld_out) {
  __shared__ float red[32];
  const float4* row = reinterpret_cast<const float4*>(s + static_cast<int64_t>(blockIdx.x) * cols);
  TO* out = p + static_cast<int64_t>(blockIdx.x) * ld_out;
  const int nv = cols / 4;
  float4 v[NV];
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int i = threadIdx.x + k * 256;
    v[k] = i < nv ? row[i] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    m = fmaxf(m, fmaxf(fmaxf(v[k].x, v[k].y), fmaxf(v[k].z, v[k].w)));
  }
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    v[k].x = expf(v[k].x - m);  // (-inf - m = -inf: padding lanes give 0)
    v[k].y = expf(v[k].y - m);
    v[k].z = expf(v[k].z - m);
    v[k].w = expf(v[k].w - m);
    sum += (v[k].x + v[k].y) + (v[k].z + v[k].w);
  }
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float inv = 1.f / tot;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int i = threadIdx.x + k * 256;
    if (i < nv) {
      const float o4[4] = {v[k].x * inv, v[k].y * inv, v[k].z * inv, v[k].w * inv};
      if constexpr (sizeof(TO) == 2) {
        uint2 u;
        reinterpret_cast<__nv_bfloat162*>(&u)[0] = __floats2bfloat162_rn(o4[0], o4[1]);
        reinterpret_cast<__nv_bfloat162*>(&u)[1] = __floats2bfloat162_rn(o4[2], o4[3]);
        *reinterpret_cast<uint2*>(out + 4 * i) = u;
      } else {
        *reinterpret_cast<float4*>(out + 4 * i) = make_float4(o4[0], o4[1], o4[2], o4[3]);
      }
    }
  }
  for (int i = cols + threadIdx.x; i < ld_out; i += 256) out[i] = from_f<TO>(0.f);
}

cudaError_t launch_softmax_rows(const float* s_in, void* p_out, int p_f32, int rows, int cols, int ld_out,
                                cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (cols > 0 && cols <= 4096 && cols % 4 == 0 && ld_out % 4 == 0) {
    const int nv = (cols / 4 + 255) / 256;  // float4 vectors per thread
#define VAE_SMX(NV)                                                                                                   \
  if (p_f32) softmax_rows_reg_kernel<float, NV><<<rows, 256, 0, s>>>(s_in, static_cast<float*>(p_out), cols, ld_out); \
  else softmax_rows_reg_kernel<__nv_bfloat16, NV><<<rows, 256, 0, s>>>(s_in, static_cast<__nv_bfloat16*>(p_out), cols, ld_out);
    switch (nv) {
      case 1: VAE_SMX(1) break;
      case 2: VAE_SMX(2) break;
      case 3: VAE_SMX(3) break;
      default: VAE_SMX(4) break;
    }
#undef VAE_SMX
    return cudaGetLastError();
  }
  if (p_f32) softmax_rows_kernel<float><<<rows, 256, 0, s>>>(s_in, static_cast<float*>(p_out), cols, ld_out);
  else softmax_rows_kernel<__nv_bfloat16><<<rows, 256, 0, s>>>(s_in, static_cast<__nv_bfloat16*>(p_out), cols, ld_out);
  return cudaGetLastError();
}

// CUDA-core batched GEMM, 32 x 32 output tile per block, fp32
__global__ void __launch_bounds__(256) gemm_simt_kernel(const float* A, const float* Bm, float* D, const float* bias,
                                                        const float* res, int M, int N, int K, int64_t sa, int64_t sb,
                                                        int64_t sd, int64_t ldb_n, int64_t ldb_k, float alpha) {
  __shared__ float As[32][33], Bs[32][33];
  const int bz = blockIdx.z;
  const float* a = A + bz * sa;
  const float* bmat = Bm + bz * sb;
  const int m0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;  // 32 x 8
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k0 = 0; k0 < K; k0 += 32) {
    for (int r = ty; r < 32; r += 8) {
      const int m = m0 + r, k = k0 + tx, n = n0 + r;
      As[r][tx] = (m < M && k < K) ? a[static_cast<int64_t>(m) * K + k] : 0.f;
      Bs[r][tx] = (n < N && k < K) ? bmat[n * ldb_n + k * ldb_k] : 0.f;
    }
    __syncthreads();
    for (int k = 0; k < 32; ++k) {
      const float bv = Bs[tx][k];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = fmaf(As[ty + 8 * i][k], bv, acc[i]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 8 * i, n = n0 + tx;
    if (m < M && n < N) {
      const int64_t o = bz * sd + static_cast<int64_t>(m) * N + n;
      float v = acc[i] * alpha + (bias ? bias[n] : 0.f);
      if (res) v += res[o];
      D[o] = v;
    }
  }
}

cudaError_t launch_gemm_simt(const float* A, const float* Bm, float* D, const float* bias, const float* residual,
                             int M, int N, int K, int batch, int64_t sa, int64_t sb, int64_t sd, int64_t ldb_n,
                             int64_t ldb_k, float alpha, cudaStream_t s) {
  if (M <= 0 || N <= 0 || batch <= 0) return cudaSuccess;
  dim3 grid((N + 31) / 32, (M + 31) / 32, batch);
  gemm_simt_kernel<<<grid, 256, 0, s>>>(A, Bm, D, bias, residual, M, N, K, sa, sb, sd, ldb_n, ldb_k, alpha);
  return cudaGetLastError();
}

template <typename TI, typename TO>
__global__ void cast_frames_kernel(const TI* x, int xTa, TO* y, int yTa, int T, int64_t fe, int64_t n, uint32_t* fault) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = i % fe;
    const int64_t f = i / fe;
    const int64_t t = f % T, b = f / T;
    const float v = to_f<TI>(x[(b * xTa + t) * fe + e]);
    if (sizeof(TO) == 1 && !(fabsf(v) <= 448.f)) raise_fault(fault, FAULT_RANGE, 23);
    y[(b * yTa + t) * fe + e] = from_f<TO>(v);
  }
}

// 8 consecutive elements per thread (frame_elems a multiple of 8): one 16- or 32-byte load, one store
template <typename TI, typename TO>
__global__ void cast_frames8_kernel(const TI* x, int xTa, TO* y, int yTa, int T, int64_t fv, int64_t nv, uint32_t* fault) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nv;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = i % fv;
    const int64_t f = i / fv;
    const int64_t t = f % T, b = f / T;
    float v[8];
    load8(x + ((b * xTa + t) * fv + e) * 8, v);
    vstore8(y + ((b * yTa + t) * fv + e) * 8, v, fault);
  }
}

cudaError_t launch_cast_frames(const void* x, int x_f32, int x_T_alloc, void* y, int y_kind, int y_T_alloc, int B, int T,
                               int64_t frame_elems, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(B) * T * frame_elems;
  if (n <= 0) return cudaSuccess;
  if (frame_elems % 8 == 0) {
    const int64_t fv = frame_elems / 8, nv = n / 8;
    const int blocks8 = static_cast<int>(std::min<int64_t>((nv + 255) / 256, 152 * 16));
    uint32_t* f8 = fault_word();
    const float* xf = static_cast<const float*>(x);
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
#define VAE_CAST8(XP, TO) \
  cast_frames8_kernel<<<blocks8, 256, 0, s>>>(XP, x_T_alloc, static_cast<TO*>(y), y_T_alloc, T, fv, nv, f8)
    if (x_f32) {
      if (y_kind == 1) VAE_CAST8(xf, float);
      else if (y_kind == 2) VAE_CAST8(xf, __nv_fp8_e4m3);
      else VAE_CAST8(xf, __nv_bfloat16);
    } else {
      if (y_kind == 1) VAE_CAST8(xb, float);
      else if (y_kind == 2) VAE_CAST8(xb, __nv_fp8_e4m3);
      else VAE_CAST8(xb, __nv_bfloat16);
    }
#undef VAE_CAST8
    return cudaGetLastError();
  }
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 152 * 64));
  const float* xf = static_cast<const float*>(x);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  uint32_t* fault = fault_word();
  const int y_f32 = y_kind == 1;
  if (y_kind == 2) {
    __nv_fp8_e4m3* y8 = static_cast<__nv_fp8_e4m3*>(y);
    if (x_f32) cast_frames_kernel<<<blocks, 256, 0, s>>>(xf, x_T_alloc, y8, y_T_alloc, T, frame_elems, n, fault);
    else cast_frames_kernel<<<blocks, 256, 0, s>>>(xb, x_T_alloc, y8, y_T_alloc, T, frame_elems, n, fault);
    return cudaGetLastError();
  }
  if (x_f32 && y_f32) cast_frames_kernel<<<blocks, 256, 0, s>>>(xf, x_T_alloc, static_cast<float*>(y), y_T_alloc, T, frame_elems, n, fault);
  else if (x_f32) cast_frames_kernel<<<blocks, 256, 0, s>>>(xf, x_T_alloc, static_cast<__nv_bfloat16*>(y), y_T_alloc, T, frame_elems, n, fault);
  else if (y_f32) cast_frames_kernel<<<blocks, 256, 0, s>>>(xb, x_T_alloc, static_cast<float*>(y), y_T_alloc, T, frame_elems, n, fault);
  else cast_frames_kernel<<<blocks, 256, 0, s>>>(xb, x_T_alloc, static_cast<__nv_bfloat16*>(y), y_T_alloc, T, frame_elems, n, fault);
  return cudaGetLastError();
}

// [batch, rows, cols] -> [batch, cols, ld] with ld = rows rounded up to 64 (zero padded)
__global__ void transpose_kernel(const __nv_bfloat16* in, __nv_bfloat16* out, int rows, int cols, int ld) {
  __shared__ __nv_bfloat16 tile[32][33];
  const int bz = blockIdx.z;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const __nv_bfloat16* ib = in + static_cast<int64_t>(bz) * rows * cols;
  __nv_bfloat16* ob = out + static_cast<int64_t>(bz) * cols * ld;
  for (int k = threadIdx.y; k < 32; k += blockDim.y) {
    const int r = r0 + k, c = c0 + threadIdx.x;
    tile[k][threadIdx.x] = (r < rows && c < cols) ? ib[static_cast<int64_t>(r) * cols + c] : f2bf(0.f);
  }
  __syncthreads();
  for (int k = threadIdx.y; k < 32; k += blockDim.y) {
    const int c = c0 + k, r = r0 + threadIdx.x;
    if (c < cols && r < ld) ob[static_cast<int64_t>(c) * ld + r] = tile[threadIdx.x][k];
  }
}

cudaError_t launch_transpose_bf16(const void* in, void* out, int batch, int rows, int cols, cudaStream_t s) {
  const int ld = (rows + 63) / 64 * 64;
  dim3 grid((cols + 31) / 32, (ld + 31) / 32, batch);
  transpose_kernel<<<grid, dim3(32, 8), 0, s>>>(static_cast<const __nv_bfloat16*>(in), static_cast<__nv_bfloat16*>(out),
                                                rows, cols, ld);
  return cudaGetLastError();
}

// ============================================================================ encoder layouts
template <typename TO>
__global__ void pixels_to_cl_kernel(const float* v, int B, int C, int T, int H, int W, int ph, int pw, int h0, int nh,
                                    int w0, int nw, int C_pad, TO* y, int yTa, uint32_t* fault) {
  const int64_t n = static_cast<int64_t>(B) * T * nh * nw * C_pad;
  const int Cf = C * ph * pw;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int k = static_cast<int>(i % C_pad);
    int64_t r = i / C_pad;
    const int xx = static_cast<int>(r % nw);
    r /= nw;
    const int yy = static_cast<int>(r % nh);
    r /= nh;
    const int t = static_cast<int>(r % T);
    const int b = static_cast<int>(r / T);
    float val = 0.f;
    if (k < Cf) {
      const int c = k / (ph * pw), dy = (k / pw) % ph, dx = k % pw;
      val = v[((static_cast<int64_t>(b) * C + c) * T + t) * H * static_cast<int64_t>(W) +
              static_cast<int64_t>((h0 + yy) * ph + dy) * W + (w0 + xx) * pw + dx];
    }
    if (sizeof(TO) == 1 && !(fabsf(val) <= 448.f)) raise_fault(fault, FAULT_RANGE, 24);
    y[(((static_cast<int64_t>(b) * yTa + t) * nh + yy) * nw + xx) * C_pad + k] = from_f<TO>(val);
  }
}

// pw == 4, C_pad == 64: one thread per output pixel: C*ph float4 reads (the 4 adjacent pixels of one
// (c, dy); consecutive threads take consecutive output columns, so every read is coalesced) and the
// whole 64-channel pixel written as 16-byte vectors (consecutive threads, consecutive pixels)
template <typename TO>
__global__ void pixels_to_cl64_kernel(const float* v, int B, int C, int T, int H, int W, int ph, int h0, int nh, int w0,
                                      int nw, TO* y, int yTa, uint32_t* fault) {
  const int runs = C * ph;  // (c, dy) pairs, <= 16
  const int64_t n = static_cast<int64_t>(B) * T * nh * nw;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int xx = static_cast<int>(i % nw);
    int64_t r = i / nw;
    const int yy = static_cast<int>(r % nh);
    r /= nh;
    const int t = static_cast<int>(r % T);
    const int b = static_cast<int>(r / T);
    float o[64];
#pragma unroll
    for (int g = 0; g < 16; ++g) {
      float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
      if (g < runs) {
        const int c = g / ph, dy = g - (g / ph) * ph;
        q = *reinterpret_cast<const float4*>(v + ((static_cast<int64_t>(b) * C + c) * T + t) * H * static_cast<int64_t>(W) +
                                             static_cast<int64_t>((h0 + yy) * ph + dy) * W +
                                             static_cast<int64_t>(w0 + xx) * 4);
      }
      o[4 * g] = q.x; o[4 * g + 1] = q.y; o[4 * g + 2] = q.z; o[4 * g + 3] = q.w;
    }
    TO* dst = y + (((static_cast<int64_t>(b) * yTa + t) * nh + yy) * nw + xx) * 64;
#pragma unroll
    for (int k = 0; k < 64; k += 8) vstore8(dst + k, o + k, fault);
  }
}

cudaError_t launch_pixels_to_cl(const float* v, int B, int C, int T, int H, int W, int ph, int pw, int h0, int nh,
                                int w0, int nw, int C_pad, void* y, int y_kind, int y_T_alloc, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(B) * T * nh * nw * C_pad;
  if (n <= 0) return cudaSuccess;
  if (pw == 4 && C_pad == 64 && C * ph <= 16 && W % 4 == 0 && (reinterpret_cast<uintptr_t>(v) & 15u) == 0) {
    const int64_t np = static_cast<int64_t>(B) * T * nh * nw;
    const int blocks4 = static_cast<int>(std::min<int64_t>((np + 255) / 256, 152 * 16));
    uint32_t* f4 = fault_word();
    if (y_kind == 1)
      pixels_to_cl64_kernel<<<blocks4, 256, 0, s>>>(v, B, C, T, H, W, ph, h0, nh, w0, nw, static_cast<float*>(y),
                                                    y_T_alloc, f4);
    else if (y_kind == 2)
      pixels_to_cl64_kernel<<<blocks4, 256, 0, s>>>(v, B, C, T, H, W, ph, h0, nh, w0, nw,
                                                    static_cast<__nv_fp8_e4m3*>(y), y_T_alloc, f4);
    else
      pixels_to_cl64_kernel<<<blocks4, 256, 0, s>>>(v, B, C, T, H, W, ph, h0, nh, w0, nw,
                                                    static_cast<__nv_bfloat16*>(y), y_T_alloc, f4);
    return cudaGetLastError();
  }
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 152 * 64));
  uint32_t* f = fault_word();
  if (y_kind == 1)
    pixels_to_cl_kernel<<<blocks, 256, 0, s>>>(v, B, C, T, H, W, ph, pw, h0, nh, w0, nw, C_pad, static_cast<float*>(y),
                                               y_T_alloc, f);
  else if (y_kind == 2)
    pixels_to_cl_kernel<<<blocks, 256, 0, s>>>(v, B, C, T, H, W, ph, pw, h0, nh, w0, nw, C_pad,
                                               static_cast<__nv_fp8_e4m3*>(y), y_T_alloc, f);
  else
    pixels_to_cl_kernel<<<blocks, 256, 0, s>>>(v, B, C, T, H, W, ph, pw, h0, nh, w0, nw, C_pad,
                                               static_cast<__nv_bfloat16*>(y), y_T_alloc, f);
  return cudaGetLastError();
}

// one thread per output element (consecutive threads write consecutive channels)
template <typename TI, typename TO>
__global__ void fold_frames_kernel(const TI* x, int xTa, int B, int T, int H, int W, int C, int st, int sh, int sw,
                                   TO* y, int yTa, uint32_t* fault) {
  const int S = st * sh * sw;
  const int To = (T + st - 1) / st, Ho = H / sh, Wo = W / sw, Co = C * S;
  const int64_t n = static_cast<int64_t>(B) * To * Ho * Wo * Co;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int k = static_cast<int>(i % Co);
    int64_t r = i / Co;
    const int xo = static_cast<int>(r % Wo);
    r /= Wo;
    const int yo = static_cast<int>(r % Ho);
    r /= Ho;
    const int to = static_cast<int>(r % To);
    const int b = static_cast<int>(r / To);
    const int c = k / S, sub = k - (k / S) * S;
    const int dt = sub / (sh * sw), dy = (sub / sw) % sh, dx = sub % sw;
    const int ti = max(st * to + dt - (st - 1), 0);
    const float val =
        to_f<TI>(x[(((static_cast<int64_t>(b) * xTa + ti) * H + (sh * yo + dy)) * W + (sw * xo + dx)) * C + c]);
    if (sizeof(TO) == 1 && !(fabsf(val) <= 448.f)) raise_fault(fault, FAULT_RANGE, 25);
    y[(((static_cast<int64_t>(b) * yTa + to) * Ho + yo) * Wo + xo) * Co + k] = from_f<TO>(val);
  }
}

// 4 consecutive input channels as floats (one 16- or 8-byte load)
VAE_DEV void load4f(const float* p, float* v) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
VAE_DEV void load4f(const __nv_bfloat16* p, float* v) {
  const uint2 a = *reinterpret_cast<const uint2*>(p);
  const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a.x));
  const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a.y));
  v[0] = lo.x; v[1] = lo.y; v[2] = hi.x; v[3] = hi.y;
}

// one thread per (output pixel, run of 4 input channels c0..c0+3): S vector reads (one per sub-position,
// consecutive threads reading consecutive channels of the same input pixel) and one contiguous run of
// 4*S output channels c*S + sub written as 16-byte vectors; 32-bit index arithmetic once per thread
template <typename TI, typename TO, int S>
__global__ void fold_frames_v_kernel(const TI* x, int xTa, int B, int T, int H, int W, int C, int st, int sh, int sw,
                                     TO* y, int yTa, uint32_t* fault) {
  constexpr int CPT = 4;
  const int To = (T + st - 1) / st, Ho = H / sh, Wo = W / sw;
  const int team = C / CPT;
  const int n = B * To * Ho * Wo * team;  // < 2^30 (the launcher checks)
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int j = i % team;
    int r = i / team;
    const int xo = r % Wo;
    r /= Wo;
    const int yo = r % Ho;
    r /= Ho;
    const int to = r % To;
    const int b = r / To;
    const int c0 = j * CPT;
    float v[S][CPT];
#pragma unroll
    for (int sub = 0; sub < S; ++sub) {
      const int dt = sub / (sh * sw), dy = (sub / sw) % sh, dx = sub % sw;
      const int ti = max(st * to + dt - (st - 1), 0);
      load4f(x + ((static_cast<int64_t>(b) * xTa + ti) * H + (sh * yo + dy)) * static_cast<int64_t>(W) * C +
                 static_cast<int64_t>(sw * xo + dx) * C + c0,
             v[sub]);
    }
    float o[CPT * S];
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc)
#pragma unroll
      for (int sub = 0; sub < S; ++sub) o[cc * S + sub] = v[sub][cc];
    TO* dst = y + (((static_cast<int64_t>(b) * yTa + to) * Ho + yo) * Wo + xo) * static_cast<int64_t>(C) * S +
              static_cast<int64_t>(c0) * S;
#pragma unroll
    for (int q = 0; q < CPT * S; q += 8) vstore8(dst + q, o + q, fault);
  }
}

cudaError_t launch_fold_frames(const void* x, int x_f32, int x_T_alloc, int B, int T, int H, int W, int C, int st,
                               int sh, int sw, void* y, int y_kind, int y_T_alloc, cudaStream_t s) {
  if (st < 1 || sh < 1 || sw < 1 || H % sh || W % sw) return cudaErrorInvalidValue;
  const int S = st * sh * sw;
  const int64_t nv = static_cast<int64_t>(B) * ((T + st - 1) / st) * (H / sh) * (W / sw) * (C / 4);
  if ((S == 4 || S == 8) && C % 4 == 0 && nv < (1LL << 30)) {
    if (nv <= 0) return cudaSuccess;
    const int bl = static_cast<int>(std::min<int64_t>((nv + 255) / 256, 152 * 16));
    uint32_t* fs = fault_word();
#define VAE_FOLDV(TI, TO, SS)                                                                                       \
  fold_frames_v_kernel<TI, TO, SS><<<bl, 256, 0, s>>>(static_cast<const TI*>(x), x_T_alloc, B, T, H, W, C, st, sh, sw, \
                                                      static_cast<TO*>(y), y_T_alloc, fs)
#define VAE_FOLDV_T(TI, SS)                                   \
  if (y_kind == 1) VAE_FOLDV(TI, float, SS);                  \
  else if (y_kind == 2) VAE_FOLDV(TI, __nv_fp8_e4m3, SS);     \
  else VAE_FOLDV(TI, __nv_bfloat16, SS);
    if (x_f32) {
      if (S == 4) { VAE_FOLDV_T(float, 4) } else { VAE_FOLDV_T(float, 8) }
    } else {
      if (S == 4) { VAE_FOLDV_T(__nv_bfloat16, 4) } else { VAE_FOLDV_T(__nv_bfloat16, 8) }
    }
#undef VAE_FOLDV_T
#undef VAE_FOLDV
    return cudaGetLastError();
  }
  const int64_t n = static_cast<int64_t>(B) * ((T + st - 1) / st) * (H / sh) * (W / sw) * C * st * sh * sw;
  if (n <= 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 152 * 64));
  uint32_t* f = fault_word();
#define VAE_FOLD(TI, TO)                                                                                          \
  fold_frames_kernel<<<blocks, 256, 0, s>>>(static_cast<const TI*>(x), x_T_alloc, B, T, H, W, C, st, sh, sw,       \
                                            static_cast<TO*>(y), y_T_alloc, f)
  if (x_f32) {
    if (y_kind == 1) VAE_FOLD(float, float);
    else if (y_kind == 2) VAE_FOLD(float, __nv_fp8_e4m3);
    else VAE_FOLD(float, __nv_bfloat16);
  } else {
    if (y_kind == 1) VAE_FOLD(__nv_bfloat16, float);
    else if (y_kind == 2) VAE_FOLD(__nv_bfloat16, __nv_fp8_e4m3);
    else VAE_FOLD(__nv_bfloat16, __nv_bfloat16);
  }
#undef VAE_FOLD
  return cudaGetLastError();
}

__global__ void stride2_weights_kernel(const float* w, int C_out, int C_in, float* out) {
  const int64_t n = static_cast<int64_t>(C_out) * 4 * C_in * 27;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int tap = static_cast<int>(i % 27);
    const int k = static_cast<int>((i / 27) % (4 * C_in));
    const int o = static_cast<int>(i / (27LL * 4 * C_in));
    const int kt = tap / 9, kh = (tap / 3) % 3, kw = tap % 3;
    const int c = k / 4, dy = (k / 2) % 2, dx = k % 2;
    const int sy = 2 * (kh - 1) + dy, sx = 2 * (kw - 1) + dx;
    float val = 0.f;
    if (kt == 2 && kh >= 1 && kw >= 1 && sy <= 2 && sx <= 2) val = w[((static_cast<int64_t>(o) * C_in + c) * 3 + sy) * 3 + sx];
    out[i] = val;
  }
}

cudaError_t launch_stride2_weights(const float* w, int C_out, int C_in, float* out, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(C_out) * 4 * C_in * 27;
  if (n <= 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 152 * 64));
  stride2_weights_kernel<<<blocks, 256, 0, s>>>(w, C_out, C_in, out);
  return cudaGetLastError();
}

// ============================================================================ weight packing
// bf16 K-major [N_pad, 27 * C_in_pad]; row n' = sub * (C_out/S) + c holds PyTorch channel c * S + sub
// (natural: row n' holds channel n', for convs that store NCTHW pixels)
// The tf32 high part of an fp32 value: its 13 low mantissa bits cleared (so whatever a tf32 consumer does
// with those bits, it sees exactly this value); the remainder x - hi is exact in fp32.
VAE_DEV float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xffffe000u); }

__global__ void pack_tf32_kernel(const float* w, int C_out, int C_in, int C_in_pad, int N_pad, int S, int natural,
                                 float* out) {
  const int64_t n = static_cast<int64_t>(N_pad) * 27 * C_in_pad;
  const int Cd = C_out / S;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int ci = static_cast<int>(i % C_in_pad);
    const int tap = static_cast<int>((i / C_in_pad) % 27);
    const int np = static_cast<int>(i / (27LL * C_in_pad));
    float v = 0.f;
    if (np < C_out && ci < C_in) {
      const int sub = np / Cd, c = np % Cd;
      const int co = natural ? np : c * S + sub;
      v = w[(static_cast<int64_t>(co) * C_in + ci) * 27 + tap];
    }
    const float hi = tf32_hi(v);
    out[i] = hi;
    out[n + i] = v - hi;
  }
}

cudaError_t launch_pack_weights_tf32(const float* w, int C_out, int C_in, int C_in_pad, int N_pad, int S, void* out,
                                     cudaStream_t s, int natural) {
  const int64_t n = static_cast<int64_t>(N_pad) * 27 * C_in_pad;
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 152 * 64));
  pack_tf32_kernel<<<blocks, 256, 0, s>>>(w, C_out, C_in, C_in_pad, N_pad, S, natural, static_cast<float*>(out));
  return cudaGetLastError();
}

// 4 elements per thread (n % 4 == 0, 16-byte aligned arrays) or one
__global__ void split_tf32_kernel(const float* x, float* hi, float* lo, int64_t n) {
  const int64_t n4 = (n % 4 == 0) ? n / 4 : 0;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 v = reinterpret_cast<const float4*>(x)[i];
    const float4 h = make_float4(tf32_hi(v.x), tf32_hi(v.y), tf32_hi(v.z), tf32_hi(v.w));
    reinterpret_cast<float4*>(hi)[i] = h;
    reinterpret_cast<float4*>(lo)[i] = make_float4(v.x - h.x, v.y - h.y, v.z - h.z, v.w - h.w);
  }
  if (n4 == 0)
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      const float h = tf32_hi(x[i]);
      hi[i] = h;
      lo[i] = x[i] - h;
    }
}

cudaError_t launch_split_tf32(const float* x, float* hi, float* lo, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const bool vec = n % 4 == 0 && (reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(hi) |
                                  reinterpret_cast<uintptr_t>(lo)) % 16 == 0;
  if (!vec && n % 4 == 0) return cudaErrorMisalignedAddress;
  const int64_t work = n % 4 == 0 ? n / 4 : n;
  const int blocks = static_cast<int>(std::min<int64_t>((work + 255) / 256, 152 * 16));
  split_tf32_kernel<<<blocks, 256, 0, s>>>(x, hi, lo, n);
  return cudaGetLastError();
}

__global__ void pack_bf16_kernel(const float* w, int C_out, int C_in, int C_in_pad, int N_pad, int S, int natural,
                                 __nv_bfloat16* out) {
  const int64_t n = static_cast<int64_t>(N_pad) * 27 * C_in_pad;
  const int Cd = C_out / S;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int ci = static_cast<int>(i % C_in_pad);
    const int tap = static_cast<int>((i / C_in_pad) % 27);
    const int np = static_cast<int>(i / (27LL * C_in_pad));
    float v = 0.f;
    if (np < C_out && ci < C_in) {
      const int sub = np / Cd, c = np % Cd;
      const int co = natural ? np : c * S + sub;
      v = w[(static_cast<int64_t>(co) * C_in + ci) * 27 + tap];
    }
    out[i] = f2bf(v);
  }
}

// tap-stacked packing of a narrow conv: [3 kt][kTapRows][C_in_pad], row (kh*3 + kw) * kTapMaxN + np
__global__ void pack_tap_bf16_kernel(const float* w, int C_out, int C_in, int C_in_pad, int S, int natural,
                                     __nv_bfloat16* out) {
  const int64_t n = 3LL * kTapRows * C_in_pad;
  const int Cd = C_out / S;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int ci = static_cast<int>(i % C_in_pad);
    const int row = static_cast<int>((i / C_in_pad) % kTapRows);
    const int kt = static_cast<int>(i / (static_cast<int64_t>(kTapRows) * C_in_pad));
    const int t9 = row / kTapMaxN, np = row % kTapMaxN;
    float v = 0.f;
    if (t9 < 9 && np < C_out && ci < C_in) {
      const int sub = np / Cd, c = np % Cd;
      const int co = natural ? np : c * S + sub;
      v = w[(static_cast<int64_t>(co) * C_in + ci) * 27 + kt * 9 + t9];
    }
    out[i] = f2bf(v);
  }
}

cudaError_t launch_pack_weights_bf16(const float* w, int C_out, int C_in, int C_in_pad, int N_pad, int S, void* out,
                                     cudaStream_t s, int natural, int tap_stacked) {
  if (tap_stacked) {
    if (C_out > kTapMaxN) return cudaErrorInvalidValue;
    const int64_t n = 3LL * kTapRows * C_in_pad;
    const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 152 * 64));
    pack_tap_bf16_kernel<<<blocks, 256, 0, s>>>(w, C_out, C_in, C_in_pad, S, natural, static_cast<__nv_bfloat16*>(out));
    return cudaGetLastError();
  }
  const int64_t n = static_cast<int64_t>(N_pad) * 27 * C_in_pad;
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 152 * 64));
  pack_bf16_kernel<<<blocks, 256, 0, s>>>(w, C_out, C_in, C_in_pad, N_pad, S, natural,
                                          static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

// e4m3 K-major [N_pad, 27 * C_in_pad] with the bf16 packing's row order; one block per packed row: the
// row's scale is max|w| / 448 (1 for an all-zero or padding row), its bytes round w / scale to nearest
// even.  The scales follow the bytes at fp8_scale_offset().
size_t fp8_scale_offset(int N_pad, int C_in_pad) {
  return (static_cast<size_t>(N_pad) * 27 * C_in_pad + 255) & ~size_t(255);
}

__global__ void __launch_bounds__(256) pack_fp8_kernel(const float* w, int C_out, int C_in, int C_in_pad, int S,
                                                        int natural, __nv_fp8_e4m3* out, float* scales) {
  __shared__ float red[8];
  const int np = blockIdx.x;
  const int Cd = C_out / S;
  const int64_t K = 27LL * C_in_pad;
  const bool real = np < C_out;
  const int co = real ? (natural ? np : (np % Cd) * S + np / Cd) : 0;
  const float* wr = w + static_cast<int64_t>(co) * C_in * 27;  // [C_in, 27] of output channel co
  float m = 0.f;
  if (real)
    for (int64_t i = threadIdx.x; i < 27LL * C_in; i += blockDim.x) m = fmaxf(m, fabsf(wr[i]));
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.f;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
  const float scale = m > 0.f ? m / 448.f : 1.f;
  if (threadIdx.x == 0) scales[np] = scale;
  for (int64_t i = threadIdx.x; i < K; i += blockDim.x) {
    const int ci = static_cast<int>(i % C_in_pad);
    const int tap = static_cast<int>(i / C_in_pad);
    const float v = (real && ci < C_in) ? wr[static_cast<int64_t>(ci) * 27 + tap] / scale : 0.f;
    out[static_cast<int64_t>(np) * K + i] = from_f<__nv_fp8_e4m3>(fminf(fmaxf(v, -448.f), 448.f));
  }
}

cudaError_t launch_pack_weights_fp8(const float* w, int C_out, int C_in, int C_in_pad, int N_pad, int S, void* out,
                                    cudaStream_t s, int natural) {
  if (N_pad <= 0) return cudaSuccess;
  pack_fp8_kernel<<<N_pad, 256, 0, s>>>(w, C_out, C_in, C_in_pad, S, natural, static_cast<__nv_fp8_e4m3*>(out),
                                        reinterpret_cast<float*>(static_cast<char*>(out) + fp8_scale_offset(N_pad, C_in_pad)));
  return cudaGetLastError();
}

// fp32 [27, C_in, C_out] (PyTorch channel order)
__global__ void pack_f32_kernel(const float* w, int C_out, int C_in, float* out) {
  const int64_t n = 27LL * C_in * C_out;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int co = static_cast<int>(i % C_out);
    const int ci = static_cast<int>((i / C_out) % C_in);
    const int tap = static_cast<int>(i / (static_cast<int64_t>(C_out) * C_in));
    out[i] = w[(static_cast<int64_t>(co) * C_in + ci) * 27 + tap];
  }
}

cudaError_t launch_pack_weights_f32(const float* w, int C_out, int C_in, void* out, cudaStream_t s) {
  const int64_t n = 27LL * C_in * C_out;
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 152 * 64));
  pack_f32_kernel<<<blocks, 256, 0, s>>>(w, C_out, C_in, static_cast<float*>(out));
  return cudaGetLastError();
}

__global__ void to_bf16_kernel(const float* w, int64_t n, __nv_bfloat16* out) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[i] = f2bf(w[i]);
}

cudaError_t launch_pack_matrix_bf16(const float* w, int rows, int cols, void* out, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(rows) * cols;
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 152 * 64));
  to_bf16_kernel<<<blocks, 256, 0, s>>>(w, n, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

// ============================================================================ watchdog self-test
__global__ void watchdog_kernel(uint32_t* fault, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, fault, limit_ns, 99);  // nothing ever arrives
  __syncthreads();
}

cudaError_t launch_watchdog_test(uint64_t limit_ns, cudaStream_t s) {
  watchdog_kernel<<<1, 32, 0, s>>>(fault_word(), limit_ns);
  return cudaGetLastError();
}

}  // namespace vae
