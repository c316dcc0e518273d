// Internal launcher interface shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/vaedec.h"

namespace vae {

constexpr int kMaxP = VAE_MAX_PATCHES;

// Device fault word of the current device (4 x u32, see common.cuh).
uint32_t* fault_word();
// Default bound of every in-kernel wait, nanoseconds.
uint64_t wait_limit_ns();

// Tensor-core (tcgen05) convolution / GEMM.  All pointers device.
struct ConvTcArgs {
  int mode;  // 0 = causal conv3d (implicit GEMM over 27 taps), 1 = batched GEMM
  // conv geometry
  int B, T, H, W;       // output frames / rows / cols before depth-to-space
  int C_in_pad;         // channels of x (multiple of 64)
  int T_in;             // frames readable from x (T + cache_frames)
  int x_T_alloc;        // frames between consecutive batch items of x (>= T_in)
  int cache_frames;     // 0 or 2
  int nph, npw;
  const int* ph_edges;  // host arrays nph+1 / npw+1
  const int* pw_edges;
  // gemm geometry
  int M, K, batch;
  int64_t stride_a, stride_b, stride_d;
  float alpha;
  // operands
  const void* x;        // conv: x channels-last bf16; gemm: A
  const void* w;        // conv: packed weights bf16 [N_pad, 27*C_in_pad]; gemm: B [N, K]
  int N_real, N_pad;
  const float* bias;    // conv: PyTorch channel order (index c*S + sub); gemm: [N]
  const void* residual; int res_f32; int res_T_alloc;  // residual [B, res_T_alloc, H, W, N] (0 = T)
  void* y; int out_f32; int out_ncthw; int y_T_alloc;    // y frames per batch item (0 = T_out)
  int64_t ldd;                                           // gemm: row stride of D (0 = N_real)
  int d2s_t, d2s_h, d2s_w, drop_first;
  // fused group-norm statistics of y (nullptr = none): exact per-patch sums, see norm.cu
  void* gn_partials; int gn_groups;
  // optional second copy of y (channels-last, y2_T_alloc frames per batch item): bf16, or e4m3 with y2_fp8
  void* y2; int y2_T_alloc; int y2_fp8;
  // conv mode, e4m3 operands: x and w hold e4m3 bytes (C_in_pad a multiple of 128) and the product of
  // output channel n (packed row order) is multiplied by wscale[n] (its weights' scale)
  int fp8; const float* wscale;
  // weight rows in PyTorch channel order (packed with natural != 0); required for NCTHW outputs
  int natural;
  // conv mode, weights packed tap-stacked (see kTapRows): all 9 spatial taps in one MMA
  int tap_stacked;
  // conv mode, fp32 operands as 3 x TF32 products (kind::tf32): x holds the tf32 high parts of the
  // fp32 input and x_lo the remainders (same layout); w holds [2][N_pad][27 * C_in_pad] fp32 (high
  // parts, then remainders); each product is a_hi b_hi + a_hi b_lo + a_lo b_hi; C_in_pad % 32 == 0
  int tf32;
  const void* x_lo;
};

// Narrow bf16 convs (at most kTapMaxN output channels) pack their weights tap-stacked: for each temporal
// tap kt one K-major tile of kTapRows rows, row (kh*3 + kw) * kTapMaxN + n holding output column n of
// spatial tap (kh, kw) (zero rows beyond 9 * kTapMaxN and beyond the real columns): [3][kTapRows][C_in_pad].
constexpr int kTapMaxN = 12;
constexpr int kTapRows = 112;  // 9 * 12 = 108 rounded up to a multiple of 16
inline bool conv_tap_stacked(int N_real, int fp8) { return !fp8 && N_real <= kTapMaxN; }
cudaError_t launch_conv_tc(const ConvTcArgs& a, cudaStream_t s);

// CUDA-core convolution (any channel count, fp32 or bf16 storage, fp32 accumulation).
struct ConvSimtArgs {
  int B, T, H, W, C_in, C_out, T_in, x_T_alloc, cache_frames;
  const void* x; int x_f32;
  const float* w;  // [27, C_in, C_out] fp32
  const float* bias;
  const void* residual; int res_f32; int res_T_alloc;
  void* y; int out_f32; int out_ncthw; int y_T_alloc;
  int d2s_t, d2s_h, d2s_w, drop_first;
  int nph, npw; const int* ph_edges; const int* pw_edges;
};
cudaError_t launch_conv_simt(const ConvSimtArgs& a, cudaStream_t s);

// Weight packing.  Rows are ordered (depth-to-space sub-position, channel) so that a 32-column epilogue
// chunk is 32 channels of one sub-position; natural != 0 keeps PyTorch's channel order (c*S + sub),
// which convs storing NCTHW pixels use (a chunk then holds whole runs of horizontally adjacent pixels).
cudaError_t launch_pack_weights_bf16(const float* w, int C_out, int C_in, int C_in_pad, int N_pad, int S,
                                     void* out, cudaStream_t s, int natural = 0, int tap_stacked = 0);
cudaError_t launch_pack_weights_f32(const float* w, int C_out, int C_in, void* out, cudaStream_t s);
// fp32 weights for the 3 x TF32 conv: the bf16 packing's rows, K-major fp32 [2][N_pad][27 * C_in_pad]:
// high parts (the fp32 value with its 13 low mantissa bits cleared), then the exact remainders.
cudaError_t launch_pack_weights_tf32(const float* w, int C_out, int C_in, int C_in_pad, int N_pad, int S, void* out,
                                     cudaStream_t s, int natural = 0);
// x = hi + lo exactly, hi = x with its 13 low mantissa bits cleared (a tf32 value), n elements.
cudaError_t launch_split_tf32(const float* x, float* hi, float* lo, int64_t n, cudaStream_t s);
cudaError_t launch_pack_matrix_bf16(const float* w, int rows, int cols, void* out, cudaStream_t s);
// e4m3 K-major [N_pad, 27 * C_in_pad] (rows as the bf16 packing), each row scaled by its own
// scale = max|w| / 448, followed at fp8_scale_offset() bytes by the float scales [N_pad].
size_t fp8_scale_offset(int N_pad, int C_in_pad);
cudaError_t launch_pack_weights_fp8(const float* w, int C_out, int C_in, int C_in_pad, int N_pad, int S, void* out,
                                    cudaStream_t s, int natural = 0);

// Group norm.
struct GnArgs {
  int B, T, H, W, C, groups;
  float eps;
  int silu;
  int nph, npw; const int* ph_edges; const int* pw_edges;
  const void* x; int x_f32; int x_T_alloc;  // frames per batch item in memory (0 = T)
  void* y; int y_f32; int y_T_alloc;
  int y_fp8;               // y holds e4m3 conv operands (round to nearest, |y| > 448 flags VAE_ERR_RANGE)
  const float* gamma; const float* beta;
  void* partials;          // gn_workspace_bytes: [nph*npw, B, T, groups] GnPartial, then [B*T, C] float2
};
size_t gn_partials_bytes(int nph, int npw, int B, int T, int groups);
// partials followed (256-aligned) by the per-(frame, channel) affine of the finalize step
size_t gn_workspace_bytes(int nph, int npw, int B, int T, int groups, int C);
cudaError_t launch_gn_stats(const GnArgs& a, cudaStream_t s);  // clears and fills partials
cudaError_t launch_gn_apply(const GnArgs& a, cudaStream_t s);
// Channel RMS norm (+ SiLU when a.silu) per pixel; uses B..C, eps, silu, x*, y*, gamma, beta of a.
bool rms_supported(int C);
cudaError_t launch_rms(const GnArgs& a, cudaStream_t s);

// Layout helpers.
// Latent box [B, C, t0:t0+nt, h0:h0+nh, w0:w0+nw] of an NCTHW fp32 tensor [B, C, T, H, W] ->
// channels-last [B, y_T_alloc, nh, nw, C_pad] (frames 0..nt-1 of each batch item), zero channels >= C.
cudaError_t launch_latent_to_cl(const float* z, int B, int C, int T, int H, int W, int t0, int nt, int h0, int nh, int w0,
                                int nw, int C_pad, void* y, int y_f32, int y_T_alloc, cudaStream_t s);
cudaError_t launch_d2s(const void* x, void* y, int B, int T, int H, int W, int C, int st, int sh, int sw,
                       int drop_first, int f32, cudaStream_t s);
// Pixels NCTHW fp32 [B, C, T, H, W] -> channels-last [B, y_T_alloc, nh, nw, C_pad] (frames 0..T-1) of
// the space-to-depth box (h0, nh, w0, nw in folded units) with fold (1, ph, pw): channel
// c*ph*pw + dy*pw + dx <- pixel (c, t, ph*(h0+y)+dy, pw*(w0+x)+dx); channels >= C*ph*pw are 0.
// y_kind: 0 bf16, 1 fp32, 2 e4m3.
cudaError_t launch_pixels_to_cl(const float* v, int B, int C, int T, int H, int W, int ph, int pw, int h0, int nh,
                                int w0, int nw, int C_pad, void* y, int y_kind, int y_T_alloc, cudaStream_t s);
// Causal space-to-depth of a channels-last tensor [B, x_T_alloc, H, W, C] (frames 0..T-1) into
// [B, y_T_alloc, H/sh, W/sw, C*st*sh*sw]: channel c*S + dt*sh*sw + dy*sw + dx of output frame t' <- input
// (max(st*t' + dt - (st-1), 0), sh*y+dy, sw*x+dx, c); (T + st - 1) / st output frames.
cudaError_t launch_fold_frames(const void* x, int x_f32, int x_T_alloc, int B, int T, int H, int W, int C, int st,
                               int sh, int sw, void* y, int y_kind, int y_T_alloc, cudaStream_t s);
// The stride-2 down-sampler's weights w [C_out, C_in, 3, 3] as a stride-1 3x3x3 causal conv over the
// (1,2,2)-folded input: out [C_out, 4*C_in, 3, 3, 3] with out[o, c*4 + dy*2 + dx, 2, kh, kw] =
// w[o, c, 2(kh-1)+dy, 2(kw-1)+dx] for kh, kw >= 1 where that index is <= 2, and 0 elsewhere.
cudaError_t launch_stride2_weights(const float* w, int C_out, int C_in, float* out, cudaStream_t s);
cudaError_t launch_copy_frames(const void* src, int src_T, int src_t0, void* dst, int dst_T, int dst_t0, int n_frames,
                               int B, int64_t frame_bytes, cudaStream_t s);

// Tile blend.
cudaError_t launch_blend(const void* const* tiles, const vae_tile_t* meta, int n_tiles, void* out,
                         const vae_blend_desc_t& d, cudaStream_t s);

// CUDA-core batched GEMM (fp32 storage): D[b] = alpha * A[b] B[b]^T + bias[n] + residual, with
// B element (n, k) at B + n*ldb_n + k*ldb_k.  A [M, K] row-major, D/residual [M, N] row-major.
cudaError_t launch_gemm_simt(const float* A, const float* Bm, float* D, const float* bias, const float* residual,
                             int M, int N, int K, int batch, int64_t sa, int64_t sb, int64_t sd, int64_t ldb_n,
                             int64_t ldb_k, float alpha, cudaStream_t s);
// Cast / copy a channels-last tensor between frame layouts and dtypes (y_kind: 0 bf16, 1 fp32, 2 e4m3).
cudaError_t launch_cast_frames(const void* x, int x_f32, int x_T_alloc, void* y, int y_kind, int y_T_alloc, int B, int T,
                               int64_t frame_elems, cudaStream_t s);

// Softmax over rows of an fp32 matrix, written as bf16 (attention probabilities).
cudaError_t launch_softmax_rows(const float* s_in, void* p_out, int p_f32, int rows, int cols, int ld_out, cudaStream_t s);
// Channels-last bf16 [N, C] -> transposed copy [C, N] (per batch).
cudaError_t launch_transpose_bf16(const void* in, void* out, int batch, int rows, int cols, cudaStream_t s);

cudaError_t launch_watchdog_test(uint64_t limit_ns, cudaStream_t s);

// Op-level error reporting (records the message for vae_last_error(NULL, ...)) and the group-norm
// descriptor checks shared by the group-norm entry points.
vae_status_t op_error(vae_status_t code, const char* msg);
vae_status_t validate_gn_desc(const void* x, const void* y, const vae_gn_desc_t* d);

}  // namespace vae
