/*
 * vaedec.h -- C ABI of the GB300 (sm_103a) patched / tiled causal video-VAE decoder.
 *
 * The library turns a video-diffusion latent [B, C, T, h, w] into pixels [B, 3, T', H, W]
 * through a causal-Conv3d residual decoder.  The decode can be split into spatial patches; each
 * patch is computed by its own thread blocks, reads its halo rows straight from the neighbouring
 * patch, and contributes per-patch partial sums to every group norm.  The patched result equals
 * the unpatched one bit for bit.  Tiled decode with linear overlap blending is also provided.
 *
 * Sources (page titles; the section is given with each entry point):
 *   [DV]  DistVAE PR #14 "Add tiled VAE parallelism & extended model support"
 *   [TP]  TensorRT-LLM PR #15753 "LTX-2 tile-parallel VAE decode"
 *   [WAN] TensorRT-LLM PR #16066 "ParallelVAE_TrtllmWan for native Wan VAE"
 *   [ENC] vllm-omni PR #4831 "VAE tiling parallel encode for LTX-2"
 *
 * Conventions (all entry points):
 *   - Device pointers are CUDA device addresses on the current device, 16-byte aligned, and the
 *     tensors they point at are dense (no strides).  Host pointers are marked "host".
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Every GPU
 *     entry point only enqueues work on `stream` and returns; nothing inside synchronises the host
 *     unless stated.  Results are valid once the stream has reached the call's work.
 *   - The caller owns every buffer it passes.  The library never frees caller memory.
 *   - Errors: arguments are validated on the host before any launch; a call that returns an error
 *     enqueued nothing.  A device-side watchdog (every wait inside a kernel is bounded) records a
 *     fault word instead of hanging; `vae_last_error` synchronises the device and reports it as
 *     VAE_ERR_TIMEOUT or VAE_ERR_RANGE.
 *   - Layouts: "channels-last" means [B, T, H, W, C] with C contiguous (the layout of all
 *     activations, following the channels-last halo fix of [WAN]); "NCTHW" means [B, C, T, H, W]
 *     (the latent and the decoded pixels, PyTorch's Conv3d layout).
 *   - Handles are not thread-safe; separate handles are independent.
 */
#ifndef VAEDEC_H
#define VAEDEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  VAE_OK = 0,
  VAE_ERR_INVALID_ARG = 1,      /* a null pointer, a negative or inconsistent size */
  VAE_ERR_UNSUPPORTED = 2,      /* a configuration this library refuses rather than answers wrongly */
  VAE_ERR_PATCH_TOO_NARROW = 3, /* a patch narrower than the convolution's reach ([DV] narrow-patch commit) */
  VAE_ERR_ALIGNMENT = 4,        /* a pointer that is not 16-byte aligned */
  VAE_ERR_OOM = 5,              /* a library-owned allocation failed */
  VAE_ERR_CUDA = 6,             /* a CUDA runtime call failed */
  VAE_ERR_TIMEOUT = 7,          /* a bounded wait inside a kernel ran out (device watchdog) */
  VAE_ERR_RANGE = 8             /* a group-norm input with |x| >= 8192 (outside the exact-sum range), or an
                                   e4m3 conv operand with |x| > 448 (stored saturated) */
} vae_status_t;

/* Storage / arithmetic types.  VAE_FP8 is e4m3 (1 sign, 4 exponent, 3 mantissa bits; largest finite
 * value 448) for convolution operands, multiplied on the tcgen05 tensor cores (kind::f8f6f4, fp32
 * accumulation); the low-precision conv of [WAN]'s reviewer comment (FP4 conv quantisation with the
 * RMSNorm/SiLU -> quantisation fusion), here at 8 bits.  Weights are e4m3 with one fp32 scale per
 * output channel (max |w| / 448) applied in the conv epilogue; activations are stored unscaled
 * (round to nearest even; a value beyond +-448 is saturated and flags VAE_ERR_RANGE).  As a decoder
 * dtype: the residual blocks' and up-samplers' convs whose input channels are a multiple of 128 take
 * e4m3 operands written by the norm (norm + SiLU -> quantisation in one pass) or by the last residual
 * block's conv epilogue; conv_in, conv_out and attention stay as in bf16 mode, the residual stream and
 * conv1's output are stored in bf16; pixels are bf16.  Accuracy bar against the fp32 oracle: relative L2 <= 0.15 and PSNR >= 35 dB
 * (each e4m3 rounding has unit roundoff 2^-4; the same rounding points emulated in the oracle give
 * relative L2 0.05-0.07 on small decoders and 0.094 on the first frame of the Wan-shaped decode). */
typedef enum { VAE_BF16 = 0, VAE_FP32 = 1, VAE_FP8 = 2, VAE_FP32_TC = 3 } vae_dtype_t;

/* The decoder's norm family.  VAE_NORM_GROUP: per-frame group norm whose statistics span patches
 * ([DV] PatchGroupNorm commit).  VAE_NORM_CHANNEL_RMS: a channel RMS norm per pixel, the norm of the
 * Wan / Qwen-Image, HunyuanVideo 1.5 and LTX-2 decoders, which reduces over channels only and so
 * needs nothing from other patches ([DV] Qwen-Image, HunyuanVideo/1.5 and LTX-2 adapter commits). */
typedef enum { VAE_NORM_GROUP = 0, VAE_NORM_CHANNEL_RMS = 1 } vae_norm_t;

#define VAE_MAX_STAGES 8
#define VAE_MAX_PATCHES 64 /* per axis */
#define VAE_MAX_TILES 512

/* Structured error report: callers need not parse text ([DV] tile-planner commit exposes the row
 * count and processing factor as fields for the same reason). */
typedef struct {
  int code;          /* vae_status_t of the last failure */
  int rows;          /* VAE_ERR_PATCH_TOO_NARROW: rows of the offending patch */
  int factor;        /* VAE_ERR_PATCH_TOO_NARROW: the reach it needed */
  char message[256]; /* human-readable detail */
} vae_error_info_t;

/* ------------------------------------------------------------------------------------------ */
/* Decoder                                                                                     */
/* ------------------------------------------------------------------------------------------ */

/* Architecture of a causal video-VAE decoder ([DV] Wan and LTX-2 adapter commits, [WAN]):
 *   conv_in (latent_c -> stage_c[0]) -> mid_res residual blocks -> [mid attention]
 *   -> per stage i: n_res[i] residual blocks, then (i < n_stages-1) the up-sampling conv
 *      stage_c[i] -> up_t*up_h*up_w*stage_c[i+1] and depth-to-space
 *   -> group norm + SiLU -> conv_out (stage_c[last] -> out_c*out_d2s_t*out_d2s_h*out_d2s_w)
 *   -> final depth-to-space.
 * Every conv is 3x3x3, stride 1, causal in time (2 copies of frame 0 in front, or the 2 cached
 * frames in a chunked decode), zero-padded by 1 in space.  A residual block is
 * x + conv2(SiLU(GN2(conv1(SiLU(GN1(x)))))).  Group norm statistics are per (batch, frame, group),
 * population variance, eps inside the square root.  The attention is one head over each frame's
 * H*W tokens with 1x1 q/k/v/o projections, scale 1/sqrt(C), on GN(x) without SiLU, plus residual.
 * dtype: VAE_BF16 stores activations in bf16 (fp32 accumulation, statistics and blend),
 * VAE_FP32 stores everything in fp32 and runs on the CUDA cores (fp32 FMAs in a fixed order): the
 * parity mode, max relative error <= 1e-4 against the fp64 oracle.
 * VAE_FP32_TC (decoder / encoder dtype only) is VAE_FP32 with the convs whose input channels are a
 * multiple of 32 on the tcgen05 tensor cores as three TF32 products per fp32 product (kind::tf32: the
 * high part of each operand is the value with its 13 low mantissa bits cleared, the remainder is exact
 * in fp32, and a_hi b_hi + a_hi b_lo + a_lo b_hi goes into the fp32 accumulator), about 70x faster;
 * the tensor cores' accumulation over 27 * C_in terms leaves relative errors near 3e-4 at 1024
 * channels (measured on the LTX-shaped 720p decode), so it is a fast fp32 reference, not the parity
 * mode.  Its workspace holds two more copies (high parts, remainders) of the largest conv input.
 * norm_type: VAE_NORM_GROUP (gn_groups, gn_eps as above), or VAE_NORM_CHANNEL_RMS: every norm above
 * becomes x * rsqrt(mean over channels of x^2 + gn_eps) * gamma + beta per pixel (gn_groups is then
 * ignored; stage channels must be multiples of 8 and at most 1024 with C/8 a power of two or a
 * multiple of 32). */
typedef struct {
  int latent_c;
  int n_stages;
  int stage_c[VAE_MAX_STAGES];
  int n_res[VAE_MAX_STAGES];
  int up_t[VAE_MAX_STAGES], up_h[VAE_MAX_STAGES], up_w[VAE_MAX_STAGES];
  int mid_res;
  int mid_attn;
  int gn_groups;
  float gn_eps;
  int out_c;
  int out_d2s_t, out_d2s_h, out_d2s_w;
  vae_dtype_t dtype;
  vae_norm_t norm_type;
} vae_config_t;

typedef struct vae_decoder vae_decoder_t; /* opaque */

/* Number of parameter tensors `vae_decoder_create` expects for `cfg` (host only). */
vae_status_t vae_decoder_n_weights(const vae_config_t* cfg, int* n_weights);

/* Create a decoder.  `weights` (host array of n_weights device pointers) lists the parameters
 * as fp32 device tensors in declaration order:
 *   conv_in.{weight [C0, latent_c, 3,3,3], bias [C0]};
 *   per mid residual block r, then per stage i and residual block r:
 *     norm1.{gamma, beta}, conv1.{weight, bias}, norm2.{gamma, beta}, conv2.{weight, bias};
 *   (mid_attn) mid.attn.norm.{gamma, beta}, then q, k, v, o: {weight [C, C], bias [C]}
 *     (the attention parameters come after the mid residual blocks, before stage 0);
 *   stage i < n_stages-1: up.{weight [s*C_{i+1}, C_i, 3,3,3], bias};
 *   head.norm.{gamma, beta}, head.conv.{weight, bias}.
 * Conv weights use PyTorch's [C_out, C_in, k_t, k_h, k_w] layout.  The library copies and repacks
 * them into its own buffers (K-major bf16 for the tensor-core path), so the caller may free its
 * tensors once the call returns.  Allocates device memory; synchronises the device. */
vae_status_t vae_decoder_create(const vae_config_t* cfg, const void* const* weights, int n_weights,
                                vae_decoder_t** out);

/* Free everything the handle owns (synchronises the device). */
void vae_decoder_destroy(vae_decoder_t* dec);

/* Allocate the workspace for a latent shape (host array [B, C, T, h, w]) and patch grid up front,
 * so that later `vae_decode` calls of that size or smaller allocate nothing (and can be captured
 * in a CUDA graph).  `vae_decode` calls it itself when the workspace is too small. */
vae_status_t vae_decoder_reserve(vae_decoder_t* dec, const int64_t latent_shape[5], int n_patch_h,
                                 int n_patch_w);

/* Decode a whole latent.  latent: fp32 NCTHW [B, latent_c, T, h, w] (device); out: NCTHW
 * [B, out_c, s_t*(T-1)+1, s_h*h, s_w*w] (device) in the config's dtype.  The latent's h and w are
 * split into n_patch_h x n_patch_w patches by the band rule ([DV] Patchify commit: the first
 * h % n_patch_h bands get one extra latent row); every layer keeps those bands, scaled.  Patch
 * counts change no output bit.  A band narrower than one latent row returns
 * VAE_ERR_PATCH_TOO_NARROW.  Resets the temporal caches. */
vae_status_t vae_decode(vae_decoder_t* dec, const void* latent, const int64_t latent_shape[5], void* out,
                        int n_patch_h, int n_patch_w, void* stream);

/* Chunked temporal decode ([DV] Wan adapter commit: a per-conv temporal cache threads through a
 * chunked decode).  Call with first_chunk=1 for the chunk holding latent frame 0, then in order
 * with first_chunk=0.  Each causal conv keeps the last 2 frames of its input inside the handle.
 * A first chunk of n latent frames yields s_t*(n-1)+1 output frames, a later one s_t*n.  The
 * concatenated outputs equal `vae_decode` of the whole latent bit for bit. */
vae_status_t vae_decode_chunk(vae_decoder_t* dec, const void* latent_chunk, const int64_t chunk_shape[5],
                              int first_chunk, void* out_chunk, int n_patch_h, int n_patch_w, void* stream);

/* Decode from host memory to host memory, through the chunked temporal decode above ([DV] Wan adapter
 * commit): latent_host is the NCTHW fp32 latent [B, C, T, h, w] and
 * out_host the NCTHW pixels (bf16, or fp32 for the fp32 dtypes) [B, out_c, T', H, W], both in host
 * memory (page-locked for the copies to overlap; pageable memory works, serialised).  The latent goes
 * in and the pixels come out in the temporal chunks of vae_decode_chunk (chunk 0 = latent frame 0, then
 * frames_per_chunk frames; 0 picks about five chunks), copied on an internal stream while `stream`
 * decodes the neighbouring chunk, through two device buffers per direction; `stream` waits for the
 * last copy, so the pixels are in out_host once the work on `stream` completes.  The result equals
 * `vae_decode` of the same latent bit for bit (chunked == whole).  Resets the temporal caches;
 * allocates the chunk buffers and the workspace before enqueuing anything. */
vae_status_t vae_decode_host(vae_decoder_t* dec, const void* latent_host, const int64_t latent_shape[5],
                             void* out_host, int n_patch_h, int n_patch_w, int frames_per_chunk, void* stream);

/* Overlap-tiled decode ([TP] Approach): tiles of tile_thw latent frames/rows/cols overlapping by
 * ovl_thw (host arrays) are planned with `vae_tile_plan`, each decoded causally on its own, and
 * blended with `vae_tile_blend`.  The result differs from `vae_decode` inside overlaps by design.
 * Tiles of one latent shape are decoded together as one batch (up to 16 GiB of workspace per batch);
 * each tile's pixels are bit-identical to `vae_decode` of that tile's latent box on its own. */
vae_status_t vae_decode_tiled(vae_decoder_t* dec, const void* latent, const int64_t latent_shape[5],
                              void* out, const int tile_thw[3], const int ovl_thw[3], void* stream);

/* Per-kernel timing of the decoder's launches (profiling aid).  While enabled, every kernel the
 * handle enqueues is bracketed by CUDA events on its stream and tagged with its kernel class and its
 * algorithmic work (conv/GEMM FLOPs = 2 * MACs of the real channel counts; norm/blend bytes = the
 * reads and writes the operation needs).  Enabling creates events per launch: do not enable it
 * inside a CUDA-graph capture. */
typedef struct {
  char name[32];   /* kernel class: conv_tc (tensor-core convs but the pixel head), conv_head (the
                      tensor-core conv_out), conv_simt, gn_stats, gn_apply, gemm_tc, gemm_simt, softmax,
                      transpose, cast, copy, latent, blend, rms_norm */
  int launches;    /* launches since the last read */
  double ms;       /* summed device time of those launches */
  double flops;    /* summed algorithmic FLOPs */
  double bytes;    /* summed algorithmic DRAM bytes */
} vae_prof_t;

vae_status_t vae_decoder_profile(vae_decoder_t* dec, int enable);

/* Synchronises the device, folds the recorded launches into per-class totals (at most *n entries;
 * *n returns the count) and starts a new recording. */
vae_status_t vae_decoder_profile_read(vae_decoder_t* dec, vae_prof_t* out, int* n);

/* Last failure of `dec` (or of the op-level calls when dec is NULL).  Synchronises the device and
 * folds in the device fault word (VAE_ERR_TIMEOUT / VAE_ERR_RANGE), then clears it. */
vae_status_t vae_last_error(vae_decoder_t* dec, vae_error_info_t* info);

/* ------------------------------------------------------------------------------------------ */
/* Encoder                                                                                     */
/* ------------------------------------------------------------------------------------------ */

/* Down-sampler kinds ([DV] encoder commits): VAE_DOWN_FOLD, a stride-1 causal conv to
 * stage_c[i+1] / (down_t*down_h*down_w) channels followed by space-to-depth (HunyuanVideo 1.5,
 * LTX-2); VAE_DOWN_STRIDE, one zero row below and one zero column to the right, then a 3x3 stride-2
 * conv of each frame to stage_c[i+1] channels (Qwen-Image / Wan 2.1, AutoencoderKL; down factors
 * (1, 2, 2)). */
typedef enum { VAE_DOWN_FOLD = 0, VAE_DOWN_STRIDE = 1 } vae_down_t;

/* Architecture of a causal video-VAE encoder, the decoder read backwards ([DV] encoder commits):
 *   pixels [B, pix_c, T, H, W] -> space-to-depth by (1, patch_h, patch_w) (patchify, optional)
 *   -> conv_in (pix_c*patch_h*patch_w -> stage_c[0]) -> per stage i: n_res[i] residual blocks, then
 *      (i < n_stages-1) the down-sampler to stage_c[i+1] -> mid_res residual blocks
 *   -> norm + SiLU -> conv_out (stage_c[last] -> 2 * latent_c moments: mean and log-variance).
 * Space-to-depth moves position (c, s_t t + dt, s_h y + dy, s_w x + dx) to channel
 * c*(s_t s_h s_w) + dt s_h s_w + dy s_w + dx; a temporal fold first puts s_t - 1 copies of frame 0 in
 * front (causal: the first frame folds into one latent frame, T -> (T - 1)/s_t + 1).  Convs, residual
 * blocks, norms and dtypes are as in the decoder (VAE_FP8: e4m3 operands for the residual blocks' and
 * down-samplers' convs whose input channels are a multiple of 128). */
typedef struct {
  int pix_c;
  int patch_h, patch_w;
  int n_stages;
  int stage_c[VAE_MAX_STAGES];
  int n_res[VAE_MAX_STAGES];
  int down_kind[VAE_MAX_STAGES];
  int down_t[VAE_MAX_STAGES], down_h[VAE_MAX_STAGES], down_w[VAE_MAX_STAGES];
  int mid_res;
  int gn_groups;
  float gn_eps;
  int latent_c;
  vae_dtype_t dtype;
  vae_norm_t norm_type;
} vae_encoder_config_t;

typedef struct vae_encoder vae_encoder_t; /* opaque */

/* Number of parameter tensors `vae_encoder_create` expects for `cfg` (host only). */
vae_status_t vae_encoder_n_weights(const vae_encoder_config_t* cfg, int* n_weights);

/* Create an encoder.  `weights` (host array of n_weights device fp32 pointers, 16-byte aligned) in
 * declaration order: conv_in.{weight,bias}; per stage i: per residual block norm1.{gamma,beta},
 * conv1.{weight,bias}, norm2.{gamma,beta}, conv2.{weight,bias}; then (i < n_stages-1) down.{weight,bias}
 * ([C_next/S, C_i, 3, 3, 3] for VAE_DOWN_FOLD, [C_next, C_i, 3, 3] for VAE_DOWN_STRIDE); then the mid
 * residual blocks; head.norm.{gamma,beta}; head.conv.{weight,bias} ([2*latent_c, C_last, 3, 3, 3]).
 * The weights are copied (and repacked); the caller may free them afterwards.  Synchronises. */
vae_status_t vae_encoder_create(const vae_encoder_config_t* cfg, const void* const* weights, int n_weights,
                                vae_encoder_t** enc);

/* Encode pixels (device fp32 NCTHW [B, pix_c, T, H, W], T = 1 + s_t*k, H and W multiples of the
 * total spatial factor) into moments (device fp32 NCTHW [B, 2*latent_c, (T-1)/s_t + 1, H/s_h, W/s_w]),
 * split into n_patch_h x n_patch_w spatial patches cut on the latent grid ([DV] Patchify commit: bands
 * in whole multiples of what the encoder narrows the axis by, first bands one latent row larger).
 * Every kernel of a layer covers all patches; halo rows are read from the neighbour in place, so a
 * strided down-sampler's halo follows the patch's place in the global stride grid.  The result does
 * not depend on the patch grid (bit for bit).  Stream-ordered; the workspace grows on first use. */
vae_status_t vae_encode(vae_encoder_t* enc, const void* video, const int64_t video_shape[5], void* moments,
                        int n_patch_h, int n_patch_w, void* stream);

/* Overlap-tiled encode ([ENC] encode_tile_split / exec / merge): spatial tiles planned on the latent grid
 * by the tile plan's rule (tile_hw latent rows/cols, overlap ovl_hw), each tile's pixels encoded on
 * their own, the latent tiles blended with the decode's ramps and normalised weighted sum (in latent
 * units, the whole clip in time).  Same shapes as vae_encode.  Tiles of one shape are encoded together
 * as one batch (up to 16 GiB of workspace per batch), each bit-identical to encoding it on its own. */
vae_status_t vae_encode_tiled(vae_encoder_t* enc, const void* video, const int64_t video_shape[5], void* moments,
                              const int tile_hw[2], const int ovl_hw[2], void* stream);

/* Per-kernel timing of the encoder's launches, as vae_decoder_profile / vae_decoder_profile_read. */
vae_status_t vae_encoder_profile(vae_encoder_t* enc, int enable);
vae_status_t vae_encoder_profile_read(vae_encoder_t* enc, vae_prof_t* out, int* n);

/* Last failure of `enc`, as vae_last_error. */
vae_status_t vae_encoder_last_error(vae_encoder_t* enc, vae_error_info_t* info);

void vae_encoder_destroy(vae_encoder_t* enc);

/* ------------------------------------------------------------------------------------------ */
/* Host plans (pure integer, no GPU needed)                                                    */
/* ------------------------------------------------------------------------------------------ */

/* Band edges of n patches over `length` latent rows at a layer of the given scale ([DV] Patchify
 * commit): edges[0..n] (host), edges[i+1]-edges[i] = scale * (ceil or floor of length/n), the
 * larger bands first.  A band narrower than `reach` returns VAE_ERR_PATCH_TOO_NARROW. */
vae_status_t vae_patch_edges(int length, int n, int scale, int reach, int* edges);

/* One tile of an overlap-tiled decode. */
typedef struct {
  int lat[6]; /* t0, nt, h0, nh, w0, nw: the tile's latent box */
  int pix[6]; /* t0, nt, h0, nh, w0, nw: its output pixel box (causal time: first latent frame -> 1 frame) */
  int ovl[6]; /* overlap with the previous / next tile along t, h, w, in output pixels (0 at image borders) */
} vae_tile_t;

/* Tile plan ([TP] Approach; [ENC] LTX-2.5 grid: 576 px with tile 512 / stride 448 is 2 x 2).
 * Per axis: starts 0, S-O, 2(S-O), ... until a tile reaches the end; the last is clipped.
 * Spatial pixels = scale_s * latent; temporal pixels of a tile starting at t0 with n frames are
 * [scale_t*t0, scale_t*(t0+n-1)] when causal_t, else scale_t * latent.  Tiles in raster order
 * (t, h, w).  tiles: host array of capacity *n_tiles (in: capacity, out: count). */
vae_status_t vae_tile_plan(const int lat_thw[3], const int tile_thw[3], const int ovl_thw[3], int scale_t,
                           int scale_s, int causal_t, vae_tile_t* tiles, int* n_tiles);

/* ------------------------------------------------------------------------------------------ */
/* Op-level entry points                                                                       */
/* ------------------------------------------------------------------------------------------ */

/* Causal Conv3d descriptor.  Output frames T, rows H, cols W before depth-to-space. */
typedef struct {
  int B, T, H, W;
  int C_in, C_out;       /* C_out counts conv output channels (before depth-to-space) */
  int cache_frames;      /* 0: x holds T frames, frame 0 is repeated twice in front (causal pad);
                            2: x holds 2 cached frames followed by the T frames */
  int n_patch_h, n_patch_w;
  int patch_h_edges[VAE_MAX_PATCHES + 1]; /* ascending, 0 .. H (band edges at this layer) */
  int patch_w_edges[VAE_MAX_PATCHES + 1]; /* ascending, 0 .. W */
  int d2s_t, d2s_h, d2s_w; /* depth-to-space fused into the store (1,1,1 = none) */
  int drop_first;          /* with d2s_t > 1: drop the first d2s_t-1 output frames */
  int out_ncthw;           /* 1: y is NCTHW pixels; 0: y is channels-last */
  vae_dtype_t in_dtype;    /* x (and the packed weights) */
  vae_dtype_t out_dtype;   /* y */
  vae_dtype_t res_dtype;   /* residual */
} vae_conv_desc_t;

/* Bytes of the packed weight buffer for `d`. */
size_t vae_conv3d_packed_bytes(const vae_conv_desc_t* d);

/* Repack an fp32 PyTorch-layout weight [C_out, C_in, 3, 3, 3] (device) into the library layout
 * (device, vae_conv3d_packed_bytes(d) bytes, caller-owned): for bf16 a K-major [N_pad, 27*C_in_pad]
 * matrix whose rows are ordered (depth-to-space sub-position, channel) so that the fused
 * depth-to-space stores contiguous channels; for fp8 the same matrix in e4m3 bytes, each row divided
 * by its scale max|row| / 448, followed (at the next 256-byte boundary) by the fp32 scales [N_pad];
 * for fp32 [27, C_in, C_out].  With out_ncthw the bf16 / fp8 rows keep PyTorch's channel order (so the
 * conv's store writes runs of horizontally adjacent pixels); pack and conv must use the same out_ncthw.
 * bf16 convs with C_out <= 12 pack tap-stacked instead: [3 (k_t)][112][C_in], row (k_h*3 + k_w)*12 + n
 * holding packed column n (same order as above) of that spatial tap, zero rows elsewhere, so that one
 * tensor-core instruction covers all 9 spatial taps of a narrow conv. */
vae_status_t vae_conv3d_pack_weights(const float* w, const vae_conv_desc_t* d, void* w_packed, void* stream);

/* Causal Conv3d ([DV] PatchConv3d padding commit, HunyuanVideo/LTX-2 commits): for every output
 * voxel y[b,t,h,w,co] = bias[co] + sum_{kt,kh,kw,ci} W[co,ci,kt,kh,kw] * x[b, t-2+kt, h-1+kh, w-1+kw, ci]
 * with t-2+kt clamped at 0 (or read from the 2 cached frames), zero outside the image, plus
 * residual[b,t,h,w,co] when `residual` is non-NULL, then depth-to-space.  x: channels-last
 * [B, cache_frames+T, H, W, C_in]; bias fp32 [C_out] or NULL; residual channels-last [B,T,H,W,C_out]
 * or NULL (only without depth-to-space); y: [B, T', H*d2s_h, W*d2s_w, C_out/(d2s)] channels-last or
 * NCTHW, T' = d2s_t*T - (drop_first ? d2s_t-1 : 0).  Each patch's outputs are computed by blocks
 * that own that patch; their halo taps read the neighbour patch's rows in place.  bf16 inputs with
 * C_in % 64 == 0 run on the tcgen05 tensor-core kernel, the rest on a CUDA-core kernel; e4m3 inputs
 * (in_dtype VAE_FP8, C_in % 128 == 0, weights packed for VAE_FP8) run on the tensor cores with e4m3
 * products (kind::f8f6f4), each output channel's sum multiplied by its weight scale before the bias.
 * y must not alias x or residual. */
vae_status_t vae_conv3d_causal(const void* x, const void* w_packed, const float* bias, const void* residual,
                               void* y, const vae_conv_desc_t* d, void* stream);

/* PatchGroupNorm (+ SiLU) descriptor. */
typedef struct {
  int B, T, H, W, C;
  int groups;
  float eps;
  int silu; /* 1: y = SiLU(norm(x)); 0: y = norm(x) */
  int n_patch_h, n_patch_w;
  int patch_h_edges[VAE_MAX_PATCHES + 1];
  int patch_w_edges[VAE_MAX_PATCHES + 1];
  vae_dtype_t in_dtype, out_dtype;
} vae_gn_desc_t;

/* out_dtype VAE_FP8: y is written as e4m3 operands of a following fp8 conv (in_dtype bf16 or fp32). */

/* Bytes of scratch `vae_patch_groupnorm_silu` needs for `d`. */
size_t vae_patch_groupnorm_workspace_bytes(const vae_gn_desc_t* d);

/* PatchGroupNorm + SiLU ([DV] PatchGroupNorm commit: the exact global mean and the population
 * variance of each group, divide by the count, no Bessel correction, merged from per-patch sums).
 * Statistics per (b, t, group) over the group's C/groups channels and all H x W pixels.  Each
 * patch accumulates exact integer partial sums of x*2^18 and (x*2^18)^2 (so |x| < 8192, else
 * VAE_ERR_RANGE is flagged); the per-patch sums are merged in patch order; mean and variance
 * follow in fp64 from the exact totals.  Integer sums make the result independent of the patch
 * count and of the order blocks run in.  y = SiLU((x - mean) * rsqrt(var + eps) * gamma + beta).
 * x, y: channels-last [B, T, H, W, C] (y may alias x); gamma, beta: fp32 [C]; workspace: device
 * scratch of vae_patch_groupnorm_workspace_bytes(d) bytes, cleared by the call. */
vae_status_t vae_patch_groupnorm_silu(const void* x, const float* gamma, const float* beta, void* y,
                                      void* workspace, const vae_gn_desc_t* d, void* stream);

/* Bytes of the fixed device array that vae_patch_groupnorm_silu_noalloc uses as scratch (4 MiB). */
#define VAE_GN_NOALLOC_SCRATCH_BYTES (4 << 20)

/* PatchGroupNorm + SiLU without any allocation, for callers that cannot allocate device memory: hosts
 * whose own pool allocator owns the whole device and that pass a plugin only its input and output
 * buffers, or loops in which a cudaMalloc (which can synchronise the device) is not allowed.  The pages
 * have no counterpart of this entry point; it computes exactly what vae_patch_groupnorm_silu computes
 * (same kernels, same result), but its scratch -- the per-patch partial sums and the per-frame affine,
 * vae_patch_groupnorm_workspace_bytes(d) bytes -- lives in a fixed device array of
 * VAE_GN_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads the library holds until
 * the process exits.  A descriptor needing more scratch than that returns VAE_ERR_UNSUPPORTED and
 * launches nothing.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before any stream capture.
 * Every call shares the one array and leaves its contents behind; each call clears the partial sums it
 * needs before using them, but calls whose GPU work overlaps (e.g. on two streams, or from two host
 * threads) race on the array: serialise them.  No cudaMalloc, cudaFree or allocating library routine is
 * called.  x, y, gamma, beta, d: as for vae_patch_groupnorm_silu. */
vae_status_t vae_patch_groupnorm_silu_noalloc(const void* x, const float* gamma, const float* beta, void* y,
                                              const vae_gn_desc_t* d, void* stream);

/* Channel RMS norm descriptor: x, y channels-last [B, T, H, W, C] (out_dtype VAE_FP8: e4m3 y). */
typedef struct {
  int B, T, H, W, C;
  float eps;
  int silu;
  vae_dtype_t in_dtype, out_dtype;
} vae_rms_desc_t;

/* Channel RMS norm + optional SiLU ([DV] Qwen-Image, HunyuanVideo/1.5 and LTX-2 adapter commits:
 * the norm reduces over channels, so a patch needs nothing from its neighbours).  Per pixel
 * y = x * r * gamma + beta with r = 1 / sqrt(mean over the C channels of x^2 + eps) (fp32 sums in a
 * fixed order per pixel, so the result does not depend on any patch grid), then SiLU when silu != 0.
 * x, y: 16-byte aligned device pointers (y may alias x); gamma, beta: fp32 [C], 32-byte aligned.
 * C: a multiple of 8, at most 1024, with C/8 a power of two or a multiple of 32 (else
 * VAE_ERR_UNSUPPORTED).  Enqueued on `stream`; nothing is allocated. */
vae_status_t vae_channel_rmsnorm_silu(const void* x, const float* gamma, const float* beta, void* y,
                                      const vae_rms_desc_t* d, void* stream);

/* Depth-to-space descriptor: x [B, T, H, W, C*s_t*s_h*s_w] channels-last. */
typedef struct {
  int B, T, H, W, C;
  int s_t, s_h, s_w;
  int drop_first;
  vae_dtype_t dtype;
} vae_d2s_desc_t;

/* Depth-to-space ([DV] LTX-2 commit: channels move into space, one input position per output):
 * channel c*(s_t s_h s_w) + dt*s_h*s_w + dy*s_w + dx of (t, h, w) goes to channel c of
 * (s_t*t+dt, s_h*h+dy, s_w*w+dx); with drop_first the first s_t-1 output frames are dropped.
 * y: [B, s_t*T - drop, s_h*H, s_w*W, C] channels-last. */
vae_status_t vae_upsample_d2s(const void* x, void* y, const vae_d2s_desc_t* d, void* stream);

/* Tile-blend descriptor: output NCTHW [B, C, T, H, W]. */
typedef struct {
  int B, C, T, H, W;
  vae_dtype_t tile_dtype, out_dtype;
} vae_blend_desc_t;

/* Overlap blend ([TP] Approach: each tile weighted by a mask assembled from 1-D parts, summed next
 * to the weights, divided): out = sum_i w_i x_i / sum_i w_i in fp32, tiles in the given (raster)
 * order; w_i is the outer product of per-axis ramps: over a P-pixel overlap with the previous tile
 * the weight rises as (y+1)/(P+1), over one with the next it falls as (n-y)/(P+1), elsewhere 1.
 * Each output pixel gathers the tiles covering it, so no accumulation buffer is needed.
 * tiles: host array of n_tiles device pointers, tile i NCTHW [B, C, pix nt, nh, nw];
 * meta: host array of n_tiles vae_tile_t (pix and ovl used); every output pixel must be covered. */
vae_status_t vae_tile_blend(const void* const* tiles, const vae_tile_t* meta, int n_tiles, void* out,
                            const vae_blend_desc_t* d, void* stream);

/* Batched bf16 GEMM on the tcgen05 tensor cores (the attention's products):
 * D[b] = alpha * A[b] (M x K, row-major) * B[b]^T (B[b] is N x K, row-major) + bias (fp32 [N] or
 * NULL), fp32 accumulation, D (M x N row-major) in out_dtype.  K % 64 == 0, N % 16 == 0;
 * strides in elements between batches. */
vae_status_t vae_gemm_bf16(const void* A, const void* B, void* D, const float* bias, int M, int N, int K,
                           int batch, int64_t stride_a, int64_t stride_b, int64_t stride_d, float alpha,
                           vae_dtype_t out_dtype, void* stream);

/* Watchdog self-test: launches a kernel that waits on a barrier nothing will complete, bounded
 * by timeout_us; returns VAE_ERR_TIMEOUT after synchronising (the context stays usable), or
 * VAE_OK if the wait was not bounded as it should be. */
vae_status_t vae_watchdog_selftest(int timeout_us, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* VAEDEC_H */
