// C ABI of libvaedec: argument checks, host plans, the decoder handle and its layer schedule.
//
// The decoder runs the layer sequence of the causal video-VAE decoders described in DistVAE PR #14
// "Add tiled VAE parallelism & extended model support" (Wan, LTX-2 adapter commits) and TensorRT-LLM
// PR #16066 "ParallelVAE_TrtllmWan for native Wan VAE", split into spatial patches: the band rule of
// the Patchify commit fixes the patch edges at the latent grid, every layer keeps those bands scaled
// by its up-sampling factor, and every kernel of a layer covers all patches at once (a halo read
// needs the neighbour's previous layer, so layers are synchronous).  Chunked temporal decode keeps
// per-conv 2-frame caches in the handle; tiled decode follows TensorRT-LLM PR #15753 "LTX-2
// tile-parallel VAE decode".  Everything is stream-ordered; nothing here synchronises the host
// except create/destroy/reserve (allocation) and vae_last_error.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"

namespace vae {

__device__ uint32_t g_fault[4];

uint32_t* fault_word() {
  static uint32_t* ptrs[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fault) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(p);
  }
  return ptrs[dev];
}

uint64_t wait_limit_ns() { return 2000000000ull; }

}  // namespace vae

using namespace vae;

// ================================================================================ errors
struct vae_decoder;
namespace {

vae_error_info_t g_last{};  // op-level calls
std::mutex g_last_mu;

vae_status_t set_err(vae_error_info_t* e, vae_status_t code, int rows, int factor, const char* fmt, ...) {
  vae_error_info_t tmp{};
  tmp.code = code;
  tmp.rows = rows;
  tmp.factor = factor;
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(tmp.message, sizeof(tmp.message), fmt, ap);
  va_end(ap);
  if (e) {
    *e = tmp;
  } else {
    std::lock_guard<std::mutex> lk(g_last_mu);
    g_last = tmp;
  }
  return code;
}

#define CK(call)                                                                               \
  do {                                                                                         \
    cudaError_t _e = (call);                                                                   \
    if (_e != cudaSuccess)                                                                     \
      return set_err(ERRP, _e == cudaErrorMemoryAllocation ? VAE_ERR_OOM : VAE_ERR_CUDA, 0, 0, \
                     "%s failed: %s", #call, cudaGetErrorString(_e));                          \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int round_up(int x, int m) { return (x + m - 1) / m * m; }

vae_status_t band_edges(int length, int n, int scale, int reach, int* edges, vae_error_info_t* e) {
  if (length <= 0 || n <= 0 || scale <= 0 || n > VAE_MAX_PATCHES)
    return set_err(e, VAE_ERR_INVALID_ARG, 0, 0, "bad band request: length %d, n %d, scale %d", length, n, scale);
  const int q = length / n, r = length % n;
  edges[0] = 0;
  for (int i = 0; i < n; ++i) {
    const int sz = (i < r ? q + 1 : q) * scale;
    if (sz < reach)
      return set_err(e, VAE_ERR_PATCH_TOO_NARROW, sz, reach,
                     "patch %d has %d rows, narrower than the kernel reach %d", i, sz, reach);
    edges[i + 1] = edges[i] + sz;
  }
  return VAE_OK;
}

}  // namespace

// ================================================================================ decoder
namespace {

// bf16 mode keeps the residual stream and the first conv's output (the two group-norm inputs
// that are not conv operands) in fp32; conv operands are bf16.  fp8 mode stores both in bf16: next to
// the e4m3 operands' rounding the bf16 storage is small (oracle emulation, mini decoders: rel-L2
// 0.0678 -> 0.0694 and 0.0495 -> 0.0498), and the norms' passes move 2 bytes per element, not 4.
constexpr bool kResidF32 = true;
constexpr bool kC1F32 = true;

struct ConvL {
  int C_in = 0, C_out = 0, C_in_pad = 0, N_pad = 0, st = 1, sh = 1, sw = 1;
  bool tc = false;
  bool fp8 = false;        // e4m3 operands and weights (fp8 decoders)
  bool natural = false;    // weight rows in PyTorch channel order (convs that store NCTHW pixels)
  bool tap = false;        // narrow bf16 conv: weights packed tap-stacked (all 9 spatial taps in one MMA)
  bool tf32 = false;       // fp32 decoder on the tensor cores: 3 TF32 products per fp32 product
  float* wscale = nullptr; // fp8: per-output-channel weight scales (inside the packed weight buffer)
  void* w = nullptr;       // packed weights
  float* bias = nullptr;   // fp32 [C_out]
  void* cache = nullptr;   // [B, 2, H, W, C_in_pad] (chunked decode)
  size_t cache_bytes = 0;
};
struct NormL {
  float* gamma = nullptr;
  float* beta = nullptr;
  int C = 0;
};
struct ResL {
  NormL n1, n2;
  ConvL c1, c2;
};
struct AttnL {
  NormL n;
  void* w[4] = {nullptr, nullptr, nullptr, nullptr};  // q, k, v, o: bf16 (or fp32) [C, C]
  float* b[4] = {nullptr, nullptr, nullptr, nullptr};
};

struct Level {  // one spatial/temporal scale of the decode
  int T, H, W, C;
  int ph[VAE_MAX_PATCHES + 1], pw[VAE_MAX_PATCHES + 1];
};

}  // namespace

struct vae_decoder {
  vae_config_t cfg{};
  bool f32 = false;  // fp32 storage mode
  bool f8 = false;   // e4m3 operands for the residual blocks' and up-samplers' convs
  bool f32tc = false;  // fp32 storage with the convs as three TF32 products on the tensor cores
  ConvL conv_in;
  std::vector<ResL> mid;
  bool has_attn = false;
  AttnL attn;
  std::vector<std::vector<ResL>> stages;
  std::vector<ConvL> ups;
  NormL head_norm;
  ConvL head;
  std::vector<void*> owned;  // every cudaMalloc of the handle
  // workspace
  void* ws = nullptr;
  size_t ws_bytes = 0;
  int64_t ws_shape[5] = {0, 0, 0, 0, 0};
  int ws_nph = 0, ws_npw = 0;
  bool caches_ready = false;
  int64_t cache_shape[5] = {0, 0, 0, 0, 0};
  int cache_nph = 0, cache_npw = 0;
  // tiled decode tile storage
  void* tiles = nullptr;
  size_t tiles_bytes = 0;
  // host-buffer decode: the copy stream, double-buffered latent / pixel chunks, and its events
  cudaStream_t copy_stream = nullptr;
  void* hb_lat[2] = {nullptr, nullptr};
  void* hb_out[2] = {nullptr, nullptr};
  size_t hb_lat_bytes = 0, hb_out_bytes = 0;
  cudaEvent_t hb_ev[8] = {};  // [0,1] latent in, [2,3] chunk decoded, [4,5] pixels out, [6] start, [7] end
  bool hb_ready = false;
  vae_error_info_t err{};
  // profiling: events around every launch while enabled
  bool prof = false;
  struct Rec {
    int kind;
    cudaEvent_t a, b;
    double flops, bytes;
  };
  std::vector<Rec> recs;
};

namespace {

// conv_head: the tensor-core conv_out (pixel head), timed apart from the other convs
enum Kind { K_CONV_TC, K_CONV_SIMT, K_GN_STATS, K_GN_APPLY, K_GEMM_TC, K_GEMM_SIMT, K_SOFTMAX, K_TRANSPOSE, K_CAST,
            K_COPY, K_LATENT, K_BLEND, K_RMS, K_CONV_HEAD, K_COUNT };
const char* kKindNames[K_COUNT] = {"conv_tc", "conv_simt", "gn_stats", "gn_apply", "gemm_tc", "gemm_simt",
                                   "softmax", "transpose", "cast", "copy", "latent", "blend", "rms_norm",
                                   "conv_head"};

// Brackets one launch with events when the handle is profiling.
struct Prof {
  vae_decoder* d;
  cudaStream_t s;
  int kind;
  double fl, by;
  cudaEvent_t a = nullptr;
  Prof(vae_decoder* dd, cudaStream_t ss, int k, double flops, double bytes) : d(dd), s(ss), kind(k), fl(flops), by(bytes) {
    if (d && d->prof && cudaEventCreate(&a) == cudaSuccess) cudaEventRecord(a, s);
  }
  ~Prof() {
    if (!a) return;
    cudaEvent_t b = nullptr;
    if (cudaEventCreate(&b) != cudaSuccess) {
      cudaEventDestroy(a);
      return;
    }
    cudaEventRecord(b, s);
    d->recs.push_back({kind, a, b, fl, by});
  }
};

#define ERRP (&d->err)

template <typename T>
vae_status_t dalloc(vae_decoder* d, T** p, size_t bytes) {
  void* q = nullptr;
  cudaError_t e = cudaMalloc(&q, std::max<size_t>(bytes, 256));
  if (e != cudaSuccess) return set_err(&d->err, VAE_ERR_OOM, 0, 0, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
  d->owned.push_back(q);
  *p = static_cast<T*>(q);
  return VAE_OK;
}

int act_bytes(const vae_decoder* d) { return d->f32 ? 4 : 2; }
// bytes of one element of conv c's operand (e4m3 convs of an fp8 decoder take 1)
int op_bytes(const vae_decoder* d, const ConvL& c) { return c.fp8 ? 1 : act_bytes(d); }
int res_bytes(const vae_decoder* d) { return (d->f32 || (kResidF32 && !d->f8)) ? 4 : 2; }
int c1_bytes(const vae_decoder* d) { return (d->f32 || (kC1F32 && !d->f8)) ? 4 : 2; }

vae_status_t make_conv(vae_decoder* d, ConvL& c, const float* w, const float* b, int C_in, int C_out, int st, int sh,
                       int sw, bool pad_input = false, bool allow_fp8 = false, bool natural = false) {
  c.C_in = C_in;
  c.C_out = C_out;
  c.st = st; c.sh = sh; c.sw = sw;
  const int S = st * sh * sw;
  if (C_out % S) return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "conv out channels %d not divisible by %d", C_out, S);
  // tensor cores take 64-channel K blocks (32 fp32 channels for the 3 x TF32 products of fp32
  // decoders); the latent is zero-padded up to them when it is converted
  const int kb = d->f32 ? 32 : 64;
  c.tc = (!d->f32 || d->f32tc) && (C_in % kb == 0 || pad_input);
  c.tf32 = d->f32 && c.tc;
  c.C_in_pad = c.tc ? round_up(C_in, kb) : C_in;
  c.fp8 = d->f8 && allow_fp8 && c.tc && C_in % 128 == 0;
  c.natural = natural;
  if (c.fp8) {
    c.N_pad = round_up(C_out, 16);
    const size_t off = fp8_scale_offset(c.N_pad, c.C_in_pad);
    vae_status_t s = dalloc(d, &c.w, off + static_cast<size_t>(c.N_pad) * 4);
    if (s) return s;
    c.wscale = reinterpret_cast<float*>(static_cast<char*>(c.w) + off);
    CK(launch_pack_weights_fp8(w, C_out, C_in, c.C_in_pad, c.N_pad, S, c.w, nullptr, natural));
  } else if (c.tf32) {
    c.N_pad = round_up(C_out, 16);
    vae_status_t s = dalloc(d, &c.w, 2ull * c.N_pad * 27 * c.C_in_pad * 4);
    if (s) return s;
    CK(launch_pack_weights_tf32(w, C_out, C_in, c.C_in_pad, c.N_pad, S, c.w, nullptr, natural));
  } else if (c.tc) {
    c.N_pad = round_up(C_out, 16);
    c.tap = conv_tap_stacked(C_out, 0);
    const size_t bytes = c.tap ? 3ull * kTapRows * c.C_in_pad * 2 : static_cast<size_t>(c.N_pad) * 27 * c.C_in_pad * 2;
    vae_status_t s = dalloc(d, &c.w, bytes);
    if (s) return s;
    CK(launch_pack_weights_bf16(w, C_out, C_in, c.C_in_pad, c.N_pad, S, c.w, nullptr, natural, c.tap));
  } else {
    const size_t bytes = 27ull * C_in * C_out * 4;
    vae_status_t s = dalloc(d, &c.w, bytes);
    if (s) return s;
    CK(launch_pack_weights_f32(w, C_out, C_in, c.w, nullptr));
  }
  vae_status_t s = dalloc(d, &c.bias, C_out * 4ull);
  if (s) return s;
  CK(cudaMemcpy(c.bias, b, C_out * 4ull, cudaMemcpyDeviceToDevice));
  return VAE_OK;
}

vae_status_t make_norm(vae_decoder* d, NormL& n, const float* g, const float* b, int C) {
  n.C = C;
  vae_status_t s = dalloc(d, &n.gamma, C * 4ull);
  if (s) return s;
  s = dalloc(d, &n.beta, C * 4ull);
  if (s) return s;
  CK(cudaMemcpy(n.gamma, g, C * 4ull, cudaMemcpyDeviceToDevice));
  CK(cudaMemcpy(n.beta, b, C * 4ull, cudaMemcpyDeviceToDevice));
  return VAE_OK;
}

int count_weights(const vae_config_t& c) {
  int n = 2;
  n += 8 * c.mid_res;
  if (c.mid_attn) n += 2 + 8;
  for (int i = 0; i < c.n_stages; ++i) {
    n += 8 * c.n_res[i];
    if (i + 1 < c.n_stages) n += 2;
  }
  n += 4;
  return n;
}

vae_status_t check_config(const vae_config_t* c, vae_error_info_t* e) {
  if (!c) return set_err(e, VAE_ERR_INVALID_ARG, 0, 0, "null config");
  const bool rms = c->norm_type == VAE_NORM_CHANNEL_RMS;
  if (c->norm_type != VAE_NORM_GROUP && !rms) return set_err(e, VAE_ERR_INVALID_ARG, 0, 0, "unknown norm type");
  if (c->n_stages < 1 || c->n_stages > VAE_MAX_STAGES || c->latent_c <= 0 || (!rms && c->gn_groups <= 0) || c->out_c <= 0 ||
      c->mid_res < 0 || c->out_d2s_t < 1 || c->out_d2s_h < 1 || c->out_d2s_w < 1 ||
      (c->dtype != VAE_BF16 && c->dtype != VAE_FP32 && c->dtype != VAE_FP8 && c->dtype != VAE_FP32_TC))
    return set_err(e, VAE_ERR_INVALID_ARG, 0, 0, "invalid decoder config");
  if (c->out_d2s_t != 1) return set_err(e, VAE_ERR_UNSUPPORTED, 0, 0, "temporal depth-to-space in conv_out is not supported");
  for (int i = 0; i < c->n_stages; ++i) {
    const int C = c->stage_c[i];
    if (rms) {
      if (C <= 0 || c->n_res[i] < 0) return set_err(e, VAE_ERR_INVALID_ARG, 0, 0, "stage %d channels", i);
      if (!rms_supported(C)) return set_err(e, VAE_ERR_UNSUPPORTED, 0, 0, "stage %d: RMS norm over %d channels not supported", i, C);
    } else {
    if (C <= 0 || C % c->gn_groups || c->n_res[i] < 0) return set_err(e, VAE_ERR_INVALID_ARG, 0, 0, "stage %d channels", i);
    const int cpg = C / c->gn_groups;
    if (C % 8 || C > 6144 || !(cpg % 8 == 0 || 8 % cpg == 0))
      return set_err(e, VAE_ERR_UNSUPPORTED, 0, 0, "stage %d: %d channels / %d groups not supported", i, C, c->gn_groups);
    }
    if (i + 1 < c->n_stages && (c->up_t[i] < 1 || c->up_t[i] > 2 || c->up_h[i] < 1 || c->up_w[i] < 1 || c->up_h[i] != c->up_w[i]))
      return set_err(e, VAE_ERR_UNSUPPORTED, 0, 0, "up-sampler %d factors", i);
  }
  if (c->out_d2s_h != c->out_d2s_w) return set_err(e, VAE_ERR_UNSUPPORTED, 0, 0, "non-square final depth-to-space");
  return VAE_OK;
}

#undef ERRP

}  // namespace

extern "C" vae_status_t vae_decoder_n_weights(const vae_config_t* cfg, int* n_weights) {
  vae_status_t s = check_config(cfg, nullptr);
  if (s) return s;
  if (!n_weights) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null n_weights");
  *n_weights = count_weights(*cfg);
  return VAE_OK;
}

namespace {
// Every device allocation of a handle (weights, workspace, caches, tile storage).
void release_memory(vae_decoder* d) {
  cudaDeviceSynchronize();
  for (void* p : d->owned) cudaFree(p);
  d->owned.clear();
  if (d->ws) cudaFree(d->ws);
  if (d->tiles) cudaFree(d->tiles);
  d->ws = d->tiles = nullptr;
  d->ws_bytes = d->tiles_bytes = 0;
  for (int i = 0; i < 2; ++i) {
    if (d->hb_lat[i]) cudaFree(d->hb_lat[i]);
    if (d->hb_out[i]) cudaFree(d->hb_out[i]);
    d->hb_lat[i] = d->hb_out[i] = nullptr;
  }
  d->hb_lat_bytes = d->hb_out_bytes = 0;
  if (d->hb_ready) {
    for (cudaEvent_t& e : d->hb_ev) cudaEventDestroy(e);
    cudaStreamDestroy(d->copy_stream);
    d->copy_stream = nullptr;
    d->hb_ready = false;
  }
}
}  // namespace

extern "C" void vae_decoder_destroy(vae_decoder_t* d) {
  if (!d) return;
  release_memory(d);
  delete d;
}

extern "C" vae_status_t vae_decoder_create(const vae_config_t* cfg, const void* const* weights, int n_weights,
                                           vae_decoder_t** out) {
  if (!out) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null out");
  *out = nullptr;
  vae_status_t s = check_config(cfg, nullptr);
  if (s) return s;
  if (!weights || n_weights != count_weights(*cfg))
    return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "expected %d weight tensors, got %d", count_weights(*cfg), n_weights);
  for (int i = 0; i < n_weights; ++i)
    if (!weights[i] || !aligned16(weights[i]))
      return set_err(nullptr, weights[i] ? VAE_ERR_ALIGNMENT : VAE_ERR_INVALID_ARG, 0, 0, "weight %d pointer", i);
  vae_decoder* d = new vae_decoder();
  d->cfg = *cfg;
  d->f32 = cfg->dtype == VAE_FP32 || cfg->dtype == VAE_FP32_TC;
  d->f32tc = cfg->dtype == VAE_FP32_TC;
  d->f8 = cfg->dtype == VAE_FP8;
  int k = 0;
  auto W = [&](void) { return static_cast<const float*>(weights[k++]); };
  auto res_block = [&](ResL& r, int C) -> vae_status_t {
    const float *g1 = W(), *b1 = W(), *w1 = W(), *bb1 = W(), *g2 = W(), *b2 = W(), *w2 = W(), *bb2 = W();
    vae_status_t st = make_norm(d, r.n1, g1, b1, C);
    if (!st) st = make_conv(d, r.c1, w1, bb1, C, C, 1, 1, 1, false, true);
    if (!st) st = make_norm(d, r.n2, g2, b2, C);
    if (!st) st = make_conv(d, r.c2, w2, bb2, C, C, 1, 1, 1, false, true);
    return st;
  };
  const int C0 = cfg->stage_c[0];
  {
    const float* w = W();
    const float* b = W();
    s = make_conv(d, d->conv_in, w, b, cfg->latent_c, C0, 1, 1, 1, true);
  }
  d->mid.resize(cfg->mid_res);
  for (int r = 0; r < cfg->mid_res && !s; ++r) s = res_block(d->mid[r], C0);
  d->has_attn = cfg->mid_attn != 0;
  if (d->has_attn && !s) {
    const float* g = W();
    const float* b = W();
    s = make_norm(d, d->attn.n, g, b, C0);
    for (int q = 0; q < 4 && !s; ++q) {
      const float* w = W();
      const float* bb = W();
      s = dalloc(d, &d->attn.w[q], static_cast<size_t>(C0) * C0 * (d->f32 ? 4 : 2));
      if (!s) s = dalloc(d, &d->attn.b[q], C0 * 4ull);
      if (!s) {
        cudaError_t e = d->f32 ? cudaMemcpy(d->attn.w[q], w, static_cast<size_t>(C0) * C0 * 4, cudaMemcpyDeviceToDevice)
                               : launch_pack_matrix_bf16(w, C0, C0, d->attn.w[q], nullptr);
        if (e == cudaSuccess) e = cudaMemcpy(d->attn.b[q], bb, C0 * 4ull, cudaMemcpyDeviceToDevice);
        if (e != cudaSuccess) s = set_err(&d->err, VAE_ERR_CUDA, 0, 0, "attention weights: %s", cudaGetErrorString(e));
      }
    }
    if (!s && (C0 % 64 || C0 % 16)) s = set_err(&d->err, VAE_ERR_UNSUPPORTED, 0, 0, "attention channels %d", C0);
  }
  d->stages.resize(cfg->n_stages);
  d->ups.resize(std::max(0, cfg->n_stages - 1));
  for (int i = 0; i < cfg->n_stages && !s; ++i) {
    d->stages[i].resize(cfg->n_res[i]);
    for (int r = 0; r < cfg->n_res[i] && !s; ++r) s = res_block(d->stages[i][r], cfg->stage_c[i]);
    if (i + 1 < cfg->n_stages && !s) {
      const float* w = W();
      const float* b = W();
      const int S = cfg->up_t[i] * cfg->up_h[i] * cfg->up_w[i];
      s = make_conv(d, d->ups[i], w, b, cfg->stage_c[i], S * cfg->stage_c[i + 1], cfg->up_t[i], cfg->up_h[i], cfg->up_w[i],
                    false, true);
    }
  }
  if (!s) {
    const int CL = cfg->stage_c[cfg->n_stages - 1];
    const float* g = W();
    const float* b = W();
    s = make_norm(d, d->head_norm, g, b, CL);
    const float* w = W();
    const float* bb = W();
    const int S = cfg->out_d2s_t * cfg->out_d2s_h * cfg->out_d2s_w;
    if (!s)
      s = make_conv(d, d->head, w, bb, CL, cfg->out_c * S, cfg->out_d2s_t, cfg->out_d2s_h, cfg->out_d2s_w, false, false,
                    true);
  }
  if (!s) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) s = set_err(&d->err, VAE_ERR_CUDA, 0, 0, "weight packing: %s", cudaGetErrorString(e));
  }
  if (s) {
    {
      std::lock_guard<std::mutex> lk(g_last_mu);
      g_last = d->err;
    }
    vae_decoder_destroy(d);
    return s;
  }
  *out = d;
  return VAE_OK;
}

// ------------------------------------------------------------------------------ workspace plan
namespace {

struct Plan {
  std::vector<Level> lv;  // level i = stage i; lv[n_stages] = pixel level of conv_out's output
  int Tlat, h, w, B, nph, npw;
  bool first;
  // buffer sizes in bytes
  size_t x_bytes, hin_bytes, c1_bytes, gn_bytes, lat_bytes;
  size_t split_bytes = 0;  // fp32 decoders: each of the high-part and remainder copies of a conv input
  size_t attn_tok, attn_tokp;  // tokens per frame and padded
  size_t q_bytes, s_bytes, p_bytes, vt_bytes;
};

vae_status_t make_plan(vae_decoder* d, int B, int Tlat, int h, int w, int nph, int npw, bool first, Plan& p) {
  const vae_config_t& c = d->cfg;
  p.B = B; p.Tlat = Tlat; p.h = h; p.w = w; p.nph = nph; p.npw = npw; p.first = first;
  p.lv.clear();
  int T = Tlat, sh = 1, sw = 1;
  for (int i = 0; i < c.n_stages; ++i) {
    Level L{};
    L.T = T; L.H = h * sh; L.W = w * sw; L.C = c.stage_c[i];
    vae_status_t s = band_edges(h, nph, sh, 1, L.ph, &d->err);
    if (s) return s;
    s = band_edges(w, npw, sw, 1, L.pw, &d->err);
    if (s) return s;
    p.lv.push_back(L);
    if (i + 1 < c.n_stages) {
      T = c.up_t[i] * T - (first ? c.up_t[i] - 1 : 0);
      sh *= c.up_h[i];
      sw *= c.up_w[i];
    }
  }
  {
    Level L{};
    L.T = T; L.H = h * sh * c.out_d2s_h; L.W = w * sw * c.out_d2s_w; L.C = c.out_c;
    vae_status_t s = band_edges(h, nph, sh * c.out_d2s_h, 1, L.ph, &d->err);
    if (!s) s = band_edges(w, npw, sw * c.out_d2s_w, 1, L.pw, &d->err);
    if (s) return s;
    p.lv.push_back(L);
  }
  const int ab = act_bytes(d), rb = res_bytes(d), cb = c1_bytes(d);
  p.x_bytes = p.hin_bytes = p.c1_bytes = p.gn_bytes = 0;
  for (int i = 0; i < c.n_stages; ++i) {
    const Level& L = p.lv[i];
    const size_t px = static_cast<size_t>(B) * L.H * L.W;
    p.x_bytes = std::max(p.x_bytes, px * L.T * L.C * rb);
    p.hin_bytes = std::max(p.hin_bytes, px * (L.T + 2) * L.C * ab);
    p.c1_bytes = std::max(p.c1_bytes, px * std::max<size_t>(static_cast<size_t>(L.T) * cb, (L.T + 2ull) * ab) * L.C);
    const int groups = c.norm_type == VAE_NORM_GROUP ? c.gn_groups : 0;  // RMS norms keep no partial sums
    p.gn_bytes = std::max(p.gn_bytes, gn_workspace_bytes(nph, npw, B, L.T, groups, L.C));
  }
  const int Clat = d->conv_in.C_in_pad;
  p.lat_bytes = static_cast<size_t>(B) * (Tlat + 2) * h * w * Clat * ab;
  p.hin_bytes = std::max(p.hin_bytes, p.lat_bytes);
  p.split_bytes = d->f32 ? p.hin_bytes : 0;  // every conv input lives in hin
  p.attn_tok = static_cast<size_t>(h) * w;
  p.attn_tokp = round_up(static_cast<int>(p.attn_tok), 64);
  if (d->has_attn) {
    const size_t F = static_cast<size_t>(B) * Tlat, C0 = c.stage_c[0];
    p.q_bytes = F * p.attn_tok * C0 * ab;
    p.vt_bytes = F * C0 * p.attn_tokp * ab;
    p.s_bytes = F * p.attn_tok * p.attn_tok * 4;
    p.p_bytes = F * p.attn_tok * p.attn_tokp * ab;
  } else {
    p.q_bytes = p.vt_bytes = p.s_bytes = p.p_bytes = 0;
  }
  return VAE_OK;
}

size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

struct Bufs {
  char *x, *hin, *c1, *gn, *q, *k, *v, *vt, *s, *p, *o, *hi, *lo;
};

size_t ws_total(const Plan& p) {
  return align_up(p.x_bytes) + align_up(p.hin_bytes) + align_up(p.c1_bytes) + align_up(p.gn_bytes) +
         4 * align_up(p.q_bytes) + align_up(p.vt_bytes) + align_up(p.s_bytes) + align_up(p.p_bytes) +
         2 * align_up(p.split_bytes) + 256;
}

Bufs carve(void* base, const Plan& p) {
  Bufs b{};
  char* c = static_cast<char*>(base);
  b.x = c; c += align_up(p.x_bytes);
  b.hin = c; c += align_up(p.hin_bytes);
  b.c1 = c; c += align_up(p.c1_bytes);
  b.gn = c; c += align_up(p.gn_bytes);
  b.q = c; c += align_up(p.q_bytes);
  b.k = c; c += align_up(p.q_bytes);
  b.v = c; c += align_up(p.q_bytes);
  b.o = c; c += align_up(p.q_bytes);
  b.vt = c; c += align_up(p.vt_bytes);
  b.s = c; c += align_up(p.s_bytes);
  b.p = c; c += align_up(p.p_bytes);
  b.hi = c; c += align_up(p.split_bytes);
  b.lo = c;
  return b;
}

#define ERRP (&d->err)

vae_status_t ensure_ws(vae_decoder* d, const Plan& p) {
  const size_t need = ws_total(p);
  if (need <= d->ws_bytes) return VAE_OK;
  if (d->ws) {
    CK(cudaDeviceSynchronize());
    cudaFree(d->ws);
    d->ws = nullptr;
    d->ws_bytes = 0;
  }
  CK(cudaMalloc(&d->ws, need));
  d->ws_bytes = need;
  return VAE_OK;
}

// all convs of the decoder in schedule order (for cache allocation)
template <typename F>
void for_each_conv(vae_decoder* d, F f) {
  f(d->conv_in, 0);
  for (auto& r : d->mid) { f(r.c1, 0); f(r.c2, 0); }
  for (size_t i = 0; i < d->stages.size(); ++i) {
    for (auto& r : d->stages[i]) { f(r.c1, static_cast<int>(i)); f(r.c2, static_cast<int>(i)); }
    if (i + 1 < d->stages.size()) f(d->ups[i], static_cast<int>(i));
  }
  f(d->head, static_cast<int>(d->stages.size()) - 1);
}

vae_status_t ensure_caches(vae_decoder* d, const Plan& p) {
  bool ok = d->caches_ready;
  vae_status_t st = VAE_OK;
  for_each_conv(d, [&](ConvL& c, int lvl) {
    const Level& L = p.lv[lvl];
    const size_t need = static_cast<size_t>(p.B) * 2 * L.H * L.W * c.C_in_pad * op_bytes(d, c);
    if (c.cache_bytes < need) ok = false;
  });
  if (ok) return VAE_OK;
  CK(cudaDeviceSynchronize());
  for_each_conv(d, [&](ConvL& c, int lvl) {
    if (st) return;
    const Level& L = p.lv[lvl];
    const size_t need = static_cast<size_t>(p.B) * 2 * L.H * L.W * c.C_in_pad * op_bytes(d, c);
    if (c.cache_bytes >= need) return;
    void* q = nullptr;
    if (cudaMalloc(&q, need) != cudaSuccess) {
      st = set_err(&d->err, VAE_ERR_OOM, 0, 0, "cache allocation of %zu bytes failed", need);
      return;
    }
    d->owned.push_back(q);
    c.cache = q;
    c.cache_bytes = need;
  });
  if (!st) d->caches_ready = true;
  return st;
}

// ------------------------------------------------------------------------------ layer runners
struct Ctx {
  vae_decoder* d;
  const Plan* p;
  Bufs b;
  cudaStream_t s;
  bool chunked;                      // keep per-conv caches
  const void* stats_src = nullptr;   // tensor whose group-norm partial sums the last conv produced
};

// Where a conv writes and what its epilogue fuses.
struct ConvOut {
  void* y = nullptr;
  int y_f32 = 0, y_T_alloc = 0, out_ncthw = 0;
  const void* residual = nullptr;
  int res_f32 = 0;
  int drop_first = 0;
  const Level* stats_level = nullptr;  // fuse group-norm partial sums of y at this level (nullptr = no)
  void* y2 = nullptr;                  // copy of y behind 2 cache frames (next conv's operand) ...
  int y2_fp8 = 0;                      // ... in e4m3 (else bf16)
};

// Run conv `c` at level L.  `in` is its input buffer (conv operand dtype, B x (2+T) frames, frames 0..1
// the temporal cache).
vae_status_t run_conv(Ctx& x, ConvL& c, const Level& L, char* in, const ConvOut& o) {
  vae_decoder* d = x.d;
  const int B = x.p->B, T = L.T, Ta = T + 2;
  const int64_t frame_bytes = static_cast<int64_t>(L.H) * L.W * c.C_in_pad * op_bytes(d, c);
  const bool use_cache = x.chunked && !x.p->first;
  x.stats_src = nullptr;
  void* y = o.y;
  const int y_f32 = o.y_f32, y_T_alloc = o.y_T_alloc, out_ncthw = o.out_ncthw, res_f32 = o.res_f32;
  const void* residual = o.residual;
  const int drop_first = o.drop_first;
  if (use_cache) {
    Prof pr(d, x.s, K_COPY, 0, 4.0 * B * frame_bytes);
    CK(launch_copy_frames(c.cache, 2, 0, in, Ta, 0, 2, B, frame_bytes, x.s));
  }
  const double conv_flops = 2.0 * 27 * c.C_in * c.C_out * static_cast<double>(B) * T * L.H * L.W;
  const char* xin = in + (use_cache ? 0 : 2 * frame_bytes);
  const int cache_frames = use_cache ? 2 : 0;
  if (c.tc) {
    ConvTcArgs a{};
    a.mode = 0;
    a.B = B; a.T = T; a.H = L.H; a.W = L.W;
    a.C_in_pad = c.C_in_pad; a.T_in = T + cache_frames; a.x_T_alloc = Ta; a.cache_frames = cache_frames;
    a.nph = x.p->nph; a.npw = x.p->npw; a.ph_edges = L.ph; a.pw_edges = L.pw;
    a.x = xin; a.w = c.w; a.N_real = c.C_out; a.N_pad = c.N_pad; a.bias = c.bias;
    a.residual = residual; a.res_f32 = res_f32; a.res_T_alloc = T;
    a.y = y; a.out_f32 = y_f32; a.out_ncthw = out_ncthw; a.y_T_alloc = y_T_alloc;
    a.d2s_t = c.st; a.d2s_h = c.sh; a.d2s_w = c.sw; a.drop_first = drop_first;
    a.fp8 = c.fp8; a.wscale = c.wscale; a.natural = c.natural; a.tap_stacked = c.tap;
    if (c.tf32) {
      // 3 x TF32: split the whole input (cache frames included) into high parts and remainders
      const int64_t n = static_cast<int64_t>(B) * Ta * (frame_bytes / 4);
      if (static_cast<size_t>(n) * 4 > x.p->split_bytes)
        return set_err(&d->err, VAE_ERR_UNSUPPORTED, 0, 0, "conv input larger than the split buffers");
      {
        Prof pr(d, x.s, K_CAST, 0, 12.0 * n);
        CK(launch_split_tf32(reinterpret_cast<const float*>(in), reinterpret_cast<float*>(x.b.hi),
                             reinterpret_cast<float*>(x.b.lo), n, x.s));
      }
      a.tf32 = 1;
      a.x = x.b.hi + (xin - in);
      a.x_lo = x.b.lo + (xin - in);
    }
    const int Cd = c.C_out / (c.st * c.sh * c.sw);
    const int G = d->cfg.gn_groups;  // (ignored, possibly 0, by channel-RMS decoders)
    const int cpg = (G > 0 && Cd % G == 0) ? Cd / G : 0;
    // fused sums cost one warp reduction per group per 32 columns: worth it from 16 channels per group
    const bool fuse = o.stats_level && d->cfg.norm_type == VAE_NORM_GROUP && !out_ncthw && Cd % 32 == 0 && cpg >= 16 &&
                      (cpg < 32 ? 32 % cpg == 0 : cpg % 32 == 0);
    if (fuse) {
      CK(cudaMemsetAsync(x.b.gn, 0, gn_partials_bytes(x.p->nph, x.p->npw, B, o.stats_level->T, G), x.s));
      a.gn_partials = x.b.gn;
      a.gn_groups = G;
    }
    if (o.y2) {
      const int64_t f2 = static_cast<int64_t>(L.H) * c.sh * L.W * c.sw * Cd * (o.y2_fp8 ? 1 : 2);
      a.y2 = static_cast<char*>(o.y2) + 2 * f2;
      a.y2_T_alloc = (o.stats_level ? o.stats_level->T : T) + 2;
      a.y2_fp8 = o.y2_fp8;
    }
    {
      Prof pr(d, x.s, &c == &d->head ? K_CONV_HEAD : K_CONV_TC, conv_flops, 0);
      CK(launch_conv_tc(a, x.s));
    }
    if (fuse) x.stats_src = y;
  } else {
    ConvSimtArgs a{};
    a.B = B; a.T = T; a.H = L.H; a.W = L.W; a.C_in = c.C_in; a.C_out = c.C_out;
    a.T_in = T + cache_frames; a.x_T_alloc = Ta; a.cache_frames = cache_frames;
    a.x = xin; a.x_f32 = d->f32; a.w = static_cast<const float*>(c.w); a.bias = c.bias;
    a.residual = residual; a.res_f32 = res_f32; a.res_T_alloc = T;
    a.y = y; a.out_f32 = y_f32; a.out_ncthw = out_ncthw; a.y_T_alloc = y_T_alloc;
    a.d2s_t = c.st; a.d2s_h = c.sh; a.d2s_w = c.sw; a.drop_first = drop_first;
    a.nph = x.p->nph; a.npw = x.p->npw; a.ph_edges = L.ph; a.pw_edges = L.pw;
    Prof pr(d, x.s, K_CONV_SIMT, conv_flops, 0);
    CK(launch_conv_simt(a, x.s));
  }
  if (x.chunked) {
    Prof pr(d, x.s, K_COPY, 0, 4.0 * B * frame_bytes);
    // keep the last 2 frames of this conv's (padded) input sequence for the next chunk
    if (use_cache || T >= 2) {
      const int last = 2 + T;  // frames [last-2, last) of the input are the newest two
      CK(launch_copy_frames(in, Ta, last - 2, c.cache, 2, 0, 2, B, frame_bytes, x.s));
    } else {  // first chunk of one frame: the padded sequence ends x0, x0
      CK(launch_copy_frames(in, Ta, 2, c.cache, 2, 0, 1, B, frame_bytes, x.s));
      CK(launch_copy_frames(in, Ta, 2, c.cache, 2, 1, 1, B, frame_bytes, x.s));
    }
  }
  return VAE_OK;
}

// GN (+SiLU) of src (B x T frames, dtype src_f32) into hin frames [2, 2+T), in the operand type of the
// conv that reads them (out_fp8: e4m3)
vae_status_t run_gn(Ctx& x, const NormL& n, const Level& L, const void* src, int src_f32, int silu, bool out_fp8) {
  vae_decoder* d = x.d;
  GnArgs g{};
  g.B = x.p->B; g.T = L.T; g.H = L.H; g.W = L.W; g.C = L.C; g.groups = d->cfg.gn_groups;
  g.eps = d->cfg.gn_eps; g.silu = silu;
  g.nph = x.p->nph; g.npw = x.p->npw; g.ph_edges = L.ph; g.pw_edges = L.pw;
  g.x = src; g.x_f32 = src_f32; g.x_T_alloc = L.T;
  const int ob = out_fp8 ? 1 : act_bytes(d);
  const int64_t frame_bytes = static_cast<int64_t>(L.H) * L.W * L.C * ob;
  g.y = x.b.hin + 2 * frame_bytes; g.y_f32 = d->f32; g.y_T_alloc = L.T + 2; g.y_fp8 = out_fp8;
  g.gamma = n.gamma; g.beta = n.beta;
  g.partials = x.b.gn;
  const double elems = static_cast<double>(g.B) * L.T * L.H * L.W * L.C;
  if (d->cfg.norm_type == VAE_NORM_CHANNEL_RMS) {  // per pixel: no statistics pass
    Prof pr(d, x.s, K_RMS, 0, elems * ((src_f32 ? 4 : 2) + ob));
    CK(launch_rms(g, x.s));
    return VAE_OK;
  }
  if (x.stats_src != src) {  // not already summed by the producing conv's epilogue
    Prof pr(d, x.s, K_GN_STATS, 0, elems * (src_f32 ? 4 : 2));
    CK(launch_gn_stats(g, x.s));
  }
  {
    Prof pr(d, x.s, K_GN_APPLY, 0, elems * ((src_f32 ? 4 : 2) + ob));
    CK(launch_gn_apply(g, x.s));
  }
  return VAE_OK;
}

// One residual block.  With up_copy, conv2 also stores a copy of the new residual stream into the
// conv1 buffer (behind 2 cache frames) for the up-sampling conv that follows, in that conv's operand
// type (e4m3 when up_fp8, else bf16); *copied says so.
vae_status_t run_resblock(Ctx& x, ResL& r, const Level& L, bool up_copy = false, bool* copied = nullptr,
                          bool up_fp8 = false) {
  vae_decoder* d = x.d;
  const int rf = res_bytes(d) == 4, cf = c1_bytes(d) == 4;
  vae_status_t s = run_gn(x, r.n1, L, x.b.x, rf, 1, r.c1.fp8);
  ConvOut o1;
  o1.y = x.b.c1; o1.y_f32 = cf; o1.y_T_alloc = L.T; o1.stats_level = &L;
  if (!s) s = run_conv(x, r.c1, L, x.b.hin, o1);
  if (!s) s = run_gn(x, r.n2, L, x.b.c1, cf, 1, r.c2.fp8);
  ConvOut o2;  // in-place residual add
  o2.y = x.b.x; o2.y_f32 = rf; o2.y_T_alloc = L.T; o2.residual = x.b.x; o2.res_f32 = rf; o2.stats_level = &L;
  const bool cp = up_copy && r.c2.tc && !d->f32 && L.C % 32 == 0;
  if (cp) {
    o2.y2 = x.b.c1;
    o2.y2_fp8 = up_fp8;
  }
  if (!s) s = run_conv(x, r.c2, L, x.b.hin, o2);
  if (copied) *copied = cp && !s;
  return s;
}

vae_status_t run_attention(Ctx& x, const Level& L) {
  vae_decoder* d = x.d;
  const int C = L.C, F = x.p->B * L.T;
  const int tok = L.H * L.W, tokp = static_cast<int>(x.p->attn_tokp);
  const int rf = res_bytes(d) == 4;
  x.stats_src = nullptr;
  // GN without SiLU into hn (= buffer q's neighbour o, reused before O is produced)
  {
    GnArgs g{};
    g.B = x.p->B; g.T = L.T; g.H = L.H; g.W = L.W; g.C = C; g.groups = d->cfg.gn_groups;
    g.eps = d->cfg.gn_eps; g.silu = 0;
    g.nph = x.p->nph; g.npw = x.p->npw; g.ph_edges = L.ph; g.pw_edges = L.pw;
    g.x = x.b.x; g.x_f32 = rf; g.x_T_alloc = L.T;
    g.y = x.b.o; g.y_f32 = d->f32; g.y_T_alloc = L.T;
    g.gamma = d->attn.n.gamma; g.beta = d->attn.n.beta;
    g.partials = x.b.gn;
    const double elems = static_cast<double>(g.B) * L.T * L.H * L.W * C;
    if (d->cfg.norm_type == VAE_NORM_CHANNEL_RMS) {
      Prof pr(d, x.s, K_RMS, 0, elems * ((rf ? 4 : 2) + act_bytes(d)));
      CK(launch_rms(g, x.s));
    } else {
      {
        Prof pr(d, x.s, K_GN_STATS, 0, elems * (rf ? 4 : 2));
        CK(launch_gn_stats(g, x.s));
      }
      {
        Prof pr(d, x.s, K_GN_APPLY, 0, elems * ((rf ? 4 : 2) + act_bytes(d)));
        CK(launch_gn_apply(g, x.s));
      }
    }
  }
  const float scale = 1.0f / std::sqrt(static_cast<float>(C));
  const int64_t M = static_cast<int64_t>(F) * tok;
  if (d->f32) {
    const float* hn = reinterpret_cast<const float*>(x.b.o);
    float* qkv[3] = {reinterpret_cast<float*>(x.b.q), reinterpret_cast<float*>(x.b.k), reinterpret_cast<float*>(x.b.v)};
    for (int i = 0; i < 3; ++i)
      CK(launch_gemm_simt(hn, static_cast<const float*>(d->attn.w[i]), qkv[i], d->attn.b[i], nullptr, static_cast<int>(M), C,
                          C, 1, 0, 0, 0, C, 1, 1.0f, x.s));
    float* S = reinterpret_cast<float*>(x.b.s);
    CK(launch_gemm_simt(qkv[0], qkv[1], S, nullptr, nullptr, tok, tok, C, F, static_cast<int64_t>(tok) * C,
                        static_cast<int64_t>(tok) * C, static_cast<int64_t>(tok) * tok, C, 1, scale, x.s));
    float* P = reinterpret_cast<float*>(x.b.p);
    CK(launch_softmax_rows(S, P, 1, F * tok, tok, tok, x.s));
    // O = P V: B element (n = c, k = token) = V[token * C + c]
    float* O = reinterpret_cast<float*>(x.b.o);
    CK(launch_gemm_simt(P, qkv[2], O, nullptr, nullptr, tok, C, tok, F, static_cast<int64_t>(tok) * tok,
                        static_cast<int64_t>(tok) * C, static_cast<int64_t>(tok) * C, 1, C, 1.0f, x.s));
    float* X = reinterpret_cast<float*>(x.b.x);
    CK(launch_gemm_simt(O, static_cast<const float*>(d->attn.w[3]), X, d->attn.b[3], X, static_cast<int>(M), C, C, 1, 0,
                        0, 0, C, 1, 1.0f, x.s));
    return VAE_OK;
  }
  auto gemm = [&](const void* A, const void* Bm, void* D, const float* bias, int Mm, int N, int K, int batch,
                  int64_t sa, int64_t sb, int64_t sd, int64_t ldd, float alpha, int out_f32, const void* res,
                  int r_f32) -> vae_status_t {
    ConvTcArgs a{};
    a.mode = 1;
    a.M = Mm; a.K = K; a.batch = batch; a.stride_a = sa; a.stride_b = sb; a.stride_d = sd; a.alpha = alpha;
    a.x = A; a.w = Bm; a.N_real = N; a.N_pad = round_up(N, 16); a.bias = bias;
    a.residual = res; a.res_f32 = r_f32; a.y = D; a.out_f32 = out_f32; a.ldd = ldd;
    a.d2s_t = a.d2s_h = a.d2s_w = 1;
    Prof pr(d, x.s, K_GEMM_TC, 2.0 * Mm * N * K * batch, 0);
    CK(launch_conv_tc(a, x.s));
    return VAE_OK;
  };
  vae_status_t s = VAE_OK;
  char* qkv[3] = {x.b.q, x.b.k, x.b.v};
  for (int i = 0; i < 3 && !s; ++i)
    s = gemm(x.b.o, d->attn.w[i], qkv[i], d->attn.b[i], static_cast<int>(M), C, C, 1, 0, 0, 0, 0, 1.0f, 0, nullptr, 0);
  if (s) return s;
  {
    Prof pr(d, x.s, K_TRANSPOSE, 0, 2.0 * F * tok * C * 2);
    CK(launch_transpose_bf16(x.b.v, x.b.vt, F, tok, C, x.s));  // V^T [F, C, tokp], zero padded
  }
  s = gemm(x.b.q, x.b.k, x.b.s, nullptr, tok, tok, C, F, static_cast<int64_t>(tok) * C, static_cast<int64_t>(tok) * C,
           static_cast<int64_t>(tok) * tok, 0, scale, 1, nullptr, 0);
  if (s) return s;
  {
    Prof pr(d, x.s, K_SOFTMAX, 0, static_cast<double>(F) * tok * (tok * 4.0 + tokp * 2.0));
    CK(launch_softmax_rows(reinterpret_cast<const float*>(x.b.s), x.b.p, 0, F * tok, tok, tokp, x.s));
  }
  s = gemm(x.b.p, x.b.vt, x.b.o, nullptr, tok, C, tokp, F, static_cast<int64_t>(tok) * tokp,
           static_cast<int64_t>(C) * tokp, static_cast<int64_t>(tok) * C, 0, 1.0f, 0, nullptr, 0);
  if (s) return s;
  return gemm(x.b.o, d->attn.w[3], x.b.x, d->attn.b[3], static_cast<int>(M), C, C, 1, 0, 0, 0, 0, 1.0f, rf, x.b.x, rf);
}

// Decode one chunk (or the whole latent) into out (NCTHW, out_T_alloc frames per (b, c)).
// lat_full = (T, H, W) of the latent tensor, lat_box = (t0, h0, w0) of the decoded box.
// Decode p.B = n_boxes x B_lat items: the latent boxes lat_boxes[3 i .. 3 i + 2] (t0, h0, w0) of the B_lat items
// of `latent` (full extent lat_full), box after box along the batch (tiles of one shape decode together).
vae_status_t run_decode(vae_decoder* d, const Plan& p, const float* latent, const int lat_full[3], const int* lat_boxes,
                        int n_boxes, void* out, int out_T_alloc, bool chunked, cudaStream_t s) {
  Ctx x{d, &p, carve(d->ws, p), s, chunked};
  const vae_config_t& c = d->cfg;
  const int rf = res_bytes(d) == 4;
  vae_status_t st = VAE_OK;
  // latent box NCTHW fp32 -> channels-last conv input (frames 2.. of hin), channels zero-padded
  {
    const Level& L0 = p.lv[0];
    const int Cp = d->conv_in.C_in_pad;
    const int64_t fb = static_cast<int64_t>(p.h) * p.w * Cp * act_bytes(d);
    if (n_boxes < 1 || p.B % n_boxes) return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "bad latent box batch");
    const int Bl = p.B / n_boxes;
    for (int i = 0; i < n_boxes; ++i) {
      const int* bx = lat_boxes + 3 * i;
      Prof pr(d, s, K_LATENT, 0, static_cast<double>(Bl) * p.Tlat * p.h * p.w * (c.latent_c * 4.0 + Cp * act_bytes(d)));
      CK(launch_latent_to_cl(latent, Bl, c.latent_c, lat_full[0], lat_full[1], lat_full[2], bx[0], p.Tlat, bx[1], p.h,
                             bx[2], p.w, Cp, x.b.hin + 2 * fb + static_cast<int64_t>(i) * Bl * (p.Tlat + 2) * fb, d->f32,
                             p.Tlat + 2, s));
    }
    ConvOut o;
    o.y = x.b.x; o.y_f32 = rf; o.y_T_alloc = L0.T; o.stats_level = &L0;
    st = run_conv(x, d->conv_in, L0, x.b.hin, o);
    if (st) return st;
  }
  for (auto& r : d->mid) {
    st = run_resblock(x, r, p.lv[0]);
    if (st) return st;
  }
  if (d->has_attn) {
    st = run_attention(x, p.lv[0]);
    if (st) return st;
  }
  for (int i = 0; i < c.n_stages; ++i) {
    const Level& L = p.lv[i];
    bool copied = false;
    for (size_t r = 0; r < d->stages[i].size(); ++r) {
      const bool last = r + 1 == d->stages[i].size() && i + 1 < c.n_stages;
      st = run_resblock(x, d->stages[i][r], L, last, &copied, last && d->ups[i].fp8);
      if (st) return st;
    }
    if (i + 1 < c.n_stages) {
      // conv input = the residual stream in the conv dtype, behind 2 cache frames: either the copy
      // the last conv2 stored, or a cast of the residual stream
      const int64_t fe = static_cast<int64_t>(L.H) * L.W * L.C;
      char* in = x.b.c1;
      if (!copied) {
        in = x.b.hin;
        const int ob = op_bytes(d, d->ups[i]);
        Prof pr(d, s, K_CAST, 0, static_cast<double>(p.B) * L.T * fe * (res_bytes(d) + ob));
        CK(launch_cast_frames(x.b.x, rf, L.T, x.b.hin + 2 * fe * ob, d->ups[i].fp8 ? 2 : (d->f32 ? 1 : 0), L.T + 2, p.B,
                              L.T, fe, s));
      }
      ConvOut o;
      o.y = x.b.x; o.y_f32 = rf; o.y_T_alloc = p.lv[i + 1].T; o.drop_first = p.first ? 1 : 0;
      o.stats_level = &p.lv[i + 1];
      st = run_conv(x, d->ups[i], L, in, o);
      if (st) return st;
    }
  }
  const Level& LL = p.lv[c.n_stages - 1];
  st = run_gn(x, d->head_norm, LL, x.b.x, rf, 1, d->head.fp8);
  if (st) return st;
  ConvOut o;
  o.y = out; o.y_f32 = d->f32; o.y_T_alloc = out_T_alloc; o.out_ncthw = 1; o.drop_first = p.first ? 1 : 0;
  return run_conv(x, d->head, LL, x.b.hin, o);
}

vae_status_t check_shape(vae_decoder* d, const int64_t* shp, int nph, int npw) {
  if (!shp) return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "null shape");
  if (shp[0] <= 0 || shp[1] != d->cfg.latent_c || shp[2] <= 0 || shp[3] <= 0 || shp[4] <= 0)
    return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "latent shape mismatch");
  if (shp[0] > 64 || shp[2] > 4096 || shp[3] > 8192 || shp[4] > 8192)
    return set_err(&d->err, VAE_ERR_UNSUPPORTED, 0, 0, "latent too large");
  if (nph < 1 || npw < 1 || nph > VAE_MAX_PATCHES || npw > VAE_MAX_PATCHES)
    return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "patch counts %d x %d", nph, npw);
  return VAE_OK;
}

vae_status_t check_gn_range(vae_decoder* d, const Plan& p) {
  // exact integer group sums need fewer than 2^23 elements per (frame, group)
  if (d->cfg.norm_type != VAE_NORM_GROUP) return VAE_OK;
  for (int i = 0; i < d->cfg.n_stages; ++i) {
    const Level& L = p.lv[i];
    const double n = static_cast<double>(L.C / d->cfg.gn_groups) * L.H * L.W;
    if (n >= 8388608.0)
      return set_err(&d->err, VAE_ERR_UNSUPPORTED, 0, 0, "group of %.0f elements exceeds the exact-sum range", n);
  }
  return VAE_OK;
}

}  // namespace

extern "C" vae_status_t vae_decoder_reserve(vae_decoder_t* d, const int64_t shp[5], int nph, int npw) {
  if (!d) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null decoder");
  vae_status_t s = check_shape(d, shp, nph, npw);
  if (s) return s;
  Plan p;
  s = make_plan(d, static_cast<int>(shp[0]), static_cast<int>(shp[2]), static_cast<int>(shp[3]),
                static_cast<int>(shp[4]), nph, npw, false, p);
  if (s) return s;
  return ensure_ws(d, p);
}

extern "C" vae_status_t vae_decode(vae_decoder_t* d, const void* latent, const int64_t shp[5], void* out, int nph,
                                   int npw, void* stream) {
  if (!d) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null decoder");
  if (!latent || !out) return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "null latent or out");
  if (!aligned16(latent) || !aligned16(out)) return set_err(&d->err, VAE_ERR_ALIGNMENT, 0, 0, "latent/out not 16-byte aligned");
  vae_status_t s = check_shape(d, shp, nph, npw);
  if (s) return s;
  Plan p;
  s = make_plan(d, static_cast<int>(shp[0]), static_cast<int>(shp[2]), static_cast<int>(shp[3]),
                static_cast<int>(shp[4]), nph, npw, true, p);
  if (s) return s;
  s = check_gn_range(d, p);
  if (s) return s;
  s = ensure_ws(d, p);
  if (s) return s;
  const int full[3] = {static_cast<int>(shp[2]), static_cast<int>(shp[3]), static_cast<int>(shp[4])};
  const int box[3] = {0, 0, 0};
  return run_decode(d, p, static_cast<const float*>(latent), full, box, 1, out, p.lv.back().T, false,
                    static_cast<cudaStream_t>(stream));
}

extern "C" vae_status_t vae_decode_chunk(vae_decoder_t* d, const void* latent, const int64_t shp[5], int first_chunk,
                                         void* out, int nph, int npw, void* stream) {
  if (!d) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null decoder");
  if (!latent || !out) return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "null latent or out");
  if (!aligned16(latent) || !aligned16(out)) return set_err(&d->err, VAE_ERR_ALIGNMENT, 0, 0, "latent/out not 16-byte aligned");
  vae_status_t s = check_shape(d, shp, nph, npw);
  if (s) return s;
  if (!first_chunk && !d->caches_ready)
    return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "a later chunk came before the first chunk");
  if (!first_chunk && (shp[0] != d->cache_shape[0] || shp[3] != d->cache_shape[3] || shp[4] != d->cache_shape[4] ||
                       nph != d->cache_nph || npw != d->cache_npw))
    return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "chunk shape or patch grid differs from the first chunk");
  Plan p;
  s = make_plan(d, static_cast<int>(shp[0]), static_cast<int>(shp[2]), static_cast<int>(shp[3]),
                static_cast<int>(shp[4]), nph, npw, first_chunk != 0, p);
  if (s) return s;
  s = check_gn_range(d, p);
  if (s) return s;
  Plan pmax;  // caches and workspace sized for a non-first chunk of this size
  s = make_plan(d, static_cast<int>(shp[0]), static_cast<int>(shp[2]), static_cast<int>(shp[3]),
                static_cast<int>(shp[4]), nph, npw, false, pmax);
  if (s) return s;
  s = ensure_ws(d, pmax);
  if (s) return s;
  if (first_chunk) d->caches_ready = false;
  s = ensure_caches(d, p);
  if (s) return s;
  for (int i = 0; i < 5; ++i) d->cache_shape[i] = shp[i];
  d->cache_nph = nph;
  d->cache_npw = npw;
  const int full[3] = {static_cast<int>(shp[2]), static_cast<int>(shp[3]), static_cast<int>(shp[4])};
  const int box[3] = {0, 0, 0};
  return run_decode(d, p, static_cast<const float*>(latent), full, box, 1, out, p.lv.back().T, true,
                    static_cast<cudaStream_t>(stream));
}

// Decode from and to host memory: temporal chunks (chunk 0 = latent frame 0, then frames_per_chunk frames)
// go through vae_decode_chunk on `stream`, while a second stream copies the next latent chunk in and the
// previous chunk's pixels out (double-buffered device chunks), so the copies overlap the decode.
extern "C" vae_status_t vae_decode_host(vae_decoder_t* d, const void* latent_host, const int64_t shp[5],
                                        void* out_host, int nph, int npw, int frames_per_chunk, void* stream) {
  if (!d) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null decoder");
  if (!latent_host || !out_host || !shp) return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "null argument");
  vae_status_t s = check_shape(d, shp, nph, npw);
  if (s) return s;
  const vae_config_t& c = d->cfg;
  int st = c.out_d2s_t, ss = c.out_d2s_h;
  for (int i = 0; i + 1 < c.n_stages; ++i) {
    st *= c.up_t[i];
    ss *= c.up_h[i];
  }
  const int B = static_cast<int>(shp[0]), Cl = static_cast<int>(shp[1]), T = static_cast<int>(shp[2]);
  const int h = static_cast<int>(shp[3]), w = static_cast<int>(shp[4]);
  const int per = frames_per_chunk > 0 ? frames_per_chunk : std::max(1, (T - 1 + 4) / 5);
  const int To = st * (T - 1) + 1, Ho = ss * h, Wo = ss * w, Co = c.out_c;
  const size_t ob = d->f32 ? 4 : 2;
  const size_t lat_frame = static_cast<size_t>(h) * w * 4, out_frame = static_cast<size_t>(Ho) * Wo * ob;
  const int max_lat = std::min(per, std::max(T - 1, 1)), max_out = std::max(1, st * max_lat);
  const size_t lat_bytes = static_cast<size_t>(B) * Cl * max_lat * lat_frame;
  const size_t out_bytes = static_cast<size_t>(B) * Co * max_out * out_frame;
  // everything allocated before anything is enqueued: the chunk buffers, and the workspace of the
  // largest chunk (so no chunk call has to grow it in the middle of the stream)
  if (!d->hb_ready) {
    CK(cudaStreamCreateWithFlags(&d->copy_stream, cudaStreamNonBlocking));
    for (cudaEvent_t& e : d->hb_ev) CK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    d->hb_ready = true;
  }
  if (d->hb_lat_bytes < lat_bytes || d->hb_out_bytes < out_bytes) {
    CK(cudaDeviceSynchronize());
    for (int i = 0; i < 2; ++i) {
      if (d->hb_lat[i]) cudaFree(d->hb_lat[i]);
      if (d->hb_out[i]) cudaFree(d->hb_out[i]);
      d->hb_lat[i] = d->hb_out[i] = nullptr;
    }
    d->hb_lat_bytes = d->hb_out_bytes = 0;
    for (int i = 0; i < 2; ++i) {
      CK(cudaMalloc(&d->hb_lat[i], lat_bytes));
      CK(cudaMalloc(&d->hb_out[i], out_bytes));
    }
    d->hb_lat_bytes = lat_bytes;
    d->hb_out_bytes = out_bytes;
  }
  {
    Plan pmax;
    s = make_plan(d, B, max_lat, h, w, nph, npw, false, pmax);
    if (!s) s = ensure_ws(d, pmax);
    if (s) return s;
  }
  cudaStream_t cs = static_cast<cudaStream_t>(stream), cp = d->copy_stream;
  cudaEvent_t* ev = d->hb_ev;
  CK(cudaEventRecord(ev[6], cs));  // the copies start after what `stream` already holds
  CK(cudaStreamWaitEvent(cp, ev[6], 0));
  const char* lat = static_cast<const char*>(latent_host);
  char* out = static_cast<char*>(out_host);
  int t0 = 0;
  for (int i = 0; t0 < T; ++i) {
    const int n = i == 0 ? 1 : std::min(per, T - t0);
    const int buf = i & 1;
    // latent frames [t0, t0 + n) of every (b, c) plane -> hb_lat[buf] (free once chunk i - 2 decoded)
    if (i >= 2) CK(cudaStreamWaitEvent(cp, ev[2 + buf], 0));
    CK(cudaMemcpy2DAsync(d->hb_lat[buf], n * lat_frame, lat + t0 * lat_frame, T * lat_frame, n * lat_frame,
                         static_cast<size_t>(B) * Cl, cudaMemcpyHostToDevice, cp));
    CK(cudaEventRecord(ev[buf], cp));
    // decode the chunk into hb_out[buf] (free once chunk i - 2's pixels are out)
    CK(cudaStreamWaitEvent(cs, ev[buf], 0));
    if (i >= 2) CK(cudaStreamWaitEvent(cs, ev[4 + buf], 0));
    const int64_t cshp[5] = {B, Cl, n, h, w};
    s = vae_decode_chunk(d, d->hb_lat[buf], cshp, i == 0, d->hb_out[buf], nph, npw, stream);
    if (s) return s;
    CK(cudaEventRecord(ev[2 + buf], cs));
    // its pixel frames [f0, f0 + nf) of every (b, c) plane -> out_host
    const int f0 = i == 0 ? 0 : 1 + st * (t0 - 1), nf = i == 0 ? 1 : st * n;
    CK(cudaStreamWaitEvent(cp, ev[2 + buf], 0));
    CK(cudaMemcpy2DAsync(out + f0 * out_frame, To * out_frame, d->hb_out[buf], nf * out_frame, nf * out_frame,
                         static_cast<size_t>(B) * Co, cudaMemcpyDeviceToHost, cp));
    CK(cudaEventRecord(ev[4 + buf], cp));
    t0 += n;
  }
  CK(cudaEventRecord(ev[7], cp));  // `stream` ends with the last copy
  CK(cudaStreamWaitEvent(cs, ev[7], 0));
  return VAE_OK;
}

#undef ERRP

// ================================================================================ tile plan
extern "C" vae_status_t vae_tile_plan(const int lat[3], const int tile[3], const int ovl[3], int scale_t, int scale_s,
                                      int causal_t, vae_tile_t* tiles, int* n_tiles) {
  if (!lat || !tile || !ovl || !n_tiles || scale_t < 1 || scale_s < 1)
    return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "tile plan arguments");
  int starts[3][4096], ext[3][4096], cnt[3];
  int px0[3][4096], pxn[3][4096];
  for (int a = 0; a < 3; ++a) {
    if (lat[a] <= 0 || tile[a] <= 0 || ovl[a] < 0 || ovl[a] >= tile[a])
      return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "axis %d: length %d tile %d overlap %d", a, lat[a], tile[a], ovl[a]);
    const int stride = tile[a] - ovl[a];
    int n = 0, s = 0;
    while (true) {
      if (n >= 4096) return set_err(nullptr, VAE_ERR_UNSUPPORTED, 0, 0, "too many tiles on axis %d", a);
      starts[a][n] = s;
      ext[a][n] = std::min(tile[a], lat[a] - s);
      ++n;
      if (s + tile[a] >= lat[a]) break;
      s += stride;
    }
    cnt[a] = n;
    const int sc = a == 0 ? scale_t : scale_s;
    for (int i = 0; i < n; ++i) {
      px0[a][i] = sc * starts[a][i];
      pxn[a][i] = (a == 0 && causal_t) ? sc * (ext[a][i] - 1) + 1 : sc * ext[a][i];
    }
  }
  const long total = static_cast<long>(cnt[0]) * cnt[1] * cnt[2];
  if (!tiles) {
    *n_tiles = static_cast<int>(std::min<long>(total, 0x7fffffff));
    return VAE_OK;
  }
  if (total > *n_tiles) {
    *n_tiles = static_cast<int>(std::min<long>(total, 0x7fffffff));
    return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "tile array holds %d, plan needs %ld", *n_tiles, total);
  }
  int k = 0;
  for (int it = 0; it < cnt[0]; ++it)
    for (int ih = 0; ih < cnt[1]; ++ih)
      for (int iw = 0; iw < cnt[2]; ++iw) {
        vae_tile_t& t = tiles[k++];
        const int idx[3] = {it, ih, iw};
        for (int a = 0; a < 3; ++a) {
          const int i = idx[a];
          t.lat[2 * a] = starts[a][i];
          t.lat[2 * a + 1] = ext[a][i];
          t.pix[2 * a] = px0[a][i];
          t.pix[2 * a + 1] = pxn[a][i];
          t.ovl[2 * a] = i > 0 ? px0[a][i - 1] + pxn[a][i - 1] - px0[a][i] : 0;
          t.ovl[2 * a + 1] = i + 1 < cnt[a] ? px0[a][i] + pxn[a][i] - px0[a][i + 1] : 0;
        }
      }
  *n_tiles = k;
  return VAE_OK;
}

extern "C" vae_status_t vae_patch_edges(int length, int n, int scale, int reach, int* edges) {
  if (!edges) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null edges");
  return band_edges(length, n, scale, reach, edges, nullptr);
}

#define ERRP (&d->err)
extern "C" vae_status_t vae_decode_tiled(vae_decoder_t* d, const void* latent, const int64_t shp[5], void* out,
                                         const int tile_thw[3], const int ovl_thw[3], void* stream) {
  if (!d) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null decoder");
  if (!latent || !out || !tile_thw || !ovl_thw) return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "null argument");
  if (!aligned16(latent) || !aligned16(out)) return set_err(&d->err, VAE_ERR_ALIGNMENT, 0, 0, "latent/out not 16-byte aligned");
  vae_status_t s = check_shape(d, shp, 1, 1);
  if (s) return s;
  const vae_config_t& c = d->cfg;
  int st = c.out_d2s_t, ss = c.out_d2s_h;
  for (int i = 0; i + 1 < c.n_stages; ++i) {
    st *= c.up_t[i];
    ss *= c.up_h[i];
  }
  const int lat[3] = {static_cast<int>(shp[2]), static_cast<int>(shp[3]), static_cast<int>(shp[4])};
  std::vector<vae_tile_t> tl(VAE_MAX_TILES);
  int n = VAE_MAX_TILES;
  constexpr size_t kTileBatchWorkspace = 16ull << 30;  // workspace budget of one batch of equal-shape tiles
  s = vae_tile_plan(lat, tile_thw, ovl_thw, st, ss, 1, tl.data(), &n);
  if (s) return set_err(&d->err, s, 0, 0, "tile plan failed (%d tiles max)", VAE_MAX_TILES);
  const int B = static_cast<int>(shp[0]);
  const int ob = d->f32 ? 4 : 2;
  auto tile_bytes = [&](int i) {
    return static_cast<size_t>(B) * c.out_c * tl[i].pix[1] * tl[i].pix[3] * tl[i].pix[5] * ob;
  };
  // Tiles of one latent shape decode together as one batch of K x B items (each item's arithmetic is
  // the same whatever else is in the batch), K bounded by the workspace budget; a batch's tile outputs
  // are contiguous, in the batch's tile order.
  std::vector<std::vector<int>> batches;
  {
    std::vector<char> taken(n, 0);
    for (int i = 0; i < n; ++i) {
      if (taken[i]) continue;
      std::vector<int> grp;
      for (int j = i; j < n; ++j)
        if (!taken[j] && tl[j].lat[1] == tl[i].lat[1] && tl[j].lat[3] == tl[i].lat[3] && tl[j].lat[5] == tl[i].lat[5]) {
          grp.push_back(j);
          taken[j] = 1;
        }
      int K = tile_bytes(i) % 256 == 0 ? static_cast<int>(grp.size()) : 1;
      while (K > 1) {
        Plan pk;
        s = make_plan(d, K * B, tl[i].lat[1], tl[i].lat[3], tl[i].lat[5], 1, 1, true, pk);
        if (s) return s;
        if (ws_total(pk) <= kTileBatchWorkspace) break;
        --K;
      }
      for (size_t a = 0; a < grp.size(); a += K)
        batches.emplace_back(grp.begin() + a, grp.begin() + std::min(grp.size(), a + K));
    }
  }
  // storage for every decoded tile (the blend gathers them); workspace for the largest batch first, so
  // the loop below allocates nothing
  size_t total = 0;
  std::vector<size_t> boff(batches.size());
  for (size_t b = 0; b < batches.size(); ++b) {
    boff[b] = total;
    total += align_up(batches[b].size() * tile_bytes(batches[b][0]));
    Plan pb;
    const vae_tile_t& t = tl[batches[b][0]];
    s = make_plan(d, static_cast<int>(batches[b].size()) * B, t.lat[1], t.lat[3], t.lat[5], 1, 1, true, pb);
    if (s) return s;
    s = ensure_ws(d, pb);
    if (s) return s;
  }
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  if (d->tiles_bytes < total) {
    CK(cudaDeviceSynchronize());
    if (d->tiles) cudaFree(d->tiles);
    d->tiles = nullptr;
    d->tiles_bytes = 0;
    CK(cudaMalloc(&d->tiles, total));
    d->tiles_bytes = total;
  }
  char* base = static_cast<char*>(d->tiles);
  std::vector<const void*> ptrs(n);
  const int full[3] = {lat[0], lat[1], lat[2]};
  for (size_t b = 0; b < batches.size(); ++b) {
    const std::vector<int>& bt = batches[b];
    const int K = static_cast<int>(bt.size());
    const vae_tile_t& t = tl[bt[0]];
    Plan p;
    s = make_plan(d, K * B, t.lat[1], t.lat[3], t.lat[5], 1, 1, true, p);
    if (s) return s;
    s = check_gn_range(d, p);
    if (s) return s;
    s = ensure_ws(d, p);
    if (s) return s;
    std::vector<int> boxes(3 * K);
    for (int k = 0; k < K; ++k) {
      boxes[3 * k] = tl[bt[k]].lat[0];
      boxes[3 * k + 1] = tl[bt[k]].lat[2];
      boxes[3 * k + 2] = tl[bt[k]].lat[4];
      ptrs[bt[k]] = base + boff[b] + k * tile_bytes(bt[k]);
    }
    s = run_decode(d, p, static_cast<const float*>(latent), full, boxes.data(), K, base + boff[b], p.lv.back().T, false,
                   strm);
    if (s) return s;
  }
  vae_blend_desc_t bd{};
  bd.B = B; bd.C = c.out_c;
  bd.T = st * (lat[0] - 1) + 1; bd.H = ss * lat[1]; bd.W = ss * lat[2];
  bd.tile_dtype = bd.out_dtype = d->f32 ? VAE_FP32 : VAE_BF16;
  {
    double by = static_cast<double>(B) * c.out_c * bd.T * bd.H * bd.W * ob;
    for (int i = 0; i < n; ++i) by += static_cast<double>(B) * c.out_c * tl[i].pix[1] * tl[i].pix[3] * tl[i].pix[5] * ob;
    Prof pr(d, strm, K_BLEND, 0, by);
    CK(launch_blend(ptrs.data(), tl.data(), n, out, bd, strm));
  }
  return VAE_OK;
}

extern "C" vae_status_t vae_decoder_profile(vae_decoder_t* d, int enable) {
  if (!d) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null decoder");
  d->prof = enable != 0;
  return VAE_OK;
}

extern "C" vae_status_t vae_decoder_profile_read(vae_decoder_t* d, vae_prof_t* out, int* n) {
  if (!d || !out || !n) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null argument");
  CK(cudaDeviceSynchronize());
  vae_prof_t acc[K_COUNT];
  memset(acc, 0, sizeof(acc));
  for (auto& r : d->recs) {
    float ms = 0.f;
    cudaEventElapsedTime(&ms, r.a, r.b);
    vae_prof_t& e = acc[r.kind];
    e.launches += 1;
    e.ms += ms;
    e.flops += r.flops;
    e.bytes += r.bytes;
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  d->recs.clear();
  int k = 0;
  for (int i = 0; i < K_COUNT && k < *n; ++i) {
    if (!acc[i].launches) continue;
    out[k] = acc[i];
    snprintf(out[k].name, sizeof(out[k].name), "%s", kKindNames[i]);
    ++k;
  }
  *n = k;
  return VAE_OK;
}
#undef ERRP

// ================================================================================ encoder
// The encoder runs the decoder's layers read backwards ([DV] encoder commits): the same convs, norms and
// residual blocks (through an embedded decoder core that holds the norm configuration, dtype, error
// record, profiling and allocations), with down-samplers in place of up-samplers.
struct vae_encoder {
  vae_decoder core;
  vae_encoder_config_t ecfg{};
  ConvL conv_in;
  std::vector<std::vector<ResL>> stages;
  std::vector<ConvL> downs;
  std::vector<ResL> mid;
  NormL head_norm;
  ConvL head;
};

namespace {

int count_enc_weights(const vae_encoder_config_t& c) {
  int n = 2;
  for (int i = 0; i < c.n_stages; ++i) {
    n += 8 * c.n_res[i];
    if (i + 1 < c.n_stages) n += 2;
  }
  return n + 8 * c.mid_res + 4;
}

vae_status_t check_enc_config(const vae_encoder_config_t* c) {
  if (!c) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null encoder config");
  const bool rms = c->norm_type == VAE_NORM_CHANNEL_RMS;
  if ((c->norm_type != VAE_NORM_GROUP && !rms) || c->n_stages < 1 || c->n_stages > VAE_MAX_STAGES || c->pix_c <= 0 ||
      c->patch_h < 1 || c->patch_w < 1 || c->latent_c <= 0 || c->mid_res < 0 || (!rms && c->gn_groups <= 0) ||
      (c->dtype != VAE_BF16 && c->dtype != VAE_FP32 && c->dtype != VAE_FP8 && c->dtype != VAE_FP32_TC))
    return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "invalid encoder config");
  for (int i = 0; i < c->n_stages; ++i) {
    const int C = c->stage_c[i];
    if (C <= 0 || c->n_res[i] < 0) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "stage %d channels", i);
    if (rms ? !rms_supported(C)
            : (C % c->gn_groups || C % 8 || C > 6144 || !((C / c->gn_groups) % 8 == 0 || 8 % (C / c->gn_groups) == 0)))
      return set_err(nullptr, VAE_ERR_UNSUPPORTED, 0, 0, "stage %d: %d channels not supported by its norm", i, C);
    if (i + 1 < c->n_stages) {
      const int st = c->down_t[i], sh = c->down_h[i], sw = c->down_w[i];
      if (c->down_kind[i] == VAE_DOWN_FOLD) {
        if (st < 1 || st > 2 || sh < 1 || sw < 1 || c->stage_c[i + 1] % (st * sh * sw))
          return set_err(nullptr, VAE_ERR_UNSUPPORTED, 0, 0, "fold down-sampler %d factors", i);
      } else if (c->down_kind[i] == VAE_DOWN_STRIDE) {
        if (st != 1 || sh != 2 || sw != 2)
          return set_err(nullptr, VAE_ERR_UNSUPPORTED, 0, 0, "the strided down-sampler %d takes factors (1, 2, 2)", i);
      } else {
        return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "down-sampler %d kind", i);
      }
    }
  }
  return VAE_OK;
}

struct EncPlan {
  Plan p;                 // B, patch grid, buffer sizes (no attention); p.lv = one level per stage
  int T0, H0, W0, Cin;    // the patchified pixels (conv_in's input)
};

// Levels: stage i at T_i x H_i x W_i; bands cut on the latent grid, scaled by what stage i still narrows.
vae_status_t make_enc_plan(vae_encoder* e, int B, int T, int H, int W, int nph, int npw, EncPlan& ep) {
  const vae_encoder_config_t& c = e->ecfg;
  vae_decoder* d = &e->core;
  int st_tot = 1, sh_tot = c.patch_h, sw_tot = c.patch_w;
  for (int i = 0; i + 1 < c.n_stages; ++i) {
    st_tot *= c.down_t[i];
    sh_tot *= c.down_h[i];
    sw_tot *= c.down_w[i];
  }
  if (H % sh_tot || W % sw_tot || (T - 1) % st_tot)
    return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0,
                   "video %dx%dx%d: frames - 1 must divide by %d and rows / cols by %d / %d", T, H, W, st_tot, sh_tot,
                   sw_tot);
  const int h_lat = H / sh_tot, w_lat = W / sw_tot;
  Plan& p = ep.p;
  p.B = B; p.nph = nph; p.npw = npw; p.first = true;
  p.Tlat = (T - 1) / st_tot + 1; p.h = h_lat; p.w = w_lat;
  p.lv.clear();
  ep.T0 = T; ep.H0 = H / c.patch_h; ep.W0 = W / c.patch_w;
  ep.Cin = c.pix_c * c.patch_h * c.patch_w;
  int Ti = T, sh = sh_tot / c.patch_h, sw = sw_tot / c.patch_w;
  for (int i = 0; i < c.n_stages; ++i) {
    Level L{};
    L.T = Ti; L.H = h_lat * sh; L.W = w_lat * sw; L.C = c.stage_c[i];
    vae_status_t s = band_edges(h_lat, nph, sh, 1, L.ph, &d->err);
    if (!s) s = band_edges(w_lat, npw, sw, 1, L.pw, &d->err);
    if (s) return s;
    p.lv.push_back(L);
    if (i + 1 < c.n_stages) {
      Ti = (Ti + c.down_t[i] - 1) / c.down_t[i];
      sh /= c.down_h[i];
      sw /= c.down_w[i];
    }
  }
  const int ab = act_bytes(d), rb = res_bytes(d), cb = c1_bytes(d);
  p.x_bytes = p.hin_bytes = p.c1_bytes = p.gn_bytes = 0;
  p.hin_bytes = static_cast<size_t>(B) * (T + 2) * ep.H0 * ep.W0 * e->conv_in.C_in_pad * ab;
  for (int i = 0; i < c.n_stages; ++i) {
    const Level& L = p.lv[i];
    const size_t px = static_cast<size_t>(B) * L.H * L.W;
    p.x_bytes = std::max(p.x_bytes, px * L.T * L.C * rb);
    p.hin_bytes = std::max(p.hin_bytes, px * (L.T + 2) * L.C * ab);
    p.c1_bytes = std::max(p.c1_bytes, px * L.T * L.C * cb);
    const int groups = c.norm_type == VAE_NORM_GROUP ? c.gn_groups : 0;
    p.gn_bytes = std::max(p.gn_bytes, gn_workspace_bytes(nph, npw, B, L.T, groups, L.C));
    if (i + 1 < c.n_stages) {
      const Level& N = p.lv[i + 1];
      if (c.down_kind[i] == VAE_DOWN_FOLD)  // the down conv's unfolded output
        p.c1_bytes = std::max(p.c1_bytes, px * L.T * e->downs[i].C_out * rb);
      else                                  // the (1,2,2)-folded input of the strided conv
        p.hin_bytes = std::max(p.hin_bytes, static_cast<size_t>(B) * (N.T + 2) * N.H * N.W * 4 * L.C * ab);
    }
    if (c.norm_type == VAE_NORM_GROUP &&
        static_cast<double>(L.C / c.gn_groups) * L.H * L.W >= 8388608.0)
      return set_err(&d->err, VAE_ERR_UNSUPPORTED, 0, 0, "stage %d: group exceeds the exact-sum range", i);
  }
  p.lat_bytes = 0;
  p.split_bytes = d->f32 ? p.hin_bytes : 0;  // every conv input lives in hin
  p.attn_tok = p.attn_tokp = 0;
  p.q_bytes = p.vt_bytes = p.s_bytes = p.p_bytes = 0;
  return VAE_OK;
}

#define ERRP (&d->err)
// Encode the pixel box rows [h0, h0 + H), cols [w0, w0 + W) (pixel units) of video [B, pix_c, T, Hf, Wf]
// into moments NCTHW fp32 [B, 2*latent_c, T', h, w].
// Encode ep.p.B = n_boxes x B_v items: the pixel boxes (h0, w0) = boxes[2 i], boxes[2 i + 1] of the B_v videos
// (full frames Hf x Wf), box after box along the batch.
vae_status_t run_encode(vae_encoder* e, const EncPlan& ep, const float* video, int Hf, int Wf, const int* boxes,
                        int n_boxes, float* out, cudaStream_t s) {
  vae_decoder* d = &e->core;
  const vae_encoder_config_t& c = e->ecfg;
  const Plan& p = ep.p;
  Ctx x{d, &p, carve(d->ws, p), s, false};
  const int rf = res_bytes(d) == 4;
  auto kind_of = [&](const ConvL& cv) { return cv.fp8 ? 2 : (d->f32 ? 1 : 0); };
  {
    const Level& L0 = p.lv[0];
    const int ob = op_bytes(d, e->conv_in);
    const int64_t fb = static_cast<int64_t>(ep.H0) * ep.W0 * e->conv_in.C_in_pad * ob;
    if (n_boxes < 1 || p.B % n_boxes) return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "bad pixel box batch");
    const int Bv = p.B / n_boxes;
    for (int i = 0; i < n_boxes; ++i) {
      const int h0 = boxes[2 * i], w0 = boxes[2 * i + 1];
      Prof pr(d, s, K_LATENT, 0, static_cast<double>(Bv) * ep.T0 * ep.H0 * ep.W0 * (ep.Cin * 4.0 + e->conv_in.C_in_pad * ob));
      CK(launch_pixels_to_cl(video, Bv, c.pix_c, ep.T0, Hf, Wf, c.patch_h, c.patch_w, h0 / c.patch_h, ep.H0,
                             w0 / c.patch_w, ep.W0, e->conv_in.C_in_pad,
                             x.b.hin + 2 * fb + static_cast<int64_t>(i) * Bv * (ep.T0 + 2) * fb, kind_of(e->conv_in),
                             ep.T0 + 2, s));
    }
    ConvOut o;
    o.y = x.b.x; o.y_f32 = rf; o.y_T_alloc = L0.T; o.stats_level = &L0;
    vae_status_t st = run_conv(x, e->conv_in, L0, x.b.hin, o);
    if (st) return st;
  }
  for (int i = 0; i < c.n_stages; ++i) {
    const Level& L = p.lv[i];
    for (auto& r : e->stages[i]) {
      vae_status_t st = run_resblock(x, r, L);
      if (st) return st;
    }
    if (i + 1 == c.n_stages) break;
    const Level& N = p.lv[i + 1];
    ConvL& dc = e->downs[i];
    const int ob = op_bytes(d, dc);
    if (c.down_kind[i] == VAE_DOWN_FOLD) {
      // stride-1 conv of the residual stream (cast to the conv's operand type), then the fold
      const int64_t fe = static_cast<int64_t>(L.H) * L.W * L.C;
      {
        Prof pr(d, s, K_CAST, 0, static_cast<double>(p.B) * L.T * fe * (res_bytes(d) + ob));
        CK(launch_cast_frames(x.b.x, rf, L.T, x.b.hin + 2 * fe * ob, kind_of(dc), L.T + 2, p.B, L.T, fe, s));
      }
      ConvOut od;
      od.y = x.b.c1; od.y_f32 = rf; od.y_T_alloc = L.T;
      vae_status_t st = run_conv(x, dc, L, x.b.hin, od);
      if (st) return st;
      Prof pr(d, s, K_COPY, 0, 2.0 * p.B * L.T * L.H * L.W * dc.C_out * res_bytes(d));
      CK(launch_fold_frames(x.b.c1, rf, L.T, p.B, L.T, L.H, L.W, dc.C_out, c.down_t[i], c.down_h[i], c.down_w[i], x.b.x,
                            rf ? 1 : 0, N.T, s));
      x.stats_src = nullptr;
    } else {
      // fold (1, 2, 2) into the conv's operand type, then the stride-1 conv with rearranged weights
      const int64_t fe2 = static_cast<int64_t>(N.H) * N.W * 4 * L.C;
      {
        Prof pr(d, s, K_COPY, 0, static_cast<double>(p.B) * N.T * fe2 * (res_bytes(d) + ob));
        CK(launch_fold_frames(x.b.x, rf, L.T, p.B, L.T, L.H, L.W, L.C, 1, 2, 2, x.b.hin + 2 * fe2 * ob, kind_of(dc),
                              N.T + 2, s));
      }
      ConvOut od;
      od.y = x.b.x; od.y_f32 = rf; od.y_T_alloc = N.T; od.stats_level = &N;
      vae_status_t st = run_conv(x, dc, N, x.b.hin, od);
      if (st) return st;
    }
  }
  const Level& LL = p.lv[c.n_stages - 1];
  for (auto& r : e->mid) {
    vae_status_t st = run_resblock(x, r, LL);
    if (st) return st;
  }
  vae_status_t st = run_gn(x, e->head_norm, LL, x.b.x, rf, 1, e->head.fp8);
  if (st) return st;
  ConvOut o;
  o.y = out; o.y_f32 = 1; o.y_T_alloc = LL.T; o.out_ncthw = 1;
  return run_conv(x, e->head, LL, x.b.hin, o);
}
#undef ERRP

vae_status_t check_video(vae_encoder* e, const int64_t* shp, int nph, int npw) {
  vae_decoder* d = &e->core;
  if (!shp) return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "null shape");
  if (shp[0] <= 0 || shp[1] != e->ecfg.pix_c || shp[2] <= 0 || shp[3] <= 0 || shp[4] <= 0)
    return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "video shape mismatch");
  if (shp[0] > 64 || shp[2] > 4096 || shp[3] > 16384 || shp[4] > 16384)
    return set_err(&d->err, VAE_ERR_UNSUPPORTED, 0, 0, "video too large");
  if (nph < 1 || npw < 1 || nph > VAE_MAX_PATCHES || npw > VAE_MAX_PATCHES)
    return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "patch counts %d x %d", nph, npw);
  return VAE_OK;
}

}  // namespace

extern "C" vae_status_t vae_encoder_n_weights(const vae_encoder_config_t* cfg, int* n_weights) {
  vae_status_t s = check_enc_config(cfg);
  if (s) return s;
  if (!n_weights) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null n_weights");
  *n_weights = count_enc_weights(*cfg);
  return VAE_OK;
}

extern "C" void vae_encoder_destroy(vae_encoder_t* e) {
  if (!e) return;
  release_memory(&e->core);
  delete e;
}

extern "C" vae_status_t vae_encoder_create(const vae_encoder_config_t* cfg, const void* const* weights, int n_weights,
                                           vae_encoder_t** out) {
  if (!out) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null out");
  *out = nullptr;
  vae_status_t s = check_enc_config(cfg);
  if (s) return s;
  if (!weights || n_weights != count_enc_weights(*cfg))
    return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "expected %d weight tensors, got %d", count_enc_weights(*cfg),
                   n_weights);
  for (int i = 0; i < n_weights; ++i)
    if (!weights[i] || !aligned16(weights[i]))
      return set_err(nullptr, weights[i] ? VAE_ERR_ALIGNMENT : VAE_ERR_INVALID_ARG, 0, 0, "weight %d pointer", i);
  vae_encoder* e = new vae_encoder();
  e->ecfg = *cfg;
  vae_decoder* d = &e->core;
  d->cfg.gn_groups = cfg->gn_groups;
  d->cfg.gn_eps = cfg->gn_eps;
  d->cfg.norm_type = cfg->norm_type;
  d->cfg.dtype = cfg->dtype;
  d->f32 = cfg->dtype == VAE_FP32 || cfg->dtype == VAE_FP32_TC;
  d->f32tc = cfg->dtype == VAE_FP32_TC;
  d->f8 = cfg->dtype == VAE_FP8;
  int k = 0;
  auto W = [&](void) { return static_cast<const float*>(weights[k++]); };
  auto res_block = [&](ResL& r, int C) -> vae_status_t {
    const float *g1 = W(), *b1 = W(), *w1 = W(), *bb1 = W(), *g2 = W(), *b2 = W(), *w2 = W(), *bb2 = W();
    vae_status_t st = make_norm(d, r.n1, g1, b1, C);
    if (!st) st = make_conv(d, r.c1, w1, bb1, C, C, 1, 1, 1, false, true);
    if (!st) st = make_norm(d, r.n2, g2, b2, C);
    if (!st) st = make_conv(d, r.c2, w2, bb2, C, C, 1, 1, 1, false, true);
    return st;
  };
  {
    const float* w = W();
    const float* b = W();
    s = make_conv(d, e->conv_in, w, b, cfg->pix_c * cfg->patch_h * cfg->patch_w, cfg->stage_c[0], 1, 1, 1, true);
  }
  e->stages.resize(cfg->n_stages);
  e->downs.resize(std::max(0, cfg->n_stages - 1));
  float* tmp = nullptr;  // rearranged stride-2 weights
  for (int i = 0; i < cfg->n_stages && !s; ++i) {
    const int C = cfg->stage_c[i];
    e->stages[i].resize(cfg->n_res[i]);
    for (int r = 0; r < cfg->n_res[i] && !s; ++r) s = res_block(e->stages[i][r], C);
    if (i + 1 < cfg->n_stages && !s) {
      const float* w = W();
      const float* b = W();
      const int Cn = cfg->stage_c[i + 1];
      if (cfg->down_kind[i] == VAE_DOWN_FOLD) {
        const int S = cfg->down_t[i] * cfg->down_h[i] * cfg->down_w[i];
        s = make_conv(d, e->downs[i], w, b, C, Cn / S, 1, 1, 1, false, true);
      } else {
        if (!tmp) s = dalloc(d, &tmp, static_cast<size_t>(Cn) * 4 * C * 27 * 4);  // freed with the handle
        cudaError_t ce = s ? cudaSuccess : launch_stride2_weights(w, Cn, C, tmp, nullptr);
        if (ce != cudaSuccess) s = set_err(&d->err, VAE_ERR_CUDA, 0, 0, "stride-2 weights: %s", cudaGetErrorString(ce));
        if (!s) s = make_conv(d, e->downs[i], tmp, b, 4 * C, Cn, 1, 1, 1, false, true);
        if (!s && cudaDeviceSynchronize() != cudaSuccess) s = set_err(&d->err, VAE_ERR_CUDA, 0, 0, "weight packing");
        tmp = nullptr;  // the next strided down-sampler (if any) gets its own scratch
      }
    }
  }
  const int CL = cfg->stage_c[cfg->n_stages - 1];
  e->mid.resize(cfg->mid_res);
  for (int r = 0; r < cfg->mid_res && !s; ++r) s = res_block(e->mid[r], CL);
  if (!s) {
    const float* g = W();
    const float* b = W();
    s = make_norm(d, e->head_norm, g, b, CL);
    const float* w = W();
    const float* bb = W();
    if (!s) s = make_conv(d, e->head, w, bb, CL, 2 * cfg->latent_c, 1, 1, 1, false, false, true);
  }
  if (!s) {
    cudaError_t ce = cudaDeviceSynchronize();
    if (ce != cudaSuccess) s = set_err(&d->err, VAE_ERR_CUDA, 0, 0, "weight packing: %s", cudaGetErrorString(ce));
  }
  if (s) {
    {
      std::lock_guard<std::mutex> lk(g_last_mu);
      g_last = d->err;
    }
    vae_encoder_destroy(e);
    return s;
  }
  *out = e;
  return VAE_OK;
}

#define ERRP (&e->core.err)
extern "C" vae_status_t vae_encode(vae_encoder_t* e, const void* video, const int64_t shp[5], void* moments, int nph,
                                   int npw, void* stream) {
  if (!e) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null encoder");
  if (!video || !moments) return set_err(&e->core.err, VAE_ERR_INVALID_ARG, 0, 0, "null video or moments");
  if (!aligned16(video) || !aligned16(moments))
    return set_err(&e->core.err, VAE_ERR_ALIGNMENT, 0, 0, "video/moments not 16-byte aligned");
  vae_status_t s = check_video(e, shp, nph, npw);
  if (s) return s;
  EncPlan ep;
  s = make_enc_plan(e, static_cast<int>(shp[0]), static_cast<int>(shp[2]), static_cast<int>(shp[3]),
                    static_cast<int>(shp[4]), nph, npw, ep);
  if (s) return s;
  s = ensure_ws(&e->core, ep.p);
  if (s) return s;
  const int box0[2] = {0, 0};
  return run_encode(e, ep, static_cast<const float*>(video), static_cast<int>(shp[3]), static_cast<int>(shp[4]), box0, 1,
                    static_cast<float*>(moments), static_cast<cudaStream_t>(stream));
}

extern "C" vae_status_t vae_encode_tiled(vae_encoder_t* e, const void* video, const int64_t shp[5], void* moments,
                                         const int tile_hw[2], const int ovl_hw[2], void* stream) {
  if (!e) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null encoder");
  vae_decoder* d = &e->core;
  if (!video || !moments || !tile_hw || !ovl_hw) return set_err(&d->err, VAE_ERR_INVALID_ARG, 0, 0, "null argument");
  if (!aligned16(video) || !aligned16(moments))
    return set_err(&d->err, VAE_ERR_ALIGNMENT, 0, 0, "video/moments not 16-byte aligned");
  vae_status_t s = check_video(e, shp, 1, 1);
  if (s) return s;
  EncPlan whole;
  s = make_enc_plan(e, static_cast<int>(shp[0]), static_cast<int>(shp[2]), static_cast<int>(shp[3]),
                    static_cast<int>(shp[4]), 1, 1, whole);
  if (s) return s;
  const int B = static_cast<int>(shp[0]);
  const int sh_tot = static_cast<int>(shp[3]) / whole.p.h, sw_tot = static_cast<int>(shp[4]) / whole.p.w;
  const int lat[3] = {whole.p.Tlat, whole.p.h, whole.p.w};
  const int tile[3] = {whole.p.Tlat, tile_hw[0], tile_hw[1]};
  const int ovl[3] = {0, ovl_hw[0], ovl_hw[1]};
  std::vector<vae_tile_t> tl(VAE_MAX_TILES);
  int n = VAE_MAX_TILES;
  constexpr size_t kTileBatchWorkspace = 16ull << 30;  // workspace budget of one batch of equal-shape tiles
  s = vae_tile_plan(lat, tile, ovl, 1, 1, 0, tl.data(), &n);
  if (s) return set_err(&d->err, s, 0, 0, "tile plan failed (%d tiles max)", VAE_MAX_TILES);
  const int M = 2 * e->ecfg.latent_c;
  auto tile_bytes = [&](int i) { return static_cast<size_t>(B) * M * tl[i].pix[1] * tl[i].pix[3] * tl[i].pix[5] * 4; };
  // tiles of one shape encode together as one batch (within the workspace budget), outputs contiguous
  std::vector<std::vector<int>> batches;
  {
    std::vector<char> taken(n, 0);
    for (int i = 0; i < n; ++i) {
      if (taken[i]) continue;
      std::vector<int> grp;
      for (int j = i; j < n; ++j)
        if (!taken[j] && tl[j].lat[3] == tl[i].lat[3] && tl[j].lat[5] == tl[i].lat[5]) {
          grp.push_back(j);
          taken[j] = 1;
        }
      int K = tile_bytes(i) % 256 == 0 ? static_cast<int>(grp.size()) : 1;
      while (K > 1) {
        EncPlan pk;
        s = make_enc_plan(e, K * B, static_cast<int>(shp[2]), tl[i].lat[3] * sh_tot, tl[i].lat[5] * sw_tot, 1, 1, pk);
        if (s) return s;
        if (ws_total(pk.p) <= kTileBatchWorkspace) break;
        --K;
      }
      for (size_t a = 0; a < grp.size(); a += K)
        batches.emplace_back(grp.begin() + a, grp.begin() + std::min(grp.size(), a + K));
    }
  }
  size_t total = 0;
  std::vector<size_t> boff(batches.size());
  for (size_t b = 0; b < batches.size(); ++b) {  // workspace before anything is enqueued
    boff[b] = total;
    total += align_up(batches[b].size() * tile_bytes(batches[b][0]));
    const vae_tile_t& t = tl[batches[b][0]];
    EncPlan pb;
    s = make_enc_plan(e, static_cast<int>(batches[b].size()) * B, static_cast<int>(shp[2]), t.lat[3] * sh_tot,
                      t.lat[5] * sw_tot, 1, 1, pb);
    if (!s) s = ensure_ws(d, pb.p);
    if (s) return s;
  }
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  if (d->tiles_bytes < total) {
    CK(cudaDeviceSynchronize());
    if (d->tiles) cudaFree(d->tiles);
    d->tiles = nullptr;
    d->tiles_bytes = 0;
    CK(cudaMalloc(&d->tiles, total));
    d->tiles_bytes = total;
  }
  char* base = static_cast<char*>(d->tiles);
  std::vector<const void*> ptrs(n);
  for (size_t b = 0; b < batches.size(); ++b) {
    const std::vector<int>& bt = batches[b];
    const int K = static_cast<int>(bt.size());
    const vae_tile_t& t = tl[bt[0]];
    EncPlan ep;
    s = make_enc_plan(e, K * B, static_cast<int>(shp[2]), t.lat[3] * sh_tot, t.lat[5] * sw_tot, 1, 1, ep);
    if (!s) s = ensure_ws(d, ep.p);
    if (s) return s;
    std::vector<int> boxes(2 * K);
    for (int k = 0; k < K; ++k) {
      boxes[2 * k] = tl[bt[k]].lat[2] * sh_tot;
      boxes[2 * k + 1] = tl[bt[k]].lat[4] * sw_tot;
      ptrs[bt[k]] = base + boff[b] + k * tile_bytes(bt[k]);
    }
    s = run_encode(e, ep, static_cast<const float*>(video), static_cast<int>(shp[3]), static_cast<int>(shp[4]),
                   boxes.data(), K, reinterpret_cast<float*>(base + boff[b]), strm);
    if (s) return s;
  }
  vae_blend_desc_t bd{};
  bd.B = B; bd.C = M; bd.T = lat[0]; bd.H = lat[1]; bd.W = lat[2];
  bd.tile_dtype = bd.out_dtype = VAE_FP32;
  Prof pr(d, strm, K_BLEND, 0, 8.0 * B * M * lat[0] * lat[1] * lat[2]);
  CK(launch_blend(ptrs.data(), tl.data(), n, moments, bd, strm));
  return VAE_OK;
}
#undef ERRP

extern "C" vae_status_t vae_encoder_profile(vae_encoder_t* e, int enable) {
  if (!e) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null encoder");
  return vae_decoder_profile(&e->core, enable);
}

extern "C" vae_status_t vae_encoder_profile_read(vae_encoder_t* e, vae_prof_t* out, int* n) {
  if (!e) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null encoder");
  return vae_decoder_profile_read(&e->core, out, n);
}

extern "C" vae_status_t vae_encoder_last_error(vae_encoder_t* e, vae_error_info_t* info) {
  if (!e) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null encoder");
  return vae_last_error(&e->core, info);
}

// ================================================================================ op level
#define ERRP nullptr
namespace {
vae_status_t check_edges(int n, const int* e, int extent, const char* what) {
  if (n < 1 || n > VAE_MAX_PATCHES) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "%s: %d patches", what, n);
  if (e[0] != 0 || e[n] != extent) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "%s edges must span 0..%d", what, extent);
  for (int i = 0; i < n; ++i)
    if (e[i + 1] - e[i] < 1)
      return set_err(nullptr, VAE_ERR_PATCH_TOO_NARROW, e[i + 1] - e[i], 1, "%s patch %d has %d rows", what, i, e[i + 1] - e[i]);
  return VAE_OK;
}
bool conv_tc_ok(const vae_conv_desc_t* d) { return d->in_dtype == VAE_BF16 && d->C_in % 64 == 0; }
bool conv_fp8(const vae_conv_desc_t* d) { return d->in_dtype == VAE_FP8; }
int conv_npad(const vae_conv_desc_t* d) { return (d->C_out + 15) / 16 * 16; }
}  // namespace

extern "C" size_t vae_conv3d_packed_bytes(const vae_conv_desc_t* d) {
  if (!d || d->C_in <= 0 || d->C_out <= 0) return 0;
  if (conv_fp8(d)) return fp8_scale_offset(conv_npad(d), d->C_in) + static_cast<size_t>(conv_npad(d)) * 4;
  if (conv_tc_ok(d) && conv_tap_stacked(d->C_out, 0)) return 3ull * kTapRows * d->C_in * 2;
  if (conv_tc_ok(d)) return static_cast<size_t>(conv_npad(d)) * 27 * d->C_in * 2;
  return 27ull * d->C_in * d->C_out * 4;
}

extern "C" vae_status_t vae_conv3d_pack_weights(const float* w, const vae_conv_desc_t* d, void* w_packed, void* stream) {
  if (!w || !d || !w_packed) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null argument");
  const int S = d->d2s_t * d->d2s_h * d->d2s_w;
  if (S < 1 || d->C_out % S) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "C_out %% depth-to-space");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (conv_fp8(d) && d->C_in % 128)
    return set_err(nullptr, VAE_ERR_UNSUPPORTED, 0, 0, "fp8 convs need C_in %% 128 == 0 (got %d)", d->C_in);
  if (conv_fp8(d))
    CK(launch_pack_weights_fp8(w, d->C_out, d->C_in, d->C_in, conv_npad(d), S, w_packed, s, d->out_ncthw));
  else if (conv_tc_ok(d))
    CK(launch_pack_weights_bf16(w, d->C_out, d->C_in, d->C_in, conv_npad(d), S, w_packed, s, d->out_ncthw,
                                conv_tap_stacked(d->C_out, 0)));
  else CK(launch_pack_weights_f32(w, d->C_out, d->C_in, w_packed, s));
  return VAE_OK;
}

extern "C" vae_status_t vae_conv3d_causal(const void* x, const void* w_packed, const float* bias, const void* residual,
                                          void* y, const vae_conv_desc_t* d, void* stream) {
  if (!x || !w_packed || !y || !d) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null argument");
  if (!aligned16(x) || !aligned16(y) || !aligned16(w_packed) || (residual && !aligned16(residual)))
    return set_err(nullptr, VAE_ERR_ALIGNMENT, 0, 0, "pointers must be 16-byte aligned");
  if (d->B <= 0 || d->T <= 0 || d->H <= 0 || d->W <= 0 || d->C_in <= 0 || d->C_out <= 0 ||
      (d->cache_frames != 0 && d->cache_frames != 2) || d->d2s_t < 1 || d->d2s_h < 1 || d->d2s_w < 1)
    return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "bad conv descriptor");
  const int S = d->d2s_t * d->d2s_h * d->d2s_w;
  if (d->C_out % S) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "C_out not divisible by the depth-to-space factor");
  if (residual && S != 1) return set_err(nullptr, VAE_ERR_UNSUPPORTED, 0, 0, "residual with depth-to-space");
  if (d->in_dtype != VAE_BF16 && d->in_dtype != VAE_FP32 && d->in_dtype != VAE_FP8)
    return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "bad input dtype");
  if (d->out_dtype == VAE_FP8 || d->res_dtype == VAE_FP8)
    return set_err(nullptr, VAE_ERR_UNSUPPORTED, 0, 0, "conv outputs and residuals are bf16 or fp32");
  if (conv_fp8(d) && d->C_in % 128)
    return set_err(nullptr, VAE_ERR_UNSUPPORTED, 0, 0, "fp8 convs need C_in %% 128 == 0 (got %d)", d->C_in);
  vae_status_t st = check_edges(d->n_patch_h, d->patch_h_edges, d->H, "height");
  if (!st) st = check_edges(d->n_patch_w, d->patch_w_edges, d->W, "width");
  if (st) return st;
  if ((x == y) || (residual && residual == y && S != 1)) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "y aliases x");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (conv_tc_ok(d) || conv_fp8(d)) {
    ConvTcArgs a{};
    if (conv_fp8(d)) {
      a.fp8 = 1;
      a.wscale = reinterpret_cast<const float*>(static_cast<const char*>(w_packed) + fp8_scale_offset(conv_npad(d), d->C_in));
    }
    a.mode = 0;
    a.B = d->B; a.T = d->T; a.H = d->H; a.W = d->W; a.C_in_pad = d->C_in;
    a.T_in = d->T + d->cache_frames; a.x_T_alloc = a.T_in; a.cache_frames = d->cache_frames;
    a.nph = d->n_patch_h; a.npw = d->n_patch_w; a.ph_edges = d->patch_h_edges; a.pw_edges = d->patch_w_edges;
    a.x = x; a.w = w_packed; a.N_real = d->C_out; a.N_pad = conv_npad(d); a.bias = bias;
    a.residual = residual; a.res_f32 = d->res_dtype == VAE_FP32;
    a.y = y; a.out_f32 = d->out_dtype == VAE_FP32; a.out_ncthw = d->out_ncthw;
    a.d2s_t = d->d2s_t; a.d2s_h = d->d2s_h; a.d2s_w = d->d2s_w; a.drop_first = d->drop_first;
    a.natural = d->out_ncthw;
    a.tap_stacked = !a.fp8 && conv_tap_stacked(d->C_out, 0);
    CK(launch_conv_tc(a, s));
  } else {
    ConvSimtArgs a{};
    a.B = d->B; a.T = d->T; a.H = d->H; a.W = d->W; a.C_in = d->C_in; a.C_out = d->C_out;
    a.T_in = d->T + d->cache_frames; a.x_T_alloc = a.T_in; a.cache_frames = d->cache_frames;
    a.x = x; a.x_f32 = d->in_dtype == VAE_FP32; a.w = static_cast<const float*>(w_packed); a.bias = bias;
    a.residual = residual; a.res_f32 = d->res_dtype == VAE_FP32;
    a.y = y; a.out_f32 = d->out_dtype == VAE_FP32; a.out_ncthw = d->out_ncthw;
    a.d2s_t = d->d2s_t; a.d2s_h = d->d2s_h; a.d2s_w = d->d2s_w; a.drop_first = d->drop_first;
    a.nph = d->n_patch_h; a.npw = d->n_patch_w; a.ph_edges = d->patch_h_edges; a.pw_edges = d->patch_w_edges;
    CK(launch_conv_simt(a, s));
  }
  return VAE_OK;
}

extern "C" size_t vae_patch_groupnorm_workspace_bytes(const vae_gn_desc_t* d) {
  if (!d || d->B <= 0 || d->T <= 0 || d->groups <= 0 || d->n_patch_h <= 0 || d->n_patch_w <= 0) return 0;
  return gn_workspace_bytes(d->n_patch_h, d->n_patch_w, d->B, d->T, d->groups, d->C);
}

namespace {
vae_status_t check_gn_desc(const vae_gn_desc_t* d) {
  if (d->B <= 0 || d->T <= 0 || d->H <= 0 || d->W <= 0 || d->C <= 0 || d->groups <= 0 || d->C % d->groups)
    return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "bad group-norm descriptor");
  if ((d->in_dtype != VAE_BF16 && d->in_dtype != VAE_FP32) ||
      (d->out_dtype != VAE_BF16 && d->out_dtype != VAE_FP32 && d->out_dtype != VAE_FP8))
    return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "bad group-norm dtypes");
  const int cpg = d->C / d->groups;
  if (d->C % 8 || d->C > 6144 || d->groups > 1024 || !(cpg % 8 == 0 || 8 % cpg == 0))
    return set_err(nullptr, VAE_ERR_UNSUPPORTED, 0, 0, "%d channels in %d groups not supported", d->C, d->groups);
  if (static_cast<double>(cpg) * d->H * d->W >= 8388608.0)
    return set_err(nullptr, VAE_ERR_UNSUPPORTED, 0, 0, "group larger than the exact-sum range (2^23 elements)");
  vae_status_t st = check_edges(d->n_patch_h, d->patch_h_edges, d->H, "height");
  if (!st) st = check_edges(d->n_patch_w, d->patch_w_edges, d->W, "width");
  return st;
}
}  // namespace

namespace vae {
vae_status_t op_error(vae_status_t code, const char* msg) { return set_err(nullptr, code, 0, 0, "%s", msg); }
vae_status_t validate_gn_desc(const void* x, const void* y, const vae_gn_desc_t* d) {
  if (!aligned16(x) || !aligned16(y)) return set_err(nullptr, VAE_ERR_ALIGNMENT, 0, 0, "pointers must be 16-byte aligned");
  return check_gn_desc(d);
}
}  // namespace vae

extern "C" vae_status_t vae_patch_groupnorm_silu(const void* x, const float* gamma, const float* beta, void* y,
                                                 void* workspace, const vae_gn_desc_t* d, void* stream) {
  if (!x || !gamma || !beta || !y || !workspace || !d) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null argument");
  if (!aligned16(x) || !aligned16(y) || !aligned16(workspace))
    return set_err(nullptr, VAE_ERR_ALIGNMENT, 0, 0, "pointers must be 16-byte aligned");
  vae_status_t st = check_gn_desc(d);
  if (st) return st;
  GnArgs g{};
  g.B = d->B; g.T = d->T; g.H = d->H; g.W = d->W; g.C = d->C; g.groups = d->groups; g.eps = d->eps; g.silu = d->silu;
  g.nph = d->n_patch_h; g.npw = d->n_patch_w; g.ph_edges = d->patch_h_edges; g.pw_edges = d->patch_w_edges;
  g.x = x; g.x_f32 = d->in_dtype == VAE_FP32; g.y = y; g.y_f32 = d->out_dtype == VAE_FP32;
  g.y_fp8 = d->out_dtype == VAE_FP8;
  g.gamma = gamma; g.beta = beta; g.partials = workspace;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CK(launch_gn_stats(g, s));
  CK(launch_gn_apply(g, s));
  return VAE_OK;
}

extern "C" vae_status_t vae_channel_rmsnorm_silu(const void* x, const float* gamma, const float* beta, void* y,
                                                 const vae_rms_desc_t* d, void* stream) {
  if (!x || !gamma || !beta || !y || !d) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null argument");
  if (!aligned16(x) || !aligned16(y) || (reinterpret_cast<uintptr_t>(gamma) & 31) ||
      (reinterpret_cast<uintptr_t>(beta) & 31))
    return set_err(nullptr, VAE_ERR_ALIGNMENT, 0, 0, "x, y must be 16-byte and gamma, beta 32-byte aligned");
  if (d->B <= 0 || d->T <= 0 || d->H <= 0 || d->W <= 0 || d->C <= 0 || !(d->eps >= 0.f))
    return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "bad RMS-norm descriptor");
  if ((d->in_dtype != VAE_BF16 && d->in_dtype != VAE_FP32) ||
      (d->out_dtype != VAE_BF16 && d->out_dtype != VAE_FP32 && d->out_dtype != VAE_FP8))
    return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "bad dtype");
  if (!rms_supported(d->C)) return set_err(nullptr, VAE_ERR_UNSUPPORTED, 0, 0, "RMS norm over %d channels not supported", d->C);
  GnArgs g{};
  g.B = d->B; g.T = d->T; g.H = d->H; g.W = d->W; g.C = d->C; g.eps = d->eps; g.silu = d->silu;
  g.x = x; g.x_f32 = d->in_dtype == VAE_FP32; g.y = y; g.y_f32 = d->out_dtype == VAE_FP32;
  g.y_fp8 = d->out_dtype == VAE_FP8;
  g.gamma = gamma; g.beta = beta;
  CK(launch_rms(g, static_cast<cudaStream_t>(stream)));
  return VAE_OK;
}

extern "C" vae_status_t vae_upsample_d2s(const void* x, void* y, const vae_d2s_desc_t* d, void* stream) {
  if (!x || !y || !d) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null argument");
  if (d->B <= 0 || d->T <= 0 || d->H <= 0 || d->W <= 0 || d->C <= 0 || d->s_t < 1 || d->s_h < 1 || d->s_w < 1)
    return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "bad depth-to-space descriptor");
  if (x == y) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "y aliases x");
  CK(launch_d2s(x, y, d->B, d->T, d->H, d->W, d->C, d->s_t, d->s_h, d->s_w, d->drop_first, d->dtype == VAE_FP32,
                static_cast<cudaStream_t>(stream)));
  return VAE_OK;
}

extern "C" vae_status_t vae_tile_blend(const void* const* tiles, const vae_tile_t* meta, int n_tiles, void* out,
                                       const vae_blend_desc_t* d, void* stream) {
  if (!tiles || !meta || !out || !d || n_tiles <= 0) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null argument");
  if (n_tiles > VAE_MAX_TILES) return set_err(nullptr, VAE_ERR_UNSUPPORTED, 0, 0, "more than %d tiles", VAE_MAX_TILES);
  if (d->B <= 0 || d->C <= 0 || d->T <= 0 || d->H <= 0 || d->W <= 0)
    return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "bad blend descriptor");
  for (int i = 0; i < n_tiles; ++i) {
    const int* p = meta[i].pix;
    if (!tiles[i] || p[1] <= 0 || p[3] <= 0 || p[5] <= 0 || p[0] < 0 || p[2] < 0 || p[4] < 0 || p[0] + p[1] > d->T ||
        p[2] + p[3] > d->H || p[4] + p[5] > d->W)
      return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "tile %d box outside the output", i);
    for (int k = 0; k < 6; ++k)
      if (meta[i].ovl[k] < 0 || meta[i].ovl[k] > 65535) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "tile %d overlap", i);
  }
  CK(launch_blend(tiles, meta, n_tiles, out, *d, static_cast<cudaStream_t>(stream)));
  return VAE_OK;
}

extern "C" vae_status_t vae_gemm_bf16(const void* A, const void* Bm, void* D, const float* bias, int M, int N, int K,
                                      int batch, int64_t sa, int64_t sb, int64_t sd, float alpha, vae_dtype_t out_dtype,
                                      void* stream) {
  if (!A || !Bm || !D) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "null argument");
  if (M <= 0 || N <= 0 || K <= 0 || batch <= 0 || K % 64 || N % 16 || (batch > 1 && (sa % 8 || sb % 8)))
    return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "gemm sizes (K %% 64, N %% 16)");
  if (!aligned16(A) || !aligned16(Bm) || !aligned16(D)) return set_err(nullptr, VAE_ERR_ALIGNMENT, 0, 0, "alignment");
  ConvTcArgs a{};
  a.mode = 1;
  a.M = M; a.K = K; a.batch = batch; a.stride_a = batch > 1 ? sa : static_cast<int64_t>(M) * K;
  a.stride_b = batch > 1 ? sb : static_cast<int64_t>(N) * K; a.stride_d = sd; a.alpha = alpha;
  a.x = A; a.w = Bm; a.N_real = N; a.N_pad = N; a.bias = bias;
  a.y = D; a.out_f32 = out_dtype == VAE_FP32;
  a.d2s_t = a.d2s_h = a.d2s_w = 1;
  CK(launch_conv_tc(a, static_cast<cudaStream_t>(stream)));
  return VAE_OK;
}

extern "C" vae_status_t vae_watchdog_selftest(int timeout_us, void* stream) {
  if (timeout_us <= 0 || timeout_us > 10000000) return set_err(nullptr, VAE_ERR_INVALID_ARG, 0, 0, "timeout_us");
  CK(launch_watchdog_test(static_cast<uint64_t>(timeout_us) * 1000ull, static_cast<cudaStream_t>(stream)));
  CK(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  vae_error_info_t info{};
  return vae_last_error(nullptr, &info);
}
#undef ERRP

extern "C" vae_status_t vae_last_error(vae_decoder_t* d, vae_error_info_t* info) {
  vae_error_info_t out{};
  if (d) out = d->err;
  else {
    std::lock_guard<std::mutex> lk(g_last_mu);
    out = g_last;
  }
  int dev_count = 0;
  if (cudaGetDeviceCount(&dev_count) == cudaSuccess && dev_count > 0) {
    cudaError_t e = cudaDeviceSynchronize();
    uint32_t* fw = fault_word();
    uint32_t host[4] = {0, 0, 0, 0};
    if (e == cudaSuccess && fw) e = cudaMemcpy(host, fw, sizeof(host), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
      out.code = VAE_ERR_CUDA;
      snprintf(out.message, sizeof(out.message), "CUDA error: %s", cudaGetErrorString(e));
    } else if (host[0] != 0) {
      out.code = static_cast<int>(host[0]);
      out.rows = 0;
      out.factor = 0;
      snprintf(out.message, sizeof(out.message), "device fault %u at site %u (block %u)", host[0], host[1], host[2]);
      const uint32_t zero[4] = {0, 0, 0, 0};
      cudaMemcpy(fw, zero, sizeof(zero), cudaMemcpyHostToDevice);
    }
  }
  if (info) *info = out;
  if (d) d->err = vae_error_info_t{};
  else {
    std::lock_guard<std::mutex> lk(g_last_mu);
    g_last = vae_error_info_t{};
  }
  return static_cast<vae_status_t>(out.code);
}
