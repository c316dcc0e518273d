// Causal Conv3d as an implicit GEMM on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// Computes, for every output voxel of every patch,
//   y[b,t,h,w,co] = bias[co] + sum_{kt,kh,kw,ci} W[co,ci,kt,kh,kw] * x[b, max(t-2+kt,0), h-1+kh, w-1+kw, ci]
// (+ residual, then depth-to-space), the causal convolution of the video-VAE decoders in DistVAE
// PR #14 "Add tiled VAE parallelism & extended model support" (PatchConv3d padding commit: zero
// padding at image edges, halo rows from the neighbour patch at interior edges; the temporal pad is
// one-sided, frames repeated).
//
// GEMM view: M = output pixels of one frame tile (128 or 256 = rows_t x cols_t pixels of one patch),
// N = output channels (tile BN <= 256), K = 27 taps x C_in, walked tap-major in 64-channel blocks.
// Per K block one TMA box load brings the tap-shifted 128 x 64 input tile (5-D tensor map over the
// channels-last activation; out-of-image rows and columns arrive as zeros, the causal time index is
// clamped at frame 0 or points into the 2 cached frames) and one brings the BN x 64 weight tile.
// Halo taps of a tile at an interior patch edge land in the neighbouring patch's rows of the same
// activation, so halo rows are read in place.  The M tile never crosses a patch edge, so every block
// writes to exactly one patch.  There is no split-K and the K order is fixed, so each output's sum
// runs in the same order whatever the patch grid: outputs are bit-identical across patch counts.
//
// Warp roles (192 threads): warp 0 issues TMA loads into a STAGES-deep shared-memory ring, warp 1
// owns the tensor memory and issues tcgen05.mma (128 x BN x 16, bf16 -> fp32 accumulators in TMEM),
// warps 2-5 drain TMEM with tcgen05.ld and run the epilogue (bias, residual, depth-to-space scatter,
// bf16/fp32 store, optional fused group-norm partial sums).  Every mbarrier wait is bounded.
//
// Launch forms: for weight tiles 128 or 256 wide (convs and unbatched GEMMs) CTAs run in clusters
// of 2 and the pair's two M tiles run as one cta_group::2 MMA (each CTA loads its own A tiles and
// half of the weight tile into its own shared memory; two 64-channel k blocks per stage where they
// fit).  Other weight widths and batched GEMMs run one CTA per tile, each loading its whole weight
// tile.  Every operand load is a plain TMA load into the issuing CTA's shared memory.
// Convs at most 64 channels wide (the Wan pixel head, 64-channel stages) use halo mode: one box of (rows_t + 2) rows of 16
// pixels per (kt, channel chunk) feeds all 9 spatial taps.  The three horizontal taps are stacked
// along N (one MMA of N = 3 x BN per tap row kh, its A rows starting kh box rows down), so each A row
// read from shared memory serves three taps; accumulator row m then holds, for box pixel m, its
// contribution to the outputs one and two columns to its left, and the epilogue adds rows m, m + 1
// and m + 2 (same 16-lane half-warp) with warp shuffles.  The producer and the MMA issuer advance
// ring slot, phase and tap with counters (no divisions on their single-thread critical paths).
#include <cuda.h>

#include <algorithm>
#include <cstdio>
#include <mutex>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace vae {

struct TcParams {
  int mode;  // 0 conv, 1 gemm
  int B, T, H, W, T_in, cache_frames, C_in_pad;
  int res_T_alloc, y_T_alloc;
  int64_t ldd;
  int rows_t, cols_t, n_trows, n_tcols;
  int nph, npw;
  int trow_prefix[kMaxP + 1], tcol_prefix[kMaxP + 1];
  int ph_edges[kMaxP + 1], pw_edges[kMaxP + 1];
  int M, K, batch, m_tiles_per_batch;
  int64_t stride_d;
  float alpha;
  int num_kb, cchunks;
  int N_real, BN, n_ntiles, tmem_cols, stages;
  int msub;  // 128-pixel MMA sub-tiles per tile (2 when BN <= 128: both share each weight tile)
  int ks;    // k blocks (64 channels of one tap) per shared-memory stage: 1 or 2
  // halo mode (narrow convs): one stage = one (kt, 64-channel chunk) halo box of (rows_t + 2) x 16
  // pixels (rows_t = 8 x msub output rows of cols_t = 14 pixels) that all 9 spatial taps read in place,
  // plus those taps' weight tiles ([kh][kw][BN rows]: the 3 kw tiles of one kh form one N = 3 BN operand)
  // halo = 2, tap-stacked (at most kTapMaxN output channels): a box of 16 x 16 pixels (14 x 14 outputs)
  // and one tile of kTapRows weight rows holding all 9 spatial taps, so each MMA is N = kTapRows wide;
  // the epilogue adds the taps' partial sums of neighbouring pixels (kw: warp shuffles within a box
  // row; kh: through scratch shared memory at scratch_off, 2 x kTapMaxN floats per box pixel)
  int halo;
  uint32_t halo_a_bytes, halo_tx, halo_stage, scratch_off;
  const float* bias;
  const void* residual;
  int res_f32;
  void* y;
  int out_f32, out_ncthw;
  int d2s_t, d2s_h, d2s_w, drop, C_d2s, S;
  int T_out, H_out, W_out;
  void* gn_partials;
  int gn_groups, gn_cpg;
  void* y2;          // optional copy of y (channels-last), y2_T_alloc frames per batch item: bf16, or e4m3
  int y2_T_alloc, y2_fp8;
  int fp8;           // e4m3 operands (kind::f8f6f4); kc = channels per 128-byte k block (64 bf16, 128 e4m3)
  int kc;
  int tf32;          // fp32 operands as 3 TF32 products (kc = 32); the weights' remainder rows start at w_lo_row
  int w_lo_row;
  const float* wscale;  // fp8: per-output-channel weight scale (packed row order)
  int natural;       // weight rows (and so accumulator columns) in PyTorch channel order c * S + sub
  int n_tiles;
  int pair;          // 1: CTAs run in clusters of 2 on adjacent M tiles of one N tile as one cta_group::2
                     // MMA, each loading half of the weight tile into its own shared memory
  int n_mtiles, seq_count;
  int npc;           // N tiles per work chunk (divides n_ntiles)
  uint32_t* fault;
  uint64_t limit_ns;
};

namespace {

constexpr int kThreads = 192;
constexpr int kBlockM = 128;
constexpr int kBlockK = 64;
constexpr uint32_t kABytes = kBlockM * kBlockK * 2;  // 16 KB
constexpr int kTapBoxPx = 256;                      // tap-stacked box: 16 rows x 16 pixels

// named barrier 1 over the 4 epilogue warps (barrier 0 is __syncthreads)
VAE_DEV void epi_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// the same barrier, returning whether pred held in every one of the 128 threads
VAE_DEV bool epi_bar_and(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred))
      : "memory");
  return r != 0;
}

VAE_DEV int find_band(const int* prefix, int n, int idx) {
  int i = 0;
  while (i + 1 < n && prefix[i + 1] <= idx) ++i;
  return i;
}

// Group-norm partial sums of one (patch, b, t, group): exact integer sums of q = round(x * 2^18) and of
// q^2, the latter kept as two 64-bit sums (of the low 32 bits and of the rest of every contribution,
// sum q^2 = s2a + s2b * 2^32) so that every update is a plain fire-and-forget atomic add.  Layout must
// match GnPartial in norm.cu.
struct GnPart {
  unsigned long long s1;   // two's complement int64 sum of q
  unsigned long long s2a;  // sum of (contribution mod 2^32)
  unsigned long long s2b;  // sum of (contribution >> 32)
  unsigned long long pad;
};

VAE_DEV void gn_accumulate(GnPart* dst, long long s1, unsigned long long lo, unsigned long long hi) {
  atomicAdd(&dst->s1, static_cast<unsigned long long>(s1));
  atomicAdd(&dst->s2a, lo & 0xffffffffull);
  atomicAdd(&dst->s2b, (lo >> 32) | (hi << 32));
}

}  // namespace

struct TileCoord {
  int b, t, h0, w0, h_end, w_end, patch, m0, bat, n0;
  bool dummy;  // pair mode, odd M-tile count: this CTA computes a copy of the last tile and stores nothing
};

VAE_DEV TileCoord mn_coord(const TcParams& p, int mt, int ntile);

// Work order of the persistent loop: chunks of npc N tiles (whose weights fit in L2 together)
// outermost, then M tiles, then the N tiles of the chunk, so CTAs running at the same time share A
// tiles and their weights stay cached.  In conv mode M tiles run spatial-major and frame-minor: CTAs
// running together read one spatial region of consecutive frames, so the three temporal taps of a
// frame are served from L2.  Pair mode gives CTA `rank` M tile 2i + rank of entry i.
VAE_DEV TileCoord seq_coord(const TcParams& p, int seq, int rank) {
  const int nin = seq % p.npc;
  const int rest = seq / p.npc;
  const int mcount = p.pair ? (p.n_mtiles + 1) / 2 : p.n_mtiles;
  const int mi = rest % mcount;
  const int ntile = (rest / mcount) * p.npc + nin;
  int mt = p.pair ? 2 * mi + rank : mi;
  const bool dummy = mt >= p.n_mtiles;
  if (dummy) mt = p.n_mtiles - 1;
  TileCoord c = mn_coord(p, mt, ntile);
  c.dummy = dummy;
  return c;
}

VAE_DEV TileCoord mn_coord(const TcParams& p, int mt, int ntile) {
  TileCoord c{};
  c.n0 = ntile * p.BN;
  if (p.mode == 0) {
    const int frames = p.B * p.T;
    const int frame = mt % frames;
    const int r = mt / frames;
    const int tr = r / p.n_tcols, tc = r - (r / p.n_tcols) * p.n_tcols;
    const int pi = find_band(p.trow_prefix, p.nph, tr);
    const int pj = find_band(p.tcol_prefix, p.npw, tc);
    c.b = frame / p.T;
    c.t = frame - c.b * p.T;
    c.h0 = p.ph_edges[pi] + (tr - p.trow_prefix[pi]) * p.rows_t;
    c.w0 = p.pw_edges[pj] + (tc - p.tcol_prefix[pj]) * p.cols_t;
    c.h_end = p.ph_edges[pi + 1];
    c.w_end = p.pw_edges[pj + 1];
    c.patch = pi * p.npw + pj;
  } else {
    c.bat = mt / p.m_tiles_per_batch;
    c.m0 = (mt - c.bat * p.m_tiles_per_batch) * kBlockM * p.msub;
  }
  return c;
}

// Exact group sums of one 32-column chunk (STEP channels per group inside the chunk, unrolled so the
// values stay in registers): q = round(x * 2^18) into an int64 sum, q^2 into a 128-bit sum, warp-
// reduced across the 32 rows of this warp, then added to the (patch, b, t, group) slot.
template <int STEP>
VAE_DEV void gn_chunk_sums(const TcParams& p, const TileCoord& tc, const float* v, bool st_ok, int to, int c,
                           int lane) {
#pragma unroll
  for (int i0 = 0; i0 < 32; i0 += STEP) {
    long long s1 = 0;
    unsigned long long lo = 0, hi = 0;
    if (st_ok) {
#pragma unroll
      for (int i = i0; i < i0 + STEP; ++i) {
        const float xv = v[i];
        if (!(fabsf(xv) < 8192.f)) raise_fault(p.fault, FAULT_RANGE, 20);
        const int qv = __float2int_rn(fminf(fmaxf(xv, -8191.f), 8191.f) * 262144.f);
        s1 += qv;
        const unsigned long long sq = static_cast<unsigned long long>(static_cast<long long>(qv) * qv);
        lo += sq;
        if (lo < sq) ++hi;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const long long o1 = __shfl_xor_sync(0xffffffffu, s1, off);
      const unsigned long long olo = __shfl_xor_sync(0xffffffffu, lo, off);
      const unsigned long long ohi = __shfl_xor_sync(0xffffffffu, hi, off);
      s1 += o1;
      const unsigned long long nlo = lo + olo;
      hi += ohi + (nlo < lo ? 1ull : 0ull);
      lo = nlo;
    }
    if (lane == 0 && to >= 0 && (s1 != 0 || lo != 0 || hi != 0)) {
      const int g = (c + i0) / p.gn_cpg;
      GnPart* parts = static_cast<GnPart*>(p.gn_partials);
      const int64_t slot = ((static_cast<int64_t>(tc.patch) * p.B + tc.b) * p.T_out + to) * p.gn_groups + g;
      gn_accumulate(parts + slot, s1, lo, hi);
    }
  }
}

// NCTHW pixels with the natural channel order n = c*S + dt*sh*sw + dy*sw + dx: each run of SW columns is a
// segment of SW horizontally adjacent output pixels of one (c, frame, row), stored as one vector (coalesced
// across the warp, whose lanes hold adjacent input columns).
template <int SW>
VAE_DEV void ncthw_store_runs(const TcParams& p, const TileCoord& tc, int h, int w, int nb, const float* v) {
  const int sh = p.d2s_h;
#pragma unroll
  for (int i = 0; i < 32; i += SW) {
    const int n = nb + i;
    if (n >= p.N_real) break;
    const int c = n / p.S, sub = n - c * p.S;
    const int dt = sub / (sh * SW), dy = (sub - dt * sh * SW) / SW;
    const int to = p.d2s_t * tc.t + dt - p.drop;
    if (to < 0) continue;
    float o[SW];
#pragma unroll
    for (int dx = 0; dx < SW; ++dx)
      o[dx] = v[i + dx] * (p.wscale ? p.wscale[n + dx] : 1.f) + (p.bias ? p.bias[n + dx] : 0.f);
    if (p.residual) {  // (depth-to-space factor 1 only)
      const int64_t ridx = (((static_cast<int64_t>(tc.b) * p.res_T_alloc + tc.t) * p.H + h) * p.W + w) * p.N_real + n;
#pragma unroll
      for (int dx = 0; dx < SW; ++dx)
        o[dx] += p.res_f32 ? static_cast<const float*>(p.residual)[ridx + dx]
                           : bf2f(static_cast<const __nv_bfloat16*>(p.residual)[ridx + dx]);
    }
    const int64_t oidx =
        (((static_cast<int64_t>(tc.b) * p.C_d2s + c) * p.y_T_alloc + to) * p.H_out + (h * sh + dy)) * p.W_out + w * SW;
    if (p.out_f32) {
      float* y = static_cast<float*>(p.y) + oidx;
      if constexpr (SW == 4) *reinterpret_cast<float4*>(y) = make_float4(o[0], o[1], o[2], o[3]);
      else if constexpr (SW == 2) *reinterpret_cast<float2*>(y) = make_float2(o[0], o[1]);
      else y[0] = o[0];
    } else {
      __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.y) + oidx;
      if constexpr (SW == 4) {
        uint2 u;
        reinterpret_cast<__nv_bfloat162*>(&u)[0] = __floats2bfloat162_rn(o[0], o[1]);
        reinterpret_cast<__nv_bfloat162*>(&u)[1] = __floats2bfloat162_rn(o[2], o[3]);
        *reinterpret_cast<uint2*>(y) = u;
      } else if constexpr (SW == 2) {
        *reinterpret_cast<__nv_bfloat162*>(y) = __floats2bfloat162_rn(o[0], o[1]);
      } else {
        y[0] = f2bf(o[0]);
      }
    }
  }
}

// Epilogue of one 32-column chunk held by this thread (one accumulator row).
VAE_DEV void epilogue_chunk(const TcParams& p, const TileCoord& tc, int m, int nb, float* v, int lane) {
  if (tc.dummy) return;
  const int sh = p.d2s_h, sw = p.d2s_w;
  if (p.mode == 1) {
    // ---- GEMM epilogue: D[bat, row, n] = alpha * acc + bias[n] (+ residual)
    const int row = tc.m0 + m;
    const bool valid = row < p.M;
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = v[i] * p.alpha + (p.bias ? p.bias[min(nb + i, p.N_real - 1)] : 0.f);
    if (!valid) return;
    const int64_t base = static_cast<int64_t>(tc.bat) * p.stride_d + static_cast<int64_t>(row) * p.ldd;
    if (p.residual) {
      for (int i = 0; i < 32 && nb + i < p.N_real; ++i)
        v[i] += p.res_f32 ? static_cast<const float*>(p.residual)[base + nb + i]
                          : bf2f(static_cast<const __nv_bfloat16*>(p.residual)[base + nb + i]);
    }
    if (p.N_real % 32 == 0) {
      if (p.out_f32) {
        float* o = static_cast<float*>(p.y) + base + nb;
#pragma unroll
        for (int i = 0; i < 32; i += 8) store8(o + i, v + i);
      } else {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.y) + base + nb;
#pragma unroll
        for (int i = 0; i < 32; i += 8) store8(o + i, v + i);
      }
    } else {
      for (int i = 0; i < 32 && nb + i < p.N_real; ++i) {
        if (p.out_f32) static_cast<float*>(p.y)[base + nb + i] = v[i];
        else static_cast<__nv_bfloat16*>(p.y)[base + nb + i] = f2bf(v[i]);
      }
    }
    return;
  }
  // ---- conv epilogue (halo mode: row m = box pixel (m / 16, m % 16) of the sub-tiles; columns 14, 15
  // of each box row are halo and store nothing)
  const int hm = p.halo ? (m >> 4) : m / p.cols_t;
  const int wm = p.halo ? (m & 15) : m % p.cols_t;
  const int h = tc.h0 + hm;
  const int w = tc.w0 + wm;
  const bool valid = (h < tc.h_end) && (w < tc.w_end) && wm < p.cols_t && (!p.halo || hm < p.rows_t);
  const bool vec = !p.out_ncthw && (p.C_d2s % 32 == 0);
  if (vec) {
    const int sub = nb / p.C_d2s;
    const int c = nb - sub * p.C_d2s;
    if (p.wscale) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] *= p.wscale[nb + i];
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] += p.bias ? p.bias[(c + i) * p.S + sub] : 0.f;
    const int dt = sub / (sh * sw);
    const int rem = sub - dt * sh * sw;
    const int dy = rem / sw, dx = rem - (rem / sw) * sw;
    const int to = p.d2s_t * tc.t + dt - p.drop;
    if (valid && p.residual) {
      const int64_t ridx =
          (((static_cast<int64_t>(tc.b) * p.res_T_alloc + tc.t) * p.H + h) * p.W + w) * p.N_real + nb;
      float r8[8];
#pragma unroll
      for (int i = 0; i < 32; i += 8) {
        if (p.res_f32) load8(static_cast<const float*>(p.residual) + ridx + i, r8);
        else load8(static_cast<const __nv_bfloat16*>(p.residual) + ridx + i, r8);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[i + k] += r8[k];
      }
    }
    const bool st_ok = valid && to >= 0;
    if (st_ok) {
      const int64_t oidx =
          (((static_cast<int64_t>(tc.b) * p.y_T_alloc + to) * p.H_out + (h * sh + dy)) * p.W_out + (w * sw + dx)) *
              p.C_d2s + c;
      if (p.out_f32) {
        float* o = static_cast<float*>(p.y) + oidx;
#pragma unroll
        for (int i = 0; i < 32; i += 8) store8(o + i, v + i);
      } else {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.y) + oidx;
#pragma unroll
        for (int i = 0; i < 32; i += 8) store8(o + i, v + i);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = bf2f(f2bf(v[i]));  // statistics see the stored values
      }
      if (p.y2) {  // copy in the next conv's operand type (bf16 or e4m3)
        const int64_t o2 =
            (((static_cast<int64_t>(tc.b) * p.y2_T_alloc + to) * p.H_out + (h * sh + dy)) * p.W_out + (w * sw + dx)) *
                p.C_d2s + c;
        if (p.y2_fp8) {
          __nv_fp8_e4m3* o = static_cast<__nv_fp8_e4m3*>(p.y2) + o2;
          bool ok = true;
#pragma unroll
          for (int i = 0; i < 32; i += 8) ok = store8_e4m3(o + i, v + i) && ok;
          if (!ok) raise_fault(p.fault, FAULT_RANGE, 21);
        } else {
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.y2) + o2;
#pragma unroll
          for (int i = 0; i < 32; i += 8) store8(o + i, v + i);
        }
      }
    }
    if (p.gn_partials) {
      // exact per-patch group sums of the stored values (all lanes share sub, frame `to` and the group)
      switch (min(p.gn_cpg, 32)) {
        case 4: gn_chunk_sums<4>(p, tc, v, st_ok, to, c, lane); break;
        case 8: gn_chunk_sums<8>(p, tc, v, st_ok, to, c, lane); break;
        case 16: gn_chunk_sums<16>(p, tc, v, st_ok, to, c, lane); break;
        default: gn_chunk_sums<32>(p, tc, v, st_ok, to, c, lane); break;
      }
    }
  } else if (p.out_ncthw && p.natural && (sw == 1 || sw == 2 || sw == 4)) {
    if (!valid) return;
    if (sw == 4) ncthw_store_runs<4>(p, tc, h, w, nb, v);
    else if (sw == 2) ncthw_store_runs<2>(p, tc, h, w, nb, v);
    else ncthw_store_runs<1>(p, tc, h, w, nb, v);
  } else {
    // generic scalar path (NCTHW pixels, or channel counts not a multiple of 32)
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int n = nb + i;
      if (n >= p.N_real) continue;
      const int sub = p.natural ? n % p.S : n / p.C_d2s;
      const int c = p.natural ? n / p.S : n - sub * p.C_d2s;
      float val = v[i] * (p.wscale ? p.wscale[n] : 1.f) + (p.bias ? p.bias[c * p.S + sub] : 0.f);
      const int dt = sub / (sh * sw);
      const int rem = sub - dt * sh * sw;
      const int dy = rem / sw, dx = rem - (rem / sw) * sw;
      const int to = p.d2s_t * tc.t + dt - p.drop;
      if (!valid || to < 0) continue;
      if (p.residual) {
        const int64_t ridx = (((static_cast<int64_t>(tc.b) * p.res_T_alloc + tc.t) * p.H + h) * p.W + w) * p.N_real + n;
        val += p.res_f32 ? static_cast<const float*>(p.residual)[ridx]
                         : bf2f(static_cast<const __nv_bfloat16*>(p.residual)[ridx]);
      }
      const int ho = h * sh + dy, wo = w * sw + dx;
      int64_t oidx;
      if (p.out_ncthw)
        oidx = (((static_cast<int64_t>(tc.b) * p.C_d2s + c) * p.y_T_alloc + to) * p.H_out + ho) * p.W_out + wo;
      else
        oidx = (((static_cast<int64_t>(tc.b) * p.y_T_alloc + to) * p.H_out + ho) * p.W_out + wo) * p.C_d2s + c;
      if (p.out_f32) static_cast<float*>(p.y)[oidx] = val;
      else static_cast<__nv_bfloat16*>(p.y)[oidx] = f2bf(val);
    }
  }
}

// Persistent kernel: each block walks tiles blockIdx.x, blockIdx.x + gridDim.x, ...  The shared-
// memory ring runs continuously across tiles; two TMEM accumulators let the epilogue of one tile
// overlap the MMAs of the next.
//
// kPair (conv mode, clusters of 2): the two CTAs' M tiles run as ONE tcgen05 MMA of 256 x BN
// (cta_group::2).  Each CTA loads its own 128-pixel A tiles and one half (BN/2 rows) of the weight
// tile; the leader's full barrier counts both CTAs' bytes, the leader alone issues the MMAs, and its
// commits free the stage and hand the accumulator to the epilogues in both CTAs.  Each SM then takes
// in half as many weight bytes per MMA as a CTA that holds the whole weight tile.
// kOp, the operand kind (a template parameter so that each kernel's single-thread MMA issue loop carries
// no test of it): 0 bf16 (kind::f16), 1 e4m3 (kind::f8f6f4), 2 fp32 as three TF32 products
// (kind::tf32: a_hi b_hi + a_hi b_lo + a_lo b_hi, the high parts and remainders loaded as separate
// tiles, tmA2 the remainders of x; 32 fp32 channels per 128-byte k block).
template <bool kPair, int kOp>
__global__ void __launch_bounds__(kThreads, 1)
    conv_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ TcParams p) {
  constexpr bool kF8 = kOp == 1;
  constexpr bool kT32 = kOp == 2;
  constexpr uint32_t kParts = kT32 ? 2u : 1u;  // high parts and remainders
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // one stage = ks k blocks: [A of k block 0 .. ks-1][B of k block 0 .. ks-1]; with kT32 each A and B
  // block holds the high-part tile, then the remainder tile
  const uint32_t b_half = static_cast<uint32_t>(kPair ? p.BN / 2 : p.BN) * kBlockK * 2;
  const uint32_t a_half = kABytes * static_cast<uint32_t>(p.msub);
  const uint32_t b_bytes = b_half * kParts;  // per k block
  const uint32_t a_bytes = a_half * kParts;  // per k block
  const int ks = p.ks;
  const bool halo = !kPair && p.halo;
  const uint32_t stage_bytes = halo ? p.halo_stage : static_cast<uint32_t>(ks) * (a_bytes + b_bytes);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + p.stages * stage_bytes);
  uint64_t* empty_bar = full_bar + p.stages;
  uint64_t* accf_bar = empty_bar + p.stages;  // [2] accumulator full (MMA -> epilogue)
  uint64_t* acce_bar = accf_bar + 2;          // [2] accumulator empty (epilogue -> MMA)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce_bar + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int acc_stride = p.tmem_cols / 2;
  const int rank = p.pair ? static_cast<int>(cluster_ctarank()) : 0;
  const int seq0 = p.pair ? blockIdx.x >> 1 : blockIdx.x;
  const int seq_step = p.pair ? gridDim.x >> 1 : gridDim.x;
  const uint16_t pair_mask = 0x3;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);  // MMA pairs: the leader's commit frees the stage in both CTAs
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accf_bar[a], 1);
      mbar_init(&acce_bar[a], kPair ? 2 * 4 : 4 * 32);  // MMA pairs: one arrival per epilogue warp of each CTA
    }
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if constexpr (kT32) tma_prefetch_desc(&tmA2);
  }
  if (warp == 1) {
    if constexpr (kPair) tmem_alloc_pair(tmem_slot, static_cast<uint32_t>(p.tmem_cols));
    else tmem_alloc(tmem_slot, static_cast<uint32_t>(p.tmem_cols));
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the peer's barriers (and, for MMA pairs, its tensor memory) exist before anything targets them
  if (p.pair) cluster_sync();

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if constexpr (!kPair) {
      if (p.halo) {
        if (lane == 0) {
          const int stages = p.stages, cchunks = p.cchunks;
          const uint32_t wt_bytes = static_cast<uint32_t>(p.BN) * kBlockK * 2;
          int kc = 0, s = 0;
          uint32_t ph = 0;
          bool ok = true;
          for (int seq = seq0; seq < p.seq_count && ok; seq += seq_step) {
            const TileCoord tc = seq_coord(p, seq, rank);
            for (int kt = 0; kt < 3 && ok; ++kt) {
              const int ti = max(tc.t + kt - 2 + p.cache_frames, 0);
              for (int cc = 0; cc < cchunks; ++cc, ++kc) {
                if (kc >= stages && !mbar_wait(&empty_bar[s], ph ^ 1u, p.fault, p.limit_ns, 1)) {
                  ok = false;
                  break;
                }
                uint8_t* a_dst = smem + s * stage_bytes;
                uint8_t* b_dst = a_dst + p.halo_a_bytes;
                mbar_arrive_expect_tx(&full_bar[s], p.halo_tx);
                tma_load_5d(a_dst, &tmA, &full_bar[s], cc * kBlockK, tc.w0 - 1, tc.h0 - 1, ti, tc.b);
                if (p.halo == 2) {
                  tma_load_2d(b_dst, &tmB, &full_bar[s], cc * kBlockK, kt * kTapRows);
                } else {
#pragma unroll 1
                  for (int t9 = 0; t9 < 9; ++t9)
                    tma_load_2d(b_dst + t9 * wt_bytes, &tmB, &full_bar[s], (kt * 9 + t9) * p.C_in_pad + cc * kBlockK,
                                tc.n0);
                }
                if (++s == stages) {
                  s = 0;
                  ph ^= 1u;
                }
              }
            }
          }
          for (int k = max(0, kc - p.stages); k < kc; ++k)
            mbar_wait(&full_bar[k % p.stages], (k / p.stages) & 1, p.fault, p.limit_ns, 2);
        }
      }
    }
    if (lane == 0 && !halo) {
      // per-k-block state advances by counters (no divisions on this thread's critical path)
      const int stages = p.stages, num_st = p.num_kb / ks, cchunks = p.cchunks;
      int kc = 0;        // stages filled so far (all tiles)
      int s = 0;         // ring slot of the next k block
      uint32_t ph = 0;   // parity of that slot's current use
      bool ok = true;
      for (int seq = seq0; seq < p.seq_count && ok; seq += seq_step) {
        const TileCoord tc = seq_coord(p, seq, rank);
        int cc = 0, kt = 0, kh = 0, kw = 0, kcol = 0;  // kcol = tap * C_in_pad + cc * kc
        int kb = 0;                                    // k block (GEMM mode)
        for (int st = 0; st < num_st; ++st, ++kc) {
          if (kc >= stages && !mbar_wait(&empty_bar[s], ph ^ 1u, p.fault, p.limit_ns, 1)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = smem + s * stage_bytes;
          uint8_t* b_dst = a_dst + ks * a_bytes;
          if (p.mode == 0) {
            uint32_t fb = 0;
            if constexpr (kPair) {
              // both CTAs' tiles complete on the leader's barrier (the leader alone runs the MMAs)
              fb = cluster_map(smem_u32(&full_bar[s]), 0);
              if (rank == 0) mbar_arrive_expect_tx(&full_bar[s], 2 * stage_bytes);
            } else {
              mbar_arrive_expect_tx(&full_bar[s], stage_bytes);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              if (j == ks) break;
              const int ti = max(tc.t + kt - 2 + p.cache_frames, 0);
              uint8_t* aj = a_dst + j * a_bytes;
              uint8_t* bj = b_dst + j * b_bytes;
              if constexpr (kPair) {
                tma_load_5d_pair(aj, &tmA, fb, cc * p.kc, tc.w0 + kw - 1, tc.h0 + kh - 1, ti, tc.b);
                tma_load_2d_pair(bj, &tmB, fb, kcol, tc.n0 + rank * (p.BN / 2));
                if constexpr (kT32) {
                  tma_load_5d_pair(aj + a_half, &tmA2, fb, cc * p.kc, tc.w0 + kw - 1, tc.h0 + kh - 1, ti, tc.b);
                  tma_load_2d_pair(bj + b_half, &tmB, fb, kcol, p.w_lo_row + tc.n0 + rank * (p.BN / 2));
                }
              } else {
                tma_load_5d(aj, &tmA, &full_bar[s], cc * p.kc, tc.w0 + kw - 1, tc.h0 + kh - 1, ti, tc.b);
                tma_load_2d(bj, &tmB, &full_bar[s], kcol, tc.n0);
                if constexpr (kT32) {
                  tma_load_5d(aj + a_half, &tmA2, &full_bar[s], cc * p.kc, tc.w0 + kw - 1, tc.h0 + kh - 1, ti, tc.b);
                  tma_load_2d(bj + b_half, &tmB, &full_bar[s], kcol, p.w_lo_row + tc.n0);
                }
              }
              // next (tap, channel chunk): channel chunks innermost, then kw, kh, kt
              kcol += p.kc;
              if (++cc == cchunks) {
                cc = 0;
                if (++kw == 3) {
                  kw = 0;
                  if (++kh == 3) {
                    kh = 0;
                    ++kt;
                  }
                }
              }
            }
          } else {
            // GEMM mode: ks consecutive k blocks per stage
            uint32_t fb = 0;
            if constexpr (kPair) {
              fb = cluster_map(smem_u32(&full_bar[s]), 0);
              if (rank == 0) mbar_arrive_expect_tx(&full_bar[s], 2 * stage_bytes);
            } else {
              mbar_arrive_expect_tx(&full_bar[s], stage_bytes);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              if (j == ks) break;
              uint8_t* aj = a_dst + j * a_bytes;
              uint8_t* bj = b_dst + j * b_bytes;
              if constexpr (kPair) {
                tma_load_3d_pair(aj, &tmA, fb, kb * kBlockK, tc.m0, tc.bat);
                tma_load_3d_pair(bj, &tmB, fb, kb * kBlockK, tc.n0 + rank * (p.BN / 2), tc.bat);
              } else {
                tma_load_3d(aj, &tmA, &full_bar[s], kb * kBlockK, tc.m0, tc.bat);
                tma_load_3d(bj, &tmB, &full_bar[s], kb * kBlockK, tc.n0, tc.bat);
              }
              ++kb;
            }
          }
          if (++s == stages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // drain: every issued load has landed before the block may exit (an MMA pair's follower sees
      // that through the empty barriers below: the leader consumed its tiles)
      if (!kPair || rank == 0)
        for (int k = max(0, kc - p.stages); k < kc; ++k)
          mbar_wait(&full_bar[k % p.stages], (k / p.stages) & 1, p.fault, p.limit_ns, 2);
      // MMA pair: the leader's MMAs have released every stage, so no commit arrival is still on its way
      if (kPair)
        for (int k = max(0, kc - p.stages); k < kc; ++k)
          mbar_wait(&empty_bar[k % p.stages], (k / p.stages) & 1, p.fault, p.limit_ns, 7);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if constexpr (!kPair) {
      if (p.halo) {
        if (lane == 0) {
          // tap row kh, sub-tile sub: A = the 128 box pixels from box row sub * 8 + kh on (8 box rows of
          // 16 pixels, 2048 B each, so every start is 1024-byte aligned), B = the kw = 0, 1, 2 weight tiles of
          // kh (3 BN rows), D = 3 BN columns of the sub-tile's accumulator
          // (tap-stacked: A = the 128 box pixels from box row sub * 8, B = all 9 taps' kTapRows rows)
          const bool tap = p.halo == 2;
          const uint32_t n3 = 3u * static_cast<uint32_t>(p.BN);
          const uint32_t idesc = idesc_bf16_f32(kBlockM, tap ? static_cast<uint32_t>(kTapRows) : n3);
          const int stages = p.stages, num_st = 3 * p.cchunks, msub = p.msub;
          const uint32_t smem_base = smem_u32(smem);
          const uint32_t wt_bytes = static_cast<uint32_t>(p.BN) * kBlockK * 2;
          int s = 0, it = 0;
          uint32_t ph = 0;
          bool ok = true;
          for (int seq = seq0; seq < p.seq_count && ok; seq += seq_step, ++it) {
            const int acc = it & 1, u = it >> 1;
            if (u > 0 && !mbar_wait(&acce_bar[acc], (u - 1) & 1, p.fault, p.limit_ns, 6)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * acc_stride);
            for (int st = 0; st < num_st; ++st) {
              if (!mbar_wait(&full_bar[s], ph, p.fault, p.limit_ns, 3)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t a_addr = smem_base + static_cast<uint32_t>(s) * stage_bytes;
              const uint32_t b_addr = a_addr + p.halo_a_bytes;
              if (tap) {
                const uint64_t bdesc = sdesc_kmajor_sw128(b_addr);
                for (int sub = 0; sub < msub; ++sub) {
                  const uint64_t adesc = sdesc_kmajor_sw128(a_addr + static_cast<uint32_t>(sub) * kBlockM * 128u);
                  const uint32_t d_sub = d_tmem + static_cast<uint32_t>(sub * kTapRows);
#pragma unroll
                  for (int k = 0; k < kBlockK / 16; ++k)
                    tc_mma_bf16(d_sub, adesc + static_cast<uint64_t>(2 * k), bdesc + static_cast<uint64_t>(2 * k),
                                idesc, (st == 0 && k == 0) ? 0u : 1u);
                }
              }
#pragma unroll 1
              for (uint32_t kh = 0; kh < (tap ? 0u : 3u); ++kh) {
                const uint64_t bdesc = sdesc_kmajor_sw128(b_addr + kh * 3u * wt_bytes);
                for (int sub = 0; sub < msub; ++sub) {
                  const uint32_t row0 = (static_cast<uint32_t>(sub) * 8u + kh) * 16u;
                  const uint64_t adesc = sdesc_kmajor_sw128(a_addr + row0 * 128u);
                  const uint32_t d_sub = d_tmem + static_cast<uint32_t>(sub) * n3;
#pragma unroll
                  for (int k = 0; k < kBlockK / 16; ++k)
                    tc_mma_bf16(d_sub, adesc + static_cast<uint64_t>(2 * k), bdesc + static_cast<uint64_t>(2 * k),
                                idesc, (st == 0 && kh == 0 && k == 0) ? 0u : 1u);
                }
              }
              tc_commit(&empty_bar[s]);
              if (++s == stages) {
                s = 0;
                ph ^= 1u;
              }
            }
            tc_commit(&accf_bar[acc]);
          }
        }
      }
    }
    if (lane == 0 && (!kPair || rank == 0) && !halo) {
      const uint32_t mm = kPair ? 2 * kBlockM : kBlockM;
      constexpr bool fp8 = kF8;
      const uint32_t idesc = fp8    ? idesc_e4m3_f32(mm, static_cast<uint32_t>(p.BN))
                             : kT32 ? idesc_tf32_f32(mm, static_cast<uint32_t>(p.BN))
                                    : idesc_bf16_f32(mm, static_cast<uint32_t>(p.BN));
      const int stages = p.stages, num_st = p.num_kb / ks, msub = p.msub;
      const uint32_t smem_base = smem_u32(smem);
      const uint32_t sub_cols = static_cast<uint32_t>(p.BN);
      int s = 0, it = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int seq = seq0; seq < p.seq_count && ok; seq += seq_step, ++it) {
        const int acc = it & 1, u = it >> 1;
        if (u > 0 && !mbar_wait(&acce_bar[acc], (u - 1) & 1, p.fault, p.limit_ns, 6)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * acc_stride);
        for (int st = 0; st < num_st; ++st) {
          if (!mbar_wait(&full_bar[s], ph, p.fault, p.limit_ns, 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_base + static_cast<uint32_t>(s) * stage_bytes;
          const uint32_t b_addr = a_addr + static_cast<uint32_t>(ks) * a_bytes;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (j == ks) break;
            const uint64_t bdesc = sdesc_kmajor_sw128(b_addr + static_cast<uint32_t>(j) * b_bytes);
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
              if (sub == msub) break;
              const uint64_t adesc =
                  sdesc_kmajor_sw128(a_addr + static_cast<uint32_t>(j) * a_bytes + static_cast<uint32_t>(sub) * kABytes);
              const uint32_t d_sub = d_tmem + static_cast<uint32_t>(sub) * sub_cols;
              const uint32_t first = (st == 0 && j == 0) ? 1u : 0u;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                // advance 32 B along K inside the 128-byte swizzle atom: 16 bf16, 32 e4m3 or 8 tf32 per MMA
                const uint32_t accum = (first && k == 0) ? 0u : 1u;
                const uint64_t ak = adesc + static_cast<uint64_t>(2 * k), bk = bdesc + static_cast<uint64_t>(2 * k);
                if constexpr (kT32) {
                  // the remainder tiles sit a_half / b_half bytes after the high parts (16-byte units)
                  const uint64_t akl = ak + static_cast<uint64_t>(a_half >> 4);
                  const uint64_t bkl = bk + static_cast<uint64_t>(b_half >> 4);
                  if constexpr (kPair) {
                    tc_mma_tf32_pair(d_sub, ak, bk, idesc, accum);
                    tc_mma_tf32_pair(d_sub, ak, bkl, idesc, 1u);
                    tc_mma_tf32_pair(d_sub, akl, bk, idesc, 1u);
                  } else {
                    tc_mma_tf32(d_sub, ak, bk, idesc, accum);
                    tc_mma_tf32(d_sub, ak, bkl, idesc, 1u);
                    tc_mma_tf32(d_sub, akl, bk, idesc, 1u);
                  }
                } else if constexpr (kPair && fp8) tc_mma_e4m3_pair(d_sub, ak, bk, idesc, accum);
                else if constexpr (kPair) tc_mma_bf16_pair(d_sub, ak, bk, idesc, accum);
                else if constexpr (fp8) tc_mma_e4m3(d_sub, ak, bk, idesc, accum);
                else tc_mma_bf16(d_sub, ak, bk, idesc, accum);
              }
            }
          }
          if constexpr (kPair) tc_commit_pair_arrive_both(&empty_bar[s], pair_mask);
          else tc_commit(&empty_bar[s]);
          if (++s == stages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if constexpr (kPair) tc_commit_pair_arrive_both(&accf_bar[acc], pair_mask);
        else tc_commit(&accf_bar[acc]);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int m = q * 32 + lane;
    int it = 0;
    if (!kPair && p.halo == 2) {
      // tap-stacked: accumulator row p = box pixel (p / 16, p % 16), column (kh * 3 + kw) * kTapMaxN + n.
      // R_kh(p) = sum over kw of row p + kw, column tap(kh, kw) (shuffles within the 16-lane box row);
      // output (r, c) = R_0(p) + R_1(p + 16) + R_2(p + 32), the last two through scratch[kh - 1][n][p].
      float* scr = reinterpret_cast<float*>(smem + p.scratch_off);
      for (int seq = seq0; seq < p.seq_count; seq += seq_step, ++it) {
        const int acc = it & 1, u = it >> 1;
        const bool got = mbar_wait(&accf_bar[acc], u & 1, p.fault, p.limit_ns, 5);
        if (!epi_bar_and(got)) break;  // the four warps leave together, so no later barrier waits alone
        tc_fence_after();
        const TileCoord tc = seq_coord(p, seq, rank);
        float r0[2][kTapMaxN];
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
#pragma unroll
          for (int kh = 0; kh < 3; ++kh) {
            const int c0 = kh * 3 * kTapMaxN, lo = c0 / 16 * 16;
            uint32_t raw[48];
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * acc_stride + sub * kTapRows + lo);
            tmem_ld_32x32b_x16(taddr, raw);
            tmem_ld_32x32b_x16(taddr + 16u, raw + 16);
            tmem_ld_32x32b_x16(taddr + 32u, raw + 32);
            tmem_ld_wait();
#pragma unroll
            for (int n = 0; n < kTapMaxN; ++n) {
              const int o = c0 - lo + n;
              float v = __uint_as_float(raw[o]);
              v += __shfl_down_sync(0xffffffffu, __uint_as_float(raw[o + kTapMaxN]), 1);
              v += __shfl_down_sync(0xffffffffu, __uint_as_float(raw[o + 2 * kTapMaxN]), 2);
              if (kh == 0) r0[sub][n] = v;
              else scr[((kh - 1) * kTapMaxN + n) * kTapBoxPx + sub * kBlockM + m] = v;
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&acce_bar[acc]);  // every TMEM read of this accumulator is done
        epi_bar_sync();
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          const int px = sub * kBlockM + m;
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
          if ((px >> 4) < 14 && (px & 15) < 14) {  // an output pixel: px + 32 stays inside the box
#pragma unroll
            for (int n = 0; n < kTapMaxN; ++n)
              v[n] = r0[sub][n] + scr[n * kTapBoxPx + px + 16] + scr[(kTapMaxN + n) * kTapBoxPx + px + 32];
          }
          epilogue_chunk(p, tc, px, tc.n0, v, lane);  // (n0 = 0: one weight tile)
        }
        epi_bar_sync();  // scratch is read before the next tile writes it
      }
    }
    for (int seq = seq0; seq < p.seq_count && !(!kPair && p.halo == 2); seq += seq_step, ++it) {
      const int acc = it & 1, u = it >> 1;
      if (!mbar_wait(&accf_bar[acc], u & 1, p.fault, p.limit_ns, 5)) break;
      tc_fence_after();
      const TileCoord tc = seq_coord(p, seq, rank);
      const int nchunks = (p.BN + 31) / 32;
      if (!kPair && p.halo) {
        // output (r, c) of the sub-tile = sum over kw of accumulator row (r, c + kw), columns kw * BN + n
        const int n3 = 3 * p.BN;
        for (int sub = 0; sub < p.msub; ++sub) {
          for (int j = 0; j < nchunks; ++j) {
            float v[32];
#pragma unroll
            for (int kw = 0; kw < 3; ++kw) {
              uint32_t raw[32];
              const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                     static_cast<uint32_t>(acc * acc_stride + sub * n3 + kw * p.BN + j * 32);
              if (p.BN - j * 32 >= 32) {
                tmem_ld_32x32b_x32(taddr, raw);
              } else {
                tmem_ld_32x32b_x16(taddr, raw);
#pragma unroll
                for (int i = 16; i < 32; ++i) raw[i] = 0u;
              }
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                float f = __uint_as_float(raw[i]);
                if (kw) f = __shfl_down_sync(0xffffffffu, f, kw);
                v[i] = kw ? v[i] + f : f;
              }
            }
            if (sub == p.msub - 1 && j == nchunks - 1) {
              tc_fence_before();
              mbar_arrive(&acce_bar[acc]);
            }
            const int nb = tc.n0 + j * 32;
            if (nb < p.N_real) epilogue_chunk(p, tc, sub * kBlockM + m, nb, v, lane);
          }
        }
        continue;
      }
      for (int sub = 0; sub < p.msub; ++sub) {
        for (int j = 0; j < nchunks; ++j) {
          uint32_t raw[32];
          tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                 static_cast<uint32_t>(acc * acc_stride + sub * p.BN + j * 32),
                             raw);
          tmem_ld_wait();
          if (sub == p.msub - 1 && j == nchunks - 1) {
            // every TMEM read of this accumulator is done: hand it back to the MMA warp
            tc_fence_before();
            if constexpr (kPair) {
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster(cluster_map(smem_u32(&acce_bar[acc]), 0));
            } else {
              mbar_arrive(&acce_bar[acc]);
            }
          }
          const int nb = tc.n0 + j * 32;
          if (nb >= p.N_real) continue;
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(raw[i]);
          epilogue_chunk(p, tc, sub * kBlockM + m, nb, v, lane);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (kPair) tmem_dealloc_pair(tmem_base, static_cast<uint32_t>(p.tmem_cols));
    else tmem_dealloc(tmem_base, static_cast<uint32_t>(p.tmem_cols));
  }
  if (p.pair) cluster_sync();  // neither CTA leaves while the other may still write into it
}

// ================================================================================ host side
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// esz: element bytes (1 = e4m3 bytes, 2 = bf16, 4 = fp32)
bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
              const uint32_t* box, int esz = 2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  const CUtensorMapDataType dt = esz == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : esz == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                            : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = fn(m, dt, rank,
                  const_cast<void*>(base), d, s, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int pick_cols(const int* pw, int npw) {
  // tile width (pixels) that wastes the fewest M rows over the patch widths; ties -> 16
  static const int cand[4] = {16, 8, 32, 64};
  int best = 16;
  long best_tiles = -1;
  for (int ci = 0; ci < 4; ++ci) {
    const int cw = cand[ci];
    long tiles = 0;
    for (int j = 0; j < npw; ++j) tiles += (pw[j + 1] - pw[j] + cw - 1) / cw;
    const long area = tiles * cw;  // pixels computed per tile-row band
    if (best_tiles < 0 || area < best_tiles) {
      best_tiles = area;
      best = cw;
    }
  }
  return best;
}

}  // namespace

namespace {
// Convs and unbatched GEMMs whose weight tile is 128 or 256 channels wide run each pair's two M tiles
// as one cta_group::2 MMA, each CTA holding half of the weight tile (measured on one GB300: op conv
// 512->512 1311 -> 1386 TFLOP/s).
bool mma_pair_enabled() { return true; }
// Convs at most 64 channels wide load one halo box per (kt, channel chunk) that the 9 spatial taps share,
// and stack the 3 horizontal taps along N (measured on one GB300: Wan 256->12 head on 81x352x640
// 16.35 -> 8.19 ms, 64->64 conv on 41x176x320 0.84 -> 0.51 ms).
bool halo_mode_enabled() { return true; }
constexpr int kHaloCols = 14;  // output columns of a tile: box rows of 16 pixels (14 + 2 halo)
}  // namespace

namespace {
// Per-device launch facts, filled once per device under a lock (several host threads may launch).
struct DevLaunch {
  bool ready = false;
  int n_sm = 0;
  int max_clusters = 0;          // clusters of 2 resident at once for the pair kernel ...
  size_t max_clusters_smem = 0;  // ... at this dynamic shared-memory size ...
  const void* max_clusters_kern = nullptr;  // ... for this kernel
};
std::mutex g_dev_mu;
DevLaunch g_dev[64];
}  // namespace

cudaError_t launch_conv_tc(const ConvTcArgs& a, cudaStream_t stream) {
  TcParams p{};  // per call: concurrent launches from several host threads never share it
  p.mode = a.mode;
  p.N_real = a.N_real;
  if (a.N_pad <= 256) {
    p.BN = a.N_pad;
  } else {
    p.BN = 256;
  }
  if (p.BN % 16 != 0 || p.BN < 16) return cudaErrorInvalidValue;
  p.n_ntiles = (a.N_pad + p.BN - 1) / p.BN;
  p.msub = p.BN <= 128 ? 2 : 1;
  // clusters of 2 run one cta_group::2 MMA over two adjacent M tiles of one weight tile (a batched GEMM
  // has a different B per batch item, so only unbatched GEMMs pair up)
  p.fp8 = a.fp8 ? 1 : 0;
  p.tf32 = a.tf32 ? 1 : 0;
  p.kc = p.fp8 ? 128 : p.tf32 ? 32 : 64;
  if (p.fp8 && (a.mode != 0 || !a.wscale || a.C_in_pad % 128 != 0)) return cudaErrorInvalidValue;
  if (p.tf32 && (a.mode != 0 || p.fp8 || !a.x_lo || a.tap_stacked || a.C_in_pad % 32 != 0)) return cudaErrorInvalidValue;
  p.w_lo_row = a.N_pad;
  p.wscale = p.fp8 ? a.wscale : nullptr;
  // (NCTHW pixel outputs wider than 16 channels only with vector stores (natural channel order): with
  // scalar stores the epilogue outlasts the shorter MMA phase; measured on one GB300: LTX 128->48 head
  // 3.66 ms per tap, 5.73 ms in halo mode with scalar stores)
  p.halo = (a.mode == 0 && p.BN <= 64 && !p.fp8 && !p.tf32 && (!a.out_ncthw || a.natural || a.N_real <= 16) &&
            halo_mode_enabled())
               ? 1
               : 0;
  if (a.tap_stacked) {  // weights packed tap-stacked (the caller decides, as it packs them)
    if (a.mode != 0 || p.fp8 || a.N_real > kTapMaxN || p.BN != 16 || !halo_mode_enabled()) return cudaErrorInvalidValue;
    p.halo = 2;
  }
  // halo mode: sub-tiles of 8 x 16 box pixels; two accumulators of msub x 3 BN columns must fit TMEM
  if (p.halo == 1) p.msub = 2 * 2 * 3 * p.BN <= 512 ? 2 : 1;
  if (p.halo == 2) p.msub = 2;
  const bool mma_pair =
      mma_pair_enabled() && (p.BN == 256 || p.BN == 128) && (a.mode == 0 || a.batch == 1) && !p.halo;
  const bool want_pair = mma_pair;
  p.tmem_cols = 32;
  while (p.tmem_cols < 2 * p.msub * (p.halo == 2 ? kTapRows : p.halo ? 3 * p.BN : p.BN)) p.tmem_cols <<= 1;
  if (p.tmem_cols > 512) return cudaErrorInvalidValue;
  const uint32_t kb_bytes = (kABytes * p.msub + static_cast<uint32_t>(mma_pair ? p.BN / 2 : p.BN) * kBlockK * 2) *
                            (p.tf32 ? 2u : 1u);  // (3 x TF32: high parts and remainders)
  // MMA pairs take two k blocks per stage (half the barrier round trips per MMA) where two such stages
  // fit; measured on one GB300: +11% on a 512->512 conv (3 stages), +12% on 128->128 (2 stages)
  // (a conv's 27 taps x cchunks k blocks split evenly into pairs when cchunks is even)
  const int kb_even = a.mode == 0 ? (a.C_in_pad / p.kc) % 2 == 0 : (a.K / kBlockK) % 2 == 0;
  p.ks = (mma_pair && kb_even && 2u * 2u * kb_bytes <= 200u * 1024u) ? 2 : 1;
  uint32_t stage_bytes = static_cast<uint32_t>(p.ks) * kb_bytes;
  if (p.halo == 1) {
    // box of (8 msub + 2) x 16 pixels x 64 channels, then the 9 taps' BN x 64 weight tiles
    const uint32_t box = static_cast<uint32_t>(8 * p.msub + 2) * (kHaloCols + 2) * kBlockK * 2;
    p.halo_a_bytes = (box + 1023u) & ~1023u;
    p.halo_tx = box + 9u * static_cast<uint32_t>(p.BN) * kBlockK * 2;
    p.halo_stage = p.halo_a_bytes + 9u * static_cast<uint32_t>(p.BN) * kBlockK * 2;
  } else if (p.halo == 2) {
    // box of 16 x 16 pixels x 64 channels, then one kTapRows x 64 tap-stacked weight tile
    const uint32_t box = static_cast<uint32_t>(kTapBoxPx) * kBlockK * 2;
    p.halo_a_bytes = box;
    p.halo_tx = box + static_cast<uint32_t>(kTapRows) * kBlockK * 2;
    p.halo_stage = p.halo_tx;
  }
  if (p.halo) {
    p.ks = 1;
    stage_bytes = p.halo_stage;
  }
  p.stages = std::min(8, static_cast<int>((200u * 1024u) / stage_bytes));
  if (p.stages < 2) return cudaErrorInvalidValue;
  // barriers after the stages, then (tap-stacked) the epilogue's exchange of the kh = 1, 2 partial sums
  p.scratch_off = static_cast<uint32_t>(p.stages) * stage_bytes + (2u * p.stages + 4u) * 8u + 16u;
  const uint32_t scratch_bytes = p.halo == 2 ? 2u * kTapMaxN * kTapBoxPx * 4u : 0u;
  p.bias = a.bias;
  p.residual = a.residual;
  p.res_f32 = a.res_f32;
  p.y = a.y;
  p.out_f32 = a.out_f32;
  p.out_ncthw = a.out_ncthw;
  p.natural = a.natural;
  p.fault = fault_word();
  p.limit_ns = wait_limit_ns();

  CUtensorMap tmA, tmB, tmA2;
  memset(&tmA2, 0, sizeof(tmA2));
  long long n_blocks;
  if (a.mode == 0) {
    p.B = a.B; p.T = a.T; p.H = a.H; p.W = a.W; p.T_in = a.T_in; p.cache_frames = a.cache_frames;
    p.C_in_pad = a.C_in_pad;
    if (a.C_in_pad % p.kc != 0 || a.nph > kMaxP || a.npw > kMaxP) return cudaErrorInvalidValue;
    p.nph = a.nph; p.npw = a.npw;
    for (int i = 0; i <= a.nph; ++i) p.ph_edges[i] = a.ph_edges[i];
    for (int j = 0; j <= a.npw; ++j) p.pw_edges[j] = a.pw_edges[j];
    p.cols_t = p.halo ? kHaloCols : pick_cols(a.pw_edges, a.npw);
    p.rows_t = p.halo == 2 ? 14 : p.halo ? 8 * p.msub : kBlockM * p.msub / p.cols_t;
    p.trow_prefix[0] = 0;
    for (int i = 0; i < a.nph; ++i)
      p.trow_prefix[i + 1] = p.trow_prefix[i] + (a.ph_edges[i + 1] - a.ph_edges[i] + p.rows_t - 1) / p.rows_t;
    p.tcol_prefix[0] = 0;
    for (int j = 0; j < a.npw; ++j)
      p.tcol_prefix[j + 1] = p.tcol_prefix[j] + (a.pw_edges[j + 1] - a.pw_edges[j] + p.cols_t - 1) / p.cols_t;
    p.n_trows = p.trow_prefix[a.nph];
    p.n_tcols = p.tcol_prefix[a.npw];
    p.cchunks = a.C_in_pad / p.kc;
    p.num_kb = 27 * p.cchunks;
    p.d2s_t = a.d2s_t; p.d2s_h = a.d2s_h; p.d2s_w = a.d2s_w;
    p.S = a.d2s_t * a.d2s_h * a.d2s_w;
    p.C_d2s = a.N_real / p.S;
    p.drop = a.drop_first ? a.d2s_t - 1 : 0;
    p.T_out = a.d2s_t * a.T - p.drop;
    p.H_out = a.H * a.d2s_h;
    p.W_out = a.W * a.d2s_w;
    p.res_T_alloc = a.res_T_alloc ? a.res_T_alloc : a.T;
    p.y_T_alloc = a.y_T_alloc ? a.y_T_alloc : p.T_out;
    if (a.residual && p.S != 1) return cudaErrorInvalidValue;
    p.gn_partials = a.gn_partials;
    p.gn_groups = a.gn_groups;
    p.gn_cpg = a.gn_groups ? p.C_d2s / a.gn_groups : 0;
    if (a.gn_partials && (p.C_d2s % 32 != 0 || a.out_ncthw || (p.gn_cpg < 32 ? 32 % p.gn_cpg : p.gn_cpg % 32) != 0))
      return cudaErrorInvalidValue;
    const uint64_t C = a.C_in_pad;
    const uint64_t eb = p.fp8 ? 1 : p.tf32 ? 4 : 2;  // bytes per operand element
    const uint64_t xTa = a.x_T_alloc ? a.x_T_alloc : a.T_in;
    uint64_t dims[5] = {C, (uint64_t)a.W, (uint64_t)a.H, (uint64_t)a.T_in, (uint64_t)a.B};
    uint64_t strides[4] = {C * eb, C * eb * a.W, C * eb * a.W * a.H, C * eb * a.W * a.H * xTa};
    uint32_t box[5] = {(uint32_t)p.kc, (uint32_t)p.cols_t, (uint32_t)p.rows_t, 1u, 1u};
    if (p.halo) {
      box[1] = static_cast<uint32_t>(p.cols_t + 2);
      box[2] = static_cast<uint32_t>(p.rows_t + 2);
    }
    if (!make_map(&tmA, a.x, 5, dims, strides, box, static_cast<int>(eb))) return cudaErrorInvalidValue;
    if (p.tf32 && !make_map(&tmA2, a.x_lo, 5, dims, strides, box, 4)) return cudaErrorInvalidValue;
    const uint64_t K = 27ull * C;
    uint64_t wd[2] = {K, (uint64_t)a.N_pad};
    uint64_t ws[1] = {K * eb};
    uint32_t wb[2] = {(uint32_t)p.kc, (uint32_t)(want_pair ? p.BN / 2 : p.BN)};
    if (p.halo == 2) {  // [3 kt][kTapRows][C]: one kTapRows-row tile per (kt, channel chunk)
      wd[0] = C;
      wd[1] = 3ull * kTapRows;
      ws[0] = C * eb;
      wb[1] = static_cast<uint32_t>(kTapRows);
    }
    if (p.tf32) wd[1] = 2ull * a.N_pad;  // high parts, then remainders
    if (!make_map(&tmB, a.w, 2, wd, ws, wb, static_cast<int>(eb))) return cudaErrorInvalidValue;
    n_blocks = static_cast<long long>(a.B) * a.T * p.n_trows * p.n_tcols * p.n_ntiles;
  } else {
    p.M = a.M; p.K = a.K; p.batch = a.batch; p.stride_d = a.stride_d; p.alpha = a.alpha;
    p.ldd = a.ldd ? a.ldd : a.N_real;
    if (a.K % 64 != 0) return cudaErrorInvalidValue;
    p.m_tiles_per_batch = (a.M + kBlockM * p.msub - 1) / (kBlockM * p.msub);
    p.num_kb = a.K / kBlockK;
    p.S = 1; p.C_d2s = a.N_real; p.d2s_t = p.d2s_h = p.d2s_w = 1;
    const int64_t sa = a.batch > 1 ? a.stride_a : static_cast<int64_t>(a.M) * a.K;
    const int64_t sb = a.batch > 1 ? a.stride_b : static_cast<int64_t>(a.N_real) * a.K;
    if (sa % 8 || sb % 8 || a.K % 8) return cudaErrorInvalidValue;
    uint64_t ad[3] = {(uint64_t)a.K, (uint64_t)a.M, (uint64_t)a.batch};
    uint64_t as[2] = {(uint64_t)a.K * 2, (uint64_t)sa * 2};
    uint32_t ab[3] = {64u, static_cast<uint32_t>(kBlockM * p.msub), 1u};
    if (!make_map(&tmA, a.x, 3, ad, as, ab)) return cudaErrorInvalidValue;
    // B rows beyond N_real read as zeros (never the next batch item's rows)
    uint64_t bd[3] = {(uint64_t)a.K, (uint64_t)a.N_real, (uint64_t)a.batch};
    uint64_t bs[2] = {(uint64_t)a.K * 2, (uint64_t)sb * 2};
    uint32_t bb[3] = {64u, (uint32_t)(want_pair ? p.BN / 2 : p.BN), 1u};
    if (!make_map(&tmB, a.w, 3, bd, bs, bb)) return cudaErrorInvalidValue;
    n_blocks = static_cast<long long>(a.batch) * p.m_tiles_per_batch * p.n_ntiles;
  }
  if (n_blocks <= 0) return cudaSuccess;
  if (n_blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  p.n_tiles = static_cast<int>(n_blocks);
  p.y2 = a.y2;
  p.y2_T_alloc = a.y2_T_alloc ? a.y2_T_alloc : p.T_out;
  p.y2_fp8 = a.y2_fp8;
  if (a.y2 && (p.out_ncthw || p.C_d2s % 32 != 0)) return cudaErrorInvalidValue;
  int dev = 0;
  {
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  }
  const size_t smem = 1024 + static_cast<size_t>(p.scratch_off) + scratch_bytes;
  if (smem > 227u * 1024u) return cudaErrorInvalidValue;
  int n_sm = 0;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevLaunch& dl = g_dev[dev];
    if (!dl.ready) {
      if (cudaDeviceGetAttribute(&dl.n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || dl.n_sm <= 0)
        dl.n_sm = 148;
      for (auto* k : {conv_tc_kernel<false, 0>, conv_tc_kernel<true, 0>, conv_tc_kernel<false, 1>,
                      conv_tc_kernel<true, 1>, conv_tc_kernel<false, 2>, conv_tc_kernel<true, 2>}) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
      }
      dl.ready = true;
    }
    n_sm = dl.n_sm;
  }
  p.n_mtiles = static_cast<int>(n_blocks / p.n_ntiles);
  p.pair = want_pair ? 1 : 0;
  {
    // N tiles per chunk: as many as keep the chunk's weights within ~48 MB of L2
    const double w_tile =
        static_cast<double>(p.BN) * (a.mode == 0 ? 27.0 * a.C_in_pad : static_cast<double>(a.K)) *
        (p.fp8 ? 1.0 : p.tf32 ? 8.0 : 2.0);
    int npc = p.n_ntiles;
    if (a.mode == 0) {
      npc = 1;
      for (int d = 1; d <= p.n_ntiles; ++d)
        if (p.n_ntiles % d == 0 && d * w_tile <= 48.0 * 1024 * 1024) npc = d;
    }
    p.npc = npc;
  }
  if (!p.pair) {
    p.seq_count = p.n_tiles;
    const long long grid = std::min<long long>(n_blocks, n_sm);
    const unsigned g = static_cast<unsigned>(grid);
    if (p.fp8) conv_tc_kernel<false, 1><<<g, kThreads, smem, stream>>>(tmA, tmB, tmA2, p);
    else if (p.tf32) conv_tc_kernel<false, 2><<<g, kThreads, smem, stream>>>(tmA, tmB, tmA2, p);
    else conv_tc_kernel<false, 0><<<g, kThreads, smem, stream>>>(tmA, tmB, tmA2, p);
    return cudaGetLastError();
  }
  p.seq_count = (p.n_mtiles + 1) / 2 * p.n_ntiles;
  auto* kern = p.fp8 ? conv_tc_kernel<true, 1> : p.tf32 ? conv_tc_kernel<true, 2> : conv_tc_kernel<true, 0>;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int max_clusters = 0;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevLaunch& dl = g_dev[dev];
    if (dl.max_clusters <= 0 || dl.max_clusters_smem != smem ||
        dl.max_clusters_kern != reinterpret_cast<const void*>(kern)) {
      cfg.gridDim = dim3(2 * (n_sm / 2));
      int mc = 0;
      if (cudaOccupancyMaxActiveClusters(&mc, kern, &cfg) != cudaSuccess || mc <= 0) mc = n_sm / 2;
      dl.max_clusters = mc;
      dl.max_clusters_smem = smem;
      dl.max_clusters_kern = reinterpret_cast<const void*>(kern);
    }
    max_clusters = dl.max_clusters;
  }
  const long long clusters = std::min<long long>(p.seq_count, max_clusters);
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmA2, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace vae
