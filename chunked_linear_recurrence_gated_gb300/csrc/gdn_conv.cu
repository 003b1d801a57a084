// Causal short convolution with carried boundary state (include/gdn_conv.h):
// the auxiliary local-convolution states a chunk carries besides S_in / S_out
// (StateFlow review, "What carries the argument"; footnote to its Section 3.1
// as quoted in the referee report, major comment 1), read as the causal
// depthwise convolution of a Gated DeltaNet layer's q / k / v projections.
//
// HBM-bound: every thread owns 4 channels over a run of tokens, keeps the last
// W - 1 inputs in registers as a sliding window, and reads each input row once
// (plus a W - 1 row halo per tile), with enough loads in flight to cover the
// memory latency: the forward keeps two groups of G_F tokens outstanding, the
// backward loads LA_B tokens ahead. Consecutive threads take consecutive
// channel groups, so every warp load is one contiguous 256-byte (bf16) or
// 512-byte (fp32) segment.
#include <stdint.h>

#include <algorithm>

#include <type_traits>

#include "../../include/gdn_conv.h"
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int CONV_TT_MIN = 64;  // shortest forward tile (the launch sizes tiles to fill the GPU once)
constexpr int CONV_TTB = 256;  // shortest backward tile (one dw / db partial each)
constexpr int CONV_NT = 128;   // threads per block

constexpr int CV = 4;          // channels per thread
constexpr int G_F = 8;         // tokens per load group, two groups in flight (forward)
constexpr int LA_B = 8;        // tokens loaded ahead of their use in the backward's interior

// 4 channels: 16 bytes of fp32 or 8 bytes of bf16
__device__ __forceinline__ void ld_vec(const float* p, float* v) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  v[0] = a.x;
  v[1] = a.y;
  v[2] = a.z;
  v[3] = a.w;
}
__device__ __forceinline__ void st_vec(float* p, const float* v) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void ld_vec(const __nv_bfloat16* p, float* v) {
  const uint2 a = *reinterpret_cast<const uint2*>(p);
  v[0] = __uint_as_float(a.x << 16);
  v[1] = __uint_as_float(a.x & 0xffff0000u);
  v[2] = __uint_as_float(a.y << 16);
  v[3] = __uint_as_float(a.y & 0xffff0000u);
}
__device__ __forceinline__ void st_vec(__nv_bfloat16* p, const float* v) {
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]);
  const __nv_bfloat162 h1 = __floats2bfloat162_rn(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) =
      make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
}
// 4 channels as loaded (unconverted): float4 for fp32, uint2 for bf16
template <typename T>
using RawVec = typename std::conditional<std::is_same<T, float>::value, float4, uint2>::type;
template <typename T>
__device__ __forceinline__ RawVec<T> ld_raw(const T* p) {
  return *reinterpret_cast<const RawVec<T>*>(p);
}
__device__ __forceinline__ void cvt_raw(const float4& a, float* v) {
  v[0] = a.x;
  v[1] = a.y;
  v[2] = a.z;
  v[3] = a.w;
}
__device__ __forceinline__ void cvt_raw(const uint2& a, float* v) {
  v[0] = __uint_as_float(a.x << 16);
  v[1] = __uint_as_float(a.x & 0xffff0000u);
  v[2] = __uint_as_float(a.y << 16);
  v[3] = __uint_as_float(a.y & 0xffff0000u);
}
__device__ __forceinline__ void zero_vec(float* v) {
#pragma unroll
  for (int i = 0; i < CV; ++i) v[i] = 0.f;
}

__device__ __forceinline__ float act_fwd(float z, int act) {
  return act ? __fdividef(z, 1.f + __expf(-z)) : z;
}
// d act / dz
__device__ __forceinline__ float act_grad(float z, int act) {
  if (!act) return 1.f;
  const float s = __fdividef(1.f, 1.f + __expf(-z));
  return s * (1.f + z * (1.f - s));
}

// x_ext[s + W - 1] for x index s: x[s] (0 <= s < T), the incoming state for
// -(W-1) <= s < 0 (zero when absent), zero elsewhere.
template <typename T, int W>
__device__ __forceinline__ void ld_ext(const T* xrow0, const T* srow0, int s, int Tn, int C,
                                       float* v) {
  if (s >= 0 && s < Tn)
    ld_vec(xrow0 + (size_t)s * C, v);
  else if (s < 0 && s >= -(W - 1) && srow0)
    ld_vec(srow0 + (size_t)(s + W - 1) * C, v);
  else
    zero_vec(v);
}

// One tile of tt tokens per block row; the launch picks tt (a multiple of
// 2 G_F) so that the tiles of a call fill the GPU's resident blocks once.
template <typename T, int W>
__global__ void __launch_bounds__(CONV_NT) k_conv_fwd(int Tn, int tt, int C, int act, const T* __restrict__ x,
                                                      const float* __restrict__ w,
                                                      const float* __restrict__ b,
                                                      const T* __restrict__ s_in, T* __restrict__ y,
                                                      T* __restrict__ s_out) {
  const int c0 = (blockIdx.y * CONV_NT + threadIdx.x) * CV;
  if (c0 >= C) return;
  const int bb = blockIdx.z;
  const T* xr = x + (size_t)bb * Tn * C + c0;
  const T* sr = s_in ? s_in + (size_t)bb * (W - 1) * C + c0 : nullptr;
  float wr[CV][W], br[CV];
#pragma unroll
  for (int v = 0; v < CV; ++v) {
#pragma unroll
    for (int j = 0; j < W; ++j) wr[v][j] = w[(size_t)(c0 + v) * W + j];
    br[v] = b ? b[c0 + v] : 0.f;
  }
  const int t0 = blockIdx.x * tt, t1 = min(t0 + tt, Tn);
  float xw[W - 1][CV];  // x[t - W + 1 .. t - 1]
#pragma unroll
  for (int j = 0; j < W - 1; ++j) ld_ext<T, W>(xr, sr, t0 - (W - 1) + j, Tn, C, xw[j]);
  T* yr = y + (size_t)bb * Tn * C + c0;
  // two groups of G tokens in flight: the next group's loads are issued
  // before the current group is computed
  RawVec<T> xa[G_F], xb[G_F];  // kept as loaded; converted when used
  const bool full = t1 - t0 == tt;
  auto load_group = [&](RawVec<T>* xg, int t) {
#pragma unroll
    for (int u = 0; u < G_F; ++u)
      if (full || t + u < t1) xg[u] = ld_raw(xr + (size_t)(t + u) * C);
  };
  auto compute_group = [&](const RawVec<T>* xg, int t) {
#pragma unroll
    for (int u = 0; u < G_F; ++u) {
      float xc[CV];
      if (full || t + u < t1) {
        cvt_raw(xg[u], xc);
        float out[CV];
#pragma unroll
        for (int v = 0; v < CV; ++v) {
          float z = br[v];
#pragma unroll
          for (int j = 0; j < W - 1; ++j) z = fmaf(wr[v][j], xw[j][v], z);
          z = fmaf(wr[v][W - 1], xc[v], z);
          out[v] = act_fwd(z, act);
        }
        st_vec(yr + (size_t)(t + u) * C, out);
      } else {
        zero_vec(xc);
      }
#pragma unroll
      for (int j = 0; j < W - 2; ++j)
#pragma unroll
        for (int v = 0; v < CV; ++v) xw[j][v] = xw[j + 1][v];
#pragma unroll
      for (int v = 0; v < CV; ++v) xw[W - 2][v] = xc[v];
    }
  };
  load_group(xa, t0);
  for (int t = t0; t < t1; t += 2 * G_F) {
    if (t + G_F < t1) load_group(xb, t + G_F);
    compute_group(xa, t);
    if (t + 2 * G_F < t1) load_group(xa, t + 2 * G_F);
    if (t + G_F < t1) compute_group(xb, t + G_F);
  }
  if (s_out && blockIdx.x == gridDim.x - 1) {
    // state_out[i] = x_ext[T + i]
    T* so = s_out + (size_t)bb * (W - 1) * C + c0;
#pragma unroll
    for (int i = 0; i < W - 1; ++i) {
      float v[CV];
      ld_ext<T, W>(xr, sr, Tn + i - (W - 1), Tn, C, v);
      st_vec(so + (size_t)i * C, v);
    }
  }
}

// One tile of ttb tokens per block row: g = dy * act'(z) with z
// recomputed, dx (lagging W - 1 tokens behind g), this tile's dw / db partial
// sums, and (tile 0) dstate_in; the last W - 1 positions of x_ext also
// receive dstate_out.
template <typename T, int W>
__global__ void __launch_bounds__(CONV_NT) k_conv_bwd(int Tn, int ttb, int C, int act, const T* __restrict__ x,
                                                      const float* __restrict__ w,
                                                      const float* __restrict__ b,
                                                      const T* __restrict__ s_in,
                                                      const T* __restrict__ dy,
                                                      const T* __restrict__ ds_out,
                                                      T* __restrict__ dx, T* __restrict__ ds_in,
                                                      float* __restrict__ part) {
  const int c0 = (blockIdx.y * CONV_NT + threadIdx.x) * CV;
  if (c0 >= C) return;
  const int bb = blockIdx.z, tile = blockIdx.x, ntiles = gridDim.x;
  const T* xr = x + (size_t)bb * Tn * C + c0;
  const T* sr = s_in ? s_in + (size_t)bb * (W - 1) * C + c0 : nullptr;
  const T* gr = dy + (size_t)bb * Tn * C + c0;
  const T* dsr = ds_out ? ds_out + (size_t)bb * (W - 1) * C + c0 : nullptr;
  T* dxr = dx + (size_t)bb * Tn * C + c0;
  T* dsi = ds_in ? ds_in + (size_t)bb * (W - 1) * C + c0 : nullptr;
  float wr[CV][W], br[CV];
#pragma unroll
  for (int v = 0; v < CV; ++v) {
#pragma unroll
    for (int j = 0; j < W; ++j) wr[v][j] = w[(size_t)(c0 + v) * W + j];
    br[v] = b ? b[c0 + v] : 0.f;
  }
  const int s0 = tile * ttb, s1 = min(s0 + ttb, Tn);
  const int e0 = tile == 0 ? -(W - 1) : s0;  // first emitted index (tile 0 also emits dstate_in)
  const int tb = e0, te = s1 + (W - 1);
  float xw[W - 1][CV], gw[W - 1][CV], pw[CV][W], pb[CV];
#pragma unroll
  for (int j = 0; j < W - 1; ++j) {
    ld_ext<T, W>(xr, sr, tb - (W - 1) + j, Tn, C, xw[j]);
    zero_vec(gw[j]);
  }
  zero_vec(pb);
#pragma unroll
  for (int v = 0; v < CV; ++v)
#pragma unroll
    for (int j = 0; j < W; ++j) pw[v][j] = 0.f;
  // One token t: g[t] (zero outside [0, T)), this tile's partial sums, and
  // dx_ext at x index t - (W - 1). GENERAL handles the tile's edges; the
  // interior (g computed, owned, emitted into dx, no dstate_out) skips the tests.
  auto step = [&](int t, const float* xc, const float* dd, auto general) {
    constexpr bool GEN = decltype(general)::value;
    float g[CV];
    if (!GEN || (t >= 0 && t < Tn)) {
      const bool own = !GEN || (t >= s0 && t < s1);
#pragma unroll
      for (int v = 0; v < CV; ++v) {
        float z = br[v];
#pragma unroll
        for (int j = 0; j < W - 1; ++j) z = fmaf(wr[v][j], xw[j][v], z);
        z = fmaf(wr[v][W - 1], xc[v], z);
        g[v] = dd[v] * act_grad(z, act);
        if (own) {
          pb[v] += g[v];
#pragma unroll
          for (int j = 0; j < W - 1; ++j) pw[v][j] = fmaf(g[v], xw[j][v], pw[v][j]);
          pw[v][W - 1] = fmaf(g[v], xc[v], pw[v][W - 1]);
        }
      }
    } else {
      zero_vec(g);
    }
    const int s = t - (W - 1);
    if (!GEN || (s >= e0 && s < s1)) {
      float o[CV];
#pragma unroll
      for (int v = 0; v < CV; ++v) {
        float a = wr[v][0] * g[v];
#pragma unroll
        for (int j = 1; j < W; ++j) a = fmaf(wr[v][j], gw[W - 1 - j][v], a);
        o[v] = a;
      }
      const int p = s + W - 1;  // index in x_ext
      if (GEN && dsr && p >= Tn) {
        float e[CV];
        ld_vec(dsr + (size_t)(p - Tn) * C, e);
#pragma unroll
        for (int v = 0; v < CV; ++v) o[v] += e[v];
      }
      if (!GEN || s >= 0)
        st_vec(dxr + (size_t)s * C, o);
      else if (dsi)
        st_vec(dsi + (size_t)p * C, o);
    }
#pragma unroll
    for (int j = 0; j < W - 2; ++j)
#pragma unroll
      for (int v = 0; v < CV; ++v) {
        xw[j][v] = xw[j + 1][v];
        gw[j][v] = gw[j + 1][v];
      }
#pragma unroll
    for (int v = 0; v < CV; ++v) {
      xw[W - 2][v] = xc[v];
      gw[W - 2][v] = g[v];
    }
  };
  auto general_range = [&](int ta, int tz) {
    for (int t = ta; t < tz; ++t) {
      float xc[CV], dd[CV];
      ld_ext<T, W>(xr, sr, t, Tn, C, xc);
      if (t >= 0 && t < Tn)
        ld_vec(gr + (size_t)t * C, dd);
      else
        zero_vec(dd);
      step(t, xc, dd, std::true_type());
    }
  };
  // interior: 0 <= t - (W - 1), s0 <= t - (W - 1), t < s1 (<= T)
  const int m0 = max(tb + (W - 1), W - 1), m1 = max(m0, s1);
  general_range(tb, min(m0, te));
  int t = m0;
  for (; t + LA_B <= m1; t += LA_B) {
    float xc[LA_B][CV], dd[LA_B][CV];
#pragma unroll
    for (int u = 0; u < LA_B; ++u) {
      ld_vec(xr + (size_t)(t + u) * C, xc[u]);
      ld_vec(gr + (size_t)(t + u) * C, dd[u]);
    }
#pragma unroll
    for (int u = 0; u < LA_B; ++u) step(t + u, xc[u], dd[u], std::false_type());
  }
  for (; t < m1; ++t) {
    float xc[CV], dd[CV];
    ld_vec(xr + (size_t)t * C, xc);
    ld_vec(gr + (size_t)t * C, dd);
    step(t, xc, dd, std::false_type());
  }
  general_range(max(m1, min(m0, te)), te);
  float* pp = part + (((size_t)bb * ntiles + tile) * C + c0) * (W + 1);
#pragma unroll
  for (int v = 0; v < CV; ++v) {
#pragma unroll
    for (int j = 0; j < W; ++j) pp[v * (W + 1) + j] = pw[v][j];
    pp[v * (W + 1) + W] = pb[v];
  }
}

// dw[c][j] (j < W) and db[c] (j == W): the partials of every (sequence, tile)
// summed in a fixed order.
__global__ void k_conv_reduce(int nparts, int C, int W, const float* __restrict__ part,
                              float* __restrict__ dw, float* __restrict__ db) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int n = C * (W + 1);
  if (i >= n) return;
  float a = 0.f;
  for (int k = 0; k < nparts; ++k) a += part[(size_t)k * n + i];
  const int c = i / (W + 1), j = i % (W + 1);
  if (j < W)
    dw[(size_t)c * W + j] = a;
  else if (db)
    db[c] = a;
}

// ------------------------------------------------------------------ host side
struct ConvPlan {
  int B, T, C, W, act, vec;
  bool bf16;
  int ntiles_f, ntiles_b, cblocks;
};

gdn_status plan(const gdn_conv_shape* s, ConvPlan* p) {
  if (!s) return GDN_ERR_INVALID_ARG;
  if (s->B < 1 || s->B > 65535 || s->T < 0 || s->C < 1) return GDN_ERR_INVALID_ARG;
  if (s->act != GDN_CONV_ACT_NONE && s->act != GDN_CONV_ACT_SILU) return GDN_ERR_INVALID_ARG;
  if (s->dtype != GDN_DTYPE_F32 && s->dtype != GDN_DTYPE_BF16) return GDN_ERR_UNSUPPORTED;
  if (s->W < 2 || s->W > 8) return GDN_ERR_UNSUPPORTED;
  p->bf16 = s->dtype == GDN_DTYPE_BF16;
  p->vec = CV;
  if (s->C % CV) return GDN_ERR_UNSUPPORTED;
  if ((long long)s->B * s->T > (1ll << 31) - 1 || (long long)s->T * s->C > (1ll << 40))
    return GDN_ERR_INVALID_ARG;
  p->B = s->B;
  p->T = s->T;
  p->C = s->C;
  p->W = s->W;
  p->act = s->act;
  p->ntiles_f = s->T > 0 ? (s->T + CONV_TT_MIN - 1) / CONV_TT_MIN : 1;  // at most
  p->ntiles_b = s->T > 0 ? (s->T + CONV_TTB - 1) / CONV_TTB : 1;
  const int groups = s->C / p->vec;
  p->cblocks = (groups + CONV_NT - 1) / CONV_NT;
  if (p->ntiles_f > 0x7fffffff / 2 || p->cblocks > 65535) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

size_t ws_bytes(const ConvPlan& p) {
  const size_t n = (size_t)p.B * p.ntiles_b * p.C * (p.W + 1) * sizeof(float);
  return (n + 255) & ~(size_t)255;
}

bool al(const void* q, size_t a) { return q == nullptr || ((uintptr_t)q % a) == 0; }

template <typename T, int W>
cudaError_t launch_fwd(const ConvPlan& p, const void* x, const float* w, const float* b,
                       const void* s_in, void* y, void* s_out, cudaStream_t st) {
  // tiles per block row: as many as the GPU holds resident blocks (divided
  // over the block rows), so the launch runs in one wave; at least CONV_TT_MIN
  // tokens per tile. The forward has no cross-tile sums, so the tiling does
  // not change any result.
  int dev = 0, sms = 0, occ = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) || (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) ||
      (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_conv_fwd<T, W>, CONV_NT, 0)))
    return e;
  const long long rows = (long long)p.cblocks * p.B;
  const long long per_row = std::max<long long>(1, (long long)std::max(occ, 1) * sms / rows);
  long long tt = (p.T + per_row - 1) / per_row;
  tt = std::max<long long>(CONV_TT_MIN, (tt + 2 * G_F - 1) / (2 * G_F) * (2 * G_F));
  const int ntiles = p.T > 0 ? (int)((p.T + tt - 1) / tt) : 1;
  prof_mark(st, "conv_fwd");
  k_conv_fwd<T, W><<<dim3(ntiles, p.cblocks, p.B), CONV_NT, 0, st>>>(
      p.T, (int)tt, p.C, p.act, (const T*)x, w, b, (const T*)s_in, (T*)y, (T*)s_out);
  prof_mark(st, nullptr);
  return cudaGetLastError();
}

template <typename T, int W>
cudaError_t launch_bwd(const ConvPlan& p, const void* x, const float* w, const float* b,
                       const void* s_in, const void* dy, const void* ds_out, void* dx, float* dw,
                       float* db, void* ds_in, float* part, cudaStream_t st) {
  // tiles as for the forward (one wave), at least CONV_TTB tokens each, so the
  // partial sums fit the workspace sized for CONV_TTB-token tiles
  int dev = 0, sms = 0, occ = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) || (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) ||
      (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_conv_bwd<T, W>, CONV_NT, 0)))
    return e;
  const long long rows = (long long)p.cblocks * p.B;
  const long long per_row = std::max<long long>(1, (long long)std::max(occ, 1) * sms / rows);
  long long tt = (p.T + per_row - 1) / per_row;
  tt = std::max<long long>(CONV_TTB, (tt + LA_B - 1) / LA_B * LA_B);
  const int ntiles = p.T > 0 ? (int)((p.T + tt - 1) / tt) : 1;
  prof_mark(st, "conv_bwd");
  k_conv_bwd<T, W><<<dim3(ntiles, p.cblocks, p.B), CONV_NT, 0, st>>>(
      p.T, (int)tt, p.C, p.act, (const T*)x, w, b, (const T*)s_in, (const T*)dy, (const T*)ds_out,
      (T*)dx, (T*)ds_in, part);
  if ((e = cudaGetLastError())) return e;
  prof_mark(st, "conv_reduce");
  const int n = p.C * (p.W + 1);
  k_conv_reduce<<<(n + 255) / 256, 256, 0, st>>>(p.B * ntiles, p.C, p.W, part, dw, db);
  prof_mark(st, nullptr);
  return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_fwd(const ConvPlan& p, const void* x, const float* w, const float* b,
                         const void* s_in, void* y, void* s_out, cudaStream_t st) {
  switch (p.W) {
    case 2: return launch_fwd<T, 2>(p, x, w, b, s_in, y, s_out, st);
    case 3: return launch_fwd<T, 3>(p, x, w, b, s_in, y, s_out, st);
    case 4: return launch_fwd<T, 4>(p, x, w, b, s_in, y, s_out, st);
    case 5: return launch_fwd<T, 5>(p, x, w, b, s_in, y, s_out, st);
    case 6: return launch_fwd<T, 6>(p, x, w, b, s_in, y, s_out, st);
    case 7: return launch_fwd<T, 7>(p, x, w, b, s_in, y, s_out, st);
    default: return launch_fwd<T, 8>(p, x, w, b, s_in, y, s_out, st);
  }
}

template <typename T>
cudaError_t dispatch_bwd(const ConvPlan& p, const void* x, const float* w, const float* b,
                         const void* s_in, const void* dy, const void* ds_out, void* dx, float* dw,
                         float* db, void* ds_in, float* part, cudaStream_t st) {
  switch (p.W) {
    case 2: return launch_bwd<T, 2>(p, x, w, b, s_in, dy, ds_out, dx, dw, db, ds_in, part, st);
    case 3: return launch_bwd<T, 3>(p, x, w, b, s_in, dy, ds_out, dx, dw, db, ds_in, part, st);
    case 4: return launch_bwd<T, 4>(p, x, w, b, s_in, dy, ds_out, dx, dw, db, ds_in, part, st);
    case 5: return launch_bwd<T, 5>(p, x, w, b, s_in, dy, ds_out, dx, dw, db, ds_in, part, st);
    case 6: return launch_bwd<T, 6>(p, x, w, b, s_in, dy, ds_out, dx, dw, db, ds_in, part, st);
    case 7: return launch_bwd<T, 7>(p, x, w, b, s_in, dy, ds_out, dx, dw, db, ds_in, part, st);
    default: return launch_bwd<T, 8>(p, x, w, b, s_in, dy, ds_out, dx, dw, db, ds_in, part, st);
  }
}

}  // namespace
}  // namespace gdn

extern "C" {

size_t gdn_conv_workspace_bytes(const gdn_conv_shape* shape) {
  gdn::ConvPlan p;
  if (gdn::plan(shape, &p) != GDN_OK) return 0;
  return gdn::ws_bytes(p);
}

gdn_status gdn_conv_fwd(const gdn_conv_shape* shape, const void* x, const float* w,
                        const float* b, const void* state_in, void* y, void* state_out,
                        void* stream) {
  using namespace gdn;
  ConvPlan p;
  gdn_status s = plan(shape, &p);
  if (s != GDN_OK) return s;
  const bool any = p.T > 0;
  if ((any && (!x || !y)) || !w) return GDN_ERR_INVALID_ARG;
  if (!al(x, 16) || !al(y, 16) || !al(state_in, 16) || !al(state_out, 16) || !al(w, 4) ||
      !al(b, 4))
    return GDN_ERR_INVALID_ARG;
  if (state_out && state_out == state_in) return GDN_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const cudaError_t e = p.bf16 ? dispatch_fwd<__nv_bfloat16>(p, x, w, b, state_in, y, state_out, st)
                               : dispatch_fwd<float>(p, x, w, b, state_in, y, state_out, st);
  return e ? GDN_ERR_CUDA : GDN_OK;
}

gdn_status gdn_conv_bwd(const gdn_conv_shape* shape, const void* x, const float* w,
                        const float* b, const void* state_in, const void* dy,
                        const void* dstate_out, void* dx, float* dw, float* db, void* dstate_in,
                        void* workspace, size_t workspace_bytes, void* stream) {
  using namespace gdn;
  ConvPlan p;
  gdn_status s = plan(shape, &p);
  if (s != GDN_OK) return s;
  const bool any = p.T > 0;
  if ((any && (!x || !dy || !dx)) || !w || !dw || (db && !b)) return GDN_ERR_INVALID_ARG;
  if (!al(x, 16) || !al(dy, 16) || !al(dx, 16) || !al(state_in, 16) || !al(dstate_out, 16) ||
      !al(dstate_in, 16) || !al(w, 4) || !al(b, 4) || !al(dw, 4) || !al(db, 4))
    return GDN_ERR_INVALID_ARG;
  if (!workspace || !al(workspace, 256) || workspace_bytes < ws_bytes(p)) return GDN_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  float* part = (float*)workspace;
  const cudaError_t e =
      p.bf16 ? dispatch_bwd<__nv_bfloat16>(p, x, w, b, state_in, dy, dstate_out, dx, dw, db,
                                           dstate_in, part, st)
             : dispatch_bwd<float>(p, x, w, b, state_in, dy, dstate_out, dx, dw, db, dstate_in,
                                   part, st);
  return e ? GDN_ERR_CUDA : GDN_OK;
}

}  // extern "C"
