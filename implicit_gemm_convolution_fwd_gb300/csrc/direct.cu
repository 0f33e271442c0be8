// FP32 FFMA direct convolution for small reductions (tiny C_in or kernel),
// where a tensor-core tile would be mostly padding.
//
// The sum is the one written out on the l1_p60 page (turn 1, generic kernel)
// and the l1_p76 page (turn 2): y[n,o,p] = b[o] + sum_{c,k} w[o,c,k] *
// x[n,c,p*stride + k*dilation - pad], taps outside the input reading zero.
//
// Work split: one thread owns R consecutive output positions along W of one
// (n, od, oh) row and CO output channels (a register tile of CO x R
// accumulators), so every weight read from shared memory feeds R FMAs and
// every input value feeds CO FMAs.  A CTA shares one channel block; its
// weights for a chunk of input channels are staged in shared memory and read
// as warp-wide broadcasts.  Input values come through the read-only cache:
// neighbouring threads read overlapping windows of the same rows.
#include <cuda_runtime.h>
#include <stdint.h>

#include "conv_internal.cuh"
#include "debug_check.cuh"

namespace convfwd {
namespace {

constexpr int kThreads = 128;
constexpr int kCO = 8;             // output channels per thread (and per CTA)
constexpr int kR = 4;              // output positions along W per thread
constexpr int kSmemFloats = 8192;  // 32 KB weight chunk

struct DirectParams {
  const float *__restrict__ x;
  const float *__restrict__ w;
  const float *__restrict__ bias;
  float *__restrict__ y;
  Geom g;
  int64_t items;  // N * OD * OH * ceil(OW / R)
  int owg;        // ceil(OW / R)
  int cchunk;     // input channels per weight chunk
  int kblocks;    // channel blocks of kCO per group: ceil(K / kCO)
  int64_t x_elems, w_elems, y_elems;  // extents the debug build's device checks use
};

__global__ void __launch_bounds__(kThreads) direct_ffma_kernel(const DirectParams p) {
  __shared__ __align__(16) float ws[kSmemFloats];  // [cc][tap][kCO]
  const Geom &g = p.g;
  const int taps = g.KD * g.KH * g.KW;
  // blockIdx.y = (group, channel block within the group); o0 is the block's
  // first output channel within its group
  const int grp = blockIdx.y / p.kblocks;
  const int o0 = (blockIdx.y - grp * p.kblocks) * kCO;
  const int64_t ob = (int64_t)grp * g.K;  // the group's first output channel in y and w

  const int64_t item = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const bool active = item < p.items;
  int64_t rest = active ? item : 0;
  const int owg = (int)(rest % p.owg);
  rest /= p.owg;
  const int oh = (int)(rest % g.OH);
  rest /= g.OH;
  const int od = (int)(rest % g.OD);
  const int64_t n = rest / g.OD;
  const int ow0 = owg * kR;

  float acc[kCO][kR];
#pragma unroll
  for (int o = 0; o < kCO; ++o)
#pragma unroll
    for (int r = 0; r < kR; ++r) acc[o][r] = 0.f;

  const int64_t HW = (int64_t)g.H * g.W;
  for (int64_t c0 = 0; c0 < g.C; c0 += p.cchunk) {
    const int cc_n = (int)((g.C - c0) < p.cchunk ? (g.C - c0) : p.cchunk);
    __syncthreads();
    // stage weights w[o0+o][c0+cc][tap] -> ws[(cc*taps + tap)*kCO + o]
    for (int i = threadIdx.x; i < cc_n * taps * kCO; i += kThreads) {
      const int o = i % kCO;
      const int ct = i / kCO;  // cc*taps + tap
      const int64_t og = o0 + o;
      const int64_t wi = ((ob + og) * g.C + c0) * taps + ct;
      ws[i] = (og < g.K && CONV_DBG_OK(wi, p.w_elems, kStatusBoundsW)) ? p.w[wi] : 0.f;
    }
    __syncthreads();
    if (!active) continue;
    for (int cc = 0; cc < cc_n; ++cc) {
      const float *xc = p.x + n * g.x_batch_stride() + ((grp * g.C + c0 + cc) * g.D) * HW;
      for (int kd = 0; kd < g.KD; ++kd) {
        const int id = od * g.SD + kd * g.DD - g.PD;
        if ((unsigned)id >= (unsigned)g.D) continue;
        for (int kh = 0; kh < g.KH; ++kh) {
          const int ih = oh * g.SH + kh * g.DH - g.PH;
          if ((unsigned)ih >= (unsigned)g.H) continue;
          const float *row = xc + (int64_t)id * HW + (int64_t)ih * g.W;
          const float *wt = ws + ((cc * g.KD + kd) * g.KH + kh) * g.KW * kCO;
          for (int kw = 0; kw < g.KW; ++kw) {
            float xv[kR];
#pragma unroll
            for (int r = 0; r < kR; ++r) {
              const int iw = (ow0 + r) * g.SW + kw * g.DW - g.PW;
              xv[r] = ((unsigned)iw < (unsigned)g.W && CONV_DBG_OK(row + iw - p.x, p.x_elems, kStatusBoundsX))
                          ? __ldg(row + iw)
                          : 0.f;
            }
            const float4 wa = *reinterpret_cast<const float4 *>(wt + kw * kCO);
            const float4 wb = *reinterpret_cast<const float4 *>(wt + kw * kCO + 4);
            const float wv[kCO] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int o = 0; o < kCO; ++o)
#pragma unroll
              for (int r = 0; r < kR; ++r) acc[o][r] = fmaf(wv[o], xv[r], acc[o][r]);
          }
        }
      }
    }
  }
  if (!active) return;
  const int64_t osp = (int64_t)g.OD * g.OH * g.OW;
#pragma unroll
  for (int o = 0; o < kCO; ++o) {
    const int64_t og = o0 + o;
    if (og >= g.K) break;
    const float b = p.bias ? __ldg(p.bias + ob + og) : 0.f;
    float *yo = p.y + n * g.y_batch_stride() + (ob + og) * osp + ((int64_t)od * g.OH + oh) * g.OW;
#pragma unroll
    for (int r = 0; r < kR; ++r)
      if (ow0 + r < g.OW && CONV_DBG_OK(yo + ow0 + r - p.y, p.y_elems, kStatusBoundsY)) yo[ow0 + r] = acc[o][r] + b;
  }
}

// Depthwise-style groups (one input channel per group, fewer than kCO output
// channels per group): the channel tile above would leave most of its lanes
// idle, so each thread here computes kR consecutive outputs of one output
// channel, reading that channel's taps through the read-only cache.  Grid:
// one 1-D range per (n, output channel) plane, blocks_per_plane blocks each.
__global__ void __launch_bounds__(kThreads) depthwise_kernel(const DirectParams p, int64_t items_per_plane,
                                                             int64_t blocks_per_plane) {
  const Geom &g = p.g;
  const int64_t plane = blockIdx.x / blocks_per_plane;  // n * (G * K) + oc
  const int64_t item = (blockIdx.x - plane * blocks_per_plane) * kThreads + threadIdx.x;
  if (item >= items_per_plane) return;
  const int64_t GK = g.G * g.K;
  const int64_t n = plane / GK;
  const int64_t oc = plane - n * GK;
  const int64_t grp = oc / g.K;  // its input channel (one per group)
  int64_t rest = item;
  const int owg = (int)(rest % p.owg);
  rest /= p.owg;
  const int oh = (int)(rest % g.OH);
  const int od = (int)(rest / g.OH);
  const int ow0 = owg * kR;
  const int taps = g.KD * g.KH * g.KW;
  const int64_t HW = (int64_t)g.H * g.W;
  const float *xc = p.x + n * g.x_batch_stride() + grp * g.C * g.D * HW;
  const float *wo = p.w + oc * taps;
  const float b = p.bias ? __ldg(p.bias + oc) : 0.f;
  float acc[kR];
#pragma unroll
  for (int r = 0; r < kR; ++r) acc[r] = 0.f;
  for (int kd = 0; kd < g.KD; ++kd) {
    const int id = od * g.SD + kd * g.DD - g.PD;
    if ((unsigned)id >= (unsigned)g.D) continue;
    for (int kh = 0; kh < g.KH; ++kh) {
      const int ih = oh * g.SH + kh * g.DH - g.PH;
      if ((unsigned)ih >= (unsigned)g.H) continue;
      const float *row = xc + (int64_t)id * HW + (int64_t)ih * g.W;
      const float *wt = wo + (kd * g.KH + kh) * g.KW;
      for (int kw = 0; kw < g.KW; ++kw) {
        const float wv = CONV_DBG_OK(wt + kw - p.w, p.w_elems, kStatusBoundsW) ? __ldg(wt + kw) : 0.f;
#pragma unroll
        for (int r = 0; r < kR; ++r) {
          const int iw = (ow0 + r) * g.SW + kw * g.DW - g.PW;
          if ((unsigned)iw < (unsigned)g.W && CONV_DBG_OK(row + iw - p.x, p.x_elems, kStatusBoundsX))
            acc[r] = fmaf(wv, __ldg(row + iw), acc[r]);
        }
      }
    }
  }
  float *yo = p.y + n * g.y_batch_stride() + oc * g.out_spatial() + ((int64_t)od * g.OH + oh) * g.OW;
#pragma unroll
  for (int r = 0; r < kR; ++r)
    if (ow0 + r < g.OW && CONV_DBG_OK(yo + ow0 + r - p.y, p.y_elems, kStatusBoundsY)) yo[ow0 + r] = acc[r] + b;
}

// Depthwise-style groups with stride 1 and dilation 1 (the common case): a
// block computes a 4 x 8 x 32 output tile of one (n, output channel) plane
// from its input tile staged in shared memory (zero padding filled in), each
// thread 4 consecutive outputs along W; every input value is read from global
// memory once per tile instead of once per tap.
constexpr int kDwTD = 4, kDwTH = 8, kDwTW = 32, kDwMaxK = 7;
constexpr int kDwThreads = kDwTD * kDwTH * (kDwTW / kR);  // 256
constexpr int kDwTile = (kDwTD + kDwMaxK - 1) * (kDwTH + kDwMaxK - 1) * (kDwTW + kDwMaxK - 1);

__global__ void __launch_bounds__(kDwThreads) depthwise_tiled_kernel(const DirectParams p, int tiles_d, int tiles_h,
                                                                     int tiles_w) {
  __shared__ float xs[kDwTile];
  __shared__ float ws[kDwMaxK * kDwMaxK * kDwMaxK];
  const Geom &g = p.g;
  const int64_t tiles = (int64_t)tiles_d * tiles_h * tiles_w;
  const int64_t plane = blockIdx.x / tiles;  // n * (G * K) + oc
  int64_t tl = blockIdx.x - plane * tiles;
  const int tw = (int)(tl % tiles_w);
  tl /= tiles_w;
  const int th = (int)(tl % tiles_h);
  const int td = (int)(tl / tiles_h);
  const int64_t GK = g.G * g.K;
  const int64_t n = plane / GK;
  const int64_t oc = plane - n * GK;
  const int64_t grp = oc / g.K;
  const int taps = g.KD * g.KH * g.KW;
  const int64_t HW = (int64_t)g.H * g.W;
  const float *xc = p.x + n * g.x_batch_stride() + grp * g.C * g.D * HW;
  // input tile origin and extents (stride 1, dilation 1)
  const int d0 = td * kDwTD - g.PD, h0 = th * kDwTH - g.PH, w0 = tw * kDwTW - g.PW;
  const int ID = kDwTD + g.KD - 1, IH = kDwTH + g.KH - 1, IW = kDwTW + g.KW - 1;
  // rows of the input tile, 4 at a time, 64 columns per row per pass (IW <= 38)
  for (int r = threadIdx.x >> 6; r < ID * IH; r += kDwThreads >> 6) {
    const int id = r / IH, ih = r - id * IH;
    const int d = d0 + id, h = h0 + ih;
    const bool row_in = (unsigned)d < (unsigned)g.D && (unsigned)h < (unsigned)g.H;
    const float *src = xc + (int64_t)d * HW + (int64_t)h * g.W;
    const int iw = threadIdx.x & 63;
    if (iw < IW) {
      const int w = w0 + iw;
      const bool in = row_in && (unsigned)w < (unsigned)g.W && CONV_DBG_OK(src + w - p.x, p.x_elems, kStatusBoundsX);
      if (CONV_DBG_OK(r * IW + iw, kDwTile, kStatusBoundsShared)) xs[r * IW + iw] = in ? __ldg(src + w) : 0.f;
    }
  }
  for (int i = threadIdx.x; i < taps; i += kDwThreads)
    ws[i] = CONV_DBG_OK(oc * taps + i, p.w_elems, kStatusBoundsW) ? __ldg(p.w + oc * taps + i) : 0.f;
  __syncthreads();
  const int t = threadIdx.x;
  const int lw = (t % (kDwTW / kR)) * kR, lh = (t / (kDwTW / kR)) % kDwTH, ld = t / ((kDwTW / kR) * kDwTH);
  const int od = td * kDwTD + ld, oh = th * kDwTH + lh, ow0 = tw * kDwTW + lw;
  if (od >= g.OD || oh >= g.OH || ow0 >= g.OW) return;
  float acc[kR];
#pragma unroll
  for (int r = 0; r < kR; ++r) acc[r] = 0.f;
  for (int kd = 0; kd < g.KD; ++kd)
    for (int kh = 0; kh < g.KH; ++kh) {
      const float *row = xs + ((ld + kd) * IH + (lh + kh)) * IW + lw;
      const float *wt = ws + (kd * g.KH + kh) * g.KW;
      float xv[kR + kDwMaxK - 1];
#pragma unroll
      for (int j = 0; j < kR + kDwMaxK - 1; ++j)
        if (j < kR + g.KW - 1) xv[j] = row[j];
#pragma unroll
      for (int kw = 0; kw < kDwMaxK; ++kw) {
        if (kw >= g.KW) break;
        const float wv = wt[kw];
#pragma unroll
        for (int r = 0; r < kR; ++r) acc[r] = fmaf(wv, xv[r + kw], acc[r]);
      }
    }
  const float b = p.bias ? __ldg(p.bias + oc) : 0.f;
  float *yo = p.y + n * g.y_batch_stride() + oc * g.out_spatial() + ((int64_t)od * g.OH + oh) * g.OW;
#pragma unroll
  for (int r = 0; r < kR; ++r)
    if (ow0 + r < g.OW && CONV_DBG_OK(yo + ow0 + r - p.y, p.y_elems, kStatusBoundsY)) yo[ow0 + r] = acc[r] + b;
}

}  // namespace

bool direct_supported(const Geom &g, const char **why) {
  if ((int64_t)g.taps() * kCO > kSmemFloats) {
    *why = "direct path: kernel volume above 1024 taps";
    return false;
  }
  if (g.G * ((g.K + kCO - 1) / kCO) > 65535) {
    *why = "direct path: more than 65535 blocks of 8 output channels (over all groups)";
    return false;
  }
  const int64_t items = g.N * (int64_t)g.OD * g.OH * ((g.OW + kR - 1) / kR);
  if (g.C == 1 && g.K < kCO) {
    const int64_t per_plane = ((int64_t)g.OD * g.OH * ((g.OW + kR - 1) / kR) + kThreads - 1) / kThreads;
    if (g.N * g.G * g.K * per_plane > 0x7fffffff) {
      *why = "direct path: too many output blocks for one depthwise grid";
      return false;
    }
    return true;
  }
  if ((items + kThreads - 1) / kThreads > 0x7fffffff) {
    *why = "direct path: too many output rows for one grid";
    return false;
  }
  return true;
}

cudaError_t launch_direct_ffma(const float *x, const float *w, const float *bias, float *y, const Geom &g,
                               cudaStream_t stream) {
  DirectParams p;
  p.x = x;
  p.w = w;
  p.bias = bias;
  p.y = y;
  p.g = g;
  p.owg = (g.OW + kR - 1) / kR;
  // the kernels index whole tensors (all groups) from these pointers
  p.x_elems = g.N * g.x_batch_stride() - debug_x_shrink();
  p.w_elems = g.G * g.K * g.C * g.taps();
  p.y_elems = g.N * g.y_batch_stride();
  CONV_PLAN_CHECK(!g.cl && (int64_t)g.taps() * kCO <= kSmemFloats);
  const bool unit = g.SD == 1 && g.SH == 1 && g.SW == 1 && g.DD == 1 && g.DH == 1 && g.DW == 1;
  // the tiled kernel when a tile row is mostly used (output width >= 24)
  if (g.C == 1 && g.K < kCO && unit && g.KD <= kDwMaxK && g.KH <= kDwMaxK && g.KW <= kDwMaxK && g.OW >= 24) {
    const int td = (g.OD + kDwTD - 1) / kDwTD, th = (g.OH + kDwTH - 1) / kDwTH, tw = (g.OW + kDwTW - 1) / kDwTW;
    const int64_t blocks = g.N * g.G * g.K * (int64_t)td * th * tw;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    CONV_PLAN_CHECK((kDwTD + g.KD - 1) * (kDwTH + g.KH - 1) * (kDwTW + g.KW - 1) <= kDwTile && g.taps() <= 343);
    depthwise_tiled_kernel<<<(unsigned)blocks, kDwThreads, 0, stream>>>(p, td, th, tw);
    return cudaGetLastError();
  }
  if (g.C == 1 && g.K < kCO) {
    const int64_t items = (int64_t)g.OD * g.OH * p.owg;
    const int64_t bpp = (items + kThreads - 1) / kThreads;
    const int64_t blocks = g.N * g.G * g.K * bpp;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    depthwise_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(p, items, bpp);
    return cudaGetLastError();
  }
  p.items = g.N * (int64_t)g.OD * g.OH * p.owg;
  const int taps = g.taps();
  p.cchunk = (int)(g.C < kSmemFloats / (taps * kCO) ? g.C : kSmemFloats / (taps * kCO));
  const int64_t gx = (p.items + kThreads - 1) / kThreads;
  p.kblocks = (int)((g.K + kCO - 1) / kCO);
  const int64_t gy = g.G * p.kblocks;
  if (gx > 0x7fffffff || gy > 65535) return cudaErrorInvalidConfiguration;
  CONV_PLAN_CHECK(p.cchunk >= 1 && (int64_t)p.cchunk * taps * kCO <= kSmemFloats);
  dim3 grid((unsigned)gx, (unsigned)gy);
  direct_ffma_kernel<<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace convfwd
