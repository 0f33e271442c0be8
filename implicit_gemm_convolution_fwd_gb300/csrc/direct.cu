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
      ws[i] = og < g.K ? p.w[((ob + og) * g.C + c0) * taps + ct] : 0.f;
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
              xv[r] = ((unsigned)iw < (unsigned)g.W) ? __ldg(row + iw) : 0.f;
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
      if (ow0 + r < g.OW) yo[ow0 + r] = acc[o][r] + b;
  }
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
  p.items = g.N * (int64_t)g.OD * g.OH * p.owg;
  const int taps = g.taps();
  p.cchunk = (int)(g.C < kSmemFloats / (taps * kCO) ? g.C : kSmemFloats / (taps * kCO));
  const int64_t gx = (p.items + kThreads - 1) / kThreads;
  p.kblocks = (int)((g.K + kCO - 1) / kCO);
  const int64_t gy = g.G * p.kblocks;
  if (gx > 0x7fffffff || gy > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)gx, (unsigned)gy);
  direct_ffma_kernel<<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace convfwd
