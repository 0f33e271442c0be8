// Fused Conv3d -> min over output depth -> softmax over channels, following
// the l2_p24 page (Conv3d -> torch.min(dim=2) -> torch.softmax(dim=1)),
// turns 1-2: for every (n, h, w) column the conv is evaluated at every output
// depth, a running minimum per channel is kept, and the channel softmax is
// taken with the maximum subtracted.  The 5-D conv intermediate never leaves
// registers.
//
// Mapping: one warp owns NROW output rows (n, oh) and a tile of NOWG*R output
// columns; lane = (row, channel group, column group).  A thread keeps a CO x R
// register tile (CO output channels x R consecutive columns) of conv sums for
// the current depth plus the running minima.  Weights for all channels sit in
// shared memory laid out [tap][channel group][CO], so one lane's CO weights are
// three 16-byte broadcast reads.  Input rows are read through the read-only
// cache (the whole input of the benchmark workload fits in L2), R+KW-1 values
// per (c, kd, kh) row feeding KW*R*CO FMAs.  The channel softmax runs across
// the NCG lanes that hold one column's channels with xor-shuffles; lanes of
// padding channels contribute -inf to the max and 0 to the sum.
//
// min(conv + b) == min(conv) + b exactly in fp32 (x -> fl(x + b) is monotone),
// so the bias is added once after the depth loop.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "conv_internal.cuh"

namespace convfwd {
namespace {

constexpr int kCO = 12;  // channels per thread
constexpr int kR = 4;    // columns per thread
constexpr int kMaxKW = 7;
constexpr int kMaxSmemBytes = 200 * 1024;

struct FusedParams {
  const float *__restrict__ x;
  const float *__restrict__ w;
  const float *__restrict__ bias;
  float *__restrict__ y;
  Geom g;
  int64_t rows;   // N * OH
  int coltiles;   // ceil(OW / (NOWG * R))
};

// NCG channel groups per warp, NROW rows per warp, KWT = compile-time kernel
// width (0: runtime, <= kMaxKW), VEC = 16-byte input loads (needs W % 4 == 0,
// aligned x, KWT == 3).
template <int NCG, int NROW, int KWT, bool VEC>
__global__ void __launch_bounds__(32, 14) fused_min_softmax_kernel(const FusedParams p) {
  constexpr int NOWG = 32 / (NCG * NROW);
  constexpr int NCH = NCG * kCO;  // channel slots in the warp
  constexpr int XW = KWT ? (kR + KWT - 1) : (kR + kMaxKW - 1);
  extern __shared__ __align__(16) float ws[];  // [C*taps][NCG][kCO]

  const Geom &g = p.g;
  const int KW = KWT ? KWT : g.KW;
  const int taps = g.KD * g.KH * KW;

  // ---- stage weights: ws[(c*taps + t)*NCH + o] = w[o][c][t], zero for o >= K
  {
    const int total = (int)(g.C * taps) * NCH;
    for (int i = threadIdx.x; i < total; i += 32) {
      const int o = i % NCH;
      const int ct = i / NCH;
      ws[i] = o < g.K ? p.w[(int64_t)o * g.C * taps + ct] : 0.f;
    }
  }
  __syncwarp();

  const int lane = threadIdx.x;
  const int owg = lane % NOWG;
  const int cg = (lane / NOWG) % NCG;
  const int rr = lane / (NOWG * NCG);
  const int tile = blockIdx.x % p.coltiles;
  const int64_t row = (int64_t)(blockIdx.x / p.coltiles) * NROW + rr;
  const bool row_ok = row < p.rows;
  const int64_t rowc = row_ok ? row : p.rows - 1;
  const int64_t n = rowc / g.OH;
  const int oh = (int)(rowc % g.OH);
  const int ow0 = (tile * NOWG + owg) * kR;

  const int64_t HW = (int64_t)g.H * g.W;
  const float *xn = p.x + n * g.C * g.D * HW + (int64_t)oh * g.W + ow0;

  float mins[kCO][kR];
#pragma unroll
  for (int o = 0; o < kCO; ++o)
#pragma unroll
    for (int r = 0; r < kR; ++r) mins[o][r] = INFINITY;

  for (int od = 0; od < g.OD; ++od) {
    float acc[kCO][kR];
#pragma unroll
    for (int o = 0; o < kCO; ++o)
#pragma unroll
      for (int r = 0; r < kR; ++r) acc[o][r] = 0.f;

    for (int c = 0; c < g.C; ++c) {
      for (int kd = 0; kd < g.KD; ++kd) {
        const float *plane = xn + ((int64_t)c * g.D + od + kd) * HW;
        const float *wrow = ws + ((c * g.KD + kd) * g.KH) * KW * NCH + cg * kCO;
#pragma unroll 3
        for (int kh = 0; kh < g.KH; ++kh) {
          const float *xr = plane + (int64_t)kh * g.W;
          float xv[XW];
          if (VEC) {
            // W % 4 == 0 and ow0 % 4 == 0: a 4-wide group is either fully
            // inside the row or fully past its end
            if (ow0 < g.W) {
              const float4 a = __ldg(reinterpret_cast<const float4 *>(xr));
              xv[0] = a.x, xv[1] = a.y, xv[2] = a.z, xv[3] = a.w;
            } else {
              xv[0] = 0.f, xv[1] = 0.f, xv[2] = 0.f, xv[3] = 0.f;
            }
            if (ow0 + 4 < g.W) {
              const float2 b = __ldg(reinterpret_cast<const float2 *>(xr + 4));
              xv[4] = b.x, xv[5] = b.y;
            } else {
              xv[4] = 0.f, xv[5] = 0.f;
            }
          } else {
#pragma unroll
            for (int j = 0; j < XW; ++j)
              xv[j] = (j < kR + KW - 1 && ow0 + j < g.W) ? __ldg(xr + j) : 0.f;
          }
          const float *wt = wrow + kh * KW * NCH;
#pragma unroll
          for (int kw = 0; kw < (KWT ? KWT : kMaxKW); ++kw) {
            if (!KWT && kw >= KW) break;
            const float4 w0 = *reinterpret_cast<const float4 *>(wt + kw * NCH);
            const float4 w1 = *reinterpret_cast<const float4 *>(wt + kw * NCH + 4);
            const float4 w2 = *reinterpret_cast<const float4 *>(wt + kw * NCH + 8);
            const float wv[kCO] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w, w2.x, w2.y, w2.z, w2.w};
#pragma unroll
            for (int o = 0; o < kCO; ++o)
#pragma unroll
              for (int r = 0; r < kR; ++r) acc[o][r] = fmaf(wv[o], xv[r + kw], acc[o][r]);
          }
        }
      }
    }
#pragma unroll
    for (int o = 0; o < kCO; ++o)
#pragma unroll
      for (int r = 0; r < kR; ++r) mins[o][r] = fminf(mins[o][r], acc[o][r]);
  }

  // ---- channel softmax for each of the R columns
  const int64_t OHW = (int64_t)g.OH * g.OW;
#pragma unroll
  for (int r = 0; r < kR; ++r) {
    float v[kCO];
    float mx = -INFINITY;
#pragma unroll
    for (int o = 0; o < kCO; ++o) {
      const int oc = cg * kCO + o;
      v[o] = oc < g.K ? mins[o][r] + (p.bias ? __ldg(p.bias + oc) : 0.f) : -INFINITY;
      mx = fmaxf(mx, v[o]);
    }
#pragma unroll
    for (int m = NOWG; m < NOWG * NCG; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    float s = 0.f;
#pragma unroll
    for (int o = 0; o < kCO; ++o) {
      v[o] = expf(v[o] - mx);  // padding channels: exp(-inf) = 0
      s += v[o];
    }
#pragma unroll
    for (int m = NOWG; m < NOWG * NCG; m <<= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
    const int ow = ow0 + r;
    if (row_ok && ow < g.OW) {
      float *yo = p.y + n * g.K * OHW + (int64_t)oh * g.OW + ow;
#pragma unroll
      for (int o = 0; o < kCO; ++o) {
        const int oc = cg * kCO + o;
        if (oc < g.K) yo[(int64_t)oc * OHW] = v[o] / s;
      }
    }
  }
}

template <int NCG, int NROW, int KWT, bool VEC>
cudaError_t launch_t(const FusedParams &p0, cudaStream_t stream) {
  constexpr int NOWG = 32 / (NCG * NROW);
  FusedParams p = p0;
  p.coltiles = (p.g.OW + NOWG * kR - 1) / (NOWG * kR);
  const int64_t rowgroups = (p.rows + NROW - 1) / NROW;
  const int64_t blocks = rowgroups * p.coltiles;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const size_t smem = sizeof(float) * (size_t)(p.g.C * p.g.taps()) * NCG * kCO;
  auto kern = fused_min_softmax_kernel<NCG, NROW, KWT, VEC>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)blocks, 32, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int NCG, int NROW>
cudaError_t launch_ncg(const FusedParams &p, cudaStream_t stream) {
  const Geom &g = p.g;
  if (g.KW == 3) {
    const bool vec = (g.W % 4 == 0) && (((uintptr_t)p.x & 15u) == 0);
    return vec ? launch_t<NCG, NROW, 3, true>(p, stream) : launch_t<NCG, NROW, 3, false>(p, stream);
  }
  return launch_t<NCG, NROW, 0, false>(p, stream);
}

int pick_ncg(int64_t K) {
  if (K <= kCO) return 1;
  if (K <= 2 * kCO) return 2;
  if (K <= 4 * kCO) return 4;
  return 8;
}

}  // namespace

bool fused_supported(const Geom &g, const char **why) {
  if (g.K > 8 * kCO) {
    *why = "fused path: C_out above 96";
    return false;
  }
  if (g.KW > kMaxKW) {
    *why = "fused path: kernel width above 7";
    return false;
  }
  const int ncg = pick_ncg(g.K);
  if ((int64_t)g.C * g.taps() * ncg * kCO * 4 > kMaxSmemBytes) {
    *why = "fused path: weights exceed the shared-memory budget";
    return false;
  }
  return true;
}

cudaError_t launch_fused_min_softmax(const float *x, const float *w, const float *bias, float *y,
                                     const Geom &g, cudaStream_t stream) {
  FusedParams p;
  p.x = x;
  p.w = w;
  p.bias = bias;
  p.y = y;
  p.g = g;
  p.rows = g.N * (int64_t)g.OH;
  p.coltiles = 1;
  switch (pick_ncg(g.K)) {
    case 1: return launch_ncg<1, 4>(p, stream);
    case 2: return launch_ncg<2, 2>(p, stream);
    case 4: return launch_ncg<4, 1>(p, stream);
    default: return launch_ncg<8, 1>(p, stream);
  }
}

}  // namespace convfwd
