// Peak-rate microbenchmarks of the two pipes the convolution kernels run on:
// the 5th-generation tensor cores (tcgen05.mma, kind::tf32 or kind::f16 with
// BF16 operands, fp32 accumulation in TMEM) and the FP32 FMA units (scalar
// fma.rn.f32 and packed fma.rn.f32x2).  They give the roofline denominators
// for the convolution kernels, measured on the GPU at hand and at the clock it
// runs, instead of spec-sheet figures.
//
// Tensor cores: one persistent CTA per SM; `issuers` warps each issue `iters`
// back-to-back MMAs (M = 128, K = 32 bytes of operand per row, N as asked)
// from one elected lane on operands resident in shared memory (B, and A for
// the SS form) or tensor memory (A for the TS form).  Each issuer commits once
// at the end and waits, bounded, for its MMAs.  FFMA: every thread runs
// independent multiply-add chains over registers.  Both kernels record per
// CTA the SM clock counter and the device global timer (ns) at start and end,
// so the host gets the span of the run and the SM clock during it.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <algorithm>
#include <vector>

#include "../../include/convfwd.h"
#include "conv_internal.cuh"
#include "sm100_ptx.cuh"

namespace convfwd {
namespace {

constexpr int kPeakMaxCtas = 4096;
constexpr long long kPeakWaitCycles = 1ll << 32;

// per-CTA stamps: clock64 start/end, %globaltimer start/end; and a status word
__device__ unsigned long long g_peak_clk[2][kPeakMaxCtas];
__device__ unsigned long long g_peak_ns[2][kPeakMaxCtas];
__device__ unsigned int g_peak_status;
__device__ float g_peak_sink;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

constexpr int kMmaThreads = 128;
constexpr int kMmaSmem = 120 * 1024;  // keeps one CTA per SM: its 512 TMEM columns never contend

// kind 0: kind::tf32 (K = 8); kind 1: kind::f16 with BF16 operands (K = 16).
// A (128 rows) and B (n rows) are 32-byte rows in the K-major no-swizzle
// core-matrix layout: LBO 128 bytes (the two 16-byte halves of a row), SBO
// 256 bytes (consecutive 8-row groups).
template <int KIND>
__global__ void __launch_bounds__(kMmaThreads, 1) mma_rate_kernel(int n, int issuers, int a_in_tmem, int iters) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *a_s = smem;            // 128 x 32 bytes
  uint8_t *b_s = smem + 4096;     // n x 32 bytes (n <= 256)
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 4096 + 8192);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 4);
  const int tid = threadIdx.x, warp = tid >> 5;

  // operand values: small, varied, exactly representable in the operand type
  for (int i = tid; i < (4096 + 8192) / 4; i += kMmaThreads) {
    const float v = 0.25f + 0.0625f * (float)((i * 7 + 3) % 13);
    uint32_t bits = __float_as_uint(v);
    if (KIND == 1) bits = (bits >> 16) | (bits & 0xffff0000u);  // two bf16 copies of v
    reinterpret_cast<uint32_t *>(smem)[i] = bits;
  }
  ptx::fence_proxy_async_smem();
  if (warp == 0) ptx::tmem_alloc(ptx::smem_addr(tmem_slot), 512);
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) ptx::mbar_init(ptx::smem_addr(bars + i), 1);
    ptx::fence_mbar_init();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // A for the TS form: TMEM columns 480..487 (8 columns of 32 bits = one 32-byte row per lane)
  const uint32_t a_tmem = tmem + 480u;
  if (a_in_tmem) {
    uint32_t v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = reinterpret_cast<const uint32_t *>(a_s)[(tid * 8 + j) % 1024];
    ptx::tmem_st8(tmem + ((uint32_t)(warp * 32) << 16) + 480u, v);
    ptx::tmem_wait_st();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();

  const uint32_t idesc = KIND == 0 ? ptx::idesc_tf32(128, (uint32_t)n) : ptx::idesc_bf16(128, (uint32_t)n);
  const uint64_t a_desc = ptx::smem_desc_noswizzle(ptx::smem_addr(a_s), 128, 256);
  const uint64_t b_desc = ptx::smem_desc_noswizzle(ptx::smem_addr(b_s), 128, 256);
  // distinct accumulators while they fit below column 480, shared beyond
  int n_acc = 480 / n;
  if (n_acc < 1) n_acc = 1;
  if (warp < issuers) {
    const uint32_t d = tmem + (uint32_t)((warp % n_acc) * n);
    const uint32_t bar = ptx::smem_addr(bars + warp);
    __syncwarp();
    const unsigned long long c0 = clock64(), t0 = globaltimer_ns();
    if (ptx::elect_one()) {
      for (int i = 0; i < iters; ++i) {
        if (KIND == 0) {
          if (a_in_tmem)
            ptx::mma_tf32_ts(d, a_tmem, b_desc, idesc, i > 0);
          else
            ptx::mma_tf32_ss(d, a_desc, b_desc, idesc, i > 0);
        } else {
          if (a_in_tmem)
            ptx::mma_f16_ts(d, a_tmem, b_desc, idesc, i > 0);
          else
            ptx::mma_f16_ss(d, a_desc, b_desc, idesc, i > 0);
        }
      }
      ptx::mma_commit(bar);
    }
    __syncwarp();
    bool done = false;
    const long long w0 = clock64();
    while (!(done = ptx::mbar_try_wait(bar, 0)) && clock64() - w0 < kPeakWaitCycles) {
    }
    const unsigned long long c1 = clock64(), t1 = globaltimer_ns();
    if (!done && (tid & 31) == 0) atomicOr(&g_peak_status, 1u);
    if (warp == 0 && (tid & 31) == 0 && blockIdx.x < kPeakMaxCtas) {
      g_peak_clk[0][blockIdx.x] = c0;
      g_peak_clk[1][blockIdx.x] = c1;
      g_peak_ns[0][blockIdx.x] = t0;
      g_peak_ns[1][blockIdx.x] = t1;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

constexpr int kFmaThreads = 512;
constexpr int kFmaChains = 16;  // independent fp32 multiply-add chains per thread (8 float pairs when packed)

template <bool PACKED>
__global__ void __launch_bounds__(kFmaThreads) ffma_rate_kernel(int iters, float m, float c) {
  float a[kFmaChains];
#pragma unroll
  for (int j = 0; j < kFmaChains; ++j) a[j] = (float)(threadIdx.x + j) * 1e-3f;
  const unsigned long long c0 = clock64(), t0 = globaltimer_ns();
  if (PACKED) {
    uint64_t acc[kFmaChains / 2], mm, cc;
    asm("mov.b64 %0, {%1, %1};" : "=l"(mm) : "f"(m));
    asm("mov.b64 %0, {%1, %1};" : "=l"(cc) : "f"(c));
#pragma unroll
    for (int j = 0; j < kFmaChains / 2; ++j) asm("mov.b64 %0, {%1, %2};" : "=l"(acc[j]) : "f"(a[2 * j]), "f"(a[2 * j + 1]));
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int j = 0; j < kFmaChains / 2; ++j) asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(acc[j]) : "l"(mm), "l"(cc));
    }
#pragma unroll
    for (int j = 0; j < kFmaChains / 2; ++j) asm("mov.b64 {%0, %1}, %2;" : "=f"(a[2 * j]), "=f"(a[2 * j + 1]) : "l"(acc[j]));
  } else {
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int j = 0; j < kFmaChains; ++j) asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(a[j]) : "f"(m), "f"(c));
    }
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kFmaChains; ++j) s += a[j];
  __syncthreads();
  const unsigned long long c1 = clock64(), t1 = globaltimer_ns();
  if (s == 1234.5678f) g_peak_sink = s;  // keeps the chains live
  if (threadIdx.x == 0 && blockIdx.x < kPeakMaxCtas) {
    g_peak_clk[0][blockIdx.x] = c0;
    g_peak_clk[1][blockIdx.x] = c1;
    g_peak_ns[0][blockIdx.x] = t0;
    g_peak_ns[1][blockIdx.x] = t1;
  }
}

// Span (s) from the earliest start to the latest end, the median per-CTA SM
// clock (MHz) = clock cycles / global-timer ns over each CTA's own run, and
// the median per-CTA cycle count.
cudaError_t read_stamps(int ctas, double *span_s, double *mhz, double *median_cycles) {
  std::vector<unsigned long long> clk(2 * kPeakMaxCtas), ns(2 * kPeakMaxCtas);
  cudaError_t e = cudaMemcpyFromSymbol(clk.data(), g_peak_clk, sizeof(g_peak_clk));
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(ns.data(), g_peak_ns, sizeof(g_peak_ns));
  if (e != cudaSuccess) return e;
  unsigned long long t_first = ~0ull, t_last = 0;
  std::vector<double> r(ctas), cyc(ctas);
  for (int i = 0; i < ctas; ++i) {
    const unsigned long long s0 = ns[i], s1 = ns[kPeakMaxCtas + i];
    t_first = std::min(t_first, s0);
    t_last = std::max(t_last, s1);
    cyc[i] = (double)(clk[kPeakMaxCtas + i] - clk[i]);
    r[i] = s1 > s0 ? cyc[i] / (double)(s1 - s0) * 1e3 : 0.0;
  }
  auto median = [](std::vector<double> &v) {
    std::sort(v.begin(), v.end());
    const size_t k = v.size();
    return k ? (k % 2 ? v[k / 2] : 0.5 * (v[k / 2 - 1] + v[k / 2])) : 0.0;
  };
  *span_s = t_last > t_first ? (double)(t_last - t_first) * 1e-9 : 0.0;
  *mhz = median(r);
  *median_cycles = median(cyc);
  return cudaSuccess;
}

bool g_mma_attr[64][2] = {};

}  // namespace
}  // namespace convfwd

using namespace convfwd;

namespace {
int peak_fail(int st, const char *msg) { return report_error(st, "%s", msg); }
int peak_cuda(cudaError_t e, const char *where) {
  return report_error(CONV_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

// Launch `launch` once untimed and once timed with events on `stream`.
template <class F>
int timed_twice(F launch, cudaStream_t stream, float *event_ms) {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaError_t e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  if (e == cudaSuccess) e = launch();
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaEventRecord(e0, stream);
  if (e == cudaSuccess) e = launch();
  if (e == cudaSuccess) e = cudaEventRecord(e1, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaEventElapsedTime(event_ms, e0, e1);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  return e == cudaSuccess ? CONV_OK : peak_cuda(e, "peak microbenchmark");
}
}  // namespace

extern "C" {

int conv_peak_mma(int kind, int n, int issuers, int a_in_tmem, int iters, conv_peak_result_t *out,
                  conv_stream_t stream) {
  report_error(CONV_OK, "%s", "");
  if (!out) return peak_fail(CONV_ERR_NULL, "conv_peak_mma: out is NULL");
  if (kind != 0 && kind != 1) return peak_fail(CONV_ERR_ARG, "conv_peak_mma: kind must be 0 (tf32) or 1 (bf16)");
  if (n < 16 || n > 256 || n % 16 != 0) return peak_fail(CONV_ERR_ARG, "conv_peak_mma: n must be 16..256, a multiple of 16");
  if (issuers < 1 || issuers > 4) return peak_fail(CONV_ERR_ARG, "conv_peak_mma: issuers must be 1..4");
  if (iters < 1 || iters > (1 << 18)) return peak_fail(CONV_ERR_ARG, "conv_peak_mma: iters must be 1..262144");
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return peak_cuda(e, "conv_peak_mma: device query");
  if (dev < 0 || dev >= 64 || sms > kPeakMaxCtas) return peak_fail(CONV_ERR_UNSUPPORTED, "conv_peak_mma: device index or SM count out of range");
  if (!g_mma_attr[dev][kind]) {
    e = cudaFuncSetAttribute(kind ? mma_rate_kernel<1> : mma_rate_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMmaSmem);
    if (e != cudaSuccess) return peak_cuda(e, "conv_peak_mma: cudaFuncSetAttribute");
    g_mma_attr[dev][kind] = true;
  }
  const unsigned zero = 0;
  e = cudaMemcpyToSymbol(g_peak_status, &zero, sizeof(zero));
  if (e != cudaSuccess) return peak_cuda(e, "conv_peak_mma: status reset");
  cudaStream_t s = (cudaStream_t)stream;
  float ms = 0.f;
  int st = timed_twice(
      [&]() {
        if (kind)
          mma_rate_kernel<1><<<sms, kMmaThreads, kMmaSmem, s>>>(n, issuers, a_in_tmem, iters);
        else
          mma_rate_kernel<0><<<sms, kMmaThreads, kMmaSmem, s>>>(n, issuers, a_in_tmem, iters);
        return cudaGetLastError();
      },
      s, &ms);
  if (st != CONV_OK) return st;
  unsigned status = 0;
  e = cudaMemcpyFromSymbol(&status, g_peak_status, sizeof(status));
  if (e != cudaSuccess) return peak_cuda(e, "conv_peak_mma: status read");
  if (status) return peak_fail(CONV_ERR_CUDA, "conv_peak_mma: a wait for the MMAs gave up");
  double span = 0, mhz = 0, cyc = 0;
  e = read_stamps(sms, &span, &mhz, &cyc);
  if (e != cudaSuccess) return peak_cuda(e, "conv_peak_mma: reading the stamps");
  const double k = kind ? 16.0 : 8.0;
  out->flops = 2.0 * 128.0 * n * k * (double)iters * issuers * sms;
  out->seconds = span;
  out->event_ms = ms;
  out->sm_mhz = mhz;
  out->cycles_per_op = cyc / ((double)iters * issuers);  // SM cycles per MMA on one SM
  out->ctas = sms;
  return CONV_OK;
}

int conv_peak_ffma(int packed, int iters, conv_peak_result_t *out, conv_stream_t stream) {
  report_error(CONV_OK, "%s", "");
  if (!out) return peak_fail(CONV_ERR_NULL, "conv_peak_ffma: out is NULL");
  if (iters < 1 || iters > (1 << 20)) return peak_fail(CONV_ERR_ARG, "conv_peak_ffma: iters must be 1..1048576");
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, packed ? ffma_rate_kernel<true> : ffma_rate_kernel<false>,
                                                      kFmaThreads, 0);
  if (e != cudaSuccess) return peak_cuda(e, "conv_peak_ffma: device query");
  const int ctas = sms * (per_sm > 0 ? per_sm : 1);
  if (ctas > kPeakMaxCtas) return peak_fail(CONV_ERR_UNSUPPORTED, "conv_peak_ffma: too many CTAs");
  cudaStream_t s = (cudaStream_t)stream;
  float ms = 0.f;
  int st = timed_twice(
      [&]() {
        if (packed)
          ffma_rate_kernel<true><<<ctas, kFmaThreads, 0, s>>>(iters, 0.999f, 1e-3f);
        else
          ffma_rate_kernel<false><<<ctas, kFmaThreads, 0, s>>>(iters, 0.999f, 1e-3f);
        return cudaGetLastError();
      },
      s, &ms);
  if (st != CONV_OK) return st;
  double span = 0, mhz = 0, cyc = 0;
  e = read_stamps(ctas, &span, &mhz, &cyc);
  if (e != cudaSuccess) return peak_cuda(e, "conv_peak_ffma: reading the stamps");
  out->flops = 2.0 * (double)kFmaThreads * ctas * (double)iters * 4 * kFmaChains;
  out->seconds = span;
  out->event_ms = ms;
  out->sm_mhz = mhz;
  // SM cycles per FMA instruction per SM (a packed instruction counts once and does two)
  const double instr_per_sm = (double)kFmaThreads * (per_sm > 0 ? per_sm : 1) * iters * 4 * kFmaChains / (packed ? 2 : 1) / 32.0;
  out->cycles_per_op = cyc / instr_per_sm;
  out->ctas = ctas;
  return CONV_OK;
}

}  // extern "C"
