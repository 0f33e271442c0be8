// Fused Conv3d -> min over output depth -> softmax over channels, following
// the l2_p24 page (Conv3d -> torch.min(dim=2) -> torch.softmax(dim=1)),
// turns 1-2: for every (n, h, w) column the conv is evaluated at every output
// depth, a running minimum per channel is kept, and the channel softmax is
// taken with the maximum subtracted.  The 5-D conv intermediate never leaves
// registers.  The page's module takes the min dimension as a constructor
// argument; the generic kernel also reduces over height or width (min_dim 3,
// 4) by giving the spatial axes roles: R (reduced), A (rows), B (columns).
//
// Mapping: one warp owns NROW output rows (n, oa) and a tile of NOWG*R output
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
#include "debug_check.cuh"

namespace convfwd {
namespace {

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

constexpr int kCO = 12;  // channels per thread
constexpr int kR = 4;    // columns per thread
constexpr int kMaxKW = 7;
constexpr int kMaxSmemBytes = 200 * 1024;
// A lane reads input columns ow0 .. ow0 + 5 of a shared row (ow0 <= 28) whatever
// the input width, so the last row of a ring can be over-read by up to 26
// floats when the row pitch is short; the shared-memory allocation carries
// this many floats of slack past the last ring.
constexpr int kRingSlackFloats = 32;

// The three spatial output axes in the roles the kernel gives them: R is the
// reduced (min) axis, A the row axis and B the column axis (consecutive
// columns per thread).  For the page's min over depth, (R, A, B) = (D, H, W).
struct FusedParams {
  const float *__restrict__ x;
  const float *__restrict__ w;
  const float *__restrict__ bias;
  float *__restrict__ y;
  Geom g;
  int64_t rows;    // N * OA
  int coltiles;    // ceil(OB / (NOWG * R))
  int OR, OA, OB;  // output extents along R, A, B
  int KR, KA, KB;  // kernel extents along R, A, B
  int IB;          // input extent along B
  int64_t sR, sA;  // input strides (elements) along R and A
  int sB;          // input stride along B (1, or W when B is H)
  int wR, wA, wB;  // weight offsets (within one input channel's taps) per step along R, A, B
  int64_t x_elems, w_elems, y_elems;  // extents the debug build's device checks use
};

// NCG channel groups per warp, NROW rows per warp, KWT = compile-time kernel
// extent along the column axis (0: runtime, <= kMaxKW), VEC = 16-byte input
// loads (needs unit column stride, input extent along B % 4 == 0, aligned x,
// KWT == 3).
template <int NCG, int NROW, int KWT, bool VEC>
__global__ void __launch_bounds__(32, 14) fused_min_softmax_kernel(const FusedParams p) {
  constexpr int NOWG = 32 / (NCG * NROW);
  constexpr int NCH = NCG * kCO;  // channel slots in the warp
  constexpr int XW = KWT ? (kR + KWT - 1) : (kR + kMaxKW - 1);
  extern __shared__ __align__(16) float ws[];  // [C*taps][NCG][kCO]

  const Geom &g = p.g;
  const int KW = KWT ? KWT : p.KB;  // kernel extent along the column axis
  const int taps = g.KD * g.KH * g.KW;

  // ---- stage weights: ws[((c*KR + kr)*KA + ka)*KB + kb][o] = w[o][c][tap (kr, ka, kb)],
  // zero for o >= K
  {
    const int total = (int)(g.C * taps) * NCH;
    for (int i = threadIdx.x; i < total; i += 32) {
      const int o = i % NCH;
      const int ct = i / NCH;
      const int c = ct / taps, t = ct - c * taps;
      const int kr = t / (p.KA * KW), rem = t - kr * p.KA * KW;
      const int ka = rem / KW, kb = rem - ka * KW;
      const int64_t wi = (int64_t)o * g.C * taps + c * taps + kr * p.wR + ka * p.wA + kb * p.wB;
      ws[i] = (o < g.K && CONV_DBG_OK(wi, p.w_elems, kStatusBoundsW)) ? p.w[wi] : 0.f;
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
  const int64_t n = rowc / p.OA;
  const int oa = (int)(rowc % p.OA);
  const int ob0 = (tile * NOWG + owg) * kR;

  const int64_t HW = (int64_t)g.H * g.W;
  const float *xn = p.x + n * g.C * g.D * HW + (int64_t)oa * p.sA + (int64_t)ob0 * p.sB;

  float mins[kCO][kR];
#pragma unroll
  for (int o = 0; o < kCO; ++o)
#pragma unroll
    for (int r = 0; r < kR; ++r) mins[o][r] = INFINITY;

  for (int orr = 0; orr < p.OR; ++orr) {
    float acc[kCO][kR];
#pragma unroll
    for (int o = 0; o < kCO; ++o)
#pragma unroll
      for (int r = 0; r < kR; ++r) acc[o][r] = 0.f;

    for (int c = 0; c < g.C; ++c) {
      for (int kr = 0; kr < p.KR; ++kr) {
        const float *plane = xn + (int64_t)c * g.D * HW + (int64_t)(orr + kr) * p.sR;
        const float *wrow = ws + ((c * p.KR + kr) * p.KA) * KW * NCH + cg * kCO;
#pragma unroll 3
        for (int ka = 0; ka < p.KA; ++ka) {
          const float *xr = plane + (int64_t)ka * p.sA;
          float xv[XW];
          if (VEC) {
            // unit column stride, IB % 4 == 0 and ob0 % 4 == 0: a 4-wide group
            // is either fully inside the row or fully past its end
            if (ob0 < p.IB && CONV_DBG_OK(xr - p.x, p.x_elems, kStatusBoundsX) &&
                CONV_DBG_OK(xr + 3 - p.x, p.x_elems, kStatusBoundsX)) {
              const float4 a = __ldg(reinterpret_cast<const float4 *>(xr));
              xv[0] = a.x, xv[1] = a.y, xv[2] = a.z, xv[3] = a.w;
            } else {
              xv[0] = 0.f, xv[1] = 0.f, xv[2] = 0.f, xv[3] = 0.f;
            }
            if (ob0 + 4 < p.IB && CONV_DBG_OK(xr + 5 - p.x, p.x_elems, kStatusBoundsX)) {
              const float2 b = __ldg(reinterpret_cast<const float2 *>(xr + 4));
              xv[4] = b.x, xv[5] = b.y;
            } else {
              xv[4] = 0.f, xv[5] = 0.f;
            }
          } else {
#pragma unroll
            for (int j = 0; j < XW; ++j)
              xv[j] = (j < kR + KW - 1 && ob0 + j < p.IB &&
                       CONV_DBG_OK(xr + (int64_t)j * p.sB - p.x, p.x_elems, kStatusBoundsX))
                          ? __ldg(xr + (int64_t)j * p.sB)
                          : 0.f;
          }
          const float *wt = wrow + ka * KW * NCH;
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
  const int64_t OAB = (int64_t)p.OA * p.OB;
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
    const int ob = ob0 + r;
    if (row_ok && ob < p.OB) {
      float *yo = p.y + n * g.K * OAB + (int64_t)oa * p.OB + ob;
#pragma unroll
      for (int o = 0; o < kCO; ++o) {
        const int oc = cg * kCO + o;
        if (oc < g.K && CONV_DBG_OK(yo + (int64_t)oc * OAB - p.y, p.y_elems, kStatusBoundsY))
          yo[(int64_t)oc * OAB] = v[o] / s;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Staged variant for the common shape (C_out <= 24, output width <= 32, KW = 3):
// one persistent CTA per SM owns a contiguous block of (n, oh) output rows
// (26 at a time, one per warp).  The input rows that block needs are streamed
// through a ring of KD + 2*NB - 1 depth planes in shared memory with cp.async:
// while the block computes NB output depths from the planes it holds, the next
// NB planes land in the other slots, so the block synchronises once per NB
// depths and the FMA loop reads x from shared memory.
// A lane holds 6 channels x 4 columns (lane = channel group x column group),
// which keeps registers low enough for 26 warps per SM to hide shared-memory
// latency; the min / softmax epilogue is as above.
constexpr int kSWarps = 26;
constexpr int kSThreads = kSWarps * 32;
constexpr int kSRows = kSWarps;      // output rows per block
constexpr int kSCO = 6;              // channels per lane
constexpr int kSNcg = 4;             // 4 x 6 = 24 channel slots
constexpr int kSWTap = 8;            // floats per (row, channel group, tap): 6 channels + 2 pad
constexpr int kSWStride = 3 * kSWTap;  // floats per (row, channel group)
constexpr int kSWRow = kSNcg * kSWStride;  // floats per (c, kd, kh) weight row
constexpr int kSMaxSrows = 128;      // shared rows per channel per plane (output rows + halos)

struct StagedParams {
  const float *__restrict__ x;
  const float *__restrict__ w;
  const float *__restrict__ bias;
  float *__restrict__ y;
  Geom g;
  int64_t rows;          // N * OA
  // axis roles as in FusedParams, with the column axis always W: (R, A) =
  // (D, H) for the min over depth, (H, D) for the min over height
  int OR, OA;            // output extents along R and A
  int KR, KA;            // kernel extents along R and A
  int IR;                // input extent along R (planes)
  int64_t sR, sA;        // input strides along R and A
  int wR, wA;            // weight offsets per step along R and A
  int WP;                // shared-memory row pitch (floats): W rounded up to 4, plus 4
  int srows_max;         // shared-memory rows per channel per plane
  int ring;              // planes in the ring (KD + 2 * nb - 1)
  int nb;                // output depths computed between two block-wide barriers
  int vec;               // 16-byte copies are legal
  uint32_t w_floats;     // weight region size (floats, multiple of 4)
  uint32_t slot_floats;  // one plane: C * srows_max * WP
  int64_t x_elems, w_elems, y_elems;  // extents the debug build's device checks use
};

// Packed fp32 pairs (two adjacent output channels) for fma.rn.f32x2.
__device__ __forceinline__ unsigned long long pack2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack2(unsigned long long r, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
// acc += w * x for both halves (round to nearest, no flush), one instruction.
__device__ __forceinline__ void fma2(unsigned long long &acc, unsigned long long w, unsigned long long x) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(w), "l"(x));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const float *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const float *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// Wait until at most n of this thread's cp.async groups are pending (n clamped to [0, 7]).
__device__ __forceinline__ void cp_async_wait_pending(int n) {
  switch (n < 0 ? 0 : n) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
  }
}

// CT, KDT, KHT, WPT, SRT: compile-time C_in, KR, KA (the kernel extents along
// the reduced and row axes: KD, KH for the min over depth), shared row pitch
// and shared rows per channel (0 = runtime); the benchmark shape is
// specialised so that every shared-memory offset in the FMA loop is an
// immediate.  Names below follow the min over depth (planes = depth).
// SKIP: warps without a row of the block skip the FMA work (worth it when the
// CTAs' row shares are well below the warp count; it costs a few registers).
template <int CT, int KDT, int KHT, int WPT, int SRT, bool SKIP>
__global__ void __launch_bounds__(kSThreads, 1) fused_min_softmax_staged_kernel(const StagedParams p) {
  constexpr int NOWG = 8;
  extern __shared__ __align__(16) float sm[];
  float *ws = sm;                 // [(c*KD + kd)*KH + kh][4 channel groups][kw][6 channels + 2 pad]
  float *ring = sm + p.w_floats;  // [ring][C][srows_max][WP]
  __shared__ int64_t srow_src[kSMaxSrows];  // input-row base offset of each shared row
  __shared__ int nsrows_s;

  const Geom &g = p.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = CT ? CT : (int)g.C, KD = KDT ? KDT : p.KR, KH = KHT ? KHT : p.KA;
  const int WP = WPT ? WPT : p.WP, SR = SRT ? SRT : p.srows_max;
  const int taps = KD * KH * 3;
  const int64_t HW = (int64_t)g.H * g.W;

  __shared__ float bias_s[kSNcg * kSCO];
  // weights (and bias) -> shared memory; run once, after the first input
  // planes are requested, so that both loads are in flight together
  auto stage_weights = [&]() {
    for (int i = tid; i < C * KD * KH * kSWRow; i += kSThreads) {
      const int row = i / kSWRow, rem = i - row * kSWRow;
      const int cgi = rem / kSWStride, jj = rem - cgi * kSWStride;
      float v = 0.f;
      const int kw = jj / kSWTap, o = jj - kw * kSWTap, oc = cgi * kSCO + o;
      if (o < kSCO && oc < g.K) {
        const int c = row / (KD * KH), rem2 = row - c * KD * KH;
        const int kr = rem2 / KH, ka = rem2 - kr * KH;
        const int64_t wi = (int64_t)oc * C * taps + c * taps + kr * p.wR + ka * p.wA + kw;
        if (CONV_DBG_OK(wi, p.w_elems, kStatusBoundsW)) v = p.w[wi];
      }
      ws[i] = v;
    }
    if (tid < kSNcg * kSCO) bias_s[tid] = (p.bias && tid < g.K) ? __ldg(p.bias + tid) : 0.f;
  };
  bool weights_staged = false;
  // The ring is not cleared: the padding columns past W feed only output
  // columns >= OW, which are never stored, and each column's softmax is
  // independent of the others.

  const int owg = lane & 7, cg = lane >> 3;
  const int ow0 = owg * 4;
  const int64_t r_begin = (int64_t)blockIdx.x * p.rows / gridDim.x;
  const int64_t r_end = (int64_t)(blockIdx.x + 1) * p.rows / gridDim.x;
  const uint32_t ring_addr = (uint32_t)__cvta_generic_to_shared(ring);
  const int WQ = p.vec ? g.W / 4 : g.W;  // copy units per row

  for (int64_t r0 = r_begin; r0 < r_end; r0 += kSRows) {
    const int nrows = (int)min64(kSRows, r_end - r0);
    const int64_t n0 = r0 / p.OA;
    __syncthreads();  // the previous block's readers are done with the ring and the row table
    // Shared rows: per image the block touches, its output rows plus KH - 1
    // halo rows.  Thread s fills entry s by walking the (at most a few)
    // image segments of the block.
    const int oh_lo0 = (int)(r0 - n0 * p.OA);
    if (tid < kSMaxSrows) {
      int start = 0, rem = nrows, lo = oh_lo0;
      int64_t n = n0;
      while (rem > 0) {
        const int cnt = min(rem, p.OA - lo);
        const int len = cnt + KH - 1;
        if (tid < start + len) {
          srow_src[tid] = n * g.C * g.D * HW + (int64_t)(lo + tid - start) * p.sA;
          break;
        }
        start += len;
        rem -= cnt;
        ++n;
        lo = 0;
      }
      if (tid == 0) {
        int total = 0;
        for (int rr = nrows, l = oh_lo0; rr > 0; l = 0) {
          const int cnt = min(rr, p.OA - l);
          total += cnt + KH - 1;
          rr -= cnt;
        }
        nsrows_s = total;
      }
    }
    __syncthreads();
    const int nsrows = nsrows_s;

    // Copies of one input plane: thread -> (shared row s, 16-byte unit q),
    // looping over the C channels (fixed strides), so that issuing a plane
    // costs a few instructions per copy and no divisions.
    const int per_plane_sq = nsrows * WQ;
    const int sq0 = tid;
    const int s0 = sq0 < per_plane_sq ? sq0 / WQ : 0, q0 = sq0 - s0 * WQ;
    const int64_t src0 = sq0 < per_plane_sq ? srow_src[s0] + (int64_t)q0 * (p.vec ? 4 : 1) : 0;
    const uint32_t dst0 = 4u * (uint32_t)(s0 * p.WP) + (p.vec ? 16u : 4u) * (uint32_t)q0;
    const int64_t c_stride_src = (int64_t)g.D * HW;
    const uint32_t c_stride_dst = 4u * (uint32_t)(p.srows_max * p.WP);
    int slot_of_next = 0;  // ring slot of the next plane issued (planes are issued in order)
    // one copy of x[src] into the ring (the debug build checks both ends)
    auto copy_in = [&](uint32_t dst, const float *src) {
#ifdef CONVFWD_DEBUG
      const uint32_t nb = p.vec ? 16u : 4u;
      if (!CONV_DBG_OK(src - p.x, p.x_elems, kStatusBoundsX) ||
          !CONV_DBG_OK(src + nb / 4 - 1 - p.x, p.x_elems, kStatusBoundsX) ||
          !CONV_DBG_OK(dst - ring_addr + nb - 1, 4ll * p.ring * p.slot_floats, kStatusBoundsShared))
        return;
#endif
      if (p.vec)
        cp_async16(dst, src);
      else
        cp_async4(dst, src);
    };
    auto issue_plane = [&](int dd) {
      const uint32_t slot = ring_addr + 4u * (uint32_t)slot_of_next * p.slot_floats;
      slot_of_next = (slot_of_next + 1 == p.ring) ? 0 : slot_of_next + 1;
      const int64_t dd_off = (int64_t)dd * p.sR;
      if (sq0 < per_plane_sq) {
        const float *src = p.x + src0 + dd_off;
        uint32_t dst = slot + dst0;
        for (int c = 0; c < C; ++c, src += c_stride_src, dst += c_stride_dst) copy_in(dst, src);
      }
      // rare: more (row, unit) pairs than threads
      for (int i = sq0 + kSThreads; i < per_plane_sq; i += kSThreads) {
        const int si = i / WQ, qi = i - si * WQ;
        const float *src = p.x + srow_src[si] + dd_off + (int64_t)qi * (p.vec ? 4 : 1);
        uint32_t dst = slot + 4u * (uint32_t)(si * p.WP) + (p.vec ? 16u : 4u) * (uint32_t)qi;
        for (int c = 0; c < C; ++c, src += c_stride_src, dst += c_stride_dst) copy_in(dst, src);
      }
      cp_async_commit();
    };
    // the first group's planes: 0 .. nb + KD - 2, one commit group per plane
    int issued = 0;  // commit groups issued in this block (one per plane)
    for (int dd = 0; dd < p.nb + KD - 1 && dd < p.IR; ++dd, ++issued) issue_plane(dd);
    if (!weights_staged) {
      stage_weights();
      weights_staged = true;
    }

    // this lane's output row and its shared-memory row
    const int lr = warp;
    const bool row_ok = lr < nrows;
    const int lrc = row_ok ? lr : nrows - 1;
    const int64_t rabs = r0 + lrc;
    const int64_t n = rabs / p.OA;
    const int oh = (int)(rabs - n * p.OA);
    const int my_srow = lrc + (KH - 1) * (int)(n - n0);

    float mins[kSCO][kR];
#pragma unroll
    for (int o = 0; o < kSCO; ++o)
#pragma unroll
      for (int r = 0; r < kR; ++r) mins[o][r] = INFINITY;

    int s_od = 0;  // ring slot of plane od
    for (int od = 0; od < p.OR; ++od) {
      if ((od % p.nb) == 0 && od > 0) {
        cp_async_wait_all();
        __syncthreads();  // this group's planes are in; the previous group's slots are free
        for (int dd = od + p.nb + KD - 1; dd < od + 2 * p.nb + KD - 1 && dd < p.IR; ++dd) issue_plane(dd);
      } else if (od == 0) {
        // first group: depth 0 starts as soon as its KD planes are in ...
        cp_async_wait_pending(issued - KD);
        __syncthreads();
        for (int dd = p.nb + KD - 1; dd < 2 * p.nb + KD - 1 && dd < p.IR; ++dd, ++issued) issue_plane(dd);
      } else if (od == 1) {
        // ... and depth 1 waits for the rest of the group's planes
        cp_async_wait_pending(issued - (int)min64(p.nb + KD - 1, p.IR));
        __syncthreads();
      }
      // with SKIP, a warp without a row of this block (the CTA's share is
      // smaller than its warp count) only takes part in the copies and barriers
      if (!SKIP || row_ok) {
        // acc2[op][r]: channels (2*op, 2*op + 1) at column r, packed
        unsigned long long acc2[kSCO / 2][kR];
#pragma unroll
        for (int op = 0; op < kSCO / 2; ++op)
#pragma unroll
          for (int r = 0; r < kR; ++r) acc2[op][r] = 0ull;
        const float *xlane = ring + (size_t)my_srow * WP + ow0;
        const float *wlane = ws + cg * kSWStride;
#pragma unroll
        for (int kd = 0; kd < (KDT ? KDT : 1); ++kd) {
          for (int kdr = KDT ? kd : 0; kdr < (KDT ? kd + 1 : KD); ++kdr) {
            int slot = s_od + kdr;
            if (slot >= p.ring) slot -= p.ring;
            const float *xplane = xlane + (size_t)slot * p.slot_floats;
#pragma unroll
            for (int c = 0; c < (CT ? CT : 1); ++c) {
              for (int cr = CT ? c : 0; cr < (CT ? c + 1 : C); ++cr) {
                const float *xc = xplane + cr * SR * WP;
                const float *wc = wlane + ((cr * KD + kdr) * KH) * kSWRow;
#pragma unroll
                for (int kh = 0; kh < (KHT ? KHT : 1); ++kh) {
                  for (int khr = KHT ? kh : 0; khr < (KHT ? kh + 1 : KH); ++khr) {
                    const float *xr = xc + khr * WP;
                    const float4 a = *reinterpret_cast<const float4 *>(xr);
                    const float2 b2 = *reinterpret_cast<const float2 *>(xr + 4);
                    // each input value duplicated into both halves of a pair
                    const unsigned long long xx[6] = {pack2(a.x, a.x), pack2(a.y, a.y), pack2(a.z, a.z),
                                                      pack2(a.w, a.w), pack2(b2.x, b2.x), pack2(b2.y, b2.y)};
                    const float *wt = wc + khr * kSWRow;
#pragma unroll
                    for (int kw = 0; kw < 3; ++kw) {
                      // the tap's 6 channel weights are 3 aligned pairs in shared memory
                      const ulonglong2 q0 = *reinterpret_cast<const ulonglong2 *>(wt + kw * kSWTap);
                      const unsigned long long q1 = *reinterpret_cast<const unsigned long long *>(wt + kw * kSWTap + 4);
                      const unsigned long long wp[kSCO / 2] = {q0.x, q0.y, q1};
#pragma unroll
                      for (int op = 0; op < kSCO / 2; ++op)
#pragma unroll
                        for (int r = 0; r < kR; ++r) fma2(acc2[op][r], wp[op], xx[r + kw]);
                    }
                  }
                }
              }
            }
          }
        }
#pragma unroll
        for (int op = 0; op < kSCO / 2; ++op)
#pragma unroll
          for (int r = 0; r < kR; ++r) {
            float c0, c1;
            unpack2(acc2[op][r], c0, c1);
            mins[2 * op][r] = fminf(mins[2 * op][r], c0);
            mins[2 * op + 1][r] = fminf(mins[2 * op + 1][r], c1);
          }
      }
      s_od = (s_od + 1 == p.ring) ? 0 : s_od + 1;
    }

    // channel softmax per column across the 4 channel-group lanes (xor 8, 16)
    const int64_t OHW = (int64_t)p.OA * g.OW;
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      float v[kSCO];
      float mx = -INFINITY;
#pragma unroll
      for (int o = 0; o < kSCO; ++o) {
        const int oc = cg * kSCO + o;
        v[o] = oc < g.K ? mins[o][r] + bias_s[oc] : -INFINITY;
        mx = fmaxf(mx, v[o]);
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, NOWG));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2 * NOWG));
      float ssum = 0.f;
#pragma unroll
      for (int o = 0; o < kSCO; ++o) {
        v[o] = __expf(v[o] - mx);
        ssum += v[o];
      }
      ssum += __shfl_xor_sync(0xffffffffu, ssum, NOWG);
      ssum += __shfl_xor_sync(0xffffffffu, ssum, 2 * NOWG);
      const float inv = 1.f / ssum;
      const int ow = ow0 + r;
      if (row_ok && ow < g.OW) {
        float *yo = p.y + n * g.K * OHW + (int64_t)oh * g.OW + ow;
#pragma unroll
        for (int o = 0; o < kSCO; ++o) {
          const int oc = cg * kSCO + o;
          if (oc < g.K && CONV_DBG_OK(yo + (int64_t)oc * OHW - p.y, p.y_elems, kStatusBoundsY))
            yo[(int64_t)oc * OHW] = v[o] * inv;
        }
      }
    }
  }
  cp_async_wait_all();
}

// Shared-memory plan of the staged variant; false when it does not apply.
// Batched transpose of the last two dims, in [B][R][C] -> out [B][C][R], in
// 32 x 32 tiles through shared memory (both sides coalesced).  Block 32 x 8.
__global__ void __launch_bounds__(256) transpose_last2_kernel(const float *__restrict__ in, float *__restrict__ out,
                                                             int64_t B, int R, int C) {
  __shared__ float t[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int64_t b = blockIdx.z; b < B; b += gridDim.z) {
    const float *src = in + b * (int64_t)R * C;
    float *dst = out + b * (int64_t)R * C;
    for (int i = threadIdx.y; i < 32; i += 8) {
      const int r = r0 + i, c = c0 + (int)threadIdx.x;
      if (r < R && c < C && CONV_DBG_OK(b * (int64_t)R * C + (int64_t)r * C + c, B * (int64_t)R * C, kStatusBoundsX))
        t[i][threadIdx.x] = src[(int64_t)r * C + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += 8) {
      const int c = c0 + i, r = r0 + (int)threadIdx.x;
      if (r < R && c < C && CONV_DBG_OK(b * (int64_t)R * C + (int64_t)c * R + r, B * (int64_t)R * C, kStatusBoundsWs))
        dst[(int64_t)c * R + r] = t[threadIdx.x][i];
    }
    __syncthreads();
  }
}

cudaError_t launch_transpose_last2(const float *in, float *out, int64_t B, int R, int C, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const dim3 grid((unsigned)((C + 31) / 32), (unsigned)((R + 31) / 32), (unsigned)(B < 65535 ? B : 65535));
  transpose_last2_kernel<<<grid, dim3(32, 8), 0, stream>>>(in, out, B, R, C);
  return cudaGetLastError();
}

// The same problem with H and W exchanged (x and w transposed in their last two dims).
Geom swap_hw(const Geom &g) {
  Geom t = g;
  t.H = g.W, t.W = g.H, t.OH = g.OW, t.OW = g.OH, t.KH = g.KW, t.KW = g.KH;
  t.SH = g.SW, t.SW = g.SH, t.PH = g.PW, t.PW = g.PH, t.DH = g.DW, t.DW = g.DH;
  return t;
}

// The staged kernel's axis fields for the min over depth (2) or height (3).
void staged_axes(const Geom &g, int min_dim, StagedParams *sp) {
  const int64_t HW = (int64_t)g.H * g.W;
  if (min_dim == 2) {
    sp->OR = g.OD, sp->OA = g.OH, sp->KR = g.KD, sp->KA = g.KH, sp->IR = g.D;
    sp->sR = HW, sp->sA = g.W, sp->wR = g.KH * g.KW, sp->wA = g.KW;
  } else {
    sp->OR = g.OH, sp->OA = g.OD, sp->KR = g.KH, sp->KA = g.KD, sp->IR = g.H;
    sp->sR = g.W, sp->sA = HW, sp->wR = g.KW, sp->wA = g.KH * g.KW;
  }
}

bool staged_plan(const Geom &g, const float *x, StagedParams *sp) {
  // sp's axis fields (OR, OA, KR, KA, IR, sR, sA, wR, wA) are filled by the caller
  if (g.K > kSNcg * kSCO || g.OW > 32 || g.KW != 3) return false;
  const int64_t seg = (kSRows - 1) / sp->OA + 2;  // images a block of kSRows rows can touch
  const int64_t srows64 = kSRows + (int64_t)(sp->KA - 1) * seg;
  if (srows64 > kSMaxSrows) return false;
  const int srows = (int)srows64;
  const int WP = (g.W + 3) / 4 * 4 + 4;
  const int64_t w_floats = (int64_t)g.C * sp->KR * sp->KA * kSWRow;
  const int64_t slot = (int64_t)g.C * srows * WP;
  // output depths per block-wide barrier: the largest of 4, 2, 1 whose ring
  // (KD + 2 * nb - 1 planes) fits (6 measured no faster than 4)
  int nb = 0, ring = 0;
  for (const int cand : {4, 2, 1}) {
    ring = sp->KR + 2 * cand - 1;
    const int64_t bytes = 4 * ((w_floats + 3) / 4 * 4 + ring * slot + kRingSlackFloats);
    if (bytes <= kMaxSmemBytes) {
      nb = cand;
      break;
    }
  }
  if (nb < 1) return false;
  sp->nb = nb;
  sp->WP = WP;
  sp->srows_max = srows;
  sp->ring = ring;
  sp->vec = (g.W % 4 == 0) && ((((uintptr_t)x) & 15u) == 0);
  sp->w_floats = (uint32_t)((w_floats + 3) / 4 * 4);
  sp->slot_floats = (uint32_t)slot;
  return true;
}

// Byte offsets of the transposed copies of x and w in the workspace of the min
// over width (256-byte sections).
size_t transpose_x_bytes(const Geom &g) { return ((size_t)g.N * g.C * g.in_spatial() * 4 + 255) / 256 * 256; }
size_t transpose_w_bytes(const Geom &g) { return ((size_t)g.K * g.C * g.taps() * 4 + 255) / 256 * 256; }

template <int NCG, int NROW, int KWT, bool VEC>
cudaError_t launch_t(const FusedParams &p0, cudaStream_t stream) {
  constexpr int NOWG = 32 / (NCG * NROW);
  FusedParams p = p0;
  p.coltiles = (p.OB + NOWG * kR - 1) / (NOWG * kR);
  const int64_t rowgroups = (p.rows + NROW - 1) / NROW;
  const int64_t blocks = rowgroups * p.coltiles;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const size_t smem = sizeof(float) * (size_t)(p.g.C * p.g.taps()) * NCG * kCO;
  CONV_PLAN_CHECK(smem <= (size_t)kMaxSmemBytes && p.g.K <= NCG * kCO && (!KWT || KWT == p.KB));
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
  if (p.KB == 3) {
    const bool vec = p.sB == 1 && (p.IB % 4 == 0) && (p.sA % 4 == 0) && (p.sR % 4 == 0) &&
                     (((int64_t)p.g.D * p.g.H * p.g.W) % 4 == 0) && (((uintptr_t)p.x & 15u) == 0);
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

namespace {
// One thread per (image, position): the channel softmax of a [N][C][plane]
// tensor in place; consecutive threads take consecutive positions, so each
// channel's reads and writes are coalesced.
__global__ void __launch_bounds__(256) channel_softmax_kernel(float *__restrict__ y, int64_t N, int64_t C,
                                                              int64_t plane) {
  const int64_t total = N * plane;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = i / plane, pos = i - n * plane;
    float *q = y + n * C * plane + pos;
    if (!CONV_DBG_OK(q - y, N * C * plane, kStatusBoundsY) ||
        !CONV_DBG_OK(q + (C - 1) * plane - y, N * C * plane, kStatusBoundsY))
      continue;
    float mx = -INFINITY;
    for (int64_t c = 0; c < C; ++c) mx = fmaxf(mx, q[c * plane]);
    float sum = 0.f;
    for (int64_t c = 0; c < C; ++c) sum += expf(q[c * plane] - mx);
    const float inv = 1.f / sum;
    for (int64_t c = 0; c < C; ++c) q[c * plane] = expf(q[c * plane] - mx) * inv;
  }
}
}  // namespace

cudaError_t launch_channel_softmax(float *y, int64_t N, int64_t C, int64_t plane, cudaStream_t stream) {
  const int64_t total = N * plane;
  if (total == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t want = (total + 255) / 256, cap = (int64_t)sms * 8;
  channel_softmax_kernel<<<(unsigned)(want < cap ? want : cap), 256, 0, stream>>>(y, N, C, plane);
  return cudaGetLastError();
}

Geom swap_hw_geom(const Geom &g) { return swap_hw(g); }
size_t transposed_x_bytes(const Geom &g) { return transpose_x_bytes(g); }
size_t transposed_hw_bytes(const Geom &g) { return transpose_x_bytes(g) + transpose_w_bytes(g); }

cudaError_t transpose_hw(const float *x, const float *w, float *ws, const Geom &g, cudaStream_t stream) {
  cudaError_t e = launch_transpose_last2(x, ws, g.N * g.C * g.D, g.H, g.W, stream);
  if (e == cudaSuccess) e = launch_transpose_last2(w, ws + transpose_x_bytes(g) / 4, g.K * g.C * g.KD, g.KH, g.KW, stream);
  return e;
}

bool fused_supported(const Geom &g, int min_dim, const char **why) {
  if (g.K > 8 * kCO) {
    *why = "fused path: C_out above 96";
    return false;
  }
  // the kernel's column axis is W, or H when the min runs over W
  if ((min_dim == 4 ? g.KH : g.KW) > kMaxKW) {
    *why = "fused path: kernel extent along the output's last axis above 7";
    return false;
  }
  const int ncg = pick_ncg(g.K);
  if ((int64_t)g.C * g.taps() * ncg * kCO * 4 > kMaxSmemBytes) {
    *why = "fused path: weights exceed the shared-memory budget";
    return false;
  }
  return true;
}

size_t fused_transpose_bytes(const Geom &g, int min_dim) {
  if (min_dim != 4) return 0;
  // the min over width of (x, w) is the min over height of (x, w) with H and
  // W exchanged, which the staged kernel runs when its shape limits allow
  const Geom t = swap_hw(g);
  StagedParams sp;
  staged_axes(t, 3, &sp);
  if (!staged_plan(t, nullptr, &sp)) return 0;
  return transpose_x_bytes(g) + transpose_w_bytes(g);
}


cudaError_t launch_fused_min_softmax(const float *x, const float *w, const float *bias, float *y,
                                     const Geom &g, int min_dim, cudaStream_t stream, float *ws) {
  if (min_dim == 4 && ws && fused_transpose_bytes(g, 4) > 0) {
    // min over width: transpose x and w in their last two dims into ws, then
    // the min over height of the transposed problem on the staged kernel; its
    // output [N, C_out, OD, OW'] with OW' = OH is exactly y's layout
    const cudaError_t e = transpose_hw(x, w, ws, g, stream);
    if (e != cudaSuccess) return e;
    return launch_fused_min_softmax(ws, ws + transpose_x_bytes(g) / 4, bias, y, swap_hw(g), 3, stream, nullptr);
  }
  FusedParams p;
  p.x = x;
  p.w = w;
  p.bias = bias;
  p.y = y;
  p.g = g;
  p.coltiles = 1;
  // Axis roles.  Tensor dim min_dim of [N, C, D, H, W] is reduced; the output
  // keeps the other two spatial axes in order, the last one contiguous.
  const int64_t HW = (int64_t)g.H * g.W;
  if (min_dim == 2) {  // (R, A, B) = (D, H, W)
    p.OR = g.OD, p.OA = g.OH, p.OB = g.OW;
    p.KR = g.KD, p.KA = g.KH, p.KB = g.KW;
    p.IB = g.W, p.sR = HW, p.sA = g.W, p.sB = 1;
    p.wR = g.KH * g.KW, p.wA = g.KW, p.wB = 1;
  } else if (min_dim == 3) {  // (H, D, W)
    p.OR = g.OH, p.OA = g.OD, p.OB = g.OW;
    p.KR = g.KH, p.KA = g.KD, p.KB = g.KW;
    p.IB = g.W, p.sR = g.W, p.sA = HW, p.sB = 1;
    p.wR = g.KW, p.wA = g.KH * g.KW, p.wB = 1;
  } else {  // min_dim 4: (W, D, H)
    p.OR = g.OW, p.OA = g.OD, p.OB = g.OH;
    p.KR = g.KW, p.KA = g.KD, p.KB = g.KH;
    p.IB = g.H, p.sR = 1, p.sA = HW, p.sB = g.W;
    p.wR = 1, p.wA = g.KH * g.KW, p.wB = g.KW;
  }
  p.rows = g.N * (int64_t)p.OA;
  p.x_elems = g.N * g.C * g.in_spatial() - debug_x_shrink();
  p.w_elems = g.K * g.C * g.taps();
  p.y_elems = g.N * g.K * (int64_t)p.OA * p.OB;
  CONV_PLAN_CHECK(p.OR >= 1 && p.OA >= 1 && p.OB >= 1 && p.KB <= kMaxKW && g.G == 1 && !g.cl);
  CONV_PLAN_CHECK((int64_t)p.OR * p.OA * p.OB == g.out_spatial());
  StagedParams sp;
  // the staged kernel keeps W as its column axis: the min over depth or height
  if (min_dim != 4) staged_axes(g, min_dim, &sp);
  if (min_dim != 4 && staged_plan(g, x, &sp)) {
    sp.x = x;
    sp.w = w;
    sp.bias = bias;
    sp.y = y;
    sp.g = g;
    sp.rows = p.rows;
    sp.x_elems = p.x_elems;
    sp.w_elems = p.w_elems;
    sp.y_elems = p.y_elems;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const size_t smem = 4 * ((size_t)sp.w_floats + (size_t)sp.ring * sp.slot_floats + kRingSlackFloats);
    CONV_PLAN_CHECK(smem <= (size_t)kMaxSmemBytes && sp.nb >= 1 && sp.ring == sp.KR + 2 * sp.nb - 1);
    CONV_PLAN_CHECK(sp.srows_max <= kSMaxSrows && sp.WP >= g.W + 4 && g.KW == 3 && g.K <= kSNcg * kSCO);
    CONV_PLAN_CHECK(!sp.vec || ((g.W % 4) == 0 && ((uintptr_t)x & 15u) == 0));
    // the benchmark shape (C_in 3, kernel 3^3, W 32 -> pitch 36) is specialised: 30 shared
    // rows for the min over depth (blocks span <= 2 images of 30 rows), 32 over height (22)
    const bool spec3 = g.C == 3 && sp.KR == 3 && sp.KA == 3 && sp.WP == 36;
    auto kern = (spec3 && sp.srows_max == 30)   ? fused_min_softmax_staged_kernel<3, 3, 3, 36, 30, false>
                : (spec3 && sp.srows_max == 32) ? fused_min_softmax_staged_kernel<3, 3, 3, 36, 32, true>
                                                : fused_min_softmax_staged_kernel<0, 0, 0, 0, 0, true>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // every SM gets a contiguous share of the rows (processed 26 at a time)
    const int grid = (int)(p.rows < sms ? p.rows : sms);
    kern<<<grid, kSThreads, smem, stream>>>(sp);
    return cudaGetLastError();
  }
  switch (pick_ncg(g.K)) {
    case 1: return launch_ncg<1, 4>(p, stream);
    case 2: return launch_ncg<2, 2>(p, stream);
    case 4: return launch_ncg<4, 1>(p, stream);
    default: return launch_ncg<8, 1>(p, stream);
  }
}

}  // namespace convfwd
