// Implicit-GEMM forward convolution on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators), fp32-accurate through a 3xTF32 split.
//
// The GEMM view is the one the l1_p60 page (turn 1) uses to size the problem:
// rows = output positions (N x OD x OH x OW), columns = output channels, and
// the reduction runs over K = C_in x KD x KH x KW taps of
//   y[n,o,p] = b[o] + sum_{c,k} w[o,c,k] * x[n,c, p*stride + k*dilation - pad]
// (zero padding: taps outside the input contribute 0).  The im2col matrix is
// never materialised in memory: producer warps gather it straight from x
// into tensor memory.
//
// Per CTA (persistent, one per SM, 768 threads):
//   warps 0-3    epilogue: tcgen05.ld the accumulator, add bias, store y
//                (each warp store covers 32 consecutive output positions of
//                one channel, i.e. 128 contiguous bytes)
//   warps 4-19   producers, four groups of four warps.  A thread owns one
//                output position (one TMEM lane) of a 128-row tile; it
//                gathers the position's receptive field for a chunk of K,
//                splits every value into TF32 hi + lo (hi = top 10 mantissa
//                bits, lo = exact remainder) and writes both to TMEM with
//                tcgen05.st.
//   warps 20-23  one per tile slot: the whole warp runs the slot's chunk loop
//                and one elected lane issues its MMAs:
//                D += A_hi*B_hi + A_hi*B_lo + A_lo*B_hi   (M=128, N=C_out pad 32, K=8 per MMA)
// A slot is an independent tile pipeline: its own issuing warp, TMEM
// accumulator and two A stages.  A thread needs ~120-145 cycles to issue one
// tcgen05.mma with N <= 128, so several issuing threads are what keeps the
// tensor pipe busy: four slots when C_out pads to <= 64, else two (TMEM holds
// 512 columns).  Consecutive tiles of a CTA rotate over the slots.
// A (im2col tile) comes from TMEM, B (weights, split hi/lo once per CTA) from
// shared memory in the K-major no-swizzle core-matrix layout.  Hand-off
// between roles uses mbarriers; tcgen05.commit signals MMA completion.  Every
// wait is bounded: on timeout the kernel raises a flag, lets the other roles
// fall through, drains its MMAs and frees TMEM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <atomic>

#include "conv_internal.cuh"
#include "debug_check.cuh"
#include "sm100_ptx.cuh"

namespace convfwd {

__device__ unsigned int g_device_status = 0;

namespace {

constexpr int kTileM = 128;
constexpr int kEpiWarps = 4;
constexpr int kProdGroups = 4;                         // one TMEM A stage per group
constexpr int kMaxSlots = 4;                           // tile pipelines; consecutive tiles rotate over them
constexpr int kMmaWarp = kEpiWarps + 4 * kProdGroups;  // 20: first of the issuer warps (one per slot)
constexpr int kThreads = (kMmaWarp + kMaxSlots) * 32;  // 768
constexpr int kChunkMax = 32;                          // K columns per chunk (registers hold one chunk)
constexpr int kUnit = 16;                              // reduction columns per gather / TMEM store
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxNpad = 128;
constexpr int kMaxSmem = 227 * 1024;
constexpr int kMinSmem = 116 * 1024;  // keeps one CTA per SM, so TMEM allocation never contends
constexpr int kMaxStages = 2 * kMaxSlots;     // two A stages per slot
// a_full, a_empty [stages], d_full, d_empty [slots], b_full [stages] (streamed weights), drain [slots]
constexpr int kNumBars = 3 * kMaxStages + 3 * kMaxSlots;
constexpr long long kWaitLimitCycles = 1ll << 32;  // about two seconds

struct IgemmParams {
  const float *__restrict__ x;
  const float *__restrict__ w;
  const float *__restrict__ bias;
  float *__restrict__ y;
  // the BF16 kernel's tensors (bfloat16 bit patterns); unused by the 3xTF32 kernel
  const uint16_t *__restrict__ xh;
  const uint16_t *__restrict__ wh;
  const uint16_t *__restrict__ bh;
  uint16_t *__restrict__ yh;
  Geom g;
  int64_t M_total;  // N * OD * OH * OW
  int64_t osp;      // OD * OH * OW
  int64_t tiles;    // ceil(M_total / 128)
  int Kred;         // reduction columns of this pass (all of C_in * taps when one pass holds them)
  int Kfull;        // the whole reduction length C_in * taps (row length of w)
  int k_begin;      // first reduction column of this pass
  int accumulate;   // later passes add the accumulator to y instead of the bias
  int64_t y_chans;  // channels per image of y (batch / position stride; all groups and blocks)
  int Kpad;         // padded reduction length of this pass (multiple of 32)
  int Npad;         // C_out rounded up to 32
  int KC;           // K columns per pipeline chunk (multiple of 16)
  int nchunks;      // ceil(Kpad / KC)
  int nslots;       // tile slots (2 or 4), each with an MMA-issuing warp and an accumulator
  int tap_major;    // reduction ordered (tap, c) instead of (c, tap); padded convs with C_in % 4 == 0,
                    // and always for channels-last tensors
  int vec4;         // channels last with 16-byte aligned groups of 4 channels: float4 gathers
  int vec8;         // ... and 32-byte aligned groups of 8 channels: one 32-byte load per 8 columns
                    // (the host picks the kernel instance with that gather form: VEC 1 / 2)
  int vec_store;    // channels last with 16-byte aligned output rows: float4 stores
  uint32_t b_bytes; // Npad * Kpad * 4; with streamed weights the whole B stage region
  // streamed weights: B chunks prepared once (hi then lo, each in the core-matrix
  // layout of one chunk) in a workspace and copied per chunk into the A stage's
  // twin B stage with a bulk copy
  const float *__restrict__ wsp;  // this launch's chunks: chunk q at wsp + q * sb_stage_bytes / 4
  uint32_t sb_stage_bytes;        // 2 * Npad * KC * 4
  // clock cycles after which a pipeline wait gives up (kWaitLimitCycles unless
  // a test shortened it); the waits that guard TMEM release always use
  // kWaitLimitCycles
  long long wait_limit;
  // fused conv3d -> min over depth -> channel softmax (the FUSED kernel): a
  // column is a block of 128 consecutive (image, kept-plane position) pairs
  // of the flattened N x plane index (a block may span two images, so no
  // column is ragged but the last); each CTA runs its columns' R tiles along
  // the reduced dim back to back
  int64_t columns;  // ceil(N * plane / 128)
  // the reduced output axis rdim (0 = depth, 1 = height, 2 = width) has R
  // positions; the kept plane (the other two axes in order, A x nB
  // positions) is what y holds per image and channel
  int R;
  int rdim;
  int64_t plane;
  int nB;
  int fused_min_only;  // a 32-channel block of a wider layer: write min + bias, no softmax
  // fused_slab_kernel: slab columns (padded to 16 / real), the kernel extent
  // along the reduced axis, ring slabs
  int slab_cols, slab_real, slab_kr, nslabs;
  // elements addressable from x / w (or wh) / y (or yh) / wsp as this launch
  // receives them: what the debug build's device checks test indices against
  int64_t x_elems, w_elems, y_elems, ws_elems;
};

struct Plan {
  int Kred, Kpad, Npad, KC, nchunks, nslots, tap_major;
  int kpass;    // reduction columns per pass (multiple of 32); Kred when one pass holds them all
  int npasses;  // ceil(Kred / kpass)
  size_t smem;  // shared memory of a full pass
};

// g.K is the output channels of one launch (<= 128; the host splits wider
// layers into channel blocks).  A reduction whose weights (hi + lo) exceed
// shared memory runs in passes of kpass columns, the later ones adding into y.
bool make_plan(const Geom &g, Plan *pl, const char **why) {
  if (g.K > kMaxNpad) {
    *why = "C_out above 128 in one launch";
    return false;
  }
  if (g.KD > 32 || g.KH > 32 || g.KW > 32) {
    *why = "a kernel dimension above 32";
    return false;
  }
  const int64_t HW = (int64_t)g.H * g.W, DHW = HW * g.D;
  const int64_t tap_span = (int64_t)(g.KD - 1) * g.DD * HW + (int64_t)(g.KH - 1) * g.DH * g.W + (int64_t)(g.KW - 1) * g.DW;
  const int64_t max_off = g.cl ? tap_span * g.G * g.C + (g.C - 1) : (g.C - 1) * DHW + tap_span;
  if (max_off >= (int64_t)1 << 31) {
    *why = "receptive-field offsets of one image exceed 2^31 elements";
    return false;
  }
  const int64_t kred = g.C * (int64_t)g.KD * g.KH * g.KW;
  pl->Kred = (int)kred;
  pl->Kpad = (int)((kred + 31) / 32 * 32);
  pl->Npad = (int)((g.K + 31) / 32 * 32);
  // Reduction order.  (c, kd, kh, kw) keeps a row of KW taps contiguous; with
  // C_in a multiple of 4 the order (kd, kh, kw, c) instead makes every group
  // of 4 consecutive columns share one tap, so a position near the border
  // tests the tap's bounds once per group rather than once per column.  It is
  // used only for padded convolutions: without padding nearly every warp takes
  // the unchecked path, where the channel-major order reads x with better
  // locality (consecutive columns hit the same cache lines).
  pl->tap_major = (g.C % 4 == 0 && (g.PD > 0 || g.PH > 0 || g.PW > 0)) ? 1 : 0;
  // Channels-last tensors: (tap, c) is the weights' memory order and makes
  // consecutive columns consecutive addresses.
  if (g.cl) pl->tap_major = 1;
  // TMEM: one accumulator of Npad columns per slot, then two A stages per
  // slot of KC hi + KC lo columns.  Four slots (four MMA instruction streams)
  // when the accumulators leave room for 16-column stages, else two.
  pl->nslots = (kMaxSlots * pl->Npad + 2 * kMaxSlots * 2 * kUnit <= (int)kTmemCols) ? kMaxSlots : 2;
  int kc = (int)((kTmemCols - pl->nslots * pl->Npad) / (2 * 2 * pl->nslots)) / kUnit * kUnit;
  if (kc > kChunkMax) kc = kChunkMax;
  if (kc > pl->Kpad) kc = pl->Kpad;
  pl->KC = kc;
  // columns per pass: B hi + lo (8 * Npad bytes per column) and the two
  // tables (8 bytes per column) beside the bias and the barriers
  const size_t fixed = (size_t)pl->Npad * 4 + 16 + kNumBars * 8 + 16;
  const int kmax = (int)((kMaxSmem - fixed) / ((size_t)8 * pl->Npad + 8)) / 32 * 32;
  if (kmax < 32) {
    *why = "no reduction pass fits in shared memory";
    return false;
  }
  pl->kpass = pl->Kpad < kmax ? pl->Kpad : kmax;
  pl->npasses = (pl->Kred + pl->kpass - 1) / pl->kpass;
  if (pl->npasses > 1) pl->Kpad = pl->kpass;
  pl->nchunks = (pl->Kpad + kc - 1) / kc;
  const size_t smem = (size_t)2 * pl->Npad * pl->Kpad * 4 + (size_t)pl->Kpad * 8 + fixed;
  pl->smem = smem < (size_t)kMinSmem ? (size_t)kMinSmem : smem;
  return true;
}

// The CTA's tile order: its it-th tile (it = 0, 1, ...) is tile_of(p, it),
// cyclic over the grid so that all SMs sweep the output together.  FUSED:
// the CTA takes columns blockIdx.x, + gridDim.x, ... and runs each column's
// OD depth tiles consecutively; tile id = column * OD + depth.
template <bool FUSED = false>
__device__ __forceinline__ int64_t tile_of(const IgemmParams &p, int64_t it) {
  if (FUSED) {
    const int64_t od = p.R, c = it / od;
    return (blockIdx.x + c * (int64_t)gridDim.x) * od + (it - c * od);
  }
  return blockIdx.x + it * (int64_t)gridDim.x;
}
template <bool FUSED = false>
__device__ __forceinline__ int64_t cta_tile_count(const IgemmParams &p) {
  if (FUSED) return (p.columns - blockIdx.x + gridDim.x - 1) / gridDim.x * p.R;
  return (p.tiles - blockIdx.x + gridDim.x - 1) / gridDim.x;
}

// Bounded mbarrier wait.  Returns false (and raises the abort flag plus the
// device status bit on timeout) when the phase did not complete.  The first
// test is inline; the polling loop, which reads the abort flag and the clock
// every 16 polls (every poll when a test has shortened the limit: one poll
// can block for a few thousand cycles), is out of line so that the roles'
// loops stay short.
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             long long limit, uint32_t site) {
  const long long t0 = clock64();
  const uint32_t check_mask = limit < kWaitLimitCycles ? 0u : 15u;
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & check_mask) == 0) {
      if (*abort_flag) return false;
      if (clock64() - t0 > limit) {
        *abort_flag = 1;
        atomicOr(&g_device_status, kStatusIgemmWatchdog | site);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           long long limit, uint32_t site) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  return wait_phase_slow(bar, parity, abort_flag, limit, site);
}

__device__ __forceinline__ uint32_t tf32_hi_bits(float v) { return __float_as_uint(v) & 0xffffe000u; }

// The n lowest bits set, 0 <= n <= 32 (a kernel extent of 32 taps fills the word).
__device__ __forceinline__ uint32_t low_bits(int n) { return n >= 32 ? 0xffffffffu : (1u << n) - 1u; }

// Columns per in-bounds test of the tested gather: with a tap-major
// reduction over a channel count that is a multiple of 4, the largest of 16,
// 8, 4 dividing C_in (every aligned block of that many columns shares a tap);
// else 1.  The host picks the kernel instance with the same value.
__host__ __device__ __forceinline__ int test_group_cols(int tap_major, int C) {
  return (tap_major && C % 4 == 0) ? (C % 16 == 0 ? 16 : C % 8 == 0 ? 8 : 4) : 1;
}

// One producer thread's output position within a tile.
struct PosInfo {
  const float *xo;      // x at the receptive field's origin (may lie in the padding)
  int64_t xoff;         // the same as an element offset from x
  uint32_t dm, hm, wm;  // bit k set: tap k along D / H / W lands inside the input
  bool valid;           // the position exists (last tile may be partial)
  bool warp_full;       // every lane's receptive field is entirely inside the input
#ifdef CONVFWD_DEBUG
  int64_t xn;           // elements of x the launch may read
#endif
};

// x[xoff + o] (the debug build first checks that the index lies in x)
__device__ __forceinline__ float ldx(const PosInfo &ps, int32_t o) {
#ifdef CONVFWD_DEBUG
  if (!CONV_DBG_OK(ps.xoff + o, ps.xn, kStatusBoundsX)) return 0.f;
#endif
  return __ldg(ps.xo + o);
}

// An output position as mixed-radix digits (image, od, oh, ow); n >= N means
// past the last position.
struct OutPos {
  int64_t n;
  int od, oh, ow;
};

// The digits of flat output index m (divisions).
__device__ __forceinline__ OutPos decode_out(const IgemmParams &p, int64_t m) {
  const Geom &g = p.g;
  OutPos o;
  if (m < ((int64_t)1 << 31) && p.osp < ((int64_t)1 << 31)) {  // 32-bit divisions when they fit
    const uint32_t mm = (uint32_t)m, osp = (uint32_t)p.osp, OHW = (uint32_t)g.OH * (uint32_t)g.OW;
    const uint32_t n32 = mm / osp, pp = mm - n32 * osp;
    o.n = n32;
    o.od = (int)(pp / OHW);
    const uint32_t rem = pp - (uint32_t)o.od * OHW;
    o.oh = (int)(rem / (uint32_t)g.OW);
    o.ow = (int)(rem - (uint32_t)o.oh * (uint32_t)g.OW);
  } else {
    const int64_t OHW = (int64_t)g.OH * g.OW;
    o.n = m / p.osp;
    const int64_t pp = m - o.n * p.osp;
    o.od = (int)(pp / OHW);
    const int rem = (int)(pp - (int64_t)o.od * OHW);
    o.oh = rem / g.OW;
    o.ow = rem - o.oh * g.OW;
  }
  return o;
}

template <bool FUSED = false>
__device__ __forceinline__ PosInfo position_info(const IgemmParams &p, bool valid, int64_t n, int od, int oh,
                                                 int ow);

// The producer-side description of row t of a tile (FUSED: the tile's column
// and reduced index; otherwise 128 consecutive flat output positions).
template <bool FUSED = false>
__device__ __forceinline__ PosInfo decode_position(const IgemmParams &p, int64_t tile, int t) {
  const Geom &g = p.g;
  bool valid;
  int64_t n = 0;
  int od = 0, oh = 0, ow = 0;
  if (FUSED) {
    // tile = column * R + r; row t is entry column * 128 + t of the
    // flattened (image, kept-plane position) index, at index r of the
    // reduced dim; the output coordinates follow from (r, a, b) directly
    const int64_t col = tile / p.R;
    const int64_t r = tile - col * p.R, flat = col * kTileM + t;
    valid = flat < g.N * p.plane;
    int64_t img = 0, pp = 0, a = 0, bb = 0;
    if (valid) {
      if (g.N * p.plane < ((int64_t)1 << 31)) {  // 32-bit divisions when every index fits
        const uint32_t f32 = (uint32_t)flat, pl = (uint32_t)p.plane, nb = (uint32_t)p.nB;
        const uint32_t i32 = f32 / pl, q32 = f32 - i32 * pl, a32 = q32 / nb;
        img = i32, pp = q32, a = a32, bb = q32 - a32 * nb;
      } else {
        img = flat / p.plane, pp = flat - img * p.plane, a = pp / p.nB, bb = pp - a * p.nB;
      }
    }
    // the reduced axis is D, H or W (rdim 0, 1, 2); the kept A and B axes are the other two, in order
    n = img;
    od = (int)(p.rdim == 0 ? r : a);
    oh = (int)(p.rdim == 1 ? r : (p.rdim == 0 ? a : bb));
    ow = (int)(p.rdim == 2 ? r : bb);
  } else {
    const OutPos o = decode_out(p, tile * kTileM + t);
    valid = o.n < g.N;
    if (valid) n = o.n, od = o.od, oh = o.oh, ow = o.ow;
  }
  return position_info<FUSED>(p, valid, n, od, oh, ow);
}

// Receptive-field origin, border masks and the warp-wide interior test of
// output position (n, od, oh, ow); an invalid position reads nothing.
template <bool FUSED>
__device__ __forceinline__ PosInfo position_info(const IgemmParams &p, bool valid, int64_t n, int od, int oh,
                                                 int ow) {
  const Geom &g = p.g;
  PosInfo ps;
  ps.valid = valid;
  const int id0 = od * g.SD - g.PD, ih0 = oh * g.SH - g.PH, iw0 = ow * g.SW - g.PW;
  uint32_t dm = 0, hm = 0, wm = 0;
  if (FUSED || (g.PD == 0 && g.PH == 0 && g.PW == 0)) {
    // no padding: every tap of a valid position lies inside the input (the
    // output size is the largest for which the last tap of the last position does)
    dm = low_bits(g.KD), hm = low_bits(g.KH), wm = low_bits(g.KW);
  } else {
    for (int k = 0; k < g.KD; ++k) dm |= (uint32_t)((unsigned)(id0 + k * g.DD) < (unsigned)g.D) << k;
    for (int k = 0; k < g.KH; ++k) hm |= (uint32_t)((unsigned)(ih0 + k * g.DH) < (unsigned)g.H) << k;
    for (int k = 0; k < g.KW; ++k) wm |= (uint32_t)((unsigned)(iw0 + k * g.DW) < (unsigned)g.W) << k;
  }
  ps.dm = dm;
  ps.hm = hm;
  ps.wm = wm;
  const bool full = ps.valid && dm == low_bits(g.KD) && hm == low_bits(g.KH) && wm == low_bits(g.KW);
  ps.warp_full = __all_sync(0xffffffffu, full);
  const int64_t HW = (int64_t)g.H * g.W;
  const int64_t pos = (int64_t)id0 * HW + (int64_t)ih0 * g.W + iw0;  // may be negative (padding)
  const int64_t xoff = g.cl ? (n * HW * g.D + pos) * (g.G * g.C) : n * g.x_batch_stride() + pos;
  ps.xoff = xoff;
  ps.xo = p.x + (ps.valid ? xoff : 0);
#ifdef CONVFWD_DEBUG
  ps.xn = p.x_elems;
#endif
  return ps;
}

// 16 consecutive reduction columns [k0, k0 + 16) of one output position.
// toff[k]: input offset of column k from the receptive field's origin;
// ttap[k]: kd | kh << 8 | kw << 16 (bit 31: padding column past Kred).
// tg (4, 8 or 16): the reduction runs tap by tap over a channel count that is
// a multiple of tg, so every aligned group of tg columns shares one tap (and
// padding columns come in whole groups): one in-bounds test per group.
// tg = 1: a group of 4 can straddle two taps whose tests differ, and each
// column is tested on its own.
// Warps whose receptive fields are all inside the input read four offsets per
// 16-byte shared load and skip every bounds test; only a unit that reaches the
// padding columns checks them.
// VEC (compile time: each form is its own kernel instance, so that the
// N C D H W gather is compiled without the channels-last forms): 2 = 32-byte
// loads of 8 channels, 1 = 16-byte loads of 4 (channels last), 0 = one load
// per value (any layout).
template <int VEC>
__device__ __forceinline__ void gather_cols(const PosInfo &ps, const int32_t *toff, const uint32_t *ttap, int k0,
                                            int Kred, int tg, float (&v)[kUnit]) {
  if constexpr (VEC == 2) {
    // channels last, C % 8 == 0: columns 8q .. 8q+7 are 8 consecutive channels
    // of one tap, 32-byte aligned: one 32-byte load per group (half the load
    // instructions, and L1 tag lookups, of the 16-byte form)
    bool in = false;
#pragma unroll
    for (int q = 0; q < kUnit / 8; ++q) {
      const int k = k0 + 8 * q;
      if (ps.warp_full) {
        in = k < Kred;
      } else if (q == 0 || tg == 8) {
        const uint32_t e = ttap[k];
        const uint32_t kd = e & 0xffu, kh = (e >> 8) & 0xffu, kw = (e >> 16) & 0xffu;
        in = ps.valid && !(e >> 31) && (((ps.dm >> kd) & (ps.hm >> kh) & (ps.wm >> kw)) & 1u);
      }
      float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#ifdef CONVFWD_DEBUG
      if (in) in = CONV_DBG_OK(ps.xoff + toff[k], ps.xn, kStatusBoundsX) &&
                   CONV_DBG_OK(ps.xoff + toff[k] + 7, ps.xn, kStatusBoundsX);
#endif
      if (in) ptx::ldg_nc_v8(ps.xo + toff[k], a);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[8 * q + j] = a[j];
    }
  } else if constexpr (VEC == 1) {
    // channels last, C % 4 == 0: columns 4q .. 4q+3 are 4 consecutive channels
    // of one tap, 16-byte aligned; one 16-byte load per group, and one test
    // per tg-column block of one tap
    bool in = false;
#pragma unroll
    for (int q = 0; q < kUnit / 4; ++q) {
      const int k = k0 + 4 * q;
      if (ps.warp_full) {
        in = k < Kred;
      } else if (q == 0 || tg == 4 || (q == 2 && tg == 8)) {
        const uint32_t e = ttap[k];
        const uint32_t kd = e & 0xffu, kh = (e >> 8) & 0xffu, kw = (e >> 16) & 0xffu;
        in = ps.valid && !(e >> 31) && (((ps.dm >> kd) & (ps.hm >> kh) & (ps.wm >> kw)) & 1u);
      }
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#ifdef CONVFWD_DEBUG
      if (in) in = CONV_DBG_OK(ps.xoff + toff[k], ps.xn, kStatusBoundsX) &&
                   CONV_DBG_OK(ps.xoff + toff[k] + 3, ps.xn, kStatusBoundsX);
#endif
      if (in) a = __ldg(reinterpret_cast<const float4 *>(ps.xo + toff[k]));
      v[4 * q + 0] = a.x;
      v[4 * q + 1] = a.y;
      v[4 * q + 2] = a.z;
      v[4 * q + 3] = a.w;
    }
  } else {
  if (ps.warp_full) {
    const int4 *o4 = reinterpret_cast<const int4 *>(toff + k0);
    if (k0 + kUnit <= Kred) {
#pragma unroll
      for (int q = 0; q < kUnit / 4; ++q) {
        const int4 o = o4[q];
        v[4 * q + 0] = ldx(ps, o.x);
        v[4 * q + 1] = ldx(ps, o.y);
        v[4 * q + 2] = ldx(ps, o.z);
        v[4 * q + 3] = ldx(ps, o.w);
      }
    } else {
      // the unit reaching the padding columns: groups of 4 wholly past the
      // reduction load nothing (a warp-uniform branch)
#pragma unroll
      for (int q = 0; q < kUnit / 4; ++q) {
        const int k = k0 + 4 * q;
        if (k >= Kred) {
          v[4 * q + 0] = v[4 * q + 1] = v[4 * q + 2] = v[4 * q + 3] = 0.f;
          continue;
        }
        const int4 o = o4[q];
        v[4 * q + 0] = ldx(ps, o.x);
        v[4 * q + 1] = k + 1 < Kred ? ldx(ps, o.y) : 0.f;
        v[4 * q + 2] = k + 2 < Kred ? ldx(ps, o.z) : 0.f;
        v[4 * q + 3] = k + 3 < Kred ? ldx(ps, o.w) : 0.f;
      }
    }
  } else if (tg >= 4) {
    // columns 4q .. 4q+3 of the unit share one tap, and so do the groups of
    // one tg-column block (padding columns come in whole groups, since Kred
    // is then a multiple of tg): a test where a block starts
    const int4 *o4 = reinterpret_cast<const int4 *>(toff + k0);
    bool in = false;
#pragma unroll
    for (int q = 0; q < kUnit / 4; ++q) {
      if (q == 0 || tg == 4 || (q == 2 && tg == 8)) {
        const uint32_t e = ttap[k0 + 4 * q];
        const uint32_t kd = e & 0xffu, kh = (e >> 8) & 0xffu, kw = (e >> 16) & 0xffu;
        in = ps.valid && !(e >> 31) && (((ps.dm >> kd) & (ps.hm >> kh) & (ps.wm >> kw)) & 1u);
      }
      const int4 o = o4[q];
      v[4 * q + 0] = in ? ldx(ps, o.x) : 0.f;
      v[4 * q + 1] = in ? ldx(ps, o.y) : 0.f;
      v[4 * q + 2] = in ? ldx(ps, o.z) : 0.f;
      v[4 * q + 3] = in ? ldx(ps, o.w) : 0.f;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kUnit; ++j) {
      const uint32_t e = ttap[k0 + j];
      const uint32_t kd = e & 0xffu, kh = (e >> 8) & 0xffu, kw = (e >> 16) & 0xffu;
      const bool in = ps.valid && !(e >> 31) && (((ps.dm >> kd) & (ps.hm >> kh) & (ps.wm >> kw)) & 1u);
      v[j] = in ? ldx(ps, toff[k0 + j]) : 0.f;
    }
  }
  }
}

// The fused epilogue (warps 0-3).  Lane tid owns entry column * 128 + tid of
// the flattened (image, kept-plane position) index; over the column's R tiles
// along the reduced dim it keeps min_r conv[n, o, r, pos] for each channel
// o < K <= 32, then adds the bias (min(z + b) = min(z) + b: x -> fl(x + b) is
// monotone), takes the softmax over o with the maximum subtracted, and writes
// y[n, o, pos]: a warp store covers 32 consecutive positions of one channel.
// Tiles rotate over nslots accumulators (tile it in accumulator it % nslots).
__device__ __forceinline__ void fused_epilogue(const IgemmParams &p, uint32_t tmem, uint32_t bar_d_full,
                                               uint32_t bar_d_empty, volatile int *abort_flag, const float *bias_s,
                                               int nslots, int warp, int tid) {
  const Geom &g = p.g;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const int64_t my_tiles = cta_tile_count<true>(p);
  const int R = p.R, K = g.K;  // R: the reduced extent (depth, height or width)
  const int64_t plane = p.plane;
  float mn[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) mn[j] = 0.f;
  for (int64_t it = 0; it < my_tiles; ++it) {
    const uint32_t b = (uint32_t)(it % nslots), rb = (uint32_t)(it / nslots);
    const bool ok = wait_phase(bar_d_full + 8 * b, rb & 1, abort_flag, p.wait_limit, kWaitSiteDFull);
    if (!__all_sync(0xffffffffu, ok)) break;
    ptx::tc_fence_after();
    const int64_t d = it % R;
    // the accumulator in two halves of 16 columns (fewer live registers)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t v[16];
      ptx::tmem_ld16(tmem + lane_base + b * p.Npad + 16 * h, v);
      ptx::tmem_wait_ld();
      if (d == 0) {
#pragma unroll
        for (int j = 0; j < 16; ++j) mn[16 * h + j] = __uint_as_float(v[j]);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) mn[16 * h + j] = fminf(mn[16 * h + j], __uint_as_float(v[j]));
      }
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(bar_d_empty + 8 * b);
    if (d == R - 1) {
      const int64_t flat = tile_of<true>(p, it) / R * kTileM + tid;
      if (flat < g.N * plane) {
        const int64_t img = flat / plane, pp = flat - img * plane;
        // y[n, o, pos]; images are y_chans channels apart (all blocks of a wider layer)
        float *yp = p.y + img * p.y_chans * plane + pp;
#ifdef CONVFWD_DEBUG
        {
          const int64_t i0 = img * p.y_chans * plane + pp;
          if (!CONV_DBG_OK(i0, p.y_elems, kStatusBoundsY) ||
              !CONV_DBG_OK(i0 + (int64_t)(K - 1) * plane, p.y_elems, kStatusBoundsY))
            continue;
        }
#endif
        if (p.fused_min_only) {
          // one block of a layer wider than 32 channels: the softmax over all
          // of them runs afterwards as a pass of its own
          float *q = yp;  // stepped: 32 hoisted 64-bit addresses would spill
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j < K) *q = mn[j] + bias_s[j];
            q += plane;
          }
        } else {
          float mx = -INFINITY;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            mn[j] += bias_s[j];
            if (j < K) mx = fmaxf(mx, mn[j]);
          }
          float sum = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            mn[j] = j < K ? expf(mn[j] - mx) : 0.f;
            sum += mn[j];
          }
          const float inv = 1.f / sum;
          float *q = yp;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j < K) __stcs(q, mn[j] * inv);
            q += plane;
          }
        }
      }
    }
  }
}

// CH: register buffer of one chunk (>= KC): 16 for four slots, 32 for two.
// ACC: a later reduction pass (adds into y; instantiated separately so that
// the single-pass kernels keep their registers).  SB: streamed weights (see
// IgemmParams::wsp): no resident weight matrix, any reduction length in one pass.
// FUSED: the conv3d -> min over depth -> channel softmax of the l2_p24 page
// (turns 1-2): a tile is 128 (image, plane position) pairs at one depth, the
// depth tiles of a column consecutive, and an epilogue that keeps each
// position's running minimum over depth in registers and writes only the
// softmax of the last one.  VEC: the gather form (see gather_cols).  TG: the
// columns per in-bounds test fixed at compile time (0: read at run time).
template <int CH, bool ACC, bool SB, bool FUSED = false, int VEC = 0, int TG = 0>
__global__ void __launch_bounds__(kThreads, 1) igemm_3xtf32_kernel(const IgemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Geom &g = p.g;
  if constexpr (TG != 0) {
    // an instance compiled for another test group does no work and reports
    // like a kernel that gave up (the host never launches one)
    if (TG != test_group_cols(p.tap_major, g.C)) {
      if (threadIdx.x == 0) atomicOr(&g_device_status, kStatusIgemmWatchdog);
      return;
    }
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint8_t *b_hi = smem;              // resident weights: hi [Npad x Kpad]; streamed: the B stages
  uint8_t *b_lo = smem + p.b_bytes;  // resident weights: lo
  int32_t *toff = reinterpret_cast<int32_t *>(smem + (SB ? 1 : 2) * (size_t)p.b_bytes);  // [Kpad]
  uint32_t *ttap = reinterpret_cast<uint32_t *>(toff + p.Kpad);                // [Kpad]
  float *bias_s = reinterpret_cast<float *>(ttap + p.Kpad);
  uint64_t *bars = reinterpret_cast<uint64_t *>((reinterpret_cast<uintptr_t>(bias_s + p.Npad) + 15) & ~(uintptr_t)15);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  const uint32_t bar_a_full = ptx::smem_addr(bars + 0);                                // [stages]
  const uint32_t bar_a_empty = ptx::smem_addr(bars + kMaxStages);                      // [stages]
  const uint32_t bar_d_full = ptx::smem_addr(bars + 2 * kMaxStages);                   // [slots]
  const uint32_t bar_d_empty = ptx::smem_addr(bars + 2 * kMaxStages + kMaxSlots);      // [slots]
  const uint32_t bar_b_full = ptx::smem_addr(bars + 2 * kMaxStages + 2 * kMaxSlots);      // [stages]
  const uint32_t bar_drain = ptx::smem_addr(bars + 3 * kMaxStages + 2 * kMaxSlots);       // [slots]
  const int nslots = p.nslots;

  const uint32_t SBO = (uint32_t)p.Kpad * 32;  // bytes between 8-row groups of B
  const int taps = g.KD * g.KH * g.KW;
  const int64_t HW = (int64_t)g.H * g.W, DHW = HW * g.D;

  // ---- weights -> shared memory, split into TF32 hi / lo.  Word i of the
  // core-matrix layout holds B[n][k] with n = 8*(cm / (Kpad/4)) + row,
  // k = 4*(cm % (Kpad/4)) + col, so consecutive threads write consecutive
  // words (conflict-free).
  {
    const int kq = p.Kpad / 4;
    const int words = SB ? 0 : p.Npad * p.Kpad;  // streamed weights arrive per chunk
    for (int i = tid; i < words; i += kThreads) {
      const int cm = i >> 5, r = (i >> 2) & 7, cw = i & 3;
      const int n = (cm / kq) * 8 + r, k = (cm % kq) * 4 + cw;
      // w is [C_out][C_in][taps]; GEMM column kg = k_begin + k maps to (c, t) by the reduction order
      const int kg = p.k_begin + k;
      int kmem = kg;
      if (p.tap_major && !g.cl && k < p.Kred) {
        const int t = kg / g.C;
        kmem = (kg - t * g.C) * taps + t;
      }
      float v = 0.f;
      if (n < g.K && k < p.Kred && CONV_DBG_OK((int64_t)n * p.Kfull + kmem, p.w_elems, kStatusBoundsW))
        v = __ldg(p.w + (int64_t)n * p.Kfull + kmem);
      const float hi = __uint_as_float(tf32_hi_bits(v));
      reinterpret_cast<float *>(b_hi)[i] = hi;
      reinterpret_cast<float *>(b_lo)[i] = v - hi;
    }
    // ---- reduction column -> (input offset, tap coordinates)
    for (int kk = tid; kk < p.Kpad; kk += kThreads) {
      if (kk < p.Kred) {
        const int kg = p.k_begin + kk;
        int c, t;
        if (p.tap_major) {
          t = kg / g.C;
          c = kg - t * g.C;
        } else {
          c = kg / taps;
          t = kg - c * taps;
        }
        const int kw = t % g.KW, khd = t / g.KW;
        const int kd = khd / g.KH, kh = khd - kd * g.KH;
        const int64_t tpos = (int64_t)kd * g.DD * HW + (int64_t)kh * g.DH * g.W + (int64_t)kw * g.DW;
        toff[kk] = (int32_t)(g.cl ? tpos * (g.G * g.C) + c : c * DHW + tpos);
        ttap[kk] = (uint32_t)kd | ((uint32_t)kh << 8) | ((uint32_t)kw << 16);
      } else {
        toff[kk] = 0;
        ttap[kk] = 0x80000000u;  // padding: contributes zero
      }
    }
    for (int i = tid; i < p.Npad; i += kThreads)
      bias_s[i] = (p.bias && !ACC && i < g.K) ? __ldg(p.bias + i) : 0.f;
  }
  ptx::fence_proxy_async_smem();
  if (warp == kMmaWarp) ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
  if (tid == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      ptx::mbar_init(bar_a_full + 8 * s, 128);
      ptx::mbar_init(bar_a_empty + 8 * s, 1);
      ptx::mbar_init(bar_b_full + 8 * s, 1);
    }
    for (int b = 0; b < kMaxSlots; ++b) {
      ptx::mbar_init(bar_drain + 8 * b, 1);
      ptx::mbar_init(bar_d_full + 8 * b, 1);
      ptx::mbar_init(bar_d_empty + 8 * b, 128);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // slot b's accumulator at column b * Npad; A stage s: hi at a_col0 + 2*KC*s, lo at + KC.
  // Slot b owns stages 2b and 2b + 1; it is served by kProdGroups / nslots
  // producer groups.
  const uint32_t a_col0 = (uint32_t)(nslots * p.Npad);

  if (FUSED && warp < kEpiWarps) {
    fused_epilogue(p, tmem, bar_d_full, bar_d_empty, abort_flag, bias_s, nslots, warp, tid);
  } else if (warp < kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int64_t my_tiles = cta_tile_count(p);
    for (int64_t it = 0; it < my_tiles; ++it) {
      const int64_t tile = tile_of(p, it);
      const uint32_t b = (uint32_t)(it % nslots), rb = (uint32_t)(it / nslots);
      bool ok = wait_phase(bar_d_full + 8 * b, rb & 1, abort_flag, p.wait_limit, kWaitSiteDFull);
      if (!__all_sync(0xffffffffu, ok)) break;
      ptx::tc_fence_after();
      const int64_t m = tile * kTileM + tid;
      const bool valid = m < p.M_total;
      int64_t n = 0, pp = 0;
      if (valid) {
        if (p.M_total < ((int64_t)1 << 31)) {
          n = (uint32_t)m / (uint32_t)p.osp;
          pp = m - n * p.osp;
        } else {
          n = m / p.osp;
          pp = m - n * p.osp;
        }
      }
      // y[n, o, pos] (batch stride spans all groups' channels), or y[n, pos, o] channels last
      float *yp = g.cl ? p.y + (n * p.osp + pp) * p.y_chans : p.y + n * p.y_chans * p.osp + pp;
      // y[n, c0 + j, pos] = accumulator column c0 + j + bias, j < 32: a warp
      // store covers 32 consecutive positions of one channel.
      auto store32 = [&](const uint32_t (&v)[32], int c0) {
#ifdef CONVFWD_DEBUG
        {
          // this lane's stores of channels c0 .. c0 + 31 (< K): first and last index
          const int64_t i0 = (yp - p.y) + (g.cl ? (int64_t)c0 : (int64_t)c0 * p.osp);
          const int nk = min(32, (int)g.K - c0);
          const int64_t i1 = i0 + (int64_t)(nk - 1) * (g.cl ? 1 : p.osp);
          if (nk > 0 && (!CONV_DBG_OK(i0, p.y_elems, kStatusBoundsY) || !CONV_DBG_OK(i1, p.y_elems, kStatusBoundsY)))
            return;
        }
#endif
        if (ACC) {
          // a later reduction pass: add to what the earlier passes stored
          const int64_t ostride = g.cl ? 1 : p.osp;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int o = c0 + j;
            if (o < g.K) yp[o * ostride] += __uint_as_float(v[j]);
          }
          return;
        }
        if (g.cl) {
          // one position's channels are contiguous: 16-byte stores when aligned
          if (p.vec_store && c0 + 32 <= g.K) {
            float4 *q4 = reinterpret_cast<float4 *>(yp + c0);
            const float4 *b4 = reinterpret_cast<const float4 *>(bias_s + c0);
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const float4 bb = b4[j4];
              __stcs(q4 + j4, make_float4(__uint_as_float(v[4 * j4 + 0]) + bb.x, __uint_as_float(v[4 * j4 + 1]) + bb.y,
                                          __uint_as_float(v[4 * j4 + 2]) + bb.z, __uint_as_float(v[4 * j4 + 3]) + bb.w));
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int o = c0 + j;
              if (o < g.K) __stcs(yp + o, __uint_as_float(v[j]) + bias_s[o]);
            }
          }
          return;
        }
        if (c0 + 32 <= g.K) {
          float *q = yp + (int64_t)c0 * p.osp;
          const float4 *b4 = reinterpret_cast<const float4 *>(bias_s + c0);
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 bb = b4[j4];
            __stcs(q, __uint_as_float(v[4 * j4 + 0]) + bb.x);
            q += p.osp;
            __stcs(q, __uint_as_float(v[4 * j4 + 1]) + bb.y);
            q += p.osp;
            __stcs(q, __uint_as_float(v[4 * j4 + 2]) + bb.z);
            q += p.osp;
            __stcs(q, __uint_as_float(v[4 * j4 + 3]) + bb.w);
            q += p.osp;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int o = c0 + j;
            if (o < g.K) __stcs(yp + (int64_t)o * p.osp, __uint_as_float(v[j]) + bias_s[o]);
          }
        }
      };
      // 32 accumulator columns at a time; the accumulator is released after
      // the last read, before the last stores.
      for (int c0 = 0; c0 < p.Npad; c0 += 32) {
        uint32_t v[32];
        ptx::tmem_ld32(tmem + lane_base + b * p.Npad + c0, v);
        ptx::tmem_wait_ld();
        if (c0 + 32 >= p.Npad) {
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar_d_empty + 8 * b);
        }
        if (valid) store32(v, c0);
      }
    }
  } else if (warp < kMmaWarp) {
    // ------------------------------------------------------------ producers
    // Group grp serves slot grp / gps (the CTA's tiles it = slot, slot +
    // nslots, ...): it takes the slot's chunks lg = sel, sel + gps, ... and
    // puts chunk lg in the slot's stage lg & 1.  A chunk's loads are issued
    // before waiting for its stage to drain.
    const int grp = (warp - kEpiWarps) >> 2;
    const int gps = kProdGroups / nslots;  // producer groups per slot (1 or 2)
    const int slot = grp / gps, sel = grp - slot * gps;
    const int t = tid - 32 * kEpiWarps - 128 * grp;  // TMEM lane / row of the tile
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int64_t my_tiles = cta_tile_count<FUSED>(p);
    const int64_t slot_tiles = (my_tiles - slot + nslots - 1) / nslots;  // it = slot, slot + nslots, ...
    // columns per in-bounds test of the tested gather: the largest of 16, 8, 4
    // dividing C_in when the reduction is tap-major (warp-uniform)
    const int tg = TG != 0 ? TG : test_group_cols(p.tap_major, g.C);  // compile time where TG is given
    // Chunk q of a tile: gather its K columns into registers (loads only).
    auto gather_chunk = [&](const PosInfo &ps, int q, float (&v)[CH]) {
      const int k0 = q * p.KC;
      const int ncols = min(p.KC, p.Kpad - k0);
#pragma unroll
      for (int u = 0; u < CH / kUnit; ++u) {
        if (u * kUnit < ncols) {
          float (&vu)[kUnit] = *reinterpret_cast<float (*)[kUnit]>(v + u * kUnit);
          gather_cols<VEC>(ps, toff, ttap, k0 + u * kUnit, p.Kred, tg, vu);
        }
      }
    };
    // Slot-local chunk lg (= chunk q of its tile): wait for its stage to
    // drain, split into hi / lo, store both to TMEM and signal the issuer.
    // The lo part overwrites v in place (keeps the chunk within the register
    // budget without spills).  False when the wait timed out.  full: the
    // chunk is known to hold KC columns (no per-unit column test).
    // streamed weights: the group's thread 0 brings chunk q's B into the
    // stage; it remembers its last copy to wait for it before leaving
    int sb_last_stage = -1;
    uint32_t sb_last_parity = 0;
    auto put_chunk = [&](uint32_t lg, int q, float (&v)[CH], bool full = false) -> bool {
      const int stage = 2 * slot + (int)(lg & 1);
      const uint32_t a_hi_col = a_col0 + (uint32_t)(2 * p.KC * stage);
      const uint32_t a_lo_col = a_hi_col + (uint32_t)p.KC;
      const int ncols = min(p.KC, p.Kpad - q * p.KC);
      const uint32_t r = (uint32_t)(lg >> 1);
      const bool ok = wait_phase(bar_a_empty + 8 * stage, (r & 1) ^ 1, abort_flag, p.wait_limit, kWaitSiteAEmpty);
      if (!__all_sync(0xffffffffu, ok)) return false;
      ptx::tc_fence_after();
      if (SB && t == 0) {
        // the stage's MMAs are done: its B half is free too
        const int64_t w0 = (int64_t)q * (p.sb_stage_bytes / 4);
        if (CONV_DBG_OK(w0 + p.sb_stage_bytes / 4 - 1, p.ws_elems, kStatusBoundsWs)) {
          ptx::mbar_arrive_expect_tx(bar_b_full + 8 * stage, p.sb_stage_bytes);
          ptx::bulk_copy_g2s(ptx::smem_addr(b_hi + (size_t)stage * p.sb_stage_bytes), p.wsp + w0, p.sb_stage_bytes,
                             bar_b_full + 8 * stage);
        } else {
          ptx::mbar_arrive(bar_b_full + 8 * stage);  // (debug build) the copy is dropped
        }
        sb_last_stage = stage;
        sb_last_parity = r & 1;
      }
#pragma unroll
      for (int u = 0; u < CH / kUnit; ++u) {
        if (full || u * kUnit < ncols) {
#pragma unroll
          for (int h = 0; h < kUnit; h += 8) {
            uint32_t tmp[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) tmp[j] = tf32_hi_bits(v[u * kUnit + h + j]);
            ptx::tmem_st8(tmem + lane_base + a_hi_col + (uint32_t)(u * kUnit + h), tmp);
#pragma unroll
            for (int j = 0; j < 8; j += 2)
              ptx::sub_f32x2(v[u * kUnit + h + j], v[u * kUnit + h + j + 1], __uint_as_float(tmp[j]),
                             __uint_as_float(tmp[j + 1]), v[u * kUnit + h + j], v[u * kUnit + h + j + 1]);
            ptx::tmem_st8(tmem + lane_base + a_lo_col + (uint32_t)(u * kUnit + h),
                          *reinterpret_cast<const uint32_t (*)[8]>(v + u * kUnit + h));
          }
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar_a_full + 8 * stage);
      return true;
    };
    // full chunks of a warp whose receptive fields are all inside the input:
    // four offsets per shared load, no tests
    auto gather_full = [&](const PosInfo &ps, int q, float (&v)[CH]) {
      const int4 *o4 = reinterpret_cast<const int4 *>(toff + q * CH);
#pragma unroll
      for (int i = 0; i < CH / 4; ++i) {
        const int4 o = o4[i];
        v[4 * i + 0] = ldx(ps, o.x);
        v[4 * i + 1] = ldx(ps, o.y);
        v[4 * i + 2] = ldx(ps, o.z);
        v[4 * i + 3] = ldx(ps, o.w);
      }
    };
    const int nfull = (p.KC == CH && VEC == 0) ? p.Kred / CH : 0;  // chunks entirely inside the reduction
    bool aborted = false;
    for (int64_t li = 0; li < slot_tiles && !aborted; ++li) {
      const PosInfo ps = decode_position<FUSED>(p, tile_of<FUSED>(p, li * nslots + slot), t);
      // slot-local index of the tile's first chunk; only its low bits matter
      // (stage and phase parity), so 32-bit arithmetic (wrapping) serves
      const uint32_t lg0 = (uint32_t)li * (uint32_t)p.nchunks;
      // this group's chunks of the tile: lg = lg0 + q with lg = sel (mod gps)
      int q = (int)((sel - (int)(lg0 % (uint32_t)gps) + gps) % gps);
      if (CH == 16 && ps.warp_full) {
        for (; q < nfull; q += gps) {
          float v[CH];
          gather_full(ps, q, v);
          if (!put_chunk(lg0 + q, q, v, true)) {
            aborted = true;
            break;
          }
        }
        if (aborted) break;
      }
      for (; q < p.nchunks; q += gps) {
        float v[CH];
        // 32-column chunks have no loop of their own (a second copy of the
        // loop spills): interior warps pick the unchecked gather per chunk
        if (CH == 32 && ps.warp_full && q < nfull)
          gather_full(ps, q, v);
        else
          gather_chunk(ps, q, v);
        if (!put_chunk(lg0 + q, q, v)) {
          aborted = true;
          break;
        }
      }
    }
    if (SB && sb_last_stage >= 0) {
      // no bulk copy of ours may still be landing when the CTA exits (bounded)
      const long long t0 = clock64();
      while (!ptx::mbar_try_wait(bar_b_full + 8 * sb_last_stage, sb_last_parity) && clock64() - t0 < kWaitLimitCycles) {
      }
    }
  } else if (warp >= kMmaWarp && warp - kMmaWarp < nslots) {
    // ------------------------------------------------------------ MMA issuers
    // One warp per slot, on different SM sub-partitions: a thread cannot issue
    // a tcgen05.mma much faster than one per ~140 cycles, so the slots keep
    // two or four instruction streams (tiles) in flight.  The whole warp runs
    // the loop (its values stay warp-uniform); one elected lane issues.
    // Per K-step: D += A_hi*B_hi + A_hi*B_lo + A_lo*B_hi.
    const int slot = __shfl_sync(0xffffffffu, warp - kMmaWarp, 0);
    const uint32_t idesc = ptx::idesc_tf32(kTileM, (uint32_t)p.Npad);
    const uint32_t bhi = ptx::smem_addr(b_hi), blo = ptx::smem_addr(b_lo);
    const uint32_t d_tmem = tmem + (uint32_t)(slot * p.Npad);
    const int64_t my_tiles = cta_tile_count<FUSED>(p);
    bool aborted = false;
    for (int64_t it = slot; it < my_tiles && !aborted; it += nslots) {
      const int64_t li = it / nslots;
      if (!__all_sync(0xffffffffu, wait_phase(bar_d_empty + 8 * slot, ((uint32_t)li & 1) ^ 1, abort_flag, p.wait_limit,
                                                  kWaitSiteDEmpty))) break;
      ptx::tc_fence_after();
      for (int q = 0; q < p.nchunks; ++q) {
        const uint32_t lg = (uint32_t)li * (uint32_t)p.nchunks + (uint32_t)q;
        const uint32_t s = (uint32_t)(2 * slot + (int)(lg & 1)), r = (uint32_t)(lg >> 1);
        bool ok = wait_phase(bar_a_full + 8 * s, r & 1, abort_flag, p.wait_limit, kWaitSiteAFull);
        if (SB && ok) ok = wait_phase(bar_b_full + 8 * s, r & 1, abort_flag, p.wait_limit, kWaitSiteBFull);
        if (!__all_sync(0xffffffffu, ok)) {
          aborted = true;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a_hi = tmem + a_col0 + 2u * (uint32_t)p.KC * s;
        const uint32_t a_lo = a_hi + (uint32_t)p.KC;
        const int k0 = q * p.KC;
        const int ksteps = min(p.KC, p.Kpad - k0) / 8;
        // streamed: the stage holds chunk q only (hi, then lo), 8-row groups KC * 32 bytes apart
        const uint32_t sb_hi = bhi + s * p.sb_stage_bytes, sb_lo = sb_hi + p.sb_stage_bytes / 2;
        if (ptx::elect_one()) {
          for (int ks = 0; ks < ksteps; ++ks) {
            const uint32_t kbyte = (uint32_t)(k0 + ks * 8) * 32u;  // (k/4) core matrices of 128 B
            const uint64_t dh = SB ? ptx::smem_desc_noswizzle(sb_hi + 256u * ks, 128, (uint32_t)p.KC * 32)
                                   : ptx::smem_desc_noswizzle(bhi + kbyte, 128, SBO);
            const uint64_t dl = SB ? ptx::smem_desc_noswizzle(sb_lo + 256u * ks, 128, (uint32_t)p.KC * 32)
                                   : ptx::smem_desc_noswizzle(blo + kbyte, 128, SBO);
            ptx::mma_tf32_ts(d_tmem, a_hi + 8 * ks, dh, idesc, (q | ks) != 0);
            ptx::mma_tf32_ts(d_tmem, a_hi + 8 * ks, dl, idesc, 1);
            ptx::mma_tf32_ts(d_tmem, a_lo + 8 * ks, dh, idesc, 1);
          }
          ptx::mma_commit(bar_a_empty + 8 * s);
        }
        __syncwarp();
      }
      if (aborted) break;
      if (ptx::elect_one()) ptx::mma_commit(bar_d_full + 8 * slot);
      __syncwarp();
    }
    if (*abort_flag) {
      // drain: every MMA this warp issued completes before TMEM is released
      if (ptx::elect_one()) {
        ptx::mma_commit(bar_drain + 8 * slot);
        const long long t0 = clock64();
        while (!ptx::mbar_try_wait(bar_drain + 8 * slot, 0) && clock64() - t0 < kWaitLimitCycles) {
        }
      }
      __syncwarp();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Streamed weights, prepared once per call: chunk q of the reduction (KC
// columns) as the tensor cores read it from shared memory, hi then lo, each
// [Npad x KC] in core matrices of 8 rows x 4 floats (LBO 128 bytes along K,
// SBO KC * 32 bytes along N).  Column kg maps to w's memory order as in the
// kernel's resident staging.
__global__ void split_weights_kernel(const float *__restrict__ w, float *__restrict__ ws, int K, int C, int taps,
                                     int Kfull, int Npad, int KC, int nchunks, int tap_major, int64_t w_elems,
                                     int64_t ws_elems) {
  const int64_t per_chunk = (int64_t)Npad * KC;
  const int64_t total = per_chunk * nchunks;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int q = (int)(i / per_chunk);
    const int e = (int)(i - (int64_t)q * per_chunk);
    const int n = e / KC, kl = e - n * KC;
    const int kg = q * KC + kl;
    float v = 0.f;
    if (n < K && kg < Kfull) {
      int kmem = kg;
      if (tap_major) {
        const int t = kg / C;
        kmem = (kg - t * C) * taps + t;
      }
      if (CONV_DBG_OK((int64_t)n * Kfull + kmem, w_elems, kStatusBoundsW)) v = __ldg(w + (int64_t)n * Kfull + kmem);
    }
    const float hi = __uint_as_float(tf32_hi_bits(v));
    const int64_t o = ((int64_t)(n / 8) * (KC / 4) + kl / 4) * 32 + (n % 8) * 4 + (kl % 4);
    const int64_t c0 = (int64_t)q * 2 * per_chunk;
    if (!CONV_DBG_OK(c0 + o, ws_elems, kStatusBoundsWs) || !CONV_DBG_OK(c0 + per_chunk + o, ws_elems, kStatusBoundsWs))
      continue;
    float *chunk = ws + c0;
    chunk[o] = hi;
    chunk[per_chunk + o] = v - hi;
  }
}

// The fused op with slabs (launched when a slab fits: see fused_slab_plan).
// Along the reduced axis, tile d of a column reads input planes d .. d + KR - 1
// (KR: the kernel extent along that axis; stride 1, no padding).  The
// receptive-field columns one plane contributes, (c, ka, kb) over the other
// two kernel dims -- a slab -- are the same for the KR tiles that read the
// plane, so each plane's slab is gathered once into a ring of NS slabs in TMEM
// and tile d accumulates sum_kr A(slab d + kr) * B_kr, with B_kr the weights
// at kernel offset kr along the reduced axis (resident in shared memory, split
// into TF32 hi / lo).  The four producer groups fill slabs round-robin; a
// slab's ring slot is free again once its KR readers' MMAs have completed
// (edge planes with fewer readers pre-arrive the missing counts).  The
// epilogue is the fused one; the MMAs are the 3xTF32 products of the main
// kernel.
__global__ void __launch_bounds__(kThreads, 1) fused_slab_kernel(const IgemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Geom &g = p.g;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int Sp = p.slab_cols, Sc = p.slab_real, KR = p.slab_kr, NS = p.nslabs;
  const int rd = p.rdim;
  const int KA = rd == 0 ? g.KH : g.KD, KB = rd == 2 ? g.KH : g.KW;
  const int64_t HW = (int64_t)g.H * g.W, DHW = HW * g.D;
  // input strides along the reduced axis and the kept A and B axes
  const int64_t sRin = rd == 0 ? HW : rd == 1 ? (int64_t)g.W : 1;
  const int64_t sAin = rd == 0 ? (int64_t)g.W : HW;
  const int64_t sBin = rd == 2 ? (int64_t)g.W : 1;
  const uint32_t blk_bytes = (uint32_t)(p.Npad * Sp * 4);  // one weight block (hi or lo)

  uint8_t *b_hi = smem;                 // [KR][Npad x Sp] core-matrix layout
  uint8_t *b_lo = smem + p.b_bytes;     // b_bytes = KR * blk_bytes
  int32_t *toff = reinterpret_cast<int32_t *>(smem + 2 * (size_t)p.b_bytes);  // [Sp]
  float *bias_s = reinterpret_cast<float *>(toff + Sp);
  uint64_t *bars = reinterpret_cast<uint64_t *>((reinterpret_cast<uintptr_t>(bias_s + p.Npad) + 15) & ~(uintptr_t)15);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  const uint32_t bar_s_full = ptx::smem_addr(bars + 0);                           // [NS]
  const uint32_t bar_s_empty = ptx::smem_addr(bars + kMaxStages);                 // [NS]
  const uint32_t bar_d_full = ptx::smem_addr(bars + 2 * kMaxStages);              // [slots]
  const uint32_t bar_d_empty = ptx::smem_addr(bars + 2 * kMaxStages + kMaxSlots);  // [slots]
  const uint32_t bar_drain = ptx::smem_addr(bars + 3 * kMaxStages + 2 * kMaxSlots);
  constexpr int nslots = kMaxSlots;

  // ---- weights: block kr, word i -> B[n][k] as in the main kernel (Kpad = Sp)
  {
    const int kq = Sp / 4, per_blk = p.Npad * Sp;
    const int taps = g.KD * g.KH * g.KW;
    for (int i = tid; i < KR * per_blk; i += kThreads) {
      const int blk = i / per_blk, e = i - blk * per_blk;
      const int cm = e >> 5, r = (e >> 2) & 7, cw = e & 3;
      const int n = (cm / kq) * 8 + r, k = (cm % kq) * 4 + cw;
      float v = 0.f;
      if (n < g.K && k < Sc) {
        const int c = k / (KA * KB), rem = k - c * KA * KB, ka = rem / KB, kb = rem - ka * KB;
        const int kd = rd == 0 ? blk : ka, kh = rd == 0 ? ka : rd == 1 ? blk : kb, kw = rd == 2 ? blk : kb;
        const int64_t wi = (int64_t)n * p.Kfull + (int64_t)c * taps + (kd * g.KH + kh) * g.KW + kw;
        if (CONV_DBG_OK(wi, p.w_elems, kStatusBoundsW)) v = __ldg(p.w + wi);
      }
      const float hi = __uint_as_float(tf32_hi_bits(v));
      reinterpret_cast<float *>(b_hi)[i] = hi;
      reinterpret_cast<float *>(b_lo)[i] = v - hi;
    }
    for (int k = tid; k < Sp; k += kThreads) {
      int32_t o = 0;
      if (k < Sc) {
        const int c = k / (KA * KB), rem = k - c * KA * KB, ka = rem / KB, kb = rem - ka * KB;
        o = (int32_t)(c * DHW + ka * sAin + kb * sBin);
      }
      toff[k] = o;
    }
    for (int i = tid; i < p.Npad; i += kThreads) bias_s[i] = (p.bias && i < g.K) ? __ldg(p.bias + i) : 0.f;
  }
  ptx::fence_proxy_async_smem();
  if (warp == kMmaWarp) ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
  if (tid == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      ptx::mbar_init(bar_s_full + 8 * s, 128);
      ptx::mbar_init(bar_s_empty + 8 * s, (uint32_t)KR);
    }
    for (int b = 0; b < kMaxSlots; ++b) {
      ptx::mbar_init(bar_drain + 8 * b, 1);
      ptx::mbar_init(bar_d_full + 8 * b, 1);
      ptx::mbar_init(bar_d_empty + 8 * b, 128);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM: accumulator b at column b * Npad; slab s at slab_col0 + 2 * Sp * s (hi), + Sp (lo)
  const uint32_t slab_col0 = (uint32_t)(nslots * p.Npad);
  const int64_t ncols = (p.columns - blockIdx.x + gridDim.x - 1) / gridDim.x;  // this CTA's columns
  const int P = p.R + KR - 1;                                                   // input planes per column

  if (warp < kEpiWarps) {
    fused_epilogue(p, tmem, bar_d_full, bar_d_empty, abort_flag, bias_s, nslots, warp, tid);
  } else if (warp < kMmaWarp) {
    // ------------------------------------------------------------ producers
    const int grp = (warp - kEpiWarps) >> 2;
    const int t = tid - 32 * kEpiWarps - 128 * grp;  // TMEM lane / row of the tile
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    int64_t cur_j = -1, base = 0;
    bool valid = false;
    const int64_t total = ncols * P;
    for (int64_t sidx = grp; sidx < total; sidx += kProdGroups) {
      const int64_t j = sidx / P;
      const int pl = (int)(sidx - j * P);
      if (j != cur_j) {
        // row t of column j: entry col * 128 + t of the flattened (image, kept position) index
        cur_j = j;
        const int64_t flat = (blockIdx.x + j * (int64_t)gridDim.x) * kTileM + t;
        valid = flat < g.N * p.plane;
        const int64_t img = valid ? flat / p.plane : 0, pp = valid ? flat - img * p.plane : 0;
        const int64_t a = pp / p.nB, bb = pp - a * p.nB;
        base = img * g.x_batch_stride() + a * sAin + bb * sBin;
      }
      const int64_t xoff = base + (int64_t)pl * sRin;
      const uint32_t s = (uint32_t)(sidx % NS), q = (uint32_t)(sidx / NS);
      const bool ok = wait_phase(bar_s_empty + 8 * s, (q & 1) ^ 1, abort_flag, p.wait_limit, kWaitSiteAEmpty);
      if (!__all_sync(0xffffffffu, ok)) break;
      ptx::tc_fence_after();
      const uint32_t col = slab_col0 + 2u * (uint32_t)Sp * s;
      const float *xo = p.x + (valid ? xoff : 0);
      for (int u = 0; u < Sp / kUnit; ++u) {
        float v[kUnit];
        const int4 *o4 = reinterpret_cast<const int4 *>(toff + u * kUnit);
#pragma unroll
        for (int q = 0; q < kUnit / 4; ++q) {
          // four offsets per shared load; columns past the slab (and invalid rows) read nothing
          const int k = u * kUnit + 4 * q;
          const int4 o = o4[q];
          const int oo[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x = 0.f;
            if (valid && k + e < Sc && CONV_DBG_OK(xoff + oo[e], p.x_elems, kStatusBoundsX)) x = __ldg(xo + oo[e]);
            v[4 * q + e] = x;
          }
        }
#pragma unroll
        for (int h = 0; h < kUnit; h += 8) {
          uint32_t tmp[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) tmp[jj] = tf32_hi_bits(v[h + jj]);
          ptx::tmem_st8(tmem + lane_base + col + (uint32_t)(u * kUnit + h), tmp);
#pragma unroll
          for (int jj = 0; jj < 8; jj += 2)
            ptx::sub_f32x2(v[h + jj], v[h + jj + 1], __uint_as_float(tmp[jj]), __uint_as_float(tmp[jj + 1]), v[h + jj],
                           v[h + jj + 1]);
          ptx::tmem_st8(tmem + lane_base + col + (uint32_t)(Sp + u * kUnit + h),
                        *reinterpret_cast<const uint32_t (*)[8]>(v + h));
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar_s_full + 8 * s);
      if (t == 0) {
        // planes near a column's ends have fewer than KR reader tiles:
        // complete the slot's empty phase for the missing ones
        const int first = pl - KR + 1 > 0 ? pl - KR + 1 : 0, last = pl < p.R - 1 ? pl : p.R - 1;
        for (int m = last - first + 1; m < KR; ++m) ptx::mbar_arrive(bar_s_empty + 8 * s);
      }
    }
  } else if (warp >= kMmaWarp && warp - kMmaWarp < nslots) {
    // ------------------------------------------------------------ MMA issuers
    // warp b issues tiles it = b, b + nslots, ...: tile (j, d) = (it / R, it % R)
    // sums the 3xTF32 products of slabs j * P + d + kr with weight blocks kr
    const int slot = __shfl_sync(0xffffffffu, warp - kMmaWarp, 0);
    const uint32_t idesc = ptx::idesc_tf32(kTileM, (uint32_t)p.Npad);
    const uint32_t bhi = ptx::smem_addr(b_hi), blo = ptx::smem_addr(b_lo);
    const uint32_t d_tmem = tmem + (uint32_t)(slot * p.Npad);
    const int64_t my_tiles = ncols * p.R;
    bool aborted = false;
    for (int64_t it = slot; it < my_tiles && !aborted; it += nslots) {
      const int64_t li = it / nslots;
      if (!__all_sync(0xffffffffu, wait_phase(bar_d_empty + 8 * slot, ((uint32_t)li & 1) ^ 1, abort_flag,
                                                  p.wait_limit, kWaitSiteDEmpty))) break;
      ptx::tc_fence_after();
      const int64_t j = it / p.R, d = it - j * p.R;
      for (int kr = 0; kr < KR; ++kr) {
        const int64_t sidx = j * P + d + kr;
        const uint32_t s = (uint32_t)(sidx % NS), q = (uint32_t)(sidx / NS);
        if (!__all_sync(0xffffffffu, wait_phase(bar_s_full + 8 * s, q & 1, abort_flag, p.wait_limit, kWaitSiteAFull))) {
          aborted = true;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a_hi = tmem + slab_col0 + 2u * (uint32_t)Sp * s;
        const uint32_t a_lo = a_hi + (uint32_t)Sp;
        if (ptx::elect_one()) {
          for (int ks = 0; ks < Sp / 8; ++ks) {
            const uint64_t dh = ptx::smem_desc_noswizzle(bhi + kr * blk_bytes + 256u * ks, 128, (uint32_t)Sp * 32);
            const uint64_t dl = ptx::smem_desc_noswizzle(blo + kr * blk_bytes + 256u * ks, 128, (uint32_t)Sp * 32);
            ptx::mma_tf32_ts(d_tmem, a_hi + 8 * ks, dh, idesc, (kr | ks) != 0);
            ptx::mma_tf32_ts(d_tmem, a_hi + 8 * ks, dl, idesc, 1);
            ptx::mma_tf32_ts(d_tmem, a_lo + 8 * ks, dh, idesc, 1);
          }
          ptx::mma_commit(bar_s_empty + 8 * s);
        }
        __syncwarp();
      }
      if (aborted) break;
      if (ptx::elect_one()) ptx::mma_commit(bar_d_full + 8 * slot);
      __syncwarp();
    }
    if (*abort_flag) {
      // drain: every MMA this warp issued completes before TMEM is released
      if (ptx::elect_one()) {
        ptx::mma_commit(bar_drain + 8 * slot);
        const long long t0 = clock64();
        while (!ptx::mbar_try_wait(bar_drain + 8 * slot, 0) && clock64() - t0 < kWaitLimitCycles) {
        }
      }
      __syncwarp();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

#include "igemm_bf16.cuh"

// The plain-convolution kernel instance for a launch: a later reduction pass
// (per-value gather, run-time test group), else by gather form (vec 2 / 1)
// and, for the per-value form, by test group (16 / 8 / 4 compiled in; 1 and
// the streamed weights' 8 and 4 read at run time).
using IgemmKern = void (*)(const IgemmParams);
template <int CH, bool SB>
IgemmKern pick_plain(bool acc, int vec, int tg) {
  if constexpr (!SB) {
    if (acc) return igemm_3xtf32_kernel<CH, true, false>;
  }
  if (vec == 2) return igemm_3xtf32_kernel<CH, false, SB, false, 2>;
  if (vec == 1) return igemm_3xtf32_kernel<CH, false, SB, false, 1>;
  if (tg == 16) return igemm_3xtf32_kernel<CH, false, SB, false, 0, 16>;
  if constexpr (!SB) {
    if (tg == 8) return igemm_3xtf32_kernel<CH, false, false, false, 0, 8>;
    if (tg == 4) return igemm_3xtf32_kernel<CH, false, false, false, 0, 4>;
  }
  return igemm_3xtf32_kernel<CH, false, SB>;
}

int g_num_sms[64] = {0};
// the pipeline waits' limit for the next launches (set_wait_limit)
std::atomic<long long> g_wait_limit{kWaitLimitCycles};
bool g_attr_bf16_set[64] = {false};
bool g_attr_f16_set[64] = {false};
bool g_attr_set[64] = {false};
bool g_attr_fused_set[64] = {false};

// Elements addressable from a launch's x pointer (the group's first channel)
// to the last element the launch may read; the debug build's test hook can
// shrink it.
int64_t x_extent(const Geom &g) {
  const int64_t dhw = g.in_spatial();
  const int64_t n = g.cl ? (g.N * dhw - 1) * g.G * g.C + g.C : (g.N - 1) * g.x_batch_stride() + g.C * dhw;
  const int64_t s = debug_x_shrink();
  return n > s ? n - s : 0;
}
// The same for y: kb channels of `plane` positions per image, images y_chans
// channels apart.
int64_t y_extent(const Geom &g, int64_t y_chans, int64_t kb, int64_t plane) {
  return g.cl ? (g.N * plane - 1) * y_chans + kb : (g.N - 1) * y_chans * plane + kb * plane;
}
// TMEM columns a plan uses: one accumulator per slot plus two A stages (hi + lo) per slot.
int tmem_cols_used(int nslots, int npad, int kc) { return nslots * npad + nslots * 2 * 2 * kc; }

}  // namespace

bool igemm_supported(const Geom &g, const char **why) {
  Plan pl;
  Geom gb = g;
  if (gb.K > kMaxNpad) gb.K = kMaxNpad;  // wider layers run in channel blocks of 128
  return make_plan(gb, &pl, why);
}

int igemm_launches(const Geom &g) {
  Plan pl;
  Geom gb = g;
  if (gb.K > kMaxNpad) gb.K = kMaxNpad;
  const char *why = "";
  if (!make_plan(gb, &pl, &why)) return 0;
  return (int)((g.K + kMaxNpad - 1) / kMaxNpad) * pl.npasses;
}

// Workspace bytes for streamed weights (one group), or 0 when the layer does
// not need them (its weights fit in shared memory, or it spans channel blocks).
size_t igemm_stream_bytes_one_group(const Geom &g) {
  if (g.K > kMaxNpad) return 0;
  Plan pl;
  const char *why = "";
  // channels-last layers stream their weights even when they would fit:
  // the freed shared memory becomes L1 for the gather, which re-reads each
  // tap's channel line (sweep b 0.564 -> 0.527 ms)
  if (!make_plan(g, &pl, &why) || (pl.npasses <= 1 && !g.cl)) return 0;
  const int64_t kfull = g.C * (int64_t)g.taps();
  const int64_t kpad = (kfull + 31) / 32 * 32;
  const size_t smem = (size_t)pl.nslots * 2 * 2 * pl.Npad * pl.KC * 4 + (size_t)kpad * 8 + (size_t)pl.Npad * 4 +
                      16 + kNumBars * 8 + 16;
  if (smem > (size_t)kMaxSmem) return 0;  // the column tables alone would not fit
  return (size_t)pl.Npad * kpad * 8;
}

cudaError_t launch_igemm_3xtf32(const float *x, const float *w, const float *bias, float *y, const Geom &g,
                                cudaStream_t stream, float *ws) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (g_num_sms[dev] == 0) {
    e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  if (!g_attr_set[dev]) {
    const void *kerns[] = {
        (const void *)igemm_3xtf32_kernel<16, false, false>, (const void *)igemm_3xtf32_kernel<32, false, false>,
        (const void *)igemm_3xtf32_kernel<16, true, false>, (const void *)igemm_3xtf32_kernel<32, true, false>,
        (const void *)igemm_3xtf32_kernel<16, false, true>, (const void *)igemm_3xtf32_kernel<32, false, true>,
        (const void *)igemm_3xtf32_kernel<16, false, false, false, 1>,
        (const void *)igemm_3xtf32_kernel<32, false, false, false, 1>,
        (const void *)igemm_3xtf32_kernel<16, false, true, false, 1>,
        (const void *)igemm_3xtf32_kernel<32, false, true, false, 1>,
        (const void *)igemm_3xtf32_kernel<16, false, false, false, 2>,
        (const void *)igemm_3xtf32_kernel<32, false, false, false, 2>,
        (const void *)igemm_3xtf32_kernel<16, false, true, false, 2>,
        (const void *)igemm_3xtf32_kernel<32, false, true, false, 2>,
        (const void *)igemm_3xtf32_kernel<16, false, false, false, 0, 16>,
        (const void *)igemm_3xtf32_kernel<32, false, false, false, 0, 16>,
        (const void *)igemm_3xtf32_kernel<16, false, true, false, 0, 16>,
        (const void *)igemm_3xtf32_kernel<32, false, true, false, 0, 16>,
        (const void *)igemm_3xtf32_kernel<16, false, false, false, 0, 8>,
        (const void *)igemm_3xtf32_kernel<32, false, false, false, 0, 8>,
        (const void *)igemm_3xtf32_kernel<16, false, false, false, 0, 4>,
        (const void *)igemm_3xtf32_kernel<32, false, false, false, 0, 4>};
    for (const void *k : kerns) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
      if (e != cudaSuccess) return e;
    }
    g_attr_set[dev] = true;
  }
  const int64_t osp = (int64_t)g.OD * g.OH * g.OW;
  const int64_t kfull = g.C * (int64_t)g.taps();
  if (ws && igemm_stream_bytes_one_group(g) > 0) {
    // streamed weights: prepare the chunks, then one pass over the whole reduction
    Plan pl;
    const char *why = "";
    if (!make_plan(g, &pl, &why)) return cudaErrorInvalidValue;
    const int kpad = (int)((kfull + 31) / 32 * 32);
    const int nchunks = kpad / pl.KC;
    const int64_t total = (int64_t)pl.Npad * pl.KC * nchunks;
    const int threads = 256;
    const int64_t blocks64 = (total + threads - 1) / threads;
    const int blocks = (int)(blocks64 < 4096 ? blocks64 : 4096);
    CONV_PLAN_CHECK(nchunks * pl.KC == kpad && pl.KC % 16 == 0);
    CONV_PLAN_CHECK(tmem_cols_used(pl.nslots, pl.Npad, pl.KC) <= (int)kTmemCols);
    CONV_PLAN_CHECK(((uintptr_t)ws & 15u) == 0);
    split_weights_kernel<<<blocks, threads, 0, stream>>>(w, ws, (int)g.K, (int)g.C, g.taps(), (int)kfull, pl.Npad,
                                                         pl.KC, nchunks, pl.tap_major && !g.cl, g.K * kfull,
                                                         2 * total);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    IgemmParams p = {};
    p.wait_limit = g_wait_limit.load();
    p.x = x;
    p.w = w;
    p.bias = bias;
    p.y = y;
    p.g = g;
    p.osp = osp;
    p.M_total = g.N * p.osp;
    p.tiles = (p.M_total + kTileM - 1) / kTileM;
    p.Kred = (int)kfull;
    p.Kfull = (int)kfull;
    p.k_begin = 0;
    p.accumulate = 0;
    p.y_chans = g.G * g.K;
    p.Kpad = kpad;
    p.Npad = pl.Npad;
    p.KC = pl.KC;
    p.nchunks = nchunks;
    p.nslots = pl.nslots;
    p.tap_major = pl.tap_major;
    p.vec4 = (g.cl && g.C % 4 == 0 && (g.G * g.C) % 4 == 0 && ((uintptr_t)x & 15u) == 0) ? 1 : 0;
    p.vec8 = (p.vec4 && g.C % 8 == 0 && (g.G * g.C) % 8 == 0 && ((uintptr_t)x & 31u) == 0) ? 1 : 0;
    p.vec_store = (g.cl && (g.G * g.K) % 4 == 0 && ((uintptr_t)y & 15u) == 0) ? 1 : 0;
    p.wsp = ws;
    p.sb_stage_bytes = (uint32_t)(2 * pl.Npad * pl.KC * 4);
    p.b_bytes = (uint32_t)(pl.nslots * 2) * p.sb_stage_bytes;
    p.x_elems = x_extent(g);
    p.w_elems = g.K * kfull;
    p.y_elems = y_extent(g, p.y_chans, g.K, osp);
    p.ws_elems = 2 * total;
    const size_t smem_need = (size_t)p.b_bytes + (size_t)kpad * 8 + (size_t)pl.Npad * 4 + 16 + kNumBars * 8 + 16;
    const size_t smem = smem_need < (size_t)kMinSmem ? (size_t)kMinSmem : smem_need;
    const int64_t grid = p.tiles < g_num_sms[dev] ? p.tiles : g_num_sms[dev];
    CONV_PLAN_CHECK(smem <= (size_t)kMaxSmem && p.sb_stage_bytes % 16 == 0 && grid >= 1);
    CONV_PLAN_CHECK(!p.vec8 || (((uintptr_t)x & 31u) == 0 && p.tap_major && kfull % 8 == 0));
    const int vec = p.vec8 ? 2 : p.vec4 ? 1 : 0;
    const int tg = test_group_cols(p.tap_major, g.C);
    const IgemmKern kern = pl.KC <= 16 ? pick_plain<16, true>(false, vec, tg) : pick_plain<32, true>(false, vec, tg);
    kern<<<(unsigned)grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
  }
  // Output channels in blocks of at most 128 (one accumulator tile), each over
  // the reduction in passes that fit shared memory; every launch is a whole
  // persistent kernel on views of w, bias and y.
  for (int64_t o0 = 0; o0 < g.K; o0 += kMaxNpad) {
    Geom gb = g;
    gb.K = g.K - o0 < kMaxNpad ? g.K - o0 : kMaxNpad;
    Plan pl;
    const char *why = "";
    if (!make_plan(gb, &pl, &why)) return cudaErrorInvalidValue;
    for (int pass = 0; pass < pl.npasses; ++pass) {
      const int k_begin = pass * pl.kpass;
      const int kred = (int)(kfull - k_begin < pl.kpass ? kfull - k_begin : pl.kpass);
      IgemmParams p = {};
      p.wait_limit = g_wait_limit.load();
      p.x = x;
      p.w = w + o0 * kfull;
      p.bias = bias ? bias + o0 : nullptr;
      p.y = y + (g.cl ? o0 : o0 * osp);
      p.g = gb;
      p.osp = osp;
      p.M_total = g.N * p.osp;
      p.tiles = (p.M_total + kTileM - 1) / kTileM;
      p.Kred = kred;
      p.Kfull = (int)kfull;
      p.k_begin = k_begin;
      p.accumulate = pass > 0;
      p.y_chans = g.G * g.K;
      p.Kpad = (kred + 31) / 32 * 32;
      p.Npad = pl.Npad;
      p.KC = pl.KC;
      p.nchunks = (p.Kpad + pl.KC - 1) / pl.KC;
      p.nslots = pl.nslots;
      p.tap_major = pl.tap_major;
      p.vec4 = (g.cl && g.C % 4 == 0 && (g.G * g.C) % 4 == 0 && ((uintptr_t)x & 15u) == 0) ? 1 : 0;
      p.vec8 = (p.vec4 && g.C % 8 == 0 && (g.G * g.C) % 8 == 0 && ((uintptr_t)x & 31u) == 0) ? 1 : 0;
      p.vec_store = (g.cl && (g.G * g.K) % 4 == 0 && ((uintptr_t)p.y & 15u) == 0) ? 1 : 0;
      p.b_bytes = (uint32_t)((size_t)pl.Npad * p.Kpad * 4);
      p.x_elems = x_extent(g);
      p.w_elems = gb.K * kfull;
      p.y_elems = y_extent(g, p.y_chans, gb.K, osp);
      const size_t smem_need = (size_t)2 * pl.Npad * p.Kpad * 4 + (size_t)p.Kpad * 8 + (size_t)pl.Npad * 4 + 16 +
                               kNumBars * 8 + 16;
      const size_t smem = smem_need < (size_t)kMinSmem ? (size_t)kMinSmem : smem_need;
      const int64_t grid = p.tiles < g_num_sms[dev] ? p.tiles : g_num_sms[dev];
        CONV_PLAN_CHECK(smem <= (size_t)kMaxSmem && grid >= 1 && kred > 0);
      CONV_PLAN_CHECK(p.Kpad % 32 == 0 && p.nchunks * p.KC >= p.Kpad && p.KC % 16 == 0);
      CONV_PLAN_CHECK(tmem_cols_used(pl.nslots, pl.Npad, pl.KC) <= (int)kTmemCols);
      CONV_PLAN_CHECK(k_begin + kred <= kfull && (o0 + gb.K) <= g.K);
      CONV_PLAN_CHECK(!p.vec4 || ((uintptr_t)x & 15u) == 0);
      CONV_PLAN_CHECK(!p.vec8 || (((uintptr_t)x & 31u) == 0 && p.tap_major && k_begin % 8 == 0 && kred % 8 == 0));
      // the vector gathers serve single-pass launches; reduction passes
      // (rare: weights beyond shared memory without a streaming block) take
      // the per-value gather, which serves any layout
      const int vec = pl.npasses != 1 ? 0 : p.vec8 ? 2 : p.vec4 ? 1 : 0;
      const int tg = pl.npasses != 1 ? 0 : test_group_cols(p.tap_major, g.C);
      const IgemmKern kern =
          pl.KC <= 16 ? pick_plain<16, false>(pass > 0, vec, tg) : pick_plain<32, false>(pass > 0, vec, tg);
      kern<<<(unsigned)grid, kThreads, smem, stream>>>(p);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

void describe_igemm_plan(const Geom &g, bool streamed, char *buf, size_t n) {
  Plan pl;
  Geom gb = g;
  if (gb.K > kMaxNpad) gb.K = kMaxNpad;
  const char *why = "";
  if (!make_plan(gb, &pl, &why)) {
    snprintf(buf, n, "unsupported (%s)", why);
    return;
  }
  const int64_t tiles = (g.N * g.out_spatial() + kTileM - 1) / kTileM;
  const int64_t blocks = (g.K + kMaxNpad - 1) / kMaxNpad;
  snprintf(buf, n,
           "tiles=%lld Kred=%d Kpad=%d Npad=%d KC=%d slots=%d order=%s passes=%d channel_blocks=%lld weights=%s "
           "smem=%zu",
           (long long)tiles, pl.Kred, pl.Kpad, pl.Npad, pl.KC, pl.nslots, pl.tap_major ? "tap-major" : "channel-major",
           streamed ? 1 : pl.npasses, (long long)blocks, streamed ? "streamed" : "resident", pl.smem);
}

bool igemm_fused_supported(const Geom &g, int min_dim, const char **why) {
  Plan pl;
  if (min_dim < 2 || min_dim > 4) {
    *why = "tensor-core fused path: min_dim must be 2, 3 or 4";
    return false;
  }
  if (g.cl) {
    *why = "tensor-core fused path: channels-last input";
    return false;
  }
  if (g.SD != 1 || g.SH != 1 || g.SW != 1 || g.PD || g.PH || g.PW || g.DD != 1 || g.DH != 1 || g.DW != 1 || g.G != 1) {
    *why = "tensor-core fused path: stride 1, no padding, dilation 1 and one group only";
    return false;
  }
  // layers wider than 32 channels run in blocks of 32 (the epilogue holds one
  // position's channels in registers), then a channel-softmax pass
  Geom gb = g;
  if (gb.K > 32) gb.K = 32;
  if (!make_plan(gb, &pl, why)) return false;
  if (pl.KC != 16) {
    *why = "tensor-core fused path: no 16-column stages";
    return false;
  }
  if (pl.npasses != 1 && igemm_stream_bytes_one_group(gb) == 0) {
    *why = "tensor-core fused path: the weights neither fit in shared memory nor stream";
    return false;
  }
  return true;
}

size_t igemm_fused_stream_bytes(const Geom &g) {
  Plan pl;
  Geom gb = g;
  if (gb.K > 32) gb.K = 32;  // per channel block, reused block after block
  const char *why = "";
  if (!make_plan(gb, &pl, &why) || pl.npasses == 1) return 0;
  return igemm_stream_bytes_one_group(gb);
}

cudaError_t launch_igemm_fused_min_softmax(const float *x, const float *w, const float *bias, float *y, const Geom &g,
                                           int min_dim, cudaStream_t stream, float *ws, bool min_only,
                                           int64_t y_chans) {
  Plan pl;
  const char *why = "";
  if (g.K > 32 || !igemm_fused_supported(g, min_dim, &why) || !make_plan(g, &pl, &why)) return cudaErrorInvalidValue;
  const bool streamed = pl.npasses != 1;
  if (streamed && !ws) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (g_num_sms[dev] == 0) {
    e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  if (!g_attr_fused_set[dev]) {
    e = cudaFuncSetAttribute(igemm_3xtf32_kernel<16, false, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fused_slab_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(igemm_3xtf32_kernel<16, false, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kMaxSmem);
    if (e != cudaSuccess) return e;
    g_attr_fused_set[dev] = true;
  }
  const int64_t kfull = g.C * (int64_t)g.taps();
  IgemmParams p = {};
  p.wait_limit = g_wait_limit.load();
  p.x = x;
  p.w = w;
  p.bias = bias;
  p.y = y;
  p.g = g;
  p.osp = (int64_t)g.OD * g.OH * g.OW;
  p.M_total = g.N * p.osp;
  // the reduced axis and the kept plane (the other two axes, in order)
  p.rdim = min_dim - 2;
  if (min_dim == 2) {
    p.R = g.OD, p.nB = g.OW, p.plane = (int64_t)g.OH * g.OW;
  } else if (min_dim == 3) {
    p.R = g.OH, p.nB = g.OW, p.plane = (int64_t)g.OD * g.OW;
  } else {
    p.R = g.OW, p.nB = g.OH, p.plane = (int64_t)g.OD * g.OH;
  }
  p.columns = (g.N * p.plane + kTileM - 1) / kTileM;
  p.tiles = p.columns * p.R;
  p.Kfull = (int)kfull;
  p.k_begin = 0;
  p.accumulate = 0;
  p.y_chans = y_chans > 0 ? y_chans : g.K;
  p.fused_min_only = min_only ? 1 : 0;
  p.Npad = pl.Npad;
  p.KC = pl.KC;
  p.nslots = pl.nslots;
  p.tap_major = pl.tap_major;
  const int64_t grid = p.columns < g_num_sms[dev] ? p.columns : g_num_sms[dev];
  p.x_elems = x_extent(g);
  p.w_elems = g.K * kfull;
  p.y_elems = (g.N - 1) * p.y_chans * p.plane + g.K * p.plane;
  CONV_PLAN_CHECK(grid >= 1 && p.R >= 1 && p.columns * kTileM >= g.N * p.plane);
  CONV_PLAN_CHECK(p.plane * p.R == p.osp && p.nB >= 1 && p.plane % p.nB == 0);
  CONV_PLAN_CHECK(tmem_cols_used(pl.nslots, pl.Npad, pl.KC) <= (int)kTmemCols);
  if (streamed) {
    // the whole reduction in one pass, its weights split once into ws and
    // brought in chunk by chunk (as for the plain conv's streamed weights)
    const int kpad = (int)((kfull + 31) / 32 * 32);
    const int nchunks = kpad / pl.KC;
    const int64_t total = (int64_t)pl.Npad * pl.KC * nchunks;
    const int threads = 256;
    const int64_t blocks64 = (total + threads - 1) / threads;
    const int blocks = (int)(blocks64 < 4096 ? blocks64 : 4096);
    CONV_PLAN_CHECK(nchunks * pl.KC == kpad && ((uintptr_t)ws & 15u) == 0);
    split_weights_kernel<<<blocks, threads, 0, stream>>>(w, ws, (int)g.K, (int)g.C, g.taps(), (int)kfull, pl.Npad,
                                                         pl.KC, nchunks, pl.tap_major, g.K * kfull, 2 * total);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    p.Kred = (int)kfull;
    p.Kpad = kpad;
    p.nchunks = nchunks;
    p.wsp = ws;
    p.sb_stage_bytes = (uint32_t)(2 * pl.Npad * pl.KC * 4);
    p.b_bytes = (uint32_t)(pl.nslots * 2) * p.sb_stage_bytes;
    p.ws_elems = 2 * total;
    const size_t smem_need = (size_t)p.b_bytes + (size_t)kpad * 8 + (size_t)pl.Npad * 4 + 16 + kNumBars * 8 + 16;
    const size_t smem = smem_need < (size_t)kMinSmem ? (size_t)kMinSmem : smem_need;
    CONV_PLAN_CHECK(smem <= (size_t)kMaxSmem);
    igemm_3xtf32_kernel<16, false, true, true><<<(unsigned)grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
  }
  p.Kred = pl.Kred;
  p.Kpad = pl.Kpad;
  p.nchunks = pl.nchunks;
  // slabs: each input plane along the reduced axis gathered once (a slab of
  // C_in x KA x KB columns, padded to 16) and read by the KR tiles that need
  // it, when a ring of KR + 3 slabs (four tiles in flight) fits in TMEM
  // beside the four accumulators
  {
    const int kr = min_dim == 2 ? g.KD : min_dim == 3 ? g.KH : g.KW;
    const int ka = min_dim == 2 ? g.KH : g.KD, kb = min_dim == 4 ? g.KH : g.KW;
    const int64_t sc = g.C * (int64_t)ka * kb;
    const int sp = (int)((sc + 15) / 16 * 16);
    int ns = sp > 0 ? (int)((kTmemCols - kMaxSlots * pl.Npad) / (2 * sp)) : 0;
    if (ns > kMaxStages) ns = kMaxStages;
    // (the min over width reaches here as a min over height of transposed
    // copies; read directly, along W, it keeps the chunked kernel)
    if (min_dim != 4 && sc <= 32 && pl.nslots == kMaxSlots && ns >= kr + kMaxSlots - 1) {
      p.slab_cols = sp;
      p.slab_real = (int)sc;
      p.slab_kr = kr;
      p.nslabs = ns;
      p.b_bytes = (uint32_t)((size_t)kr * pl.Npad * sp * 4);
      const size_t need = 2 * (size_t)p.b_bytes + (size_t)sp * 4 + (size_t)pl.Npad * 4 + 16 + kNumBars * 8 + 16;
      const size_t smem = need < (size_t)kMinSmem ? (size_t)kMinSmem : need;
      CONV_PLAN_CHECK(smem <= (size_t)kMaxSmem && kMaxSlots * pl.Npad + 2 * sp * ns <= (int)kTmemCols);
      CONV_PLAN_CHECK(p.R + kr - 1 == (min_dim == 2 ? g.D : min_dim == 3 ? g.H : g.W));
      fused_slab_kernel<<<(unsigned)grid, kThreads, smem, stream>>>(p);
      return cudaGetLastError();
    }
  }
  p.b_bytes = (uint32_t)((size_t)pl.Npad * pl.Kpad * 4);
  CONV_PLAN_CHECK(pl.smem <= (size_t)kMaxSmem && pl.npasses == 1);
  igemm_3xtf32_kernel<16, false, false, true><<<(unsigned)grid, kThreads, pl.smem, stream>>>(p);
  return cudaGetLastError();
}

bool igemm_bf16_supported(const Geom &g, const char **why) {
  PlanBf16 pl;
  Geom gb = g;
  if (gb.K > kMaxNpad) gb.K = kMaxNpad;  // wider layers run in channel blocks of 128
  return make_plan_bf16(gb, &pl, why);
}

size_t igemm_bf16_stream_bytes(const Geom &g) {
  PlanBf16 pl;
  Geom gb = g;
  if (gb.K > kMaxNpad) gb.K = kMaxNpad;
  const char *why = "";
  if (!make_plan_bf16(gb, &pl, &why) || !pl.streamed) return 0;
  return (size_t)pl.Npad * pl.Kpad * 2;
}

cudaError_t launch_igemm_bf16(const uint16_t *x, const uint16_t *w, const uint16_t *bias, uint16_t *y, const Geom &g,
                              bool fp16, cudaStream_t stream, uint16_t *ws) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (g_num_sms[dev] == 0) {
    e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  bool &attr_set = fp16 ? g_attr_f16_set[dev] : g_attr_bf16_set[dev];
  if (!attr_set) {
    const void *kerns[2][5] = {
        {(const void *)igemm_bf16_kernel<false, false>, (const void *)igemm_bf16_kernel<false, true>,
         (const void *)igemm_bf16_kernel<false, false, 16>, (const void *)igemm_bf16_kernel<false, false, 8>,
         (const void *)igemm_bf16_kernel<false, false, 4>},
        {(const void *)igemm_bf16_kernel<true, false>, (const void *)igemm_bf16_kernel<true, true>,
         (const void *)igemm_bf16_kernel<true, false, 16>, (const void *)igemm_bf16_kernel<true, false, 8>,
         (const void *)igemm_bf16_kernel<true, false, 4>}};
    for (const void *k : kerns[fp16 ? 1 : 0]) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
      if (e != cudaSuccess) return e;
    }
    attr_set = true;
  }
  const int64_t osp = (int64_t)g.OD * g.OH * g.OW;
  const int64_t kfull = g.C * (int64_t)g.taps();
  // output channels in blocks of at most 128 (one accumulator tile), each a
  // whole persistent launch on views of w, bias and y
  for (int64_t o0 = 0; o0 < g.K; o0 += kMaxNpad) {
    Geom gb = g;
    gb.K = g.K - o0 < kMaxNpad ? g.K - o0 : kMaxNpad;
    PlanBf16 pl;
    const char *why = "";
    if (!make_plan_bf16(gb, &pl, &why)) return cudaErrorInvalidValue;
    if (pl.streamed && !ws) return cudaErrorInvalidValue;
    if (pl.streamed) {
      // the block's weights in chunk order into ws (reused block after block, in stream order)
      const int64_t total = (int64_t)pl.Npad * kBfChunk * pl.nchunks;
      const int64_t blocks64 = (total + 255) / 256;
      CONV_PLAN_CHECK(((uintptr_t)ws & 15u) == 0 && pl.nchunks * kBfChunk == pl.Kpad);
      split_weights_bf16_kernel<<<(unsigned)(blocks64 < 4096 ? blocks64 : 4096), 256, 0, stream>>>(
          w + o0 * kfull, ws, (int)gb.K, (int)g.C, g.taps(), (int)kfull, pl.Npad, pl.nchunks, pl.tap_major,
          gb.K * kfull, total);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    IgemmParams p = {};
    p.wait_limit = g_wait_limit.load();
    p.xh = x;
    p.wh = w + o0 * kfull;
    p.bh = bias ? bias + o0 : nullptr;
    p.yh = y + o0 * osp;
    p.g = gb;
    p.osp = osp;
    p.M_total = g.N * p.osp;
    p.tiles = (p.M_total + kTileM - 1) / kTileM;
    p.Kred = pl.Kred;
    p.Kfull = pl.Kred;
    p.y_chans = g.G * g.K;
    p.Kpad = pl.Kpad;
    p.Npad = pl.Npad;
    p.KC = kBfChunk;
    p.nchunks = pl.nchunks;
    p.nslots = pl.nslots;
    p.tap_major = pl.tap_major;
    p.b_bytes = (uint32_t)((size_t)pl.Npad * pl.Kpad * 2);
    if (pl.streamed) {
      p.wsp = reinterpret_cast<const float *>(ws);
      p.sb_stage_bytes = (uint32_t)(pl.Npad * kBfChunk * 2);
      p.b_bytes = (uint32_t)(pl.nslots * 2) * p.sb_stage_bytes;
      p.ws_elems = (int64_t)pl.Npad * kBfChunk * pl.nchunks;
    }
    p.x_elems = x_extent(g);
    p.w_elems = gb.K * kfull;
    p.y_elems = y_extent(g, p.y_chans, gb.K, osp);
    const int64_t grid = p.tiles < g_num_sms[dev] ? p.tiles : g_num_sms[dev];
    CONV_PLAN_CHECK(pl.smem <= (size_t)kMaxSmem && grid >= 1 && pl.Kred == kfull && !g.cl);
    CONV_PLAN_CHECK(pl.nchunks * kBfChunk >= pl.Kpad && pl.nslots * pl.Npad + pl.nslots * 2 * 16 <= (int)kTmemCols);
    // resident weights: the instance with the test group compiled in (16 / 8 / 4)
    const int tg = pl.streamed ? 0 : test_group_cols(p.tap_major, g.C);
    auto pick = [&](auto half) -> IgemmKern {
      constexpr bool H = decltype(half)::value;
      if (pl.streamed) return igemm_bf16_kernel<H, true>;
      if (tg == 16) return igemm_bf16_kernel<H, false, 16>;
      if (tg == 8) return igemm_bf16_kernel<H, false, 8>;
      if (tg == 4) return igemm_bf16_kernel<H, false, 4>;
      return igemm_bf16_kernel<H, false>;
    };
    const IgemmKern kern = fp16 ? pick(std::true_type{}) : pick(std::false_type{});
    kern<<<(unsigned)grid, kThreads, pl.smem, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

void set_wait_limit(long long cycles) { g_wait_limit.store(cycles > 0 ? cycles : kWaitLimitCycles); }

cudaError_t read_and_clear_device_status(unsigned *flags) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero));
  *flags = v;
  return e;
}

}  // namespace convfwd
