// 16-bit variant of the implicit-GEMM kernel: x, w and bias in bfloat16 (or
// float16, template HALF), the products and their sum in fp32 (tensor-core
// accumulator), y rounded once to the input type (round to nearest even) at
// the store.  The conv sum is the one in
// the l1_p60 page (turn 1); the pages weigh BF16 against fp32 accuracy and
// keep fp32, so this path is the lower-precision option next to 3xTF32.
//
// Structure as the 3xTF32 kernel (same warp roles, slots, tables and waits);
// what changes:
//   * no hi/lo split: a gathered value is stored once, two bf16 per 32-bit
//     TMEM column, so one 32-column chunk of K fills 16 TMEM columns;
//   * one tcgen05.mma kind::f16 per 16 reduction columns (K = 16);
//   * B holds one bf16 copy of the weights: core matrices of 8 rows x 8 bf16,
//     LBO = 128 bytes along K, SBO = Kpad * 16 bytes along N.
// This file is included inside igemm_tcgen05.cu's anonymous namespace.

constexpr int kBfChunk = 32;  // reduction columns per chunk (16 TMEM columns)

struct PlanBf16 {
  int Kred, Kpad, Npad, nchunks, nslots, tap_major;
  int streamed;  // the weights exceed shared memory: chunk by chunk from a workspace
  size_t smem;
};

bool make_plan_bf16(const Geom &g, PlanBf16 *pl, const char **why) {
  if (g.K > kMaxNpad) {
    *why = "C_out (per group) above 128";
    return false;
  }
  if (g.KD > 32 || g.KH > 32 || g.KW > 32) {
    *why = "a kernel dimension above 32";
    return false;
  }
  if (g.cl) {
    *why = "channels-last layout is fp32 only";
    return false;
  }
  const int64_t HW = (int64_t)g.H * g.W, DHW = HW * g.D;
  const int64_t max_off = (g.C - 1) * DHW + (int64_t)(g.KD - 1) * g.DD * HW + (int64_t)(g.KH - 1) * g.DH * g.W +
                          (int64_t)(g.KW - 1) * g.DW;
  if (max_off >= (int64_t)1 << 31) {
    *why = "receptive-field offsets of one image exceed 2^31 elements";
    return false;
  }
  const int64_t kred = g.C * (int64_t)g.KD * g.KH * g.KW;
  pl->Kred = (int)kred;
  pl->Kpad = (int)((kred + kBfChunk - 1) / kBfChunk * kBfChunk);
  pl->Npad = (int)((g.K + 31) / 32 * 32);
  // TMEM: one accumulator of Npad columns per slot, two A stages of 16 columns per slot
  pl->nslots = (kMaxSlots * pl->Npad + 2 * kMaxSlots * (kBfChunk / 2) <= (int)kTmemCols) ? kMaxSlots : 2;
  pl->nchunks = pl->Kpad / kBfChunk;
  pl->tap_major = (g.C % 4 == 0 && (g.PD > 0 || g.PH > 0 || g.PW > 0)) ? 1 : 0;
  const size_t fixed = (size_t)pl->Kpad * 8 + (size_t)pl->Npad * 4 + 16 + kNumBars * 8 + 16;
  size_t smem = (size_t)pl->Npad * pl->Kpad * 2 + fixed;
  pl->streamed = 0;
  if (smem > (size_t)kMaxSmem) {
    // streamed weights: two B stages per slot of one chunk each (Npad x 32 bf16)
    smem = (size_t)pl->nslots * 2 * pl->Npad * kBfChunk * 2 + fixed;
    if (smem > (size_t)kMaxSmem) {
      *why = "the reduction's column tables exceed shared memory";
      return false;
    }
    pl->streamed = 1;
  }
  pl->smem = smem < (size_t)kMinSmem ? (size_t)kMinSmem : smem;
  return true;
}

// x[xoff + o] as a zero-extended 16-bit pattern (the debug build first checks
// that the index lies in x)
__device__ __forceinline__ uint32_t ldxh(const PosInfo &ps, const uint16_t *xo, int32_t o) {
#ifdef CONVFWD_DEBUG
  if (!CONV_DBG_OK(ps.xoff + o, ps.xn, kStatusBoundsX)) return 0u;
#endif
  return (uint32_t)__ldg(xo + o);
}

// 16 consecutive reduction columns of one output position as bf16 bit
// patterns (zero-extended to 32 bits); same tables and paths as gather_cols.
__device__ __forceinline__ void gather_cols_bf16(const PosInfo &ps, const uint16_t *xo, const int32_t *toff,
                                                 const uint32_t *ttap, int k0, int Kred, int tg,
                                                 uint32_t (&v)[kUnit]) {
  if (ps.warp_full) {
    const int4 *o4 = reinterpret_cast<const int4 *>(toff + k0);
#pragma unroll
    for (int q = 0; q < kUnit / 4; ++q) {
      const int4 o = o4[q];
      const int k = k0 + 4 * q;
      v[4 * q + 0] = k + 0 < Kred ? ldxh(ps, xo, o.x) : 0u;
      v[4 * q + 1] = k + 1 < Kred ? ldxh(ps, xo, o.y) : 0u;
      v[4 * q + 2] = k + 2 < Kred ? ldxh(ps, xo, o.z) : 0u;
      v[4 * q + 3] = k + 3 < Kred ? ldxh(ps, xo, o.w) : 0u;
    }
  } else if (tg >= 4) {
    // tap-major over C_in a multiple of tg: one test per tg-column block
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
      v[4 * q + 0] = in ? ldxh(ps, xo, o.x) : 0u;
      v[4 * q + 1] = in ? ldxh(ps, xo, o.y) : 0u;
      v[4 * q + 2] = in ? ldxh(ps, xo, o.z) : 0u;
      v[4 * q + 3] = in ? ldxh(ps, xo, o.w) : 0u;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kUnit; ++j) {
      const uint32_t e = ttap[k0 + j];
      const uint32_t kd = e & 0xffu, kh = (e >> 8) & 0xffu, kw = (e >> 16) & 0xffu;
      const bool in = ps.valid && !(e >> 31) && (((ps.dm >> kd) & (ps.hm >> kh) & (ps.wm >> kw)) & 1u);
      v[j] = in ? ldxh(ps, xo, toff[k0 + j]) : 0u;
    }
  }
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

template <bool HALF>
__device__ __forceinline__ float bits16_to_float(unsigned short b) {
  return HALF ? __half2float(__ushort_as_half(b)) : bf16_bits_to_float(b);
}
template <bool HALF>
__device__ __forceinline__ unsigned short float_to_bits16(float f) {
  return HALF ? __half_as_ushort(__float2half_rn(f)) : __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Streamed weights, prepared once per call: chunk q of the reduction (32
// columns) as the tensor cores read it from shared memory, [Npad x 32] 16-bit
// values in core matrices of 8 rows x 8 (LBO 128 bytes along K, SBO 512 bytes
// along N); column kg maps to w's memory order as in the resident staging.
__global__ void split_weights_bf16_kernel(const uint16_t *__restrict__ w, uint16_t *__restrict__ ws, int K, int C,
                                          int taps, int Kfull, int Npad, int nchunks, int tap_major, int64_t w_elems,
                                          int64_t ws_elems) {
  const int64_t per_chunk = (int64_t)Npad * kBfChunk;
  const int64_t total = per_chunk * nchunks;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int q = (int)(i / per_chunk);
    const int e = (int)(i - (int64_t)q * per_chunk);
    const int cm = e >> 6, r = (e >> 3) & 7, col = e & 7;  // core matrix (8 x 8), row, column
    const int n = (cm / (kBfChunk / 8)) * 8 + r, k = (cm % (kBfChunk / 8)) * 8 + col;
    const int kg = q * kBfChunk + k;
    uint16_t v = 0;
    if (n < K && kg < Kfull) {
      int kmem = kg;
      if (tap_major) {
        const int t = kg / C;
        kmem = (kg - t * C) * taps + t;
      }
      if (CONV_DBG_OK((int64_t)n * Kfull + kmem, w_elems, kStatusBoundsW)) v = __ldg(w + (int64_t)n * Kfull + kmem);
    }
    if (CONV_DBG_OK(i, ws_elems, kStatusBoundsWs)) ws[i] = v;
  }
}

// HALF = false: bfloat16 tensors; true: float16 tensors (A and B always of one type).
// SB: streamed weights (p.wsp: the prepared chunks, p.sb_stage_bytes each).
// TG: the tested gather's columns per in-bounds test fixed at compile time
// (0: read at run time), as in the 32-bit kernel.
template <bool HALF, bool SB, int TG = 0>
__global__ void __launch_bounds__(kThreads, 1) igemm_bf16_kernel(const IgemmParams p) {
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

  uint8_t *b_s = smem;  // resident weights, or (SB) one B stage per A stage
  int32_t *toff = reinterpret_cast<int32_t *>(smem + p.b_bytes);  // [Kpad]
  uint32_t *ttap = reinterpret_cast<uint32_t *>(toff + p.Kpad);    // [Kpad]
  float *bias_s = reinterpret_cast<float *>(ttap + p.Kpad);
  uint64_t *bars = reinterpret_cast<uint64_t *>((reinterpret_cast<uintptr_t>(bias_s + p.Npad) + 15) & ~(uintptr_t)15);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  const uint32_t bar_a_full = ptx::smem_addr(bars + 0);
  const uint32_t bar_a_empty = ptx::smem_addr(bars + kMaxStages);
  const uint32_t bar_d_full = ptx::smem_addr(bars + 2 * kMaxStages);
  const uint32_t bar_d_empty = ptx::smem_addr(bars + 2 * kMaxStages + kMaxSlots);
  const uint32_t bar_b_full = ptx::smem_addr(bars + 2 * kMaxStages + 2 * kMaxSlots);  // [stages] (SB)
  const uint32_t bar_drain = ptx::smem_addr(bars + 3 * kMaxStages + 2 * kMaxSlots);  // [slots]
  const int nslots = p.nslots;

  const uint32_t SBO = (uint32_t)p.Kpad * 16;  // bytes between 8-row groups of B
  const int taps = g.KD * g.KH * g.KW;
  const int64_t HW = (int64_t)g.H * g.W, DHW = HW * g.D;

  // ---- weights -> shared memory as bf16 pairs.  32-bit word i of the
  // core-matrix layout holds B[n][k], B[n][k+1] with n = 8*(cm / (Kpad/8)) +
  // row, k = 8*(cm % (Kpad/8)) + 2*pair (cm = i / 32, row = (i / 4) % 8,
  // pair = i % 4): consecutive threads write consecutive words.
  {
    const int kq8 = p.Kpad / 8;
    const int words = SB ? 0 : p.Npad * p.Kpad / 2;  // streamed weights arrive per chunk
    for (int i = tid; i < words; i += kThreads) {
      const int cm = i >> 5, r = (i >> 2) & 7, pr = i & 3;
      const int n = (cm / kq8) * 8 + r, k = (cm % kq8) * 8 + pr * 2;
      uint32_t word = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int kk = k + h;
        if (n < g.K && kk < p.Kred) {
          int kmem = kk;
          if (p.tap_major) {
            const int t = kk / g.C;
            kmem = (kk - t * g.C) * taps + t;
          }
          if (CONV_DBG_OK((int64_t)n * p.Kred + kmem, p.w_elems, kStatusBoundsW))
            word |= (uint32_t)__ldg(p.wh + (int64_t)n * p.Kred + kmem) << (16 * h);
        }
      }
      reinterpret_cast<uint32_t *>(b_s)[i] = word;
    }
    for (int kk = tid; kk < p.Kpad; kk += kThreads) {
      if (kk < p.Kred) {
        int c, t;
        if (p.tap_major) {
          t = kk / g.C;
          c = kk - t * g.C;
        } else {
          c = kk / taps;
          t = kk - c * taps;
        }
        const int kw = t % g.KW, khd = t / g.KW;
        const int kd = khd / g.KH, kh = khd - kd * g.KH;
        toff[kk] = (int32_t)(c * DHW + (int64_t)kd * g.DD * HW + (int64_t)kh * g.DH * g.W + (int64_t)kw * g.DW);
        ttap[kk] = (uint32_t)kd | ((uint32_t)kh << 8) | ((uint32_t)kw << 16);
      } else {
        toff[kk] = 0;
        ttap[kk] = 0x80000000u;
      }
    }
    for (int i = tid; i < p.Npad; i += kThreads)
      bias_s[i] = (p.bh && i < g.K) ? bits16_to_float<HALF>(__ldg(p.bh + i)) : 0.f;
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
  // slot b: accumulator at column b * Npad; A stage s (2 per slot) at a_col0 + 16 * s
  const uint32_t a_col0 = (uint32_t)(nslots * p.Npad);

  if (warp < kEpiWarps) {
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
        n = m / p.osp;
        pp = m - n * p.osp;
      }
      uint16_t *yp = p.yh + n * p.y_chans * p.osp + pp;  // images y_chans channels apart (all groups and blocks)
      for (int c0 = 0; c0 < p.Npad; c0 += 32) {
        uint32_t v[32];
        ptx::tmem_ld32(tmem + lane_base + b * p.Npad + c0, v);
        ptx::tmem_wait_ld();
        if (c0 + 32 >= p.Npad) {
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar_d_empty + 8 * b);
        }
#ifdef CONVFWD_DEBUG
        if (valid) {
          // this lane's stores of channels c0 .. c0 + 31 (< K): first and last index
          const int64_t i0 = (yp - p.yh) + (int64_t)c0 * p.osp;
          const int nk = min(32, (int)g.K - c0);
          if (nk > 0 && (!CONV_DBG_OK(i0, p.y_elems, kStatusBoundsY) ||
                         !CONV_DBG_OK(i0 + (int64_t)(nk - 1) * p.osp, p.y_elems, kStatusBoundsY)))
            continue;
        }
#endif
        if (valid) {
          uint16_t *q = yp + (int64_t)c0 * p.osp;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (c0 + j < g.K) {
              __stcs(reinterpret_cast<unsigned short *>(q),
                     float_to_bits16<HALF>(__uint_as_float(v[j]) + bias_s[c0 + j]));
            }
            q += p.osp;
          }
        }
      }
    }
  } else if (warp < kMmaWarp) {
    // ------------------------------------------------------------ producers
    const int grp = (warp - kEpiWarps) >> 2;
    const int gps = kProdGroups / nslots;
    const int slot = grp / gps, sel = grp - slot * gps;
    const int t = tid - 32 * kEpiWarps - 128 * grp;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int64_t my_tiles = cta_tile_count(p);
    const int64_t slot_tiles = (my_tiles - slot + nslots - 1) / nslots;
    // columns per in-bounds test of the tested gather (tap-major: the largest
    // of 16, 8, 4 dividing C_in; else each column)
    const int tg = TG != 0 ? TG : test_group_cols(p.tap_major, g.C);  // compile time where TG is given
    // streamed weights: the group's thread 0 brings chunk q's B into the stage
    // and remembers its last copy, to wait for it before leaving
    int sb_last_stage = -1;
    uint32_t sb_last_parity = 0;
    bool aborted = false;
    for (int64_t li = 0; li < slot_tiles && !aborted; ++li) {
      const PosInfo ps = decode_position(p, tile_of(p, li * nslots + slot), t);
      const uint16_t *xo = p.xh + (ps.valid ? ps.xoff : 0);
      // slot-local index of the tile's first chunk; only its low bits matter
      // (stage and phase parity), so 32-bit arithmetic (wrapping) serves
      const uint32_t lg0 = (uint32_t)li * (uint32_t)p.nchunks;
      // chunk q (slot-local lg = lg0 + q): wait for its stage, store, signal the issuer
      auto put = [&](int q, const uint32_t (&packed)[kBfChunk / 2]) -> bool {
        const uint32_t lg = lg0 + (uint32_t)q;
        const int stage = 2 * slot + (int)(lg & 1);
        const uint32_t r = (uint32_t)(lg >> 1);
        const bool ok = wait_phase(bar_a_empty + 8 * stage, (r & 1) ^ 1, abort_flag, p.wait_limit, kWaitSiteAEmpty);
        if (!__all_sync(0xffffffffu, ok)) return false;
        ptx::tc_fence_after();
        if (SB && t == 0) {
          // the stage's MMAs are done: its B half is free too
          const int64_t e0 = (int64_t)q * (p.sb_stage_bytes / 2);  // 16-bit elements
          if (CONV_DBG_OK(e0 + p.sb_stage_bytes / 2 - 1, p.ws_elems, kStatusBoundsWs)) {
            ptx::mbar_arrive_expect_tx(bar_b_full + 8 * stage, p.sb_stage_bytes);
            ptx::bulk_copy_g2s(ptx::smem_addr(b_s + (size_t)stage * p.sb_stage_bytes),
                               reinterpret_cast<const uint8_t *>(p.wsp) + (size_t)q * p.sb_stage_bytes,
                               p.sb_stage_bytes, bar_b_full + 8 * stage);
          } else {
            ptx::mbar_arrive(bar_b_full + 8 * stage);  // (debug build) the copy is dropped
          }
          sb_last_stage = stage;
          sb_last_parity = r & 1;
        }
        ptx::tmem_st16(tmem + lane_base + a_col0 + (uint32_t)(16 * stage), packed);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_a_full + 8 * stage);
        return true;
      };
      int q = (int)((sel - (int)(lg0 % (uint32_t)gps) + gps) % gps);
      if (ps.warp_full) {
        // full chunks of an interior warp: four offsets per shared load, no tests
        const int nfull = p.Kred / kBfChunk;
        for (; q < nfull; q += gps) {
          uint32_t packed[kBfChunk / 2];
          const int4 *o4 = reinterpret_cast<const int4 *>(toff + q * kBfChunk);
#pragma unroll
          for (int i = 0; i < kBfChunk / 4; ++i) {
            const int4 o = o4[i];
            packed[2 * i] = __byte_perm(ldxh(ps, xo, o.x), ldxh(ps, xo, o.y), 0x5410);
            packed[2 * i + 1] = __byte_perm(ldxh(ps, xo, o.z), ldxh(ps, xo, o.w), 0x5410);
          }
          if (!put(q, packed)) {
            aborted = true;
            break;
          }
        }
        if (aborted) break;
      }
      for (; q < p.nchunks; q += gps) {
        const int k0 = q * kBfChunk;
        uint32_t packed[kBfChunk / 2];
#pragma unroll
        for (int u = 0; u < kBfChunk / kUnit; ++u) {
          uint32_t v[kUnit];
          gather_cols_bf16(ps, xo, toff, ttap, k0 + u * kUnit, p.Kred, tg, v);
#pragma unroll
          for (int j = 0; j < kUnit / 2; ++j) packed[u * (kUnit / 2) + j] = __byte_perm(v[2 * j], v[2 * j + 1], 0x5410);
        }
        if (!put(q, packed)) {
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
    // the whole warp runs the loop (warp-uniform values); one elected lane issues
    const int slot = __shfl_sync(0xffffffffu, warp - kMmaWarp, 0);
    const uint32_t idesc = HALF ? ptx::idesc_f16(kTileM, (uint32_t)p.Npad) : ptx::idesc_bf16(kTileM, (uint32_t)p.Npad);
    const uint32_t bsa = ptx::smem_addr(b_s);
    const uint32_t d_tmem = tmem + (uint32_t)(slot * p.Npad);
    const int64_t my_tiles = cta_tile_count(p);
    bool aborted = false;
    for (int64_t it = slot; it < my_tiles && !aborted; it += nslots) {
      const int64_t li = it / nslots;
      if (!__all_sync(0xffffffffu, wait_phase(bar_d_empty + 8 * slot, ((uint32_t)li & 1) ^ 1, abort_flag, p.wait_limit,
                                                  kWaitSiteDEmpty))) break;
      ptx::tc_fence_after();
      for (int q = 0; q < p.nchunks; ++q) {
        const uint32_t lg = (uint32_t)li * (uint32_t)p.nchunks + (uint32_t)q;
        const uint32_t s = (uint32_t)(2 * slot + (int)(lg & 1)), r = lg >> 1;
        bool ok = wait_phase(bar_a_full + 8 * s, r & 1, abort_flag, p.wait_limit, kWaitSiteAFull);
        if (SB && ok) ok = wait_phase(bar_b_full + 8 * s, r & 1, abort_flag, p.wait_limit, kWaitSiteBFull);
        if (!__all_sync(0xffffffffu, ok)) {
          aborted = true;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a = tmem + a_col0 + 16u * s;
        if (ptx::elect_one()) {
#pragma unroll
          for (int ks = 0; ks < kBfChunk / 16; ++ks) {
            const uint32_t kbyte = (uint32_t)((q * kBfChunk + ks * 16) / 8) * 128u;  // core matrices along K
            // streamed: the stage holds chunk q only, 8-row groups 512 bytes apart
            const uint64_t bd = SB ? ptx::smem_desc_noswizzle(bsa + s * p.sb_stage_bytes + 256u * ks, 128, 512)
                                   : ptx::smem_desc_noswizzle(bsa + kbyte, 128, SBO);
            ptx::mma_f16_ts(d_tmem, a + 8u * ks, bd, idesc, (q | ks) != 0);
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
