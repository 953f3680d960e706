// Small-T rungs: T = 1 ("gemv"), T = 2..8 ("small_t"), T = 9..16
// ("small_t_tiled").
//
//   y[t][n] = sum_g s[n][g] * sum_{k in g} w[n][k] * x[t][k]   (fp32 out)
//
// These rungs stream 2-bit weights, so the design goal is the weight stream at
// HBM speed with as few instructions per weight as possible (GB300 has ~1.5
// fp32 lane-ops per weight at full HBM rate; a CUDA-core or mma.sync GEMV
// spends more than that on decode and fragment traffic alone).
//
// 1. Activation split (xprep_kernel, once per call).  Per token and per
//    128-wide group, x is scaled by a power of two 2^p so that the group's
//    absmax lies in [128, 256), then split exactly into two fp8 e4m3 pieces
//    x 2^p = h1 + h2 (h1 = RN_e4m3(x 2^p), h2 = RN_e4m3(x 2^p - h1)).  A bf16
//    value has 8 significant bits and each piece holds 4, so the split is
//    exact for every element within 2^-10 of its group's absmax; smaller ones
//    keep an absolute error below 2^-10 * 2^-p.  The pieces are the columns of
//    the MMA's B operand (column piece * H + token), written straight into the
//    tcgen05 K-major shared-memory layout, one contiguous block per 512-wide k
//    stage, followed by the per-(group, token) factors f = 2^(3-p).
// 2. Weights as fp8, decoded into tensor memory.  The packed code puts each
//    weight's nonzero bit and sign bit at the 2^-3 exponent bit and the sign
//    bit of an e4m3 byte once shifted, so one shift and one AND turn a packed
//    word into four exact e4m3 values w/8.  Each decode thread owns one of
//    the CTA's 128 rows (one TMEM lane) and stores its decoded row chunk with
//    tcgen05.st into a double-buffered A operand in TMEM.
// 3. One thread issues tcgen05.mma kind::f8f6f4 (A in TMEM, B in shared
//    memory, fp32 accumulator in TMEM), one 128 x N x 128 accumulator per
//    128-wide group; the decode threads read it back with tcgen05.ld and fold
//    it into their row's running sums with s[n][g] * f[g][token].
//
// Pipeline (one CTA per SM, persistent; TMEM 512 columns):
//   warp 4   producer: one 2D TMA box of packed weights (128 rows x 128 B,
//            128-byte swizzle) + one bulk copy of the stage's activation block
//            + cp.async of the stage's fp16 scales, into a ring of stages;
//   warps 0-3 decode stage i into A[i & 1], then fold stage i-1;
//   warp 5   allocates TMEM and issues the MMAs of stage i once A[i & 1] is
//            full and D[i & 1] has been drained.
// The (row block, 512-wide k stage) units are cut into equal contiguous
// ranges, one per CTA, so every SM streams the same bytes; a row block that
// straddles two CTAs is finished with fp32 atomics into a y the prep kernel
// zeroed.  The main kernel is a programmatic dependent of the prep kernel, so
// its prologue and first weight loads overlap the prep.
//
// The pages' kernel for this band (the "small_t" rung of the
// "ninfer-perf-tuning" skill page, sections 2 and 6) decodes through a LUT
// into warp-level MMAs with one warp per 16 rows over all of K.  On GB300 the
// warp-level MMA path is instruction-bound well below the HBM rate, so here
// the decode is a mask, the multiply is tcgen05, and the grid is balanced over
// (rows x k) instead of rows alone.
#include "tern_device.cuh"
#include "tern_internal.h"

#include <cuda_fp8.h>

namespace tern {
namespace {

constexpr int kRows = 128;       // rows per CTA row block (MMA M, TMEM lanes)
constexpr int kDecWarps = 8;     // two decode threads per row (groups split in halves)
constexpr int kThreads = (kDecWarps + 2) * 32;
constexpr int kProducerWarp = kDecWarps;
constexpr int kMmaWarp = kDecWarps + 1;
constexpr uint32_t kXLbo = 128;            // K-direction core-matrix stride in the B block
constexpr uint32_t kXSbo = kSTStageK / 16 * 128;  // N-direction stride (512 k per stage)

template <int TT>
struct TC {
  static constexpr int kH = TT <= 8 ? 8 : 16;  // B columns per piece
  static constexpr int kNC = 2 * kH;           // MMA N: 16 or 32
  static constexpr int kXFrag = kNC * kSTStageK;
  static constexpr int kXF = 4 * kH * 4;       // f[group 4][kH] fp32
  static constexpr int kXBytes = kXFrag + kXF;
  static constexpr int kStages = kNC == 16 ? 6 : 5;
  static constexpr int kWBytes = kRows * 128;
  static constexpr int kSBytes = kRows * 8;
  static constexpr int kWOff = 0;  // 1024-aligned for the 128-byte swizzle
  static constexpr int kXOff = kWOff + kStages * kWBytes;
  static constexpr int kSOff = kXOff + kStages * kXBytes;
  static constexpr int kBarOff = kSOff + kStages * kSBytes;
  // full, empty, afull[2], mdone[2], dfree[2], xch_full, xch_empty
  static constexpr int kNumBars = 2 * kStages + 8;
  static constexpr int kTmemSlot = kBarOff + kNumBars * 8;
  static constexpr int kXchOff = kTmemSlot + 16;             // partial sums [TT][128] fp32
  static constexpr int kBytes = kXchOff + TT * kRows * 4;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kACol = 0;    // A[2]: 128 columns each (512 k of e4m3)
  static constexpr uint32_t kDCol = 256;  // D[2]: 4 groups x kNC columns each
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kDCol + 2 * 4 * kNC <= kTmemCols, "TMEM budget");
  static_assert(kXBytes % 16 == 0, "bulk copy size");
};

// ------------------------------------------------------------------ prep
// One warp per (token slot t < H, 128-wide group).  Lane l holds k = 4l .. 4l+3
// of the group.  Slot order inside each 16-wide block of k is the transpose
// the decoder produces: slot 4i + b holds k = 4b + i.
template <int TT>
__global__ void __launch_bounds__(256) xprep_kernel(const uint16_t* __restrict__ x,
                                                    uint8_t* __restrict__ out, float* y, int K,
                                                    int N, int tok0, int Tt, int KS, int zero_y) {
  grid_dependents_launch();
  using C = TC<TT>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int task = blockIdx.x * 8 + warp;
  const int groups = 4 * KS;
  if (task < C::kH * groups) {
    const int t = task / groups;
    const int gi = task % groups;
    const int ks = gi >> 2, jg = gi & 3;
    const int kbase = gi * 128 + 4 * lane;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (t < Tt && kbase < K) {
      const uint2 raw =
          *reinterpret_cast<const uint2*>(x + static_cast<size_t>(tok0 + t) * K + kbase);
      v[0] = __uint_as_float(raw.x << 16);
      v[1] = __uint_as_float(raw.x & 0xFFFF0000u);
      v[2] = __uint_as_float(raw.y << 16);
      v[3] = __uint_as_float(raw.y & 0xFFFF0000u);
    }
    float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    int p = 0;
    float f = 0.f;
    if (m > 0.f) {
      int e;
      (void)frexpf(m, &e);  // m = fr * 2^e, fr in [0.5, 1)
      p = 8 - e;            // m * 2^p in [128, 256)
      f = ldexpf(1.0f, 3 - p);
    }
    uint8_t* st = out + static_cast<size_t>(ks) * C::kXBytes;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float xs = ldexpf(v[i], p);
      const __nv_fp8_storage_t h1 = __nv_cvt_float_to_fp8(xs, __NV_SATFINITE, __NV_E4M3);
      const float h1f = __half2float(__half(__nv_cvt_fp8_to_halfraw(h1, __NV_E4M3)));
      const __nv_fp8_storage_t h2 = __nv_cvt_float_to_fp8(xs - h1f, __NV_SATFINITE, __NV_E4M3);
      // k = 4 lane + i: 16-block lane/4, position b = lane%4, i -> slot 4i + b
      const int slot = 128 * jg + 16 * (lane >> 2) + 4 * i + (lane & 3);
#pragma unroll
      for (int piece = 0; piece < 2; ++piece) {
        const int n = piece * C::kH + t;
        const int off = (n >> 3) * kXSbo + (slot >> 4) * kXLbo + (n & 7) * 16 + (slot & 15);
        st[off] = piece ? h2 : h1;
      }
    }
    if (lane == 0) reinterpret_cast<float*>(st + C::kXFrag)[jg * C::kH + t] = f;
  }
  if (zero_y) {
    const long long total = static_cast<long long>(Tt) * N;
    float* yt = y + static_cast<size_t>(tok0) * N;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
      yt[i] = 0.f;
  }
}

// ------------------------------------------------------------------ main
template <int TT>
__global__ void __launch_bounds__(kThreads, 1)
    smallt_kernel(const __grid_constant__ CUtensorMap tmW, const uint16_t* __restrict__ scales,
                  const uint8_t* __restrict__ xprep, float* __restrict__ y, int K, int N,
                  int tok0, int Tt, int KS, long long U, int* err) {
  using C = TC<TT>;
  constexpr int S = C::kStages;
  constexpr int H = C::kH;
  constexpr int NC = C::kNC;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + S;
  uint64_t* afull = empty + S;
  uint64_t* mdone = afull + 2;
  uint64_t* dfree = mdone + 2;
  uint64_t* xch_full = dfree + 2;
  uint64_t* xch_empty = xch_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kTmemSlot);
  float* xbuf = reinterpret_cast<float*>(smem + C::kXchOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = K >> 7;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 32);          // producer lanes (+ TMA / bulk bytes)
      mbar_init(&empty[s], kDecWarps);  // stage folded
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&afull[b], kDecWarps);  // A[b] decoded
      mbar_init(&mdone[b], 1);          // MMAs reading A[b] / writing D[b] done (commit)
      mbar_init(&dfree[b], kDecWarps);  // D[b] drained
    }
    mbar_init(xch_full, kDecWarps / 2);   // upper decode half's partial sums written
    mbar_init(xch_empty, kDecWarps / 2);  // ... and consumed
    fence_mbar_init();
    prefetch_tensormap(&tmW);
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  const long long P = gridDim.x;
  const long long begin = U * blockIdx.x / P;
  const long long end = U * (blockIdx.x + 1) / P;
  const int nunits = static_cast<int>(end - begin);
  // first unit's (row block, k stage); later ones advance incrementally
  const int rb0 = static_cast<int>(begin / KS);
  const int ks0 = static_cast<int>(begin - static_cast<long long>(rb0) * KS);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    int it = 0;
    bool dep_ready = false;
    int rb = rb0, ks = ks0;
    for (; it < nunits; ++it) {
      const int s = it % S;
      if (it >= S && !__all_sync(0xffffffffu, mbar_wait(&empty[s], ((it / S) & 1) ^ 1, err))) break;
      uint8_t* xs = smem + C::kXOff + s * C::kXBytes;
      if (lane == 0) {
        mbar_expect_tx(&full[s], C::kWBytes + C::kXBytes);
        tma_load_2d(smem + C::kWOff + s * C::kWBytes, &tmW, ks * 128, rb * kRows, &full[s]);
        if (!dep_ready) {
          grid_dependency_wait();  // the activation blocks come from the prep kernel
          dep_ready = true;
        }
        bulk_load(xs, xprep + static_cast<size_t>(ks) * C::kXBytes, C::kXBytes, &full[s]);
      }
      // fp16 scales of groups 4 ks .. 4 ks + 3 for rows lane + 32 i
      uint2* sb = reinterpret_cast<uint2*>(smem + C::kSOff + s * C::kSBytes);
      const int g0 = ks * 4;
      if ((G & 3) == 0) {
#pragma unroll
        for (int i = 0; i < kRows / 32; ++i) {
          const int r = lane + 32 * i;
          const int n = rb * kRows + r;
          const bool in = n < N;
          cp_async_8(&sb[r], scales + static_cast<size_t>(in ? n : 0) * G + g0, in ? 8u : 0u);
        }
        cp_async_mbar_arrive(&full[s]);
      } else {
#pragma unroll
        for (int i = 0; i < kRows / 32; ++i) {
          const int r = lane + 32 * i;
          const int n = rb * kRows + r;
          uint2 v = make_uint2(0, 0);
          if (n < N) {
            const uint16_t* src = scales + static_cast<size_t>(n) * G + g0;
            uint32_t h[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) h[j] = (g0 + j < G) ? src[j] : 0u;
            v = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
          }
          sb[r] = v;
        }
        mbar_arrive(&full[s]);
      }
      if (++ks == KS) {
        ks = 0;
        ++rb;
      }
    }
    // Stay until this CTA's copies have landed (bounded).
    for (int d = (it > S ? it - S : 0); d < it; ++d)
      if (!mbar_wait(&full[d % S], (d / S) & 1, err)) break;
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop so that addresses and descriptors stay
    // warp-uniform; one elected lane issues.
    const bool leader = elect_one();
    constexpr uint32_t idesc = idesc_e4m3_f32(kRows, NC);
    // Descriptor of stage 0's B block; a stage / k chunk only moves the start
    // address field (address >> 4 in the low bits).
    const uint64_t desc0 = smem_desc_kmajor(smem_addr(smem + C::kXOff), kXLbo, kXSbo);
    int it = 0;
    int ks = ks0;
    for (; it < nunits; ++it) {
      const int b = it & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&afull[b], (it >> 1) & 1, err))) break;
      if (it >= 2 && !__all_sync(0xffffffffu, mbar_wait(&dfree[b], ((it >> 1) & 1) ^ 1, err)))
        break;
      tc_fence_after();
      const uint64_t dstage = desc0 + static_cast<uint64_t>(((it % S) * C::kXBytes) >> 4);
      const uint32_t dcol = tbase + C::kDCol + b * 4 * NC;
      const uint32_t acol = tbase + C::kACol + b * 128;
      const int ng = G - 4 * ks < 4 ? G - 4 * ks : 4;
      if (leader) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          if (g < ng) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f8f6f4_ts(dcol + g * NC, acol + g * 32 + kk * 8,
                            dstage + static_cast<uint64_t>(((8 * g + 2 * kk) * kXLbo) >> 4), idesc,
                            kk > 0);
          }
        }
        mma_commit(&mdone[b]);
      }
      __syncwarp();
      if (++ks == KS) ks = 0;
    }
    // Before TMEM is released, the last MMAs issued must have completed.
    for (int d = (it > 2 ? it - 2 : 0); d < it; ++d)
      if (!mbar_wait(&mdone[d & 1], (d >> 1) & 1, err)) break;
  } else {
    // ------------------------------------------------------------ decode + fold
    // Warp w owns TMEM lane quarter q = w % 4 (rows 32 q .. 32 q + 31) and the
    // two groups 2 h, 2 h + 1 (h = w / 4) of every stage.
    const int q = warp & 3;
    const int h = warp >> 2;
    const int r = q * 32 + lane;  // row within the block == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    float yacc[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) yacc[t] = 0.f;
    int cur_rb = -1;
    bool cur_from_start = false;
    int cur_last_ks = -1;
    bool dep_ready = false;
    bool ok = true;
    int nflush = 0;

    // Both halves hold partial sums of the same rows: the upper half hands its
    // sums over through shared memory, the lower half adds and writes y.
    auto flush = [&](int rb, bool whole) -> bool {
      if (!dep_ready) {
        grid_dependency_wait();  // y was zeroed by the prep kernel
        dep_ready = true;
      }
      bool fine = true;
      if (h == 1) {
        if (nflush > 0)
          fine = __all_sync(0xffffffffu, mbar_wait(xch_empty, (nflush - 1) & 1, err));
        if (fine) {
#pragma unroll
          for (int t = 0; t < TT; ++t) xbuf[t * kRows + r] = yacc[t];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(xch_full);
      } else {
        fine = __all_sync(0xffffffffu, mbar_wait(xch_full, nflush & 1, err));
        if (fine) {
          const int n = rb * kRows + r;
#pragma unroll
          for (int t = 0; t < TT; ++t) {
            const float v = yacc[t] + xbuf[t * kRows + r];
            if (n < N && t < Tt) {
              float* dst = y + static_cast<size_t>(tok0 + t) * N + n;
              if (whole) *dst = v;
              else atomicAdd(dst, v);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(xch_empty);
      }
#pragma unroll
      for (int t = 0; t < TT; ++t) yacc[t] = 0.f;
      ++nflush;
      return fine;
    };

    auto fold = [&](int j, int rb, int ks) -> bool {
      const int b = j & 1;
      const int s = j % S;
      if (!__all_sync(0xffffffffu, mbar_wait(&mdone[b], (j >> 1) & 1, err))) return false;
      tc_fence_after();
      if (rb != cur_rb) {
        if (cur_rb >= 0 && !flush(cur_rb, cur_from_start && cur_last_ks == KS - 1)) return false;
        cur_rb = rb;
        cur_from_start = (ks == 0);
      }
      cur_last_ks = ks;
      const int ng = G - 4 * ks < 4 ? G - 4 * ks : 4;
      // scales of groups 2h, 2h+1 for this row
      const uint32_t sw =
          *reinterpret_cast<const uint32_t*>(smem + C::kSOff + s * C::kSBytes + r * 8 + 4 * h);
      const float* fv =
          reinterpret_cast<const float*>(smem + C::kXOff + s * C::kXBytes + C::kXFrag);
      // Only the accumulator columns that carry tokens are read back (TMEM
      // loads are the scarce resource of this loop): piece 0 of token t is
      // column t, piece 1 is column H + t.
      uint32_t d[2][NC];
#pragma unroll
      for (int gg = 0; gg < 2; ++gg) {
        const int g = 2 * h + gg;
        if (g < ng) {
          const uint32_t dbase = tbase + lane_off + C::kDCol + (b * 4 + g) * NC;
          if constexpr (TT == 1) {
            tmem_ld1(dbase, d[gg][0]);
            tmem_ld1(dbase + H, d[gg][H]);
          } else if constexpr (TT == 4) {
            tmem_ld4(dbase, d[gg]);
            tmem_ld4(dbase + H, d[gg] + H);
          } else {
            tmem_ld16(dbase, d[gg]);
            if constexpr (NC == 32) tmem_ld16(dbase + 16, d[gg] + 16);
          }
        }
      }
      tmem_wait_ld();
#pragma unroll
      for (int gg = 0; gg < 2; ++gg) {
        const int g = 2 * h + gg;
        if (g < ng) {
          const float sg = __half2float(__ushort_as_half(
              static_cast<unsigned short>(gg ? (sw >> 16) : (sw & 0xFFFFu))));
#pragma unroll
          for (int t = 0; t < TT; ++t)
            yacc[t] = fmaf(sg * fv[g * H + t],
                           __uint_as_float(d[gg][t]) + __uint_as_float(d[gg][H + t]), yacc[t]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&dfree[b]);
        mbar_arrive(&empty[s]);
      }
      return true;
    };

    int it = 0;
    int rb = rb0, ks = ks0, prb = rb0, pks = ks0;  // this unit and the previous one
    for (; it < nunits && ok; ++it) {
      const int s = it % S;
      const int b = it & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (it / S) & 1, err))) {
        ok = false;
        break;
      }
      // A[b] is free: the MMAs of unit it-2 completed (waited in fold(it-2)).
      const uint8_t* wrow = smem + C::kWOff + s * C::kWBytes + r * 128;
      const int ng = G - 4 * ks < 4 ? G - 4 * ks : 4;
#pragma unroll
      for (int gg = 0; gg < 2; ++gg) {
        const int g = 2 * h + gg;
        if (g < ng) {
          const uint4 c0 = lds_v4(wrow + (((2 * g) ^ (r & 7)) << 4));
          const uint4 c1 = lds_v4(wrow + (((2 * g + 1) ^ (r & 7)) << 4));
          const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          uint32_t a[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            a[4 * j + 0] = decode_e4m3<0>(w[j]);
            a[4 * j + 1] = decode_e4m3<1>(w[j]);
            a[4 * j + 2] = decode_e4m3<2>(w[j]);
            a[4 * j + 3] = decode_e4m3<3>(w[j]);
          }
          tmem_st32(tbase + lane_off + C::kACol + b * 128 + g * 32, a);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&afull[b]);
      if (it >= 1 && !fold(it - 1, prb, pks)) {
        ok = false;
        break;
      }
      prb = rb;
      pks = ks;
      if (++ks == KS) {
        ks = 0;
        ++rb;
      }
    }
    if (ok && nunits > 0 && fold(nunits - 1, prb, pks) && cur_rb >= 0)
      flush(cur_rb, cur_from_start && cur_last_ks == KS - 1);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tbase, C::kTmemCols);
}

template <int TT>
cudaError_t set_attr_one() {
  return cudaFuncSetAttribute(smallt_kernel<TT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TC<TT>::kAlloc);
}

template <int TT>
cudaError_t launch_tt(const CUtensorMap* tmW, const uint16_t* scales, const uint16_t* x,
                      uint8_t* xprep, float* y, int K, int N, int tok0, int Tt, int num_sms,
                      int* err, cudaStream_t stream) {
  using C = TC<TT>;
  const int KS = (K + kSTStageK - 1) / kSTStageK;
  const long long NB = (N + kRows - 1) / kRows;
  const long long U = NB * KS;
  long long P = num_sms;  // one CTA per SM: each holds all 512 TMEM columns
  if (P > U) P = U;
  // Does the split of U units over P CTAs cut a row block between two CTAs?
  bool cut = false;
  for (long long p = 1; p < P && !cut; ++p) cut = (U * p / P) % KS != 0;

  const int tasks = C::kH * 4 * KS;
  xprep_kernel<TT><<<(tasks + 7) / 8, 256, 0, stream>>>(x, xprep, y, K, N, tok0, Tt, KS,
                                                         cut ? 1 : 0);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(P));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, smallt_kernel<TT>, *tmW, scales,
                            static_cast<const uint8_t*>(xprep), y, K, N, tok0, Tt, KS, U, err);
}

}  // namespace

size_t smallt_xprep_bytes(int tt, int K) {
  const int KS = (K + kSTStageK - 1) / kSTStageK;
  int per = 0;
  switch (tt) {
    case 1: per = TC<1>::kXBytes; break;
    case 4: per = TC<4>::kXBytes; break;
    case 8: per = TC<8>::kXBytes; break;
    default: per = TC<16>::kXBytes; break;
  }
  return static_cast<size_t>(per) * KS;
}

int smallt_rows(int) { return kRows; }

cudaError_t smallt_set_attributes() {
  cudaError_t e;
  if ((e = set_attr_one<1>()) != cudaSuccess) return e;
  if ((e = set_attr_one<4>()) != cudaSuccess) return e;
  if ((e = set_attr_one<8>()) != cudaSuccess) return e;
  if ((e = set_attr_one<16>()) != cudaSuccess) return e;
  return cudaSuccess;
}

int smallt_ctas_per_sm(int) { return 1; }

cudaError_t launch_smallt(int tt, const CUtensorMap* tmW, const uint16_t* scales,
                          const uint16_t* x, uint8_t* xprep, float* y, int K, int N, int tok0,
                          int Tt, int num_sms, int ctas_per_sm, int* err, cudaStream_t stream) {
  (void)ctas_per_sm;
  switch (tt) {
    case 1: return launch_tt<1>(tmW, scales, x, xprep, y, K, N, tok0, Tt, num_sms, err, stream);
    case 4: return launch_tt<4>(tmW, scales, x, xprep, y, K, N, tok0, Tt, num_sms, err, stream);
    case 8: return launch_tt<8>(tmW, scales, x, xprep, y, K, N, tok0, Tt, num_sms, err, stream);
    default:
      return launch_tt<16>(tmW, scales, x, xprep, y, K, N, tok0, Tt, num_sms, err, stream);
  }
}

}  // namespace tern
