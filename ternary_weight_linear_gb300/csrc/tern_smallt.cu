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
// 1. Activation split.  Per token and per 128-wide group, x is scaled by a
//    power of two 2^p so that the group's absmax lies in [128, 256), then
//    split exactly into two fp8 e4m3 pieces x 2^p = h1 + h2
//    (h1 = RN_e4m3(x 2^p), h2 = RN_e4m3(x 2^p - h1)).  A bf16 value has 8
//    significant bits and each piece holds 4, so the split is exact for every
//    element within 2^-10 of its group's absmax; smaller ones keep an
//    absolute error below 2^-10 * 2^-p.  The pieces are the columns of the
//    MMA's B operand (column piece * H + token) in the tcgen05 K-major
//    shared-memory layout, one block per 1024-wide k stage, with the
//    per-(group, token) factors f = 2^(3-p).  At T = 1 four warps of the
//    main kernel build the blocks of every stage the CTA visits once, into
//    shared memory where they stay (a compact layout: see kX1Lbo); for wider
//    token tiles a prep kernel builds all blocks once per call and the main
//    kernel copies each stage's block in with its weights.
// 2. Weights as fp8, decoded into tensor memory.  The packed code puts each
//    weight's nonzero bit and sign bit at the 2^-3 exponent bit and the sign
//    bit of an e4m3 byte once shifted, so one shift and one AND turn a packed
//    word into four exact e4m3 values w/8.  Decode threads own rows of the
//    CTA's 128-row block (one TMEM lane each) and store decoded row chunks
//    with tcgen05.st into the A operand in TMEM.
// 3. One thread issues tcgen05.mma kind::f8f6f4 (A in TMEM, B in shared
//    memory, fp32 accumulator in TMEM), one 128 x N x 128 accumulator per
//    128-wide group; fold threads read it back with tcgen05.ld and fold it
//    into their row's running sums with s[n][g] * f[g][token].
//
// Pipeline (one CTA per SM, persistent; TMEM 512 columns):
//   warp 16    producer: two 2D TMA boxes of packed weights (128 rows x 128 B
//              each, 128-byte swizzle) per stage into the weight ring (plus,
//              for T > 1, a bulk copy of the stage's activation block); the
//              stage's fp16 scales (cp.async) into a longer scale ring;
//   warps 19-22 (T = 1) build the resident activation blocks and factors;
//   warps 0-7  decode (four groups of 32 rows per warp) into A slots;
//   warps 17-18 issue the MMAs of half-stage 0 / 1 of every stage once its
//              A slot is full and its D slot has been drained (warp 17 also
//              allocates TMEM);
//   warps 8-15 fold D slots into per-row running sums (two threads per row,
//              one per half-stage) and write y at the end of each row block.
//
// Work split: the (row block, 1024-wide k stage) units are cut into equal
// contiguous ranges, one per CTA, so every SM streams the same bytes.  A row
// block whole inside one CTA is written to y directly.  A row block split
// between CTAs is summed with fp32 atomics into y: at its start every CTA
// zeroes the y rows of its split row blocks and counts itself in the
// workspace's arrival counter, and it adds into y only once the counter
// shows that all CTAs of the launch have zeroed (by then, in practice, long
// since true).  The atomics make the order of those few additions, and so
// the last bits of split rows, vary from run to run.
//
// A stage is 1024 k: two 128-byte weight boxes per row, eight groups; a
// half-stage is one box, four groups.  TMEM is used in half-stage slots: the
// decode warps of groups 0-3 and of groups 4-7 each fill their own A slot,
// the MMAs of a half-stage write their own D slot, so decode, MMA and fold
// can run half-stages apart; each A slot is filled and released in two
// halves (groups 0-1, 2-3), so a half-stage's MMAs overlap the decoding of
// its next use.  (Doubling the stage from 512 k halved every role's barrier
// hand-offs per byte, which bound the pipeline.)
//
// Calls chain by programmatic dependent launch: every kernel lets the next one
// launch as soon as all of its CTAs run; the next kernel's CTAs set up, warm
// L2 with their first weight tiles and wait for the previous grid before they
// read anything it may have written (weights, x) or write y / the workspace.
// Every ring of slots has an even length, so a slot only ever holds
// half-stages of one parity (one decode half, one MMA issuer, one fold half):
// a waiter's barrier is then never two phases behind it.
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
// Two fold threads per row: fold warp f owns TMEM lane quarter f % 4 and
// half-stage f / 4 (groups 2 (f / 4), 2 (f / 4) + 1) of every stage.
constexpr int kFoldWarps = 8;
constexpr int kProducerWarp = kDecWarps + kFoldWarps;
// Two MMA-issuing warps: the first issues half-stage 0 of every stage, the
// second half-stage 1, so a single issuing thread never paces the tensor pipe.
constexpr int kMmaWarp = kProducerWarp + 1;
constexpr int kMmaWarps = 2;
constexpr int kXWarp0 = kMmaWarp + kMmaWarps;  // (T = 1) activation warps, one per group
constexpr int kGS = kSTStageK / 128;       // 128-wide groups per stage
constexpr int kGH = kGS / 2;               // groups per half-stage
constexpr int kWBoxes = kSTStageK / 512;   // 128-byte TMA boxes per stage row
static_assert(kGH == 4 && kWBoxes * 4 == kGS, "a half-stage is one weight box");
constexpr uint32_t kXLbo = 128;            // K-direction core-matrix stride in the B block
constexpr uint32_t kXSbo = kSTStageK / 16 * 128;  // N-direction stride (one stage of k)
// T = 1 activation block of one stage: only B columns 0 (h1) and 8 (h2) carry
// data.  With a 16-byte K-direction stride, column r of a core matrix aliases
// column 0 of the core matrix r steps further along K, so each piece needs a
// single row of one byte per k (plus 112 bytes of overrun): the other 14
// accumulator columns receive shifted dot products that are never read.
constexpr uint32_t kX1Lbo = 16;
constexpr uint32_t kX1Sbo = kSTStageK + 128;  // h2 row
constexpr int kX1Stage = 2 * kX1Sbo;          // bytes per stage (h1 row, h2 row, overruns)
constexpr int kX1MaxStages = kSmallTT1MaxK / kSTStageK;

template <int TT>
struct TC {
  static constexpr int kH = TT <= 8 ? 8 : 16;  // B columns per piece
  static constexpr int kNC = 2 * kH;           // MMA N: 16 or 32
  static constexpr int kXFrag = kNC * kSTStageK;  // B operand of one k stage
  static constexpr int kXF = kGS * kH * 4;        // f[group][kH] fp32
  static constexpr int kXBytes = kXFrag + kXF;    // one stage block of the prep buffer
  static constexpr bool kInKernelX = TT == 1;     // x blocks built by the main kernel
  static constexpr int kXWarps = kInKernelX ? 4 : 0;  // two groups of every stage each
  static constexpr int kThreads = (kXWarp0 + kXWarps) * 32;
  // TMEM is used in half-stage slots (kGH groups): A slots of kGH x 32
  // columns (e4m3), D slots of kGH x kNC columns.
  // Both ring lengths are even: half-stage hu uses slot hu % n, so every
  // slot only ever holds half-stages of one parity, which one decode half,
  // one MMA issuer and one fold half own.  A barrier a waiter checks is then
  // never two phases behind it (with an odd length the slot alternates
  // between the halves, and an issuer could pass a parity check while the
  // other decode half was still one phase back).
  static constexpr int kNAH = 2;
  static constexpr int kNDH = TT <= 8 ? 4 : 2;
  static_assert(kNAH % 2 == 0 && kNDH % 2 == 0, "slot rings must not mix half-stage parities");
  static constexpr int kStages = TT == 1 ? 4 : 3;  // weight (+ activation) ring
  // Scale loads run kLead units ahead of the weight loads (T = 1: the weight
  // ring does not wait for the MMAs, so the fold must never wait for scales).
  static constexpr int kLead = kInKernelX ? 2 : 0;
  // scale (+ factor) ring: held until folded, which trails the weight ring
  // by up to (kNAH + kNDH) / 2 stages
  static constexpr int kSStages = kStages + kLead + (kNAH + kNDH + 1) / 2;
  static constexpr int kWBytes = kRows * kSTStageK / 4;  // kWBoxes boxes of 128 rows x 128 B
  static constexpr int kSBytes = kRows * 2 * kGS + (kInKernelX ? 0 : kXF);  // scales [128][kGS], f
  static constexpr int kWOff = 0;  // 1024-aligned for the 128-byte swizzle
  static constexpr int kXOff = kWOff + kStages * kWBytes;  // activation ring (T > 1)
  static constexpr int kSOff = kXOff + (kInKernelX ? 0 : kStages * kXFrag);
  static constexpr int kFOff = kSOff + kSStages * kSBytes;  // (T = 1) f[stage][4]
  static constexpr int kBarOff = kFOff + (kInKernelX ? kX1MaxStages * kGS * 4 : 0);
  static constexpr int kNumBars =
      2 * kStages + 2 * kSStages + 4 * kNAH + 2 * kNDH + 8 + (kInKernelX ? kX1MaxStages : 0);
  static constexpr int kTmemSlot = kBarOff + kNumBars * 8;
  static constexpr int kFirstOff = kTmemSlot + 16;  // fold: parked first row block sums
  static constexpr int kPartOff = kFirstOff + TT * kRows * 4;  // fold: half-stage 1 sums
  static constexpr int kX1Off = (kPartOff + TT * kRows * 4 + 127) / 128 * 128;  // (T = 1)
  // shared memory for K: fixed part, the T = 1 blocks, alignment slack
  static constexpr int smem_bytes(int KS) {
    return kX1Off + (kInKernelX ? KS * kX1Stage : 0) + 1024;
  }
  static constexpr int kAllocMax = smem_bytes(kInKernelX ? kX1MaxStages : 0);
  static constexpr uint32_t kASlot = kGH * 32;     // A[kNAH] slots
  static constexpr uint32_t kDSlot = kGH * kNC;    // D[kNDH] slots
  static constexpr uint32_t kACol = 0;
  static constexpr uint32_t kDCol = kNAH * kASlot;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kDCol + kNDH * kDSlot <= kTmemCols, "TMEM budget");
  static_assert(kXFrag % 16 == 0 && kXF % 16 == 0 && kXBytes % 16 == 0, "bulk copy sizes");
  static_assert(kSBytes % 16 == 0 && kBarOff % 8 == 0, "alignment");
  static_assert(kAllocMax <= 227 * 1024, "shared memory");
};

// x 2^p -> (h1, h2), two e4m3 pieces with h1 + h2 == x 2^p for |x 2^p| < 256
// (up to the e4m3 resolution of the remainder, see above).
__device__ __forceinline__ void split_e4m3(float xs, uint8_t& h1, uint8_t& h2) {
  const __nv_fp8_storage_t a = __nv_cvt_float_to_fp8(xs, __NV_SATFINITE, __NV_E4M3);
  const float af = __half2float(__half(__nv_cvt_fp8_to_halfraw(a, __NV_E4M3)));
  h1 = a;
  h2 = __nv_cvt_float_to_fp8(xs - af, __NV_SATFINITE, __NV_E4M3);
}

// Power-of-two exponent p with m 2^p in [128, 256), and f = 2^(3-p); 0 / 0 for m = 0.
__device__ __forceinline__ void group_exponent(float m, int& p, float& f) {
  p = 0;
  f = 0.f;
  if (m > 0.f) {
    int e;
    (void)frexpf(m, &e);  // m = fr * 2^e, fr in [0.5, 1)
    p = 8 - e;
    f = ldexpf(1.0f, 3 - p);
  }
}

// CTA owning unit u when U units are cut into P equal contiguous ranges
// (CTA c holds units [U c / P, U (c + 1) / P)).
__device__ __forceinline__ int owner_of(long long u, long long U, long long P) {
  return static_cast<int>(((u + 1) * P - 1) / U);
}

// ------------------------------------------------------------------ prep
// Activation blocks of one token tile for all stages (T > 1).  One warp per
// (token slot t < H, 128-wide group).  Lane l holds k = 4l .. 4l+3 of the
// group.  Slot order inside each 16-wide block of k is the transpose the
// decoder produces: slot 4i + b holds k = 4b + i.
template <int TT>
__global__ void __launch_bounds__(256) xprep_kernel(const uint16_t* __restrict__ x,
                                                    uint8_t* __restrict__ out, int K, int tok0,
                                                    int Tt, int KS) {
  grid_dependents_launch();
  grid_dependency_wait();  // x (and this buffer's last reader) come from earlier work
  using C = TC<TT>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int task = blockIdx.x * 8 + warp;
  const int groups = kGS * KS;
  if (task >= C::kH * groups) return;
  const int t = task / groups;
  const int gi = task % groups;
  const int ks = gi / kGS, jg = gi % kGS;
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
  int p;
  float f;
  group_exponent(m, p, f);
  uint8_t* st = out + static_cast<size_t>(ks) * C::kXBytes;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint8_t hp[2];
    split_e4m3(ldexpf(v[i], p), hp[0], hp[1]);
    // k = 4 lane + i: 16-block lane/4, position b = lane%4, i -> slot 4i + b
    const int slot = 128 * jg + 16 * (lane >> 2) + 4 * i + (lane & 3);
#pragma unroll
    for (int piece = 0; piece < 2; ++piece) {
      const int n = piece * C::kH + t;
      const int off = (n >> 3) * kXSbo + (slot >> 4) * kXLbo + (n & 7) * 16 + (slot & 15);
      st[off] = hp[piece];
    }
  }
  if (lane == 0) reinterpret_cast<float*>(st + C::kXFrag)[jg * C::kH + t] = f;
}

// ------------------------------------------------------------------ main
// x: bf16 activations (read at T = 1); xprep: prep blocks (T > 1).
// arrivals: the workspace's launch-arrival counter (see the fold warps).
template <int TT>
__global__ void __launch_bounds__(TC<TT>::kThreads, 1)
    smallt_kernel(const __grid_constant__ CUtensorMap tmW, const uint16_t* __restrict__ scales,
                  const uint16_t* __restrict__ x, const uint8_t* __restrict__ xprep,
                  float* __restrict__ y, unsigned long long* __restrict__ arrivals, int K, int N,
                  int tok0, int Tt, int KS, long long U, int* err) {
  using C = TC<TT>;
  constexpr int S = C::kStages;
  constexpr int SS = C::kSStages;
  constexpr int NA = C::kNAH;
  constexpr int ND = C::kNDH;
  constexpr int H = C::kH;
  constexpr int NC = C::kNC;

  // The next kernel on the stream may launch now; it waits for this grid
  // before touching anything this one writes.
  grid_dependents_launch();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + S;     // weights decoded and activation block consumed
  uint64_t* sfull = empty + S;    // scales + factors landed
  uint64_t* sempty = sfull + SS;  // ... and folded
  // A slots are used in two halves (sub-slots 2 a and 2 a + 1: groups 0-1
  // and 2-3 of the half-stage), each with its own barriers, so the MMAs on
  // one half overlap the decoding of the other.
  uint64_t* afull = sempty + SS;     // A sub-slot written by its four decoders
  uint64_t* afree = afull + 2 * NA;  // MMAs reading A sub-slot completed
  uint64_t* mdone = afree + 2 * NA;  // MMAs writing D slot d completed
  uint64_t* dfree = mdone + ND;   // D slot d read back by the fold warps
  uint64_t* xready = dfree + ND;  // (T = 1) activation block of stage ks built
  // fold pairs: [quarter] the half-stage-1 warp's row block sums are in
  // shared memory / have been taken by the half-stage-0 warp
  uint64_t* pfull = xready + (C::kInKernelX ? kX1MaxStages : 0);
  uint64_t* pfree = pfull + 4;
  uint8_t* xres = smem + C::kX1Off;                              // (T = 1) blocks
  float* ftab = reinterpret_cast<float*>(smem + C::kFOff);       // (T = 1) f[ks][kGS]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = K >> 7;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);  // producer's expect_tx arrival
      // the decoders (+ one MMA commit per half-stage when the stage holds
      // activations)
      mbar_init(&empty[s], C::kInKernelX ? kDecWarps : kDecWarps + 2);
    }
    for (int s = 0; s < SS; ++s) {
      mbar_init(&sfull[s], 32);
      mbar_init(&sempty[s], kFoldWarps);
    }
    for (int a = 0; a < 2 * NA; ++a) {
      mbar_init(&afull[a], kDecWarps / 2);
      mbar_init(&afree[a], 1);
    }
    for (int d = 0; d < ND; ++d) {
      mbar_init(&mdone[d], 1);
      mbar_init(&dfree[d], kFoldWarps / 2);  // the four warps of its half-stage
    }
    if constexpr (C::kInKernelX)
      for (int k = 0; k < KS; ++k) mbar_init(&xready[k], kGS);  // one arrival per group
    for (int q = 0; q < 4; ++q) {
      mbar_init(&pfull[q], 1);
      mbar_init(&pfree[q], 1);
    }
    fence_mbar_init();
    prefetch_tensormap(&tmW);
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  const long long P = gridDim.x;
  const int cta = blockIdx.x;
  const long long begin = U * cta / P;
  const long long end = U * (cta + 1) / P;
  const int nunits = static_cast<int>(end - begin);
  // first unit's (row block, k stage); later ones advance incrementally
  const int rb0 = static_cast<int>(begin / KS);
  const int ks0 = static_cast<int>(begin - static_cast<long long>(rb0) * KS);
  // Every role but the producer (which first warms L2) waits for the previous
  // grid here, so that no bounded wait below starts its clock while a slow
  // predecessor is still running.
  if (warp != kProducerWarp) grid_dependency_wait();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Warm L2 with the first stages' weights and the first row block's
    // scales while the previous grid finishes; load only after it has.
    if (lane == 0) {
      int rb = rb0, ks = ks0;
      for (int it = 0; it < nunits && it < S; ++it) {
#pragma unroll
        for (int b = 0; b < kWBoxes; ++b)
          tma_prefetch_2d(&tmW, ks * (kSTStageK / 4) + 128 * b, rb * kRows);
        if (++ks == KS) {
          ks = 0;
          ++rb;
        }
      }
      const int rows = N - rb0 * kRows < kRows ? N - rb0 * kRows : kRows;
      const uint32_t sbytes = (static_cast<uint32_t>(rows) * G * 2) & ~15u;
      if (sbytes) bulk_prefetch_l2(scales + static_cast<size_t>(rb0) * kRows * G, sbytes);
    }
    grid_dependency_wait();
    // Scale stream: unit su's fp16 scales of groups kGS ks .. kGS ks + kGS - 1
    // for rows lane + 32 i (and, T > 1, its factors f), into scale ring slot
    // su % SS.
    int su = 0, srb = rb0, sks = ks0;
    auto issue_scales = [&]() -> bool {
      const int ss = su % SS;
      if (su >= SS &&
          !__all_sync(0xffffffffu, mbar_wait(&sempty[ss], ((su / SS) & 1) ^ 1, err)))
        return false;
      uint8_t* sst = smem + C::kSOff + ss * C::kSBytes;
      if constexpr (!C::kInKernelX) {
        if (lane == 0) {
          mbar_expect_tx(&sfull[ss], C::kXF);
          bulk_load(sst + kRows * 2 * kGS,
                    xprep + static_cast<size_t>(sks) * C::kXBytes + C::kXFrag, C::kXF,
                    &sfull[ss]);
        }
      }
      uint4* sb = reinterpret_cast<uint4*>(sst);
      const int g0 = sks * kGS;
      if ((G % kGS) == 0) {
        // whole 16-byte rows of scales
#pragma unroll
        for (int i = 0; i < kRows / 32; ++i) {
          const int r = lane + 32 * i;
          const int n = srb * kRows + r;
          const bool in = n < N;
          cp_async_16(&sb[r], scales + static_cast<size_t>(in ? n : 0) * G + g0, in ? 16u : 0u);
        }
        cp_async_mbar_arrive(&sfull[ss]);
      } else if ((G & 3) == 0) {
        // 8-byte halves; the second is past the row end in a short last stage
        const bool second = g0 + 4 < G;
#pragma unroll
        for (int i = 0; i < kRows / 32; ++i) {
          const int r = lane + 32 * i;
          const int n = srb * kRows + r;
          const bool in = n < N;
          const uint16_t* src = scales + static_cast<size_t>(in ? n : 0) * G + g0;
          cp_async_8(&sb[r], src, in ? 8u : 0u);
          cp_async_8(reinterpret_cast<uint8_t*>(&sb[r]) + 8, second ? src + 4 : src,
                     (in && second) ? 8u : 0u);
        }
        cp_async_mbar_arrive(&sfull[ss]);
      } else {
#pragma unroll
        for (int i = 0; i < kRows / 32; ++i) {
          const int r = lane + 32 * i;
          const int n = srb * kRows + r;
          uint32_t hv[kGS];
#pragma unroll
          for (int j = 0; j < kGS; ++j) hv[j] = 0u;
          if (n < N) {
            const uint16_t* src = scales + static_cast<size_t>(n) * G + g0;
#pragma unroll
            for (int j = 0; j < kGS; ++j) hv[j] = (g0 + j < G) ? src[j] : 0u;
          }
          sb[r] = make_uint4(hv[0] | (hv[1] << 16), hv[2] | (hv[3] << 16), hv[4] | (hv[5] << 16),
                             hv[6] | (hv[7] << 16));
        }
        mbar_arrive(&sfull[ss]);
      }
      ++su;
      if (++sks == KS) {
        sks = 0;
        ++srb;
      }
      return true;
    };
    bool ok = true;
    while (ok && su < nunits && su < C::kLead) ok = issue_scales();
    int it = 0;
    int rb = rb0, ks = ks0;
    for (; it < nunits && ok; ++it) {
      const int s = it % S;
      if (it >= S && !__all_sync(0xffffffffu, mbar_wait(&empty[s], ((it / S) & 1) ^ 1, err))) break;
      if (lane == 0) {
        // activations are resident at T = 1; for T > 1 the stage's block comes along
        mbar_arrive_expect_tx(&full[s], C::kWBytes + (C::kInKernelX ? 0 : C::kXFrag));
#pragma unroll
        for (int bx = 0; bx < kWBoxes; ++bx)
          tma_load_2d(smem + C::kWOff + s * C::kWBytes + bx * (kRows * 128), &tmW,
                      ks * (kSTStageK / 4) + 128 * bx, rb * kRows, &full[s]);
        if constexpr (!C::kInKernelX)
          bulk_load(smem + C::kXOff + s * C::kXFrag,
                    xprep + static_cast<size_t>(ks) * C::kXBytes, C::kXFrag, &full[s]);
      }
      if (su < nunits) ok = issue_scales();
      if (++ks == KS) {
        ks = 0;
        ++rb;
      }
    }
    // Stay until this CTA's copies have landed (bounded).
    for (int d = (it > S ? it - S : 0); d < it; ++d)
      if (!mbar_wait(&full[d % S], (d / S) & 1, err)) break;
    for (int d = (su > SS ? su - SS : 0); d < su; ++d)
      if (!mbar_wait(&sfull[d % SS], (d / SS) & 1, err)) break;
  } else if (warp >= kXWarp0) {
    // ------------------------------------------------------------ activations (T = 1)
    // Activation warp xw builds groups xw and xw + 4 of every stage this CTA
    // visits, in visiting order, once: lane l splits k = 128 g + 4l .. +3 of
    // the stage.  Item qi is group xw + 4 (qi & 1) of the (qi >> 1)-th stage.
    if constexpr (C::kInKernelX) {
      const int xw = warp - kXWarp0;
      grid_dependency_wait();
      const uint16_t* xt = x + static_cast<size_t>(tok0) * K;
      const int nq = nunits < KS ? nunits : KS;
      const int nitems = 2 * nq;
      // loads of the next kXLoads items stay in flight while one is built
      constexpr int kXLoads = 8;
      uint2 raw[kXLoads];
      auto load_item = [&](int qi) -> uint2 {
        const int ks = (ks0 + (qi >> 1)) % KS;
        const int k = ks * kSTStageK + 128 * (xw + 4 * (qi & 1)) + 4 * lane;
        return (qi < nitems && k < K) ? *reinterpret_cast<const uint2*>(xt + k)
                                      : make_uint2(0, 0);
      };
#pragma unroll
      for (int j = 0; j < kXLoads; ++j) raw[j] = load_item(j);
      for (int q0 = 0; q0 < nitems; q0 += kXLoads) {
#pragma unroll
        for (int j = 0; j < kXLoads; ++j) {
          const int qi = q0 + j;
          if (qi >= nitems) break;
          const int ks = (ks0 + (qi >> 1)) % KS;
          const int g = xw + 4 * (qi & 1);
          const uint2 cur = raw[j];
          raw[j] = load_item(qi + kXLoads);
          const float v[4] = {__uint_as_float(cur.x << 16), __uint_as_float(cur.x & 0xFFFF0000u),
                              __uint_as_float(cur.y << 16), __uint_as_float(cur.y & 0xFFFF0000u)};
          float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          // floor(log2 m) from the bits; p = 7 - that puts m 2^p in [128, 256)
          float sc1 = 0.f, sc2 = 0.f, f = 0.f;
          if (m > 0.f) {
            const uint32_t mb = __float_as_uint(m);
            const int el =
                (mb >> 23) ? static_cast<int>(mb >> 23) - 127 : (31 - __clz(mb)) - 149;
            const int p = 7 - el;                // in [-120, 156]
            const int p1 = p >> 1, p2 = p - p1;  // each in [-60, 78]
            sc1 = __uint_as_float(static_cast<uint32_t>(p1 + 127) << 23);
            sc2 = __uint_as_float(static_cast<uint32_t>(p2 + 127) << 23);
            // f = 2^(3-p) = 2^(el-4): a normal power of two unless el is tiny
            f = el - 4 >= -126 ? __uint_as_float(static_cast<uint32_t>(el - 4 + 127) << 23)
                               : ldexpf(1.0f, el - 4);
          }
          uint32_t h1 = 0, h2 = 0;  // byte i: piece of k = 4l + i
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const float2 xs = make_float2((v[2 * hf] * sc1) * sc2, (v[2 * hf + 1] * sc1) * sc2);
            const __nv_fp8x2_storage_t a =
                __nv_cvt_float2_to_fp8x2(xs, __NV_SATFINITE, __NV_E4M3);
            const __half2_raw ar = __nv_cvt_fp8x2_to_halfraw2(a, __NV_E4M3);
            const float2 af = __half22float2(*reinterpret_cast<const __half2*>(&ar));
            const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(
                make_float2(xs.x - af.x, xs.y - af.y), __NV_SATFINITE, __NV_E4M3);
            h1 |= static_cast<uint32_t>(a) << (16 * hf);
            h2 |= static_cast<uint32_t>(c) << (16 * hf);
          }
          // 16-block 8 g + l/4, position b = l%4: value i goes to slot 4i + b
          uint8_t* blk = xres + ks * kX1Stage + (8 * g + (lane >> 2)) * 16 + (lane & 3);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            blk[4 * i] = static_cast<uint8_t>(h1 >> (8 * i));
            blk[kX1Sbo + 4 * i] = static_cast<uint8_t>(h2 >> (8 * i));
          }
          if (lane == 0) ftab[ks * kGS + g] = f;
          fence_proxy_async_smem();  // the MMA reads the block through the async proxy
          __syncwarp();
          if (lane == 0) mbar_arrive(&xready[ks]);
        }
      }
    }
  } else if (warp >= kMmaWarp && warp < kMmaWarp + kMmaWarps) {
    // ------------------------------------------------------------ MMA issuers
    // Each warp runs its loop whole so that addresses and descriptors stay
    // warp-uniform; one elected lane issues.  Half-stage hu = 2 it + hh
    // (groups 2 hh, 2 hh + 1) uses A slot hu % NA and D slot hu % ND and is
    // issued by MMA warp hh.
    const int w = warp - kMmaWarp;
    const bool leader = elect_one();
    constexpr uint32_t idesc = idesc_e4m3_f32(kRows, NC);
    // Descriptor of stage 0's B block; a stage / k chunk only moves the start
    // address field (address >> 4 in the low bits).
    const uint64_t desc0 =
        C::kInKernelX ? smem_desc_kmajor(smem_addr(xres), kX1Lbo, kX1Sbo)
                      : smem_desc_kmajor(smem_addr(smem + C::kXOff), kXLbo, kXSbo);
    constexpr uint32_t kLbo = C::kInKernelX ? kX1Lbo : kXLbo;
    int last = -1;
    for (int hu = w; hu < 2 * nunits; hu += kMmaWarps) {
      const int it = hu >> 1, hh = hu & 1;
      const int s = it % S;
      const int ks = static_cast<int>((ks0 + it) % KS);
      const int ng = G - kGS * ks < kGS ? G - kGS * ks : kGS;
      const uint64_t dstage =
          desc0 + static_cast<uint64_t>(
                      (C::kInKernelX ? ks * kX1Stage : s * C::kXFrag) >> 4);
      if constexpr (C::kInKernelX) {
        if (!__all_sync(0xffffffffu, mbar_wait(&xready[ks], 0, err))) break;
      }
      const int a = hu % NA;
      const int d = hu % ND;
      if (hu >= ND &&
          !__all_sync(0xffffffffu, mbar_wait(&dfree[d], ((hu / ND) & 1) ^ 1, err)))
        break;
      const uint32_t dcol = tbase + C::kDCol + d * C::kDSlot;
      const uint32_t acol = tbase + C::kACol + a * C::kASlot;
      bool ok_h = true;
#pragma unroll
      for (int b = 0; b < 2; ++b) {  // the two A sub-slots of the half-stage
        if (!__all_sync(0xffffffffu, mbar_wait(&afull[2 * a + b], (hu / NA) & 1, err))) {
          ok_h = false;
          break;
        }
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int gs = 0; gs < kGH / 2; ++gs) {
            const int gg = (kGH / 2) * b + gs;
            const int g = kGH * hh + gg;
            if (g < ng) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f8f6f4_ts(dcol + gg * NC, acol + gg * 32 + kk * 8,
                              dstage + static_cast<uint64_t>(((8 * g + 2 * kk) * kLbo) >> 4),
                              idesc, kk > 0);
            }
          }
          mma_commit(&afree[2 * a + b]);
        }
        __syncwarp();
      }
      if (!ok_h) break;
      if (leader) {
        if (!C::kInKernelX) mma_commit(&empty[s]);
        mma_commit(&mdone[d]);
      }
      __syncwarp();
      last = hu;
    }
    // Before TMEM is released, this warp's last MMAs must have completed.  The
    // D slot's barrier is still at that phase: with two issuers and an even
    // ring, only this issuer's own (earlier) half-stages use the slot.
    static_assert(kMmaWarps == 2 && ND % 2 == 0, "the last-slot wait needs two issuers");
    if (last >= 0) mbar_wait(&mdone[last % ND], (last / ND) & 1, err);
  } else if (warp < kDecWarps) {
    // ------------------------------------------------------------ decode
    // Warp w owns TMEM lane quarter q = w % 4 (rows 32 q .. 32 q + 31) and the
    // four groups 4 h .. 4 h + 3 (h = w / 4, the stage's weight box h) of
    // every stage.
    const int q = warp & 3;
    const int h = warp >> 2;
    const int r = q * 32 + lane;  // row within the block == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    int ks = ks0;
    for (int it = 0; it < nunits; ++it) {
      const int s = it % S;
      const int hu = 2 * it + h;  // this warp's half-stage
      const int a = hu % NA;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (it / S) & 1, err))) break;
      // half-stage h is weight box h: groups kGH h .. kGH h + kGH - 1
      const uint8_t* wrow = smem + C::kWOff + s * C::kWBytes + h * (kRows * 128) + r * 128;
      const int ng = G - kGS * ks < kGS ? G - kGS * ks : kGS;
      bool ok_h = true;
#pragma unroll
      for (int b = 0; b < 2; ++b) {  // A sub-slot b: groups 2 b, 2 b + 1 of the half-stage
        if (hu >= NA &&
            !__all_sync(0xffffffffu, mbar_wait(&afree[2 * a + b], ((hu / NA) & 1) ^ 1, err))) {
          ok_h = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int gs = 0; gs < kGH / 2; ++gs) {
          const int gg = (kGH / 2) * b + gs;
          const int g = kGH * h + gg;
          if (g < ng) {
            const uint4 c0 = lds_v4(wrow + (((2 * gg) ^ (r & 7)) << 4));
            const uint4 c1 = lds_v4(wrow + (((2 * gg + 1) ^ (r & 7)) << 4));
            const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            uint32_t av[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              av[4 * j + 0] = decode_e4m3<0>(w[j]);
              av[4 * j + 1] = decode_e4m3<1>(w[j]);
              av[4 * j + 2] = decode_e4m3<2>(w[j]);
              av[4 * j + 3] = decode_e4m3<3>(w[j]);
            }
            tmem_st32(tbase + lane_off + C::kACol + a * C::kASlot + gg * 32, av);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[2 * a + b]);
      }
      if (!ok_h) break;
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++ks == KS) ks = 0;
    }
  } else {
    // ------------------------------------------------------------ fold
    // Fold warp f owns TMEM lane quarter fq = f % 4 (rows 32 fq .. 32 fq + 31)
    // and half-stage fh = f / 4 (groups 2 fh, 2 fh + 1) of every stage:
    // y[t][row] += s[row][g] * f[g][t] * (D[g][piece 0, t] + D[g][piece 1, t]).
    // At the end of a row block the fh = 1 warp hands its sums to the fh = 0
    // warp of the same quarter, which writes y.
    const int fq = (warp - kDecWarps) & 3;  // == warp % 4
    const int fh = (warp - kDecWarps) >> 2;
    const int r = fq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(fq * 32) << 16;
    float yacc[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) yacc[t] = 0.f;

    // Row blocks split between CTAs are summed with fp32 atomics into y.
    // Every CTA first zeroes the y rows of its split row blocks, then adds to
    // the launch-arrival counter; a CTA adds into y only once the counter
    // shows that every writing fold warp of the launch has done its zeroing.
    // Each launch adds exactly 1024 in total, so the counter is a multiple of
    // 1024 between launches and needs no reset.  (Only the fh = 0 warps write
    // y, zero and count.)
    auto is_split = [&](int rb) {
      const long long u = static_cast<long long>(rb) * KS;
      return owner_of(u, U, P) != owner_of(u + KS - 1, U, P);
    };
    grid_dependency_wait();  // y and the workspace may be in use by earlier work
    const int rb_last = static_cast<int>((end - 1) / KS);
    unsigned long long arrival_target = 0;
    if (fh == 0) {
      const int zr[2] = {rb0, rb_last};
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if ((i == 1 && rb_last == rb0) || !is_split(zr[i])) continue;
        const int n = zr[i] * kRows + r;
        if (n < N)
          for (int t = 0; t < Tt; ++t) y[static_cast<size_t>(tok0 + t) * N + n] = 0.f;
      }
      __threadfence();
      __syncwarp();
      if (lane == 0) {
        const unsigned long long add =
            (cta == 0 && fq == 0) ? 1024ull - 4ull * static_cast<unsigned long long>(P) + 1ull
                                  : 1ull;
        arrival_target = (atomicAdd(arrivals, add) & ~1023ull) + 1024ull;
      }
      arrival_target = __shfl_sync(0xffffffffu, arrival_target, 0);
    }

    // A split row block's sums are added into y only after the arrival
    // counter shows every CTA has zeroed; so that the fold never stalls on
    // that check mid-stream, the first row block's sums (when split) wait in
    // shared memory and all atomics are issued once this CTA's last unit is
    // folded.
    float* first_part = reinterpret_cast<float*>(smem + C::kFirstOff);  // [TT][128]
    float* half_part = reinterpret_cast<float*>(smem + C::kPartOff);    // [TT][128]
    bool first_parked = false;
    int nflush = 0;
    // false: a bounded wait gave up (the error word is set)
    auto flush = [&](int rb) -> bool {
      const int n = rb * kRows + r;
      if (fh == 1) {
        // hand the sums over once the previous hand-over has been taken
        if (nflush > 0 &&
            !__all_sync(0xffffffffu, mbar_wait(&pfree[fq], (nflush - 1) & 1, err)))
          return false;
#pragma unroll
        for (int t = 0; t < TT; ++t) half_part[t * kRows + r] = yacc[t];
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[fq]);
      } else {
        if (!__all_sync(0xffffffffu, mbar_wait(&pfull[fq], nflush & 1, err))) return false;
#pragma unroll
        for (int t = 0; t < TT; ++t) yacc[t] += half_part[t * kRows + r];
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfree[fq]);
        if (!is_split(rb)) {
#pragma unroll
          for (int t = 0; t < TT; ++t)
            if (n < N && t < Tt) y[static_cast<size_t>(tok0 + t) * N + n] = yacc[t];
        } else if (rb == rb0 && rb != rb_last) {
#pragma unroll
          for (int t = 0; t < TT; ++t) first_part[t * kRows + r] = yacc[t];
          first_parked = true;
        } else {
          bool fine = true;
          if (lane == 0) fine = wait_counter_at_least(arrivals, arrival_target, err);
          fine = __shfl_sync(0xffffffffu, fine ? 1 : 0, 0) != 0;
          if (fine) {
#pragma unroll
            for (int t = 0; t < TT; ++t)
              if (n < N && t < Tt) atomicAdd(&y[static_cast<size_t>(tok0 + t) * N + n], yacc[t]);
            if (first_parked) {
              const int n0 = rb0 * kRows + r;
#pragma unroll
              for (int t = 0; t < TT; ++t)
                if (n0 < N && t < Tt)
                  atomicAdd(&y[static_cast<size_t>(tok0 + t) * N + n0],
                            first_part[t * kRows + r]);
              first_parked = false;
            }
          }
        }
      }
      ++nflush;
#pragma unroll
      for (int t = 0; t < TT; ++t) yacc[t] = 0.f;
      return true;
    };

    int ks = ks0;
    bool ok = true;
    for (int j = 0; j < nunits && ok; ++j) {
      const int ss = j % SS;
      if (!__all_sync(0xffffffffu, mbar_wait(&sfull[ss], (j / SS) & 1, err))) break;
      const int ng = G - kGS * ks < kGS ? G - kGS * ks : kGS;
      const uint8_t* sst = smem + C::kSOff + ss * C::kSBytes;
      // this half-stage's kGH fp16 scales
      const uint2 s4 = lds_v2(sst + r * (2 * kGS) + fh * (2 * kGH));
      // f[g][t] at fv[g * FH + t]
      constexpr int FH = C::kInKernelX ? 1 : H;
      const float* fv = C::kInKernelX ? ftab + ks * kGS
                                      : reinterpret_cast<const float*>(sst + kRows * 2 * kGS);
      if constexpr (C::kInKernelX) {
        if (!__all_sync(0xffffffffu, mbar_wait(&xready[ks], 0, err))) break;
      }
      const int hu = 2 * j + fh;
      const int d = hu % ND;
      if (!__all_sync(0xffffffffu, mbar_wait(&mdone[d], (hu / ND) & 1, err))) break;
      tc_fence_after();
      const uint32_t dbase = tbase + lane_off + C::kDCol + d * C::kDSlot;
      // only the accumulator columns that carry tokens are read back:
      // piece 0 of token t is column t, piece 1 is H + t
      auto fold_group = [&](int gg, const uint32_t* dv) {
        const uint32_t sp = gg < 2 ? s4.x : s4.y;
        const float sg = __half2float(__ushort_as_half(
            static_cast<unsigned short>((gg & 1) ? (sp >> 16) : (sp & 0xFFFFu))));
        const int g = kGH * fh + gg;
#pragma unroll
        for (int t = 0; t < TT; ++t)
          yacc[t] = fmaf(sg * fv[g * FH + t], __uint_as_float(dv[t]) + __uint_as_float(dv[H + t]),
                         yacc[t]);
      };
      static_assert(NC == 16 || NC == 32, "accumulator width");
      static_assert(TT == 1 || TT == 4 || TT == 8 || TT == 16, "token tiles");
      if constexpr (TT >= 8) {
        // 8 or 16 tokens: one group at a time keeps the live registers down
#pragma unroll
        for (int gg = 0; gg < kGH; ++gg) {
          uint32_t dv[NC];
          const bool has = kGH * fh + gg < ng;
          if (has) {
            tmem_ld16(dbase + gg * NC, dv);
            if constexpr (NC == 32) tmem_ld16(dbase + gg * NC + 16, dv + 16);
          }
          tmem_wait_ld();
          if (gg == kGH - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&dfree[d]);
          }
          if (has) fold_group(gg, dv);
        }
      } else {
        uint32_t dv[kGH][NC];
#pragma unroll
        for (int gg = 0; gg < kGH; ++gg) {
          if (kGH * fh + gg < ng) {
            const uint32_t col = dbase + gg * NC;
            if constexpr (TT == 1) {
              tmem_ld1(col, dv[gg][0]);
              tmem_ld1(col + H, dv[gg][H]);
            } else {
              tmem_ld4(col, dv[gg]);
              tmem_ld4(col + H, dv[gg] + H);
            }
          }
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dfree[d]);
#pragma unroll
        for (int gg = 0; gg < kGH; ++gg)
          if (kGH * fh + gg < ng) fold_group(gg, dv[gg]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[ss]);
      if (++ks == KS) {
        ok = flush(static_cast<int>((begin + j) / KS));
        ks = 0;
      }
    }
    // a row block whose last stage lies beyond this CTA's range
    if (ok && ks != 0) ok = flush(rb_last);
    if (ok && fh == 0 && first_parked) {
      // the last row block was whole: add the parked first one now
      bool fine = true;
      if (lane == 0) fine = wait_counter_at_least(arrivals, arrival_target, err);
      fine = __shfl_sync(0xffffffffu, fine ? 1 : 0, 0) != 0;
      const int n0 = rb0 * kRows + r;
      if (fine)
#pragma unroll
        for (int t = 0; t < TT; ++t)
          if (n0 < N && t < Tt)
            atomicAdd(&y[static_cast<size_t>(tok0 + t) * N + n0], first_part[t * kRows + r]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tbase, C::kTmemCols);
}

template <int TT>
cudaError_t set_attr_one() {
  return cudaFuncSetAttribute(smallt_kernel<TT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TC<TT>::kAllocMax);
}

cudaLaunchConfig_t pdl_config(cudaLaunchAttribute* attr, dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <int TT>
cudaError_t launch_tt(const CUtensorMap* tmW, const uint16_t* scales, const uint16_t* x,
                      int* sync, uint8_t* work, float* y, int K, int N, int tok0, int Tt,
                      int num_sms, int* err, cudaStream_t stream) {
  using C = TC<TT>;
  const int KS = (K + kSTStageK - 1) / kSTStageK;
  const long long NB = (N + kRows - 1) / kRows;
  const long long U = NB * KS;
  long long P = num_sms;  // one CTA per SM: each holds all 512 TMEM columns
  if (P > kSmallTMaxCtas) P = kSmallTMaxCtas;
  if (P > U) P = U;
  uint8_t* xprep = work;

  cudaLaunchAttribute attr[1];
  if constexpr (!C::kInKernelX) {
    const int tasks = C::kH * kGS * KS;
    cudaLaunchConfig_t pc = pdl_config(attr, dim3((tasks + 7) / 8), dim3(256), 0, stream);
    cudaError_t e = cudaLaunchKernelEx(&pc, xprep_kernel<TT>, x, xprep, K, tok0, Tt, KS);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = pdl_config(attr, dim3(static_cast<unsigned>(P)), dim3(C::kThreads),
                                      C::smem_bytes(KS), stream);
  return cudaLaunchKernelEx(&cfg, smallt_kernel<TT>, *tmW, scales, x,
                            static_cast<const uint8_t*>(xprep), y,
                            reinterpret_cast<unsigned long long*>(sync), K, N, tok0, Tt, KS, U,
                            err);
}

}  // namespace

size_t smallt_work_bytes(int tt, int K) {
  const int KS = (K + kSTStageK - 1) / kSTStageK;
  size_t prep = 0;
  switch (tt) {
    case 1: prep = 0; break;  // built inside the main kernel
    case 4: prep = static_cast<size_t>(TC<4>::kXBytes) * KS; break;
    case 8: prep = static_cast<size_t>(TC<8>::kXBytes) * KS; break;
    default: prep = static_cast<size_t>(TC<16>::kXBytes) * KS; break;
  }
  return prep;
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

cudaError_t launch_smallt(int tt, const CUtensorMap* tmW, const uint16_t* scales,
                          const uint16_t* x, int* sync, uint8_t* work, float* y, int K, int N,
                          int tok0, int Tt, int num_sms, int* err, cudaStream_t stream) {
  switch (tt) {
    case 1:
      return launch_tt<1>(tmW, scales, x, sync, work, y, K, N, tok0, Tt, num_sms, err, stream);
    case 4:
      return launch_tt<4>(tmW, scales, x, sync, work, y, K, N, tok0, Tt, num_sms, err, stream);
    case 8:
      return launch_tt<8>(tmW, scales, x, sync, work, y, K, N, tok0, Tt, num_sms, err, stream);
    default:
      return launch_tt<16>(tmW, scales, x, sync, work, y, K, N, tok0, Tt, num_sms, err, stream);
  }
}

}  // namespace tern
