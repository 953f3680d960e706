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
// 1. Activation pieces.  Per token and per 128-wide group, x is scaled by a
//    power of two 2^p so that the group's absmax m lies in [2^14, 2^15), and
//    split into three fp8 e5m2 pieces
//        v = x 2^p,  h1 = RN(v),  h2 = RN(v - h1),  h3 = RN(v - h1 - h2)
//    (RN: nearest e5m2 value, ties to even, computed as round3).
//    A bf16 value has 8 significant bits and an e5m2 value 3, and each
//    rounding leaves a remainder at most half a step of the piece it rounds
//    to; so for every element whose exponent is at least that of m minus 21
//    (its scaled value at least 2^-7, its last bit at least 2^-14)
//    h1 + h2 + h3 == v exactly, and every nonzero piece is a normal e5m2.
//    Smaller nonzero elements ("leftovers", |x| < 2^-21 of m's binade) get no
//    pieces; the group's factor is stored negated with their sum of |x|.  The
//    fold notes such groups and, at the end of the row block, either leaves
//    them out (their bound within 2^-11 of the row block's partial sum) or
//    adds their products exactly on the CUDA cores (leftover_dot), reading
//    the group's packed weights and x again.  With bf16 activations
//    leftovers occur only in groups whose values span more than 21 binades.
//    The pieces are the columns of the MMA's B operand in the tcgen05
//    K-major shared-memory layout, one block per 1024-wide k stage, with the
//    per-(group, token) factors f = 2^(3-p).  A prep kernel builds all
//    blocks once per call; at T = 1 the main kernel copies the blocks of
//    every stage it visits once into shared memory, where they stay (a
//    compact layout: see kX1Lbo), and for wider token tiles it copies each
//    stage's block in with its weights.  At T = 1 with at most two units per
//    CTA the fold warps build the resident blocks from x instead, and the
//    prep kernel is not launched.
// 2. Weights as fp8, decoded into tensor memory.  The packed code puts each
//    weight's nonzero bit and sign bit at the 2^-3 exponent bit and the sign
//    bit of an e4m3 byte once shifted, so one shift and one AND turn a packed
//    word into four exact e4m3 values w/8.  Decode threads own rows of the
//    CTA's 128-row block (one TMEM lane each) and store decoded row chunks
//    with tcgen05.st into the A operand in TMEM.
// 3. tcgen05.mma kind::f8f6f4 (A e4m3 in TMEM, B e5m2 in shared memory, fp32
//    accumulator in TMEM): every product w/8 * piece is exact.  Fold threads
//    read the accumulators back with tcgen05.ld and fold the pieces' sums
//    into their row's running sums with s[n][g] * f[g][token].  Beside the
//    leftovers left out within their budget, the only roundings are the
//    fp32 sums.
//
// Pipeline (one CTA per SM, persistent; TMEM 512 columns):
//   warp 16    producer: two 2D TMA boxes of packed weights (128 rows x 128 B
//              each, 128-byte swizzle) per stage into the weight ring (plus,
//              for T > 1, a bulk copy of the stage's activation block); the
//              stage's fp16 scales (cp.async) into a longer scale ring.  The
//              weights and scales of the first stages are requested before
//              the previous kernel on the stream has finished (they are not
//              written by it); activations only after.
//   warps 0-7  decode (four groups of 32 rows per warp) into A sub-slots;
//              they start on the early stages before the previous grid ends;
//   warps 17-18 issue the MMAs of half-stage 0 / 1 of every stage once its
//              A sub-slot is full and its D slot has been drained (warp 17
//              also allocates TMEM);
//   warps 8-15 fold D slots into per-row running sums (two threads per row,
//              one per half-stage) and write y at the end of each row block
//              (or hand split row blocks' sums to warp 19);
//   warp 19    adds up the row blocks this CTA shares with others.
//
// Work split: the (row block, 1024-wide k stage) units are cut into equal
// contiguous ranges, one per CTA, so every SM streams the same bytes.  A row
// block whole inside one CTA is written to y directly.  A row block split
// between CTAs is reduced without waiting on other CTAs: each CTA writes its
// partial row sums to the workspace and takes a ticket; the CTA that arrives
// last adds every partial in CTA order and writes y.  (A CTA that finishes a
// row block shared with one other CTA, which started it earlier, polls the
// ticket and copies the other partial in before its own sums are ready.)
// The result does not depend on which CTA finishes last, so every output is
// reproducible bit for bit, and no CTA ever waits for another to be
// scheduled.
//
// A stage is 1024 k: two 128-byte weight boxes per row, eight groups; a
// half-stage is one box, four groups.  TMEM is used per half-stage: the
// decode warps of groups 0-3 and of groups 4-7 each fill their own ring of A
// sub-slots (two groups each), the MMAs of a half-stage write their own D
// slot, so decode, MMA and fold can run sub-slots apart.
//
// Calls chain by programmatic dependent launch: every kernel lets the next one
// launch as soon as all of its CTAs run; the next kernel's CTAs set up, load
// their first weight stages and wait for the previous grid before they read
// anything it may have written (x) or write y / the workspace.  The prep
// kernel's CTAs are small enough (4 warps, 32 registers, no shared memory)
// to sit beside a main-kernel CTA, so a prep launch never holds an SM the
// next main kernel needs.  Each A sub-slot ring and D ring belongs to one
// decode half, one MMA issuer and one fold half, so a waiter's barrier is
// never two phases behind it.
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
// half-stage f / 4 (groups 4 (f / 4) .. 4 (f / 4) + 3) of every stage.
constexpr int kFoldWarps = 8;
constexpr int kProducerWarp = kDecWarps + kFoldWarps;
// Two MMA-issuing warps: the first issues half-stage 0 of every stage, the
// second half-stage 1, so a single issuing thread never paces the tensor pipe.
constexpr int kMmaWarp = kProducerWarp + 1;
constexpr int kMmaWarps = 2;
constexpr int kXWarp0 = kMmaWarp + kMmaWarps;  // activation warps (T = 1) / split-row warp
constexpr int kGS = kSTStageK / 128;       // 128-wide groups per stage
constexpr int kGH = kGS / 2;               // groups per half-stage
constexpr int kWBoxes = kSTStageK / 512;   // 128-byte TMA boxes per stage row
static_assert(kGH == 4 && kWBoxes * 4 == kGS, "a half-stage is one weight box");
constexpr uint32_t kXLbo = 128;            // K-direction core-matrix stride in the B block
constexpr uint32_t kXSbo = kSTStageK / 16 * 128;  // N-direction stride (8 columns of one stage)
// T = 1 activation block of one stage, for an N = 16 MMA.  With a 32-byte
// K-direction core-matrix stride, columns 0 and 1 of each 8-column group are
// two interleaved byte rows and column c + 2 aliases column c one core
// matrix further along K; so three pieces need only the clean columns 0, 1
// (first group: h1, h2) and 8 (second group: h3), one byte per k each (plus
// an overrun that the never-read columns 2-7 / 9-15 reach).
constexpr uint32_t kX1Lbo = 32;
constexpr uint32_t kX1Sbo = kSTStageK / 16 * 32 + 128;  // second 8-column group
constexpr int kX1Stage = 2 * kX1Sbo;                    // bytes per stage block
// A stage's block and its groups' (f, L) pairs, as the prep kernel writes it
// and the one-token kernel keeps it resident.
constexpr int kX1Slot = kX1Stage + (kSTStageK / 128) * 8;
static_assert(kX1Sbo >= kSTStageK / 16 * 32 + 7 * 16, "the junk columns' overrun stays inside");

// Tiles that run in cluster mode (the one-token tile: at T = 4 and 16 the
// smaller, cluster-scheduled grid cost the down projection more than the
// on-chip sums saved).
constexpr bool cluster_tile(int tt) { return tt == 1; }

// Largest cluster of CTAs sharing one row block (cluster mode, T = 1).
constexpr int kMaxCl = 4;

template <int TT>
struct TC {
  // Token slots of the B operand and MMA N (= accumulator columns per group).
  //   TT = 1:  compact block, pieces in columns 0, 1, 8; N = 16.
  //   TT = 4:  piece j of token t in column 4 j + t (12 of 16); N = 16.
  //   TT = 8:  pieces 0, 1 in columns 8 j + t (N = 16); piece 2 in a block of
  //            its own (columns 0-7, 8-15 zero) whose N = 16 MMA accumulates
  //            onto the same accumulator columns as piece 0.
  //   TT = 16: pieces 0, 1 in columns 16 j + t (N = 32); piece 2 as for 8.
  static constexpr int kH = TT;
  static constexpr int kNC = TT <= 8 ? 16 : 32;
  static constexpr bool kH3 = TT >= 8;
  static constexpr int kP1 = TT == 1 ? 1 : (TT == 4 ? 4 : TT);  // piece 1's column offset
  static constexpr int kP2 = TT == 1 ? 8 : 8;                    // piece 2's (TT <= 4)
  static constexpr int kXMain = kNC * kSTStageK;                 // main B block of a stage
  static constexpr int kXFrag = kXMain + (kH3 ? 16 * kSTStageK : 0);  // + piece-2 block
  // per (group, token): the factor f, then the leftovers' sum of |x| L
  static constexpr int kXF = 2 * kGS * kH * 4;                   // f[group][kH], L[group][kH]
  // one stage of the prep buffer (T = 1: compact block + (f, L)[group])
  static constexpr int kXBytes = TT == 1 ? kX1Slot : kXFrag + kXF;
  // T = 1: the stages' blocks stay resident, copied once per call
  static constexpr bool kInKernelX = TT == 1;
  static constexpr int kXWarps = 1;  // the split-row warp
  static constexpr int kThreads = (kXWarp0 + kXWarps) * 32;
  // TMEM.  A (e4m3 weights): each half-stage (one decode half, one MMA
  // issuer) has its own ring of kNSub sub-slots of kGH / 2 groups (64
  // columns), used in order by that half alone; its decoders can run
  // kNSub / 2 units ahead of the MMAs that free the sub-slots.  A sub-slot
  // needs one A-operand load of the tensor pipe per use, and only its own
  // half ever waits on its barriers.  D (fp32 accumulators): one slot of
  // kGH x kNC columns per half-stage; the fold drains it before the next
  // unit's MMAs of that half.
  static constexpr int kNSub = TT == 16 ? 2 : 3;
  static constexpr int kNDH = 2;
  static constexpr int kStages = TT == 1 ? 5 : (TT == 16 ? 2 : 3);  // weight (+ activation) ring
  // Scale loads run kLead units ahead of the weight loads (T = 1: the weight
  // ring does not wait for the MMAs, so the fold must never wait for scales).
  static constexpr int kLead = kInKernelX ? 2 : 0;
  // Weight stages requested before the previous grid ends.  (T = 1) Only two:
  // the activation copies, issued after it, queue behind whatever is in
  // flight, and the first MMAs wait for them.
  static constexpr int kEarly = kInKernelX ? 2 : kStages;
  static_assert(2 * kEarly >= kNSub, "decoders fill the free A sub-slots from early stages only");
  // scale (+ factor) ring: held until folded, which trails the weight ring
  // by up to the A lookahead and the D slot
  static constexpr int kSStages = kStages + kLead + (kNSub + 1) / 2 + 1;
  static constexpr int kWBytes = kRows * kSTStageK / 4;  // kWBoxes boxes of 128 rows x 128 B
  static constexpr int kSBytes = kRows * 2 * kGS + (kInKernelX ? 0 : kXF);  // scales [128][kGS], f, L
  static constexpr int kWOff = 0;  // 1024-aligned for the 128-byte swizzle
  static constexpr int kXOff = kWOff + kStages * kWBytes;  // activation ring (T > 1)
  static constexpr int kSOff = kXOff + (kInKernelX ? 0 : kStages * kXFrag);
  static constexpr int kBarOff = kSOff + kSStages * kSBytes;
  static constexpr int kNumBars = 2 * kStages + 2 * kSStages + 4 * kNSub + 2 * kNDH + 8 + 2 +
                                  (kInKernelX ? kSmallTX1MaxSlots : 0) + 1;
  static constexpr int kTmemSlot = kBarOff + kNumBars * 8;
  // 16-byte aligned from here on: the regions below are read as float4 / uint2
  static constexpr int kPartOff = (kTmemSlot + 16 + 15) / 16 * 16;  // fold: half-stage 1 sums [TT][128]
  // fold: the CTA's split row blocks' sums [2][TT][128], for the split-row warp
  static constexpr int kSplitOff = kPartOff + TT * kRows * 4;
  // fold: one group of x per fold warp for exact leftovers [kFoldWarps][128] bf16
  static constexpr int kLxOff = kSplitOff + 2 * TT * kRows * 4;
  // fold: the leftover groups each fold warp has left out of its current row
  // block, decided when the row block ends [kFoldWarps][kDefer] (code, |f|)
  static constexpr int kDefer = 8;
  static constexpr int kDefOff = kLxOff + kFoldWarps * 256;
  // cluster mode (TT = 1): the other ranks' partial sums of the row block,
  // written into rank 0's shared memory [kMaxCl - 1][TT][128]
  static constexpr bool kCluster = cluster_tile(TT);
  static constexpr int kClOff = kDefOff + kFoldWarps * kDefer * 8;
  static constexpr int kX1Off =
      (kClOff + (kCluster ? (kMaxCl - 1) * TT * kRows * 4 : 0) + 127) / 128 * 128;  // (T = 1)
  // shared memory for nslots resident T = 1 blocks: fixed part, blocks, alignment slack
  static constexpr int smem_bytes(int nslots) {
    return kX1Off + (kInKernelX ? nslots * kX1Slot : 0) + 1024;
  }
  static constexpr int kAllocMax = smem_bytes(kInKernelX ? kSmallTX1MaxSlots : 0);
  static constexpr uint32_t kSubCols = (kGH / 2) * 32;  // A sub-slot
  static constexpr uint32_t kAHalf = kNSub * kSubCols;  // a half-stage's A ring
  static constexpr uint32_t kDSlot = kGH * kNC;         // D[kNDH] slots
  static constexpr uint32_t kACol = 0;
  static constexpr uint32_t kDCol = 2 * kAHalf;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kDCol + kNDH * kDSlot <= kTmemCols, "TMEM budget");
  static_assert(kXFrag % 16 == 0 && kXF % 16 == 0 && kXBytes % 16 == 0, "bulk copy sizes");
  static_assert(kSBytes % 16 == 0 && kBarOff % 8 == 0, "alignment");
  static_assert(kPartOff % 16 == 0 && kSplitOff % 16 == 0 && kLxOff % 16 == 0 &&
                    kDefOff % 16 == 0 && kClOff % 16 == 0 && kX1Off % 128 == 0,
                "vector-accessed regions must be 16-byte aligned");
  static_assert(kAllocMax <= 227 * 1024, "shared memory");
};

// Instruction descriptor for kind::f8f6f4 with A e4m3 and B e5m2, fp32
// accumulator, both operands K-major.
constexpr uint32_t idesc_e4m3_e5m2_f32(int M, int N) {
  return idesc_e4m3_f32(M, N) | (1u << 10);  // B type field (bits 10-12): e5m2
}

// Scales of a group with absmax m > 0 (finite): el = floor(log2 m); the
// pieces are cut from v = x 2^p with p = 14 - el, applied as two normal
// powers of two sc1 * sc2 (p may exceed the fp32 exponent range of one
// factor); the fold factor is f = 2^(3 - p) = 2^(el - 11) (w enters the MMA
// as w/8).
__device__ __forceinline__ void piece_band(float m, float& sc1, float& sc2, float& f) {
  const uint32_t mb = __float_as_uint(m);
  const int el = (mb >> 23) ? static_cast<int>(mb >> 23) - 127 : (31 - __clz(mb)) - 149;
  const int p = 14 - el;               // in [-113, 147]
  const int p1 = p >> 1, p2 = p - p1;  // each in [-57, 74]
  sc1 = __uint_as_float(static_cast<uint32_t>(p1 + 127) << 23);
  sc2 = __uint_as_float(static_cast<uint32_t>(p2 + 127) << 23);
  f = el - 11 >= -126 ? __uint_as_float(static_cast<uint32_t>(el - 11 + 127) << 23)
                      : ldexpf(1.0f, el - 11);  // a subnormal power of two, still exact
}

// Below this magnitude an element of the group is a leftover (2^(el - 21));
// computed the same way from |f| by the prep and by the fold.
__device__ __forceinline__ float leftover_limit(float f_abs) { return f_abs * 0x1p-10f; }

// x rounded to 3 significant bits (the e5m2 grid for |x| >= 2^-14), nearest
// with ties to even: (x + c) - c with c = 1.5 * 2^(exp(x) + 21) puts the last
// bit of the sum at 2^(exp(x) - 2).  Two fp32 adds, no conversion latency.
__device__ __forceinline__ float round3(float x) {
  const uint32_t e = __float_as_uint(x) & 0x7F800000u;
  const float c = __uint_as_float((e + (21u << 23)) | 0x00400000u);
  return __fsub_rn(__fadd_rn(x, c), c);
}

// Three e5m2 pieces of two scaled values (low byte: v.x, high byte: v.y):
// h1 = RN(v), h2 = RN(v - h1), h3 = RN(v - h1 - h2), computed in fp32 (every
// difference is exact), then packed; each piece is an exact e5m2 value.
__device__ __forceinline__ void split3_e5m2(float2 v, uint32_t& h1, uint32_t& h2, uint32_t& h3) {
  const float2 a = make_float2(round3(v.x), round3(v.y));
  const float2 r1 = make_float2(v.x - a.x, v.y - a.y);
  const float2 b = make_float2(round3(r1.x), round3(r1.y));
  const float2 r2 = make_float2(r1.x - b.x, r1.y - b.y);
  h1 = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E5M2);
  h2 = __nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E5M2);
  h3 = __nv_cvt_float2_to_fp8x2(r2, __NV_SATFINITE, __NV_E5M2);
}

// Pieces of one lane's four consecutive elements of a group (bf16 bits in
// raw), given the group's absmax m (already reduced over the warp).  Byte i of
// h1/h2/h3 is element i's piece; returns f, negated when some element of the
// group (any lane) is a leftover, and in lsum the sum of the leftovers' |x|
// over the group (0 without leftovers).  Must be called by the whole warp.
__device__ __forceinline__ float group_pieces(uint2 raw, float m, uint32_t& h1, uint32_t& h2,
                                              uint32_t& h3, float& lsum) {
  const float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                      __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
  h1 = h2 = h3 = 0u;
  lsum = 0.f;
  if (m == 0.f) return 0.f;  // warp-uniform
  float sc1, sc2, f;
  piece_band(m, sc1, sc2, f);
  const float tau = leftover_limit(f);
  bool left = false;
  float s[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool lo = v[i] != 0.f && fabsf(v[i]) < tau;
    left |= lo;
    lsum += lo ? fabsf(v[i]) : 0.f;
    s[i] = lo ? 0.f : (v[i] * sc1) * sc2;
  }
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    uint32_t a, b, c;
    split3_e5m2(make_float2(s[2 * hf], s[2 * hf + 1]), a, b, c);
    h1 |= a << (16 * hf);
    h2 |= b << (16 * hf);
    h3 |= c << (16 * hf);
  }
  if (!__any_sync(0xffffffffu, left)) {
    lsum = 0.f;
    return f;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
  return -f;
}

// The exact part of one group's dot product that the pieces leave out: the sum
// of w[n][k] * x[k] over the group's elements with 0 < |x| < tau, in fp32
// (every product is exact).  wrow: row n's 8 packed words of the group; xs:
// the group's 128 bf16 values (shared memory, two per 32-bit word).
__device__ __forceinline__ float leftover_dot(uint4 wa, uint4 wb, const uint32_t* xs, float tau) {
  const uint32_t w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
  float acc = 0.f;
#pragma unroll 1
  for (int j = 0; j < 8; ++j) {  // word j: k = 16 j .. 16 j + 15 of the group
    uint32_t wj = w[0];
#pragma unroll
    for (int u = 1; u < 8; ++u)
      if (u == j) wj = w[u];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int bit = 8 * (e >> 2) + ((e & 3) < 2 ? (e & 3) : (e & 3) + 2);
      const uint32_t xw = xs[8 * j + (e >> 1)];
      const float xf = __uint_as_float((e & 1) ? (xw & 0xFFFF0000u) : (xw << 16));
      const bool nz = (wj >> bit) & 1u;
      const bool neg = (wj >> (bit + 2)) & 1u;
      if (nz && xf != 0.f && fabsf(xf) < tau) acc += neg ? -xf : xf;
    }
  }
  return acc;
}

// CTA owning unit u when U units are cut into P equal contiguous ranges
// (CTA c holds units [U c / P, U (c + 1) / P)).
__device__ __forceinline__ int owner_of(long long u, long long U, long long P) {
  return static_cast<int>(((u + 1) * P - 1) / U);
}

// ------------------------------------------------------------------ prep
// Activation blocks of one token tile for all stages.  One warp per (token
// slot t < H, 128-wide group), kPrepWarps warps per CTA looping over the
// tasks, at most one CTA per SM: 4 warps of 32 registers and no shared memory
// fit beside a resident main-kernel CTA (640 threads of at most 96
// registers, at most 226 KB of shared memory), so a launch queued behind the
// main kernel of the previous call takes no SM from the next one.  Lane l
// holds k = 4l .. 4l+3 of the group.  Slot order inside each 16-wide block of
// k is the transpose the decoder produces: slot 4i + b holds k = 4b + i.
constexpr int kPrepWarps = 4;

// Group jg of a stage's block (at st) for token slot t, from the lane's four
// bf16 values raw.  The whole warp calls it.
__device__ __forceinline__ float lane_absmax4(uint2 raw) {
  const float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                      __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
  return fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
}

// Write group jg of a stage's block (at st) for token slot t: the lane's
// three piece bytes for its four elements (hp[j], element i in byte i), and
// (lane 0) the group's factor f and leftover sum lsum.
template <int TT>
__device__ __forceinline__ void prep_write(const uint32_t (&hp)[3], float f, float lsum,
                                           uint8_t* st, int t, int jg, int lane) {
  using C = TC<TT>;
  if constexpr (TT == 1) {
    // compact block: 16-block j = 8 jg + l/4 at bytes 32 j (piece 0), 32 j + 16
    // (piece 1) and kX1Sbo + 32 j (piece 2); position b = l%4: value i at 4i + b
    uint8_t* blk = st + 32 * (8 * jg + (lane >> 2)) + (lane & 3);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      blk[4 * e] = static_cast<uint8_t>(hp[0] >> (8 * e));
      blk[16 + 4 * e] = static_cast<uint8_t>(hp[1] >> (8 * e));
      blk[kX1Sbo + 4 * e] = static_cast<uint8_t>(hp[2] >> (8 * e));
    }
    if (lane == 0) reinterpret_cast<float2*>(st + kX1Stage)[jg] = make_float2(f, lsum);
  } else {
    auto put = [&](uint8_t* blk, int n, int slot, uint8_t b) {
      blk[(n >> 3) * kXSbo + (slot >> 4) * kXLbo + (n & 7) * 16 + (slot & 15)] = b;
    };
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // k = 4 lane + i: 16-block lane/4, position b = lane%4, i -> slot 4i + b
      const int slot = 128 * jg + 16 * (lane >> 2) + 4 * i + (lane & 3);
      const uint8_t b0 = static_cast<uint8_t>(hp[0] >> (8 * i));
      const uint8_t b1 = static_cast<uint8_t>(hp[1] >> (8 * i));
      const uint8_t b2 = static_cast<uint8_t>(hp[2] >> (8 * i));
      put(st, t, slot, b0);
      put(st, C::kP1 + t, slot, b1);
      if constexpr (C::kH3) {
        put(st + C::kXMain, t, slot, b2);
        if constexpr (TT == 8) put(st + C::kXMain, 8 + t, slot, 0);  // the block's idle columns
      } else {
        put(st, C::kP2 + t, slot, b2);
      }
    }
    if (lane == 0) {
      float* fl = reinterpret_cast<float*>(st + C::kXFrag);
      fl[jg * C::kH + t] = f;
      fl[(kGS + jg) * C::kH + t] = lsum;
    }
  }
}

// As prep_task, with the group's absmax m already reduced over the warp.
template <int TT>
__device__ __forceinline__ void prep_task_m(uint2 raw, float m, uint8_t* st, int t, int jg,
                                            int lane) {
  uint32_t hp[3];
  float lsum;
  const float f = group_pieces(raw, m, hp[0], hp[1], hp[2], lsum);
  prep_write<TT>(hp, f, lsum, st, t, jg, lane);
}

template <int TT>
__device__ __forceinline__ void prep_task(uint2 raw, uint8_t* st, int t, int jg, int lane) {
  float m = lane_absmax4(raw);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  prep_task_m<TT>(raw, m, st, t, jg, lane);
}

template <int TT>
__global__ void __launch_bounds__(kPrepWarps * 32, 16) xprep_kernel(const uint16_t* __restrict__ x,
                                                               uint8_t* __restrict__ out, int K,
                                                               int tok0, int Tt, int KS) {
  grid_dependents_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int groups = kGS * KS;
  const int tasks = TC<TT>::kH * groups;
  const int stride = gridDim.x * kPrepWarps;
  // Warm L2 with the groups of x this warp reads first (lane i: its i-th
  // task) while the previous grid finishes; a prefetch only moves lines into
  // L2, so it is harmless while x may still be being written.
  {
    const int task = blockIdx.x * kPrepWarps + warp + lane * stride;
    const int t = task / groups, kbase = (task % groups) * 128;
    if (task < tasks && t < Tt && kbase < K)
      bulk_prefetch_l2(x + static_cast<size_t>(tok0 + t) * K + kbase, 256u);
  }
  grid_dependency_wait();  // x (and this buffer's last reader) come from earlier work
  // two tasks' loads in flight before their arithmetic
  for (int t0 = blockIdx.x * kPrepWarps + warp; t0 < tasks; t0 += 2 * stride) {
    uint2 raw[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int task = t0 + u * stride;
      const int t = task / groups, kbase = (task % groups) * 128 + 4 * lane;
      raw[u] = make_uint2(0u, 0u);
      if (task < tasks && t < Tt && kbase < K)
        raw[u] = *reinterpret_cast<const uint2*>(x + static_cast<size_t>(tok0 + t) * K + kbase);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int task = t0 + u * stride;
      if (task < tasks) {
        const int gi = task % groups;
        prep_task<TT>(raw[u], out + static_cast<size_t>(gi / kGS) * TC<TT>::kXBytes,
                      task / groups, gi % kGS, lane);
      }
    }
  }
}

// int8 activations (the decode variant of the pages' int8 path): per token,
// xs = absmax / 127 and q = clamp(rint(x / xs), -127, 127) with IEEE fp32
// division, the arithmetic of tern_quant_act_s8; q is split as on the s8
// rung into p1 = 16 floor((q + 8) / 16) and p2 = q - p1, both exact in e5m2
// (multiples of 16 up to 128, integers in [-8, 7]), the third piece is zero
// and the factor is 8 xs, so the fold adds s * 8 xs * (acc / 8): the s8
// rung's value with exact integer group sums.  One CTA per (token slot,
// stage): its four warps first find the token's absmax (the whole row), then
// build the stage's eight groups, two per warp.  4 warps of 32 registers and
// 16 bytes of shared memory: it fits beside a main-kernel CTA.
template <int TT>
__global__ void __launch_bounds__(kPrepWarps * 32, 16) xprep_i8_kernel(
    const uint16_t* __restrict__ x, uint8_t* __restrict__ out, int K, int tok0, int Tt, int KS) {
  grid_dependents_launch();
  grid_dependency_wait();  // x (and this buffer's last reader) come from earlier work
  __shared__ float red[kPrepWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = K >> 7;
  const int tasks = TC<TT>::kH * KS;
  for (int task = blockIdx.x; task < tasks; task += gridDim.x) {
    const int t = task / KS, ks = task % KS;
    const uint16_t* row = x + static_cast<size_t>(tok0 + (t < Tt ? t : 0)) * K;
    float a = 0.f;
    if (t < Tt)
      for (int c = threadIdx.x; c < (K >> 3); c += kPrepWarps * 32) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + 8 * c);
        a = fmaxf(a, fmaxf(lane_absmax4(make_uint2(v.x, v.y)), lane_absmax4(make_uint2(v.z, v.w))));
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) red[warp] = a;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kPrepWarps; ++w) a = fmaxf(a, red[w]);
    __syncthreads();  // red is rewritten by the next task
    const float xs = a / 127.0f;  // IEEE single-precision division
    uint8_t* st = out + static_cast<size_t>(ks) * TC<TT>::kXBytes;
    for (int jg = warp; jg < kGS; jg += kPrepWarps) {
      const int g = ks * kGS + jg;
      uint2 raw = make_uint2(0u, 0u);
      if (t < Tt && g < G) raw = *reinterpret_cast<const uint2*>(row + g * 128 + 4 * lane);
      const float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                          __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
      uint32_t hp[3] = {0u, 0u, 0u};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        int q = 0;
        if (a > 0.f) q = static_cast<int>(fminf(fmaxf(rintf(v[i] / xs), -127.f), 127.f));
        const int h = (q + 8) >> 4;  // floor((q + 8) / 16), in [-8, 8]
        hp[0] |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(static_cast<float>(16 * h),
                                                             __NV_SATFINITE, __NV_E5M2))
                 << (8 * i);
        hp[1] |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(static_cast<float>(q - 16 * h),
                                                             __NV_SATFINITE, __NV_E5M2))
                 << (8 * i);
      }
      prep_write<TT>(hp, 8.0f * xs, 0.f, st, t, jg, lane);
    }
  }
}

// Rotated activations (the Hadamard rotation of every 1024-wide block, fused
// into the staging): one warp per (token slot, stage), the stage being one
// rotation block.  The warp loads the block with lane l holding elements
// 128 g + 4 l + i, rotates it in registers (hadamard_block_1024), scales by
// 1/32 and rounds each value once to bf16, nearest-even; lane l then holds
// exactly its four values of each of the stage's eight groups and builds
// their pieces as the unrotated kernel does.  One-warp CTAs of at most 64
// registers (at most one per SM), so they too fit beside a main-kernel CTA.
template <int TT>
__global__ void __launch_bounds__(32, 32) xprep_rot_kernel(const uint16_t* __restrict__ x,
                                                           uint8_t* __restrict__ out, int K,
                                                           int tok0, int Tt, int KS) {
  grid_dependents_launch();
  grid_dependency_wait();  // x (and this buffer's last reader) come from earlier work
  const int lane = threadIdx.x;
  const int tasks = TC<TT>::kH * KS;
  for (int task = blockIdx.x; task < tasks; task += gridDim.x) {
    const int t = task / KS, ks = task % KS;
    float v[32];
#pragma unroll
    for (int g = 0; g < kGS; ++g) {
      uint2 raw = make_uint2(0u, 0u);
      if (t < Tt)  // K is a multiple of 1024: every group of the stage exists
        raw = *reinterpret_cast<const uint2*>(x + static_cast<size_t>(tok0 + t) * K +
                                              ks * kSTStageK + 128 * g + 4 * lane);
      v[4 * g + 0] = __uint_as_float(raw.x << 16);
      v[4 * g + 1] = __uint_as_float(raw.x & 0xFFFF0000u);
      v[4 * g + 2] = __uint_as_float(raw.y << 16);
      v[4 * g + 3] = __uint_as_float(raw.y & 0xFFFF0000u);
    }
    hadamard_block_1024(v, lane);
    uint8_t* st = out + static_cast<size_t>(ks) * TC<TT>::kXBytes;
    // the eight groups' bf16 values and absmax reductions side by side (eight
    // independent shuffle chains), then their pieces
    uint2 raw[kGS];
    float m[kGS];
#pragma unroll
    for (int g = 0; g < kGS; ++g) {
      uint32_t b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        b[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v[4 * g + i] * 0.03125f));
      raw[g] = make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
      m[g] = lane_absmax4(raw[g]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int g = 0; g < kGS; ++g) m[g] = fmaxf(m[g], __shfl_xor_sync(0xffffffffu, m[g], o));
#pragma unroll
    for (int g = 0; g < kGS; ++g) prep_task_m<TT>(raw[g], m[g], st, t, g, lane);
  }
}

// ------------------------------------------------------------------ main
// The units of one CTA: a contiguous range, from stage ks0 of row block rb0.
struct Visit {
  int KS;      // k stages per row block
  int rb0;     // row block of the range's first unit, and its stage
  int ks0;
  int nunits;  // units in the range
};

// (row block, stage) of the unit at position v of the range, stepped
// incrementally.
struct Cursor {
  int rb, ks, v;
  __device__ __forceinline__ void start(const Visit& s) {
    v = 0;
    rb = s.rb0;
    ks = s.ks0;
  }
  __device__ __forceinline__ void next(const Visit& s) {
    ++v;
    if (++ks == s.KS) {
      ks = 0;
      ++rb;
    }
  }
  // this CTA's last unit of row block rb
  __device__ __forceinline__ bool ends_row_block(const Visit& s) const {
    return v == s.nunits - 1 || ks == s.KS - 1;
  }
};

// (T = 1) The CTA visits min(nunits, KS) distinct stages, a cyclic run from
// ks0; stage ks keeps its activation block in slot (ks - ks0) mod KS, and
// the i-th stage of the run is new_stage(i).
__device__ __forceinline__ int stage_slot(const Visit& s, int ks) {
  return ks >= s.ks0 ? ks - s.ks0 : ks + s.KS - s.ks0;
}
__device__ __forceinline__ int new_stage(const Visit& s, int i) {
  return i < s.KS - s.ks0 ? s.ks0 + i : i - (s.KS - s.ks0);
}

// wp: the packed weights (read again only for leftovers); x: bf16 activations
// (read at T = 1, and for leftovers); xprep: prep blocks (T > 1).
// tickets / partials: the workspace's ticket counters (one per CTA) and
// partial row sums of split row blocks.  nslots: T = 1 resident blocks;
// build_x: (T = 1) the fold warps build them from x instead of copying the
// prep kernel's.
template <int TT>
__global__ void __launch_bounds__(TC<TT>::kThreads, 1)
    smallt_kernel(const __grid_constant__ CUtensorMap tmW, const uint32_t* __restrict__ wp,
                  const uint16_t* __restrict__ scales, const uint16_t* __restrict__ x,
                  const uint8_t* __restrict__ xprep, float* __restrict__ y,
                  int* __restrict__ tickets, float* __restrict__ partials, int K, int N, int tok0,
                  int Tt, int KS, int nslots, long long U, int build_x, int cl, int* err) {
  using C = TC<TT>;
  constexpr int S = C::kStages;
  constexpr int SS = C::kSStages;
  constexpr int NSUB = C::kNSub;
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
  // [half][sub-slot]: A sub-slot written by its half's four decoders / the
  // MMAs reading it completed
  uint64_t* afull = sempty + SS;
  uint64_t* afree = afull + 2 * NSUB;
  uint64_t* mdone = afree + 2 * NSUB;  // MMAs writing D slot d completed
  uint64_t* dfree = mdone + ND;   // D slot d read back by the fold warps
  // fold pairs: [quarter] the half-stage-1 warp's row block sums are in
  // shared memory / have been taken by the half-stage-0 warp
  uint64_t* pfull = dfree + ND;
  uint64_t* pfree = pfull + 4;
  // [i] the four writing fold warps have published their partial sums of the
  // CTA's i-th split row block
  uint64_t* pub = pfree + 4;
  uint64_t* xready = pub + 2;  // (T = 1) activation block of slot q built
  // (cluster mode, rank 0) the other ranks' partial sums have landed
  uint64_t* cfull = xready + (C::kInKernelX ? kSmallTX1MaxSlots : 0);
  uint8_t* xres = smem + C::kX1Off;  // (T = 1) resident slots: block + (f, L)[kGS]
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
    for (int a = 0; a < 2 * NSUB; ++a) {
      mbar_init(&afull[a], kDecWarps / 2);
      mbar_init(&afree[a], 1);
    }
    for (int d = 0; d < ND; ++d) {
      mbar_init(&mdone[d], 1);
      mbar_init(&dfree[d], kFoldWarps / 2);  // the four warps of its half-stage
    }
    for (int q = 0; q < 4; ++q) {
      mbar_init(&pfull[q], 1);
      mbar_init(&pfree[q], 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&pub[i], 4);  // the four half-stage-0 fold warps
    if constexpr (C::kInKernelX)
      for (int q = 0; q < nslots; ++q)  // the producer's copy, or one group per fold warp
        mbar_init(&xready[q], build_x ? kFoldWarps : 1);
    // every lane of every other rank's split-row warp arrives once
    mbar_init(cfull, cl > 1 ? (cl - 1) * 32 : 1);
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
  // Work: equal contiguous ranges of the (row block, stage) units; or, in
  // cluster mode (cl > 1), row block cta / cl cut into cl contiguous stage
  // ranges, one per rank of the cluster.
  long long begin, end;
  int crank = 0;
  if (cl > 1) {
    crank = static_cast<int>(cluster_ctarank());
    const long long crb = cta / cl;
    begin = crb * KS + static_cast<long long>(KS) * crank / cl;
    end = crb * KS + static_cast<long long>(KS) * (crank + 1) / cl;
    cluster_sync_all();  // every rank's barriers are initialised before any remote arrival
  } else {
    begin = U * cta / P;
    end = U * (cta + 1) / P;
  }
  Visit vs;
  vs.KS = KS;
  vs.nunits = static_cast<int>(end - begin);
  vs.rb0 = static_cast<int>(begin / KS);
  vs.ks0 = static_cast<int>(begin - static_cast<long long>(vs.rb0) * KS);
  const int rb_last = static_cast<int>((end - 1) / KS);
  const int nunits = vs.nunits;
  const int rb0 = vs.rb0, ks0 = vs.ks0;
  auto is_split = [&](int rb) {
    const long long u = static_cast<long long>(rb) * KS;
    return owner_of(u, U, P) != owner_of(u + KS - 1, U, P);
  };
  // The CTA's split row blocks in the order the fold finishes them: the
  // first row block, then the last (either when shared with another CTA).
  int sp[2];
  int nsp = 0;
  if (cl > 1) {
    sp[nsp++] = rb0;  // the cluster's one row block
  } else {
    if (is_split(rb0)) sp[nsp++] = rb0;
    if (rb_last != rb0 && is_split(rb_last)) sp[nsp++] = rb_last;
  }

  // The roles wait for the previous grid before any bounded wait whose end
  // depends on it, so that no clock starts while a slow predecessor is still
  // running: here, except for the producer (which first requests the weights
  // of its first stages) and the decoders (which decode those stages into
  // the free A sub-slots first, and wait before the first sub-slot reuse).
  if (warp >= kDecWarps && warp != kProducerWarp) grid_dependency_wait();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Scale stream: unit su's fp16 scales of groups kGS ks .. kGS ks + kGS - 1
    // for rows lane + 32 i, into scale ring slot su % SS; for T > 1 the
    // unit's factors f and leftover sums L come with them (expected here,
    // copied by issue_f once the previous grid, which may have written them,
    // has finished).
    int su = 0;
    Cursor cs;
    cs.start(vs);
    auto issue_scales = [&]() -> bool {
      const int ss = su % SS;
      if (su >= SS &&
          !__all_sync(0xffffffffu, mbar_wait(&sempty[ss], ((su / SS) & 1) ^ 1, err)))
        return false;
      uint8_t* sst = smem + C::kSOff + ss * C::kSBytes;
      if constexpr (!C::kInKernelX) {
        if (lane == 0) mbar_expect_tx(&sfull[ss], C::kXF);
        __syncwarp();
      }
      uint4* sb = reinterpret_cast<uint4*>(sst);
      const int g0 = cs.ks * kGS;
      if ((G % kGS) == 0) {
        // whole 16-byte rows of scales
#pragma unroll
        for (int i = 0; i < kRows / 32; ++i) {
          const int r = lane + 32 * i;
          const int n = cs.rb * kRows + r;
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
          const int n = cs.rb * kRows + r;
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
          const int n = cs.rb * kRows + r;
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
      cs.next(vs);
      return true;
    };
    // (T > 1) the factors of scale unit fu, whose stage is fks
    auto issue_f = [&](int fu, int fks) {
      if constexpr (!C::kInKernelX) {
        if (lane == 0)
          bulk_load(smem + C::kSOff + (fu % SS) * C::kSBytes + kRows * 2 * kGS,
                    xprep + static_cast<size_t>(fks) * C::kXBytes + C::kXFrag, C::kXF,
                    &sfull[fu % SS]);
      }
    };
    // weights of unit it (stage ks of row block rb) into ring slot it % S; the
    // barrier also expects the stage's activation block (T > 1)
    auto issue_weights = [&](int it, int rb, int ks) {
      const int s = it % S;
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[s], C::kWBytes + (C::kInKernelX ? 0 : C::kXFrag));
#pragma unroll
        for (int bx = 0; bx < kWBoxes; ++bx)
          tma_load_2d(smem + C::kWOff + s * C::kWBytes + bx * (kRows * 128), &tmW,
                      ks * (kSTStageK / 4) + 128 * bx, rb * kRows, &full[s]);
      }
    };
    auto issue_x = [&](int it, int ks) {
      if constexpr (!C::kInKernelX) {
        if (lane == 0)
          bulk_load(smem + C::kXOff + (it % S) * C::kXFrag,
                    xprep + static_cast<size_t>(ks) * C::kXBytes, C::kXFrag, &full[it % S]);
      }
    };
    // Weights and scales are not written by the previous kernels of the
    // stream's chain, so the first stages are requested before its end.
    bool ok = true;
    const int first = nunits < C::kEarly ? nunits : C::kEarly;
    while (ok && su < nunits && su < C::kLead) ok = issue_scales();
    int it = 0;
    Cursor cw;
    cw.start(vs);
    for (; it < first && ok; ++it) {
      issue_weights(it, cw.rb, cw.ks);
      if (su < nunits) ok = issue_scales();
      cw.next(vs);
    }
    const int su_early = su;
    // (T = 1) the resident activation slots, in visiting order, unless the
    // fold warps build them
    const int nq = nunits < KS ? nunits : KS;
    if constexpr (C::kInKernelX) {
      // The fold warps read the stages' x right after the previous grid ends:
      // warm L2 with it first (a prefetch only moves lines into L2, so it is
      // harmless while an earlier kernel may still write x).
      if (build_x && lane < nq) {
        const int ks = new_stage(vs, lane);
        const int kk = K - ks * kSTStageK < kSTStageK ? K - ks * kSTStageK : kSTStageK;
        bulk_prefetch_l2(x + static_cast<size_t>(tok0) * K + static_cast<size_t>(ks) * kSTStageK,
                    static_cast<uint32_t>(kk) * 2u);
      }
    }
    grid_dependency_wait();
    if constexpr (C::kInKernelX) {
      if (!build_x && lane == 0)
        for (int q = 0; q < nq; ++q) {
          mbar_arrive_expect_tx(&xready[q], kX1Slot);
          bulk_load(xres + q * kX1Slot,
                    xprep + static_cast<size_t>(new_stage(vs, q)) * kX1Slot, kX1Slot, &xready[q]);
        }
    }
    if constexpr (!C::kInKernelX) {
      Cursor ce;
      ce.start(vs);
      for (int j = 0; j < su_early; ++j, ce.next(vs)) {
        if (j < it) issue_x(j, ce.ks);
        issue_f(j, ce.ks);
      }
    }
    for (; it < nunits && ok; ++it) {
      const int s = it % S;
      if (it >= S && !__all_sync(0xffffffffu, mbar_wait(&empty[s], ((it / S) & 1) ^ 1, err))) break;
      issue_weights(it, cw.rb, cw.ks);
      issue_x(it, cw.ks);
      if (su < nunits) {
        const int fks = cs.ks;
        const int fu = su;
        ok = issue_scales();
        if (ok) issue_f(fu, fks);
      }
      cw.next(vs);
    }
    // Stay until this CTA's copies have landed (bounded).
    for (int d = (it > S ? it - S : 0); d < it; ++d)
      if (!mbar_wait(&full[d % S], (d / S) & 1, err)) break;
    for (int d = (su > SS ? su - SS : 0); d < su; ++d)
      if (!mbar_wait(&sfull[d % SS], (d / SS) & 1, err)) break;
    if constexpr (C::kInKernelX)
      if (!build_x)
        for (int q = 0; q < nq; ++q)
          if (!mbar_wait(&xready[q], 0, err)) break;
  } else if (warp == kXWarp0) {
    // ------------------------------------------------------------ split-row sums
    // Warp kXWarp0 combines
    // the CTA's split row blocks as the fold hands over their sums, with a
    // ticket per row block (kept at the index of its first CTA).  The fold
    // never waits for any of this, and no CTA waits for another: each CTA
    // publishes its sums to the workspace and takes the ticket; the last adds
    // every partial in CTA order and writes y, so the bits do not depend on
    // which CTA finished last.  It puts the ticket back to zero for the next
    // launch.
    //   A row block shared with one other CTA and begun here is this CTA's
    // last; the other CTA starts with it and usually publishes long before
    // this one is done.  So while the fold works, this warp polls the ticket
    // and, once the other's partial is out, copies it into the free split
    // slot; the end of the row block is then an add and the stores.  (When
    // the poll finds nothing by then, the general way applies.)
    if (cl > 1) {
      // Cluster mode: rank r > 0 stores its sums into rank 0's shared memory
      // (slot r - 1) and every lane arrives on rank 0's barrier (release,
      // cluster scope); rank 0 adds the ranks' sums to 0 in rank order.
      const float* mine = reinterpret_cast<const float*>(smem + C::kSplitOff);
      const int n = sp[0] * kRows + 4 * lane;
      if (__all_sync(0xffffffffu, mbar_wait(&pub[0], 0, err))) {
        if constexpr (C::kCluster) {
          const float* buf = reinterpret_cast<const float*>(smem + C::kClOff);
          if (crank != 0) {
            const uint32_t dst = mapa_shared(
                smem_addr(smem + C::kClOff) + static_cast<uint32_t>((crank - 1) * TT * kRows * 4), 0);
            for (int t = 0; t < Tt; ++t)
              st_cluster_v4(dst + static_cast<uint32_t>((t * kRows + 4 * lane) * 4),
                            *reinterpret_cast<const float4*>(mine + t * kRows + 4 * lane));
            mbar_arrive_remote(mapa_shared(smem_addr(cfull), 0));
          } else if (__all_sync(0xffffffffu, mbar_wait_cluster(cfull, 0, err))) {
            for (int t = 0; t < Tt; ++t) {
              float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int rk = 0; rk < cl; ++rk) {
                const float* src = rk == 0 ? mine : buf + (rk - 1) * TT * kRows;
                const float4 v = *reinterpret_cast<const float4*>(src + t * kRows + 4 * lane);
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
              }
              const float a[4] = {acc.x, acc.y, acc.z, acc.w};
              float* yr = y + static_cast<size_t>(tok0 + t) * N + n;
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (n + e < N) yr[e] = a[e];
            }
          }
        }
      }
    } else {
      auto first_rb = [&](int c) { return static_cast<int>(U * c / P / KS); };
      float* split_sums = reinterpret_cast<float*>(smem + C::kSplitOff);
      for (int i = 0; i < nsp; ++i) {
        const int rb = sp[i];
        const long long u0 = static_cast<long long>(rb) * KS;
        const int c0 = owner_of(u0, U, P), c1 = owner_of(u0 + KS - 1, U, P);
        const float* mine = split_sums + i * TT * kRows;  // [TT][128] in shared memory
        const int n = rb * kRows + 4 * lane;               // lane l: rows 4l .. 4l+3
        // slot 1 - i is free here: slot 0 is published before slot 1 is
        // used, and with one split row block slot 1 is never used
        float* other = split_sums + (1 - i) * TT * kRows;
        bool early = false;
        if (c1 - c0 == 1 && cta == c0 && i == nsp - 1) {
          const unsigned long long t0 = global_timer_ns();
          bool fine = true;
          for (;;) {
            const bool ready = __any_sync(0xffffffffu, mbar_try_wait(&pub[i], 0));
            if (!early) {
              int tk = 0;
              if (lane == 0) tk = ld_acquire_gpu(&tickets[c0]);
              tk = __shfl_sync(0xffffffffu, tk, 0);
              __syncwarp();
              if (tk == 1) {  // CTA c1 has published (its first row block: slot 0)
                const float* pc = partials + static_cast<size_t>(c1) * 2 * TT * kRows + 4 * lane;
                for (int t = 0; t < Tt; ++t)
                  *reinterpret_cast<float4*>(other + t * kRows + 4 * lane) =
                      __ldcg(reinterpret_cast<const float4*>(pc + t * kRows));
                early = true;
              }
            }
            if (ready) break;
            if (early) break;  // nothing left to overlap: wait below
            if (global_timer_ns() - t0 > kWaitLimitNs) {
              if (lane == 0) atomicOr(err, kErrTimeout);
              fine = false;
              break;
            }
            __nanosleep(256);
          }
          if (!fine) break;
        }
        // (every lane acquires the fold's stores to `mine`)
        if (!__all_sync(0xffffffffu, mbar_wait(&pub[i], 0, err))) break;
        if (early) {
          // y = (0 + own) + other's: the general sum's order and bits
          for (int t = 0; t < Tt; ++t) {
            const float4 a = *reinterpret_cast<const float4*>(mine + t * kRows + 4 * lane);
            const float4 b = *reinterpret_cast<const float4*>(other + t * kRows + 4 * lane);
            const float v[4] = {(0.f + a.x) + b.x, (0.f + a.y) + b.y, (0.f + a.z) + b.z,
                                (0.f + a.w) + b.w};
            float* yr = y + static_cast<size_t>(tok0 + t) * N + n;
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (n + e < N) yr[e] = v[e];
          }
          if (lane == 0) tickets[c0] = 0;  // the other CTA has taken it: ready for the next launch
          continue;
        }
        // publish this CTA's sums (slot 0: its first row block, 1: its last)
        {
          const float4* src = reinterpret_cast<const float4*>(mine);
          float4* dst = reinterpret_cast<float4*>(
              partials + static_cast<size_t>(cta * 2 + (rb == rb0 ? 0 : 1)) * TT * kRows);
#pragma unroll
          for (int e = 0; e < TT; ++e) dst[e * 32 + lane] = src[e * 32 + lane];
          __threadfence();
          __syncwarp();
        }
        // the ticket: acquire-release at GPU scope (every lane fenced its part
        // of the partial first; a last arriver reads the others' after)
        int last = 0;
        if (lane == 0) last = atomic_add_acq_rel_gpu(&tickets[c0], 1) == c1 - c0;
        last = __shfl_sync(0xffffffffu, last, 0);
        __syncwarp();
        if (!last) continue;
        // eight float4 loads in flight at a time (up to eight tokens of
        // 8 / tokens CTAs), the CTAs' partials added in CTA order
        constexpr int kTC = TT < 8 ? TT : 8;
        constexpr int kCB = 8 / kTC;
        for (int t0 = 0; t0 < Tt; t0 += kTC) {
          float4 acc[kTC];
#pragma unroll
          for (int tj = 0; tj < kTC; ++tj) acc[tj] = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int cb = c0; cb <= c1; cb += kCB) {
            float4 v[kCB][kTC];
#pragma unroll
            for (int ci = 0; ci < kCB; ++ci) {
              const int c = cb + ci;
              const float* pc =
                  partials + static_cast<size_t>(c * 2 + (first_rb(c) == rb ? 0 : 1)) * TT * kRows +
                  4 * lane;
#pragma unroll
              for (int tj = 0; tj < kTC; ++tj)
                v[ci][tj] = c <= c1 && t0 + tj < Tt
                                ? __ldcg(reinterpret_cast<const float4*>(pc + (t0 + tj) * kRows))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int ci = 0; ci < kCB; ++ci) {
              if (cb + ci > c1) break;
#pragma unroll
              for (int tj = 0; tj < kTC; ++tj) {
                acc[tj].x += v[ci][tj].x;
                acc[tj].y += v[ci][tj].y;
                acc[tj].z += v[ci][tj].z;
                acc[tj].w += v[ci][tj].w;
              }
            }
          }
#pragma unroll
          for (int tj = 0; tj < kTC; ++tj) {
            if (t0 + tj >= Tt) continue;
            float* yr = y + static_cast<size_t>(tok0 + t0 + tj) * N + n;
            const float a[4] = {acc[tj].x, acc[tj].y, acc[tj].z, acc[tj].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (n + e < N) yr[e] = a[e];
          }
        }
        if (lane == 0) tickets[c0] = 0;  // every other CTA has taken it: ready for the next launch
      }
    }
  } else if (warp >= kMmaWarp && warp < kMmaWarp + kMmaWarps) {
    // ------------------------------------------------------------ MMA issuers
    // Each warp runs its loop whole so that addresses and descriptors stay
    // warp-uniform; one elected lane issues.  Half-stage hu = 2 it + hh
    // (groups 4 hh .. 4 hh + 3) uses A sub-slots (2 it + b) % NSUB of half
    // hh's ring (b = 0, 1) and D slot hu % ND, and is issued by MMA warp hh.
    const int w = warp - kMmaWarp;
    const bool leader = elect_one();
    constexpr uint32_t idesc = idesc_e4m3_e5m2_f32(kRows, NC);
    constexpr uint32_t idesc3 = idesc_e4m3_e5m2_f32(kRows, 16);  // piece-2 block
    // Descriptor of stage (slot) 0's B block; a stage / k chunk only moves the
    // start address field (address >> 4 in the low bits).
    const uint64_t desc0 =
        C::kInKernelX ? smem_desc_kmajor(smem_addr(xres), kX1Lbo, kX1Sbo)
                      : smem_desc_kmajor(smem_addr(smem + C::kXOff), kXLbo, kXSbo);
    constexpr uint32_t kLbo = C::kInKernelX ? kX1Lbo : kXLbo;
    int last = -1;
    Cursor cu;
    cu.start(vs);
    for (int hu = w; hu < 2 * nunits; hu += kMmaWarps, cu.next(vs)) {
      const int it = hu >> 1, hh = hu & 1;
      const int s = it % S;
      const int ks = cu.ks;
      const int ng = G - kGS * ks < kGS ? G - kGS * ks : kGS;
      const int q = stage_slot(vs, ks);  // (T = 1) resident slot
      const uint64_t dstage =
          desc0 + static_cast<uint64_t>((C::kInKernelX ? q * kX1Slot : s * C::kXFrag) >> 4);
      const uint64_t dstage3 = dstage + static_cast<uint64_t>(C::kXMain >> 4);
      if constexpr (C::kInKernelX) {
        if (!__all_sync(0xffffffffu, mbar_wait(&xready[q], 0, err))) break;
      }
      const int d = hu % ND;
      if (hu >= ND &&
          !__all_sync(0xffffffffu, mbar_wait(&dfree[d], ((hu / ND) & 1) ^ 1, err)))
        break;
      const uint32_t dcol = tbase + C::kDCol + d * C::kDSlot;
      bool ok_h = true;
#pragma unroll
      for (int b = 0; b < 2; ++b) {  // the two A sub-slots of the half-stage
        const int u = 2 * it + b, j = u % NSUB;
        uint64_t* af = &afull[hh * NSUB + j];
        if (!__all_sync(0xffffffffu, mbar_wait(af, (u / NSUB) & 1, err))) {
          ok_h = false;
          break;
        }
        tc_fence_after();
        const uint32_t acol = tbase + C::kACol + hh * C::kAHalf + j * C::kSubCols;
        if (leader) {
#pragma unroll
          for (int gs = 0; gs < kGH / 2; ++gs) {
            const int gg = (kGH / 2) * b + gs;
            const int g = kGH * hh + gg;
            if (g < ng) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t koff = static_cast<uint64_t>(((8 * g + 2 * kk) * kLbo) >> 4);
                mma_f8f6f4_ts(dcol + gg * NC, acol + gs * 32 + kk * 8, dstage + koff, idesc,
                              kk > 0);
                if constexpr (C::kH3)  // piece 2 onto piece 0's columns
                  mma_f8f6f4_ts(dcol + gg * NC, acol + gs * 32 + kk * 8, dstage3 + koff, idesc3,
                                true);
              }
            }
          }
          mma_commit(&afree[hh * NSUB + j]);
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
    Cursor cu;
    cu.start(vs);
    for (int it = 0; it < nunits; ++it, cu.next(vs)) {
      const int s = it % S;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (it / S) & 1, err))) break;
      // half-stage h is weight box h: groups kGH h .. kGH h + kGH - 1.  All
      // of this warp's packed words of the unit go to registers first, so
      // that the ring slot is handed back to the producer at once (the slot
      // of a T > 1 stage also holds the activation block: there the MMA
      // commits release it).
      const uint8_t* wrow = smem + C::kWOff + s * C::kWBytes + h * (kRows * 128) + r * 128;
      const int ng = G - kGS * cu.ks < kGS ? G - kGS * cu.ks : kGS;
      uint4 wv[kGH][2];
#pragma unroll
      for (int gg = 0; gg < kGH; ++gg) {
        wv[gg][0] = lds_v4(wrow + (((2 * gg) ^ (r & 7)) << 4));
        wv[gg][1] = lds_v4(wrow + (((2 * gg + 1) ^ (r & 7)) << 4));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      bool ok_h = true;
#pragma unroll
      for (int b = 0; b < 2; ++b) {  // groups 2 b, 2 b + 1 of the half-stage
        const int u = 2 * it + b, j = u % NSUB;  // into sub-slot j of this half's ring
        if (u == NSUB) grid_dependency_wait();  // (the early stages cover u < NSUB)
        if (u >= NSUB &&
            !__all_sync(0xffffffffu,
                        mbar_wait(&afree[h * NSUB + j], ((u / NSUB) & 1) ^ 1, err))) {
          ok_h = false;
          break;
        }
        tc_fence_after();
        const uint32_t acol = tbase + lane_off + C::kACol + h * C::kAHalf + j * C::kSubCols;
#pragma unroll
        for (int gs = 0; gs < kGH / 2; ++gs) {
          const int gg = (kGH / 2) * b + gs;
          const int g = kGH * h + gg;
          if (g < ng) {
            const uint4 c0 = wv[gg][0], c1 = wv[gg][1];
            const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            uint32_t av[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              av[4 * j + 0] = decode_e4m3<0>(w[j]);
              av[4 * j + 1] = decode_e4m3<1>(w[j]);
              av[4 * j + 2] = decode_e4m3<2>(w[j]);
              av[4 * j + 3] = decode_e4m3<3>(w[j]);
            }
            tmem_st32(acol + gs * 32, av);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[h * NSUB + j]);
      }
      if (!ok_h) break;
    }
  } else {
    // ------------------------------------------------------------ fold
    if (C::kInKernelX && build_x) {
      // (T = 1, few units per CTA) Before any accumulator is ready, fold warp
      // jg builds group jg of the activation block of every stage the CTA
      // visits, into the resident slots in visiting order (all loads first).
      const int jg = warp - kDecWarps;
      const int nq = nunits < KS ? nunits : KS;
      uint2 raw[kSmallTX1MaxSlots];
#pragma unroll
      for (int q = 0; q < kSmallTX1MaxSlots; ++q) {
        raw[q] = make_uint2(0u, 0u);
        const int gi = q < nq ? new_stage(vs, q) * kGS + jg : G;
        if (gi < G)
          raw[q] = *reinterpret_cast<const uint2*>(x + static_cast<size_t>(tok0) * K + gi * 128 +
                                                   4 * lane);
      }
#pragma unroll
      for (int q = 0; q < kSmallTX1MaxSlots; ++q) {
        if (q < nq) {
          prep_task<1>(raw[q], xres + q * kX1Slot, 0, jg, lane);
          fence_proxy_async_smem();  // the MMA reads the block through the async proxy
          __syncwarp();
          if (lane == 0) mbar_arrive(&xready[q]);
        }
      }
    }
    // Fold warp f owns TMEM lane quarter fq = f % 4 (rows 32 fq .. 32 fq + 31)
    // and half-stage fh = f / 4 (groups 4 fh .. 4 fh + 3) of every stage:
    // y[t][row] += s[row][g] * f[g][t] * (sum of the pieces' accumulators of
    // token t).  At the end of a row block the fh = 1 warp hands its sums to
    // the fh = 0 warp of the same quarter, which writes y (or, for a row
    // block shared with other CTAs, publishes them for the split-row warp).
    //
    // Leftovers (a group's elements more than 21 binades below its absmax,
    // flagged by a negative f, with their sum of |x| in L): for each output,
    // their contribution is at most s * L.  A leftover group is first left
    // out, its bound added to the row's budget lam and the group noted (up to
    // kDefer per row block; past that it is added exactly at once).  When the
    // row block ends, |yacc| of this warp's groups is a lower bound of
    // sum|s w x| over them (every term added is an exact part of y, or the
    // pieces' sum, bounded by its own sum of |s w x|); if lam is within 2^-11
    // of it the noted groups stay out: the error is below 2^-11 of
    // sum|s w x|, half the bf16 rungs' bar.  Otherwise the noted groups of
    // that token are added exactly (leftover_dot, on the group's x staged in
    // shared memory, the weights and scale read again from global memory).
    // One budget lam serves all tokens of a row: a token's own left-out
    // bounds never exceed it.
    const int fq = (warp - kDecWarps) & 3;  // == warp % 4
    const int fh = (warp - kDecWarps) >> 2;
    const int r = fq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(fq * 32) << 16;
    float yacc[TT];
    float lam = 0.f;  // leftover bounds left out so far in this row block
#pragma unroll
    for (int t = 0; t < TT; ++t) yacc[t] = 0.f;

    float* half_part = reinterpret_cast<float*>(smem + C::kPartOff);  // [TT][128]
    float* split_sums = reinterpret_cast<float*>(smem + C::kSplitOff);  // [2][TT][128]
    uint2* lx = reinterpret_cast<uint2*>(smem + C::kLxOff) + (warp - kDecWarps) * 32;
    uint2* defer = reinterpret_cast<uint2*>(smem + C::kDefOff) + (warp - kDecWarps) * C::kDefer;
    int ndef = 0;  // noted leftover groups in this row block (warp-uniform)
    // Add leftover group g (within stage ks) of token t exactly to yacc[t]
    // where pred; sg: the row's scale of the group.  The whole warp calls it.
    auto add_exact = [&](int ks, int g, int t, float f_abs, float sg, bool pred, int n) {
      if (!__any_sync(0xffffffffu, pred)) return;
      // the group's x into this warp's staging area, the row's weights at the
      // same time: one memory round trip
      const int ga = ks * kGS + g;
      const uint2 xv = *reinterpret_cast<const uint2*>(
          x + static_cast<size_t>(tok0 + t) * K + ga * 128 + 4 * lane);
      uint4 wa = make_uint4(0, 0, 0, 0), wb = wa;
      if (pred) {
        const uint4* wq =
            reinterpret_cast<const uint4*>(wp + static_cast<size_t>(n) * (K >> 4) + ga * 8);
        wa = ldg_nc_v4(wq);
        wb = ldg_nc_v4(wq + 1);
      }
      lx[lane] = xv;
      __syncwarp();
      if (pred) {
        const float d = leftover_dot(wa, wb, reinterpret_cast<const uint32_t*>(lx),
                                     leftover_limit(f_abs));
#pragma unroll
        for (int u = 0; u < TT; ++u)
          if (u == t) yacc[u] = fmaf(sg, d, yacc[u]);
      }
      __syncwarp();
    };
    // Decide the noted leftover groups of the row block ending here.
    auto settle_leftovers = [&](int rb) {
      if (ndef == 0) return;  // warp-uniform
      const int n = rb * kRows + r;
      uint32_t need = 0;  // bit t: token t's noted groups are added exactly
#pragma unroll
      for (int t = 0; t < TT; ++t)
        if (lam > 0x1p-11f * fabsf(yacc[t])) need |= 1u << t;
      __syncwarp();
#pragma unroll 1
      for (int e = 0; e < ndef; ++e) {
        const uint2 de = defer[e];
        const int t = de.x & 15, g = (de.x >> 4) & 15, ks = static_cast<int>(de.x >> 8);
        const bool pred = ((need >> t) & 1u) && n < N && t < Tt;
        float sg = 0.f;
        if (pred)
          sg = __half2float(__ushort_as_half(scales[static_cast<size_t>(n) * G + ks * kGS + g]));
        add_exact(ks, g, t, __uint_as_float(de.y), sg, pred, n);
      }
      ndef = 0;
    };
    int nflush = 0;
    int nsplit = 0;
    // Row block rb's sums are final in yacc (fh = 0 warps): a row block whole
    // in this CTA is stored; a split one's sums are published as this CTA's
    // partial (slot 0: the CTA's first row block, 1: its last) for the
    // split-row warp.  false: a bounded wait gave up.
    auto flush = [&](int rb) -> bool {
      const int n = rb * kRows + r;
      settle_leftovers(rb);
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
        if (nsplit < nsp && rb == sp[nsplit]) {
          float* mine = split_sums + nsplit * TT * kRows;
#pragma unroll
          for (int t = 0; t < TT; ++t) mine[t * kRows + r] = yacc[t];
          __syncwarp();
          if (lane == 0) mbar_arrive(&pub[nsplit]);
          ++nsplit;
        } else {
#pragma unroll
          for (int t = 0; t < TT; ++t)
            if (n < N && t < Tt) y[static_cast<size_t>(tok0 + t) * N + n] = yacc[t];
        }
      }
      ++nflush;
#pragma unroll
      for (int t = 0; t < TT; ++t) yacc[t] = 0.f;
      lam = 0.f;
      return true;
    };

    Cursor cu;
    cu.start(vs);
    bool ok = true;
    for (int j = 0; j < nunits && ok; ++j, cu.next(vs)) {
      const int ss = j % SS;
      if (!__all_sync(0xffffffffu, mbar_wait(&sfull[ss], (j / SS) & 1, err))) break;
      const int ks = cu.ks;
      const int ng = G - kGS * ks < kGS ? G - kGS * ks : kGS;
      const uint8_t* sst = smem + C::kSOff + ss * C::kSBytes;
      // this half-stage's kGH fp16 scales
      const uint2 s4 = lds_v2(sst + r * (2 * kGS) + fh * (2 * kGH));
      auto scale_of = [&](int gg) {
        const uint32_t sp2 = gg < 2 ? s4.x : s4.y;
        return __half2float(__ushort_as_half(
            static_cast<unsigned short>((gg & 1) ? (sp2 >> 16) : (sp2 & 0xFFFFu))));
      };
      const int q = stage_slot(vs, ks);  // (T = 1) resident slot
      // (f, L) of group g (within the stage), token t
      auto fl_of = [&](int g, int t) -> float2 {
        if constexpr (C::kInKernelX) {
          return reinterpret_cast<const float2*>(xres + q * kX1Slot + kX1Stage)[g];
        } else {
          const float* fl = reinterpret_cast<const float*>(sst + kRows * 2 * kGS);
          return make_float2(fl[g * H + t], fl[(kGS + g) * H + t]);
        }
      };
      if constexpr (C::kInKernelX) {
        if (!__all_sync(0xffffffffu, mbar_wait(&xready[q], 0, err))) break;
      }
      const int hu = 2 * j + fh;
      const int d = hu % ND;
      if (!__all_sync(0xffffffffu, mbar_wait(&mdone[d], (hu / ND) & 1, err))) break;
      tc_fence_after();
      const uint32_t dbase = tbase + lane_off + C::kDCol + d * C::kDSlot;
      // (warp-uniform) bit gg: group gg of the half-stage has leftovers for
      // some token (from an OR of the factors' sign bits)
      uint32_t gflag = 0;
      // Only the accumulator columns that carry tokens are read back; dv[]
      // holds them with piece j of token t at dv[PJ[j] + t].
      auto fold_group = [&](int gg, const uint32_t* dv) {
        const float sg = scale_of(gg);
        const int g = kGH * fh + gg;
        uint32_t fbits = 0;
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          float dsum;
          if constexpr (TT == 1)
            dsum = (__uint_as_float(dv[0]) + __uint_as_float(dv[1])) + __uint_as_float(dv[2]);
          else if constexpr (C::kH3)
            dsum = __uint_as_float(dv[t]) + __uint_as_float(dv[C::kP1 + t]);
          else
            dsum = (__uint_as_float(dv[t]) + __uint_as_float(dv[C::kP1 + t])) +
                   __uint_as_float(dv[C::kP2 + t]);
          const float f = fl_of(g, t).x;
          fbits |= __float_as_uint(f);
          yacc[t] = fmaf(sg * fabsf(f), dsum, yacc[t]);
        }
        gflag |= (fbits >> 31) << gg;
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
        constexpr int kDV = TT == 1 ? 3 : 12;
        uint32_t dv[kGH][kDV];
#pragma unroll
        for (int gg = 0; gg < kGH; ++gg) {
          if (kGH * fh + gg < ng) {
            const uint32_t col = dbase + gg * NC;
            if constexpr (TT == 1) {
              tmem_ld2(col, dv[gg]);            // pieces 0, 1 (columns 0, 1)
              tmem_ld1(col + C::kP2, dv[gg][2]);  // piece 2 (column 8)
            } else {
              tmem_ld4(col, dv[gg]);
              tmem_ld4(col + C::kP1, dv[gg] + 4);
              tmem_ld4(col + C::kP2, dv[gg] + 8);
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
      if (gflag) {  // rare: groups with leftovers (see above)
#pragma unroll 1
        for (int bit = 0; bit < kGH * TT; ++bit) {
          const int gg = bit / TT, t = bit % TT;
          if (!((gflag >> gg) & 1u)) continue;
          const int g = kGH * fh + gg;
          const float2 fl = fl_of(g, t);
          if (!(fl.x < 0.f)) continue;
          const float sg = scale_of(gg);
          if (ndef < C::kDefer) {
            lam += sg * fl.y;  // |leftover contribution| <= s * L
            if (lane == 0)
              defer[ndef] = make_uint2(static_cast<uint32_t>(ks << 8 | g << 4 | t),
                                       __float_as_uint(-fl.x));
            ++ndef;
          } else {
            const int n = cu.rb * kRows + r;
            add_exact(ks, g, t, -fl.x, sg, n < N && t < Tt, n);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[ss]);
      if (cu.ends_row_block(vs)) ok = flush(cu.rb);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // no CTA of a cluster leaves while another may still write its shared memory
  if (cl > 1) cluster_sync_all();
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

// Grid of the small-T kernel for (K, N): units U, CTAs P, stages KS.
// Most clusters of c CTAs of smallt_kernel<TT> that can be resident at once
// (cached per tile and size; 0 when the query fails).
template <int TT>
int max_active_clusters(int c) {
  static int cache[kMaxCl + 1] = {-1, -1, -1, -1, -1};
  if (cache[c] >= 0) return cache[c];
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(c);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(c));
  cfg.blockDim = dim3(TC<TT>::kThreads);
  cfg.dynamicSmemBytes = TC<TT>::kAllocMax;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, smallt_kernel<TT>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  cache[c] = n;
  return n;
}

int max_active_clusters_tt(int tt, int c) {
  switch (tt) {
    case 1: return max_active_clusters<1>(c);
    default: return 0;
  }
}

struct SmallTGrid {
  int KS;
  long long U, P;
  int cl;  // CTAs per row block in cluster mode, else 1
};
// Grid of the small-T kernel for tile tt: units U, CTAs P, stages KS.  A
// layer with few row blocks (each to be shared by several CTAs anyway) runs
// in cluster mode when it fits: one cluster of cl CTAs per row block, all
// clusters resident at once, so the row block's sums meet in shared memory.
SmallTGrid smallt_grid(int K, int N, int num_sms, int tt) {
  SmallTGrid g;
  g.KS = (K + kSTStageK - 1) / kSTStageK;
  const long long NB = (N + kRows - 1) / kRows;
  g.U = NB * g.KS;
  long long P = num_sms;  // one CTA per SM: each holds all 512 TMEM columns
  if (P > kSmallTMaxCtas) P = kSmallTMaxCtas;
  if (P > g.U) P = g.U;
  g.P = P;
  g.cl = 1;
  if (cluster_tile(tt) && g.KS >= 2 && 2 * NB <= P) {
    long long c = P / NB;
    if (c > kMaxCl) c = kMaxCl;
    if (c > g.KS) c = g.KS;
    while (c >= 2 && max_active_clusters_tt(tt, static_cast<int>(c)) < NB) --c;
    if (c >= 2) {
      g.cl = static_cast<int>(c);
      g.P = NB * c;
    }
  }
  return g;
}

// Units of the CTA with the most.
long long max_units_per_cta(const SmallTGrid& g) {
  return g.cl > 1 ? (g.KS + g.cl - 1) / g.cl : (g.U + g.P - 1) / g.P;
}

// Resident activation slots of the one-token kernel: the distinct stages a CTA
// visits at most.
int t1_slots(const SmallTGrid& g) {
  const long long per = max_units_per_cta(g);
  return static_cast<int>(per < g.KS ? per : g.KS);
}

template <int TT>
cudaError_t launch_tt(const CUtensorMap* tmW, const uint32_t* Wp, const uint16_t* scales,
                      const uint16_t* x, int* sync, uint8_t* work, float* y, int K, int N,
                      int tok0, int Tt, int num_sms, int act, int* err, cudaStream_t stream,
                      int* launches) {
  const bool rotate = act == kActRotated;
  using C = TC<TT>;
  const SmallTGrid g = smallt_grid(K, N, num_sms, TT);
  const int nslots = C::kInKernelX ? t1_slots(g) : 0;
  if (nslots > kSmallTX1MaxSlots) return cudaErrorInvalidValue;
  float* partials = reinterpret_cast<float*>(work);
  uint8_t* xprep = work + smallt_partials_bytes(TT);

  // (T = 1) With at most two units per CTA the call is short and the prep
  // kernel's extra dependency step costs more than building the few stages
  // in every CTA from x; with more, x is better read once by the prep kernel
  // (an L2 hit for the main kernel, whose own reads of x would queue behind
  // its weight stream).
  const int build_x = C::kInKernelX && act == kActExact && max_units_per_cta(g) <= 2 ? 1 : 0;
  cudaLaunchAttribute attr[1];
  if (act == kActInt8) {
    // one 4-warp CTA per (token slot, stage)
    const int tasks = C::kH * g.KS;
    const int blocks = tasks < num_sms ? tasks : num_sms;
    cudaLaunchConfig_t pc = pdl_config(attr, dim3(blocks), dim3(kPrepWarps * 32), 0, stream);
    cudaError_t e = cudaLaunchKernelEx(&pc, xprep_i8_kernel<TT>, x, xprep, K, tok0, Tt, g.KS);
    if (e != cudaSuccess) return e;
    ++*launches;
  } else if (rotate) {
    // one warp per (token slot, stage): the stage is one rotation block
    const int tasks = C::kH * g.KS;
    const int blocks = tasks < num_sms ? tasks : num_sms;
    cudaLaunchConfig_t pc = pdl_config(attr, dim3(blocks), dim3(32), 0, stream);
    cudaError_t e = cudaLaunchKernelEx(&pc, xprep_rot_kernel<TT>, x, xprep, K, tok0, Tt, g.KS);
    if (e != cudaSuccess) return e;
    ++*launches;
  } else if (!build_x) {
    const int tasks = C::kH * kGS * g.KS;
    int blocks = (tasks + kPrepWarps - 1) / kPrepWarps;
    if (blocks > num_sms) blocks = num_sms;
    cudaLaunchConfig_t pc = pdl_config(attr, dim3(blocks), dim3(kPrepWarps * 32), 0, stream);
    cudaError_t e = cudaLaunchKernelEx(&pc, xprep_kernel<TT>, x, xprep, K, tok0, Tt, g.KS);
    if (e != cudaSuccess) return e;
    ++*launches;
  }
  cudaLaunchAttribute mattr[2];
  cudaLaunchConfig_t cfg = pdl_config(mattr, dim3(static_cast<unsigned>(g.P)), dim3(C::kThreads),
                                      C::smem_bytes(nslots), stream);
  if (g.cl > 1) {
    mattr[1].id = cudaLaunchAttributeClusterDimension;
    mattr[1].val.clusterDim.x = static_cast<unsigned>(g.cl);
    mattr[1].val.clusterDim.y = 1;
    mattr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, smallt_kernel<TT>, *tmW, Wp, scales, x,
                         static_cast<const uint8_t*>(xprep), y, sync, partials, K, N, tok0, Tt,
                         g.KS, nslots, g.U, build_x, g.cl, err);
  if (e == cudaSuccess) ++*launches;
  return e;
}

}  // namespace

size_t smallt_partials_bytes(int tt) {
  return static_cast<size_t>(kSmallTMaxCtas) * 2 * tt * kRows * sizeof(float);
}

size_t smallt_work_bytes(int tt, int K) {
  const int KS = (K + kSTStageK - 1) / kSTStageK;
  size_t prep = 0;
  switch (tt) {
    case 1: prep = static_cast<size_t>(TC<1>::kXBytes) * KS; break;
    case 4: prep = static_cast<size_t>(TC<4>::kXBytes) * KS; break;
    case 8: prep = static_cast<size_t>(TC<8>::kXBytes) * KS; break;
    default: prep = static_cast<size_t>(TC<16>::kXBytes) * KS; break;
  }
  return smallt_partials_bytes(tt) + prep;
}

int smallt_rows(int) { return kRows; }

int smallt_gemv_tile(int K, int N, int num_sms) {
  return t1_slots(smallt_grid(K, N, num_sms, 1)) <= kSmallTX1MaxSlots ? 1 : 4;
}

cudaError_t smallt_set_attributes() {
  cudaError_t e;
  if ((e = set_attr_one<1>()) != cudaSuccess) return e;
  if ((e = set_attr_one<4>()) != cudaSuccess) return e;
  if ((e = set_attr_one<8>()) != cudaSuccess) return e;
  if ((e = set_attr_one<16>()) != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t launch_smallt(int tt, const CUtensorMap* tmW, const uint32_t* Wp,
                          const uint16_t* scales, const uint16_t* x, int* sync, uint8_t* work,
                          float* y, int K, int N, int tok0, int Tt, int num_sms, int act,
                          int* err, cudaStream_t stream, int* launches) {
  switch (tt) {
    case 1:
      return launch_tt<1>(tmW, Wp, scales, x, sync, work, y, K, N, tok0, Tt, num_sms, act, err,
                          stream, launches);
    case 4:
      return launch_tt<4>(tmW, Wp, scales, x, sync, work, y, K, N, tok0, Tt, num_sms, act, err,
                          stream, launches);
    case 8:
      return launch_tt<8>(tmW, Wp, scales, x, sync, work, y, K, N, tok0, Tt, num_sms, act, err,
                          stream, launches);
    default:
      return launch_tt<16>(tmW, Wp, scales, x, sync, work, y, K, N, tok0, Tt, num_sms, act,
                           err, stream, launches);
  }
}

}  // namespace tern
