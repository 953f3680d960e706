// s8 rung (T >= 17): int8 per-token activations x ternary weights, exact
// integer accumulation per 128-wide group, fp32 output
//     y[t][n] = xs[t] * sum_g s[n][g] * acc[t][n][g],
//     acc[t][n][g] = sum_{k in g} q[t][k] w[n][k].
//
// On 5th-generation tensor cores.  sm_103a has no integer tcgen05 MMA, so the
// integers travel as exact fp8 e4m3 values:
//   * w / 8 in {-1/8, 0, 1/8} (the packed code decodes to it with a shift and
//     an AND, as in the small-T rungs);
//   * q = p1 + p2 with p1 = 16 rint(q / 16) and p2 = q - p1, both
//     exact in e4m3 (prepared by the pieces quantiser);
// and the two pieces are fed as two halves of the contraction into the same
// fp32 accumulator, which then holds exactly acc / 8 (|acc| <= 127 * 128, far
// inside fp32's exact integer range; every product is a multiple of 1/8).
//
// Tile: 128 weight rows (MMA M, TMEM lanes) x 128 tokens (MMA N).  Per
// 128-wide group a stage holds the packed weights (TMA, 128 rows x 32 B) and
// the two piece blocks (TMA, 128 tokens x 128 B each, 128-byte swizzle, the
// canonical K-major SW128 layout of the MMA's B operand).  The stage ring in
// shared memory is deeper than the ring of A slots in TMEM (which shares the
// 512 columns with the D slots), so copies run further ahead than decodes.
// Warp roles:
//   warps 0-3   decode the group's weights into an A slot in TMEM
//               (tcgen05.st, one row per thread);
//   kFoldW warps fold: read the D slot (each warp 32 rows x kFC tokens), add
//               8 s[n][g] * D into register accumulators, and at the end of
//               the tile store y = xs[t] * acc (each warp instruction writes
//               32 consecutive floats of one token's row);
//   one warp    producer (TMA) and the tile's x_scale block;
//   two warps   issue (one thread each, alternate groups) 8 MMAs per group
//               (4 per piece, K = 32 each) into a D slot (128 columns),
//               committing to the stage's and the slot's barriers.
// Work: persistent CTAs walk the (row block, token tile) tiles with the token
// tile fastest, so CTAs that run at the same time share the row block's
// weights in L2, and the pieces of all tokens stay L2-resident.
//
// This is the "s8" prefill rung of the "ninfer-perf-tuning" skill page
// (section 2 rung map), with int8 activations as in the "NInfer sm_89 fork"
// write-up (section 9 item 2); the pages run it on int8 mma.sync.
#include "tern_device.cuh"
#include "tern_internal.h"

namespace tern {
namespace {

constexpr int kRowsS = 128;   // weight rows per tile
constexpr int kNDS = 3;       // D slots
constexpr int kDecW = 4;
constexpr int kFoldW = kS8FoldWarps;
constexpr int kProdW = kDecW + kFoldW;
constexpr int kMmaW = kProdW + 1;  // first of kMmaWarps issuers
// The issuing thread runs in step with the tensor pipe (an MMA issues about
// as fast as it executes), so its barrier waits and commits would leave the
// pipe idle; two issuers take alternate groups and cover each other's gaps.
constexpr int kMmaWarps = 2;
constexpr int kThreadsS = (kMmaW + kMmaWarps) * 32;
// An issuer's previous group (u - kMmaWarps) waited for the fold of group
// u - kMmaWarps - kNDS, so when it checks the D slot for group u the slot's
// barrier is at most one phase behind, as a parity wait requires, only while
// kMmaWarps <= kNDS.
static_assert(kMmaWarps <= kNDS, "issuers may outrun the accumulator ring's parity check");

// Layout for a token tile of TOK tokens (MMA N): 128, or 32 for T <= 32,
// and a stage ring of NST stages (36 KB of copies per 128-token stage, 12 KB
// per 32-token one).  A 32-token tile does a quarter of the MMA and fold work
// per weight byte, so the call is bound by the bytes in flight: it gets 12
// stages.  The 128-token tile runs 4, or 6 when the piece blocks are too
// large to stay in L2 (each wave of CTAs reads all of them, so they then miss
// more often).  A slots (32 TMEM columns each) take what the D slots leave.
template <int TOK, int NST>
struct SL {
  static constexpr int kStages = NST;
  static constexpr int kASlots = TOK == 32 ? 12 : 4;
  // Parity waits: an issuer's previous use of a stage or A slot was its own
  // group (the groups alternate between the issuers).  A slot a of group u
  // is free once the stage of group u - kASlots is empty (its MMAs done),
  // which needs kASlots <= kStages.
  static_assert(kStages % kMmaWarps == 0 && kASlots % kMmaWarps == 0, "issuer parity");
  static_assert(kASlots <= kStages, "A slot reuse");
  static_assert(kStages > kNDS, "the fold's parity wait on the stage ring");
  static constexpr int kFC = TOK * 4 / kFoldW;  // tokens (D columns) per fold warp
  static_assert(kFoldW % 4 == 0 && kFC % 16 == 0, "fold split");
  static constexpr int kPB = TOK * 128;   // one piece block of a group
  static constexpr int kWB = kRowsS * 32;  // packed weights of a group (4 KB)
  static constexpr int kP1Off = 0;         // 1024-aligned (128-byte swizzle atoms)
  static constexpr int kP2Off = kP1Off + kStages * kPB;
  static constexpr int kWOff = kP2Off + kStages * kPB;
  static constexpr int kXsOff = kWOff + kStages * kWB;  // x_scale of 2 tiles
  static constexpr int kBarOff = kXsOff + 2 * TOK * 4;
  static constexpr int kNumBars = 2 * kStages + kASlots + kNDS + 4 + kMmaWarps;
  static constexpr int kTmemSlot = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kTmemSlot + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kACol = 0;
  static constexpr uint32_t kDCol = kASlots * 32;
  static_assert(kP2Off % 1024 == 0 && kWOff % 1024 == 0 && kXsOff % 16 == 0, "alignment");
  static_assert(kDCol + kNDS * TOK <= 512, "TMEM budget");
  static_assert(kAlloc <= 227 * 1024, "shared memory");
};

// Shared-memory descriptor of a K-major operand in the 128-byte swizzle
// layout: rows of 128 bytes, 8-row atoms 1024 bytes apart (stride byte
// offset), layout type 2 (SWIZZLE_128B) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

template <int TOK, int NST>
__global__ void __launch_bounds__(kThreadsS, 1)
    s8tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmP1,
                const __grid_constant__ CUtensorMap tmP2, const uint16_t* __restrict__ scales,
                const float* __restrict__ x_scale, float* __restrict__ y, int T, int K, int N,
                int nfull, int chunks,
                int* __restrict__ tickets, float* __restrict__ partials, int* err) {
  using L = SL<TOK, NST>;
  grid_dependents_launch();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  // empty[s]: the stage's weights are decoded and its group's MMAs are
  // complete (so its pieces and the group's A slot have been read, and its D
  // slot holds the group's sums)
  uint64_t* empty = full + L::kStages;
  uint64_t* afull = empty + L::kStages;  // A slot written
  uint64_t* dfree = afull + L::kASlots;  // D slot read back
  uint64_t* xsfull = dfree + kNDS;     // [2] tile's x_scale landed
  uint64_t* xsfree = xsfull + 2;       // [2] ... and used
  uint64_t* mfin = xsfree + 2;         // [issuer] all of that issuer's MMAs complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  const float* xs_tile = reinterpret_cast<const float*>(smem + L::kXsOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = K >> 7;
  const int RB = (N + kRowsS - 1) / kRowsS;
  const int TB = (T + TOK - 1) / TOK;
  const int tiles = RB * TB;
  // Work items, walked by the persistent CTAs (item blockIdx.x + m gridDim.x):
  // the first nfull tiles whole, then each remaining tile as `chunks` ranges
  // of its groups.  A chunked tile's warps publish partial sums and the last
  // chunk to finish adds them in chunk order (see the fold).
  const int nitems_all = nfull + (tiles - nfull) * chunks;
  struct Item {
    int tile, g0, g1, chunk;  // chunk < 0: the whole tile
  };
  auto item_of = [&](int m) -> Item {
    const int idx = blockIdx.x + m * static_cast<int>(gridDim.x);
    Item it;
    if (idx < nfull) {
      it.tile = idx;
      it.g0 = 0;
      it.g1 = G;
      it.chunk = -1;
    } else {
      const int j = idx - nfull;
      it.tile = nfull + j / chunks;
      it.chunk = j % chunks;
      it.g0 = G * it.chunk / chunks;
      it.g1 = G * (it.chunk + 1) / chunks;
    }
    return it;
  };
  const int nitems = blockIdx.x < nitems_all
                         ? (nitems_all - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1
                         : 0;
  int units = 0;
  for (int m = 0; m < nitems; ++m) {
    const Item it = item_of(m);
    units += it.g1 - it.g0;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecW + 1);
    }
    for (int a = 0; a < L::kASlots; ++a) mbar_init(&afull[a], kDecW);
    for (int d = 0; d < kNDS; ++d) mbar_init(&dfree[d], kFoldW);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&xsfull[b], 1);
      mbar_init(&xsfree[b], kFoldW);
    }
    for (int w = 0; w < kMmaWarps; ++w) mbar_init(&mfin[w], 1);
    fence_mbar_init();
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmP1);
    prefetch_tensormap(&tmP2);
  }
  if (warp == kMmaW) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // the set-up above overlaps the previous kernel; the pieces, x_scale, y and
  // the workspace belong to it until it has finished
  grid_dependency_wait();

  if (warp == kProdW) {
    // ------------------------------------------------------------ producer
    // one thread: copies need no warp, and single-thread waits are cheapest
    if (lane == 0) {
      int u = 0, s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int m = 0; m < nitems && ok; ++m) {
        const Item itm = item_of(m);
        const int rb = itm.tile / TB, tb = itm.tile % TB;
        // this tile's x_scale block (padded to whole 16-byte chunks: the
        // workspace rounds the x_scale array up to 256 bytes)
        const int xb = m & 1;
        if (m >= 2 && !mbar_wait(&xsfree[xb], ((m >> 1) & 1) ^ 1, err)) break;
        const int cnt = T - tb * TOK < TOK ? T - tb * TOK : TOK;
        const uint32_t bytes = static_cast<uint32_t>((cnt * 4 + 15) & ~15);
        mbar_arrive_expect_tx(&xsfull[xb], bytes);
        bulk_load(smem + L::kXsOff + xb * TOK * 4, x_scale + tb * TOK, bytes, &xsfull[xb]);
        for (int g = itm.g0; g < itm.g1; ++g, ++u) {
          if (u >= L::kStages && !mbar_wait(&empty[s], ph ^ 1, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], L::kWB + 2 * L::kPB);
          tma_load_2d(smem + L::kWOff + s * L::kWB, &tmW, g * 32, rb * kRowsS, &full[s]);
          tma_load_2d(smem + L::kP1Off + s * L::kPB, &tmP1, g * 128, tb * TOK, &full[s]);
          tma_load_2d(smem + L::kP2Off + s * L::kPB, &tmP2, g * 128, tb * TOK, &full[s]);
          if (++s == L::kStages) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      // no copy of this CTA may still be in flight when it exits
      for (int v = (u > L::kStages ? u - L::kStages : 0); v < u; ++v)
        if (!mbar_wait(&full[v % L::kStages], (v / L::kStages) & 1, err)) break;
      for (int m = (nitems > 2 ? nitems - 2 : 0); m < nitems; ++m)
        if (!mbar_wait(&xsfull[m & 1], (m >> 1) & 1, err)) break;
    }
    __syncwarp();
  } else if (warp < kDecW) {
    // ------------------------------------------------------------ decode
    const int r = warp * 32 + lane;  // row of the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    int s = 0, a = 0;
    uint32_t ph = 0;
    for (int u = 0; u < units; ++u) {
      // A slot a was last read by group v = u - kASlots, whose stage's empty
      // barrier completes with those MMAs (implied by full[s] when the rings
      // have one length: the copy into stage s waited on it)
      bool ok = mbar_wait(&full[s], ph, err);
      if (L::kASlots < L::kStages && ok && u >= L::kASlots) {
        const int v = u - L::kASlots;
        ok = mbar_wait(&empty[v % L::kStages], (v / L::kStages) & 1, err);
      }
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint8_t* wrow = smem + L::kWOff + s * L::kWB + r * 32;
      const uint4 c0 = lds_v4(wrow);
      const uint4 c1 = lds_v4(wrow + 16);
      const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      uint32_t av[32];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        av[4 * j + 0] = decode_e4m3<0>(w[j]);
        av[4 * j + 1] = decode_e4m3<1>(w[j]);
        av[4 * j + 2] = decode_e4m3<2>(w[j]);
        av[4 * j + 3] = decode_e4m3<3>(w[j]);
      }
      tmem_st32(tbase + lane_off + L::kACol + a * 32, av);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&afull[a]);
        mbar_arrive(&empty[s]);
      }
      if (++s == L::kStages) {
        s = 0;
        ph ^= 1;
      }
      if (++a == L::kASlots) a = 0;
    }
  } else if (warp >= kMmaW) {
    // ------------------------------------------------------------ MMA issuers
    // one thread per issuer warp, groups u = w, w + kMmaWarps, ...; no warp
    // votes, one commit per group
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(kRowsS, TOK);
      const uint64_t desc1 = smem_desc_sw128(smem_addr(smem + L::kP1Off));
      const uint64_t desc2 = smem_desc_sw128(smem_addr(smem + L::kP2Off));
      int u = warp - kMmaW;
      for (; u < units; u += kMmaWarps) {
        const int s = u % L::kStages, a = u % L::kASlots, d = u % kNDS;
        const uint32_t aph = (u / L::kASlots) & 1, dph = (u / kNDS) & 1;
        // The decoders arrive on afull only after waiting on the stage's
        // copy, so acquiring afull orders the pieces' bytes before these
        // MMAs too (release/acquire chains are transitive).
        if (!mbar_wait(&afull[a], aph, err)) break;
        if (u >= kNDS && !mbar_wait(&dfree[d], dph ^ 1, err)) break;
        tc_fence_after();
        const uint32_t dcol = tbase + L::kDCol + d * TOK;
        const uint32_t acol = tbase + L::kACol + a * 32;
        // descriptor start addresses advance in 16-byte units: a stage is
        // kPB bytes, a K = 32 step 32 bytes inside the swizzle atom
        const uint64_t b1 = desc1 + static_cast<uint64_t>((s * L::kPB) >> 4);
        const uint64_t b2 = desc2 + static_cast<uint64_t>((s * L::kPB) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f8f6f4_ts(dcol, acol + kk * 8, b1 + 2 * kk, idesc, kk != 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_f8f6f4_ts(dcol, acol + kk * 8, b2 + 2 * kk, idesc, true);
        mma_commit(&empty[s]);  // one commit per group: the fold waits on it too
      }
      // This issuer's MMAs are complete before the CTA tears down.  (Its own
      // barrier: a stage's barrier may have moved on by two phases when the
      // other issuer's later group reused the stage.)
      mma_commit(&mfin[warp - kMmaW]);
      mbar_wait(&mfin[warp - kMmaW], 0, err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ fold
    const int fq = warp & 3;                // TMEM lane quarter
    const int hc = (warp - kDecW) >> 2;     // token block of the tile
    const int r = fq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(fq * 32) << 16;
    float acc[L::kFC];
#pragma unroll
    for (int j = 0; j < L::kFC; ++j) acc[j] = 0.f;
    // group u's sums are in D slot u % kNDS once empty[u % kStages] has
    // completed.  Parity: that barrier's next phase needs the MMAs of group
    // u + kStages, which wait for this warp's fold of group u + kStages - kNDS
    // (later than u, as kStages > kNDS).
    int d = 0, s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int m = 0; m < nitems && ok; ++m) {
      const Item itm = item_of(m);
      const int rb = itm.tile / TB, tb = itm.tile % TB;
      const int n = rb * kRowsS + r;
      const uint16_t* srow = scales + static_cast<size_t>(n < N ? n : 0) * G;
      float snext = n < N ? __half2float(__ushort_as_half(srow[itm.g0])) : 0.f;
      for (int g = itm.g0; g < itm.g1; ++g) {
        const float sg = 8.0f * snext;  // D holds acc / 8
        if (g + 1 < itm.g1) snext = n < N ? __half2float(__ushort_as_half(srow[g + 1])) : 0.f;
        if (!__all_sync(0xffffffffu, mbar_wait(&empty[s], ph, err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // kCh columns at a time: load, wait, fold (the slot is released
        // after the last load has completed)
        constexpr int kCh = L::kFC >= 32 ? 32 : L::kFC;
        const uint32_t col = tbase + lane_off + L::kDCol + d * TOK + hc * L::kFC;
#pragma unroll
        for (int c = 0; c < L::kFC / kCh; ++c) {
          uint32_t dv[kCh];
          if constexpr (kCh == 32)
            tmem_ld32(col + 32 * c, dv);
          else
            tmem_ld16(col + 16 * c, dv);
          tmem_wait_ld();
          if (c == L::kFC / kCh - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&dfree[d]);
          }
#pragma unroll
          for (int j = 0; j < kCh; ++j)
            acc[kCh * c + j] = fmaf(sg, __uint_as_float(dv[j]), acc[kCh * c + j]);
        }
        if (++d == kNDS) d = 0;
        if (++s == L::kStages) {
          s = 0;
          ph ^= 1;
        }
      }
      if (!ok) break;
      // end of the tile: y[t][n] = xs[t] * acc
      const int xb = m & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&xsfull[xb], (m >> 1) & 1, err))) break;
      const float* xst = xs_tile + xb * TOK + hc * L::kFC;
      const int t0 = tb * TOK + hc * L::kFC;
      bool store = true;
      if (itm.chunk >= 0) {
        // Chunked tile: publish this warp's partial sums (token-major, one
        // 32-row column per token), take the (tile, warp) ticket; the last
        // chunk to arrive adds every chunk's sums in chunk order.
        const int fw = warp - kDecW;
        const int ct = itm.tile - nfull;  // the tile's index among the chunked ones
        auto part = [&](int c) {
          return partials + (static_cast<size_t>(ct * chunks + c) * kFoldW + fw) * (L::kFC * 32);
        };
        float* mine = part(itm.chunk);
#pragma unroll
        for (int j = 0; j < L::kFC; ++j) mine[j * 32 + lane] = acc[j];
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0)
          last = atomic_add_acq_rel_gpu(&tickets[ct * kFoldW + fw], 1) == chunks - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        __syncwarp();
        if (last) {
          // every chunk's sums from the workspace (this one's too), added to
          // 0 in chunk order into acc (published above, so free), then
          // scaled and stored as a whole tile's: one chunk's loads in flight
          // at a time
#pragma unroll
          for (int j = 0; j < L::kFC; ++j) acc[j] = 0.f;
          for (int c = 0; c < chunks; ++c) {
            const float* pc = part(c) + lane;
#pragma unroll
            for (int j = 0; j < L::kFC; ++j) acc[j] += __ldcg(pc + j * 32);
          }
          if (lane == 0) tickets[ct * kFoldW + fw] = 0;  // every chunk has taken it
        }
        store = last != 0;
      }
      if (!store) {
#pragma unroll
        for (int j = 0; j < L::kFC; ++j) acc[j] = 0.f;
      } else {
        // plain stores: a staged block and a TMA store per warp measured
        // slower, and the stage ring gets the shared memory instead
#pragma unroll
        for (int j = 0; j < L::kFC; ++j) {
          const int t = t0 + j;
          if (n < N && t < T) y[static_cast<size_t>(t) * N + n] = xst[j] * acc[j];
          acc[j] = 0.f;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&xsfree[xb]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaW) tmem_dealloc(tbase, 512);
}

}  // namespace

// The s8 kernel's instances: (token tile, stages).
#define TERN_S8_INSTANCES(X) X(kS8SmallTileT, 12) X(kS8TileT, 4) X(kS8TileT, kS8DeepStages)

cudaError_t s8_set_attributes() {
  cudaError_t e = cudaSuccess;
#define TERN_S8_ATTR(TOK, NST)                                                             \
  if (e == cudaSuccess)                                                                    \
    e = cudaFuncSetAttribute(s8tc_kernel<TOK, NST>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             SL<TOK, NST>::kAlloc);
  TERN_S8_INSTANCES(TERN_S8_ATTR)
#undef TERN_S8_ATTR
  return e;
}

int s8_token_tile(int T) { return T <= kS8SmallTileT ? kS8SmallTileT : kS8TileT; }

int s8_stages(int T, int K, size_t l2_bytes) {
  if (s8_token_tile(T) == kS8SmallTileT) return 12;
  return 2 * static_cast<size_t>(T) * K > l2_bytes / 2 ? kS8DeepStages : 4;
}

cudaError_t launch_s8(const CUtensorMap* tmW, const CUtensorMap* tmP1, const CUtensorMap* tmP2,
                      const uint16_t* scales, const float* x_scale, float* y, int T, int K, int N,
                      int* tickets, float* partials, int num_sms, size_t l2_bytes, int* err,
                      cudaStream_t stream) {
  const int tok = s8_token_tile(T), nst = s8_stages(T, K, l2_bytes);
  const int tiles = ((N + kRowsS - 1) / kRowsS) * ((T + tok - 1) / tok);
  const TileSplit sp = tile_split(tiles, K / 128, num_sms);
  cudaLaunchAttribute attr[1];
#define TERN_S8_LAUNCH(TOK, NST)                                                            \
  if (tok == TOK && nst == NST) {                                                           \
    const cudaLaunchConfig_t cfg =                                                          \
        pdl_launch_config(attr, dim3(sp.P), dim3(kThreadsS), SL<TOK, NST>::kAlloc, stream); \
    return cudaLaunchKernelEx(&cfg, s8tc_kernel<TOK, NST>, *tmW, *tmP1, *tmP2, scales,      \
                              x_scale, y, T, K, N, sp.nfull, sp.chunks, tickets, partials,  \
                              err);                                                         \
  }
  TERN_S8_INSTANCES(TERN_S8_LAUNCH)
#undef TERN_S8_LAUNCH
  return cudaErrorInvalidConfiguration;
}

}  // namespace tern
