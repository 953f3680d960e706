// bf16 prefill rung: bf16 activations x ternary weights on the tensor cores
// with no activation quantisation,
//     y[t][n] = sum_g s[n][g] * sum_{k in g} w[n][k] * x[t][k]   (fp32 out).
//
// tcgen05.mma kind::f16 with bf16 A and B and an fp32 accumulator: every
// product w * x (w in {-1, 0, +1}) is exact, and the only roundings are the
// fp32 sums of the accumulator (one 128-wide group per accumulation) and of
// the fold.  Against the s8 rung it trades the int8 rounding of every
// activation for twice the A-operand bytes per weight and a longer decode.
//
// Operands:
//   * A (weights, TMEM): each packed word (k = 16 j .. 16 j + 15) decodes to
//     eight 32-bit columns, column 8 j + o holding bf16 w[16 j + o] (low
//     half) and w[16 j + o + 8] (high half): the two weights of a column are
//     16 bits apart in the packed word, so one shift, two masks and one
//     multiply-add make a column (decode_bf16_pair).  So the MMA's K order
//     within each 16-wide block is 16 j + p <-> k = 16 j + p / 2 + 8 (p % 2).
//   * B (activations, shared memory): x in that same K order, written once
//     per call by interleave_kernel into the workspace ([T][K] bf16), copied
//     per group as two 64-k x 128-token boxes (128-byte swizzle, the
//     canonical K-major SW128 layout).
//
// Tile: 128 weight rows (MMA M, TMEM lanes) x 128 tokens (MMA N); per
// 128-wide group 8 MMAs of K = 16.  Warp roles as in the s8 rung:
//   warps 0-3   decode the group's weights into an A slot (64 columns);
//   warps 4-11  fold: read the D slot (32 rows x 64 tokens each), add
//               s[n][g] * D into register accumulators, and at the end of the
//               tile stage y in shared memory for a TMA store;
//   warp 12     producer (TMA);
//   warps 13-14 issue the MMAs of alternate groups (one thread each).
// Persistent CTAs walk the (row block, token tile) tiles with the token tile
// fastest, so CTAs that run at the same time share the row block's weights in
// L2.
//
// This is the "wide_mma" bf16 prefill rung of the "ninfer-perf-tuning" skill
// page (section 2 rung map; section 6 gives its cost on Ada), which the pages
// price against the s8 rung; here on tcgen05.
#include "tern_device.cuh"
#include "tern_internal.h"

namespace tern {
namespace {

constexpr int kRowsB = 128;   // weight rows per tile
constexpr int kTokB = 128;    // tokens per tile
constexpr int kStagesB = 4;   // stage ring (each stage has an A slot of 64 TMEM columns)
constexpr int kNDB = 2;       // D slots (128 columns)
constexpr int kDecWB = 4;
constexpr int kFoldWB = 8;
constexpr int kFCB = kTokB * 4 / kFoldWB;  // tokens (D columns) per fold warp
static_assert(kFCB == kS8YBoxT, "the y tensor map's box is shared with the s8 rung");
constexpr int kProdWB = kDecWB + kFoldWB;
constexpr int kMmaWB = kProdWB + 1;
// Two issuers on alternate groups (the issuing thread runs in step with the
// tensor pipe, so its waits and commits would leave the pipe idle); as in the
// s8 rung, an issuer's D-slot parity check needs kMmaWarpsB <= kNDB.
constexpr int kMmaWarpsB = 2;
constexpr int kThreadsB = (kMmaWB + kMmaWarpsB) * 32;
static_assert(kMmaWarpsB <= kNDB, "issuers may outrun the accumulator ring's parity check");

struct BL {
  static constexpr int kXB = kTokB * 128;   // one x box: 64 k x 128 tokens of bf16 (16 KB)
  static constexpr int kWB = kRowsB * 32;   // packed weights of a group (4 KB)
  static constexpr int kX0Off = 0;          // 1024-aligned (128-byte swizzle atoms)
  static constexpr int kX1Off = kX0Off + kStagesB * kXB;
  static constexpr int kWOff = kX1Off + kStagesB * kXB;
  static constexpr int kYB = kFCB * 32 * 4;  // one fold warp's output block
  static constexpr int kYOff = kWOff + kStagesB * kWB;
  static constexpr int kBarOff = kYOff + kFoldWB * kYB;
  static constexpr int kNumBars = 3 * kStagesB + kNDB + kMmaWarpsB;
  static constexpr int kTmemSlot = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kTmemSlot + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kACol = 0;
  static constexpr uint32_t kDCol = kStagesB * 64;
  static_assert(kDCol + kNDB * kTokB <= 512, "TMEM budget");
  static_assert(kAlloc <= 227 * 1024, "shared memory");
};

// Instruction descriptor for kind::f16 with bf16 A and B, fp32 accumulator,
// both operands K-major: D type f32 (bits 4-5), A and B type bf16 (bits 7-9,
// 10-12), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16_ts(uint32_t d_taddr, uint32_t a_taddr, uint64_t b_desc,
                                           uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_taddr),
      "r"(a_taddr), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1 : 0)
      : "memory");
}

__device__ __forceinline__ uint64_t smem_desc_sw128_b(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Column O (0..7) of packed word w: bf16 of the weights k = 16 j + O (low
// half) and 16 j + O + 8 (high half), +1 -> 0x3F80, -1 -> 0xBF80, 0 -> 0 (the
// invalid pair decodes to 0x8000, a zero).  The low weight sits in byte O / 4
// at nonzero bit P = {0, 1, 4, 5}[O % 4] (sign two above), the high one in
// byte O / 4 + 2: 16 bits higher.
template <int O>
__device__ __forceinline__ uint32_t decode_bf16_pair(uint32_t w) {
  constexpr int i = O % 4;
  constexpr int p = 8 * (O / 4) + (i < 2 ? i : i + 2);
  const uint32_t t = w >> p;
  return (t & 0x00010001u) * 0x3F80u + ((t << 13) & 0x80008000u);
}

__global__ void __launch_bounds__(kThreadsB, 1)
    bf16tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                  const __grid_constant__ CUtensorMap tmY, const uint16_t* __restrict__ scales,
                  float* __restrict__ y, int T, int K, int N, int y_tma, int nfull, int chunks,
                  int* __restrict__ tickets, float* __restrict__ partials, int* err) {
  grid_dependents_launch();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + BL::kBarOff);
  // empty[s]: the stage's weights are decoded and its group's MMAs are
  // complete (its A slot and x boxes have been read, and its D slot holds the
  // group's sums)
  uint64_t* empty = full + kStagesB;
  uint64_t* afull = empty + kStagesB;  // A slot written
  uint64_t* dfree = afull + kStagesB;  // D slot read back
  uint64_t* mfin = dfree + kNDB;       // [issuer] all of that issuer's MMAs complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + BL::kTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = K >> 7;
  const int RB = (N + kRowsB - 1) / kRowsB;
  const int TB = (T + kTokB - 1) / kTokB;
  const int tiles = RB * TB;
  // Work items as in the s8 rung (tile_split): the first nfull tiles whole,
  // then each remaining tile as `chunks` ranges of its groups, whose partial
  // sums the last chunk to finish adds in chunk order.
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
    for (int s = 0; s < kStagesB; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecWB + 1);
      mbar_init(&afull[s], kDecWB);
    }
    for (int d = 0; d < kNDB; ++d) mbar_init(&dfree[d], kFoldWB);
    for (int w = 0; w < kMmaWarpsB; ++w) mbar_init(&mfin[w], 1);
    fence_mbar_init();
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmX);
    if (y_tma) prefetch_tensormap(&tmY);
  }
  if (warp == kMmaWB) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // the set-up above overlaps the previous kernel; the reordered x, y and the
  // workspace belong to it until it has finished
  grid_dependency_wait();

  if (warp == kProdWB) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int u = 0, s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int m = 0; m < nitems && ok; ++m) {
        const Item itm = item_of(m);
        const int rb = itm.tile / TB, tb = itm.tile % TB;
        for (int g = itm.g0; g < itm.g1; ++g, ++u) {
          if (u >= kStagesB && !mbar_wait(&empty[s], ph ^ 1, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], BL::kWB + 2 * BL::kXB);
          tma_load_2d(smem + BL::kWOff + s * BL::kWB, &tmW, g * 32, rb * kRowsB, &full[s]);
          // x boxes in bytes: k 128 g .. 128 g + 63, then + 64 .. + 127
          tma_load_2d(smem + BL::kX0Off + s * BL::kXB, &tmX, g * 256, tb * kTokB, &full[s]);
          tma_load_2d(smem + BL::kX1Off + s * BL::kXB, &tmX, g * 256 + 128, tb * kTokB, &full[s]);
          if (++s == kStagesB) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      // no copy of this CTA may still be in flight when it exits
      for (int v = (u > kStagesB ? u - kStagesB : 0); v < u; ++v)
        if (!mbar_wait(&full[v % kStagesB], (v / kStagesB) & 1, err)) break;
    }
    __syncwarp();
  } else if (warp < kDecWB) {
    // ------------------------------------------------------------ decode
    const int r = warp * 32 + lane;  // row of the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    int s = 0;
    uint32_t ph = 0;
    for (int u = 0; u < units; ++u) {
      // the copy into stage s was issued after the MMAs that last read A
      // slot s completed (the producer waited on empty[s]), so its landing
      // also frees the slot
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, err))) break;
      tc_fence_after();
      const uint8_t* wrow = smem + BL::kWOff + s * BL::kWB + r * 32;
      const uint4 c0 = lds_v4(wrow);
      const uint4 c1 = lds_v4(wrow + 16);
      const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      const uint32_t acol = tbase + lane_off + BL::kACol + s * 64;
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {  // packed words 4 hlf .. 4 hlf + 3: columns 32 hlf ..
        uint32_t av[32];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const uint32_t wj = w[4 * hlf + jj];
          av[8 * jj + 0] = decode_bf16_pair<0>(wj);
          av[8 * jj + 1] = decode_bf16_pair<1>(wj);
          av[8 * jj + 2] = decode_bf16_pair<2>(wj);
          av[8 * jj + 3] = decode_bf16_pair<3>(wj);
          av[8 * jj + 4] = decode_bf16_pair<4>(wj);
          av[8 * jj + 5] = decode_bf16_pair<5>(wj);
          av[8 * jj + 6] = decode_bf16_pair<6>(wj);
          av[8 * jj + 7] = decode_bf16_pair<7>(wj);
        }
        tmem_st32(acol + 32 * hlf, av);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&afull[s]);
        mbar_arrive(&empty[s]);
      }
      if (++s == kStagesB) {
        s = 0;
        ph ^= 1;
      }
    }
  } else if (warp >= kMmaWB) {
    // ------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kRowsB, kTokB);
      const uint64_t desc0 = smem_desc_sw128_b(smem_addr(smem + BL::kX0Off));
      const uint64_t desc1 = smem_desc_sw128_b(smem_addr(smem + BL::kX1Off));
      int u = warp - kMmaWB;
      for (; u < units; u += kMmaWarpsB) {
        const int s = u % kStagesB, d = u % kNDB;
        const uint32_t ph = (u / kStagesB) & 1, dph = (u / kNDB) & 1;
        // The decoders arrive on afull only after waiting on the stage's
        // copy, so acquiring afull orders the x boxes' bytes before these
        // MMAs too (release/acquire chains are transitive).
        if (!mbar_wait(&afull[s], ph, err)) break;
        if (u >= kNDB && !mbar_wait(&dfree[d], dph ^ 1, err)) break;
        tc_fence_after();
        const uint32_t dcol = tbase + BL::kDCol + d * kTokB;
        const uint32_t acol = tbase + BL::kACol + s * 64;
        // a K = 16 step: 32 bytes of a 128-byte swizzled row (2 descriptor
        // units), 8 A columns
        const uint64_t b0 = desc0 + static_cast<uint64_t>((s * BL::kXB) >> 4);
        const uint64_t b1 = desc1 + static_cast<uint64_t>((s * BL::kXB) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_f16_ts(dcol, acol + kk * 8, b0 + 2 * kk, idesc, kk != 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_f16_ts(dcol, acol + 32 + kk * 8, b1 + 2 * kk, idesc, true);
        mma_commit(&empty[s]);  // one commit per group: the fold waits on it too
      }
      mma_commit(&mfin[warp - kMmaWB]);
      mbar_wait(&mfin[warp - kMmaWB], 0, err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ fold
    const int fq = warp & 3;              // TMEM lane quarter
    const int hc = (warp - kDecWB) >> 2;  // token block of the tile
    const int r = fq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(fq * 32) << 16;
    float acc[kFCB];
#pragma unroll
    for (int j = 0; j < kFCB; ++j) acc[j] = 0.f;
    // group u's sums are in D slot u % kNDB once empty[u % kStagesB] has
    // completed.  Parity: that barrier's next phase needs the MMAs of group
    // u + kStagesB, which wait for this warp's fold of group
    // u + kStagesB - kNDB (later than u).
    static_assert(kStagesB > kNDB, "the fold's parity wait on the stage ring");
    int d = 0, s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int m = 0; m < nitems && ok; ++m) {
      const Item itm = item_of(m);
      const int rb = itm.tile / TB, tb = itm.tile % TB;
      const int n = rb * kRowsB + r;
      const uint16_t* srow = scales + static_cast<size_t>(n < N ? n : 0) * G;
      float snext = n < N ? __half2float(__ushort_as_half(srow[itm.g0])) : 0.f;
      for (int g = itm.g0; g < itm.g1; ++g) {
        const float sg = snext;
        if (g + 1 < itm.g1) snext = n < N ? __half2float(__ushort_as_half(srow[g + 1])) : 0.f;
        if (!__all_sync(0xffffffffu, mbar_wait(&empty[s], ph, err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t col = tbase + lane_off + BL::kDCol + d * kTokB + hc * kFCB;
#pragma unroll
        for (int c = 0; c < kFCB / 32; ++c) {
          uint32_t dv[32];
          tmem_ld32(col + 32 * c, dv);
          tmem_wait_ld();
          if (c == kFCB / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&dfree[d]);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j)
            acc[32 * c + j] = fmaf(sg, __uint_as_float(dv[j]), acc[32 * c + j]);
        }
        if (++d == kNDB) d = 0;
        if (++s == kStagesB) {
          s = 0;
          ph ^= 1;
        }
      }
      if (!ok) break;
      const int t0 = tb * kTokB + hc * kFCB;
      bool store = true;
      if (itm.chunk >= 0) {
        // chunked tile: publish, take the (tile, warp) ticket, the last adds
        // every chunk's sums to 0 in chunk order (as in the s8 rung)
        const int fw = warp - kDecWB;
        const int ct = itm.tile - nfull;
        auto part = [&](int c) {
          return partials + (static_cast<size_t>(ct * chunks + c) * kFoldWB + fw) * (kFCB * 32);
        };
        float* mine = part(itm.chunk);
#pragma unroll
        for (int j = 0; j < kFCB; ++j) mine[j * 32 + lane] = acc[j];
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0)
          last = atomic_add_acq_rel_gpu(&tickets[ct * kFoldWB + fw], 1) == chunks - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        __syncwarp();
        if (last) {
#pragma unroll
          for (int j = 0; j < kFCB; ++j) acc[j] = 0.f;
          for (int c = 0; c < chunks; ++c) {
            const float* pc = part(c) + lane;
#pragma unroll
            for (int j = 0; j < kFCB; ++j) acc[j] += __ldcg(pc + j * 32);
          }
          if (lane == 0) tickets[ct * kFoldWB + fw] = 0;  // every chunk has taken it
        }
        store = last != 0;
      }
      if (!store) {
#pragma unroll
        for (int j = 0; j < kFCB; ++j) acc[j] = 0.f;
      } else if (y_tma) {
        // stage the warp's kFCB x 32 block and store it asynchronously: the
        // next tile's groups overlap the write-back
        float* stg = reinterpret_cast<float*>(smem + BL::kYOff + (warp - kDecWB) * BL::kYB);
        if (lane == 0) bulk_wait_group_read0();  // the warp's previous block was read out
        __syncwarp();
#pragma unroll
        for (int j = 0; j < kFCB; ++j) {
          stg[j * 32 + lane] = acc[j];
          acc[j] = 0.f;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && rb * kRowsB + fq * 32 < N && t0 < T) {
          tma_store_2d(&tmY, stg, rb * kRowsB + fq * 32, t0);
          bulk_commit_group();
        }
      } else {
#pragma unroll
        for (int j = 0; j < kFCB; ++j) {
          const int t = t0 + j;
          if (n < N && t < T) y[static_cast<size_t>(t) * N + n] = acc[j];
          acc[j] = 0.f;
        }
      }
      __syncwarp();
    }
    if (lane == 0) bulk_wait_group0();  // output blocks written before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWB) tmem_dealloc(tbase, 512);
}

// x [T][K] -> xp [T][K] in the MMA's K order: within every 16-wide block,
// position 2 o + h holds k = o + 8 h (o = 0..7, h = 0, 1).  One thread per
// 16-wide block: byte permutes of two 16-byte loads.
__global__ void __launch_bounds__(256) interleave_kernel(const uint16_t* __restrict__ x,
                                                         uint16_t* __restrict__ xp,
                                                         long long blocks) {
  grid_dependents_launch();
  grid_dependency_wait();  // x and the output buffer come from earlier work
  for (long long b = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; b < blocks;
       b += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4 lo = ldg_nc_v4(x + 16 * b);      // k 0..7
    const uint4 hi = ldg_nc_v4(x + 16 * b + 8);  // k 8..15
    const uint32_t a[4] = {lo.x, lo.y, lo.z, lo.w};
    const uint32_t c[4] = {hi.x, hi.y, hi.z, hi.w};
    uint32_t o[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      o[2 * e] = __byte_perm(a[e], c[e], 0x5410);      // k = 2e, 2e + 8
      o[2 * e + 1] = __byte_perm(a[e], c[e], 0x7632);  // k = 2e + 1, 2e + 9
    }
    uint4* dst = reinterpret_cast<uint4*>(xp + 16 * b);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// The same with the Hadamard rotation first: one warp per (token,
// 1024-block), lane l holding elements 128 g + 4 l + i (hadamard_block_1024),
// each value scaled by 1/32 and rounded once to bf16; element 16 j + o + 8 h
// of the block is then in lane 4 j' + q with q = o / 4 + 2 h, so a lane with
// q < 2 takes its partner's values from lane + 2 and writes the 16-byte half
// of block j it owns.
__global__ void __launch_bounds__(256) interleave_rot_kernel(const uint16_t* __restrict__ x,
                                                             uint16_t* __restrict__ xp,
                                                             long long pairs) {
  grid_dependents_launch();
  grid_dependency_wait();  // x and the output buffer come from earlier work
  const int lane = threadIdx.x & 31;
  for (long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       w < pairs; w += (static_cast<long long>(gridDim.x) * blockDim.x) >> 5) {
    const uint16_t* src = x + w * kRotBlock;
    float v[32];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const uint2 raw = *reinterpret_cast<const uint2*>(src + 128 * g + 4 * lane);
      v[4 * g + 0] = __uint_as_float(raw.x << 16);
      v[4 * g + 1] = __uint_as_float(raw.x & 0xFFFF0000u);
      v[4 * g + 2] = __uint_as_float(raw.y << 16);
      v[4 * g + 3] = __uint_as_float(raw.y & 0xFFFF0000u);
    }
    hadamard_block_1024(v, lane);
    uint16_t* dst = xp + w * kRotBlock;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      uint32_t b[4], pb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        b[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v[4 * g + i] * 0.03125f));
        pb[i] = __shfl_down_sync(0xffffffffu, b[i], 2);  // lane + 2: the k + 8 partners
      }
      // lane l: elements 128 g + 16 (l / 4) + 4 (l % 4) + i; for l % 4 < 2 the
      // partner lane l + 2 holds those + 8
      if ((lane & 3) < 2) {
        const uint4 out = make_uint4(b[0] | (pb[0] << 16), b[1] | (pb[1] << 16),
                                     b[2] | (pb[2] << 16), b[3] | (pb[3] << 16));
        *reinterpret_cast<uint4*>(dst + 128 * g + 16 * (lane >> 2) + 8 * (lane & 3)) = out;
      }
    }
  }
}

}  // namespace

size_t bf16_smem_bytes() { return BL::kAlloc; }

cudaError_t bf16_set_attributes() {
  return cudaFuncSetAttribute(bf16tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              BL::kAlloc);
}

cudaError_t launch_interleave(const uint16_t* x, uint16_t* xp, int T, int K, int rotate,
                              int num_sms, cudaStream_t stream) {
  if (rotate) {
    const long long pairs = static_cast<long long>(T) * (K / kRotBlock);
    long long blocks = (pairs + 7) / 8;
    if (blocks > 4LL * num_sms) blocks = 4LL * num_sms;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg =
        pdl_launch_config(attr, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream);
    return cudaLaunchKernelEx(&cfg, interleave_rot_kernel, x, xp, pairs);
  }
  const long long n16 = static_cast<long long>(T) * (K / 16);
  long long blocks = (n16 + 255) / 256;
  if (blocks > 8LL * num_sms) blocks = 8LL * num_sms;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg =
      pdl_launch_config(attr, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream);
  return cudaLaunchKernelEx(&cfg, interleave_kernel, x, xp, n16);
}

cudaError_t launch_bf16(const CUtensorMap* tmW, const CUtensorMap* tmX, const CUtensorMap* tmY,
                        const uint16_t* scales, float* y, int T, int K, int N, int* tickets,
                        float* partials, int num_sms, int* err, cudaStream_t stream) {
  const int tiles = ((N + kRowsB - 1) / kRowsB) * ((T + kTokB - 1) / kTokB);
  const TileSplit sp = tile_split(tiles, K / 128, num_sms);
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg =
      pdl_launch_config(attr, dim3(sp.P), dim3(kThreadsB), BL::kAlloc, stream);
  return cudaLaunchKernelEx(&cfg, bf16tc_kernel, *tmW, *tmX, tmY ? *tmY : *tmW, scales, y, T, K,
                            N, tmY ? 1 : 0, sp.nfull, sp.chunks, tickets, partials, err);
}

}  // namespace tern
