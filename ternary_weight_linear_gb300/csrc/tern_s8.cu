// s8 rung (T >= 17): int8 per-token activations x ternary weights, exact
// integer accumulation per 128-wide group, fp32 output
//     y[t][n] = xs[t] * sum_g s[n][g] * acc[t][n][g],
//     acc[t][n][g] = sum_{k in g} q[t][k] w[n][k].
//
// On 5th-generation tensor cores.  sm_103a has no integer tcgen05 MMA, so the
// integers travel as exact fp8 e4m3 values:
//   * w / 8 in {-1/8, 0, 1/8} (the packed code decodes to it with a shift and
//     an AND, as in the small-T rungs);
//   * q = p1 + p2 with p1 = 16 floor((q + 8) / 16) and p2 = q - p1, both
//     exact in e4m3 (prepared by the pieces quantiser);
// and the two pieces are fed as two halves of the contraction into the same
// fp32 accumulator, which then holds exactly acc / 8 (|acc| <= 127 * 128, far
// inside fp32's exact integer range; every product is a multiple of 1/8).
//
// Tile: 128 weight rows (MMA M, TMEM lanes) x 128 tokens (MMA N).  Per
// 128-wide group a stage holds the packed weights (TMA, 128 rows x 32 B) and
// the two piece blocks (TMA, 128 tokens x 128 B each, 128-byte swizzle, the
// canonical K-major SW128 layout of the MMA's B operand).  Warp roles:
//   warps 0-3   decode the group's weights into an A slot in TMEM
//               (tcgen05.st, one row per thread);
//   warp 13     issues 8 MMAs per group (4 per piece, K = 32 each) into a D
//               slot (128 columns), committing to the slot's barriers;
//   warps 4-11  fold: read the D slot (each warp 32 rows x 64 tokens), add
//               8 s[n][g] * D into register accumulators, and at the end of
//               the tile write y = xs[t] * acc;
//   warp 12     producer (TMA) and the tile's x_scale block.
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
constexpr int kTokS = 128;    // tokens per tile
constexpr int kStagesS = 4;   // stage ring
constexpr int kNAS = 4;       // A slots (32 TMEM columns = one group of e4m3)
constexpr int kNDS = 2;       // D slots (128 columns)
constexpr int kDecW = 4;
constexpr int kFoldW = 8;
constexpr int kProdW = kDecW + kFoldW;
constexpr int kMmaW = kProdW + 1;
constexpr int kThreadsS = (kMmaW + 1) * 32;

struct SL {
  static constexpr int kPB = kTokS * 128;   // one piece block of a group (16 KB)
  static constexpr int kWB = kRowsS * 32;   // packed weights of a group (4 KB)
  static constexpr int kP1Off = 0;          // 1024-aligned (128-byte swizzle atoms)
  static constexpr int kP2Off = kP1Off + kStagesS * kPB;
  static constexpr int kWOff = kP2Off + kStagesS * kPB;
  static constexpr int kXsOff = kWOff + kStagesS * kWB;  // x_scale of 2 tiles
  static constexpr int kBarOff = kXsOff + 2 * kTokS * 4;
  static constexpr int kNumBars = 2 * kStagesS + 2 * kNAS + 2 * kNDS + 4;
  static constexpr int kTmemSlot = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kTmemSlot + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kACol = 0;
  static constexpr uint32_t kDCol = kNAS * 32;
  static_assert(kDCol + kNDS * kTokS <= 512, "TMEM budget");
  static_assert(kAlloc <= 227 * 1024, "shared memory");
};

// Shared-memory descriptor of a K-major operand in the 128-byte swizzle
// layout: rows of 128 bytes, 8-row atoms 1024 bytes apart (stride byte
// offset), layout type 2 (SWIZZLE_128B) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

__global__ void __launch_bounds__(kThreadsS, 1)
    s8tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmP1,
                const __grid_constant__ CUtensorMap tmP2, const uint16_t* __restrict__ scales,
                const float* __restrict__ x_scale, float* __restrict__ y, int T, int K, int N,
                int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SL::kBarOff);
  uint64_t* empty = full + kStagesS;   // weights decoded and pieces read by the MMAs
  uint64_t* afull = empty + kStagesS;  // A slot written
  uint64_t* afree = afull + kNAS;      // MMAs reading the A slot done
  uint64_t* mdone = afree + kNAS;      // MMAs writing the D slot done
  uint64_t* dfree = mdone + kNDS;      // D slot read back
  uint64_t* xsfull = dfree + kNDS;     // [2] tile's x_scale landed
  uint64_t* xsfree = xsfull + 2;       // [2] ... and used
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SL::kTmemSlot);
  const float* xs_tile = reinterpret_cast<const float*>(smem + SL::kXsOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = K >> 7;
  const int RB = (N + kRowsS - 1) / kRowsS;
  const int TB = (T + kTokS - 1) / kTokS;
  const int tiles = RB * TB;
  const int ntiles = blockIdx.x < tiles ? (tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int units = ntiles * G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecW + 1);
    }
    for (int a = 0; a < kNAS; ++a) {
      mbar_init(&afull[a], kDecW);
      mbar_init(&afree[a], 1);
    }
    for (int d = 0; d < kNDS; ++d) {
      mbar_init(&mdone[d], 1);
      mbar_init(&dfree[d], kFoldW);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&xsfull[b], 1);
      mbar_init(&xsfree[b], kFoldW);
    }
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

  if (warp == kProdW) {
    // ------------------------------------------------------------ producer
    int u = 0;
    bool ok = true;
    for (int m = 0; m < ntiles && ok; ++m) {
      const int tile = blockIdx.x + m * gridDim.x;
      const int rb = tile / TB, tb = tile % TB;
      // this tile's x_scale block (padded to whole 16-byte chunks: the
      // workspace rounds the x_scale array up to 256 bytes)
      const int xb = m & 1;
      if (m >= 2 && !__all_sync(0xffffffffu, mbar_wait(&xsfree[xb], ((m >> 1) & 1) ^ 1, err))) break;
      if (lane == 0) {
        const int cnt = T - tb * kTokS < kTokS ? T - tb * kTokS : kTokS;
        const uint32_t bytes = static_cast<uint32_t>((cnt * 4 + 15) & ~15);
        mbar_arrive_expect_tx(&xsfull[xb], bytes);
        bulk_load(smem + SL::kXsOff + xb * kTokS * 4, x_scale + tb * kTokS, bytes, &xsfull[xb]);
      }
      for (int g = 0; g < G; ++g, ++u) {
        const int s = u % kStagesS;
        if (u >= kStagesS &&
            !__all_sync(0xffffffffu, mbar_wait(&empty[s], ((u / kStagesS) & 1) ^ 1, err))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[s], SL::kWB + 2 * SL::kPB);
          tma_load_2d(smem + SL::kWOff + s * SL::kWB, &tmW, g * 32, rb * kRowsS, &full[s]);
          tma_load_2d(smem + SL::kP1Off + s * SL::kPB, &tmP1, g * 128, tb * kTokS, &full[s]);
          tma_load_2d(smem + SL::kP2Off + s * SL::kPB, &tmP2, g * 128, tb * kTokS, &full[s]);
        }
      }
    }
    // no copy of this CTA may still be in flight when it exits
    for (int d = (u > kStagesS ? u - kStagesS : 0); d < u; ++d)
      if (!mbar_wait(&full[d % kStagesS], (d / kStagesS) & 1, err)) break;
    for (int m = (ntiles > 2 ? ntiles - 2 : 0); m < ntiles; ++m)
      if (!mbar_wait(&xsfull[m & 1], (m >> 1) & 1, err)) break;
  } else if (warp < kDecW) {
    // ------------------------------------------------------------ decode
    const int r = warp * 32 + lane;  // row of the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    for (int u = 0; u < units; ++u) {
      const int s = u % kStagesS;
      const int a = u % kNAS;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (u / kStagesS) & 1, err))) break;
      if (u >= kNAS && !__all_sync(0xffffffffu, mbar_wait(&afree[a], ((u / kNAS) & 1) ^ 1, err)))
        break;
      tc_fence_after();
      const uint8_t* wrow = smem + SL::kWOff + s * SL::kWB + r * 32;
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
      tmem_st32(tbase + lane_off + SL::kACol + a * 32, av);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&afull[a]);
        mbar_arrive(&empty[s]);
      }
    }
  } else if (warp == kMmaW) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = elect_one();
    constexpr uint32_t idesc = idesc_e4m3_f32(kRowsS, kTokS);
    const uint32_t p1base = smem_addr(smem + SL::kP1Off);
    const uint32_t p2base = smem_addr(smem + SL::kP2Off);
    int u = 0;
    for (; u < units; ++u) {
      const int s = u % kStagesS;
      const int a = u % kNAS;
      const int d = u % kNDS;
      // the pieces landed (the decode warps saw it too; waiting here orders
      // the tensor core's reads after the copy for this warp as well)
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (u / kStagesS) & 1, err))) break;
      if (!__all_sync(0xffffffffu, mbar_wait(&afull[a], (u / kNAS) & 1, err))) break;
      if (u >= kNDS && !__all_sync(0xffffffffu, mbar_wait(&dfree[d], ((u / kNDS) & 1) ^ 1, err)))
        break;
      tc_fence_after();
      if (leader) {
        const uint32_t dcol = tbase + SL::kDCol + d * kTokS;
        const uint32_t acol = tbase + SL::kACol + a * 32;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          const uint32_t bb = (p ? p2base : p1base) + s * SL::kPB;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8f6f4_ts(dcol, acol + kk * 8, smem_desc_sw128(bb + kk * 32), idesc,
                          (p | kk) != 0);
        }
        mma_commit(&empty[s]);
        mma_commit(&afree[a]);
        mma_commit(&mdone[d]);
      }
      __syncwarp();
    }
    if (u > 0) mbar_wait(&mdone[(u - 1) % kNDS], ((u - 1) / kNDS) & 1, err);
  } else {
    // ------------------------------------------------------------ fold
    const int fq = warp & 3;                // TMEM lane quarter
    const int hc = (warp - kDecW) >> 2;     // token half of the tile
    const int r = fq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(fq * 32) << 16;
    float acc[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) acc[j] = 0.f;
    int u = 0;
    bool ok = true;
    for (int m = 0; m < ntiles && ok; ++m) {
      const int tile = blockIdx.x + m * gridDim.x;
      const int rb = tile / TB, tb = tile % TB;
      const int n = rb * kRowsS + r;
      const uint16_t* srow = scales + static_cast<size_t>(n < N ? n : 0) * G;
      float snext = n < N ? __half2float(__ushort_as_half(srow[0])) : 0.f;
      for (int g = 0; g < G; ++g, ++u) {
        const int d = u % kNDS;
        const float sg = 8.0f * snext;  // D holds acc / 8
        if (g + 1 < G) snext = n < N ? __half2float(__ushort_as_half(srow[g + 1])) : 0.f;
        if (!__all_sync(0xffffffffu, mbar_wait(&mdone[d], (u / kNDS) & 1, err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t dv[64];
        const uint32_t col = tbase + lane_off + SL::kDCol + d * kTokS + hc * 64;
        tmem_ld32(col, dv);
        tmem_ld32(col + 32, dv + 32);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dfree[d]);
#pragma unroll
        for (int j = 0; j < 64; ++j) acc[j] = fmaf(sg, __uint_as_float(dv[j]), acc[j]);
      }
      if (!ok) break;
      // end of the tile: y[t][n] = xs[t] * acc
      const int xb = m & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&xsfull[xb], (m >> 1) & 1, err))) break;
      const float* xst = xs_tile + xb * kTokS + hc * 64;
      const int t0 = tb * kTokS + hc * 64;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const int t = t0 + j;
        if (n < N && t < T) y[static_cast<size_t>(t) * N + n] = xst[j] * acc[j];
        acc[j] = 0.f;
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

size_t s8_smem_bytes() { return SL::kAlloc; }

cudaError_t s8_set_attributes() {
  return cudaFuncSetAttribute(s8tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              SL::kAlloc);
}

cudaError_t launch_s8(const CUtensorMap* tmW, const CUtensorMap* tmP1, const CUtensorMap* tmP2,
                      const uint16_t* scales, const float* x_scale, float* y, int T, int K, int N,
                      int num_sms, int* err, cudaStream_t stream) {
  const long long tiles = static_cast<long long>((N + kRowsS - 1) / kRowsS) *
                          ((T + kTokS - 1) / kTokS);
  const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
  s8tc_kernel<<<grid, kThreadsS, SL::kAlloc, stream>>>(*tmW, *tmP1, *tmP2, scales, x_scale, y, T,
                                                       K, N, err);
  return cudaGetLastError();
}

}  // namespace tern
