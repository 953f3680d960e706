// Small-T bf16 rungs: T = 1 ("gemv"), T = 2..8 ("small_t"), T = 9..16
// ("small_t_tiled").
//
// y[t][n] = sum_g s[n][g] * sum_{k in g} w[n][k] * x[t][k], fp32 accumulation.
//
// The work is a stream of 2-bit weights; the kernel is built to keep HBM busy:
//  * Persistent grid.  The (row block of 128 rows) x (k stage of 512) units
//    are split into equal contiguous ranges, one per CTA, so every SM streams
//    the same number of weight bytes whatever N and K are.  A row block split
//    between two CTAs is finished with fp32 atomics into a zeroed y.
//  * One producer warp per CTA: lane 0 issues one 2D TMA box (128 rows x 128
//    bytes, 128-byte swizzle) per stage into a 4-deep shared-memory ring
//    tracked by mbarriers; the other lanes stage that stage's fp16 scales and
//    re-order the stage's activations into mma B-fragment order.
//  * Four consumer warps, 32 rows each (two 16-row mma tiles): each reads its
//    packed words from shared memory, decodes them in registers into exact
//    bf16 {-1,0,+1} (two weights per lop3 + fma.bf16x2) and feeds
//    mma.sync.m16n8k16 with fp32 accumulators, one accumulator set per
//    128-wide group that is folded into the running sum with the group scale.
//  * Token tiles of 8 (NT = 1) or 16 (NT = 2) tokens share every decoded
//    weight fragment, so a call reads the weights once for up to 16 tokens.
//
// The pages' own kernel for this band (the "small_t" rung of the
// "ninfer-perf-tuning" skill page, sections 2 and 6) keeps one warp per 16
// rows over the whole K, which on GB300's 152 SMs leaves the 5120-row down
// projection with too few warps; the balanced unit split above replaces its
// row-only grid and its split-K gate.
#include "tern_device.cuh"
#include "tern_internal.h"

namespace tern {
namespace {

constexpr int kWBytes = kSTRows * 128;  // packed weights per stage
constexpr int kSBytes = kSTRows * 8;    // 4 fp16 scales per row per stage

template <int NT>
struct SmallTLayout {
  // B fragments for one stage: [group 4][chunk 8][t 4][g 8] x (8 bytes * NT)
  static constexpr int kXBytes = 4 * 8 * 4 * 8 * 8 * NT;
  static constexpr int kWOff = 0;
  static constexpr int kXOff = kWOff + kSTStages * kWBytes;
  static constexpr int kSOff = kXOff + kSTStages * kXBytes;
  static constexpr int kBarOff = kSOff + kSTStages * kSBytes;
  static constexpr int kBytes = kBarOff + 2 * kSTStages * 8;
  static constexpr int kAlloc = kBytes + 1024;  // base re-aligned to 1024 for the swizzle
};

// One decoded pair (p = 0..7) of a packed word; v6 = v >> 6, v12 = v >> 12.
template <int P>
__device__ __forceinline__ uint32_t pair_of(uint32_t v, uint32_t v6, uint32_t v12) {
  if constexpr (P < 3) return decode_pos<P>(v);
  else if constexpr (P < 6) return decode_pos<P - 3>(v6);
  else return decode_pos<P - 6>(v12);
}

template <int NT, bool kT1>
__global__ void __launch_bounds__(kSTThreads, 1)
    smallt_kernel(const __grid_constant__ CUtensorMap tmW, const uint16_t* __restrict__ scales,
                  const uint16_t* __restrict__ x, float* __restrict__ y, int T, int K, int N,
                  int tok0, int KS, long long U, int* err) {
  using L = SmallTLayout<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + kSTStages;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = K >> 7;

  // Zero the B-fragment buffers: tokens >= T and k >= K stay zero.
  {
    uint4* xb = reinterpret_cast<uint4*>(smem + L::kXOff);
    for (int i = threadIdx.x; i < kSTStages * L::kXBytes / 16; i += blockDim.x)
      xb[i] = make_uint4(0, 0, 0, 0);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSTStages; ++s) {
      mbar_init(&full[s], 32);                 // 32 producer lanes (+ TMA bytes)
      mbar_init(&empty[s], kSTConsumerWarps);  // one arrive per consumer warp
    }
    fence_mbar_init();
    prefetch_tensormap(&tmW);
  }
  __syncthreads();

  const long long P = gridDim.x;
  const long long begin = U * blockIdx.x / P;
  const long long end = U * (blockIdx.x + 1) / P;
  const int Tt = min(T - tok0, 8 * NT);  // tokens in this tile

  if (warp == kSTConsumerWarps) {
    // ------------------------------------------------------------ producer
    int iter = 0;
    for (long long u = begin; u < end; ++u, ++iter) {
      const int s = iter % kSTStages;
      const uint32_t ph = (iter / kSTStages) & 1;
      if (iter >= kSTStages && !mbar_wait(&empty[s], ph ^ 1, err)) break;
      const int rb = static_cast<int>(u / KS);
      const int ks = static_cast<int>(u % KS);
      if (lane == 0) {
        mbar_expect_tx(&full[s], kWBytes);
        tma_load_2d(smem + L::kWOff + s * kWBytes, &tmW, ks * 128, rb * kSTRows, &full[s]);
      }
      // scales: rows lane + 32 i, groups 4 ks .. 4 ks + 3
      uint2* sb = reinterpret_cast<uint2*>(smem + L::kSOff + s * kSBytes);
      const int g0 = ks * 4;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = lane + 32 * i;
        const int n = rb * kSTRows + r;
        uint2 v = make_uint2(0, 0);
        if (n < N) {
          const uint16_t* src = scales + static_cast<size_t>(n) * G + g0;
          if ((G & 3) == 0) {
            v = *reinterpret_cast<const uint2*>(src);
          } else {
            uint32_t h[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) h[j] = (g0 + j < G) ? src[j] : 0u;
            v = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
          }
        }
        sb[r] = v;
      }
      // activations: item = (token g, 32-wide k block blk)
      uint8_t* xb = smem + L::kXOff + s * L::kXBytes;
      const int items = Tt * 16;
      for (int it = lane; it < items; it += 32) {
        const int g = it >> 4;
        const int blk = it & 15;
        const int j = blk >> 2, t = blk & 3;
        const int kk = ks * kSTStageK + 128 * j + 32 * t;
        uint32_t R[16];
        if (kk < K) {
          const uint16_t* src = x + static_cast<size_t>(tok0 + g) * K + kk;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v = ldg_nc_v4(src + 8 * q);
            R[4 * q + 0] = v.x;
            R[4 * q + 1] = v.y;
            R[4 * q + 2] = v.z;
            R[4 * q + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int q = 0; q < 16; ++q) R[q] = 0u;
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t ra = R[8 * (c >> 2) + (c & 3)];
          const uint32_t rbv = R[8 * (c >> 2) + (c & 3) + 4];
          uint2 e;
          e.x = __byte_perm(ra, rbv, 0x5410);  // (x[k1], x[k1+8])
          e.y = __byte_perm(ra, rbv, 0x7632);  // (x[k1+1], x[k1+9])
          const int ent = ((j * 8 + c) * 4 + t) * 8 + (g & 7);
          *reinterpret_cast<uint2*>(xb + (ent * NT + (g >> 3)) * 8) = e;
        }
      }
      mbar_arrive(&full[s]);
    }
    // Do not leave while this CTA's copies may still be landing: wait (bounded)
    // for the last stages issued.  In the normal flow these phases are already
    // complete and the waits return at once.
    for (int d = (iter > kSTStages ? iter - kSTStages : 0); d < iter; ++d)
      if (!mbar_wait(&full[d % kSTStages], (d / kSTStages) & 1, err)) break;
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2;
  const int t = lane & 3;
  const uint32_t wbase = smem_addr(smem + L::kWOff);
  const uint32_t xbase = smem_addr(smem + L::kXOff);
  const uint32_t sbase = smem_addr(smem + L::kSOff);

  float yacc[2][NT][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) yacc[i][nt][e] = 0.f;

  int cur_rb = -1;
  bool cur_from_start = false;
  int cur_last_ks = -1;

  auto flush = [&](int rb, bool whole) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int nA = rb * kSTRows + warp * 32 + 16 * i + g;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int n = nA + ((e >> 1) << 3);
          const int tok = nt * 8 + 2 * t + (e & 1);
          if (n < N && tok < Tt) {
            float* dst = y + static_cast<size_t>(tok0 + tok) * N + n;
            if (whole) *dst = yacc[i][nt][e];
            else atomicAdd(dst, yacc[i][nt][e]);
          }
          yacc[i][nt][e] = 0.f;
        }
      }
    }
  };

  int iter = 0;
  for (long long u = begin; u < end; ++u, ++iter) {
    const int rb = static_cast<int>(u / KS);
    const int ks = static_cast<int>(u % KS);
    if (rb != cur_rb) {
      if (cur_rb >= 0) flush(cur_rb, cur_from_start && cur_last_ks == KS - 1);
      cur_rb = rb;
      cur_from_start = (ks == 0);
    }
    cur_last_ks = ks;

    const int s = iter % kSTStages;
    const uint32_t ph = (iter / kSTStages) & 1;
    if (!mbar_wait(&full[s], ph, err)) return;

    const uint32_t wst = wbase + s * kWBytes;
    const uint32_t xst = xbase + s * SmallTLayout<NT>::kXBytes;
    const uint32_t sst = sbase + s * kSBytes;

    // rows of this warp: tile i covers rows 32 warp + 16 i + {g, g + 8}
    uint2 sc[2][2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int rA = warp * 32 + 16 * i + g;
      sc[i][0] = lds_v2(sst + rA * 8);
      sc[i][1] = lds_v2(sst + (rA + 8) * 8);
    }

#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (ks * 4 + j >= G) break;
      // packed words: row r, bytes 32 j + 8 t (2 words) in swizzled layout
      uint2 wA[2], wB[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int rA = warp * 32 + 16 * i + g;
        const uint32_t off = static_cast<uint32_t>((((2 * j + (t >> 1)) ^ (rA & 7)) << 4) +
                                                   ((t & 1) << 3));
        wA[i] = lds_v2(wst + rA * 128 + off);
        wB[i] = lds_v2(wst + (rA + 8) * 128 + off);
      }
      float acc[2][NT][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[i][nt][e] = 0.f;

#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t vA[2], vB[2], vA6[2], vB6[2], vA12[2], vB12[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          vA[i] = h ? wA[i].y : wA[i].x;
          vB[i] = h ? wB[i].y : wB[i].x;
          vA6[i] = vA[i] >> 6;
          vB6[i] = vB[i] >> 6;
          vA12[i] = vA[i] >> 12;
          vB12[i] = vB[i] >> 12;
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int c = 4 * h + cc;
          const int ent = ((j * 8 + c) * 4 + t) * 8 + g;
          uint32_t b[2 * NT];
          if constexpr (NT == 1) {
            if (kT1 && g != 0) {
              b[0] = 0u;
              b[1] = 0u;
            } else {
              uint2 bv = lds_v2(xst + ent * 8);
              b[0] = bv.x;
              b[1] = bv.y;
            }
          } else {
            uint4 bv = lds_v4(xst + ent * 16);
            b[0] = bv.x;
            b[1] = bv.y;
            b[2] = bv.z;
            b[3] = bv.w;
          }
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            uint32_t a[4];
            switch (cc) {
              case 0:
                a[0] = pair_of<0>(vA[i], vA6[i], vA12[i]);
                a[1] = pair_of<0>(vB[i], vB6[i], vB12[i]);
                a[2] = pair_of<1>(vA[i], vA6[i], vA12[i]);
                a[3] = pair_of<1>(vB[i], vB6[i], vB12[i]);
                break;
              case 1:
                a[0] = pair_of<2>(vA[i], vA6[i], vA12[i]);
                a[1] = pair_of<2>(vB[i], vB6[i], vB12[i]);
                a[2] = pair_of<3>(vA[i], vA6[i], vA12[i]);
                a[3] = pair_of<3>(vB[i], vB6[i], vB12[i]);
                break;
              case 2:
                a[0] = pair_of<4>(vA[i], vA6[i], vA12[i]);
                a[1] = pair_of<4>(vB[i], vB6[i], vB12[i]);
                a[2] = pair_of<5>(vA[i], vA6[i], vA12[i]);
                a[3] = pair_of<5>(vB[i], vB6[i], vB12[i]);
                break;
              default:
                a[0] = pair_of<6>(vA[i], vA6[i], vA12[i]);
                a[1] = pair_of<6>(vB[i], vB6[i], vB12[i]);
                a[2] = pair_of<7>(vA[i], vA6[i], vA12[i]);
                a[3] = pair_of<7>(vB[i], vB6[i], vB12[i]);
                break;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[i][nt], a, b[2 * nt], b[2 * nt + 1]);
          }
        }
      }
      // fold this group into the running sums with the row scales
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t wa = (j < 2) ? sc[i][0].x : sc[i][0].y;
        const uint32_t wb = (j < 2) ? sc[i][1].x : sc[i][1].y;
        const float sA = __half2float(__ushort_as_half(static_cast<unsigned short>(
            (j & 1) ? (wa >> 16) : (wa & 0xFFFFu))));
        const float sB = __half2float(__ushort_as_half(static_cast<unsigned short>(
            (j & 1) ? (wb >> 16) : (wb & 0xFFFFu))));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          yacc[i][nt][0] = fmaf(sA, acc[i][nt][0], yacc[i][nt][0]);
          yacc[i][nt][1] = fmaf(sA, acc[i][nt][1], yacc[i][nt][1]);
          yacc[i][nt][2] = fmaf(sB, acc[i][nt][2], yacc[i][nt][2]);
          yacc[i][nt][3] = fmaf(sB, acc[i][nt][3], yacc[i][nt][3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (cur_rb >= 0) flush(cur_rb, cur_from_start && cur_last_ks == KS - 1);
}

template <int NT, bool kT1>
cudaError_t set_attr_one() {
  return cudaFuncSetAttribute(smallt_kernel<NT, kT1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              SmallTLayout<NT>::kAlloc);
}

}  // namespace

size_t smallt_smem_bytes(int nt) {
  return nt == 1 ? SmallTLayout<1>::kAlloc : SmallTLayout<2>::kAlloc;
}

cudaError_t smallt_set_attributes() {
  cudaError_t e;
  if ((e = set_attr_one<1, true>()) != cudaSuccess) return e;
  if ((e = set_attr_one<1, false>()) != cudaSuccess) return e;
  if ((e = set_attr_one<2, false>()) != cudaSuccess) return e;
  return cudaSuccess;
}

int smallt_ctas_per_sm(int nt) {
  int n = 0;
  cudaError_t e;
  if (nt == 1)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, smallt_kernel<1, false>, kSTThreads,
                                                      SmallTLayout<1>::kAlloc);
  else
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, smallt_kernel<2, false>, kSTThreads,
                                                      SmallTLayout<2>::kAlloc);
  if (e != cudaSuccess || n < 1) n = 1;
  return n;
}

cudaError_t launch_smallt(int nt, bool t1, const CUtensorMap* tmW, const uint16_t* scales,
                          const uint16_t* x, float* y, int T, int K, int N, int tok0,
                          int num_ctas, int* err, cudaStream_t stream) {
  const int KS = (K + kSTStageK - 1) / kSTStageK;
  const long long NB = (N + kSTRows - 1) / kSTRows;
  const long long U = NB * KS;
  if (num_ctas > U) num_ctas = static_cast<int>(U);
  if (nt == 1) {
    if (t1)
      smallt_kernel<1, true><<<num_ctas, kSTThreads, SmallTLayout<1>::kAlloc, stream>>>(
          *tmW, scales, x, y, T, K, N, tok0, KS, U, err);
    else
      smallt_kernel<1, false><<<num_ctas, kSTThreads, SmallTLayout<1>::kAlloc, stream>>>(
          *tmW, scales, x, y, T, K, N, tok0, KS, U, err);
  } else {
    smallt_kernel<2, false><<<num_ctas, kSTThreads, SmallTLayout<2>::kAlloc, stream>>>(
        *tmW, scales, x, y, T, K, N, tok0, KS, U, err);
  }
  return cudaGetLastError();
}

}  // namespace tern
