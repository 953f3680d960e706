// tern_pack: int8 ternary weights -> 2-bit sign-magnitude codes.
// tern_repack_t5: base-3 packed weights (five per byte) -> the same codes.
// tern_quant_act_s8: per-token absmax/127 int8 quantisation of bf16 rows.
// The s8 rung's own input: the same codes split into two exact fp8 pieces.
// tern_rotate_bf16: blockwise Hadamard rotation of bf16 activations.
#include "tern_device.cuh"
#include "tern_internal.h"

#include <cuda_fp8.h>

namespace tern {
namespace {

// Bit of weight j's "nonzero" flag inside its byte; the "negative" flag sits
// two bits higher.  Each nibble holds two weights as [nz_lo, nz_hi, neg_lo,
// neg_hi], so that one AND with 0xA0 per byte isolates one weight as the
// fp8 e4m3 encoding of w/8 (bit 5 = exponent bit for 2^-3, bit 7 = sign).
__device__ __constant__ int kPackNzBit[4] = {0, 1, 4, 5};

// One thread per packed word: 16 int8 weights in, one uint32 out.
__global__ void __launch_bounds__(256) pack_kernel(const int8_t* __restrict__ W,
                                                   uint32_t* __restrict__ Wp, long long words,
                                                   int* __restrict__ bad_count) {
  int bad = 0;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < words;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    // word i covers weights 16 i .. 16 i + 15 of the row-major [N][K] matrix
    // (K % 16 == 0, so a word never straddles two rows).
    const uint4 v = ldg_nc_v4(W + 16 * i);
    const uint32_t b[4] = {v.x, v.y, v.z, v.w};
    uint32_t word = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {      // output byte q <- weights 4q .. 4q+3
#pragma unroll
      for (int j = 0; j < 4; ++j) {    // weight j of the byte
        int w = static_cast<int8_t>((b[q] >> (8 * j)) & 0xFFu);
        if (w < -1 || w > 1) {
          ++bad;
          w = 0;
        }
        const int p = 8 * q + kPackNzBit[j];
        word |= (static_cast<uint32_t>(w != 0) << p) | (static_cast<uint32_t>(w < 0) << (p + 2));
      }
    }
    Wp[i] = word;
  }
  if (bad_count) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if ((threadIdx.x & 31) == 0 && bad) atomicAdd(bad_count, bad);
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Per-token code of v: rint(v / scale) clamped to [-127, 127], the quotient
// rounded as one IEEE single-precision division (nearest-even, as rint).
// Without a division per element: with inv = 1 / scale rounded, q0 = v * inv
// differs from v / scale by less than 128 * (2^-23 + 2^-48) < 1.53e-5 (|v| <=
// absmax, so |v / scale| < 128; two roundings of relative error 2^-24 each),
// and the rounded quotient from v / scale by at most half an ulp below 128,
// 2^-18; so the two are less than kQMargin = 2^-15 apart.  When q0 lies
// farther than kQMargin from every half-integer, both fall strictly inside
// the same rounding interval and rint(q0) is the code; otherwise the element
// takes the division.  fast: scale and 1 / scale normal (absmax >= 127 *
// 2^-126), where those relative bounds hold; else every element divides.
constexpr float kQMargin = 3.0517578125e-05f;  // 2^-15
__device__ __forceinline__ float quant_code(float v, float scale, float inv, bool fast) {
  float r;
  if (fast) {
    const float q0 = v * inv;
    r = rintf(q0);
    if (!(fabsf(q0 - r) < 0.5f - kQMargin)) r = rintf(v / scale);
  } else {
    r = rintf(v / scale);
  }
  return fminf(fmaxf(r, -127.f), 127.f);
}
// Pairs of fp32 values in one 64-bit register for the packed fp32x2
// arithmetic (each half rounded as its scalar instruction would be).
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// max of two floats that propagates NaN (IEEE maximum, not maximumNumber)
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ bool quant_fast(float scale) {
  return scale >= 1.1754943508222875e-38f && scale < 8.507059173023462e+37f;  // [2^-126, 2^126)
}

// One CTA per token.  Pass 1: absmax.  Pass 2: codes.
constexpr int kQThreads = 256;
__global__ void __launch_bounds__(kQThreads) quant_s8_kernel(const uint16_t* __restrict__ x,
                                                             int8_t* __restrict__ q,
                                                             float* __restrict__ xs, int K) {
  const int t = blockIdx.x;
  const uint16_t* row = x + static_cast<size_t>(t) * K;
  int8_t* qrow = q + static_cast<size_t>(t) * K;
  const int chunks = K >> 3;  // 8 bf16 per 16-byte chunk (K % 16 == 0)
  float a = 0.f;
  for (int c = threadIdx.x; c < chunks; c += kQThreads) {
    const uint4 v = ldg_nc_v4(row + 8 * c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) a = fmaxf(a, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  __shared__ float red[kQThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  a = red[0];
#pragma unroll
  for (int i = 1; i < kQThreads / 32; ++i) a = fmaxf(a, red[i]);
  const float scale = a / 127.0f;  // IEEE single-precision division
  if (threadIdx.x == 0) xs[t] = scale;
  const float inv = 1.0f / scale;
  const bool fast = quant_fast(scale);
  for (int c = threadIdx.x; c < chunks; c += kQThreads) {
    uint32_t out[2] = {0u, 0u};
    if (a > 0.f) {
      const uint4 v = ldg_nc_v4(row + 8 * c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float r0 = quant_code(bf16_lo(w[j]), scale, inv, fast);
        const float r1 = quant_code(bf16_hi(w[j]), scale, inv, fast);
        const uint32_t b0 = static_cast<uint32_t>(static_cast<int>(r0)) & 0xFFu;
        const uint32_t b1 = static_cast<uint32_t>(static_cast<int>(r1)) & 0xFFu;
        out[j >> 1] |= (b0 | (b1 << 8)) << (16 * (j & 1));
      }
    }
    *reinterpret_cast<uint2*>(qrow + 8 * c) = make_uint2(out[0], out[1]);
  }
}

// s8 rung input: the codes q of quant_s8_kernel (same arithmetic), split
// exactly into two fp8 e4m3 pieces p1 = 16 rint(q / 16) (ties to even) and
// p2 = q - p1 (multiples of 16 up to 128, and integers in [-8, 8]: all exact
// in e4m3), written as p1[T][K] and p2[T][K] in the decoder's k order: within
// every 16-wide block of k, byte slot 4i + b holds k = 4b + i.
// Codes and pieces of token t's row (global or shared memory): absmax, then
// the pieces of every 16-wide block.  red: kQThreads / 32 floats of shared
// memory.  Ends without a barrier.
__device__ __forceinline__ void quant_row_pieces(const uint16_t* row, int t, int K,
                                                 uint8_t* __restrict__ p1,
                                                 uint8_t* __restrict__ p2,
                                                 float* __restrict__ xs, float* red) {
  // (plain 16-byte loads: row is global or shared memory)
  auto load16 = [&](int e) { return *reinterpret_cast<const uint4*>(row + e); };
  const int chunks = K >> 3;
  float a = 0.f;
  for (int c = threadIdx.x; c < chunks; c += kQThreads) {
    const uint4 v = load16(8 * c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) a = fmaxf(a, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  a = red[0];
#pragma unroll
  for (int i = 1; i < kQThreads / 32; ++i) a = fmaxf(a, red[i]);
  const float scale = a / 127.0f;  // IEEE single-precision division
  if (threadIdx.x == 0) xs[t] = scale;
  const float inv = 1.0f / scale;
  const bool fast = quant_fast(scale);
  for (int blk = threadIdx.x; blk < (K >> 4); blk += kQThreads) {
    const uint4 v0 = load16(16 * blk);
    const uint4 v1 = load16(16 * blk + 8);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    // The 16 codes from the product (see quant_code): dmax is the largest
    // distance of a product from its nearest integer (NaN if any is NaN).
    // On the fast path |q0| < 127.0001, so the codes need no clamp.  A block
    // with any product within kQMargin of a half-integer, a row off the fast
    // path and an all-zero row take the division for all 16 (one branch per
    // block; a block needs it with probability about 1e-3).
    float r[16];
    float dmax = 0.f;
    const uint64_t inv2 = pack_f32x2(inv, inv);
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // elements 2j, 2j + 1 as one fp32 pair
      const uint64_t q2 = mul_f32x2(pack_f32x2(bf16_lo(w[j]), bf16_hi(w[j])), inv2);
      float q0a, q0b;
      unpack_f32x2(q2, q0a, q0b);
      r[2 * j] = rintf(q0a);
      r[2 * j + 1] = rintf(q0b);
      float da, db;
      unpack_f32x2(sub_f32x2(q2, pack_f32x2(r[2 * j], r[2 * j + 1])), da, db);
      dmax = fmax_nan(dmax, fabsf(da));
      dmax = fmax_nan(dmax, fabsf(db));
    }
    if (!(fast && dmax < 0.5f - kQMargin)) {
#pragma unroll
      for (int k = 0; k < 16; ++k)
        r[k] = a > 0.f ? quant_code((k & 1) ? bf16_hi(w[k >> 1]) : bf16_lo(w[k >> 1]), scale,
                                    inv, false)
                       : 0.f;
    }
    // pieces of the codes as exact floats, two at a time: p1 = 16 rint(q /
    // 16) (q / 16 + 1.5 * 2^23 rounds to an integer, ties to even), p2 = q -
    // p1 in [-8, 8]; every step is exact in fp32
    float f1[16], f2[16];
    const uint64_t c16th = pack_f32x2(0.0625f, 0.0625f), cbig = pack_f32x2(12582912.f, 12582912.f);
    const uint64_t c16 = pack_f32x2(16.f, 16.f), cneg = pack_f32x2(-201326592.f, -201326592.f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint64_t r2 = pack_f32x2(r[2 * j], r[2 * j + 1]);
      const uint64_t p12 = fma_f32x2(fma_f32x2(r2, c16th, cbig), c16, cneg);
      unpack_f32x2(p12, f1[2 * j], f1[2 * j + 1]);
      unpack_f32x2(sub_f32x2(r2, p12), f2[2 * j], f2[2 * j + 1]);
    }
    // word i of a piece block holds k = i, i + 4, i + 8, i + 12 in bytes 0..3
    // (slot 4i + b holds k = 4b + i), converted two at a time
    uint32_t o1[4], o2[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o1[i] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(f1[i], f1[i + 4]),
                                                             __NV_SATFINITE, __NV_E4M3)) |
              (static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(f1[i + 8], f1[i + 12]),
                                                              __NV_SATFINITE, __NV_E4M3))
               << 16);
      o2[i] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(f2[i], f2[i + 4]),
                                                             __NV_SATFINITE, __NV_E4M3)) |
              (static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(f2[i + 8], f2[i + 12]),
                                                              __NV_SATFINITE, __NV_E4M3))
               << 16);
    }
    const size_t off = static_cast<size_t>(t) * K + 16 * blk;
    *reinterpret_cast<uint4*>(p1 + off) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
    *reinterpret_cast<uint4*>(p2 + off) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
  }
}


// The row is read twice (absmax, then codes).  Three ways to hold it:
//   staged (K <= kRotateMaxK): persistent CTAs walk the tokens; each copies
//     its next token's row into one of two shared-memory buffers (bulk
//     copies of up to kQCopy bytes) while it quantises the current one (one
//     buffer when two do not fit: the copy then precedes each token);
//   rotate: one CTA per token Hadamard-rotates the row blockwise (each warp a
//     1024-wide block at a time, hadamard_block_1024, scaled by 1/32 and
//     rounded once to bf16, nearest-even) into shared memory;
//   otherwise one CTA per token reads global memory twice.
constexpr uint32_t kQCopy = 16384;
constexpr size_t kQSmemPerSm = 228 * 1024;  // shared memory of an SM
constexpr int kQCtasPerSm = 4;              // the kernel's registers allow four CTAs
enum : int { kQGlobal = 0, kQRotate = 1, kQStaged = 2 };
__global__ void __launch_bounds__(kQThreads) quant_pieces_kernel(const uint16_t* __restrict__ x,
                                                                 uint8_t* __restrict__ p1,
                                                                 uint8_t* __restrict__ p2,
                                                                 float* __restrict__ xs, int T,
                                                                 int K, int mode, int nbuf,
                                                                 int* err) {
  extern __shared__ __align__(16) uint16_t xrow[];
  __shared__ uint64_t row_bar[2];
  __shared__ float red[kQThreads / 32];
  grid_dependents_launch();
  grid_dependency_wait();  // x and the output buffers come from earlier work
  if (mode == kQGlobal) {
    const int t = blockIdx.x;
    quant_row_pieces(x + static_cast<size_t>(t) * K, t, K, p1, p2, xs, red);
    return;
  }
  if (mode == kQRotate) {
    const int t = blockIdx.x;
    const uint16_t* row = x + static_cast<size_t>(t) * K;
    const int lane = threadIdx.x & 31;
    for (int b = threadIdx.x >> 5; b < K / kRotBlock; b += kQThreads / 32) {
      float v[32];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const uint2 raw = *reinterpret_cast<const uint2*>(row + b * kRotBlock + 128 * g + 4 * lane);
        v[4 * g + 0] = bf16_lo(raw.x);
        v[4 * g + 1] = bf16_hi(raw.x);
        v[4 * g + 2] = bf16_lo(raw.y);
        v[4 * g + 3] = bf16_hi(raw.y);
      }
      hadamard_block_1024(v, lane);
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        uint32_t h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          h[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v[4 * g + i] * 0.03125f));
        *reinterpret_cast<uint2*>(xrow + b * kRotBlock + 128 * g + 4 * lane) =
            make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
      }
    }
    __syncthreads();
    quant_row_pieces(xrow, t, K, p1, p2, xs, red);
    return;
  }
  // staged
  const uint32_t bytes = 2u * static_cast<uint32_t>(K);  // K % 16 == 0: 16-byte multiples
  auto issue = [&](int tt, int b) {  // one thread: token tt's row into buffer b
    mbar_arrive_expect_tx(&row_bar[b], bytes);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(x + static_cast<size_t>(tt) * K);
    uint8_t* dst = reinterpret_cast<uint8_t*>(xrow + static_cast<size_t>(b) * K);
    for (uint32_t off = 0; off < bytes; off += kQCopy)
      bulk_load(dst + off, src + off, bytes - off < kQCopy ? bytes - off : kQCopy, &row_bar[b]);
  };
  if (threadIdx.x == 0) {
    mbar_init(&row_bar[0], 1);
    mbar_init(&row_bar[1], 1);
    fence_mbar_init();
    if (static_cast<int>(blockIdx.x) < T) issue(blockIdx.x, 0);
  }
  __syncthreads();  // the barriers are initialised before anyone waits on them
  int i = 0;
  for (int t = blockIdx.x; t < T; t += gridDim.x, ++i) {
    const int b = nbuf == 2 ? (i & 1) : 0;
    const uint32_t par = nbuf == 2 ? ((i >> 1) & 1) : (i & 1);
    const int tn = t + gridDim.x;
    // buffer b ^ 1 was last read in the previous iteration, which ended with
    // a barrier
    if (nbuf == 2 && threadIdx.x == 0 && tn < T) {
      fence_proxy_async_smem();
      issue(tn, b ^ 1);
    }
    const bool ok = mbar_wait(&row_bar[b], par, err);
    if (!__syncthreads_and(ok)) {
      if (threadIdx.x == 0) {  // no copy outlives the CTA
        mbar_wait(&row_bar[b], par, err);
        if (nbuf == 2 && tn < T) mbar_wait(&row_bar[b ^ 1], ((i + 1) >> 1) & 1, err);
      }
      return;
    }
    quant_row_pieces(xrow + static_cast<size_t>(b) * K, t, K, p1, p2, xs, red);
    __syncthreads();  // buffer b and red are free again
    if (nbuf == 1 && threadIdx.x == 0 && tn < T) {
      fence_proxy_async_smem();
      issue(tn, 0);
    }
  }
}

// ---------------------------------------------------------------- base-3 repack
// Base-3 layout: 26 bytes per 128-weight group, [N][K/128][26].  Byte j holds
// the group's weights 5j .. 5j+4 as sum_i (w_i + 1) 3^i, the first weight
// least significant; the last byte's digits 3 and 4 lie past the group.
// Bytes above 242 are invalid and give five zero weights.
constexpr int kT5GroupBytes = 26;
constexpr int kRepackThreads = 256;  // one 128-weight group per thread

// Each CTA stages the bytes of its kRepackThreads groups in shared memory
// with 16-byte loads (the block's first byte sits at a multiple of
// 256 * 26 = 6656 = 16 * 416 bytes), then each thread decodes one group into
// the eight 2-bit words of that group and stores them as two 16-byte vectors.
__global__ void __launch_bounds__(kRepackThreads) repack_t5_kernel(
    const uint8_t* __restrict__ P, uint32_t* __restrict__ Wp, long long groups,
    int* __restrict__ bad_count) {
  __shared__ __align__(16) uint8_t stage[kRepackThreads * kT5GroupBytes];
  const long long g0 = static_cast<long long>(blockIdx.x) * kRepackThreads;
  const long long left = groups - g0;
  const int here = left < kRepackThreads ? static_cast<int>(left) : kRepackThreads;
  const int bytes = here * kT5GroupBytes;
  const uint8_t* src = P + g0 * kT5GroupBytes;
  for (int c = threadIdx.x; c < bytes / 16; c += kRepackThreads)
    reinterpret_cast<uint4*>(stage)[c] = ldg_nc_v4(src + 16 * c);
  for (int b = (bytes / 16) * 16 + threadIdx.x; b < bytes; b += kRepackThreads) stage[b] = src[b];
  __syncthreads();

  int bad = 0;
  if (static_cast<int>(threadIdx.x) < here) {
    const uint8_t* gb = stage + threadIdx.x * kT5GroupBytes;
    uint32_t word[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < kT5GroupBytes; ++j) {
      uint32_t v = gb[j];
      if (v > 242u) {
        ++bad;
        v = 121u;  // digits 1,1,1,1,1: five zero weights
      }
#pragma unroll
      for (int i = 0; i < 5; ++i) {
        const int r = 5 * j + i;  // weight index in the group (compile-time)
        const uint32_t d = v % 3u;
        v /= 3u;
        if (r < 128) {
          // 2-bit code of w = d - 1: nonzero bit at P[r % 4] = {0, 1, 4, 5}
          // of byte (r % 16) / 4 of word r / 16, negative bit two above
          const int p = 8 * ((r % 16) / 4) + ((r % 4) < 2 ? (r % 4) : (r % 4) + 2);
          word[r / 16] |= (static_cast<uint32_t>(d != 1u) << p) |
                          (static_cast<uint32_t>(d == 0u) << (p + 2));
        }
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(Wp + (g0 + threadIdx.x) * 8);
    dst[0] = make_uint4(word[0], word[1], word[2], word[3]);
    dst[1] = make_uint4(word[4], word[5], word[6], word[7]);
  }
  if (bad_count) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if ((threadIdx.x & 31) == 0 && bad) atomicAdd(bad_count, bad);
  }
}

// ---------------------------------------------------------------- rotation
// One warp per (token, 1024-block): lane l holds elements 32 l .. 32 l + 31 of
// the block.  Index bits 0-4 are transformed inside the thread, bits 5-9
// across lanes with shuffles; each butterfly (a, b) -> (a + b, a - b) in fp32
// gives the natural-order (Sylvester) Hadamard transform.  Then * 1/32 (exact)
// and one rounding to bf16, nearest-even.  Plain loads and stores: the block
// is read whole before it is written, so xr may be x.
constexpr int kRotWarps = 8;

__global__ void __launch_bounds__(kRotWarps * 32) rotate_bf16_kernel(const uint16_t* x,
                                                                    uint16_t* xr,
                                                                    long long pairs) {
  const long long w = static_cast<long long>(blockIdx.x) * kRotWarps + (threadIdx.x >> 5);
  if (w >= pairs) return;  // whole warps leave together
  const int lane = threadIdx.x & 31;
  // x is [T][K] with K a multiple of 1024, so pair w starts at element 1024 w
  const size_t base = static_cast<size_t>(w) * kRotBlock + static_cast<size_t>(lane) * 32;
  const uint4* src = reinterpret_cast<const uint4*>(x + base);
  float v[32];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 q = src[c];
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[8 * c + 2 * e] = __uint_as_float(u[e] << 16);
      v[8 * c + 2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
    }
  }
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
    }
  }
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
    const bool upper = (lane & h) != 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], h);
      v[i] = upper ? o - v[i] : v[i] + o;
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(xr + base);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t u[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[8 * c + 2 * e] * 0.03125f));
      const uint32_t hi =
          __bfloat16_as_ushort(__float2bfloat16_rn(v[8 * c + 2 * e + 1] * 0.03125f));
      u[e] = lo | (hi << 16);
    }
    dst[c] = make_uint4(u[0], u[1], u[2], u[3]);
  }
}

}  // namespace

cudaError_t launch_pack(const int8_t* W, uint32_t* Wp, int K, int N, int* bad, int num_sms,
                        cudaStream_t stream) {
  const long long words = static_cast<long long>(N) * (K / 16);
  long long blocks = (words + 255) / 256;
  const long long cap = static_cast<long long>(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  pack_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(W, Wp, words, bad);
  return cudaGetLastError();
}

cudaError_t launch_repack_t5(const uint8_t* P, uint32_t* Wp, int K, int N, int* bad,
                             cudaStream_t stream) {
  const long long groups = static_cast<long long>(N) * (K / 128);
  const long long blocks = (groups + kRepackThreads - 1) / kRepackThreads;
  repack_t5_kernel<<<static_cast<unsigned>(blocks), kRepackThreads, 0, stream>>>(P, Wp, groups,
                                                                                  bad);
  return cudaGetLastError();
}

cudaError_t launch_rotate_bf16(const uint16_t* x, uint16_t* xr, int T, int K,
                               cudaStream_t stream) {
  const long long pairs = static_cast<long long>(T) * (K / kRotBlock);
  const long long blocks = (pairs + kRotWarps - 1) / kRotWarps;
  rotate_bf16_kernel<<<static_cast<unsigned>(blocks), kRotWarps * 32, 0, stream>>>(x, xr, pairs);
  return cudaGetLastError();
}

cudaError_t launch_quant_s8(const uint16_t* x, int8_t* q, float* xs, int T, int K,
                            cudaStream_t stream) {
  quant_s8_kernel<<<T, kQThreads, 0, stream>>>(x, q, xs, K);
  return cudaGetLastError();
}

cudaError_t quant_set_attributes() {
  return cudaFuncSetAttribute(quant_pieces_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              2 * kRotateMaxK);
}

cudaError_t launch_quant_pieces(const uint16_t* x, uint8_t* p1, uint8_t* p2, float* xs, int T,
                                int K, int rotate, int num_sms, int* err, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  if (rotate) {  // K <= kRotateMaxK: the rotated row fits
    const cudaLaunchConfig_t cfg =
        pdl_launch_config(attr, dim3(T), dim3(kQThreads), 2 * static_cast<size_t>(K), stream);
    return cudaLaunchKernelEx(&cfg, quant_pieces_kernel, x, p1, p2, xs, T, K,
                              static_cast<int>(kQRotate), 1, err);
  } else if (K <= kRotateMaxK) {
    // two row buffers when they fit the kernel's shared-memory allowance;
    // as many CTAs as fit per SM (at most kQCtasPerSm: registers)
    const int nbuf = 4 * static_cast<size_t>(K) <= 2 * static_cast<size_t>(kRotateMaxK) ? 2 : 1;
    const size_t smem = 2 * static_cast<size_t>(K) * nbuf;
    int per_sm = static_cast<int>(kQSmemPerSm / (smem + 1024));
    if (per_sm > kQCtasPerSm) per_sm = kQCtasPerSm;
    if (per_sm < 1) per_sm = 1;
    const int grid = T < per_sm * num_sms ? T : per_sm * num_sms;
    const cudaLaunchConfig_t cfg = pdl_launch_config(attr, dim3(grid), dim3(kQThreads), smem, stream);
    return cudaLaunchKernelEx(&cfg, quant_pieces_kernel, x, p1, p2, xs, T, K,
                              static_cast<int>(kQStaged), nbuf, err);
  }
  const cudaLaunchConfig_t cfg = pdl_launch_config(attr, dim3(T), dim3(kQThreads), 0, stream);
  return cudaLaunchKernelEx(&cfg, quant_pieces_kernel, x, p1, p2, xs, T, K,
                            static_cast<int>(kQGlobal), 1, err);
}

}  // namespace tern
