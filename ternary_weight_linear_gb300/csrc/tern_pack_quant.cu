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
  for (int c = threadIdx.x; c < chunks; c += kQThreads) {
    uint32_t out[2] = {0u, 0u};
    if (a > 0.f) {
      const uint4 v = ldg_nc_v4(row + 8 * c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float r0 = rintf(bf16_lo(w[j]) / scale);
        float r1 = rintf(bf16_hi(w[j]) / scale);
        r0 = fminf(fmaxf(r0, -127.f), 127.f);
        r1 = fminf(fmaxf(r1, -127.f), 127.f);
        const uint32_t b0 = static_cast<uint32_t>(static_cast<int>(r0)) & 0xFFu;
        const uint32_t b1 = static_cast<uint32_t>(static_cast<int>(r1)) & 0xFFu;
        out[j >> 1] |= (b0 | (b1 << 8)) << (16 * (j & 1));
      }
    }
    *reinterpret_cast<uint2*>(qrow + 8 * c) = make_uint2(out[0], out[1]);
  }
}

// s8 rung input: the codes q of quant_s8_kernel (same arithmetic), split
// exactly into two fp8 e4m3 pieces p1 = 16 floor((q + 8) / 16) and
// p2 = q - p1 (multiples of 16 up to 128, and integers in [-8, 7]: all exact
// in e4m3), written as p1[T][K] and p2[T][K] in the decoder's k order: within
// every 16-wide block of k, byte slot 4i + b holds k = 4b + i.
// rotate: the token's row is first Hadamard-rotated blockwise (each warp a
// 1024-wide block at a time, hadamard_block_1024, scaled by 1/32 and rounded
// once to bf16, nearest-even) into dynamic shared memory (2 K bytes), and
// quantised from there.
__global__ void __launch_bounds__(kQThreads) quant_pieces_kernel(const uint16_t* __restrict__ x,
                                                                 uint8_t* __restrict__ p1,
                                                                 uint8_t* __restrict__ p2,
                                                                 float* __restrict__ xs, int K,
                                                                 int rotate) {
  extern __shared__ __align__(16) uint16_t xrow[];
  const int t = blockIdx.x;
  const uint16_t* row = x + static_cast<size_t>(t) * K;
  if (rotate) {
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
    row = xrow;
  }
  // (plain 16-byte loads: row is global or, rotated, shared memory)
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
  __shared__ float red[kQThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  a = red[0];
#pragma unroll
  for (int i = 1; i < kQThreads / 32; ++i) a = fmaxf(a, red[i]);
  const float scale = a / 127.0f;  // IEEE single-precision division
  if (threadIdx.x == 0) xs[t] = scale;
  for (int blk = threadIdx.x; blk < (K >> 4); blk += kQThreads) {
    const uint4 v0 = load16(16 * blk);
    const uint4 v1 = load16(16 * blk + 8);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t o1[4] = {0u, 0u, 0u, 0u}, o2[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      int q = 0;
      if (a > 0.f) {
        const float v = (k & 1) ? bf16_hi(w[k >> 1]) : bf16_lo(w[k >> 1]);
        const float r = fminf(fmaxf(rintf(v / scale), -127.f), 127.f);
        q = static_cast<int>(r);
      }
      const int h = (q + 8) >> 4;  // floor((q + 8) / 16), in [-8, 8]
      const uint32_t e1 = __nv_cvt_float_to_fp8(static_cast<float>(16 * h), __NV_SATFINITE,
                                                __NV_E4M3);
      const uint32_t e2 = __nv_cvt_float_to_fp8(static_cast<float>(q - 16 * h), __NV_SATFINITE,
                                                __NV_E4M3);
      const int slot = 4 * (k & 3) + (k >> 2);  // k = 4b + i -> slot 4i + b
      o1[slot >> 2] |= e1 << (8 * (slot & 3));
      o2[slot >> 2] |= e2 << (8 * (slot & 3));
    }
    const size_t off = static_cast<size_t>(t) * K + 16 * blk;
    *reinterpret_cast<uint4*>(p1 + off) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
    *reinterpret_cast<uint4*>(p2 + off) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
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
                                int K, int rotate, cudaStream_t stream) {
  const size_t smem = rotate ? 2 * static_cast<size_t>(K) : 0;
  quant_pieces_kernel<<<T, kQThreads, smem, stream>>>(x, p1, p2, xs, K, rotate);
  return cudaGetLastError();
}

}  // namespace tern
