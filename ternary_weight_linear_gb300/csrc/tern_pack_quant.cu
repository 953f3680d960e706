// tern_pack: int8 ternary weights -> 2-bit sign-magnitude codes.
// tern_quant_act_s8: per-token absmax/127 int8 quantisation of bf16 rows.
// The s8 rung's own input: the same codes split into two exact fp8 pieces.
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
__global__ void __launch_bounds__(kQThreads) quant_pieces_kernel(const uint16_t* __restrict__ x,
                                                                 uint8_t* __restrict__ p1,
                                                                 uint8_t* __restrict__ p2,
                                                                 float* __restrict__ xs, int K) {
  const int t = blockIdx.x;
  const uint16_t* row = x + static_cast<size_t>(t) * K;
  const int chunks = K >> 3;
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
  for (int blk = threadIdx.x; blk < (K >> 4); blk += kQThreads) {
    const uint4 v0 = ldg_nc_v4(row + 16 * blk);
    const uint4 v1 = ldg_nc_v4(row + 16 * blk + 8);
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

cudaError_t launch_quant_s8(const uint16_t* x, int8_t* q, float* xs, int T, int K,
                            cudaStream_t stream) {
  quant_s8_kernel<<<T, kQThreads, 0, stream>>>(x, q, xs, K);
  return cudaGetLastError();
}

cudaError_t launch_quant_pieces(const uint16_t* x, uint8_t* p1, uint8_t* p2, float* xs, int T,
                                int K, cudaStream_t stream) {
  quant_pieces_kernel<<<T, kQThreads, 0, stream>>>(x, p1, p2, xs, K);
  return cudaGetLastError();
}

}  // namespace tern
