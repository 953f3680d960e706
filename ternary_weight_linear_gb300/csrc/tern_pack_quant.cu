// tern_pack: int8 ternary weights -> 2-bit sign-magnitude codes.
// tern_quant_act_s8: per-token absmax/127 int8 quantisation of bf16 rows.
#include "tern_device.cuh"
#include "tern_internal.h"

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

}  // namespace tern
