// Device-side building blocks shared by the rung kernels: mbarrier and TMA
// wrappers (inline PTX), bounded waits, and the 2-bit ternary decoders.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace tern {

// ---------------------------------------------------------------- error word
// One int per device; kernels OR bits into it when a bounded wait runs out.
enum : int { kErrTimeout = 1 };

// A wait gives up after this many nanoseconds of %globaltimer time.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  [[maybe_unused]] uint64_t state;
  asm volatile("mbarrier.arrive.shared::cta.b64 %0, [%1];" : "=l"(state) : "r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  [[maybe_unused]] uint64_t state;
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 %0, [%1], %2;"
               : "=l"(state)
               : "r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// kWaitLimitNs: ORs kErrTimeout into *err and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u && global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA
// 2D tiled load of a box into shared memory, completing on `bar`.
// x is the innermost coordinate (in elements of the tensor map's type).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- loads
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 lds_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// ---------------------------------------------------------------- decode
// 2-bit trit digits c = w + 1 -> bf16 pairs holding w exactly.
//
// A packed word holds 16 digits: field j (bits 2j, 2j+1) for j = 0..15.  The
// decoder yields 8 bf16x2 pairs; pair p (p = 0..7) has field p in its low half
// and field p+8 in its high half.  Method: OR the isolated field into the
// mantissa of the bf16 constant 128 (0x4300, whose unit in the last place is
// 1), giving 128 + c * 4^i for a field at mantissa position i (bits 2i,
// 2i+1, i = 0..2); one exact fused multiply-add by 4^-i and -(128 * 4^-i + 1)
// then leaves c - 1 = w.  Both halves use the same position, so one
// instruction decodes two weights.
__device__ __forceinline__ uint32_t bf16x2_fma_bits(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t lop_and_or(uint32_t v, uint32_t mask, uint32_t magic) {
  uint32_t d;
  // d = (v & mask) | magic
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(v), "r"(mask), "r"(magic));
  return d;
}

// Decode the field pair at mantissa position i (0..2) of both halves of v.
template <int I>
__device__ __forceinline__ uint32_t decode_pos(uint32_t v) {
  constexpr uint32_t kMask = 0x00030003u << (2 * I);
  // multiplier 4^-I and addend -(128 * 4^-I + 1), both exact in bf16
  constexpr uint32_t kMul = I == 0 ? 0x3F803F80u : (I == 1 ? 0x3E803E80u : 0x3D803D80u);
  constexpr uint32_t kAdd = I == 0 ? 0xC301C301u : (I == 1 ? 0xC204C204u : 0xC110C110u);
  return bf16x2_fma_bits(lop_and_or(v, kMask, 0x43004300u), kMul, kAdd);
}

// All 8 pairs of one word: out[p] = (w[field p], w[field p+8]) as bf16x2.
__device__ __forceinline__ void decode_word_bf16(uint32_t v, uint32_t out[8]) {
  const uint32_t v6 = v >> 6;
  const uint32_t v12 = v >> 12;
  out[0] = decode_pos<0>(v);
  out[1] = decode_pos<1>(v);
  out[2] = decode_pos<2>(v);
  out[3] = decode_pos<0>(v6);
  out[4] = decode_pos<1>(v6);
  out[5] = decode_pos<2>(v6);
  out[6] = decode_pos<0>(v12);
  out[7] = decode_pos<1>(v12);
}

// 4 digits of one byte (fields 0..3 of the low byte of b) -> 4 int8 w values
// (byte i = w of field i), using carry-free byte arithmetic.
__device__ __forceinline__ uint32_t decode_byte_s8(uint32_t b) {
  uint32_t x = (b | (b << 12)) & 0x000F000Fu;   // fields 0,1 -> bits 0..3; 2,3 -> 16..19
  x = (x | (x << 6)) & 0x03030303u;             // field i -> bits 8i, 8i+1
  // c - 1 per byte without borrows: ((c | 0x80) - 1) ^ 0x80
  return ((x | 0x80808080u) - 0x01010101u) ^ 0x80808080u;
}

// ---------------------------------------------------------------- MMA
__device__ __forceinline__ void mma_bf16_16816(float d[4], const uint32_t a[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_s8_16832(int d[4], const uint32_t a[4], uint32_t b0,
                                             uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Exact int -> float for |i| < 2^22 via the 1.5 * 2^23 bias.
__device__ __forceinline__ float int_to_float_exact(int i) {
  return __int_as_float(i + 0x4B400000) - 12582912.0f;
}

}  // namespace tern
