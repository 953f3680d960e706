// s8 rung (T >= 17): int8 per-token activations x ternary-as-int8 weights,
// exact int32 accumulation per 128-wide group, fp32 output
//     y[t][n] = xs[t] * sum_g s[n][g] * acc[t][n][g].
//
// Tile: 128 output rows x 128 tokens per CTA, 8 warps (2 x 4), each warp 64
// rows x 32 tokens.  Per 128-wide k group:
//   * TMA brings the group's packed weights (128 rows x 32 bytes) and its
//     activation codes (128 tokens x 128 bytes, 128-byte swizzle) into a
//     4-deep ring;
//   * all threads decode the packed weights once into an int8 tile in shared
//     memory (swizzled 16-byte chunks), shared by the four token warps;
//   * mma.sync.m16n8k32 s8 x s8 -> s32 over the group, fragments loaded with
//     ldmatrix; the per-group int32 result is exact (|acc| <= 127 * 128);
//   * the epilogue turns it into fp32 exactly (1.5 * 2^23 bias) and folds it
//     into the running sum with the row's group scale.
// This is the "s8" prefill rung of the "ninfer-perf-tuning" skill page
// (section 2 rung map; int8 m16n8k32 MMA per the "NInfer sm_89 fork"
// write-up, section 9 item 2).
#include "tern_device.cuh"
#include "tern_internal.h"

namespace tern {
namespace {

constexpr int kThreads = 256;
constexpr int kWStage = kS8TileN * 32;   // packed weights of one group
constexpr int kQStage = kS8TileT * 128;  // activation codes of one group
struct S8Layout {
  static constexpr int kQOff = 0;                                  // 1024-aligned stages
  static constexpr int kDecOff = kQOff + kS8Stages * kQStage;      // decoded int8 [128][128]
  static constexpr int kWOff = kDecOff + kS8TileN * 128;
  static constexpr int kBarOff = kWOff + kS8Stages * kWStage;
  static constexpr int kBytes = kBarOff + kS8Stages * 8;
  static constexpr int kAlloc = kBytes + 1024;
};

__global__ void __launch_bounds__(kThreads, 1)
    s8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmQ,
              const uint16_t* __restrict__ scales, const float* __restrict__ x_scale,
              float* __restrict__ y, int T, int K, int N, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S8Layout::kBarOff);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 2;  // 0..1: rows 64 wm
  const int wt = warp & 3;   // 0..3: tokens 32 wt
  const int g = lane >> 2, t4 = lane & 3;
  const int n0 = blockIdx.x * kS8TileN;
  const int t0 = blockIdx.y * kS8TileT;
  const int G = K >> 7;

  if (tid == 0) {
    for (int s = 0; s < kS8Stages; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmQ);
  }
  __syncthreads();

  auto issue = [&](int grp) {
    const int s = grp % kS8Stages;
    mbar_arrive_expect_tx(&full[s], kWStage + kQStage);
    tma_load_2d(smem + S8Layout::kWOff + s * kWStage, &tmW, grp * 32, n0, &full[s]);
    tma_load_2d(smem + S8Layout::kQOff + s * kQStage, &tmQ, grp * 128, t0, &full[s]);
  };
  int issued = 0;  // groups issued so far (meaningful in thread 0)
  if (tid == 0)
    for (; issued < kS8Stages && issued < G; ++issued) issue(issued);

  float yacc[4][4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e) yacc[a][b][e] = 0.f;

  const uint32_t dec = smem_addr(smem + S8Layout::kDecOff);
  bool ok = true;
  for (int grp = 0; grp < G; ++grp) {
    const int s = grp % kS8Stages;
    // row scales for this group (8 rows per thread), fetched before the wait
    float sc[4][2];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int n = n0 + 64 * wm + 16 * mt + g + 8 * h;
        sc[mt][h] = n < N ? __half2float(__ushort_as_half(scales[static_cast<size_t>(n) * G + grp]))
                          : 0.f;
      }
    const bool landed = mbar_wait(&full[s], (grp / kS8Stages) & 1, err);
    // decode: thread -> row tid/2, 16 packed bytes (64 weights) -> 4 chunks
    if (landed) {
      const int r = tid >> 1, hh = tid & 1;
      const uint4 pw =
          *reinterpret_cast<const uint4*>(smem + S8Layout::kWOff + s * kWStage + r * 32 + hh * 16);
      const uint32_t words[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        uint32_t d[4];
        decode_word_s8(words[m], d);  // 16 int8 weights in k order
        const uint4 o = make_uint4(d[0], d[1], d[2], d[3]);
        const int c = 4 * hh + m;
        *reinterpret_cast<uint4*>(smem + S8Layout::kDecOff + r * 128 + ((c ^ (r & 7)) << 4)) = o;
      }
    }
    // One vote per group: every thread either saw the stage land or timed out,
    // so all threads take the same branch and no barrier is left waiting.
    if (!__syncthreads_and(landed)) {
      ok = false;
      break;
    }

    int cacc[4][4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b)
#pragma unroll
        for (int e = 0; e < 4; ++e) cacc[a][b][e] = 0;

    const uint32_t qst = smem_addr(smem + S8Layout::kQOff + s * kQStage);
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
      uint32_t af[4][4];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int row = 64 * wm + 16 * mt + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int ch = 2 * kc + (lane >> 4);
        ldmatrix_x4(af[mt], dec + row * 128 + ((ch ^ (row & 7)) << 4));
      }
      uint32_t bf[4][2];
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int tok = 32 * wt + 8 * (2 * p + (lane >> 4)) + (lane & 7);
        const int ch = 2 * kc + ((lane >> 3) & 1);
        uint32_t r[4];
        ldmatrix_x4(r, qst + tok * 128 + ((ch ^ (tok & 7)) << 4));
        bf[2 * p][0] = r[0];
        bf[2 * p][1] = r[1];
        bf[2 * p + 1][0] = r[2];
        bf[2 * p + 1][1] = r[3];
      }
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) mma_s8_16832(cacc[mt][nt], af[mt], bf[nt][0], bf[nt][1]);
    }
    // exact int32 -> fp32, then fold in with the group scale
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        yacc[mt][nt][0] = fmaf(sc[mt][0], int_to_float_exact(cacc[mt][nt][0]), yacc[mt][nt][0]);
        yacc[mt][nt][1] = fmaf(sc[mt][0], int_to_float_exact(cacc[mt][nt][1]), yacc[mt][nt][1]);
        yacc[mt][nt][2] = fmaf(sc[mt][1], int_to_float_exact(cacc[mt][nt][2]), yacc[mt][nt][2]);
        yacc[mt][nt][3] = fmaf(sc[mt][1], int_to_float_exact(cacc[mt][nt][3]), yacc[mt][nt][3]);
      }
    __syncthreads();  // stage s and the decoded tile are free again
    if (tid == 0 && issued < G) issue(issued++);
  }
  if (!ok) {
    // Leave only after the copies this CTA issued have landed (bounded).
    if (tid == 0) {
      const int first = issued > kS8Stages ? issued - kS8Stages : 0;
      for (int gi = first; gi < issued; ++gi)
        if (!mbar_wait(&full[gi % kS8Stages], (gi / kS8Stages) & 1, err)) break;
    }
    return;
  }

  // y[t][n] = xs[t] * acc
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e2 = 0; e2 < 2; ++e2) {
      const int tok = t0 + 32 * wt + 8 * nt + 2 * t4 + e2;
      if (tok >= T) continue;
      const float xsv = x_scale[tok];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n = n0 + 64 * wm + 16 * mt + g + 8 * h;
          if (n < N) y[static_cast<size_t>(tok) * N + n] = xsv * yacc[mt][nt][2 * h + e2];
        }
    }
}

}  // namespace

size_t s8_smem_bytes() { return S8Layout::kAlloc; }

cudaError_t s8_set_attributes() {
  return cudaFuncSetAttribute(s8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              S8Layout::kAlloc);
}

cudaError_t launch_s8(const CUtensorMap* tmW, const CUtensorMap* tmQ, const uint16_t* scales,
                      const float* x_scale, float* y, int T, int K, int N, int* err,
                      cudaStream_t stream) {
  dim3 grid((N + kS8TileN - 1) / kS8TileN, (T + kS8TileT - 1) / kS8TileT);
  s8_kernel<<<grid, kThreads, S8Layout::kAlloc, stream>>>(*tmW, *tmQ, scales, x_scale, y, T, K, N,
                                                          err);
  return cudaGetLastError();
}

}  // namespace tern
