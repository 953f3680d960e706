// Internal interface between the C-ABI layer (tern_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tern {

// Small-T bf16 rungs: rows per CTA row block and k per pipeline stage.
constexpr int kSTRows = 128;
constexpr int kSTStageK = 512;        // 128 packed bytes per row
constexpr int kSTStages = 4;
constexpr int kSTConsumerWarps = 4;
constexpr int kSTThreads = (kSTConsumerWarps + 1) * 32;

size_t smallt_smem_bytes(int nt);

// Launch one token tile of the small-T kernel.
//   nt = 1 (8 tokens) or 2 (16 tokens); t1 = token tile known to hold one token.
//   tok0: first token of the tile.  num_ctas: persistent grid size.
cudaError_t launch_smallt(int nt, bool t1, const CUtensorMap* tmW, const uint16_t* scales,
                          const uint16_t* x, float* y, int T, int K, int N, int tok0,
                          int num_ctas, int* err, cudaStream_t stream);
cudaError_t smallt_set_attributes();
int smallt_ctas_per_sm(int nt);

// s8 rung.
constexpr int kS8TileN = 128;
constexpr int kS8TileT = 128;
constexpr int kS8Stages = 4;
size_t s8_smem_bytes();
cudaError_t s8_set_attributes();
cudaError_t launch_s8(const CUtensorMap* tmW, const CUtensorMap* tmQ, const uint16_t* scales,
                      const float* x_scale, float* y, int T, int K, int N, int* err,
                      cudaStream_t stream);

// Pack and quantise.
cudaError_t launch_pack(const int8_t* W, uint32_t* Wp, int K, int N, int* bad, int num_sms,
                        cudaStream_t stream);
cudaError_t launch_quant_s8(const uint16_t* x, int8_t* q, float* xs, int T, int K,
                            cudaStream_t stream);

}  // namespace tern
