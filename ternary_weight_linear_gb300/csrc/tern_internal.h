// Internal interface between the C-ABI layer (tern_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tern {

// Small-T rungs (T <= 16): k per pipeline stage and ring depth.  Token tiles
// are TT = 1, 4, 8 or 16 tokens.
constexpr int kSTStageK = 512;  // 128 packed bytes per row
constexpr int kSTStages = 4;

// Bytes of the activation-fragment buffer one TT tile needs for K.
size_t smallt_xprep_bytes(int tt, int K);
// Rows per CTA row block for TT (the TMA box height).
int smallt_rows(int tt);
cudaError_t smallt_set_attributes();
int smallt_ctas_per_sm(int tt);
// Launch the prep kernel and the main kernel (programmatic dependent) for
// tokens [tok0, tok0 + Tt) with Tt <= tt.  xprep: workspace of
// smallt_xprep_bytes(tt, K) bytes.
cudaError_t launch_smallt(int tt, const CUtensorMap* tmW, const uint16_t* scales,
                          const uint16_t* x, uint8_t* xprep, float* y, int K, int N, int tok0,
                          int Tt, int num_sms, int ctas_per_sm, int* err, cudaStream_t stream);

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
