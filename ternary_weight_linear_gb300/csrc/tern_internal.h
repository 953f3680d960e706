// Internal interface between the C-ABI layer (tern_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tern {

// Small-T rungs (T <= 16): k per pipeline stage.  Token tiles are TT = 1, 4,
// 8 or 16 tokens.
constexpr int kSTStageK = 1024;  // 256 packed bytes per row: two 128-byte TMA boxes
// Grid cap of the small-T kernel (one CTA per SM).
constexpr int kSmallTMaxCtas = 160;
// Most activation blocks the one-token kernel keeps resident in shared memory
// (one per distinct k stage a CTA visits); a one-token call that needs more
// runs on the four-token tile.
constexpr int kSmallTX1MaxSlots = 8;

// Workspace layout shared by all rungs: a synchronisation area of kSyncBytes
// (the small-T kernels' ticket counters, one int per CTA, which must hold
// zeros when a call starts; every call leaves them zeroed again), followed by
// the rung's scratch.
constexpr size_t kSyncBytes = 4096;
static_assert(kSmallTMaxCtas * sizeof(int) <= kSyncBytes, "sync area");

// Partial row sums of a TT tile's row blocks split between CTAs:
// [kSmallTMaxCtas][2][TT][128] fp32.
size_t smallt_partials_bytes(int tt);
// Scratch after the sync area for a TT tile and K: the partial sums, then
// (TT > 1) the activation blocks built by the prep kernel.
size_t smallt_work_bytes(int tt, int K);
// Rows per CTA row block (the TMA box height).
int smallt_rows(int tt);
// Token tile of a T = 1 call: 1 when the one-token kernel's resident
// activation blocks fit for (K, N) on num_sms SMs, else 4.
int smallt_gemv_tile(int K, int N, int num_sms);
cudaError_t smallt_set_attributes();
// Launch the small-T kernel(s) for tokens [tok0, tok0 + Tt) with Tt <= tt.
// tmW: Wp's tensor map; sync: the zeroed sync area; work:
// smallt_work_bytes(tt, K) bytes.  act: how the activations are staged
// (kActExact: exact bf16 pieces; kActRotated: the same for the
// Hadamard-rotated activations, K % 1024 == 0; kActInt8: per-token int8
// codes, the s8 definition).  Adds the number of kernels launched to
// *launches.
enum : int { kActExact = 0, kActRotated = 1, kActInt8 = 2 };
cudaError_t launch_smallt(int tt, const CUtensorMap* tmW, const uint32_t* Wp,
                          const uint16_t* scales, const uint16_t* x, int* sync, uint8_t* work,
                          float* y, int K, int N, int tok0, int Tt, int num_sms, int act,
                          int* err, cudaStream_t stream, int* launches);

// s8 rung: tiles of 128 weight rows x 128 tokens on tcgen05.
constexpr int kS8TileN = 128;
constexpr int kS8TileT = 128;
constexpr int kS8SmallTileT = 32;  // token tile of the s8 rung for T <= 32
// Chunked last wave of the s8 rung: at most this many group ranges per tile;
// the chunks' partial sums take kS8PartialBytes of workspace after the
// pieces, and their tickets the synchronisation area.
constexpr int kS8FoldWarps = 8;                          // warps folding the accumulators
constexpr int kS8YBoxT = kS8TileT * 4 / kS8FoldWarps;   // tokens per fold warp's output box
constexpr int kS8MaxChunks = 4;

// Work split of the prefill rungs (s8, bf16): P CTAs walk nfull whole tiles,
// then the rest of the tiles as `chunks` group ranges each.  Chunking applies
// when the rest fills at most half a wave, so that a fraction of a tile per
// CTA finishes the call instead of a whole tile on few SMs.
struct TileSplit {
  int P, nfull, chunks;
};
inline TileSplit tile_split(int tiles, int G, int num_sms) {
  TileSplit sp;
  const int rounds = tiles / num_sms;
  const int rest = tiles - rounds * num_sms;
  sp.nfull = tiles;
  sp.chunks = 1;
  if (rest > 0 && 2 * rest <= num_sms) {
    int c = num_sms / rest;
    if (c > kS8MaxChunks) c = kS8MaxChunks;
    if (c > G / 2) c = G / 2;
    if (c >= 2) {
      sp.nfull = rounds * num_sms;
      sp.chunks = c;
    }
  }
  const int items = sp.nfull + (tiles - sp.nfull) * sp.chunks;
  sp.P = items < num_sms ? items : num_sms;
  return sp;
}
// (at most 160 chunk items, each kS8FoldWarps blocks of kS8YBoxT x 32 floats)
constexpr size_t kS8PartialBytes =
    static_cast<size_t>(160) * kS8FoldWarps * kS8YBoxT * 32 * sizeof(float);
cudaError_t s8_set_attributes();
// Token tile the s8 rung uses for T tokens (the pieces' tensor maps' box
// height): kS8SmallTileT for T <= kS8SmallTileT, else kS8TileT.
int s8_token_tile(int T);
// Stage ring of the s8 kernel: 12 for the small token tile; for the 128-token
// tile 4, or kS8DeepStages when the piece blocks (2 T K bytes, all read while
// a wave of CTAs crosses one row block) take more than half of the L2.
constexpr int kS8DeepStages = 6;
int s8_stages(int T, int K, size_t l2_bytes);

// bf16 rung: x reordered for the MMA (xp [T][K] bf16, optionally rotated
// first), then tiles of 128 weight rows x 128 tokens on tcgen05 kind::f16.
// tmW as for s8; tmX: xp as bytes [T][2K], box 128 B x 128 rows, 128-byte
// swizzle; tmY as for s8 (or null).
cudaError_t launch_interleave(const uint16_t* x, uint16_t* xp, int T, int K, int rotate,
                              int num_sms, cudaStream_t stream);
cudaError_t launch_bf16(const CUtensorMap* tmW, const CUtensorMap* tmX, const CUtensorMap* tmY,
                        const uint16_t* scales, float* y, int T, int K, int N, int* tickets,
                        float* partials, int num_sms, int* err, cudaStream_t stream);
cudaError_t bf16_set_attributes();
// tmW: packed weights, box 32 B x kS8TileN rows, no swizzle.  tmP1 / tmP2:
// the two fp8 activation pieces [T][K], box 128 B x s8_token_tile(T) rows,
// 128-byte swizzle.  y: fp32 [T][N], stored directly.  x_scale: [T] floats,
// readable up to T rounded up to 4.
cudaError_t launch_s8(const CUtensorMap* tmW, const CUtensorMap* tmP1, const CUtensorMap* tmP2,
                      const uint16_t* scales, const float* x_scale, float* y, int T, int K, int N,
                      int* tickets, float* partials, int num_sms, size_t l2_bytes, int* err,
                      cudaStream_t stream);

// Launch configuration of a programmatic dependent launch (the kernel may
// start while the previous kernel in the stream finishes; it waits for that
// kernel's results with griddepcontrol.wait).  attr: one attribute slot.
inline cudaLaunchConfig_t pdl_launch_config(cudaLaunchAttribute* attr, dim3 grid, dim3 block,
                                            size_t smem, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Pack and quantise.
cudaError_t launch_pack(const int8_t* W, uint32_t* Wp, int K, int N, int* bad, int num_sms,
                        cudaStream_t stream);
cudaError_t launch_quant_s8(const uint16_t* x, int8_t* q, float* xs, int T, int K,
                            cudaStream_t stream);
// The s8 rung's activations: the int8 codes split into two exact e4m3 pieces.
// rotate: quantise the blockwise Hadamard rotation of x (K % 1024 == 0,
// K <= kRotateMaxK: the rotated row is staged in shared memory).
cudaError_t launch_quant_pieces(const uint16_t* x, uint8_t* p1, uint8_t* p2, float* xs, int T,
                                int K, int rotate, int num_sms, int* err, cudaStream_t stream);
cudaError_t quant_set_attributes();

// Base-3 packed weights (26 bytes per 128-weight group) -> 2-bit codes.
cudaError_t launch_repack_t5(const uint8_t* P, uint32_t* Wp, int K, int N, int* bad,
                             cudaStream_t stream);
// Blockwise (1024) Hadamard rotation of bf16 activations; xr may equal x.
constexpr int kRotBlock = 1024;
// Largest K for which tern_linear can stage rotated activations (the s8
// rung keeps a rotated token row in shared memory).
constexpr int kRotateMaxK = 65536;
cudaError_t launch_rotate_bf16(const uint16_t* x, uint16_t* xr, int T, int K,
                               cudaStream_t stream);

// Diagnostic: one kernel whose bounded wait runs out (which = 0: an mbarrier
// phase nobody completes; 1: a device counter nobody raises) and records the
// timeout in *err.
cudaError_t launch_wait_timeout_probe(int which, int* err, cudaStream_t stream);

}  // namespace tern
