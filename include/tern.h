/*
 * tern.h — C ABI of the ternary-weight linear layer for one GB300 (sm_103a).
 *
 * The layer computes y = x W^T for ternary weights W in {-1, 0, +1} with one
 * fp16 scale per 128 consecutive weights along K, for T tokens of bf16
 * activations.  Three token bands, each served by its own kernel ("rung"):
 *   T = 1        decode GEMV                           rung "gemv"
 *   T = 2..8     speculative-verify small-T tile       rung "small_t"
 *   T = 9..16    two small-T token tiles per weight    rung "small_t_tiled"
 *   T >= 17      int8 per-token activations ("s8")     rung "s8"
 * The band map, the env override and the per-rung probe follow the rung map
 * and the probe discipline of the "ninfer-perf-tuning" skill page, section 2
 * ("which rung ran" and its rung-map table); the format follows the "NInfer
 * sm_89 fork" write-up, section 9 item 2 (ternary codes plus one FP16 scale
 * per 128 weights; int8 activations with m16n8k32 int8 MMA for prefill).
 *
 * Conventions for every entry point
 *  - All array arguments are DEVICE pointers of the current CUDA device, owned
 *    by the caller.  The library never allocates or frees device memory.
 *  - `stream` is a cudaStream_t (passed as void*; NULL = legacy default
 *    stream).  Calls are asynchronous on that stream and never synchronise.
 *  - Row-major, densely packed layouts; element types are given as bit
 *    patterns so that this header needs no CUDA headers:
 *      bf16 = uint16_t (upper half of an IEEE fp32), fp16 = uint16_t (IEEE
 *      binary16), fp32 = float.
 *  - Every pointer must be 16-byte aligned (TERN_EALIGN otherwise).
 *  - Errors are returned as a negative tern_status; nothing aborts.  Launch
 *    failures return TERN_ECUDA.  Asynchronous device-side failures (a bounded
 *    wait that ran out) are recorded in a per-device error word read by
 *    tern_device_status().
 *
 * Packed weight layout (this library's format; the pages pack base-3 trits
 * five to a byte, this format spends 2 bits per weight on sign and magnitude):
 *   Wpacked is uint32 [N][K/16], i.e. K/4 bytes per row.  Byte b of row n
 *   (little-endian bytes within the words) holds weights k = 4b .. 4b+3.
 *   Weight i of a byte has its "nonzero" bit at bit P[i] and its "negative"
 *   bit at bit P[i] + 2, with P = {0, 1, 4, 5}; each nibble thus reads
 *   [nz_lo, nz_hi, neg_lo, neg_hi] from bit 0 up:
 *       (nz, neg) = (0, 0) -> 0,  (1, 0) -> +1,  (1, 1) -> -1,  (0, 1) invalid.
 *   tern_pack never writes the invalid pair; the linear kernels decode it as 0.
 *   The bit order lets the kernels turn a byte into the fp8 e4m3 encoding of
 *   w/8 with one shift and one AND.
 * Scales: fp16 [N][K/128], scale (n, g) applies to k in [128g, 128g+128).
 */
#ifndef TERN_H_
#define TERN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TERN_OK = 0,
  TERN_EINVAL = -1,   /* bad size / null pointer / unsupported shape */
  TERN_EALIGN = -2,   /* a pointer is not 16-byte aligned */
  TERN_ENOSPACE = -3, /* workspace smaller than tern_linear_workspace_bytes() */
  TERN_ENODEV = -4,   /* no usable sm_103 device current */
  TERN_ECUDA = -5,    /* a CUDA runtime call or launch failed */
  TERN_ETIMEOUT = -6  /* a device-side bounded wait ran out (see tern_device_status) */
} tern_status;

/* Rung identifiers (tern_select_rung / tern_last_rung_id). */
typedef enum {
  TERN_RUNG_GEMV = 0,
  TERN_RUNG_SMALL_T = 1,
  TERN_RUNG_SMALL_T_TILED = 2,
  TERN_RUNG_S8 = 3,
  TERN_RUNG_BF16 = 4  /* exact bf16 prefill rung; chosen by TERN_RUNG=bf16 or,
                         for T >= TERN_S8_MIN_T, TERN_PREFILL=bf16 */
} tern_rung;

/* Pack ternary int8 weights into the 2-bit layout above.
 *   W        device int8 [N][K], values in {-1, 0, +1}
 *   Wpacked  device uint32 [N][K/16], written
 *   K, N     K > 0 and K % 16 == 0; N > 0
 *   bad_count optional device int32; if not NULL, the number of inputs outside
 *            {-1, 0, +1} is ADDED to *bad_count (those inputs are packed as 0).
 * Format: "NInfer sm_89 fork" write-up, section 9 item 2 (ternary codes with
 * per-128 fp16 scales), 2-bit reading of its base-3 digit. */
int tern_pack(const int8_t* W, uint32_t* Wpacked, int K, int N, int* bad_count,
              void* stream);

/* Per-token int8 quantisation of bf16 activations ("s8" rung input).
 *   x        device bf16 [T][K]
 *   q        device int8 [T][K], written: clamp(rint(x / x_scale), -127, 127),
 *            rint = round to nearest even
 *   x_scale  device fp32 [T], written: max_k |x[t][k]| / 127 (IEEE fp32
 *            division); a token whose absmax is 0 gets x_scale 0 and q 0.
 *   T > 0, K > 0, K % 16 == 0.
 * Source: int8 activations for the prefill rung, "NInfer sm_89 fork" write-up
 * section 9 item 2 and the "s8" rung of the "ninfer-perf-tuning" skill page
 * section 2; absmax/127 with round-to-nearest-even is the reading of
 * "quantised per token". */
int tern_quant_act_s8(const uint16_t* x, int8_t* q, float* x_scale, int T,
                      int K, void* stream);

/* Convert base-3 packed weights (five per byte) to the 2-bit layout above.
 *   Pt5      device uint8 [N][K/128][26], read-only.  Each 128-weight group
 *            takes 26 bytes; byte j of a group holds the group's weights
 *            5j .. 5j+4 as the base-3 number sum_i (w_i + 1) * 3^i, the first
 *            weight least significant.  The last byte holds three weights;
 *            its two upper digits are padding and are ignored.  Bytes above
 *            242 are invalid: their weights are written as 0.
 *   Wpacked  device uint32 [N][K/16], written
 *   K, N     K > 0 and K % 128 == 0; N > 0
 *   bad_count optional device int32; if not NULL, the number of invalid bytes
 *            is ADDED to *bad_count.
 * The scales keep their [N][K/128] fp16 array.  This is a one-time,
 * memory-bound conversion for weights stored in the base-3 format; the
 * linear kernels read the 2-bit layout.
 * Format: "NInfer sm_89 fork" write-up, section 9 item 2 (base-3 codes,
 * five weights per byte, one FP16 scale per 128 weights, 1.75 bits per
 * weight: 26 bytes + 2 bytes of scale per 128 weights). */
int tern_repack_t5(const uint8_t* Pt5, uint32_t* Wpacked, int K, int N,
                   int* bad_count, void* stream);

/* Blockwise Hadamard rotation of bf16 activations:
 *   xr[t][1024 b + i] = bf16( 1/32 * sum_j (-1)^popcount(i & j) x[t][1024 b + j] )
 * for each 1024-wide block b of each token t (the orthonormal Sylvester
 * Hadamard matrix of order 1024), computed in fp32 and rounded to bf16 with
 * round-to-nearest-even.  Each output differs from the exact rotation by at
 * most half a bf16 step plus the fp32 sum error bound
 * 10 * 2^-24 * sum_j |x[t][1024 b + j]| / 32, so it is the exact value's own
 * bf16 rounding except where that value lies within the sum bound of a
 * rounding boundary.
 *   x        device bf16 [T][K], read-only
 *   xr       device bf16 [T][K], written; may be x itself (in place),
 *            otherwise it must not overlap x
 *   T > 0, K > 0, K % 1024 == 0.
 * Source: the Hadamard rotation that the "NInfer sm_89 fork" write-up
 * (section 9 item 2) fuses into the activation quantisation, over the
 * (1024-block, token) pairs of the "ninfer-perf-tuning" skill page's
 * section 6 budget table. */
int tern_rotate_bf16(const uint16_t* x, uint16_t* xr, int T, int K,
                     void* stream);

/* Bytes of the synchronisation area at the start of every workspace. */
#define TERN_SYNC_BYTES 4096u

/* Bytes of device workspace tern_linear needs for (T, K, N); the value covers
 * every rung: the synchronisation area, then for the s8 rung the int8 codes
 * split into two fp8 pieces (2 T K bytes) and the token scales, or for the
 * small-T rungs the partial row sums of row blocks that two or more CTAs
 * share and the activation blocks built per call.
 * Host-only; 0 for T < 1 or K < 1. */
size_t tern_linear_workspace_bytes(int T, int K, int N);

/* y = x W^T with group scales:
 *   y[t][n] = sum_g s[n][g] * sum_{k in g} w[n][k] * x[t][k]
 * on the bf16-activation rungs (T <= 16), and on the s8 rung (T >= 17)
 *   q, xs = tern_quant_act_s8(x)
 *   acc[t][n][g] = sum_{k in g} q[t][k] * w[n][k]   (exact integers)
 *   y[t][n]      = xs[t] * sum_g s[n][g] * acc[t][n][g]   (fp32).
 * Precision of the bf16 rungs, for every finite input: each bf16 x is cut
 * into three fp8 e5m2 pieces at a power-of-two scale per token and
 * 128-group, exactly for every element within 21 binades of the group's
 * largest, so those products w * x are formed exactly on the tensor cores.
 * The few elements further down (leftovers) are handled per row block: if
 * the bound s * sum|x| of every leftover group of a row block adds up to at
 * most 2^-11 of the row block's partial sum, they are left out, otherwise
 * they are multiplied exactly on the CUDA cores.  Beside the fp32 sums'
 * rounding the error is therefore at most 2^-11 * sum|s w x|, inside
 * |y - y_exact| <= 1e-3 * sum|s w x| + 1e-6.  Row blocks that need their
 * leftovers added read them twice (extra time, same result).
 * Results are bit-for-bit reproducible from call to call on every rung: rows
 * whose sums several CTAs share are added in a fixed CTA order.
 *   Wpacked  device uint32 [N][K/16] (layout above), read-only
 *   scales   device fp16 [N][K/128], read-only
 *   x        device bf16 [T][K], read-only
 *   y        device fp32 [T][N], written (fully overwritten)
 *   T >= 1, K >= 128 with K % 128 == 0, N >= 1
 *   workspace, workspace_bytes: device scratch of at least
 *            tern_linear_workspace_bytes(T, K, N) bytes, 16-byte aligned
 *            (TERN_ENOSPACE if smaller).  Its first TERN_SYNC_BYTES bytes are
 *            a synchronisation area (ticket counters with which the CTAs of a
 *            launch agree which of them adds up the rows they share; no CTA
 *            ever waits for another) owned by the library: zero it once
 *            before the workspace's first use (e.g. with cudaMemset), then
 *            leave it alone; every call that completes without a device-side
 *            error leaves it zeroed again.  After TERN_ETIMEOUT from
 *            tern_device_status, zero it again.  The rest of the workspace is
 *            scratch whose contents on entry are ignored.  The workspace must
 *            not be used by anything else (nor by another tern_linear call)
 *            until the call's work on `stream` has finished.
 * The small-T kernels use programmatic dependent launch: a kernel may start
 * while the previous kernel on the stream finishes, and it then already
 * reads Wpacked and scales (never x) before that kernel has completed.  So
 * Wpacked and scales must not be written by a kernel that launches its
 * dependents early and may still be running; a kernel launched without
 * programmatic dependent launch (any other library's kernel, and this
 * library's tern_pack and tern_repack_t5) has completed before the next
 * kernel starts.
 * x, y and the workspace are touched only after the previous kernel has
 * completed.
 * With TERN_ROTATE=1 in the environment the layer runs on the blockwise
 * Hadamard rotation of x (the operation of tern_rotate_bf16: each 1024-wide
 * block of each token rotated and rounded once to bf16) instead of x itself,
 * for weights stored in the rotated basis.  Every rung rotates inside its own
 * activation staging (x is never written and no extra call is made); K must
 * then be a multiple of 1024 and at most 65536, else TERN_EINVAL.  The
 * rotation's fp32 sums may round an element the other way where its exact
 * value lies within tern_rotate_bf16's stated bound of a bf16 rounding
 * boundary; otherwise the result is that of tern_linear on tern_rotate_bf16's
 * output.  Source: the rotation the "NInfer sm_89 fork" write-up (section 9
 * item 2) fuses into the activation quantisation.
 * With TERN_DECODE_ACT=int8 the T <= 16 rungs compute the s8 definition
 * instead (per-token int8 codes as tern_quant_act_s8 makes them, exact
 * integer group sums, y = xs * sum_g s * acc, held to the s8 rung's bars):
 * the int8-activation decode path of the "NInfer sm_89 fork" write-up
 * (section 9 item 2).  It has no rotated form (TERN_ROTATE with it:
 * TERN_EINVAL on those rungs).
 * The bf16 rung (TERN_RUNG=bf16, or TERN_PREFILL=bf16 for the s8 band)
 * computes the bf16-rung definition above on tcgen05 kind::f16: weights as
 * bf16 +-1, activations as they are, every product exact, fp32 sums; no
 * activation quantisation (its workspace holds x reordered for the MMA).
 * The rung is chosen from T (see tern_select_rung); TERN_RUNG forces one.
 * Every rung is correct for every T. */
int tern_linear(const uint32_t* Wpacked, const uint16_t* scales,
                const uint16_t* x, float* y, int T, int K, int N,
                void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of the fixed device scratch tern_linear_small_t_noalloc uses. */
#define TERN_NOALLOC_SCRATCH_BYTES (8u << 20)

/* tern_linear for T = 1..16 without a caller workspace and without allocating.
 *
 * The pages have no counterpart of this call; it exists for callers that
 * cannot allocate device memory or hand over a workspace: plug-in interfaces
 * that pass only input and output buffers, engines that reserve all device
 * memory at start-up and forbid allocation afterwards, and latency-critical
 * code where cudaMalloc / cudaFree would synchronise the device.
 *
 *   Wpacked, scales, x, y, T, K, N, stream: as for tern_linear.
 *   1 <= T <= 16 (TERN_EINVAL otherwise).  The rung comes from T alone:
 *   "gemv" at T = 1, "small_t" at T = 2..8, "small_t_tiled" at T = 9..16; the
 *   environment overrides of tern_linear do not apply.
 *
 * Scratch.  The call's workspace (the synchronisation area, partial sums and
 * activation blocks) lives in one file-scope device array of
 * TERN_NOALLOC_SCRATCH_BYTES (8 MiB) inside the library; every GPU that loads
 * the library holds it until the process exits.  A call whose workspace does
 * not fit returns TERN_ENOSPACE before any device work: K <= 479232 for
 * T = 1..4, K <= 219136 for T = 5..8 and K <= 118784 for T = 9..16.  The call
 * allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.
 *
 * Set-up.  The first call on a device (with that device current) looks up the
 * array's device address with cudaGetSymbolAddress and performs the library's
 * per-device set-up (kernel attributes); make that first call before any
 * stream capture.
 *
 * Sharing.  Every call on a device uses the same array, and the array keeps
 * the last call's contents.  The array is zero when the library loads; its
 * synchronisation area is left valid by every call that completes without a
 * device-side error, and every other byte a call reads it has written first,
 * so nothing needs clearing between calls.  When tern_device_status reports
 * TERN_ETIMEOUT it also zeroes the array's synchronisation area on that
 * device.  Calls whose work overlaps on the GPU (e.g. on two streams without
 * ordering between them) race on the array and give wrong results: order
 * them on one stream or with events. */
int tern_linear_small_t_noalloc(const uint32_t* Wpacked, const uint16_t* scales,
                                const uint16_t* x, float* y, int T, int K, int N,
                                void* stream);

/* Diagnostic of the failure path.  Launches one small kernel whose bounded
 * wait can never be satisfied, using the same wait code as the layer's
 * kernels:
 *   which = 0  an mbarrier phase that nothing completes
 *   which = 1  a device counter that nothing raises (a wait in global
 *              memory, the form a wait on another CTA would take)
 * After the wait limit (2 s) the kernel records the timeout in the device
 * error word and returns: nothing faults or hangs, and the context stays
 * usable.  tern_device_status() on the same stream then returns
 * TERN_ETIMEOUT and clears the word.  which outside {0, 1}: TERN_EINVAL.
 * For tests and health checks only; never needed on the layer's path. */
int tern_selftest_wait_timeout(int which, void* stream);

/* Rung the dispatcher picks for T (after env overrides).  Host-only. */
int tern_select_rung(int T);

/* Name of a rung id ("gemv", "small_t", "small_t_tiled", "s8", "bf16"), or "?". */
const char* tern_rung_name(int rung);

/* Rung launched by this thread's last successful tern_linear, or -1 / "none". */
int tern_last_rung_id(void);
const char* tern_last_rung(void);

/* Number of kernels this thread's last successful tern_linear (or
 * tern_linear_small_t_noalloc) launched: per token tile of the bandwidth
 * rungs one main kernel, plus the activation-prep kernel where the tile
 * uses one; 2 on the s8 rung (activation pieces, then the GEMM).  0 before
 * any call.  Host-only; for benchmarks and tests. */
int tern_last_launches(void);

/* Static text for a tern_status. */
const char* tern_status_string(int status);

/* Re-read the environment (TERN_RUNG, TERN_SMALL_T_MAX, TERN_TILED_MAX,
 * TERN_S8_MIN_T, TERN_PREFILL, TERN_ROTATE, TERN_DECODE_ACT, TERN_DEBUG,
 * TERN_DEBUG_MIN_T, TERN_DEBUG_BUDGET).  The
 * environment is otherwise read once per process, on first use. */
void tern_reload_env(void);

/* Synchronises `stream`, then returns and clears the current device's
 * asynchronous error word: TERN_OK, or TERN_ETIMEOUT if a kernel's bounded
 * wait ran out since the last call (in which case it also zeroes the
 * synchronisation area of tern_linear_small_t_noalloc's scratch, if that
 * scratch is set up on this device). */
int tern_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TERN_H_ */
