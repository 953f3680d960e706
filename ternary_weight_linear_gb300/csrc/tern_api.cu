// C ABI of the ternary-weight linear layer: argument checks, the T-band
// dispatcher with its environment override and per-rung debug probe, tensor
// map set-up, and the launches.
//
// Dispatcher: the rung map of the "ninfer-perf-tuning" skill page,
// section 2 — T = 1 decode entry, T = 2..8 small-T
// tile, T = 9..16 tiled small-T, T >= 17 int8 "s8" — with env-overridable
// thresholds read once per process, and a probe that prints which rung ran
// (section 2: every reachable branch reports itself), limited by a minimum T
// and a line budget.  Names of the variables are this library's own.
#include <mutex>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "tern.h"
#include "tern_internal.h"

namespace tern {

__device__ int g_device_error;  // one per device (module globals are per device)

// Fixed scratch of tern_linear_small_t_noalloc, one copy per device that loads
// the library.  In host code this name only stands in for the symbol; its
// device address comes from cudaGetSymbolAddress (noalloc_scratch below).
static __device__ __align__(256) uint8_t g_noalloc_scratch[TERN_NOALLOC_SCRATCH_BYTES];

namespace {

// ------------------------------------------------------------------ config
struct Config {
  int forced = -1;      // TERN_RUNG
  int small_t_max = 8;  // TERN_SMALL_T_MAX
  int tiled_max = 16;   // TERN_TILED_MAX
  int s8_min_t = 17;    // TERN_S8_MIN_T
  bool debug = false;   // TERN_DEBUG
  int debug_min_t = 1;  // TERN_DEBUG_MIN_T
  long debug_budget = 1000;  // TERN_DEBUG_BUDGET (lines)
  bool rotate = false;  // TERN_ROTATE: Hadamard-rotate the activations first
  bool prefill_bf16 = false;  // TERN_PREFILL=bf16: the bf16 rung for T >= s8_min_t
  bool decode_int8 = false;   // TERN_DECODE_ACT=int8: int8 activations on the T <= 16 rungs
};

std::mutex g_mu;
Config g_cfg;
bool g_cfg_loaded = false;
long g_debug_lines = 0;

int env_int(const char* name, int dflt) {
  const char* v = getenv(name);
  if (!v || !*v) return dflt;
  char* end = nullptr;
  long x = strtol(v, &end, 10);
  if (end == v) return dflt;
  return static_cast<int>(x);
}

int rung_from_name(const char* v) {
  if (!v || !*v) return -1;
  if (!strcmp(v, "gemv")) return TERN_RUNG_GEMV;
  if (!strcmp(v, "small_t")) return TERN_RUNG_SMALL_T;
  if (!strcmp(v, "small_t_tiled")) return TERN_RUNG_SMALL_T_TILED;
  if (!strcmp(v, "s8")) return TERN_RUNG_S8;
  if (!strcmp(v, "bf16")) return TERN_RUNG_BF16;
  return -1;
}

void load_config_locked() {
  Config c;
  c.forced = rung_from_name(getenv("TERN_RUNG"));
  c.small_t_max = env_int("TERN_SMALL_T_MAX", 8);
  c.tiled_max = env_int("TERN_TILED_MAX", 16);
  c.s8_min_t = env_int("TERN_S8_MIN_T", 17);
  c.debug = env_int("TERN_DEBUG", 0) != 0;
  c.debug_min_t = env_int("TERN_DEBUG_MIN_T", 1);
  c.debug_budget = env_int("TERN_DEBUG_BUDGET", 1000);
  c.rotate = env_int("TERN_ROTATE", 0) != 0;
  {
    const char* pf = getenv("TERN_PREFILL");
    c.prefill_bf16 = pf && !strcmp(pf, "bf16");
    const char* da = getenv("TERN_DECODE_ACT");
    c.decode_int8 = da && !strcmp(da, "int8");
  }
  // keep the bands well formed
  if (c.small_t_max < 1) c.small_t_max = 1;
  if (c.small_t_max > 8) c.small_t_max = 8;
  if (c.tiled_max < c.small_t_max) c.tiled_max = c.small_t_max;
  if (c.tiled_max > 16) c.tiled_max = 16;
  if (c.s8_min_t < 2) c.s8_min_t = 2;
  g_cfg = c;
  g_cfg_loaded = true;
  g_debug_lines = 0;
}

Config config() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_cfg_loaded) load_config_locked();
  return g_cfg;
}

int pick_rung(const Config& c, int T) {
  if (c.forced >= 0) return c.forced;
  if (T >= c.s8_min_t) return c.prefill_bf16 ? TERN_RUNG_BF16 : TERN_RUNG_S8;
  if (T == 1) return TERN_RUNG_GEMV;
  if (T <= c.small_t_max) return TERN_RUNG_SMALL_T;
  return TERN_RUNG_SMALL_T_TILED;  // covers T up to tiled_max and any gap below s8_min_t
}

void probe(const Config& c, int rung, int T, int K, int N) {
  if (!c.debug || T < c.debug_min_t) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_debug_lines >= c.debug_budget) return;
  ++g_debug_lines;
  const bool bw = rung != TERN_RUNG_S8 && rung != TERN_RUNG_BF16;
  fprintf(stderr, "tern: rung=%s T=%d K=%d N=%d%s%s\n", tern_rung_name(rung), T, K, N,
          c.rotate ? " rotated" : "", c.decode_int8 && bw ? " int8" : "");
  fflush(stderr);
}

thread_local int t_last_rung = -1;
thread_local int t_last_launches = 0;

// ------------------------------------------------------------------ device state
constexpr int kMaxDevices = 64;
struct DevState {
  bool ready = false;
  int sms = 0;
  size_t l2 = 0;  // L2 bytes
  int* err = nullptr;
};
DevState g_dev[kMaxDevices];
std::mutex g_dev_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int device_state(DevState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TERN_ENODEV;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevState& d = g_dev[dev];
  if (!d.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return TERN_ENODEV;
    if (prop.major != 10 || prop.minor != 3) return TERN_ENODEV;  // built for sm_103a only
    d.sms = prop.multiProcessorCount;
    d.l2 = static_cast<size_t>(prop.l2CacheSize);
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return TERN_ECUDA;
    d.err = static_cast<int*>(p);
    if (smallt_set_attributes() != cudaSuccess) return TERN_ECUDA;
    if (s8_set_attributes() != cudaSuccess) return TERN_ECUDA;
    if (quant_set_attributes() != cudaSuccess) return TERN_ECUDA;
    if (bf16_set_attributes() != cudaSuccess) return TERN_ECUDA;
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return TERN_ECUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.ready = true;
  }
  *out = &d;
  return TERN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2D uint8 tensor map: inner extent `inner` bytes, `outer` rows, row pitch `pitch` bytes.
int make_map_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch,
                uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TERN_OK : TERN_ECUDA;
}

// 2D fp32 tensor map: `inner` elements per row, `outer` rows, row pitch
// `pitch` bytes (a multiple of 16).
int make_map_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch,
                 uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TERN_OK : TERN_ECUDA;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// s8 scratch: the two fp8 pieces [T][K] each, then x_scale [T] (rounded up to
// 256 bytes, so the kernel may read it in whole 16-byte chunks), then the
// partial sums of the chunked last wave.
size_t s8_workspace_bytes(int T, int K) {
  return 2 * align_up(static_cast<size_t>(T) * K, 256) + align_up(sizeof(float) * T, 256) +
         kS8PartialBytes;
}

// K for which the activations can be staged rotated (whole 1024-wide
// rotation blocks, and a rotated s8 token row fits in shared memory).
bool rotation_shape_ok(int K) { return K % kRotBlock == 0 && K <= kRotateMaxK; }

// How the small-T rungs stage the activations under config c.
int small_t_act(const Config& c) {
  return c.decode_int8 ? kActInt8 : (c.rotate ? kActRotated : kActExact);
}

// Token tile for a rung, the tokens left, K and N: (TT, tokens in this launch).
void small_t_tile(int rung, int left, int K, int N, int num_sms, int* tt, int* take) {
  if (rung == TERN_RUNG_GEMV) {
    *tt = smallt_gemv_tile(K, N, num_sms);
    *take = 1;
  } else if (rung == TERN_RUNG_SMALL_T) {
    *take = left < 8 ? left : 8;
    *tt = *take <= 4 ? 4 : 8;
  } else {
    *take = left < 16 ? left : 16;
    *tt = 16;
  }
}

// ws: workspace whose first kSyncBytes are the zeroed sync area.
int run_small_t(DevState* d, int rung, const uint32_t* Wp, const uint16_t* s, const uint16_t* x,
                float* y, int T, int K, int N, uint8_t* ws, int act, cudaStream_t st,
                int* launches) {
  CUtensorMap tmW;
  int rc = make_map_u8(&tmW, Wp, static_cast<uint64_t>(K) / 4, static_cast<uint64_t>(N),
                       static_cast<uint64_t>(K) / 4, 128, smallt_rows(1),
                       CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != TERN_OK) return rc;
  for (int tok0 = 0; tok0 < T;) {
    int tt = 0, take = 0;
    small_t_tile(rung, T - tok0, K, N, d->sms, &tt, &take);
    if (launch_smallt(tt, &tmW, Wp, s, x, reinterpret_cast<int*>(ws), ws + kSyncBytes, y, K, N,
                      tok0, take, d->sms, act, d->err, st, launches) != cudaSuccess)
      return TERN_ECUDA;
    tok0 += take;
  }
  return TERN_OK;
}

// Scratch of tern_linear_small_t_noalloc for T tokens and K, for any (N,
// device): at T = 1 the call may run on the one-token or the four-token tile.
size_t noalloc_need(int T, int K) {
  size_t w;
  if (T == 1) {
    const size_t a = smallt_work_bytes(1, K), b = smallt_work_bytes(4, K);
    w = a > b ? a : b;
  } else {
    w = smallt_work_bytes(T <= 4 ? 4 : (T <= 8 ? 8 : 16), K);
  }
  return kSyncBytes + w;
}

// Device address of g_noalloc_scratch on the current device, looked up once
// per device with that device current.
uint8_t* g_noalloc_ptr[kMaxDevices] = {};

int noalloc_scratch(uint8_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TERN_ENODEV;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_noalloc_ptr[dev]) {
    uint8_t* p = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_noalloc_scratch) != cudaSuccess)
      return TERN_ECUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return TERN_OK;
}

}  // namespace
}  // namespace tern

using namespace tern;

extern "C" {

const char* tern_rung_name(int rung) {
  switch (rung) {
    case TERN_RUNG_GEMV: return "gemv";
    case TERN_RUNG_SMALL_T: return "small_t";
    case TERN_RUNG_SMALL_T_TILED: return "small_t_tiled";
    case TERN_RUNG_S8: return "s8";
    case TERN_RUNG_BF16: return "bf16";
    default: return "?";
  }
}

const char* tern_status_string(int st) {
  switch (st) {
    case TERN_OK: return "ok";
    case TERN_EINVAL: return "invalid argument";
    case TERN_EALIGN: return "pointer not 16-byte aligned";
    case TERN_ENOSPACE: return "workspace too small";
    case TERN_ENODEV: return "no sm_103 CUDA device current";
    case TERN_ECUDA: return "CUDA runtime error";
    case TERN_ETIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

void tern_reload_env(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  load_config_locked();
}

int tern_select_rung(int T) {
  if (T < 1) return TERN_EINVAL;
  return pick_rung(config(), T);
}

int tern_last_rung_id(void) { return t_last_rung; }
int tern_last_launches(void) { return t_last_launches; }
const char* tern_last_rung(void) { return t_last_rung < 0 ? "none" : tern_rung_name(t_last_rung); }

size_t tern_linear_workspace_bytes(int T, int K, int N) {
  (void)N;
  if (T < 1 || K < 1) return 0;
  // The sync area, then the larger rung scratch: two fp8 activation pieces
  // [T][K] + fp32 x_scale [T] (s8), or the activation blocks of the widest
  // small-T token tile.  Enough for any rung.
  const size_t a = s8_workspace_bytes(T, K);
  const size_t b = smallt_work_bytes(16, K);
  return kSyncBytes + (a > b ? a : b);
}

int tern_pack(const int8_t* W, uint32_t* Wpacked, int K, int N, int* bad_count, void* stream) {
  if (!W || !Wpacked || K <= 0 || N <= 0 || (K % 16) != 0) return TERN_EINVAL;
  if (!aligned16(W) || !aligned16(Wpacked)) return TERN_EALIGN;
  DevState* d = nullptr;
  int rc = device_state(&d);
  if (rc != TERN_OK) return rc;
  return launch_pack(W, Wpacked, K, N, bad_count, d->sms, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? TERN_OK
             : TERN_ECUDA;
}

int tern_repack_t5(const uint8_t* Pt5, uint32_t* Wpacked, int K, int N, int* bad_count,
                   void* stream) {
  if (!Pt5 || !Wpacked || K <= 0 || N <= 0 || (K % 128) != 0) return TERN_EINVAL;
  if (!aligned16(Pt5) || !aligned16(Wpacked)) return TERN_EALIGN;
  DevState* d = nullptr;
  int rc = device_state(&d);
  if (rc != TERN_OK) return rc;
  return launch_repack_t5(Pt5, Wpacked, K, N, bad_count, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? TERN_OK
             : TERN_ECUDA;
}

int tern_rotate_bf16(const uint16_t* x, uint16_t* xr, int T, int K, void* stream) {
  if (!x || !xr || T <= 0 || K <= 0 || (K % kRotBlock) != 0) return TERN_EINVAL;
  if (!aligned16(x) || !aligned16(xr)) return TERN_EALIGN;
  // in place, or no overlap at all
  const uintptr_t a = reinterpret_cast<uintptr_t>(x), b = reinterpret_cast<uintptr_t>(xr);
  const uintptr_t bytes = static_cast<uintptr_t>(T) * static_cast<uintptr_t>(K) * 2u;
  if (a != b && a < b + bytes && b < a + bytes) return TERN_EINVAL;
  DevState* d = nullptr;
  int rc = device_state(&d);
  if (rc != TERN_OK) return rc;
  return launch_rotate_bf16(x, xr, T, K, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? TERN_OK
             : TERN_ECUDA;
}

int tern_quant_act_s8(const uint16_t* x, int8_t* q, float* x_scale, int T, int K, void* stream) {
  if (!x || !q || !x_scale || T <= 0 || K <= 0 || (K % 16) != 0) return TERN_EINVAL;
  if (!aligned16(x) || !aligned16(q) || !aligned16(x_scale)) return TERN_EALIGN;
  DevState* d = nullptr;
  int rc = device_state(&d);
  if (rc != TERN_OK) return rc;
  return launch_quant_s8(x, q, x_scale, T, K, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? TERN_OK
             : TERN_ECUDA;
}

int tern_linear(const uint32_t* Wpacked, const uint16_t* scales, const uint16_t* x, float* y,
                int T, int K, int N, void* workspace, size_t workspace_bytes, void* stream) {
  if (!Wpacked || !scales || !x || !y || T < 1 || N < 1 || K < 128 || (K % 128) != 0)
    return TERN_EINVAL;
  if (!aligned16(Wpacked) || !aligned16(scales) || !aligned16(x) || !aligned16(y))
    return TERN_EALIGN;
  const Config c = config();
  if (c.rotate && !rotation_shape_ok(K)) return TERN_EINVAL;
  const int rung = pick_rung(c, T);
  // the int8 decode variant has no rotated form
  if (c.rotate && c.decode_int8 && rung != TERN_RUNG_S8 && rung != TERN_RUNG_BF16)
    return TERN_EINVAL;
  DevState* d = nullptr;
  int rc = device_state(&d);
  if (rc != TERN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int rotate = c.rotate ? 1 : 0;

  const size_t need = tern_linear_workspace_bytes(T, K, N);
  if (!workspace || workspace_bytes < need) return TERN_ENOSPACE;
  if (!aligned16(workspace)) return TERN_EALIGN;

  int launches = 0;
  switch (rung) {
    case TERN_RUNG_GEMV:
    case TERN_RUNG_SMALL_T:
    case TERN_RUNG_SMALL_T_TILED:
      rc = run_small_t(d, rung, Wpacked, scales, x, y, T, K, N, static_cast<uint8_t*>(workspace),
                       small_t_act(c), st, &launches);
      break;
    case TERN_RUNG_S8: {
      // after the sync area (whose tickets the chunked last wave uses)
      uint8_t* scratch = static_cast<uint8_t*>(workspace) + kSyncBytes;
      const size_t piece = align_up(static_cast<size_t>(T) * K, 256);
      uint8_t* p1 = scratch;
      uint8_t* p2 = scratch + piece;
      float* xs = reinterpret_cast<float*>(scratch + 2 * piece);
      if (launch_quant_pieces(x, p1, p2, xs, T, K, rotate, d->sms, d->err, st) != cudaSuccess)
        return TERN_ECUDA;
      ++launches;
      CUtensorMap tmW, tmP1, tmP2;
      rc = make_map_u8(&tmW, Wpacked, static_cast<uint64_t>(K) / 4, static_cast<uint64_t>(N),
                       static_cast<uint64_t>(K) / 4, 32, kS8TileN, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (rc != TERN_OK) return rc;
      const uint32_t tok = static_cast<uint32_t>(s8_token_tile(T));
      rc = make_map_u8(&tmP1, p1, static_cast<uint64_t>(K), static_cast<uint64_t>(T),
                       static_cast<uint64_t>(K), 128, tok, CU_TENSOR_MAP_SWIZZLE_128B);
      if (rc != TERN_OK) return rc;
      rc = make_map_u8(&tmP2, p2, static_cast<uint64_t>(K), static_cast<uint64_t>(T),
                       static_cast<uint64_t>(K), 128, tok, CU_TENSOR_MAP_SWIZZLE_128B);
      if (rc != TERN_OK) return rc;
      float* partials = reinterpret_cast<float*>(scratch + 2 * piece +
                                                 align_up(sizeof(float) * T, 256));
      rc = launch_s8(&tmW, &tmP1, &tmP2, scales, xs, y, T, K, N, static_cast<int*>(workspace),
                     partials, d->sms, d->l2, d->err, st) == cudaSuccess
               ? TERN_OK
               : TERN_ECUDA;
      ++launches;
      break;
    }
    case TERN_RUNG_BF16: {
      // after the sync area: x reordered for the MMA, 2 T K bytes (within
      // the s8 scratch the workspace size covers)
      uint16_t* xp = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + kSyncBytes);
      if (launch_interleave(x, xp, T, K, rotate, d->sms, st) != cudaSuccess) return TERN_ECUDA;
      ++launches;
      CUtensorMap tmW, tmX;
      rc = make_map_u8(&tmW, Wpacked, static_cast<uint64_t>(K) / 4, static_cast<uint64_t>(N),
                       static_cast<uint64_t>(K) / 4, 32, kS8TileN, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (rc != TERN_OK) return rc;
      rc = make_map_u8(&tmX, xp, 2 * static_cast<uint64_t>(K), static_cast<uint64_t>(T),
                       2 * static_cast<uint64_t>(K), 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
      if (rc != TERN_OK) return rc;
      CUtensorMap tmY;
      const bool y_tma = (N % 4) == 0;
      if (y_tma) {
        rc = make_map_f32(&tmY, y, static_cast<uint64_t>(N), static_cast<uint64_t>(T),
                          static_cast<uint64_t>(N) * 4, 32, kS8YBoxT);
        if (rc != TERN_OK) return rc;
      }
      // the chunked last wave's partial sums: where the s8 rung keeps its own
      float* partials = reinterpret_cast<float*>(
          static_cast<uint8_t*>(workspace) + kSyncBytes +
          2 * align_up(static_cast<size_t>(T) * K, 256) + align_up(sizeof(float) * T, 256));
      rc = launch_bf16(&tmW, &tmX, y_tma ? &tmY : nullptr, scales, y, T, K, N,
                       static_cast<int*>(workspace), partials, d->sms, d->err, st) == cudaSuccess
               ? TERN_OK
               : TERN_ECUDA;
      ++launches;
      break;
    }
    default:
      return TERN_EINVAL;
  }
  if (rc == TERN_OK) {
    t_last_rung = rung;
    t_last_launches = launches;
    probe(c, rung, T, K, N);
  }
  return rc;
}

int tern_linear_small_t_noalloc(const uint32_t* Wpacked, const uint16_t* scales,
                                const uint16_t* x, float* y, int T, int K, int N,
                                void* stream) {
  if (!Wpacked || !scales || !x || !y || T < 1 || T > 16 || N < 1 || K < 128 ||
      (K % 128) != 0)
    return TERN_EINVAL;
  if (!aligned16(Wpacked) || !aligned16(scales) || !aligned16(x) || !aligned16(y))
    return TERN_EALIGN;
  const int rung = T == 1 ? TERN_RUNG_GEMV : T <= 8 ? TERN_RUNG_SMALL_T : TERN_RUNG_SMALL_T_TILED;
  if (noalloc_need(T, K) > TERN_NOALLOC_SCRATCH_BYTES) return TERN_ENOSPACE;
  const Config c = config();
  if (c.rotate && !rotation_shape_ok(K)) return TERN_EINVAL;
  if (c.rotate && c.decode_int8) return TERN_EINVAL;
  DevState* d = nullptr;
  int rc = device_state(&d);
  if (rc != TERN_OK) return rc;
  uint8_t* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc != TERN_OK) return rc;
  int launches = 0;
  rc = run_small_t(d, rung, Wpacked, scales, x, y, T, K, N, scratch, small_t_act(c),
                   static_cast<cudaStream_t>(stream), &launches);
  if (rc == TERN_OK) {
    t_last_rung = rung;
    t_last_launches = launches;
    probe(c, rung, T, K, N);
  }
  return rc;
}

int tern_selftest_wait_timeout(int which, void* stream) {
  if (which != 0 && which != 1) return TERN_EINVAL;
  DevState* d = nullptr;
  int rc = device_state(&d);
  if (rc != TERN_OK) return rc;
  return launch_wait_timeout_probe(which, d->err, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? TERN_OK
             : TERN_ECUDA;
}

int tern_device_status(void* stream) {
  DevState* d = nullptr;
  int rc = device_state(&d);
  if (rc != TERN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return TERN_ECUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return TERN_ECUDA;
  if (v) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return TERN_ECUDA;
    // counters of an interrupted call may be left set in the no-alloc scratch
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
      uint8_t* p = nullptr;
      {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        p = g_noalloc_ptr[dev];
      }
      if (p && cudaMemsetAsync(p, 0, kSyncBytes, st) != cudaSuccess) return TERN_ECUDA;
      if (p && cudaStreamSynchronize(st) != cudaSuccess) return TERN_ECUDA;
    }
    return TERN_ETIMEOUT;
  }
  return TERN_OK;
}

}  // extern "C"
