// Host-side runtime of the library: device error word, device queries
// (once per device), TMA tensor-map encoding, status strings and the
// per-shape route selector.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.h"
#include "host.h"

namespace spg {

namespace {
constexpr int kMaxDevices = 64;
__device__ unsigned int g_error_word;

std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int> g_debug_stall{0};
std::mutex g_mu;
unsigned int* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}
}  // namespace

unsigned int* device_error_word() {
  const int d = current_device();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[d] = static_cast<unsigned int*>(p);
  }
  return g_err_ptr[d];
}

spg_status cuda_status(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return SPG_OK;
  if (std::getenv("SPG_DEBUG")) std::fprintf(stderr, "spg: %s: %s\n", where, cudaGetErrorString(e));
  return SPG_ERR_CUDA;
}

bool debug_stall_enabled() { return g_debug_stall.load(std::memory_order_relaxed) != 0; }

uint64_t wait_timeout_ns() { return g_timeout_ns.load(std::memory_order_relaxed); }

// With no visible device (host-only use of the selector) the GB300 count,
// 152, is assumed.
int num_sms() {
  constexpr int kGb300Sms = 152;
  const int d = current_device();
  if (d < 0) return kGb300Sms;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[d]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0)
      return kGb300Sms;
    g_sms[d] = n;
  }
  return g_sms[d];
}

// ------------------------------------------------------------ tensor maps
namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}
}  // namespace

bool make_tmap_3d(CUtensorMap* out, const void* base, bool bf16, uint64_t d0, uint64_t d1,
                  uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
                  uint32_t box1, int swizzle_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle_bytes == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
  else if (swizzle_bytes == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
  else if (swizzle_bytes == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
  const CUresult r =
      fn(out, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_2d_u32(CUtensorMap* out, const void* base, uint64_t d0, uint64_t d1,
                      uint64_t stride1_bytes, uint32_t box0, uint32_t box1) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  // Encoded with a third dimension of extent 1 so the kernels' 3-D TMA
  // instruction form applies to it as to every other operand.
  const cuuint64_t dims[3] = {d0, d1, 1};
  const cuuint64_t strides[2] = {stride1_bytes, stride1_bytes * d1};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(out, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- routes
// Per-shape selection.  The cost compared is the one the ninfer FP8 route
// model uses ("Routing": waves needed times the work one SM carries through
// a wave), re-derived for 152 SMs and tcgen05 tiles:
//   cost = ceil(tiles / units) * (per-SM tile work) / (per-tile efficiency)
// where a unit is an SM (one-CTA tiles) or an SM pair (two-SM tiles), the
// per-SM tile work is 128 x BN x K (plus a fixed per-tile cost for the
// epilogue tail and pipeline fill) and the efficiencies are the measured
// steady-state tensor-pipe fractions of each tile shape on GB300.  Narrow
// problems therefore fall back to narrower or one-CTA tiles, which is the
// AstrAI "small CTA below a tile-count threshold" rule in the same terms.
namespace {
struct Candidate {
  int block_m, block_n, stages;
  double eff;
  bool mn_b_ok;  // may take an N-major B operand
};
}  // namespace

spg_route select_route_internal(int kind, int64_t T, int64_t N, int64_t K, int epilogue,
                                int64_t batch, bool b_mn_major) {
  spg_route r;
  std::memset(&r, 0, sizeof r);
  r.kind = kind;
  r.acc_buffers = 2;
  r.group_m = 16;
  const int sms = num_sms();
  const int64_t nb = batch > 0 ? batch : 1;
  // SPG_FORCE_VARIANT pins the tile shape for A/B runs and tests:
  // 2sm | 2sm192 | 2sm160 | 2sm128 (pair tiles), 1sm256 | 1sm128 (one CTA).
  const char* forced_name = std::getenv("SPG_FORCE_VARIANT");
  if (forced_name && !*forced_name) forced_name = nullptr;
  const bool force_one_cta =
      forced_name && (!std::strcmp(forced_name, "1sm256") || !std::strcmp(forced_name, "1sm128"));
  if (kind == SPG_KIND_NVFP4) {
    // Two-SM 256x256 pair tile, or the one-CTA 128x128 tile when its waves
    // are cheaper (narrow T: more, smaller tiles spread the weight stream
    // over more SMs).  The one-CTA tile runs at about 0.6 of the pair tile's
    // per-SM rate on GB300.
    const int64_t t2 = ((T + 255) / 256) * ((N + 255) / 256) * nb;
    const int64_t t1 = ((T + 127) / 128) * ((N + 127) / 128) * nb;
    const double w2 = static_cast<double>((t2 + sms / 2 - 1) / (sms / 2)) * 2.0;
    const double w1 = static_cast<double>((t1 + sms - 1) / sms) * 1.0 / 0.6;
    bool one_cta = w1 < w2;
    if (forced_name) one_cta = force_one_cta;
    r.block_m = one_cta ? 128 : 256;
    r.block_n = one_cta ? 128 : 256;
    r.block_k = 256;
    r.stages = 5;
    r.acc_buffers = one_cta ? 2 : 1;
    r.variant = one_cta ? 2 : 0;
  } else {
    // Pair tiles first (widths 256/192/160/128), then one-CTA tiles.  The
    // efficiencies are steady-state tensor-pipe fractions measured on GB300
    // relative to the 256-wide pair tile.
    static const Candidate cands[] = {
        {256, 256, 6, 1.00, true},  {256, 192, 7, 0.87, false}, {256, 160, 7, 0.75, false},
        {256, 128, 8, 0.62, false}, {128, 256, 4, 0.80, true},  {128, 128, 6, 0.62, true},
    };
    constexpr int kCands = sizeof(cands) / sizeof(cands[0]);
    static const char* const kNames[kCands] = {"2sm", "2sm192", "2sm160", "2sm128", "1sm256",
                                               "1sm128"};
    const double kb = static_cast<double>((K + 127) / 128);
    const double fixed = 6.0;  // per-tile fixed cost in 128-deep K blocks
    double best = 1e300;
    int best_i = 0;
    for (int i = 0; i < kCands; ++i) {
      const Candidate& c = cands[i];
      if (forced_name && std::strcmp(forced_name, kNames[i]) != 0) continue;
      if (b_mn_major && !c.mn_b_ok) continue;
      if (epilogue == SPG_EPI_SWIGLU && c.block_n % 64 != 0) continue;
      const int units = c.block_m == 256 ? sms / 2 : sms;
      const int64_t tiles = ((T + c.block_m - 1) / c.block_m) * ((N + c.block_n - 1) / c.block_n) * nb;
      // Whole waves, plus the last partial wave shortened by the tail split
      // of the two-SM kernel (when B is K-major).
      const int ways =
          (c.block_m == 256 && !b_mn_major) ? tail_split_ways(tiles, units, c.block_n, epilogue) : 1;
      const double waves =
          static_cast<double>(tiles / units) + ((tiles % units) ? tail_item_time(ways) : 0.0);
      const double cost = waves * (c.block_n / 128.0) * (kb + fixed) / c.eff;
      if (cost < best * (1.0 - 1e-9)) {
        best = cost;
        best_i = i;
      }
    }
    r.block_m = cands[best_i].block_m;
    r.block_n = cands[best_i].block_n;
    r.stages = cands[best_i].stages;
    r.block_k = 128;
    r.variant = best_i;
  }
  const int64_t tiles = ((T + r.block_m - 1) / r.block_m) * ((N + r.block_n - 1) / r.block_n) * nb;
  r.tiles = tiles;
  const int units = r.block_m == 256 ? sms / 2 : sms;
  int64_t items = tiles;
  if (r.block_m == 256 && kind != SPG_KIND_NVFP4 && !b_mn_major) {
    const int ways = tail_split_ways(tiles, units, r.block_n, epilogue);
    items = tiles - tiles % units + (tiles % units) * ways;
  }
  const int64_t g = items < units ? items : units;
  r.grid = static_cast<int>((g < 1 ? 1 : g) * (r.block_m == 256 ? 2 : 1));
  int stage_bytes, epi_warps = 4;
  if (kind == SPG_KIND_NVFP4 && r.block_m == 256) {
    stage_bytes = 128 * 128 + 128 * 128 + 2048 + 4096;
    epi_warps = 8;
  } else if (kind == SPG_KIND_NVFP4) {
    stage_bytes = 128 * 128 + 128 * 128 + 2048 + 2048;
  } else {
    stage_bytes = 128 * 128 + (r.block_m == 256 ? r.block_n / 2 : r.block_n) * 128;
    if (r.block_m == 256) epi_warps = 4;
  }
  r.smem_bytes = 1024 + r.stages * stage_bytes + epi_warps * 2 * 2048 + 256;
  (void)epilogue;
  return r;
}

}  // namespace spg

using namespace spg;

extern "C" const char* spg_status_string(int s) {
  switch (s) {
    case SPG_OK: return "SPG_OK";
    case SPG_ERR_INVALID_ARG: return "SPG_ERR_INVALID_ARG";
    case SPG_ERR_UNSUPPORTED_SHAPE: return "SPG_ERR_UNSUPPORTED_SHAPE";
    case SPG_ERR_MISALIGNED: return "SPG_ERR_MISALIGNED";
    case SPG_ERR_CUDA: return "SPG_ERR_CUDA";
    case SPG_ERR_TIMEOUT: return "SPG_ERR_TIMEOUT";
    default: return "SPG_ERR_UNKNOWN";
  }
}

extern "C" int spg_version(void) { return 100; }

extern "C" void spg_set_wait_timeout_ns(uint64_t ns) {
  g_timeout_ns.store(ns ? ns : 1, std::memory_order_relaxed);
}

extern "C" void spg_debug_inject_stall(int enable) {
  g_debug_stall.store(enable ? 1 : 0, std::memory_order_relaxed);
}

extern "C" spg_status spg_last_device_error(spg_stream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SPG_ERR_CUDA;
  unsigned int* p = device_error_word();
  if (!p) return SPG_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return SPG_ERR_CUDA;
  if (v != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return SPG_ERR_CUDA;
    return SPG_ERR_TIMEOUT;
  }
  return SPG_OK;
}

extern "C" spg_status spg_last_device_error_code(spg_stream_t stream, uint32_t* code) {
  if (!code) return SPG_ERR_INVALID_ARG;
  *code = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SPG_ERR_CUDA;
  unsigned int* p = device_error_word();
  if (!p) return SPG_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return SPG_ERR_CUDA;
  *code = v;
  if (v != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return SPG_ERR_CUDA;
    return SPG_ERR_TIMEOUT;
  }
  return SPG_OK;
}

extern "C" spg_status spg_select_route(int kind, int64_t T, int64_t N, int64_t K, int epilogue,
                                       int64_t batch, spg_route* out) {
  if (!out || kind < 0 || kind > 2 || T < 0 || N < 0 || K < 0 || batch < 0 || epilogue < 0 ||
      epilogue > 2)
    return SPG_ERR_INVALID_ARG;
  *out = select_route_internal(kind, T, N, K, epilogue, batch, false);
  return SPG_OK;
}
