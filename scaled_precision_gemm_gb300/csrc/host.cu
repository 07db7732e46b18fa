// Host-side runtime of the library: device error word, device queries
// (once per device), TMA tensor-map encoding, status strings and the
// per-shape route selector.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "common.h"
#include "host.h"

namespace spg {

namespace {
constexpr int kMaxDevices = 64;
__device__ unsigned int g_error_word;

std::atomic<uint64_t> g_timeout_ns{2000000000ull};
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

// ---------------------------------------------------------------- routes
// Per-shape selection.  The cost compared is the one the ninfer FP8 route
// model uses ("Routing": waves needed times the work one SM carries through
// a wave), re-derived for 152 SMs and tcgen05 tiles: for each candidate tile
// width, time ~ ceil(tiles / SMs) * (tile work + fixed per-tile cost), and
// the cheapest wins.  Narrow problems (fewer tiles than SMs) prefer the
// narrower tile, which is the AstrAI "small CTA below a tile-count
// threshold" rule in the same terms.
spg_route select_route_internal(int kind, int64_t T, int64_t N, int64_t K, int epilogue,
                                int64_t batch) {
  spg_route r;
  std::memset(&r, 0, sizeof r);
  r.kind = kind;
  r.block_m = 128;
  r.acc_buffers = 2;
  const int sms = num_sms();
  const int64_t mblocks = (T + 127) / 128;
  auto tiles_for = [&](int bn) { return mblocks * ((N + bn - 1) / bn) * (batch > 0 ? batch : 1); };
  int bn = 256;
  if (kind == SPG_KIND_NVFP4) {
    bn = 128;
  } else {
    // Candidate widths 256 and 128: waves x (per-tile MMA work + a fixed
    // per-tile overhead of about 1/8 of a 256-wide K=4096 tile).
    const double kb = static_cast<double>((K + 127) / 128);
    const double overhead = 4.0;  // in units of one 128x128x128 MMA block
    double best = 1e300;
    for (int cand : {256, 128}) {
      const int64_t tiles = tiles_for(cand);
      const int64_t waves = (tiles + sms - 1) / sms;
      const double cost = static_cast<double>(waves) * (kb * (cand / 128) + overhead);
      if (cost < best - 1e-9) {
        best = cost;
        bn = cand;
      }
    }
  }
  r.block_n = bn;
  r.block_k = (kind == SPG_KIND_NVFP4) ? 256 : 128;
  if (kind == SPG_KIND_NVFP4)
    r.stages = 5;
  else
    r.stages = (bn == 256) ? 4 : 6;
  r.group_m = 16;
  r.tiles = tiles_for(bn);
  r.grid = static_cast<int>(r.tiles < sms ? r.tiles : sms);
  if (r.grid < 1) r.grid = 1;
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

extern "C" spg_status spg_select_route(int kind, int64_t T, int64_t N, int64_t K, int epilogue,
                                       int64_t batch, spg_route* out) {
  if (!out || kind < 0 || kind > 2 || T < 0 || N < 0 || K < 0 || batch < 0 || epilogue < 0 ||
      epilogue > 2)
    return SPG_ERR_INVALID_ARG;
  *out = select_route_internal(kind, T, N, K, epilogue, batch);
  return SPG_OK;
}
