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

uint32_t next_split_epoch() {
  static std::atomic<uint32_t> counter{0};
  uint32_t e = counter.fetch_add(1, std::memory_order_relaxed) + 1;
  if (e == 0) e = counter.fetch_add(1, std::memory_order_relaxed) + 1;
  return e;
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

// Encoded descriptors are cached: a GEMM call builds 3 to 6 of them, and
// eager calls with the same operands (decode steps, repeated layers) would
// otherwise re-encode them every time.  A descriptor holds nothing but the
// arguments it was encoded from, so an entry is reused exactly when every
// argument matches; a freed and re-allocated buffer at the same address with
// the same shape gets the same, still correct, descriptor.  Direct-mapped,
// kTmapCacheSize entries, one lock.
namespace {
enum TmapType : int { kTmapU8 = 0, kTmapBf16 = 1, kTmapU32 = 2 };

struct TmapKey {
  const void* base;
  uint64_t d0, d1, d2, s1, s2;
  uint32_t b0, b1;
  int type, swizzle;
  bool operator==(const TmapKey& o) const {
    return base == o.base && d0 == o.d0 && d1 == o.d1 && d2 == o.d2 && s1 == o.s1 && s2 == o.s2 &&
           b0 == o.b0 && b1 == o.b1 && type == o.type && swizzle == o.swizzle;
  }
};

struct TmapEntry {
  CUtensorMap map;
  TmapKey key;
  bool valid;
};

constexpr int kTmapCacheSize = 256;
TmapEntry g_tmap_cache[kTmapCacheSize];
std::mutex g_tmap_mu;
std::atomic<uint64_t> g_tmap_hits{0}, g_tmap_misses{0};
std::atomic<int> g_tmap_cache_on{1};

uint32_t tmap_slot(const TmapKey& k) {
  uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
  for (uint64_t v : {k.d0, k.d1, k.d2, k.s1, k.s2, uint64_t(k.b0) << 32 | k.b1,
                     uint64_t(k.type) << 8 | uint64_t(k.swizzle)})
    h = (h ^ v) * 0xBF58476D1CE4E5B9ull;
  return static_cast<uint32_t>(h >> 40) % kTmapCacheSize;
}

bool encode_tmap(CUtensorMap* out, const TmapKey& k) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {k.d0, k.d1, k.d2};
  const cuuint64_t strides[2] = {k.s1, k.s2};
  const cuuint32_t box[3] = {k.b0, k.b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (k.swizzle == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
  else if (k.swizzle == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
  else if (k.swizzle == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
  const CUtensorMapDataType dt = k.type == kTmapBf16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : k.type == kTmapU32 ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                                                      : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return fn(out, dt, 3, const_cast<void*>(k.base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool cached_tmap(CUtensorMap* out, const TmapKey& k) {
  if (!g_tmap_cache_on.load(std::memory_order_relaxed)) return encode_tmap(out, k);
  const uint32_t slot = tmap_slot(k);
  {
    std::lock_guard<std::mutex> lk(g_tmap_mu);
    const TmapEntry& e = g_tmap_cache[slot];
    if (e.valid && e.key == k) {
      *out = e.map;
      g_tmap_hits.fetch_add(1, std::memory_order_relaxed);
      return true;
    }
  }
  if (!encode_tmap(out, k)) return false;
  g_tmap_misses.fetch_add(1, std::memory_order_relaxed);
  std::lock_guard<std::mutex> lk(g_tmap_mu);
  TmapEntry& e = g_tmap_cache[slot];
  e.map = *out;
  e.key = k;
  e.valid = true;
  return true;
}
}  // namespace

bool make_tmap_3d(CUtensorMap* out, const void* base, bool bf16, uint64_t d0, uint64_t d1,
                  uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
                  uint32_t box1, int swizzle_bytes) {
  const TmapKey k{base, d0, d1, d2, stride1_bytes, stride2_bytes, box0, box1,
                  bf16 ? kTmapBf16 : kTmapU8, swizzle_bytes};
  return cached_tmap(out, k);
}

bool make_tmap_2d_u32(CUtensorMap* out, const void* base, uint64_t d0, uint64_t d1,
                      uint64_t stride1_bytes, uint32_t box0, uint32_t box1) {
  // Encoded with a third dimension of extent 1 so the kernels' 3-D TMA
  // instruction form applies to it as to every other operand.
  const TmapKey k{base, d0, d1, 1, stride1_bytes, stride1_bytes * d1, box0, box1, kTmapU32, 0};
  return cached_tmap(out, k);
}

void set_tmap_cache(bool on) {
  g_tmap_cache_on.store(on ? 1 : 0, std::memory_order_relaxed);
  if (!on) {
    std::lock_guard<std::mutex> lk(g_tmap_mu);
    for (TmapEntry& e : g_tmap_cache) e.valid = false;
  }
}

void tmap_cache_stats(uint64_t* hits, uint64_t* misses) {
  *hits = g_tmap_hits.load(std::memory_order_relaxed);
  *misses = g_tmap_misses.load(std::memory_order_relaxed);
}

// ------------------------------------------------------------ forced routes
// SPG_FORCE_VARIANT / SPG_FORCE_TAIL pin a tile shape or a tail split, and
// SPG_FORCE_GROUP_M the rasterization group, for A/B runs and tests.  They are read from the environment once, on first
// use, and again only when spg_debug_reload_env() is called, so the
// selector does no environment lookup per call.
namespace {
struct ForcedRoute {
  char variant[32];
  char tail[16];
  int group_m;  // SPG_FORCE_GROUP_M: m-blocks per rasterization group (0: the default)
};
std::mutex g_forced_mu;
ForcedRoute g_forced;
bool g_forced_loaded = false;

void copy_env(char* dst, size_t n, const char* name) {
  const char* v = std::getenv(name);
  dst[0] = 0;
  if (v) {
    std::strncpy(dst, v, n - 1);
    dst[n - 1] = 0;
  }
}

ForcedRoute forced_route() {
  std::lock_guard<std::mutex> lk(g_forced_mu);
  if (!g_forced_loaded) {
    copy_env(g_forced.variant, sizeof g_forced.variant, "SPG_FORCE_VARIANT");
    copy_env(g_forced.tail, sizeof g_forced.tail, "SPG_FORCE_TAIL");
    const char* gm = std::getenv("SPG_FORCE_GROUP_M");
    g_forced.group_m = gm ? std::atoi(gm) : 0;
    if (g_forced.group_m < 0 || g_forced.group_m > 4096) g_forced.group_m = 0;
    g_forced_loaded = true;
  }
  return g_forced;
}
}  // namespace

void reload_forced_route() {
  std::lock_guard<std::mutex> lk(g_forced_mu);
  g_forced_loaded = false;
}

bool forced_variant_is(const char* name) {
  const ForcedRoute f = forced_route();
  return std::strcmp(f.variant, name) == 0;
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
// Whether the swapped narrow-T tile is the default for this shape (T <= 128
// already checked): its 256-row weight tiles must fit one wave, and above
// T = 16 they must leave at least half of the pairs free for the K split.
// Measured on GB300 (linear / linear_add, with a workspace): N = 5120 and
// 6144 (20, 24 tiles) run 17-30% faster swapped at every T <= 128; N =
// 17408 (68 tiles, no split possible) is faster swapped at T <= 16 (23-25
// against 31 us) and slower above it (25 against 22.5 us).
bool swap_default(int64_t T, int64_t N, int pairs) {
  const int64_t tiles = (N + 255) / 256;
  if (tiles > pairs) return false;
  return T <= 16 || 2 * tiles <= pairs;
}

struct Candidate {
  int block_m, block_n, stages;
  double eff;
  bool mn_b_ok;  // may take an N-major B operand
};
}  // namespace

spg_route select_route_internal(int kind, int64_t T, int64_t N, int64_t K, int epilogue,
                                int64_t batch, bool b_mn_major, bool allow_ksplit,
                                bool allow_swap) {
  spg_route r;
  std::memset(&r, 0, sizeof r);
  r.kind = kind;
  r.acc_buffers = 2;
  // Raster group (256-row blocks per group of the tile order), swept on
  // GB300 at T = 8192 over 4..32: 16 within ~1% of the best for FP8 and the
  // NVFP4 linear_add widths; the 34816-wide NVFP4 SwiGLU ran 680 us at 32
  // against 688 at 16 (its wide rows re-read A less in taller groups).
  r.group_m = (kind == SPG_KIND_NVFP4 && N >= 16384) ? 32 : 16;
  {
    const ForcedRoute f = forced_route();
    if (f.group_m > 0) r.group_m = f.group_m;
  }
  const int sms = num_sms();
  const int pairs = sms / 2;
  const int64_t nb = batch > 0 ? batch : 1;
  // SPG_FORCE_VARIANT pins the tile shape for A/B runs and tests:
  // 2sm | 2sm192 | 2sm160 | 2sm128 (pair tiles), 1sm256 | 1sm128 (one CTA);
  // NVFP4 also 2sm_st | 2sm_cp | 2sm_mc (pair tiles), 1sm_cks | 1sm256_cks
  // (one-CTA tiles, K split inside clusters), gemv, gemv_fused.
  // SPG_FORCE_TAIL = none | n | k pins how the last partial wave is split.
  const ForcedRoute forced = forced_route();
  const char* forced_name = forced.variant[0] ? forced.variant : nullptr;
  const bool force_one_cta =
      forced_name && (!std::strcmp(forced_name, "1sm256") || !std::strcmp(forced_name, "1sm128"));
  const char* forced_tail = forced.tail[0] ? forced.tail : nullptr;
  const bool tail_n_ok = !forced_tail || !std::strcmp(forced_tail, "n");
  const bool tail_k_ok = allow_ksplit && (!forced_tail || !std::strcmp(forced_tail, "k"));
  const bool tail_none_ok = !forced_tail || !std::strcmp(forced_tail, "none");
  const int64_t nkb = kind == SPG_KIND_NVFP4 ? (K / 2 + 127) / 128 : (K + 127) / 128;
  const double kb = static_cast<double>(nkb);
  const double fixed = 6.0;  // per-tile fixed cost in 128-byte-deep K blocks
  KSplit best_ks;
  int best_ways = 1;
  int cluster_split = 1;  // variant 7: CTAs per cluster (K pieces per tile)
  // Swapped pair tile for narrow T (FP8 row-scaled linear / linear_add, and
  // the per-tensor GEMM with both operands K-major; one problem): the weight
  // rows fill the MMA's 256-row M side and the tokens its N side (64 or 128
  // wide), so every staged byte but the small token tile is weight stream,
  // where the unswapped tile stages a 256-row activation tile that is mostly
  // out-of-range padding.  SPG_FORCE_VARIANT = swap pins it; any other
  // forced variant disables it.
  const bool swap_ok = (kind == SPG_KIND_FP8_ROWSCALED || kind == SPG_KIND_FP8_TENSOR) &&
                       allow_swap && nb == 1 && epilogue != SPG_EPI_SWIGLU && !b_mn_major &&
                       T >= 1 && T <= 128;
  const bool swap = swap_ok && (forced_name ? std::strcmp(forced_name, "swap") == 0
                                            : swap_default(T, N, pairs));
  if (swap) {
    r.block_m = 256;
    r.block_n = T <= 64 ? 64 : 128;
    r.block_k = 128;
    const bool add = epilogue == SPG_EPI_ADD;
    r.stages = r.block_n == 64 ? (add ? 9 : 10) : (add ? 7 : 8);
    r.variant = 6;
    r.swap_ab = 1;
    r.tiles = (N + 255) / 256;
    r.split_n = 1;
    r.split_k = 1;
    int64_t items = r.tiles;
    // The K split, priced as for the unswapped pieces at full efficiency
    // (the pieces stream weights).  With fewer weight tiles than pairs every
    // tile is split and the pieces of a tile run as the pairs of one cluster,
    // reduced through distributed shared memory (variant 8, no workspace);
    // otherwise only the last partial wave splits, through a workspace.
    const bool cluster = r.tiles < pairs;
    const bool tail_k_cluster = !forced_tail || !std::strcmp(forced_tail, "k");
    KSplit k = (cluster ? tail_k_cluster : tail_k_ok) ? ksplit_plan(r.tiles, pairs, nkb) : KSplit();
    if (k.split_k > 1 && tail_none_ok && ksplit_piece_time(k, r.block_n) >= kb) k = KSplit();
    if (k.split_k > 1) {
      r.split_k = k.split_k;
      if (cluster)
        r.variant = 8;
      else
        r.workspace_bytes = ksplit_workspace_bytes(k, r.block_n, epilogue);
      items = r.tiles - k.tail_tiles + k.tail_tiles * k.split_k;
    }
    r.grid = static_cast<int>(2 * (items < pairs ? items : pairs));
    r.smem_bytes = 1024 + r.stages * (128 * 128 + r.block_n / 2 * 128) + 4 * 2 * 2048 +
                   (add ? 4 * (r.block_n / 32) * 2048 : 0) + 512;
    return r;
  }
  // NVFP4 at decode-sized T (1-4 tokens): the CUDA-core GEMV (variant 4;
  // two weight rows per warp, 4 warps per CTA; no workspace) where it
  // measured faster than the tile routes on GB300 (us, GEMV / best tile,
  // the one-CTA cluster K split where it applies): linear_add N = 5120,
  // K = 17408: T = 1 24.6 / 24.7, T = 2 28.7 / 26.6, T = 3 / 4 41.0 / 26.6;
  // K = 6144: T = 1-2 14.3 / 18.4, T = 3 / 4 16.4 / 18.4, 18.4 / 18.4;
  // N = 16384, K = 17408: T = 1 55.3 / 61.4, T = 2 67.6 / 61.4; the
  // 34816-wide SwiGLU 39-59 against 37-39.  Hence: N up to 16384, and T = 1
  // or K <= 8192.  SPG_FORCE_VARIANT=gemv pins it, any other forced variant
  // disables it.  Its CTAs hold the decoded activations in shared memory (34
  // bytes per token and 32 K elements), so K is bounded.
  const bool gemv_pays = N <= 16384 && (T == 1 || K <= 8192);
  const int64_t gemv_tt = T;  // token slots of the instance (1 to 4)
  if (kind == SPG_KIND_NVFP4 && nb == 1 && T >= 1 && T <= 4 &&
      gemv_tt * (K / 32) * 34 <= 200 * 1024 &&
      (forced_name ? std::strcmp(forced_name, "gemv") == 0 : gemv_pays)) {
    r.block_m = 1;
    r.block_n = 2;
    r.block_k = 32;
    r.stages = 0;
    r.acc_buffers = 0;
    r.variant = 4;
    r.tiles = N / 2;
    r.grid = static_cast<int>((N / 2 + 3) / 4);
    r.split_n = 1;
    r.split_k = 1;
    r.smem_bytes = static_cast<int32_t>(gemv_tt * (K / 32) * 34);
    return r;
  }
  if (kind == SPG_KIND_NVFP4) {
    // Two-SM 256x256 pair tile (optionally with a K split of its last
    // partial wave), or the one-CTA 128x128 tile when its waves are cheaper
    // (narrow T: more, smaller tiles spread the weight stream over more
    // SMs).  The one-CTA tile runs at about 0.6 of the pair tile's per-SM
    // rate on GB300.
    const int64_t t2 = ((T + 255) / 256) * ((N + 255) / 256) * nb;
    const int64_t t1 = ((T + 127) / 128) * ((N + 127) / 128) * nb;
    const double full2 = static_cast<double>(t2 / pairs);
    double w2 = (t2 % pairs) ? full2 + 1.0 : full2;
    KSplit ks = ksplit_plan(t2, pairs, nkb);
    // With fewer tiles than pairs the split pair tile beats the one-CTA tile
    // only while the pair tile is mostly padding (T <= 128 measured on
    // GB300: 37-41 vs 43 us at T = 16-64, 45-51 vs 43 us at T = 256).
    if (t2 < pairs && T > 128 && !forced_tail) ks = KSplit();
    if (ks.split_k > 1 && tail_k_ok) {
      const double wk = full2 + (ksplit_piece_time(ks, 256) + fixed) / (kb + fixed);
      if (wk < w2 || !tail_none_ok) {
        w2 = wk;
        best_ks = ks;
      }
    }
    w2 *= 2.0;
    const double w1 = static_cast<double>((t1 + sms - 1) / sms) * 1.0 / 0.6;
    bool one_cta = w1 < w2;
    if (forced_name) one_cta = force_one_cta;
    if (one_cta) best_ks = KSplit();
    r.block_m = one_cta ? 128 : 256;
    r.block_n = one_cta ? 128 : 256;
    r.block_k = 256;
    r.stages = 5;
    r.acc_buffers = one_cta ? 2 : 1;
    // Pair tile: scales stored into TMEM by the epilogue warps (variant 3,
    // SPG_FORCE_VARIANT=2sm_st, the default: measured on GB300 it frees the
    // tensor pipe for +5-12% over the copies) or copied by the tensor core
    // (variant 0, 2sm_cp).
    const bool st_scales = forced_name ? std::strcmp(forced_name, "2sm_cp") != 0 : true;
    const bool mc = forced_name && std::strcmp(forced_name, "2sm_mc") == 0;
    r.variant = one_cta ? 2 : (mc ? 5 : (st_scales ? 3 : 0));
    if (r.variant == 5) r.stages = 3;
    // One-CTA tiles whose K is split over the CTAs of a cluster (variant 7,
    // reduced through distributed shared memory, no workspace): 1sm_cks
    // (128 x 128 tiles) or 1sm256_cks (128 x 256).  The 128 x 128 form is
    // the default wherever every tile gets at least two pieces in one wave;
    // measured on GB300 (us, linear_add N = 5120, L2 flushed; against the
    // best other tile route): K = 17408 T = 4-64 24.6-26.6 / 34.8-38.9,
    // T = 128 26.6 / 43.0; K = 6144 T = 64-128 18.4 / 22.5.  The 128 x 256
    // form measured slower wherever both apply (34.8 / 26.6 at T = 64).
    const bool cks128 = forced_name ? !std::strcmp(forced_name, "1sm_cks") : nb == 1;
    const bool cks256 = forced_name && !std::strcmp(forced_name, "1sm256_cks");
    if (cks128 || cks256) {
      const int bn = cks256 ? 256 : 128;
      const int stages = bn == 256 ? 3 : 5;
      const int ring = stages * (128 * 128 + bn * 128 + 2048 + (bn / 128) * 2048);
      const int64_t tiles1 = ((T + 127) / 128) * ((N + bn - 1) / bn) * nb;
      const KSplit cs =
          csplit_plan(tiles1, sms, nkb, 8, bn, epilogue == SPG_EPI_SWIGLU ? 64 : 32, ring);
      if (cs.split_k > 1) {
        r.block_m = 128;
        r.block_n = bn;
        r.stages = stages;
        r.acc_buffers = 1;
        r.variant = 7;
        cluster_split = cs.split_k;
        best_ks = KSplit();
      }
    }
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
    double best = 1e300;
    int best_i = 0;
    for (int i = 0; i < kCands; ++i) {
      const Candidate& c = cands[i];
      if (forced_name && std::strcmp(forced_name, kNames[i]) != 0) continue;
      if (b_mn_major && !c.mn_b_ok) continue;
      if (epilogue == SPG_EPI_SWIGLU && c.block_n % 64 != 0) continue;
      const int units = c.block_m == 256 ? pairs : sms;
      const int64_t tiles = ((T + c.block_m - 1) / c.block_m) * ((N + c.block_n - 1) / c.block_n) * nb;
      const double full = static_cast<double>(tiles / units);
      const bool partial = (tiles % units) != 0;
      // The last partial wave: whole tiles, or (two-SM tiles) split along N
      // (K-major B only) or along K (with a workspace).
      double tail = 1e300;
      int ways = 1;
      KSplit ks;
      if (!partial) {
        tail = 0.0;
      } else {
        if (tail_none_ok || c.block_m != 256) tail = kb + fixed;
        if (c.block_m == 256 && !b_mn_major && tail_n_ok) {
          const int w = tail_split_ways(tiles, units, c.block_n, epilogue);
          if (w > 1 && tail_item_time(w) * (kb + fixed) < tail) {
            tail = tail_item_time(w) * (kb + fixed);
            ways = w;
          }
        }
        if (c.block_m == 256 && tail_k_ok) {
          const KSplit k = ksplit_plan(tiles, units, nkb);
          // With fewer tiles than pairs the pieces stream the weights rather
          // than saturate the tensor pipe, and the narrower tiles' lower
          // MMA efficiency does not show (measured on GB300, T <= 256:
          // 160-wide pieces beat 256-wide ones); cost them at full
          // efficiency (the division by c.eff below is undone).
          const double narrow = tiles < units ? c.eff : 1.0;
          if (k.split_k > 1 && (ksplit_piece_time(k, c.block_n) + fixed) * narrow < tail) {
            tail = (ksplit_piece_time(k, c.block_n) + fixed) * narrow;
            ks = k;
            ways = 1;
          }
        }
        if (tail >= 1e299) continue;  // the forced tail split does not apply
      }
      const double cost = (full * (kb + fixed) + tail) * (c.block_n / 128.0) / c.eff;
      if (cost < best * (1.0 - 1e-9)) {
        best = cost;
        best_i = i;
        best_ways = ways;
        best_ks = ks;
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
  const int units = r.block_m == 256 ? pairs : sms;
  int64_t items = tiles;
  r.split_n = 1;
  r.split_k = 1;
  r.workspace_bytes = 0;
  if (r.block_m == 256 && best_ks.split_k > 1) {
    r.split_k = best_ks.split_k;
    r.workspace_bytes = ksplit_workspace_bytes(best_ks, r.block_n, epilogue);
    items = tiles - best_ks.tail_tiles + best_ks.tail_tiles * best_ks.split_k;
  } else if (r.block_m == 256 && best_ways > 1) {
    r.split_n = best_ways;
    items = tiles - tiles % units + (tiles % units) * best_ways;
  } else if (cluster_split > 1) {
    r.split_k = cluster_split;
    items = tiles * cluster_split;  // one wave: items <= units
  }
  const int64_t g = items < units ? items : units;
  r.grid = static_cast<int>((g < 1 ? 1 : g) * (r.block_m == 256 ? 2 : 1));
  int stage_bytes, epi_warps = 4;
  if (kind == SPG_KIND_NVFP4 && r.block_m == 256) {
    // pair tiles stage half of B per CTA; the multicast tile stages all of it
    stage_bytes = 128 * 128 + (r.variant == 5 ? 2 : 1) * 128 * 128 + 2048 + 4096;
    epi_warps = 8;
  } else if (kind == SPG_KIND_NVFP4) {
    stage_bytes = 128 * 128 + r.block_n * 128 + 2048 + (r.block_n / 128) * 2048;
  } else {
    stage_bytes = 128 * 128 + (r.block_m == 256 ? r.block_n / 2 : r.block_n) * 128;
    if (r.block_m == 256) epi_warps = 4;
  }
  // barrier area: 512 bytes in the two-SM kernels, 256 in the one-CTA ones
  r.smem_bytes = 1024 + r.stages * stage_bytes + epi_warps * 2 * 2048 + (r.block_m == 256 ? 512 : 256);
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

static_assert(sizeof(spg_route) == 72, "spg_route layout (the Python binding mirrors it)");

extern "C" int spg_version(void) { return 200; }

extern "C" void spg_set_wait_timeout_ns(uint64_t ns) {
  g_timeout_ns.store(ns ? ns : 1, std::memory_order_relaxed);
}

extern "C" void spg_debug_reload_env(void) { reload_forced_route(); }

extern "C" void spg_debug_set_tmap_cache(int enable) { set_tmap_cache(enable != 0); }

extern "C" void spg_debug_tmap_cache_stats(uint64_t* hits, uint64_t* misses) {
  if (hits && misses) tmap_cache_stats(hits, misses);
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
  *out = select_route_internal(kind, T, N, K, epilogue, batch, false, false);
  return SPG_OK;
}

extern "C" spg_status spg_select_route_ws(int kind, int64_t T, int64_t N, int64_t K,
                                          int epilogue, int64_t batch, spg_route* out) {
  if (!out || kind < 0 || kind > 2 || T < 0 || N < 0 || K < 0 || batch < 0 || epilogue < 0 ||
      epilogue > 2)
    return SPG_ERR_INVALID_ARG;
  *out = select_route_internal(kind, T, N, K, epilogue, batch, false, true);
  return SPG_OK;
}

extern "C" int64_t spg_gemm_workspace_bytes(int kind, int64_t T, int64_t N, int64_t K,
                                            int epilogue, int64_t batch) {
  if (kind < 0 || kind > 2 || T <= 0 || N <= 0 || K <= 0 || batch < 0 || epilogue < 0 ||
      epilogue > 2)
    return 0;
  const int64_t b = select_route_internal(kind, T, N, K, epilogue, batch, false, true).workspace_bytes;
  if (kind != SPG_KIND_FP8_TENSOR) return b;
  // Per-tensor GEMM: enough for either B layout and for an M-major A (which
  // never takes the swapped tile).
  const int64_t n = select_route_internal(kind, T, N, K, epilogue, batch, true, true).workspace_bytes;
  const int64_t u =
      select_route_internal(kind, T, N, K, epilogue, batch, false, true, false).workspace_bytes;
  const int64_t m = b > n ? b : n;
  return m > u ? m : u;
}
