// Launch helper shared by the GEMM entry points: one function per compiled
// kernel variant, setting the dynamic shared-memory limit once per device.
#pragma once

#include <atomic>

#include "gemm_kernel.cuh"
#include "gemm_kernel_2sm.cuh"
#include "gemm_kernel_nvfp4_2sm.cuh"
#include "gemm_kernel_nvfp4_2sm_st.cuh"
#include "gemm_kernel_nvfp4_mc.cuh"
#include "host.h"

namespace spg {

struct GemmMaps {
  CUtensorMap a, b, y;
  CUtensorMap sfa, sfb;  // NVFP4 two-SM kernel only
  CUtensorMap b_narrow;  // two-SM FP8 kernel: B box of a tail-split item
  CUtensorMap r;         // linear_add residual, 32 x 32 boxes (two-SM kernels; else a copy of y)
};

template <int KIND, int EPI, int BN, int STAGES, bool A_MN, bool B_MN, int SCALE>
spg_status launch_gemm_variant(const GemmMaps& maps, const GemmParams& p, int grid,
                               cudaStream_t stream) {
  using Cfg = GemmCfg<KIND, EPI, BN, STAGES, A_MN, B_MN, SCALE>;
  auto kern = gemm_kernel<KIND, EPI, BN, STAGES, A_MN, B_MN, SCALE>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPG_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    if (cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes),
                    "cudaFuncSetAttribute") != SPG_OK)
      return SPG_ERR_CUDA;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(maps.a, maps.b, maps.y, p);
  return launch_status();
}

// One-CTA variant with the K split inside clusters: clusters of p.split_k
// CTAs, grid = p.total_items (one piece per CTA).
template <int KIND, int EPI, int BN, int STAGES, bool A_MN, bool B_MN, int SCALE>
spg_status launch_gemm_csplit_variant(const GemmMaps& maps, const GemmParams& p,
                                      cudaStream_t stream) {
  using Cfg = GemmCfg<KIND, EPI, BN, STAGES, A_MN, B_MN, SCALE, 1>;
  auto kern = gemm_kernel<KIND, EPI, BN, STAGES, A_MN, B_MN, SCALE, true>;
  if (p.split_k < 2 || p.split_k > kMaxClusterSplit || p.split_full != 0 ||
      p.total_items != p.total_tiles * p.split_k ||
      cluster_recv_bytes(BN, Cfg::kAccColsPerChunk, p.split_k) > STAGES * Cfg::kStageBytes)
    return SPG_ERR_INVALID_ARG;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPG_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    if (cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes),
                    "cudaFuncSetAttribute") != SPG_OK)
      return SPG_ERR_CUDA;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.total_items), 1, 1);
  cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.split_k);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cuda_status(cudaLaunchKernelEx(&cfg, kern, maps.a, maps.b, maps.y, p),
                  "cudaLaunchKernelEx") != SPG_OK)
    return SPG_ERR_CUDA;
  return launch_status();
}

// K split of every tile inside clusters (route variant 7): the plan the
// selector made for this shape.
inline void plan_cluster_items(GemmParams& p, const spg_route& r, int ring_bytes, int cw) {
  const KSplit k = csplit_plan(p.total_tiles, num_sms(), p.num_k_blocks, 8, r.block_n, cw,
                               ring_bytes);
  if (k.split_k != r.split_k) return;  // leaves an unsplit plan: the launcher refuses it
  p.split_k = k.split_k;
  p.kb_per_split = k.kb_per_split;
  p.split_full = 0;
  p.total_items = p.total_tiles * k.split_k;
}

// K split of every tile of a swapped pair schedule inside clusters (route
// variant 8): the selector's plan, one piece per pair.
inline void plan_pair_cluster_items(GemmParams& p, const spg_route& r, int pairs) {
  const KSplit k = ksplit_plan(p.total_tiles, pairs, p.num_k_blocks);
  if (k.split_k != r.split_k || k.tail_tiles != p.total_tiles) return;  // the launcher refuses
  p.split_k = k.split_k;
  p.kb_per_split = k.kb_per_split;
  p.split_full = 0;
  p.total_items = p.total_tiles * k.split_k;
}

// Two-SM variant: clusters of 2 CTAs, grid = 2 x pairs.  CSPLIT (swapped
// tile): clusters of 2 x p.split_k CTAs, one K piece per pair, every tile
// split (grid = 2 x p.total_items).
template <int EPI, int BN, int STAGES, bool A_MN, bool B_MN, int SCALE, bool SWAP = false,
          bool CSPLIT = false>
spg_status launch_gemm_2sm_variant(const GemmMaps& maps, const GemmParams& p, int grid,
                                   cudaStream_t stream) {
  using Cfg = Gemm2smCfg<EPI, BN, STAGES, A_MN, B_MN, SCALE, SWAP, CSPLIT>;
  auto kern = gemm_kernel_2sm<EPI, BN, STAGES, A_MN, B_MN, SCALE, SWAP, CSPLIT>;
  if (CSPLIT && (p.split_k < 2 || 2 * p.split_k > 8 || p.split_full != 0 ||
                 p.total_items != p.total_tiles * p.split_k || grid != 2 * p.total_items ||
                 cluster_recv_bytes(BN, 32, p.split_k) > STAGES * Cfg::kStageBytes))
    return SPG_ERR_INVALID_ARG;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPG_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    if (cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes),
                    "cudaFuncSetAttribute") != SPG_OK)
      return SPG_ERR_CUDA;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CSPLIT ? static_cast<unsigned>(2 * p.split_k) : 2u;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cuda_status(cudaLaunchKernelEx(&cfg, kern, maps.a, maps.b, maps.y, maps.b_narrow, maps.r, p),
                  "cudaLaunchKernelEx") != SPG_OK)
    return SPG_ERR_CUDA;
  return launch_status();
}

// Two-SM NVFP4 variant (clusters of 2 CTAs).
template <int EPI, int STAGES, bool HAS_BIAS>
spg_status launch_nvfp4_2sm_variant(const GemmMaps& maps, const GemmParams& p, int grid,
                                    cudaStream_t stream) {
  using Cfg = Nvfp4PairCfg<EPI, STAGES>;
  auto kern = gemm_kernel_nvfp4_2sm<EPI, STAGES, HAS_BIAS>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPG_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    if (cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes),
                    "cudaFuncSetAttribute") != SPG_OK)
      return SPG_ERR_CUDA;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cuda_status(cudaLaunchKernelEx(&cfg, kern, maps.a, maps.b, maps.y, maps.sfa, maps.sfb, p),
                  "cudaLaunchKernelEx") != SPG_OK)
    return SPG_ERR_CUDA;
  return launch_status();
}

// Two-SM NVFP4 variant whose scale factors are written into TMEM by warps.
template <int EPI, int STAGES, bool HAS_BIAS>
spg_status launch_nvfp4_2sm_st_variant(const GemmMaps& maps, const GemmParams& p, int grid,
                                       cudaStream_t stream) {
  using Cfg = Nvfp4StCfg<EPI, STAGES>;
  auto kern = gemm_kernel_nvfp4_2sm_st<EPI, STAGES, HAS_BIAS>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPG_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    if (cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes),
                    "cudaFuncSetAttribute") != SPG_OK)
      return SPG_ERR_CUDA;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cuda_status(cudaLaunchKernelEx(&cfg, kern, maps.a, maps.b, maps.y, maps.sfa, maps.sfb,
                                     maps.r, p),
                  "cudaLaunchKernelEx") != SPG_OK)
    return SPG_ERR_CUDA;
  return launch_status();
}

// NVFP4 on clusters of two sharing B by multicast, one-CTA MMAs.
template <int EPI, int STAGES, bool HAS_BIAS>
spg_status launch_nvfp4_mc_variant(const GemmMaps& maps, const GemmParams& p, int grid,
                                   cudaStream_t stream) {
  using Cfg = Nvfp4McCfg<EPI, STAGES>;
  auto kern = gemm_kernel_nvfp4_mc<EPI, STAGES, HAS_BIAS>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPG_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    if (cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes),
                    "cudaFuncSetAttribute") != SPG_OK)
      return SPG_ERR_CUDA;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cuda_status(cudaLaunchKernelEx(&cfg, kern, maps.a, maps.b, maps.y, maps.sfa, maps.sfb,
                                     maps.r, p),
                  "cudaLaunchKernelEx") != SPG_OK)
    return SPG_ERR_CUDA;
  return launch_status();
}

template <int KIND, int EPI, int BN, int STAGES, bool A_MN, bool B_MN, int SCALE>
constexpr int variant_smem() {
  return GemmCfg<KIND, EPI, BN, STAGES, A_MN, B_MN, SCALE>::kSmemBytes;
}

// Fill the parts of GemmParams every entry point shares.
inline void fill_common_params(GemmParams& p, const spg_route& r, int64_t M, int64_t N,
                               int64_t K_bytes, int64_t K, int64_t n_out, int64_t batch) {
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.n_out = static_cast<int>(n_out);
  p.num_m_blocks = static_cast<int>((M + r.block_m - 1) / r.block_m);
  p.num_n_blocks = static_cast<int>((N + r.block_n - 1) / r.block_n);
  p.num_k_blocks = static_cast<int>((K_bytes + 127) / 128);
  p.tiles_per_batch = p.num_m_blocks * p.num_n_blocks;
  p.total_tiles = static_cast<int>(p.tiles_per_batch * batch);
  p.group_m = r.group_m;
  p.a_batch_mul = 0;
  p.b_batch_mul = 0;
  p.row_scale = p.col_scale = p.scalar_a = p.scalar_b = nullptr;
  p.residual = nullptr;
  p.bias = nullptr;
  p.bias_scale = nullptr;
  p.bias_kind = 0;
  p.sfa = p.sfb = nullptr;
  p.sf_tiles_per_row_block = 0;
  p.split_full = p.total_tiles;
  p.split_ways = 1;
  p.split_k = 1;
  p.kb_per_split = p.num_k_blocks;
  p.total_items = p.total_tiles;
  p.ws_partial = nullptr;
  p.ws_counter = nullptr;
  p.epoch = 0;
  p.timeout_ns = wait_timeout_ns();
  // Exit waits keep a generous bound even under a short pipeline bound, so a
  // CTA never leaves with a copy or an MMA still writing its memory.
  p.drain_ns = p.timeout_ns > 1000000000ull ? p.timeout_ns : 1000000000ull;
  p.debug_stall = debug_stall_enabled() ? 1 : 0;
  p.err = device_error_word();
}

constexpr int64_t kMaxDim = 0x7FFFFFFF;

// Fused bias arguments: none, bf16 [N] (bias_scale == nullptr) or E4M3 codes
// [N] times the device scalar bias_scale.
inline spg_status set_bias(GemmParams& p, const void* bias, const float* bias_scale) {
  if (!bias) {
    if (bias_scale) return SPG_ERR_INVALID_ARG;
    return SPG_OK;
  }
  if (!aligned16(bias) || (bias_scale && !aligned16(bias_scale))) return SPG_ERR_MISALIGNED;
  p.bias = bias;
  p.bias_scale = bias_scale;
  p.bias_kind = bias_scale ? 2 : 1;
  return SPG_OK;
}

// Work items of a two-SM schedule (`units` CTA pairs) from the route's plan
// for its last partial wave: whole tiles, then that wave's tiles split
// r.split_n ways along N, or r.split_k ways along K with their partial sums
// and arrival counters in `workspace` (at least r.workspace_bytes).
inline void plan_items(GemmParams& p, const spg_route& r, int units, void* workspace) {
  const int tiles = p.total_tiles;
  if (r.split_k > 1) {
    const KSplit k = ksplit_plan(tiles, units, p.num_k_blocks);  // the selector's plan
    p.split_k = k.split_k;
    p.kb_per_split = k.kb_per_split;
    p.split_full = tiles - static_cast<int>(k.tail_tiles);
    p.total_items = p.split_full + static_cast<int>(k.tail_tiles) * k.split_k;
    p.ws_partial = static_cast<float*>(workspace);
    p.ws_counter = reinterpret_cast<unsigned long long*>(
        static_cast<char*>(workspace) + k.tail_tiles * k.split_k * 2 * 128 * int64_t(r.block_n) * 4);
    p.epoch = next_split_epoch();
  } else if (r.split_n > 1) {
    p.split_ways = r.split_n;
    p.split_full = tiles - tiles % units;
    p.total_items = p.split_full + (tiles - p.split_full) * p.split_ways;
  }
}

// Route of a GEMM entry point: with a workspace the last partial wave may be
// split along K, if the workspace is large enough for the plan.
inline spg_route route_for(int kind, int64_t T, int64_t N, int64_t K, int epilogue, int64_t batch,
                           bool b_mn, const void* workspace, int64_t workspace_bytes,
                           bool allow_swap = true) {
  spg_route r = select_route_internal(kind, T, N, K, epilogue, batch, b_mn, workspace != nullptr,
                                      allow_swap);
  if (r.workspace_bytes > workspace_bytes)
    r = select_route_internal(kind, T, N, K, epilogue, batch, b_mn, false, allow_swap);
  return r;
}

}  // namespace spg
