// NVFP4 GEMV for decode-sized T (T <= 4) on the CUDA cores, sm_103a.
//
// With a handful of tokens the NVFP4 GEMM is a stream of weight codes: a
// tensor-core tile would pad T to 128 rows and wait on its pipeline's fill
// and finish.  Here one warp owns two consecutive weight rows (a SwiGLU
// gate/up pair) and its lanes walk K in 32-element chunks (16 code bytes =
// two 16-element scale blocks), four chunks in flight per lane.
//
// Arithmetic: an E2M1 code becomes an int8 holding twice its value (a
// 16-entry table applied to four codes at a time with byte permutes; the
// activations once per CTA into shared memory, the weights as they stream),
// so a block's dot product sum_i (2 a_i)(2 w_i) is an exact integer (dp4a).  It
// is multiplied by the product of the two blocks' E4M3 scales (exact in
// fp32) and accumulated in fp32; the lanes' sums are added across the warp
// and scaled by 1/4.  The epilogue then applies gA * gW, the bias, and the
// residual or SwiGLU in the order of the tensor-core epilogue.  Relative to
// the tile kernels only the fp32 summation order differs.
//
// Scale reads follow the blocked layout (512-byte tiles of 128 rows x 64 K
// elements; row r, block b at ((r / 128) * K/64 + b / 4) * 512 + (r % 32) *
// 16 + ((r % 128) / 32) * 4 + b % 4): the two blocks of a chunk are one
// aligned 16-bit load.
#pragma once

#include <cuda_bf16.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "common.h"
#include "nvfp4_encode.cuh"
#include "ptx.cuh"

namespace spg {

struct GemvParams {
  const uint8_t* A;    // [T, K/2] codes
  const uint8_t* sfA;  // blocked scales of A
  const float* gA;
  // bf16 [T, K] activations, or nullptr.  When set, A / sfA / gA are unused:
  // every CTA quantizes X itself (global scale, block scales, codes) into
  // its shared memory, so the GEMV is the whole quantize-and-multiply
  // operator in one launch.
  const __nv_bfloat16* X;
  const uint8_t* W;    // [N, K/2] codes
  const uint8_t* sfW;  // blocked scales of W
  const float* gW;
  const void* bias;          // per weight row, or nullptr
  const float* bias_scale;   // bias_kind 2
  int bias_kind;             // 0 none, 1 bf16, 2 E4M3 x bias_scale
  const __nv_bfloat16* residual;  // [T, N] (linear_add)
  __nv_bfloat16* Y;               // [T, n_out]
  int T, N, K, n_out;
};

// Four E2M1 codes (16 bits, element i in nibble i) -> four int8 holding
// twice the values (element i in byte i).
__device__ __forceinline__ uint32_t e2m1x4_to_s8x2(uint32_t codes16) {
  const uint32_t mag = codes16 & 0x7777u;
  // twice the magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 and their negatives
  const uint32_t pos = __byte_perm(0x03020100u, 0x0C080604u, mag);
  const uint32_t neg = __byte_perm(0xFDFEFF00u, 0xF4F8FAFCu, mag);
  // byte i from neg (selector i + 4) where the code's sign bit is set
  return __byte_perm(pos, neg, 0x3210u | ((codes16 >> 1) & 0x4444u));
}

// 32 codes (one 16-byte chunk) -> 8 words of int8 (block 0 in q[0..3],
// block 1 in q[4..7]).
__device__ __forceinline__ void decode_chunk(const uint4& v, uint32_t (&q)[8]) {
  q[0] = e2m1x4_to_s8x2(v.x & 0xFFFFu);
  q[1] = e2m1x4_to_s8x2(v.x >> 16);
  q[2] = e2m1x4_to_s8x2(v.y & 0xFFFFu);
  q[3] = e2m1x4_to_s8x2(v.y >> 16);
  q[4] = e2m1x4_to_s8x2(v.z & 0xFFFFu);
  q[5] = e2m1x4_to_s8x2(v.z >> 16);
  q[6] = e2m1x4_to_s8x2(v.w & 0xFFFFu);
  q[7] = e2m1x4_to_s8x2(v.w >> 16);
}

// Byte offset of row r's scale tile base in the blocked layout (chunk 0).
__device__ __forceinline__ int gemv_sf_row_offset(int r, int kt) {
  return (r >> 7) * kt * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
}

__device__ __forceinline__ float gemv_bias(const GemvParams& p, int n) {
  if (p.bias_kind == 1)
    return __uint_as_float(uint32_t(__ldg(static_cast<const unsigned short*>(p.bias) + n)) << 16);
  const uint16_t c = __ldg(static_cast<const uint8_t*>(p.bias) + n);
  return __fmul_rn(e4m3x2_to_float2(uint16_t(c | (c << 8))).x, __ldg(p.bias_scale));
}

// CTAs per cluster of the operator form (bf16 activations quantized in the
// kernel): the cluster shares one quantization of X through distributed
// shared memory.  The kernel reads the cluster size it was launched with
// (at most kGemvMaxCluster).
constexpr int kGemvCluster = 4;  // measured against 8 on GB300: equal or faster on every decode shape
constexpr int kGemvMaxCluster = 8;

// Shared-memory bytes of the decoded activations of one CTA: per token two
// planes of K/32 16-byte words (the int8 of each chunk's two blocks) and
// K/32 pairs of E4M3 scale codes (decoded where they are used: kept as
// codes, four tokens at K = 17408 fit three CTAs per SM instead of two).
__host__ __device__ constexpr int64_t gemv_smem_bytes(int tt, int64_t K) {
  return int64_t(tt) * (K / 32) * 34;
}

__device__ __forceinline__ void st_cluster_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared::cluster.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// TT: tokens the instantiation holds (1 to 4); p.T <= TT.  Grid: one
// warp per pair of weight rows, 4 warps per CTA.  The CTA first decodes the
// activations once into shared memory (they are read by every row).
template <int EPI, int TT>
__global__ void __launch_bounds__(128, 5) gemv_nvfp4_kernel(const GemvParams p) {
  constexpr int kUnroll = 4;
  extern __shared__ uint4 gemv_smem[];
  const int lane = threadIdx.x & 31;
  const int kh = p.K / 2;
  const int nchunks = p.K / 32;
  const int kt = p.K / 64;
  uint4* aq_s = gemv_smem;  // [TT][2][nchunks]
  // [TT][nchunks] pairs of E4M3 scale codes (low byte: the chunk's first block)
  uint16_t* sa_s = reinterpret_cast<uint16_t*>(gemv_smem + 2 * TT * nchunks);
  __shared__ float red_s[4];
  __shared__ float amax_s[kGemvMaxCluster];
  float g_act = 0.f;
  if (p.X) {
    // The operator form, launched in clusters of ncta CTAs: CTA `rank`
    // takes every ncta-th share of X.  (1) Each CTA's share
    // maximum goes to every CTA of the cluster; after a cluster barrier all
    // of them hold the same global scale.  (2) Each CTA encodes its share
    // of the 32-element chunks exactly as the block quantizer does, decodes
    // them, and stores the int8 planes and block scales into the shared
    // memory of every CTA of the cluster; a second barrier publishes them.
    // A cluster spans the whole of X, so each cluster quantizes X once.
    const uint32_t rank = cluster_ctarank();
    const int ncta = int(cluster_nctarank());
    {
      // Start the warp's first two weight rows (contiguous) on their way
      // into L2 while the activations are quantized.
      const int pair0 = blockIdx.x * 4 + (threadIdx.x >> 5);
      if (pair0 * 2 < p.N) {
        const uint8_t* rows = p.W + int64_t(pair0) * 2 * kh;
        for (int off = lane * 128; off < 2 * kh; off += 32 * 128)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(rows + off));
      }
    }
    const uint4* xv = reinterpret_cast<const uint4*>(p.X);
    const int nvec = p.T * (p.K / 8);
    float a = 0.f;
    for (int i = int(rank) * blockDim.x + threadIdx.x; i < nvec; i += ncta * blockDim.x)
      a = fmaxf(a, bf16x8_amax(__ldg(xv + i)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) red_s[threadIdx.x >> 5] = a;
    __syncthreads();
    if (int(threadIdx.x) < ncta) {
      const float m = fmaxf(fmaxf(red_s[0], red_s[1]), fmaxf(red_s[2], red_s[3]));
      st_cluster_u32(mapa_shared(smem_u32(&amax_s[rank]), threadIdx.x), __float_as_uint(m));
    }
    cluster_sync();
    float m = 0.f;
    for (int r = 0; r < ncta; ++r) m = fmaxf(m, amax_s[r]);
    g_act = nvfp4_global_from_amax(m);
    const uint32_t aq_base = smem_u32(aq_s), sa_base = smem_u32(sa_s);
    const Nvfp4BlockEncoder enc(g_act);
    for (int i = int(rank) + ncta * int(threadIdx.x); i < p.T * nchunks;
         i += ncta * blockDim.x) {
      const int t = i / nchunks;
      const int c = i - t * nchunks;
      const uint4* src = xv + (int64_t(t) * p.K + int64_t(c) * 32) / 8;
      uint4 codes;
      float dec;
      const uint32_t sf0 = enc.block(__ldg(src), __ldg(src + 1), codes.x, codes.y, &dec);
      const uint32_t sf1 = enc.block(__ldg(src + 2), __ldg(src + 3), codes.z, codes.w, &dec);
      const uint16_t sa = static_cast<uint16_t>(sf0 | (sf1 << 8));
      uint32_t q[8];
      decode_chunk(codes, q);
      const uint32_t o0 = aq_base + uint32_t((t * 2) * nchunks + c) * 16u;
      const uint32_t o1 = aq_base + uint32_t((t * 2 + 1) * nchunks + c) * 16u;
      const uint32_t os = sa_base + uint32_t(t * nchunks + c) * 2u;
      for (int r = 0; r < ncta; ++r) {
        st_cluster_v4(mapa_shared(o0, r), q[0], q[1], q[2], q[3]);
        st_cluster_v4(mapa_shared(o1, r), q[4], q[5], q[6], q[7]);
        st_cluster_u16(mapa_shared(os, r), sa);
      }
    }
    cluster_sync();
  } else {
    for (int i = threadIdx.x; i < p.T * nchunks; i += blockDim.x) {
      const int t = i / nchunks;
      const int c = i - t * nchunks;
      uint32_t q[8];
      decode_chunk(__ldg(reinterpret_cast<const uint4*>(p.A + int64_t(t) * kh) + c), q);
      aq_s[(t * 2) * nchunks + c] = make_uint4(q[0], q[1], q[2], q[3]);
      aq_s[(t * 2 + 1) * nchunks + c] = make_uint4(q[4], q[5], q[6], q[7]);
      sa_s[t * nchunks + c] = __ldg(reinterpret_cast<const unsigned short*>(
          p.sfA + gemv_sf_row_offset(t, kt) + (c >> 1) * 512 + (c & 1) * 2));
    }
  }
  __syncthreads();

  // One weight-row pair per warp.  In the operator form the grid is one
  // resident wave and the warps stride over the pairs, so the in-kernel
  // quantization is paid once per CTA; otherwise the loop runs once.
  for (int pair = blockIdx.x * 4 + (threadIdx.x >> 5); pair * 2 < p.N; pair += gridDim.x * 4) {
    const int n0 = pair * 2;
    const uint4* w0 = reinterpret_cast<const uint4*>(p.W + int64_t(n0) * kh);
    const uint4* w1 = reinterpret_cast<const uint4*>(p.W + int64_t(n0 + 1) * kh);
    const int sw0 = gemv_sf_row_offset(n0, kt);
    const int sw1 = gemv_sf_row_offset(n0 + 1, kt);
    float acc[2][TT];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int t = 0; t < TT; ++t) acc[r][t] = 0.f;

    for (int c0 = lane; c0 < nchunks; c0 += 32 * kUnroll) {
      // The weight stream of kUnroll chunks first (read once: evict-first).
      uint4 wv[kUnroll][2];
      uint16_t ws[kUnroll][2];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + 32 * u;
        if (c < nchunks) {
          const int so = (c >> 1) * 512 + (c & 1) * 2;
          wv[u][0] = __ldcs(w0 + c);
          wv[u][1] = __ldcs(w1 + c);
          ws[u][0] = __ldg(reinterpret_cast<const unsigned short*>(p.sfW + sw0 + so));
          ws[u][1] = __ldg(reinterpret_cast<const unsigned short*>(p.sfW + sw1 + so));
        } else {
          wv[u][0] = wv[u][1] = make_uint4(0u, 0u, 0u, 0u);
          ws[u][0] = ws[u][1] = 0;
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + 32 * u;
        if (c >= nchunks) break;
        uint32_t wq[2][8];
        decode_chunk(wv[u][0], wq[0]);
        decode_chunk(wv[u][1], wq[1]);
        const float2 sw[2] = {e4m3x2_to_float2(ws[u][0]), e4m3x2_to_float2(ws[u][1])};
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          if (t >= p.T) break;
          const uint4 a0 = aq_s[(t * 2) * nchunks + c];
          const uint4 a1 = aq_s[(t * 2 + 1) * nchunks + c];
          const float2 sa = e4m3x2_to_float2(sa_s[t * nchunks + c]);
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            int d0 = __dp4a(int(a0.x), int(wq[r][0]), 0);
            d0 = __dp4a(int(a0.y), int(wq[r][1]), d0);
            d0 = __dp4a(int(a0.z), int(wq[r][2]), d0);
            d0 = __dp4a(int(a0.w), int(wq[r][3]), d0);
            int d1 = __dp4a(int(a1.x), int(wq[r][4]), 0);
            d1 = __dp4a(int(a1.y), int(wq[r][5]), d1);
            d1 = __dp4a(int(a1.z), int(wq[r][6]), d1);
            d1 = __dp4a(int(a1.w), int(wq[r][7]), d1);
            acc[r][t] = fmaf(float(d0), sa.x * sw[r].x, acc[r][t]);
            acc[r][t] = fmaf(float(d1), sa.y * sw[r].y, acc[r][t]);
          }
        }
      }
    }

    // Sum over the lanes (every lane ends with the totals).
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[r][t] += __shfl_xor_sync(0xffffffffu, acc[r][t], o);

    const float s = (p.X ? g_act : __ldg(p.gA)) * __ldg(p.gW);
    if constexpr (EPI == SPG_EPI_SWIGLU) {
      // rows n0 (gate) and n0 + 1 (up) give output column n0 / 2
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        if (lane == t && t < p.T) {
          float gate = (acc[0][t] * 0.25f) * s;
          float up = (acc[1][t] * 0.25f) * s;
          if (p.bias_kind) {
            gate += gemv_bias(p, n0);
            up += gemv_bias(p, n0 + 1);
          }
          const float o = __fdividef(gate, 1.f + __expf(-gate)) * up;
          p.Y[int64_t(t) * p.n_out + pair] = __float2bfloat16_rn(o);
        }
      }
    } else {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          if (lane == r * TT + t && t < p.T) {
            const int n = n0 + r;
            float v = (acc[r][t] * 0.25f) * s;
            if (p.bias_kind) v += gemv_bias(p, n);
            if constexpr (EPI == SPG_EPI_ADD)
              v += __uint_as_float(uint32_t(__ldg(reinterpret_cast<const unsigned short*>(
                                                      p.residual) +
                                                  int64_t(t) * p.N + n))
                                   << 16);
            p.Y[int64_t(t) * p.n_out + n] = __float2bfloat16_rn(v);
          }
        }
      }
    }
  }
}

// Clusters of the operator form that fit on the device at once for this
// launch configuration (0 if the query fails), cached per kernel and
// shared-memory size.
template <typename Kern>
int gemv_cluster_wave(Kern kern, const cudaLaunchConfig_t& cfg) {
  static std::mutex mu;
  static std::map<std::pair<int, size_t>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const auto key = std::make_pair(dev, cfg.dynamicSmemBytes);
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  cache[key] = n;
  return n;
}

// Launch: one warp per weight-row pair, 4 warps per CTA; the dynamic shared
// memory limit is raised once per device.
template <int EPI, int TT>
spg_status launch_gemv(const GemvParams& p, cudaStream_t s) {
  int grid = (p.N / 2 + 3) / 4;
  const int64_t smem = gemv_smem_bytes(TT, p.K);  // <= 200 KB (the route checks)
  auto kern = gemv_nvfp4_kernel<EPI, TT>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPG_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    if (cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         200 * 1024),
                    "cudaFuncSetAttribute") != SPG_OK)
      return SPG_ERR_CUDA;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  if (!p.X) {
    kern<<<grid, 128, static_cast<size_t>(smem), s>>>(p);
    return launch_status();
  }
  // Operator form: clusters of kGemvCluster CTAs, at most one resident wave
  // of them (the warps stride over the row pairs).  CTAs without a row pair
  // only take their share of the quantization.
  grid = (grid + kGemvCluster - 1) / kGemvCluster * kGemvCluster;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kGemvCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // More CTAs than one wave holds: take R = ceil(CTAs / wave) rounds of
  // pairs per warp and just enough CTAs for them (fewer CTAs also quantize
  // X fewer times).
  const int wave = gemv_cluster_wave(kern, cfg) * kGemvCluster;
  if (wave > 0 && grid > wave) {
    const int pairs = p.N / 2;
    const int rounds = (grid + wave - 1) / wave;
    const int ctas = ((pairs + rounds - 1) / rounds + 3) / 4;
    cfg.gridDim = dim3((ctas + kGemvCluster - 1) / kGemvCluster * kGemvCluster);
  }
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, p), "cudaLaunchKernelEx");
}

template <int EPI>
spg_status launch_gemv_tokens(const GemvParams& p, cudaStream_t s) {
  if (p.T == 1) return launch_gemv<EPI, 1>(p, s);
  if (p.T == 2) return launch_gemv<EPI, 2>(p, s);
  if (p.T == 3) return launch_gemv<EPI, 3>(p, s);
  return launch_gemv<EPI, 4>(p, s);
}

inline spg_status launch_gemv_epilogue(const GemvParams& p, int epilogue, cudaStream_t s) {
  switch (epilogue) {
    case SPG_EPI_LINEAR: return launch_gemv_tokens<SPG_EPI_LINEAR>(p, s);
    case SPG_EPI_ADD: return launch_gemv_tokens<SPG_EPI_ADD>(p, s);
    default: return launch_gemv_tokens<SPG_EPI_SWIGLU>(p, s);
  }
}

}  // namespace spg
