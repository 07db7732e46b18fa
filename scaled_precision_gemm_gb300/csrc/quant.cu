// Activation / weight quantizers: bf16 -> E4M3 codes with row or tensor
// scales, and bf16 -> NVFP4 (E2M1 codes, E4M3 block-16 scales in the blocked
// tile layout, fp32 global scale).
//
// All of them are streaming kernels: 16-byte vector loads of the bf16
// input, every fp32 step one correctly rounded operation so that codes and
// scales are bit-for-bit those of the plain definition, and hardware
// cvt.rn.satfinite conversions for the codes.  The per-element quotient
// x / s is the correctly rounded one, formed from a reciprocal taken once
// per scale with Markstein's correction step (ExactDivisor): an IEEE
// division per element made them instruction-bound (measured on GB300: the
// FP8 row quantizer took 88 us at T = 8192, K = 17408, against 63.5 us --
// the HBM copy rate -- with an inexact plain multiply).
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "common.h"
#include "nvfp4_encode.cuh"
#include "ptx.cuh"

namespace spg {
namespace {

__device__ __forceinline__ float vec_amax(const uint4& v) { return bf16x8_amax(v); }

// Eight bf16 divided by s (correctly rounded) -> eight E4M3 codes.  MODE 0:
// any s and x (the delayed scale may be stale); 1: s.fast and |x| <= 448 s
// (a scale taken from this data's amax); 2: the IEEE division.
template <int MODE>
__device__ __forceinline__ uint2 vec_encode_e4m3(const uint4& v, const ExactDivisor& s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = bf16_lo(w[i]), hi = bf16_hi(w[i]);
    if constexpr (MODE == 1)
      c[i] = cvt_e4m3x2(s.div_fast(lo), s.div_fast(hi));
    else if constexpr (MODE == 2)
      c[i] = cvt_e4m3x2(__fdiv_rn(lo, s.s), __fdiv_rn(hi, s.s));
    else
      c[i] = cvt_e4m3x2(s.div(lo), s.div(hi));
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <int THREADS>
__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float r = (threadIdx.x < THREADS / 32) ? red[threadIdx.x] : 0.f;
  if (w == 0) r = warp_max(r);
  if (threadIdx.x == 0) red[0] = r;
  __syncthreads();
  r = red[0];
  __syncthreads();
  return r;
}

// One CTA per row: amax over the row, s = amax/448, codes = E4M3(x/s).
// THREADS x VECS 16-byte vectors of the row stay in registers between the
// two passes; longer rows re-read their remainder.  Rows up to 8192
// elements take a 128-thread CTA, so more rows are in flight per SM
// (measured on GB300 at T = 8192: K = 5120 45 -> 33 us, K = 6144 47 -> 37 us
// against the 256-thread CTA).
template <int THREADS, int VECS>
__global__ void __launch_bounds__(THREADS) quantize_fp8_rows_kernel(
    const uint4* __restrict__ x, int64_t K, uint2* __restrict__ codes, float* __restrict__ scales) {
  __shared__ float red[THREADS / 32];
  const int64_t row = blockIdx.x;
  const int64_t nvec = K / 8;
  const uint4* xr = x + row * nvec;
  uint2* cr = codes + row * nvec;
  uint4 cache[VECS];
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < VECS; ++j) {
    const int64_t i = threadIdx.x + static_cast<int64_t>(j) * THREADS;
    if (i < nvec) {
      cache[j] = __ldg(xr + i);
      amax = fmaxf(amax, vec_amax(cache[j]));
    }
  }
  for (int64_t i = threadIdx.x + int64_t(VECS) * THREADS; i < nvec; i += THREADS)
    amax = fmaxf(amax, vec_amax(__ldg(xr + i)));
  amax = block_max<THREADS>(amax, red);
  const float s = (amax == 0.f) ? 1.f : __fdiv_rn(amax, 448.f);
  const ExactDivisor sd(s);
  // The branch is uniform over the CTA (one row, one scale).
  if (sd.fast) {
#pragma unroll
    for (int j = 0; j < VECS; ++j) {
      const int64_t i = threadIdx.x + static_cast<int64_t>(j) * THREADS;
      if (i < nvec) cr[i] = vec_encode_e4m3<1>(cache[j], sd);
    }
    for (int64_t i = threadIdx.x + int64_t(VECS) * THREADS; i < nvec; i += THREADS)
      cr[i] = vec_encode_e4m3<1>(__ldg(xr + i), sd);
  } else {
#pragma unroll
    for (int j = 0; j < VECS; ++j) {
      const int64_t i = threadIdx.x + static_cast<int64_t>(j) * THREADS;
      if (i < nvec) cr[i] = vec_encode_e4m3<2>(cache[j], sd);
    }
    for (int64_t i = threadIdx.x + int64_t(VECS) * THREADS; i < nvec; i += THREADS)
      cr[i] = vec_encode_e4m3<2>(__ldg(xr + i), sd);
  }
  if (threadIdx.x == 0) scales[row] = s;
}

// amax over a whole tensor into *amax (which the host zeroes first).
// Non-negative floats order like their bit patterns, so an unsigned
// atomicMax on the bits is a float max.
__global__ void __launch_bounds__(256) amax_kernel(const uint4* __restrict__ x, int64_t nvec,
                                                   float* __restrict__ amax) {
  __shared__ float red[8];
  float a = 0.f;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < nvec;
       i += int64_t(gridDim.x) * blockDim.x)
    a = fmaxf(a, vec_amax(__ldg(x + i)));
  a = block_max<256>(a, red);
  if (threadIdx.x == 0 && a > 0.f)
    atomicMax(reinterpret_cast<unsigned int*>(amax), __float_as_uint(a));
}

// Per-tensor E4M3 encode with s = amax/448 (1 when amax = 0).
__global__ void __launch_bounds__(256) encode_fp8_tensor_kernel(const uint4* __restrict__ x,
                                                                int64_t nvec,
                                                                const float* __restrict__ amax,
                                                                uint2* __restrict__ codes,
                                                                float* __restrict__ scale) {
  const float a = *amax;
  const float s = (a == 0.f) ? 1.f : __fdiv_rn(a, 448.f);
  const ExactDivisor sd(s);
  if (sd.fast) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < nvec;
         i += int64_t(gridDim.x) * blockDim.x)
      codes[i] = vec_encode_e4m3<1>(__ldg(x + i), sd);
  } else {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < nvec;
         i += int64_t(gridDim.x) * blockDim.x)
      codes[i] = vec_encode_e4m3<2>(__ldg(x + i), sd);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *scale = s;
}

// g = amax / (448 * 6), 1 when amax = 0.
__global__ void nvfp4_global_finalize_kernel(const float* __restrict__ amax, float* __restrict__ g) {
  *g = nvfp4_global_from_amax(*amax);
}

// NVFP4 block quantizer.  The input is walked as one flat sequence of
// 16-element blocks (rows are contiguous; a row holds K/16 of them), one
// block per lane: a warp's two 16-byte loads per step cover 1 KB spread
// over 8 cache lines, its code stores 256 contiguous bytes.  (One thread
// per 64-element group -- 16-byte loads 128 bytes apart across a warp, 32
// lines per load -- measured 86 us at T = 8192, K = 17408 on GB300, bound
// by L1 requests once the quotients were cheap.)  Each lane encodes its
// block; two shuffles gather the four scale bytes of a 64-element group
// (lanes 4j .. 4j+3) for its first lane to store as one word of the blocked
// layout.  kNvSpans steps are loaded before any is encoded.  After the data
// the grid zeroes the scale words of the padding rows.
// FROM_AMAX: gptr holds the tensor's maximum instead of g; every CTA forms g
// from it (the same value everywhere) and CTA 0 stores it to *g_out, which
// saves the global scale's separate finalize launch.
constexpr int kNvSpans = 4;

template <bool FROM_AMAX>
__global__ void __launch_bounds__(256) quantize_nvfp4_kernel(
    const uint4* __restrict__ x, uint32_t rows, uint32_t rows_pad, uint32_t upr,
    const float* __restrict__ gptr, uint2* __restrict__ codes, uint32_t* __restrict__ sf,
    float* __restrict__ g_out) {
  const uint32_t nblk = rows * upr * 4;  // host guarantees rows_pad * upr * 4 < 2^31
  const int lane = threadIdx.x & 31;
  const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t base = warp * (32 * kNvSpans);
  const float g = FROM_AMAX ? nvfp4_global_from_amax(*gptr) : *gptr;
  if (FROM_AMAX && blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
  const Nvfp4BlockEncoder enc(g);
  uint4 v[kNvSpans][2];
#pragma unroll
  for (int j = 0; j < kNvSpans; ++j) {
    const uint32_t blk = base + 32 * j + lane;
    if (blk < nblk) {
      v[j][0] = __ldg(x + 2 * int64_t(blk));
      v[j][1] = __ldg(x + 2 * int64_t(blk) + 1);
    } else {
      v[j][0] = v[j][1] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int j = 0; j < kNvSpans; ++j) {
    const uint32_t blk = base + 32 * j + lane;
    uint2 c;
    float dec;
    const uint32_t sfc = enc.block(v[j][0], v[j][1], c.x, c.y, &dec);
    uint32_t w = sfc << (8 * (lane & 3));
    w |= __shfl_xor_sync(0xffffffffu, w, 1);
    w |= __shfl_xor_sync(0xffffffffu, w, 2);
    if (blk < nblk) {
      codes[blk] = c;
      if ((lane & 3) == 0) {
        const uint32_t grp = blk >> 2;
        const uint32_t r = grp / upr, cb = grp - r * upr;
        sf[(int64_t(r >> 7) * upr + cb) * 128 + (r & 31) * 4 + ((r >> 5) & 3)] = w;
      }
    }
  }
  const uint32_t pad_words = (rows_pad - rows) * upr;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < pad_words;
       i += gridDim.x * blockDim.x) {
    const uint32_t r = rows + i / upr, cb = i % upr;
    sf[(int64_t(r >> 7) * upr + cb) * 128 + (r & 31) * 4 + ((r >> 5) & 3)] = 0u;
  }
}

// Global scale and block quantizer in one CTA, for tensors small enough
// that one SM streams them faster than four launches (memset, amax,
// finalize, encode) take to start: the CTA's maximum gives g (written to
// *g_out), then each lane encodes 16-element blocks as the block quantizer
// does (consecutive lanes on consecutive blocks, so a group's four scale
// bytes sit in lanes 4j .. 4j+3).
constexpr int kNvSmallThreads = 1024;
constexpr int64_t kNvSmallMaxElems = 72 * 1024;  // measured: one CTA wins up to ~70K elements

__global__ void __launch_bounds__(kNvSmallThreads) quantize_nvfp4_small_kernel(
    const uint4* __restrict__ x, uint32_t rows, uint32_t rows_pad, uint32_t upr,
    float* __restrict__ g_out, uint2* __restrict__ codes, uint32_t* __restrict__ sf) {
  __shared__ float red[kNvSmallThreads / 32];
  const uint32_t nblk = rows * upr * 4;
  const uint32_t nvec = nblk * 2;
  if (rows_pad != rows) {
    // Zero the scale tiles of the last row block whole (16-byte stores): its
    // padding rows stay zero, its real rows are written below, after the
    // barriers of the block maximum.  (One word per padding row and scale
    // column, each with its own index arithmetic, took ~20 us at K = 17408.)
    uint4* t = reinterpret_cast<uint4*>(sf) + ((rows_pad >> 7) - 1) * upr * 32;
    for (uint32_t i = threadIdx.x; i < upr * 32; i += kNvSmallThreads)
      t[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  float a = 0.f;
  for (uint32_t i = threadIdx.x; i < nvec; i += kNvSmallThreads) a = fmaxf(a, vec_amax(__ldg(x + i)));
  const float g = nvfp4_global_from_amax(block_max<kNvSmallThreads>(a, red));
  if (threadIdx.x == 0) *g_out = g;
  const Nvfp4BlockEncoder enc(g);
  const int lane = threadIdx.x & 31;
  // every lane of a warp takes the same number of trips (the shuffles)
  for (uint32_t base = threadIdx.x - lane; base < nblk; base += kNvSmallThreads) {
    const uint32_t blk = base + lane;
    uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
    if (blk < nblk) {
      v0 = __ldg(x + 2 * blk);
      v1 = __ldg(x + 2 * blk + 1);
    }
    uint2 c;
    float dec;
    const uint32_t sfc = enc.block(v0, v1, c.x, c.y, &dec);
    uint32_t w = sfc << (8 * (lane & 3));
    w |= __shfl_xor_sync(0xffffffffu, w, 1);
    w |= __shfl_xor_sync(0xffffffffu, w, 2);
    if (blk < nblk) {
      codes[blk] = c;
      if ((lane & 3) == 0) {
        const uint32_t grp = blk >> 2;
        const uint32_t r = grp / upr, cb = grp - r * upr;
        sf[(r >> 7) * upr * 128 + cb * 128 + (r & 31) * 4 + ((r >> 5) & 3)] = w;
      }
    }
  }
}

// Global scale and block quantizer in one cluster of up to kNvClusterMax
// CTAs, for tensors too large for one CTA but small enough that a few SMs
// stream them faster than four launches take to start.  CTA r of the
// cluster takes a contiguous run of 16-element blocks (a multiple of 32, so
// a warp's lanes hold whole 64-element groups), reduces its maximum, and
// stores it into slot r of every CTA's shared memory; after one cluster
// barrier every CTA holds all the maxima, forms the same g and encodes its
// blocks (its run is read a second time, from L2).  The scale tiles of the
// last row block are zeroed before the barrier, which orders those stores
// before the real rows' words written after it.
constexpr int kNvClusterMax = 16;
// Measured on GB300 (us, cluster / four launches): 87K elements 8.7 / 14.9,
// 279K 10.8 / 14.9, 393K 10.7 / 12.8, 786K 12.8 / 12.8, 1.1M 14.9 / 12.8.
constexpr int64_t kNvClusterMaxElems = 512 * 1024;

__global__ void __launch_bounds__(kNvSmallThreads) quantize_nvfp4_cluster_kernel(
    const uint4* __restrict__ x, uint32_t rows, uint32_t rows_pad, uint32_t upr,
    float* __restrict__ g_out, uint2* __restrict__ codes, uint32_t* __restrict__ sf) {
  __shared__ float red[kNvSmallThreads / 32];
  __shared__ float part[kNvClusterMax];
  const uint32_t ncta = cluster_nctarank(), rank = cluster_ctarank();
  const uint32_t nblk = rows * upr * 4;
  const uint32_t per = ((nblk + ncta - 1) / ncta + 31) / 32 * 32;
  const uint32_t b0 = min(rank * per, nblk), b1 = min(b0 + per, nblk);
  if (rows_pad != rows) {
    uint4* t = reinterpret_cast<uint4*>(sf) + ((rows_pad >> 7) - 1) * upr * 32;
    for (uint32_t i = rank * kNvSmallThreads + threadIdx.x; i < upr * 32;
         i += ncta * kNvSmallThreads)
      t[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  float a = 0.f;
  for (uint32_t i = 2 * b0 + threadIdx.x; i < 2 * b1; i += kNvSmallThreads)
    a = fmaxf(a, vec_amax(__ldg(x + i)));
  a = block_max<kNvSmallThreads>(a, red);
  if (threadIdx.x < ncta)
    st_cluster_u32(mapa_shared(smem_u32(&part[rank]), threadIdx.x), __float_as_uint(a));
  cluster_sync();
  float m = 0.f;
  for (uint32_t q = 0; q < ncta; ++q) m = fmaxf(m, part[q]);
  const float g = nvfp4_global_from_amax(m);
  if (rank == 0 && threadIdx.x == 0) *g_out = g;
  const Nvfp4BlockEncoder enc(g);
  const int lane = threadIdx.x & 31;
  // every lane of a warp takes the same number of trips (the shuffles)
  for (uint32_t base = b0 + threadIdx.x - lane; base < b1; base += kNvSmallThreads) {
    const uint32_t blk = base + lane;
    uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
    if (blk < b1) {
      v0 = __ldg(x + 2 * blk);
      v1 = __ldg(x + 2 * blk + 1);
    }
    uint2 c;
    float dec;
    const uint32_t sfc = enc.block(v0, v1, c.x, c.y, &dec);
    uint32_t w = sfc << (8 * (lane & 3));
    w |= __shfl_xor_sync(0xffffffffu, w, 1);
    w |= __shfl_xor_sync(0xffffffffu, w, 2);
    if (blk < b1) {
      codes[blk] = c;
      if ((lane & 3) == 0) {
        const uint32_t grp = blk >> 2;
        const uint32_t r = grp / upr, cb = grp - r * upr;
        sf[(r >> 7) * upr * 128 + cb * 128 + (r & 31) * 4 + ((r >> 5) & 3)] = w;
      }
    }
  }
}

// Cluster size for quantize_nvfp4_cluster_kernel on the current device: 16
// where such clusters can be resident (a non-portable size), else 8.
int nvfp4_cluster_ctas() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
  int c = cached[dev].load(std::memory_order_relaxed);
  if (c != 0) return c;
  c = 8;
  auto kern = quantize_nvfp4_cluster_kernel;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kNvClusterMax, 1, 1);
    cfg.blockDim = dim3(kNvSmallThreads, 1, 1);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kNvClusterMax;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n >= 1) c = kNvClusterMax;
  }
  cudaGetLastError();  // a refused query leaves no error behind
  cached[dev].store(c, std::memory_order_relaxed);
  return c;
}

// ----------------------------------------------------------------------
// Allocation-free variant of the per-tensor quantizer.  Its amax scratch is
// this file-scope device array instead of a caller-provided buffer: slots
// [0, kStaticPartials) hold one partial maximum per CTA of the first pass,
// slot kStaticPartials holds the reduced maximum.  Every slot a call reads is
// written earlier in the same call, so nothing has to be cleared between
// calls; calls that overlap on the GPU share the array and race.
constexpr int kStaticPartials = 4096;               // 16 KB of partial maxima
constexpr int64_t kStaticElemsPerPartial = 65536;   // elements one CTA reduces
constexpr int64_t kStaticMaxNumel = kStaticPartials * kStaticElemsPerPartial;
static __device__ __align__(256) float g_fp8_tensor_static_scratch[kStaticPartials + 64];

// Partial amax: CTA b reduces elements [b*65536, (b+1)*65536) into partials[b].
__global__ void __launch_bounds__(256) partial_amax_kernel(const uint4* __restrict__ x,
                                                           int64_t nvec,
                                                           float* __restrict__ partials) {
  __shared__ float red[8];
  constexpr int64_t kVecPerCta = kStaticElemsPerPartial / 8;
  const int64_t v0 = int64_t(blockIdx.x) * kVecPerCta;
  const int64_t v1 = v0 + kVecPerCta < nvec ? v0 + kVecPerCta : nvec;
  float a = 0.f;
  for (int64_t i = v0 + threadIdx.x; i < v1; i += blockDim.x) a = fmaxf(a, vec_amax(__ldg(x + i)));
  a = block_max<256>(a, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = a;
}

// Reduce partials[0, nparts) into partials[kStaticPartials] (0 when nparts == 0).
__global__ void __launch_bounds__(1024) reduce_partials_kernel(float* __restrict__ partials,
                                                               int nparts) {
  __shared__ float red[32];
  float a = 0.f;
  for (int i = threadIdx.x; i < nparts; i += blockDim.x) a = fmaxf(a, partials[i]);
  a = block_max<1024>(a, red);
  if (threadIdx.x == 0) partials[kStaticPartials] = a;
}

// ----------------------------------------------------------------------
// Delayed scaling: one kernel encodes with the scale published by the
// previous call and folds this call's amax into the history ring; its last
// block (elected by an atomic counter after a __threadfence) reduces the
// window and publishes the next scale.  Ring layout (fp32 words):
//   [0, H) history   [H] scale   [H+1] amax of the call in flight
//   [H+2] block counter (u32)   [H+3] next history index (u32)
__global__ void __launch_bounds__(256) quantize_fp8_delayed_kernel(const uint4* __restrict__ x,
                                                                  int64_t nvec,
                                                                  uint2* __restrict__ codes,
                                                                  float* __restrict__ scale_used,
                                                                  float* ring, int history) {
  __shared__ float red[8];
  __shared__ bool last;
  const float s = *reinterpret_cast<volatile float*>(ring + history);
  const ExactDivisor sd(s);
  float a = 0.f;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < nvec;
       i += int64_t(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(x + i);
    a = fmaxf(a, vec_amax(v));
    codes[i] = vec_encode_e4m3<0>(v, sd);
  }
  a = block_max<256>(a, red);
  unsigned int* amax_bits = reinterpret_cast<unsigned int*>(ring + history + 1);
  unsigned int* counter = reinterpret_cast<unsigned int*>(ring + history + 2);
  unsigned int* idx = reinterpret_cast<unsigned int*>(ring + history + 3);
  if (threadIdx.x == 0) {
    if (a > 0.f) atomicMax(amax_bits, __float_as_uint(a));
    __threadfence();
    last = atomicAdd(counter, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (last && threadIdx.x == 0) {
    __threadfence();
    const float amax = __uint_as_float(atomicExch(amax_bits, 0u));
    const unsigned int k = *reinterpret_cast<volatile unsigned int*>(idx);
    ring[k] = amax;
    float m = 0.f;
    for (int h = 0; h < history; ++h) m = fmaxf(m, reinterpret_cast<volatile float*>(ring)[h]);
    *scale_used = s;
    ring[history] = (m == 0.f) ? 1.f : __fdiv_rn(m, 448.f);
    *idx = (k + 1 == unsigned(history)) ? 0u : k + 1;
    *counter = 0u;
    __threadfence();
  }
}

__global__ void scale_ring_init_kernel(float* ring, int history, float initial_scale) {
  for (int i = threadIdx.x; i < history + 4; i += blockDim.x) {
    float v = 0.f;
    if (i == history) v = initial_scale;
    ring[i] = v;
  }
}

int grid_for(int64_t work, int threads) {
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  int64_t g = (work + threads - 1) / threads;
  if (g > cap) g = cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace
}  // namespace spg

using namespace spg;

extern "C" spg_status spg_quantize_fp8_rows(const void* x, int64_t rows, int64_t K,
                                            uint8_t* codes, float* scales, spg_stream_t stream) {
  if (rows < 0 || K < 0) return SPG_ERR_INVALID_ARG;
  if (rows == 0) return SPG_OK;
  if (!x || !codes || !scales) return SPG_ERR_INVALID_ARG;
  if (K == 0 || K % 8 != 0) return SPG_ERR_UNSUPPORTED_SHAPE;
  if (rows > 0x7FFFFFFF) return SPG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return SPG_ERR_MISALIGNED;
  const unsigned grid = static_cast<unsigned>(rows);
  const uint4* xv = static_cast<const uint4*>(x);
  uint2* cv = reinterpret_cast<uint2*>(codes);
  if (K / 8 <= 128 * 8)
    quantize_fp8_rows_kernel<128, 8><<<grid, 128, 0, stream>>>(xv, K, cv, scales);
  else
    quantize_fp8_rows_kernel<256, 9><<<grid, 256, 0, stream>>>(xv, K, cv, scales);
  return launch_status();
}

extern "C" spg_status spg_quantize_fp8_tensor(const void* x, int64_t numel, uint8_t* codes,
                                              float* scale, float* amax_scratch,
                                              spg_stream_t stream) {
  if (numel < 0) return SPG_ERR_INVALID_ARG;
  if (!scale || !amax_scratch) return SPG_ERR_INVALID_ARG;
  if (numel > 0 && (!x || !codes)) return SPG_ERR_INVALID_ARG;
  if (numel % 8 != 0) return SPG_ERR_UNSUPPORTED_SHAPE;
  if ((numel > 0 && (!aligned16(x) || !aligned16(codes))) || !aligned16(scale) ||
      !aligned16(amax_scratch))
    return SPG_ERR_MISALIGNED;
  const int64_t nvec = numel / 8;
  if (cudaMemsetAsync(amax_scratch, 0, sizeof(float), stream) != cudaSuccess) return SPG_ERR_CUDA;
  if (nvec > 0) {
    amax_kernel<<<grid_for(nvec, 256), 256, 0, stream>>>(static_cast<const uint4*>(x), nvec,
                                                          amax_scratch);
    if (launch_status() != SPG_OK) return SPG_ERR_CUDA;
  }
  encode_fp8_tensor_kernel<<<grid_for(nvec > 0 ? nvec : 1, 256), 256, 0, stream>>>(
      static_cast<const uint4*>(x), nvec, amax_scratch, reinterpret_cast<uint2*>(codes), scale);
  return launch_status();
}

extern "C" spg_status spg_nvfp4_global_scale(const void* x, int64_t numel, float* g,
                                             float* amax_scratch, spg_stream_t stream) {
  if (numel < 0 || !g || !amax_scratch) return SPG_ERR_INVALID_ARG;
  if (numel > 0 && !x) return SPG_ERR_INVALID_ARG;
  if (numel % 8 != 0) return SPG_ERR_UNSUPPORTED_SHAPE;
  if ((numel > 0 && !aligned16(x)) || !aligned16(g) || !aligned16(amax_scratch))
    return SPG_ERR_MISALIGNED;
  const int64_t nvec = numel / 8;
  if (cudaMemsetAsync(amax_scratch, 0, sizeof(float), stream) != cudaSuccess) return SPG_ERR_CUDA;
  if (nvec > 0) {
    amax_kernel<<<grid_for(nvec, 256), 256, 0, stream>>>(static_cast<const uint4*>(x), nvec,
                                                          amax_scratch);
    if (launch_status() != SPG_OK) return SPG_ERR_CUDA;
  }
  nvfp4_global_finalize_kernel<<<1, 1, 0, stream>>>(amax_scratch, g);
  return launch_status();
}

extern "C" spg_status spg_quantize_nvfp4(const void* x, int64_t rows, int64_t K, const float* g,
                                         uint8_t* codes, uint8_t* sf, spg_stream_t stream) {
  if (rows < 0 || K < 0) return SPG_ERR_INVALID_ARG;
  if (rows == 0) return SPG_OK;
  if (!x || !g || !codes || !sf) return SPG_ERR_INVALID_ARG;
  if (K == 0 || K % 64 != 0) return SPG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(sf) || !aligned16(g))
    return SPG_ERR_MISALIGNED;
  const int64_t rows_pad = (rows + 127) / 128 * 128;
  const int64_t upr = K / 64;
  // 32-bit block indices (the grid covers up to 2^31 blocks and steps past)
  if (rows_pad * upr * 4 >= (int64_t(1) << 31)) return SPG_ERR_UNSUPPORTED_SHAPE;
  const int64_t per_cta = 8 * 32 * kNvSpans;  // blocks: 8 warps x 32 lanes x kNvSpans
  const int64_t grid = (rows * upr * 4 + per_cta - 1) / per_cta;
  quantize_nvfp4_kernel<false><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
      static_cast<const uint4*>(x), static_cast<uint32_t>(rows), static_cast<uint32_t>(rows_pad),
      static_cast<uint32_t>(upr), g, reinterpret_cast<uint2*>(codes),
      reinterpret_cast<uint32_t*>(sf), nullptr);
  return launch_status();
}

extern "C" spg_status spg_quantize_nvfp4_act(const void* x, int64_t rows, int64_t K, float* g,
                                             float* amax_scratch, uint8_t* codes, uint8_t* sf,
                                             spg_stream_t stream) {
  if (rows < 0 || K < 0) return SPG_ERR_INVALID_ARG;
  if (rows == 0) return SPG_OK;
  if (!x || !g || !amax_scratch || !codes || !sf) return SPG_ERR_INVALID_ARG;
  if (K == 0 || K % 64 != 0) return SPG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(sf) || !aligned16(g) ||
      !aligned16(amax_scratch))
    return SPG_ERR_MISALIGNED;
  const int64_t rows_pad = (rows + 127) / 128 * 128;
  if (rows * K <= kNvSmallMaxElems) {
    quantize_nvfp4_small_kernel<<<1, kNvSmallThreads, 0, stream>>>(
        static_cast<const uint4*>(x), static_cast<uint32_t>(rows),
        static_cast<uint32_t>(rows_pad), static_cast<uint32_t>(K / 64), g,
        reinterpret_cast<uint2*>(codes), reinterpret_cast<uint32_t*>(sf));
    return launch_status();
  }
  if (rows * K <= kNvClusterMaxElems) {
    const int ncta = nvfp4_cluster_ctas();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ncta), 1, 1);
    cfg.blockDim = dim3(kNvSmallThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ncta);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cuda_status(cudaLaunchKernelEx(&cfg, quantize_nvfp4_cluster_kernel,
                                       static_cast<const uint4*>(x), static_cast<uint32_t>(rows),
                                       static_cast<uint32_t>(rows_pad),
                                       static_cast<uint32_t>(K / 64), g,
                                       reinterpret_cast<uint2*>(codes),
                                       reinterpret_cast<uint32_t*>(sf)),
                    "cudaLaunchKernelEx") != SPG_OK)
      return SPG_ERR_CUDA;
    return launch_status();
  }
  // Large tensors: the maximum over all SMs, then the block encoder, which
  // forms g from it (three launches with the scratch's memset).
  if (rows_pad * (K / 64) * 4 >= (int64_t(1) << 31)) return SPG_ERR_UNSUPPORTED_SHAPE;
  const int64_t nvec = rows * K / 8;
  if (cudaMemsetAsync(amax_scratch, 0, sizeof(float), stream) != cudaSuccess) return SPG_ERR_CUDA;
  amax_kernel<<<grid_for(nvec, 256), 256, 0, stream>>>(static_cast<const uint4*>(x), nvec,
                                                        amax_scratch);
  if (launch_status() != SPG_OK) return SPG_ERR_CUDA;
  const int64_t upr = K / 64;
  const int64_t per_cta = 8 * 32 * kNvSpans;
  const int64_t grid = (rows * upr * 4 + per_cta - 1) / per_cta;
  quantize_nvfp4_kernel<true><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
      static_cast<const uint4*>(x), static_cast<uint32_t>(rows), static_cast<uint32_t>(rows_pad),
      static_cast<uint32_t>(upr), amax_scratch, reinterpret_cast<uint2*>(codes),
      reinterpret_cast<uint32_t*>(sf), g);
  return launch_status();
}

extern "C" size_t spg_nvfp4_sf_bytes(int64_t rows, int64_t K) {
  if (rows <= 0 || K <= 0) return 0;
  return static_cast<size_t>((rows + 127) / 128 * 128) * static_cast<size_t>((K + 63) / 64 * 4);
}

extern "C" int64_t spg_nvfp4_sf_offset(int64_t row, int64_t kb, int64_t K) {
  if (row < 0 || kb < 0 || K <= 0 || kb >= (K + 15) / 16) return -1;
  const int64_t tiles_per_row_block = (K + 63) / 64;
  return ((row / 128) * tiles_per_row_block + kb / 4) * 512 + (row % 32) * 16 +
         ((row % 128) / 32) * 4 + (kb % 4);
}

// Allocation-free per-tensor FP8 quantizer (see include/spg.h).  The device
// address of the static scratch is looked up once per device, with that
// device current, on the first call made on it.
namespace {
std::mutex g_static_mu;
float* g_static_scratch[64] = {};

float* static_scratch_for_current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_scratch[d]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, spg::g_fp8_tensor_static_scratch) != cudaSuccess) return nullptr;
    g_static_scratch[d] = static_cast<float*>(ptr);
  }
  return g_static_scratch[d];
}
}  // namespace

extern "C" spg_status spg_quantize_fp8_tensor_noalloc(const void* x, int64_t numel,
                                                      uint8_t* codes, float* scale,
                                                      spg_stream_t stream) {
  if (numel < 0 || !scale) return SPG_ERR_INVALID_ARG;
  if (numel > 0 && (!x || !codes)) return SPG_ERR_INVALID_ARG;
  if (numel % 8 != 0 || numel > spg::kStaticMaxNumel) return SPG_ERR_UNSUPPORTED_SHAPE;
  if ((numel > 0 && (!aligned16(x) || !aligned16(codes))) || !aligned16(scale))
    return SPG_ERR_MISALIGNED;
  float* scratch = static_scratch_for_current_device();
  if (!scratch) return SPG_ERR_CUDA;
  const int64_t nvec = numel / 8;
  const int nparts = static_cast<int>((numel + spg::kStaticElemsPerPartial - 1) /
                                      spg::kStaticElemsPerPartial);
  if (nparts > 0) {
    spg::partial_amax_kernel<<<nparts, 256, 0, stream>>>(static_cast<const uint4*>(x), nvec,
                                                          scratch);
    if (launch_status() != SPG_OK) return SPG_ERR_CUDA;
  }
  spg::reduce_partials_kernel<<<1, 1024, 0, stream>>>(scratch, nparts);
  if (launch_status() != SPG_OK) return SPG_ERR_CUDA;
  spg::encode_fp8_tensor_kernel<<<spg::grid_for(nvec > 0 ? nvec : 1, 256), 256, 0, stream>>>(
      static_cast<const uint4*>(x), nvec, scratch + spg::kStaticPartials,
      reinterpret_cast<uint2*>(codes), scale);
  return launch_status();
}

extern "C" size_t spg_fp8_scale_ring_bytes(int history) {
  if (history <= 0) return 0;
  return (static_cast<size_t>(history) + 4) * sizeof(float);
}

extern "C" spg_status spg_fp8_scale_ring_init(void* ring, int history, float initial_scale,
                                              spg_stream_t stream) {
  if (!ring || history <= 0 || history > 65536 || !(initial_scale > 0.f))
    return SPG_ERR_INVALID_ARG;
  if (!aligned16(ring)) return SPG_ERR_MISALIGNED;
  spg::scale_ring_init_kernel<<<1, 256, 0, stream>>>(static_cast<float*>(ring), history,
                                                     initial_scale);
  return launch_status();
}

extern "C" spg_status spg_quantize_fp8_tensor_delayed(const void* x, int64_t numel,
                                                      uint8_t* codes, float* scale_used,
                                                      void* ring, int history,
                                                      spg_stream_t stream) {
  if (numel < 0 || !scale_used || !ring || history <= 0 || history > 65536)
    return SPG_ERR_INVALID_ARG;
  if (numel > 0 && (!x || !codes)) return SPG_ERR_INVALID_ARG;
  if (numel % 8 != 0) return SPG_ERR_UNSUPPORTED_SHAPE;
  if ((numel > 0 && (!aligned16(x) || !aligned16(codes))) || !aligned16(scale_used) ||
      !aligned16(ring))
    return SPG_ERR_MISALIGNED;
  const int64_t nvec = numel / 8;
  spg::quantize_fp8_delayed_kernel<<<spg::grid_for(nvec > 0 ? nvec : 1, 256), 256, 0, stream>>>(
      static_cast<const uint4*>(x), nvec, reinterpret_cast<uint2*>(codes), scale_used,
      static_cast<float*>(ring), history);
  return launch_status();
}
