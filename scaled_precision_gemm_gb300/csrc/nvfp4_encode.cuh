// NVFP4 encoding of bf16 values, shared by the block quantizer and by the
// GEMV that quantizes its activations itself.
//
// ninfer PR #160 "The NVFP4 TMA route reads activation scales as one tile"
// (E2M1 codes, one E4M3 scale per 16 elements, activations quantized too),
// with the two-level scale the global scale g adds: per 16-element block
//   sf   = E4M3_rne_satfinite((amax_b / 6) / g)      two IEEE divisions
//   d    = dec(sf) * g                                 one IEEE multiply
//   code = E2M1_rne_satfinite(x / d)                   0 when d == 0
// and g = amax / (448 * 6) over the whole tensor (1 when amax == 0).  Every
// fp32 step is one IEEE-rounded operation, so the codes and scales are bit
// for bit those of the plain definition.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace spg {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// x / s correctly rounded for many x and one s, from a reciprocal taken
// once: Markstein's correction step.  With y = RN(1/s) and the faithful
// q0 = RN(x * y), the remainder x - q0 * s is exact (one FMA) and
// RN(q0 + (x - q0 * s) * y) = RN(x / s) -- a quotient of two floats is never
// a tie.  The remainder is formed as q0 * s - x and subtracted, which keeps
// x = -0 giving -0 as the division does.  1/s loses precision for huge
// divisors and the remainder may underflow for tiny ones, so divisors
// outside [2^-90, 2^100] take the IEEE division (`fast` false).  With
// s >= 2^-90 a remainder can underflow only for |x| < 2^-100, where the
// quotient is below 2^-10 and every code it can round to is zero.  Checked
// against double-precision division on 2e8 random (bf16, float) pairs:
// equal wherever a code could differ.
struct ExactDivisor {
  float s, y;
  bool fast;
  __device__ __forceinline__ explicit ExactDivisor(float s_) : s(s_) {
    fast = s_ >= 0x1p-90f && s_ <= 0x1p100f;  // false for NaN too
    y = fast ? __frcp_rn(s_) : 0.f;
  }
  // Requires `fast` and a finite quotient below 2^126.
  __device__ __forceinline__ float div_fast(float x) const {
    const float q0 = __fmul_rn(x, y);
    return __fmaf_rn(-__fmaf_rn(q0, s, -x), y, q0);
  }
  // Any x: quotients of 2^126 and beyond (and NaN) come back as x * y, every
  // code saturating there as it does for the division's result.
  __device__ __forceinline__ float div(float x) const {
    if (!fast) return __fdiv_rn(x, s);
    const float q0 = __fmul_rn(x, y);
    if (!(fabsf(q0) < 0x1p126f)) return q0;
    return __fmaf_rn(-__fmaf_rn(q0, s, -x), y, q0);
  }
};

// max |x| over eight bf16 values.
__device__ __forceinline__ float bf16x8_amax(const uint4& v) {
  float a = 0.f;
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) a = fmaxf(a, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
  return a;
}

// The global scale from the tensor's amax.
__device__ __forceinline__ float nvfp4_global_from_amax(float amax) {
  return (amax == 0.f) ? 1.f : __fdiv_rn(amax, 2688.f);
}

// The block encoder for one global scale g, its divisors prepared once.
// One 16-element block (v0: elements 0-7, v1: 8-15): its eight code bytes
// (element i in nibble i of the 64 bits, low word first) and its E4M3 scale
// byte; *dec receives the scale's exact value.  (amax_b / 6) / g stays two
// IEEE divisions per block (with the reciprocal form measured no faster).
struct Nvfp4BlockEncoder {
  float g;
  __device__ __forceinline__ explicit Nvfp4BlockEncoder(float g_) : g(g_) {}

  __device__ __forceinline__ uint32_t block(const uint4& v0, const uint4& v1, uint32_t& code_lo,
                                            uint32_t& code_hi, float* dec) const {
    const float amax_b = fmaxf(bf16x8_amax(v0), bf16x8_amax(v1));
    const float t = __fdiv_rn(__fdiv_rn(amax_b, 6.f), g);
    const uint32_t sfc = cvt_e4m3x2(t, t) & 0xFFu;
    const float2 dd = e4m3x2_to_float2(static_cast<uint16_t>(sfc));  // one byte is zero
    const float sv = fmaxf(dd.x, dd.y);
    const float d = __fmul_rn(sv, g);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    // |x| <= amax_b and d >= dec(sf) * g with sf the rounded (amax_b / 6) / g,
    // so the quotients stay below 2^126.
    const ExactDivisor dv(d);
    float q[16];
    if (dv.fast) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        q[2 * i] = dv.div_fast(bf16_lo(w[i]));
        q[2 * i + 1] = dv.div_fast(bf16_hi(w[i]));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        q[2 * i] = (d == 0.f) ? 0.f : __fdiv_rn(bf16_lo(w[i]), d);
        q[2 * i + 1] = (d == 0.f) ? 0.f : __fdiv_rn(bf16_hi(w[i]), d);
      }
    }
    code_lo = cvt_e2m1x8(*reinterpret_cast<const float(*)[8]>(&q[0]));
    code_hi = cvt_e2m1x8(*reinterpret_cast<const float(*)[8]>(&q[8]));
    *dec = sv;
    return sfc;
  }
};

}  // namespace spg
